"""Benchmark of the W12 decode-GEMM on GB300.

One step = one pass of the hot path over one batch: the seven GEMMs of the
27B-class decoder layer (q 6144x5120, k/v 1024x5120, o 5120x6144, gate/up
17408x5120, down 5120x17408) at M tokens (default 1), weights resident in HBM
in W12 form, activations resident, outputs BF16.  Synthetic, seeded inputs.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle
(decode + fp64 dot products on the host cores) on a bounded sample instead.
Under torchrun every rank runs an independent replica (the path shards by
rows but the single-GPU workload is replicated: weak scaling, no collective
on the data path); value = all ranks' work / max rank time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "W12 decode-GEMM effective weight GB/s & µs/layer at M=1–32; % of HBM peak"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ("lossless_bit_weight_encode_gb300/csrc/gemm_tc.cuh",
                  "lossless_bit_weight_encode_gb300/csrc/gemv.cuh",
                  "lossless_bit_weight_encode_gb300/csrc/gemv_sm.cuh",
                  "lossless_bit_weight_encode_gb300/csrc/w12_device.cuh",
                  "lossless_bit_weight_encode_gb300/csrc/kernels.cu")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="w12", choices=["w12", "reference"])
    ap.add_argument("--m", type=int, default=1, help="tokens per GEMM (1..32)")
    ap.add_argument("--workload", default="layer", choices=["layer", "heavy", "model64", "lmhead"])
    ap.add_argument("--weights", default="w12", choices=["w12", "q8"],
                    help="w12: the lossless format; q8: the 8-bit verification copy of the same weights")
    ap.add_argument("--no-group", action="store_true",
                    help="one launch per matrix instead of q/k/v and gate/up as grouped launches")
    ap.add_argument("--graph", action="store_true", help="replay the step as a CUDA graph")
    ap.add_argument("--no-bf16", action="store_true", help="skip the cuBLAS BF16 comparator")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-baseline leg")
    ap.add_argument("--out", default=None, help="also append the JSON line to this file")
    ap.add_argument("--matrices", default=None,
                    help="comma list of layer matrices to run (profiling only; default all seven)")
    return ap.parse_args()


def kernel_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            return json.load(open(path)), "measured"
        except Exception:
            pass
    return None, "fallback"


def hbm_peak_gbs():
    peaks, kind = measured_peaks()
    if peaks:
        for key in ("hbm_gbs", "hbm_GBps", "hbm"):
            v = peaks.get(key)
            if isinstance(v, dict):
                v = v.get("burst") or v.get("value")
            if isinstance(v, (int, float)) and v > 0:
                return float(v), "of measured"
    return FALLBACK_HBM_GBS, "of fallback"


def recorded_traffic():
    """Per-launch DRAM bytes of the GEMM kernel from the committed ncu summary,
    only while the kernel sources still hash to what was profiled."""
    path = os.path.join(ROOT, "profiles", "w12_layer_m1_traffic.json")
    if not os.path.exists(path):
        return None
    try:
        rec = json.load(open(path))
    except Exception:
        return None
    if rec.get("kernel_hash") != kernel_hash():
        return None
    return rec


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        except Exception:
            pass
        finally:
            try:
                os.unlink(self.path)
            except Exception:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_median": statistics.median([float(r[3]) for r in rows
                                                     if r[3].replace(".", "").isdigit()] or [0.0])}


WORKLOAD_TEXT = {
    "layer": "layer: 27B-class decoder layer (q 6144x5120, k/v 1024x5120, o 5120x6144, gate/up 17408x5120, "
             "down 5120x17408; 340.8 M weights), weights N(0,0.02)",
    "heavy": "heavy: layer shapes, Student-t(3)*0.02 weights with 0.5% x100 outliers",
    "lmhead": "lmhead: LM head 151936x5120 (vocabulary x hidden), weights N(0,0.02), GEMM with the fused "
              "exact-argmax epilogue (per-token index and fp32 logit; logits not stored)",
    "model64": "model64: 64 layers of the 27B-class shapes chained in layer order (448 GEMMs, 21.8 G weights, "
               "32.7 GB of W12 resident), weights N(0,0.02) drawn and encoded on the GPU",
}


# ------------------------------------------------------------------ CPU oracle
class OracleSample:
    """The oracle (its own encoder for the blobs, then decode + fp64 dot
    products with OpenMP over the host cores) on a bounded sample: whole layer
    matrices in order until the time budget is spent."""

    def __init__(self, weights, xs, m):
        import oracle

        oracle.build()
        self.oracle = oracle
        self.weights, self.xs, self.m = weights, xs, m
        self.blobs = {}
        self.cores = oracle.max_threads(0)

    def run(self, max_seconds, start=0):
        """Whole matrices, cycling from `start`, until `max_seconds` of wall
        time have been spent (at least one matrix)."""
        done_w, spent, names, i = 0, 0.0, [], start
        while True:
            j = i % len(self.weights)
            name, w = self.weights[j]
            if j not in self.blobs:
                self.blobs[j] = self.oracle.encode(w)  # untimed
            t0 = time.perf_counter()
            self.oracle.w12_gemm_f64(self.xs[j], self.blobs[j], threads=0)
            spent += time.perf_counter() - t0
            done_w += w.size
            names.append(name)
            i += 1
            if spent > max_seconds:
                break
        gbs = 2.0 * done_w / spent / 1e9
        sample = (f"{len(names)} layer matrices at M={self.m} ({'+'.join(names[:7])}"
                  f"{'...' if len(names) > 7 else ''}): {done_w / 1e6:.1f} M weights in {spent:.2f} s "
                  f"(oracle encode untimed; W12 decode + fp64 dot products timed)")
        return gbs, sample, done_w, spent


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from lossless_bit_weight_encode_gb300 import workloads as wl

    if args.workload == "model64":
        # its weights come from the GPU's generator; the host-only arm times
        # the oracle on the layer workload's matrices of the same shapes
        args.workload = "layer"
    if args.workload == "lmhead":
        name, n, k = wl.LMHEAD_SHAPE
        weights = [(name, wl.gaussian_weights(n, k, seed=wl.weight_seed("lmhead", 0)))]
    else:
        weights = list(wl.layer_weights(args.workload))
    xs = [wl.activations(args.m, w.shape[1], seed=wl.activation_seed(args.workload, args.m)) for _, w in weights]
    orc = OracleSample(weights, xs, args.m)
    # one step = one layer matrix (cycling q, k, v, o, gate, up, down): a
    # bounded sample so that K + W steps stay within a few minutes
    tot_w, tot_s = 0, 0.0
    for i in range(args.warmup + args.steps):
        _, sample, w_i, s_i = orc.run(0.0, start=i)
        if i >= args.warmup:
            tot_w += w_i
            tot_s += s_i
    value = 2.0 * tot_w / tot_s / 1e9
    sample = (f"one layer matrix per step, cycling the 7 (q..down) at M={args.m}: {tot_w / 1e6:.1f} M weights "
              f"in {tot_s:.2f} s over {args.steps} steps (oracle encode untimed)")
    layer_w = sum(w.size for _, w in weights)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(2.0 * layer_w / (value * 1e9) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: 27B-class decoder layer, 7 matrices, 340.8 M weights",
                   "M": args.m, "parallelism": "host cores (OpenMP)",
                   "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": orc.cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    emit(line, args)


def emit(line, args):
    s = json.dumps(line)
    print(s, flush=True)
    if args.out:
        with open(args.out, "a") as f:
            f.write(s + "\n")


def max_over_ranks(value: float, device) -> float:
    """The largest of `value` over the ranks of the default process group (the
    job takes as long as its slowest replica); `value` itself without one."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_weight_gbs(weights_per_rank: int, world: int, ms: float) -> float:
    """Whole-job BF16-equivalent weight GB/s: every replica streams the same
    weights once per step, so the job moves world x 2 bytes per weight."""
    return world * 2.0 * weights_per_rank / (ms * 1e-3) / 1e9


# ------------------------------------------------------------------ GPU arm
def run_w12(args):
    import torch
    import torch.distributed as dist

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if args.graph:
        # stream capture needs a stream other than the legacy default one
        torch.cuda.set_stream(torch.cuda.Stream())
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    from lossless_bit_weight_encode_gb300 import Q8Weight, W12Group, W12Weight, w12
    from lossless_bit_weight_encode_gb300 import build as libbuild
    from lossless_bit_weight_encode_gb300 import workloads as wl

    libbuild.build()
    M = args.m
    nshape = len(wl.LAYER_SHAPES)
    if args.workload == "model64":
        # 64 layers drawn and encoded on the GPU (W12Weight.from_device); one
        # activation per shape, shared by every layer; one workspace per shape
        # (the launches are ordered on one stream)
        names = [f"L{layer}.{n}" for layer in range(wl.MODEL64_LAYERS) for n, _, _ in wl.LAYER_SHAPES]
        mats = []
        for layer in range(wl.MODEL64_LAYERS):
            for idx in range(nshape):
                w = wl.model64_weight_dev(layer, idx)
                mats.append(W12Weight.from_device(w))
                del w
        xs_shape = [wl.model64_activation(M, i) for i in range(nshape)]
        xs_host = [xs_shape[i % nshape] for i in range(len(mats))]
        xs_dev = [torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16) for x in xs_shape]
        xs = [xs_dev[i % nshape] for i in range(len(mats))]
        ws_shape = [mats[i].workspace(M) for i in range(nshape)]
        wss = [ws_shape[i % nshape] for i in range(len(mats))]

        def dense_weights():
            for layer in range(wl.MODEL64_LAYERS):
                for idx in range(nshape):
                    yield wl.model64_weight_dev(layer, idx)

        def cpu_weights():
            return [(n, wl.model64_weight_dev(0, i).view(torch.int16).cpu().numpy().view(np.uint16))
                    for i, (n, _, _) in enumerate(wl.LAYER_SHAPES)]
    else:
        if args.workload == "lmhead":
            name, n, k = wl.LMHEAD_SHAPE
            weights = [(name, wl.gaussian_weights(n, k, seed=wl.weight_seed("lmhead", 0)))]
        else:
            weights = list(wl.layer_weights(args.workload))
        if args.matrices:
            keep = set(args.matrices.split(","))
            weights = [(n, w) for n, w in weights if n in keep]
        names = [n for n, _ in weights]
        mats = [Q8Weight(w) if args.weights == "q8" else W12Weight(w) for _, w in weights]
        xs_host = [wl.activations(M, w.shape[1], seed=wl.activation_seed(args.workload, M)) for _, w in weights]
        # every matrix's x in one device buffer (256-byte aligned slices), so
        # that the end-to-end run brings a step's inputs in with one copy
        offs, tot = [], 0
        for x in xs_host:
            offs.append(tot)
            tot += (x.size + 127) // 128 * 128
        xpack_host = np.zeros(tot, dtype=np.uint16)
        for o, x in zip(offs, xs_host):
            xpack_host[o:o + x.size] = x.ravel()
        xpack = torch.from_numpy(xpack_host.view(np.int16)).cuda().view(torch.bfloat16)
        xs = [xpack[o:o + x.size].view(x.shape) for o, x in zip(offs, xs_host)]
        wss = [m.workspace(M) for m in mats]

        def dense_weights():
            for _, w in weights:
                yield torch.from_numpy(w.view(np.int16)).cuda().view(torch.bfloat16)

        def cpu_weights():
            return weights
    # all outputs in one device buffer: one copy brings a step's results back
    ypack = torch.empty(sum(M * m.N for m in mats), dtype=torch.bfloat16, device="cuda")
    yoffs = np.cumsum([0] + [M * m.N for m in mats])
    ys = [ypack[yoffs[i]:yoffs[i + 1]].view(M, m.N) for i, m in enumerate(mats)]
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    argmax = args.workload == "lmhead"
    if argmax:
        # the LM head: GEMM with the fused argmax epilogue (no logits stored)
        idx = torch.empty(M, dtype=torch.int32, device="cuda")
        val = torch.empty(M, dtype=torch.float32, device="cuda")
        aws = [m.argmax_workspace(M) for m in mats]
        calls = [(x.data_ptr(), m.blob.data_ptr(), m.info, M, None, idx.data_ptr(), val.data_ptr(), ws.data_ptr(),
                  ws.numel(), sh) for x, m, ws in zip(xs, mats, aws)]
        launch = w12.w12_gemm_argmax_ptr
        groups = [[i] for i in range(len(mats))]
    else:
        # q, k, v multiply the same x, and so do gate and up: one launch each
        layer_names = [n for n, _, _ in wl.LAYER_SHAPES]
        layers = len(mats) // len(layer_names)
        if args.workload == "model64":
            whole_layers = True
        else:
            whole_layers = args.workload in ("layer", "heavy") and names == layer_names
        grouped = not args.no_group and args.weights == "w12" and whole_layers
        per_layer = [[0, 1, 2], [3], [4, 5], [6]]
        groups = ([[7 * l + i for i in g] for l in range(layers) for g in per_layer] if grouped
                  else [[i] for i in range(len(mats))])
        calls = []
        group_ws = []  # keeps the group workspaces alive for the raw pointers below
        for g in groups:
            if len(g) == 1:
                i = g[0]
                calls.append((w12.w12_q8_gemm_ptr if args.weights == "q8" else w12.w12_gemm_ptr,
                              (xs[i].data_ptr(), mats[i].blob.data_ptr(), mats[i].info, ys[i].data_ptr(), M,
                               wss[i].data_ptr(), wss[i].numel(), sh)))
            else:
                grp = W12Group([mats[i] for i in g])
                gws = grp.workspace(M)
                group_ws.append((grp, gws))
                calls.append((w12.w12_gemm_group_ptr,
                              (xs[g[0]].data_ptr(), [mats[i].blob.data_ptr() for i in g], grp.infos,
                               [ys[i].data_ptr() for i in g], M, gws.data_ptr(), gws.numel(), sh)))
    if argmax:
        calls = [(launch, c) for c in calls]
        groups = [[i] for i in range(len(mats))]
    names_launch = ["+".join(names[i] for i in g) for g in groups]

    def step():
        for fn, c in calls:
            rc = fn(*c)
            if rc != 0:
                raise w12.W12Error(rc, w12.w12_last_error())

    graph = None
    if args.graph:
        step()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
        run_step = graph.replay
    else:
        run_step = step

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        run_step()
    w12.w12_check_status()
    barrier()

    # main timed region: K steps between two events
    K = args.steps
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        ev0.record()
        for _ in range(K):
            run_step()
        ev1.record()
        ev1.synchronize()
    barrier()
    ms_total = ev0.elapsed_time(ev1)
    w12.w12_check_status()
    ms_total = max_over_ranks(ms_total, "cuda")
    ms_step = ms_total / K

    # per-launch durations of the GEMM kernel (events around every launch)
    nl = len(calls)
    kp = max(10, min(K, 500 if nl <= 7 else 20))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nl + 1)] for _ in range(kp)]
    barrier()
    for k in range(kp):
        for i, (fn, c) in enumerate(calls):
            evs[k][i].record()
            rc = fn(*c)
            if rc != 0:
                raise w12.W12Error(rc, w12.w12_last_error())
        evs[k][nl].record()
    torch.cuda.synchronize()
    w12.w12_check_status()
    launch_ms = [statistics.mean(evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(kp)) for i in range(nl)]

    if args.weights == "q8":
        kernel_name = "w12_gemm_tc_kernel (Q8 copy)"
    else:
        plan0 = w12.w12_gemm_launch_info(mats[0].info, M)
        kernel_name = "w12_gemm_tc_kernel" if plan0.get("ntok") > 4 else \
            "w12_gemv_sm_kernel" if plan0.get("ctas_per_sm") == 1 else "w12_gemv_kernel"
    layer_weights = sum(m.N * m.K for m in mats)
    packed = sum(int(m.info.total_bytes) for m in mats)
    alg = [sum(int(mats[i].info.total_bytes) + 2 * M * mats[i].N for i in g) + 2 * M * mats[g[0]].K
           for g in groups]  # per launch: its blobs, one x, its outputs
    value = job_weight_gbs(layer_weights, world, ms_step)
    peak, peak_kind = hbm_peak_gbs()
    achieved = sum(alg) / (sum(launch_ms) * 1e-3) / 1e9
    traffic_rec = recorded_traffic()
    traffic = None
    if traffic_rec is not None and traffic_rec.get("M") == M and traffic_rec.get("workload") == args.workload:
        traffic = traffic_rec.get("dram_bytes_per_launch")

    # BF16 comparator (cuBLAS through torch.matmul), same shapes and x
    bf16 = None
    if not args.no_bf16:
        dense = list(dense_weights())
        # the same grouping for cuBLAS: one matmul over the concatenated weights
        wts = [torch.cat([dense[i] for i in g], dim=0) if len(g) > 1 else dense[g[0]] for g in groups]
        del dense
        xb = [xs[g[0]] for g in groups]
        outs = [torch.empty((M, w.shape[0]), dtype=torch.bfloat16, device="cuda") for w in wts]

        def bstep():
            for x, wt, o in zip(xb, wts, outs):
                torch.matmul(x, wt.t(), out=o)
                if argmax:
                    torch.argmax(o, dim=1)

        for _ in range(args.warmup):
            bstep()
        barrier()
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record()
        for _ in range(K):
            bstep()
        b1.record()
        b1.synchronize()
        bf16 = b0.elapsed_time(b1) / K
        del wts, outs

    # end to end through the public API with host buffers: x from pinned host
    # memory in, y back to pinned host memory, every step
    e2e = None
    if not args.no_e2e:
        xh = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory() for x in xs_host]
        yh = [torch.empty((M, m.N), dtype=torch.bfloat16).pin_memory() for m in mats]
        one_copy = args.workload != "model64" and not argmax
        if one_copy:
            xpack_h = torch.from_numpy(xpack_host.view(np.int16)).view(torch.bfloat16).pin_memory()
            ypack_h = torch.empty(ypack.numel(), dtype=torch.bfloat16).pin_memory()
        if argmax:
            idx_h = torch.empty(M, dtype=torch.int32).pin_memory()

        def estep():
            if one_copy:
                # the step's inputs in, its launches, its outputs out: one copy each way
                xpack.copy_(xpack_h, non_blocking=True)
                for fn, c in calls:
                    rc = fn(*c)
                    if rc != 0:
                        raise w12.W12Error(rc, w12.w12_last_error())
                ypack_h.copy_(ypack, non_blocking=True)
                return
            # x comes in once per launch (the members of a group share it)
            for (fn, c), g in zip(calls, groups):
                xs[g[0]].copy_(xh[g[0]], non_blocking=True)
                rc = fn(*c)
                if rc != 0:
                    raise w12.W12Error(rc, w12.w12_last_error())
                if argmax:
                    idx_h.copy_(idx, non_blocking=True)
                else:
                    for i in g:
                        yh[i].copy_(ys[i], non_blocking=True)

        for _ in range(args.warmup):
            estep()
        barrier()
        ke = max(10, min(K, 1000))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(ke):
            estep()
        e1.record()
        e1.synchronize()
        w12.w12_check_status()
        e_ms = max_over_ranks(e0.elapsed_time(e1) / ke, "cuda")
        e2e = {"value": round(job_weight_gbs(layer_weights, world, e_ms), 2), "unit": "GB/s",
               "h2d_bytes_per_step": int(2 * xpack_h.numel()) if one_copy else int(sum(2 * M * mats[g[0]].K for g in groups)),
               "d2h_bytes_per_step": int(4 * M) if argmax else int(sum(2 * M * m.N for m in mats)),
               "ms_per_step": round(e_ms, 5)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        orc = OracleSample(cpu_weights(), xs_host[:nshape] if args.workload == "model64" else xs_host, M)
        v, sample, _, _ = orc.run(3.0)
        cpu = {"value": round(v, 4), "unit": "GB/s", "cores": orc.cores, "kind": "oracle", "sample": sample}

    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return
    csum = clocks.summary()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {
            "workload": WORKLOAD_TEXT[args.workload],
            "M": M, "global_batch": M * world, "parallelism": f"replicas x{world}",
            "l2": f"inputs larger than L2: {packed / 1e6:.1f} MB of W12 streamed per step (L2 129 MB)",
            "launch": ("cuda graph" if graph is not None else "stream") + f" ({nl} launches per step: "
                      + ", ".join(names_launch[:7]) + ("..." if nl > 7 else "") + ")",
        },
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind, "traffic": traffic,
                     "algorithmic_bytes_per_launch": round(sum(alg) / nl),
                     "kernel": kernel_name, "launch_us": [round(v * 1e3, 2) for v in launch_ms]},
        "cpu_baseline": cpu,
        "clocks": csum,
        "e2e": e2e,
        "gpu_launches": K * nl * (2 if argmax else 1),
        "detail": {
            "us_per_layer": round(ms_step * 1e3 / (wl.MODEL64_LAYERS if args.workload == "model64" else 1), 2),
            "layers_per_step": wl.MODEL64_LAYERS if args.workload == "model64" else 1,
            "packed_GBps": round(packed / (ms_step * 1e-3) / 1e9, 1),
            "packed_frac_of_hbm_peak": round(packed / (ms_step * 1e-3) / 1e9 / peak, 4),
            "bits_per_weight": round(8.0 * packed / layer_weights, 5),
            "n_escapes": int(sum(int(getattr(m.info, "n_escapes", 0)) for m in mats)),
            "weights": args.weights,
            "per_matrix_us": {n: round(statistics.mean(launch_ms[i::nshape]) * 1e3, 2)
                              for i, (n, _, _) in enumerate(wl.LAYER_SHAPES)}
                             if args.workload == "model64" else
                             {n: round(v * 1e3, 2) for n, v in zip(names_launch, launch_ms)},
            "bf16_cublas_us_per_layer": round(bf16 * 1e3 / (wl.MODEL64_LAYERS if args.workload == "model64"
                                                            else 1), 2) if bf16 else None,
            "speedup_vs_bf16": round(bf16 / ms_step, 4) if bf16 else None,
        },
    }
    emit(line, args)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_w12(args)


if __name__ == "__main__":
    main()
