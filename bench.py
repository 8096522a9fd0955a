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
                  "lossless_bit_weight_encode_gb300/csrc/gemm_tc_sm.cuh",
                  "lossless_bit_weight_encode_gb300/csrc/gemv.cuh",
                  "lossless_bit_weight_encode_gb300/csrc/gemv_sm.cuh",
                  "lossless_bit_weight_encode_gb300/csrc/w12_device.cuh",
                  "lossless_bit_weight_encode_gb300/csrc/kernels.cu")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="w12", choices=["w12", "reference"])
    ap.add_argument("--m", type=int, default=1, help="tokens per GEMM (1..32)")
    ap.add_argument("--workload", default="layer", choices=["layer", "heavy", "model64", "lmhead", "single"])
    ap.add_argument("--weights", default="w12", choices=["w12", "q8"],
                    help="w12: the lossless format; q8: the 8-bit verification copy of the same weights")
    ap.add_argument("--no-group", action="store_true",
                    help="one launch per matrix instead of q/k/v and gate/up as grouped launches")
    ap.add_argument("--graph", action="store_true", help="replay the step as a CUDA graph")
    ap.add_argument("--no-bf16", action="store_true", help="skip the cuBLAS BF16 comparator")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-baseline leg")
    ap.add_argument("--no-detail", action="store_true",
                    help="skip the other configurations (M sweep, heavy tail, single layer, decode) that the "
                         "default layer run at M=1 adds under detail")
    ap.add_argument("--opt", action="append", default=[], metavar="NAME=VALUE",
                    help="set a library launch option (w12_set_option) for the run, e.g. --opt tc_sm=0; repeatable")
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
    "single": "single: one 1024x1024 layer, weights N(0,0.02), x[1,1024] N(0,1), PCG64 seed 0 (W then x)",
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

    def run(self, max_seconds, start=0, threads=0):
        """Whole matrices, cycling from `start`, until `max_seconds` of wall
        time have been spent (at least one matrix); `threads` OpenMP threads
        (0: all host cores)."""
        done_w, spent, names, i = 0, 0.0, [], start
        while True:
            j = i % len(self.weights)
            name, w = self.weights[j]
            if j not in self.blobs:
                self.blobs[j] = self.oracle.encode(w)  # untimed
            t0 = time.perf_counter()
            self.oracle.w12_gemm_f64(self.xs[j], self.blobs[j], threads=threads)
            spent += time.perf_counter() - t0
            done_w += w.size
            names.append(name)
            i += 1
            if spent > max_seconds:
                break
        gbs = 2.0 * done_w / spent / 1e9
        sample = (f"{len(names)} layer matrices at M={self.m} ({'+'.join(names[:7])}"
                  f"{'...' if len(names) > 7 else ''}): {done_w / 1e6:.1f} M weights in {spent:.2f} s "
                  f"(oracle encode untimed; W12 decode + fp64 dot products timed; "
                  f"{self.oracle.max_threads(threads)} threads)")
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
    elif args.workload == "single":
        w1, x1 = wl.single_case()
        weights = [("single", w1)]
    else:
        weights = list(wl.layer_weights(args.workload))
    if args.workload == "single" and args.m == 1:
        xs = [x1]
    else:
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
    sample = (f"one matrix per step, cycling {'+'.join(n for n, _ in weights)} at M={args.m}: "
              f"{tot_w / 1e6:.1f} M weights in {tot_s:.2f} s over {args.steps} steps (oracle encode untimed)")
    layer_w = sum(w.size for _, w in weights)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(2.0 * layer_w / (value * 1e9) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.workload], "M": args.m, "parallelism": "host cores (OpenMP)",
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
def bootstrap_median_ci(samples, n_boot: int = 2000, seed: int = 0):
    """Median of `samples` and a 95 % percentile-bootstrap interval for it."""
    a = np.asarray(samples, dtype=np.float64)
    rng = np.random.default_rng(seed)
    meds = np.median(a[rng.integers(0, a.size, size=(n_boot, a.size))], axis=1)
    return float(np.median(a)), float(np.percentile(meds, 2.5)), float(np.percentile(meds, 97.5))


class LayerStep:
    """The launches of one step over a list of W12 (or Q8) matrices at M
    tokens: q/k/v and gate/up grouped when the list is a whole layer (or 64),
    one launch per matrix otherwise.  Activations and outputs live in one
    device buffer each, so the end-to-end leg moves them with one copy each
    way."""

    def __init__(self, mats, names, xs_host, M, grouped, q8=False, argmax=False):
        import torch
        from lossless_bit_weight_encode_gb300 import Q8Group, W12Group, w12

        self.w12 = w12
        self.mats, self.names, self.M = mats, names, M
        self.xs_host = xs_host
        offs, tot = [], 0
        for x in xs_host:
            offs.append(tot)
            tot += (x.size + 127) // 128 * 128
        self.xpack_host = np.zeros(tot, dtype=np.uint16)
        for o, x in zip(offs, xs_host):
            self.xpack_host[o:o + x.size] = x.ravel()
        self.xpack = torch.from_numpy(self.xpack_host.view(np.int16)).cuda().view(torch.bfloat16)
        self.xs = [self.xpack[o:o + x.size].view(x.shape) for o, x in zip(offs, xs_host)]
        self.ypack = torch.empty(sum(M * m.N for m in mats), dtype=torch.bfloat16, device="cuda")
        yoffs = np.cumsum([0] + [M * m.N for m in mats])
        self.ys = [self.ypack[yoffs[i]:yoffs[i + 1]].view(M, m.N) for i, m in enumerate(mats)]
        self.argmax = argmax
        sh = torch.cuda.current_stream().cuda_stream
        self.keep = []
        if argmax:
            self.idx = torch.empty(M, dtype=torch.int32, device="cuda")
            self.val = torch.empty(M, dtype=torch.float32, device="cuda")
            self.groups = [[i] for i in range(len(mats))]
            self.calls = []
            for i, m in enumerate(mats):
                ws = m.argmax_workspace(M)
                self.calls.append((w12.w12_gemm_argmax_ptr,
                                   (self.xs[i].data_ptr(), m.blob.data_ptr(), m.info, M, None, self.idx.data_ptr(),
                                    self.val.data_ptr(), ws.data_ptr(), ws.numel(), sh)))
        else:
            n7 = len(LAYER_NAMES)
            if grouped:
                per_layer = [[0, 1, 2], [3], [4, 5], [6]]
                self.groups = [[n7 * l + i for i in g] for l in range(len(mats) // n7) for g in per_layer]
            else:
                self.groups = [[i] for i in range(len(mats))]
            self.calls = []
            for g in self.groups:
                if len(g) == 1:
                    i = g[0]
                    ws = mats[i].workspace(M)
                    self.calls.append((w12.w12_q8_gemm_ptr if q8 else w12.w12_gemm_ptr,
                                       (self.xs[i].data_ptr(), mats[i].blob.data_ptr(), mats[i].info,
                                        self.ys[i].data_ptr(), M, ws.data_ptr(), ws.numel(), sh)))
                else:
                    grp = (Q8Group if q8 else W12Group)([mats[i] for i in g])
                    gws = grp.workspace(M)
                    self.keep.append((grp, gws))
                    self.calls.append((w12.w12_q8_gemm_group_ptr if q8 else w12.w12_gemm_group_ptr,
                                       (self.xs[g[0]].data_ptr(), [mats[i].blob.data_ptr() for i in g], grp.infos,
                                        [self.ys[i].data_ptr() for i in g], M, gws.data_ptr(), gws.numel(), sh)))
        self.launch_names = ["+".join(names[i] for i in g) for g in self.groups]
        # algorithmic bytes of each launch: its blobs, one x (shared by a
        # group), its outputs (the argmax keys and results are a few bytes)
        self.alg = [sum(int(mats[i].info.total_bytes) + (0 if argmax else 2 * M * mats[i].N) for i in g)
                    + 2 * M * mats[g[0]].K for g in self.groups]
        self.packed = sum(int(m.info.total_bytes) for m in mats)
        self.weights = sum(m.N * m.K for m in mats)
        if q8:
            self.kernels = [w12.w12_q8_gemm_group_launch_info([mats[i].info for i in g], M)["kernel_name"]
                            + " (Q8 copy)" for g in self.groups]
        else:
            self.kernels = [w12.w12_gemm_group_launch_info([mats[i].info for i in g], M)["kernel_name"]
                            for g in self.groups]

    def launch_count(self) -> int:
        return len(self.calls) * (2 if self.argmax else 1)

    def run(self):
        for fn, c in self.calls:
            rc = fn(*c)
            if rc != 0:
                raise self.w12.W12Error(rc, self.w12.w12_last_error())

    def run_e2e(self, xpack_h, ypack_h, idx_h):
        """x in from pinned host memory, the launches, the outputs back."""
        self.xpack.copy_(xpack_h, non_blocking=True)
        self.run()
        if self.argmax:
            idx_h.copy_(self.idx, non_blocking=True)
        else:
            ypack_h.copy_(self.ypack, non_blocking=True)


LAYER_NAMES = ("q", "k", "v", "o", "gate", "up", "down")


def time_steps(run, K: int) -> float:
    """ms per call of `run` over K calls between two events on the current stream."""
    import torch
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        run()
    e1.record()
    e1.synchronize()
    return e0.elapsed_time(e1) / K


def step_samples(run, R: int):
    """Per-call ms of R consecutive calls (one event between each)."""
    import torch
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(R + 1)]
    evs[0].record()
    for r in range(R):
        run()
        evs[r + 1].record()
    evs[R].synchronize()
    return [evs[r].elapsed_time(evs[r + 1]) for r in range(R)]


def launch_times(step: LayerStep, reps: int):
    """Mean ms of each launch of the step, events around every launch."""
    import torch
    nl = len(step.calls)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nl + 1)] for _ in range(reps)]
    torch.cuda.synchronize()
    for k in range(reps):
        for i, (fn, c) in enumerate(step.calls):
            evs[k][i].record()
            rc = fn(*c)
            if rc != 0:
                raise step.w12.W12Error(rc, step.w12.w12_last_error())
        evs[k][nl].record()
    torch.cuda.synchronize()
    return [statistics.mean(evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(reps)) for i in range(nl)]


def cublas_ms(dense, groups, xs, K: int, warmup: int, argmax=False) -> float:
    """torch.matmul (cuBLAS BF16) over the same shapes, x and grouping."""
    import torch
    wts = [torch.cat([dense[i] for i in g], dim=0) if len(g) > 1 else dense[g[0]] for g in groups]
    xb = [xs[g[0]] for g in groups]
    outs = [torch.empty((x.shape[0], w.shape[0]), dtype=torch.bfloat16, device="cuda") for x, w in zip(xb, wts)]

    def bstep():
        for x, wt, o in zip(xb, wts, outs):
            torch.matmul(x, wt.t(), out=o)
            if argmax:
                torch.argmax(o, dim=1)

    for _ in range(warmup):
        bstep()
    return time_steps(bstep, K)


def dense_dev(weights):
    import torch
    return [torch.from_numpy(w.view(np.int16)).cuda().view(torch.bfloat16) for _, w in weights]


def sweep_point(mats, weights, xs_host, M, K, warmup, dense, q8=False):
    """µs per layer step at M tokens, the packed fraction of the HBM peak and
    the cuBLAS BF16 step on the same shapes and grouping."""
    peak, _ = hbm_peak_gbs()
    st = LayerStep(mats, [n for n, _ in weights], xs_host, M, grouped=True, q8=q8)
    for _ in range(warmup):
        st.run()
    ms = time_steps(st.run, K)
    st.w12.w12_check_status()
    med, lo, hi = bootstrap_median_ci(step_samples(st.run, max(50, K)))
    lt = launch_times(st, 20)
    st.w12.w12_check_status()
    out = {"us_per_layer": round(ms * 1e3, 2), "median_us": round(med * 1e3, 2),
           "ci95_us": [round(lo * 1e3, 2), round(hi * 1e3, 2)],
           "packed_frac_of_hbm_peak": round(st.packed / (ms * 1e-3) / 1e9 / peak, 4),
           "kernels": sorted(set(st.kernels)),
           "per_launch_us": {n: round(v * 1e3, 2) for n, v in zip(st.launch_names, lt)}}
    if dense is not None:
        b = cublas_ms(dense, st.groups, st.xs, K, warmup)
        out["bf16_cublas_us"] = round(b * 1e3, 2)
        out["speedup_vs_bf16"] = round(b / ms, 4)
    return out


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

    from lossless_bit_weight_encode_gb300 import Q8Weight, W12Weight, w12
    from lossless_bit_weight_encode_gb300 import build as libbuild
    from lossless_bit_weight_encode_gb300 import workloads as wl

    libbuild.build()
    for o in args.opt:
        name, _, value = o.partition("=")
        w12.w12_set_option(name, int(value))
    M = args.m
    K = args.steps
    nshape = len(wl.LAYER_SHAPES)
    peak, peak_kind = hbm_peak_gbs()
    if args.workload == "model64":
        # 64 layers drawn and encoded on the GPU (W12Weight.from_device); one
        # activation per shape, shared by every layer
        names = [f"L{layer}.{n}" for layer in range(wl.MODEL64_LAYERS) for n, _, _ in wl.LAYER_SHAPES]
        mats = []
        for layer in range(wl.MODEL64_LAYERS):
            for idx in range(nshape):
                w = wl.model64_weight_dev(layer, idx)
                mats.append(W12Weight.from_device(w))
                del w
        xs_shape = [wl.model64_activation(M, i) for i in range(nshape)]
        xs_host = [xs_shape[i % nshape] for i in range(len(mats))]
        step = LayerStep(mats, names, xs_host, M, grouped=not args.no_group)

        def dense_weights():
            return [wl.model64_weight_dev(layer, idx) for layer in range(wl.MODEL64_LAYERS)
                    for idx in range(nshape)]

        def cpu_weights():
            return [(n, wl.model64_weight_dev(0, i).view(torch.int16).cpu().numpy().view(np.uint16))
                    for i, (n, _, _) in enumerate(wl.LAYER_SHAPES)]
        cpu_xs = xs_shape
    elif args.workload == "single":
        # the 1024 x 1024 layer: its 1.5 MB blob fits in L2, so the step
        # rotates through enough encoded copies (3 x L2) that every call reads
        # its weights from HBM
        w, x = wl.single_case()
        base = W12Weight(w)
        l2 = torch.cuda.get_device_properties(local).L2_cache_size
        copies = max(1, -(-3 * l2 // int(base.info.total_bytes)))
        mats = [base]
        for _ in range(copies - 1):
            c = W12Weight.__new__(W12Weight)
            c.blob_host, c.info, c.N, c.K, c._ws = None, base.info, base.N, base.K, {}
            c.blob = base.blob.clone()
            mats.append(c)
        names = [f"single#{i}" for i in range(copies)]
        step = LayerStep(mats, names, [x] * copies, M, grouped=False)
        weights_single = [("single", w)]

        def dense_weights():
            d = dense_dev(weights_single)[0]
            return [d.clone() for _ in range(copies)]

        def cpu_weights():
            return weights_single
        cpu_xs = [x]
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
        q8 = args.weights == "q8"
        mats = [Q8Weight(w) if q8 else W12Weight(w) for _, w in weights]
        xs_host = [wl.activations(M, w.shape[1], seed=wl.activation_seed(args.workload, M)) for _, w in weights]
        whole = args.workload in ("layer", "heavy") and names == list(LAYER_NAMES)
        step = LayerStep(mats, names, xs_host, M, grouped=whole and not args.no_group, q8=q8,
                         argmax=args.workload == "lmhead")

        def dense_weights():
            return dense_dev(weights)

        def cpu_weights():
            return weights
        cpu_xs = xs_host

    graph = None
    run_step = step.run
    if args.graph:
        step.run()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=torch.cuda.current_stream()):
            step.run()
        run_step = graph.replay

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        run_step()
    w12.w12_check_status()
    barrier()

    # main timed region: exactly K steps between two events
    with ClockSampler(local) as clocks:
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record()
        for _ in range(K):
            run_step()
        ev1.record()
        ev1.synchronize()
        barrier()
        # per-step samples for the median and its bootstrap interval
        R = max(50, min(400, K))
        samples = step_samples(run_step, R)
    ms_total = ev0.elapsed_time(ev1)
    w12.w12_check_status()
    ms_total = max_over_ranks(ms_total, "cuda")
    ms_step = ms_total / K
    med, lo, hi = bootstrap_median_ci(samples)

    # per-launch durations (events around every launch; breaks the overlap
    # that programmatic dependent launch gives back to back)
    nl = len(step.calls)
    launch_ms = launch_times(step, max(10, min(K, 200 if nl <= 7 else 10)))
    w12.w12_check_status()
    lf = []
    for i in range(nl):
        lf.append({"launch": step.launch_names[i], "kernel": step.kernels[i], "us": round(launch_ms[i] * 1e3, 2),
                   "alg_bytes": int(step.alg[i]),
                   "frac": round(step.alg[i] / (launch_ms[i] * 1e-3) / 1e9 / peak, 4)})
    dom = max(range(nl), key=lambda i: launch_ms[i])
    achieved = step.alg[dom] / (launch_ms[dom] * 1e-3) / 1e9
    traffic_rec = recorded_traffic()
    traffic = None
    if traffic_rec is not None and traffic_rec.get("M") == M and traffic_rec.get("workload") == args.workload:
        traffic = (traffic_rec.get("per_launch_dram_bytes") or {}).get(step.launch_names[dom])

    # BF16 comparator (cuBLAS through torch.matmul), same shapes, x and grouping
    bf16 = None
    if not args.no_bf16:
        dense = dense_weights()
        bf16 = cublas_ms(dense, step.groups, step.xs, K, args.warmup, argmax=step.argmax)
        del dense

    # end to end through the public API with host buffers: x from pinned host
    # memory in, y (or the argmax index) back to pinned host memory, every step
    e2e = None
    if not args.no_e2e:
        xpack_h = torch.from_numpy(step.xpack_host.view(np.int16)).view(torch.bfloat16).pin_memory()
        ypack_h = torch.empty(step.ypack.numel(), dtype=torch.bfloat16).pin_memory()
        idx_h = torch.empty(M, dtype=torch.int32).pin_memory()

        def estep():
            step.run_e2e(xpack_h, ypack_h, idx_h)

        for _ in range(args.warmup):
            estep()
        barrier()
        e_ms = max_over_ranks(time_steps(estep, max(10, min(K, 1000))), "cuda")
        w12.w12_check_status()
        e2e = {"value": round(job_weight_gbs(step.weights, world, e_ms), 2), "unit": "GB/s",
               "h2d_bytes_per_step": int(2 * step.xpack_host.size),
               "d2h_bytes_per_step": int(4 * M) if step.argmax else int(2 * step.ypack.numel()),
               "ms_per_step": round(e_ms, 5)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        orc = OracleSample(cpu_weights(), cpu_xs, M)
        v, sample, _, _ = orc.run(3.0)
        v1, sample1, _, _ = orc.run(1.5, threads=1)
        cpu = {"value": round(v, 4), "unit": "GB/s", "cores": orc.cores, "kind": "oracle", "sample": sample,
               "value_1core": round(v1, 4), "sample_1core": sample1}

    detail_extra = {}
    if rank == 0 and world == 1 and not args.no_detail and args.workload == "layer" and args.weights == "w12" \
            and not args.matrices and M == 1:
        detail_extra = run_detail(args, mats, weights, step, bf16)

    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return
    csum = clocks.summary()
    read_ceiling = read_ceiling_gbs()
    layers = wl.MODEL64_LAYERS if args.workload == "model64" else 1
    unit_steps = len(mats) if args.workload == "single" else layers
    value = job_weight_gbs(step.weights, world, ms_step)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {
            "workload": WORKLOAD_TEXT[args.workload],
            "M": M, "global_batch": M * world, "parallelism": f"replicas x{world}",
            **({"options": args.opt} if args.opt else {}),
            "l2": (f"inputs larger than L2: {step.packed / 1e6:.1f} MB of W12 streamed per step (L2 129 MB)"
                   if args.workload != "single" else
                   f"{len(mats)} encoded copies rotated ({step.packed / 1e6:.1f} MB per step, > 3 x L2)"),
            "launch": ("cuda graph" if graph is not None else "stream") + f" ({nl} launches per step: "
                      + ", ".join(step.launch_names[:7]) + ("..." if nl > 7 else "") + ")",
        },
        "roofline": {"bound": "hbm", "kernel": step.kernels[dom], "launch": step.launch_names[dom],
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind, "traffic": traffic,
                     "algorithmic_bytes": int(step.alg[dom]),
                     "step_frac": round(step.packed / (ms_step * 1e-3) / 1e9 / peak, 4),
                     "launch_frac": lf,
                     "read_ceiling_GBps": round(read_ceiling, 1),
                     "frac_of_read_ceiling": round(achieved / read_ceiling, 4)},
        "cpu_baseline": cpu,
        "clocks": csum,
        "e2e": e2e,
        "gpu_launches": K * step.launch_count(),
        "detail": {
            "us_per_layer": round(ms_step * 1e3 / unit_steps, 3),
            "step_median_us": round(med * 1e3, 2), "step_ci95_us": [round(lo * 1e3, 2), round(hi * 1e3, 2)],
            "step_samples": len(samples),
            "layers_per_step": unit_steps,
            "packed_GBps": round(step.packed / (ms_step * 1e-3) / 1e9, 1),
            "packed_frac_of_hbm_peak": round(step.packed / (ms_step * 1e-3) / 1e9 / peak, 4),
            "bits_per_weight": round(8.0 * step.packed / step.weights, 5),
            "n_escapes": int(sum(int(getattr(m.info, "n_escapes", 0)) for m in mats)),
            "weights": args.weights,
            "per_launch_us": {n: round(v * 1e3, 2) for n, v in zip(step.launch_names[:8], launch_ms[:8])},
            "bf16_cublas_us_per_layer": round(bf16 * 1e3 / unit_steps, 3) if bf16 else None,
            "speedup_vs_bf16": round(bf16 / ms_step, 4) if bf16 else None,
            **detail_extra,
        },
    }
    emit(line, args)


def read_ceiling_gbs(nbytes: int = 2 << 30, iters: int = 20) -> float:
    """HBM read ceiling on this GPU: the library's read-stream kernel over a
    buffer larger than L2 (read once per iteration, nothing written), GB/s."""
    import torch
    from lossless_bit_weight_encode_gb300 import w12
    buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    buf.fill_(1)  # folds to 0 (an even count of equal words), never 0xFFFFFFFF
    sink = torch.zeros(4, dtype=torch.int32, device="cuda")
    sh = torch.cuda.current_stream().cuda_stream
    run = lambda: w12.w12_read_stream_ptr(buf.data_ptr(), nbytes, sink.data_ptr(), 0xFFFFFFFF, sh)
    for _ in range(3):
        run()
    ms = time_steps(run, iters)
    w12.w12_check_status()
    del buf
    return nbytes / (ms * 1e-3) / 1e9


def run_detail(args, mats, weights, step, bf16_ms):
    """The other configurations, for the record: the layer at M = 2..32, the
    heavy-tailed layer at M = 1 and 16, the single 1024 x 1024 layer, and the
    decode kernel's read + write bandwidth."""
    import torch
    from lossless_bit_weight_encode_gb300 import W12Weight, w12
    from lossless_bit_weight_encode_gb300 import workloads as wl

    peak, _ = hbm_peak_gbs()
    K = max(args.steps, 50)
    out = {}
    dense = dense_dev(weights)
    sweep = {"1": {"us_per_layer": None}}
    for M in wl.SWEEP_M:
        xs = [wl.activations(M, w.shape[1], seed=wl.activation_seed("layer", M)) for _, w in weights]
        sweep[str(M)] = sweep_point(mats, weights, xs, M, K, args.warmup, dense)
    del sweep["1"]
    out["layer_sweep"] = sweep
    del dense

    # heavy-tailed weights (escape path)
    hw = list(wl.layer_weights("heavy"))
    hmats = [W12Weight(w) for _, w in hw]
    hdense = dense_dev(hw)
    heavy = {"escape_rate": round(sum(int(m.info.n_escapes) for m in hmats) / sum(m.N * m.K for m in hmats), 6)}
    for M in wl.HEAVY_M:
        xs = [wl.activations(M, w.shape[1], seed=wl.activation_seed("heavy", M)) for _, w in hw]
        heavy[str(M)] = sweep_point(hmats, hw, xs, M, K, args.warmup, hdense)
    out["heavy"] = heavy
    del hdense, hmats

    # the single 1024 x 1024 layer at M = 1, L2 defeated by rotating copies
    w, x = wl.single_case()
    base = W12Weight(w)
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    copies = max(1, -(-3 * l2 // int(base.info.total_bytes)))
    blobs = [base.blob] + [base.blob.clone() for _ in range(copies - 1)]
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    yd = torch.empty((1, 1024), dtype=torch.bfloat16, device="cuda")
    ws = base.workspace(1)
    sh = torch.cuda.current_stream().cuda_stream
    it = [0]

    def one():
        b = blobs[it[0] % copies]
        it[0] += 1
        rc = w12.w12_gemm_ptr(xd.data_ptr(), b.data_ptr(), base.info, yd.data_ptr(), 1, ws.data_ptr(), ws.numel(),
                              sh)
        if rc != 0:
            raise w12.W12Error(rc, w12.w12_last_error())

    for _ in range(args.warmup * copies):
        one()
    ms = time_steps(one, 4 * copies)
    med, lo, hi = bootstrap_median_ci(step_samples(one, 4 * copies))
    w12.w12_check_status()
    out["single"] = {"shape": "1024x1024", "M": 1, "us": round(ms * 1e3, 3), "median_us": round(med * 1e3, 3),
                     "ci95_us": [round(lo * 1e3, 3), round(hi * 1e3, 3)], "copies_rotated": copies,
                     "packed_GBps": round(int(base.info.total_bytes) / (ms * 1e-3) / 1e9, 1),
                     "kernel": w12.w12_gemm_group_launch_info([base.info], 1)["kernel_name"]}
    del blobs

    # decode kernel: W12 -> BF16 for the gate matrix (read the blob, write
    # 2 bytes per weight)
    gate = mats[LAYER_NAMES.index("gate")]
    dec = torch.empty((gate.N, gate.K), dtype=torch.bfloat16, device="cuda")
    for _ in range(3):
        gate.decode(dec)
    ms = time_steps(lambda: gate.decode(dec), 50)
    w12.w12_check_status()
    rw = int(gate.info.total_bytes) + 2 * gate.N * gate.K
    out["decode"] = {"matrix": f"gate {gate.N}x{gate.K}", "us": round(ms * 1e3, 2), "read_write_bytes": rw,
                     "GBps": round(rw / (ms * 1e-3) / 1e9, 1), "frac_of_hbm_peak": round(rw / (ms * 1e-3) / 1e9 / peak, 4)}
    return out


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_w12(args)


if __name__ == "__main__":
    main()
