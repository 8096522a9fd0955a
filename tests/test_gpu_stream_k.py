"""Stream-K work sharing of the CUDA-core GEMV (one or two tokens): when a
single wave of CTAs holds more CTAs than there are 128-row tiles, the tiles x
segments units are cut into equal contiguous ranges, so a CTA may finish one
tile and start the next (of the same matrix or, in a group, of the next
member).  Every output meets the tolerance against the fp64 oracle, with and
without stream-K; the plan uses one full wave; results are reproducible and
the split-K counters are left at zero."""
import numpy as np
import pytest

import oracle
from lossless_bit_weight_encode_gb300 import W12Group, W12Weight, w12
from lossless_bit_weight_encode_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from gpu_util import ensure_built
    ensure_built()


def _capacity(plan):
    import torch
    return torch.cuda.get_device_properties(0).multi_processor_count * plan["ctas_per_sm"]


@pytest.fixture(params=["1", "0"], ids=["cta_per_sm", "two_ctas_per_sm"])
def gemv_kernel(request, w12_opts):
    """Both CUDA-core kernels, whichever the planner would pick."""
    w12_opts(gemv_sm=int(request.param))
    return request.param


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("shape", [(12763, 5020), (5000, 17408), (1000, 3000)])
def test_stream_k_matches_oracle(M, shape, gemv_kernel, w12_opts):
    import torch
    from gpu_util import check_tolerance, dev_to_bits, to_dev_bf16
    n, k = shape
    w = wl.heavy_tail_weights(n, k, seed=300 + n % 97)
    x = wl.activations(M, k, seed=301 + M)
    ref = oracle.gemm_f64(x, w)
    mat = W12Weight(w)
    for mode in ("1", "0"):
        w12_opts(stream_k=int(mode))
        plan = w12.w12_gemm_launch_info(mat.info, M)
        tiles, segs = int(mat.info.tiles), int(mat.info.segs)
        if mode == "1":
            expect = min(_capacity(plan), tiles * segs)
            if plan["ctas_per_sm"] == 1 and tiles * segs < 4 * expect:
                expect = max(1, tiles * segs // 4)  # at least four segments per CTA
            assert plan["ctas"] == expect, plan
        else:
            assert plan["ctas"] == tiles * plan["splits"], plan
        y = dev_to_bits(mat.gemm(to_dev_bf16(x)))
        w12.w12_check_status()
        torch.cuda.synchronize()
        check_tolerance(y, ref, f"{shape} M={M} stream_k={mode}")


@pytest.mark.parametrize("M", [1, 2])
def test_stream_k_crosses_group_members(M, gemv_kernel):
    """q/k/v-like group whose ranges end inside one member and start in the next."""
    import torch
    from gpu_util import check_tolerance, dev_to_bits, to_dev_bf16
    k = 5120
    shapes = [(2560, k), (520, k), (384, k)]
    ws = [wl.heavy_tail_weights(n, kk, seed=310 + i) for i, (n, kk) in enumerate(shapes)]
    mats = [W12Weight(w) for w in ws]
    units = sum(int(m.info.tiles) for m in mats) * int(mats[0].info.segs)
    assert units > _capacity(w12.w12_gemm_launch_info(mats[0].info, M))  # ranges cross tiles
    x = wl.activations(M, k, seed=315 + M)
    ys = W12Group(mats).gemm(to_dev_bf16(x))
    w12.w12_check_status()
    torch.cuda.synchronize()
    for i, (w, y) in enumerate(zip(ws, ys)):
        check_tolerance(dev_to_bits(y), oracle.gemm_f64(x, w), f"member {i} M={M}")


def test_stream_k_reproducible_and_counters_reset(gemv_kernel):
    import torch
    from gpu_util import dev_to_bits, to_dev_bf16
    w = wl.gaussian_weights(9000, 5120, seed=320)
    x = to_dev_bf16(wl.activations(1, 5120, seed=321))
    mat = W12Weight(w)
    y1 = dev_to_bits(mat.gemm(x))
    ws = mat.workspace(1)
    w12.w12_check_status()
    tiles = int(mat.info.tiles)
    assert int(ws[: tiles * 4].view(torch.int32).abs().sum().item()) == 0, "split-K counters not reset"
    for _ in range(3):
        assert np.array_equal(dev_to_bits(mat.gemm(x)), y1)
    w12.w12_check_status()


def test_kernel_choice(w12_opts):
    """One CTA per SM whenever one wave of ranges covers the launch, for
    Gaussian and escape-heavy weights alike, whatever the tile count."""
    import torch
    w12_opts(gemv_sm=-1)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    gauss = W12Weight(wl.gaussian_weights(2048, 1024, seed=330))
    heavy = W12Weight(wl.heavy_tail_weights(2048, 1024, seed=331))
    many = W12Weight(wl.gaussian_weights(3 * sms * 128, 512, seed=332))
    assert heavy.info.n_escapes / (2048 * 1024) > 2e-3
    for M in (1, 2):
        assert w12.w12_gemm_launch_info(gauss.info, M)["ctas_per_sm"] == 1
        assert w12.w12_gemm_launch_info(heavy.info, M)["ctas_per_sm"] == 1
        plan = w12.w12_gemm_launch_info(many.info, M)
        assert plan["ctas_per_sm"] == 1 and plan["ctas"] == sms
    w12_opts(gemv_sm=0)
    assert w12.w12_gemm_launch_info(heavy.info, 1)["ctas_per_sm"] == 2


@pytest.mark.parametrize("case", range(10))
def test_stream_k_random_shapes(case, gemv_kernel):
    """Seeded random shapes (ragged N and K, one to ~120 segments per row
    tile, one or two tokens) against the oracle, on both CUDA-core kernels."""
    import torch
    from gpu_util import check_tolerance, dev_to_bits, to_dev_bf16
    rng = np.random.default_rng(1000 + case)
    k = int(rng.integers(1, 30000))
    n = int(rng.integers(1, max(2, min(9000, 40_000_000 // k))))
    M = int(rng.integers(1, 3))
    gen = wl.heavy_tail_weights if case % 3 == 0 else wl.gaussian_weights
    w = gen(n, k, seed=1100 + case)
    x = wl.activations(M, k, seed=1200 + case)
    y = dev_to_bits(W12Weight(w).gemm(to_dev_bf16(x)))
    w12.w12_check_status()
    torch.cuda.synchronize()
    check_tolerance(y, oracle.gemm_f64(x, w), f"case {case}: {n}x{k} M={M}")


@pytest.mark.parametrize("frac", [0.02, 0.10, 1.0])
@pytest.mark.parametrize("M", [1, 2])
def test_forced_escapes_on_both_kernels(frac, M, gemv_kernel):
    """2 %, 10 % and 100 % escapes: staged and unstaged escape runs, lanes
    with several escapes, and (one CTA per SM) the counts of earlier chunks."""
    import torch
    from gpu_util import check_tolerance, dev_to_bits, to_dev_bf16
    w = wl.forced_escape_weights(640, 4096 + 96, frac, seed=int(frac * 1000) + 10 * M)
    # huge exponents overflow the sum; keep the weights finite and moderate
    e = (w >> 7) & 0xFF
    w = np.where((e > 140) | (e == 255), (w & 0x807F) | np.uint16(130 << 7), w).astype(np.uint16)
    x = wl.activations(M, w.shape[1], seed=1300 + M)
    y = dev_to_bits(W12Weight(w).gemm(to_dev_bf16(x)))
    w12.w12_check_status()
    torch.cuda.synchronize()
    check_tolerance(y, oracle.gemm_f64(x, w), f"{frac:.0%} escapes M={M}")
