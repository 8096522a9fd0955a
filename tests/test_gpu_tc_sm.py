"""The one-CTA-per-SM tensor-core kernel (3..32 tokens; sixteen decode warps
store decoded tiles into TMEM, one warp issues tcgen05.mma, four drain the
accumulators) against the fp64 oracle: stream-K ranges that end inside a
tile or a group member, ranges over many short tiles, ragged N and K, every
escape regime, fixed split-K, reproducibility and the split-K counters."""
import numpy as np
import pytest

import oracle
from lossless_bit_weight_encode_gb300 import W12Group, W12Weight, w12
from lossless_bit_weight_encode_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TC_SM = 3  # W12_KERNEL_TC_SM


@pytest.fixture(scope="module", autouse=True)
def built():
    from gpu_util import ensure_built
    ensure_built()


def _run(mat, x_bits):
    import torch
    from gpu_util import dev_to_bits, to_dev_bf16
    y = dev_to_bits(mat.gemm(to_dev_bf16(x_bits)))
    w12.w12_check_status()
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("M", [3, 8, 16, 17, 32])
@pytest.mark.parametrize("shape", [(12763, 5020), (5000, 17408), (1000, 3000), (130, 7000), (300, 33),
                                   (200000, 64)])
def test_tc_sm_matches_oracle(M, shape):
    """Ranges cross tiles (12763 x 5020), hold many short tiles (200000 x 64:
    a two-chunk segment per tile, about ten pieces per CTA, so the two
    accumulators are reused), or split one tile over several CTAs (130 x
    7000); K ragged against chunks and segments."""
    from gpu_util import check_tolerance
    n, k = shape
    w = wl.heavy_tail_weights(n, k, seed=400 + n % 97 + k % 13)
    x = wl.activations(M, k, seed=401 + M)
    mat = W12Weight(w)
    plan = w12.w12_gemm_group_launch_info([mat.info], M)
    assert plan["kernel"] == TC_SM and plan["ctas_per_sm"] == 1, plan
    assert plan["ntok"] == (16 if M <= 16 else 32)
    check_tolerance(_run(mat, x), oracle.gemm_f64(x, w), f"{shape} M={M}")


@pytest.mark.parametrize("M", [4, 16, 32])
def test_tc_sm_crosses_group_members(M):
    """q/k/v-like group whose ranges end inside one member and start in the next."""
    import torch
    from gpu_util import check_tolerance, dev_to_bits, to_dev_bf16
    k = 5120
    shapes = [(2560, k), (520, k), (384, k)]
    ws = [wl.heavy_tail_weights(n, kk, seed=410 + i) for i, (n, kk) in enumerate(shapes)]
    mats = [W12Weight(w) for w in ws]
    assert w12.w12_gemm_group_launch_info([m.info for m in mats], M)["kernel"] == TC_SM
    x = wl.activations(M, k, seed=415 + M)
    ys = W12Group(mats).gemm(to_dev_bf16(x))
    w12.w12_check_status()
    torch.cuda.synchronize()
    for i, (w, y) in enumerate(zip(ws, ys)):
        check_tolerance(dev_to_bits(y), oracle.gemm_f64(x, w), f"member {i} M={M}")


@pytest.mark.parametrize("M", [5, 32])
def test_tc_sm_reproducible_and_counters_reset(M):
    import torch
    from gpu_util import dev_to_bits, to_dev_bf16
    w = wl.gaussian_weights(9000, 5120, seed=420)
    x = to_dev_bf16(wl.activations(M, 5120, seed=421))
    mat = W12Weight(w)
    y1 = dev_to_bits(mat.gemm(x))
    ws = mat.workspace(M)
    w12.w12_check_status()
    tiles = int(mat.info.tiles)
    assert int(ws[: tiles * 4].view(torch.int32).abs().sum().item()) == 0, "split-K counters not reset"
    for _ in range(3):
        assert np.array_equal(dev_to_bits(mat.gemm(x)), y1)
    w12.w12_check_status()


@pytest.mark.parametrize("frac", [0.02, 0.10, 1.0])
@pytest.mark.parametrize("M", [4, 16, 32])
def test_tc_sm_forced_escapes(frac, M):
    """2 %, 10 % and 100 % escapes: escape runs staged in shared memory or
    read from global memory, lanes with several escapes, and the position of
    a warp's first escape counted from either end of its quarter."""
    from gpu_util import check_tolerance
    w = wl.forced_escape_weights(640, 4096 + 96, frac, seed=int(frac * 1000) + 20 * M)
    e = (w >> 7) & 0xFF
    w = np.where((e > 140) | (e == 255), (w & 0x807F) | np.uint16(130 << 7), w).astype(np.uint16)
    x = wl.activations(M, w.shape[1], seed=1400 + M)
    check_tolerance(_run(W12Weight(w), x), oracle.gemm_f64(x, w), f"{frac:.0%} escapes M={M}")


@pytest.mark.parametrize("M", [3, 32])
def test_tc_sm_fixed_split_k(M, w12_opts):
    """The same kernel with fixed split-K (one piece per CTA, grid of splits x
    tiles) when the splits option forces it."""
    from gpu_util import check_tolerance
    w12_opts(splits=3)
    w = wl.heavy_tail_weights(700, 6000, seed=430)
    x = wl.activations(M, 6000, seed=431)
    mat = W12Weight(w)
    plan = w12.w12_gemm_group_launch_info([mat.info], M)
    assert plan["kernel"] == TC_SM and plan["splits"] == 3 and plan["ctas"] == 3 * int(mat.info.tiles), plan
    check_tolerance(_run(mat, x), oracle.gemm_f64(x, w), f"fixed split-K M={M}")


@pytest.mark.parametrize("case", range(8))
def test_tc_sm_random_shapes(case):
    from gpu_util import check_tolerance
    rng = np.random.default_rng(2000 + case)
    k = int(rng.integers(1, 30000))
    n = int(rng.integers(1, max(2, min(9000, 40_000_000 // k))))
    M = int(rng.integers(3, 33))
    gen = wl.heavy_tail_weights if case % 3 == 0 else wl.gaussian_weights
    w = gen(n, k, seed=2100 + case)
    x = wl.activations(M, k, seed=2200 + case)
    check_tolerance(_run(W12Weight(w), x), oracle.gemm_f64(x, w), f"case {case}: {n}x{k} M={M}")


def test_tc_sm_small_integers_exact():
    from gpu_util import bits_to_f64
    rng = np.random.default_rng(440)
    wi = rng.integers(-8, 9, (640, 2560)).astype(np.float32)
    xi = rng.integers(-8, 9, (29, 2560)).astype(np.float32)
    y = bits_to_f64(_run(W12Weight(wl.to_bf16_bits(wi)), wl.to_bf16_bits(xi)))
    ref = (xi.astype(np.int64) @ wi.astype(np.int64).T).astype(np.float64)
    assert np.array_equal(y, bits_to_f64(wl.to_bf16_bits(ref.astype(np.float32))))
