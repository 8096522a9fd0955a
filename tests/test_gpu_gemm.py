"""GPU W12 GEMM through the C ABI against the fp64 oracle over the original
BF16 weights: tolerance on every tested output, bit-exact where the arithmetic
is exact (one-hot x, small integers), reproducible run to run, and the failure
path (bounded wait -> W12_ERR_TIMEOUT) without a fault."""
import numpy as np
import pytest

import oracle
from lossless_bit_weight_encode_gb300 import W12Weight, w12
from lossless_bit_weight_encode_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

# tensor-core variants: (kernel, A operand, token tile); "sm" is the
# one-CTA-per-SM kernel (A in TMEM), "multi" the several-CTA kernel
TC_VARIANTS = [("sm", "tmem", "32"), ("sm", "tmem", "16"), ("multi", "tmem", "32"), ("multi", "tmem", "16"),
               ("multi", "smem", "32"), ("multi", "smem", "16")]


@pytest.fixture(scope="module", autouse=True)
def built():
    from gpu_util import ensure_built
    ensure_built()


@pytest.fixture(params=TC_VARIANTS, ids=lambda v: f"{v[0]}-{v[1]}-ntok{v[2]}")
def a_operand(request, w12_opts):
    """Every tensor-core variant: one CTA per SM or several, A in TMEM or
    SMEM, 32- or 16-token tile."""
    kernel, a, ntok = request.param
    w12_opts(tc_sm=kernel == "sm", a_operand_smem=a == "smem", token_tile=int(ntok))
    return request.param


def _gemm(mat, x_bits):
    import torch
    from gpu_util import dev_to_bits, to_dev_bf16
    y = mat.gemm(to_dev_bf16(x_bits))
    w12.w12_check_status()
    torch.cuda.synchronize()
    return dev_to_bits(y)


@pytest.mark.parametrize("M", [1, 2, 3, 8, 16, 17, 31, 32])
def test_small_gemm_all_m(M, a_operand):
    from gpu_util import check_tolerance
    w = wl.gaussian_weights(384, 2048, seed=M)
    x = wl.activations(M, 2048, seed=100 + M)
    mat = W12Weight(w)
    check_tolerance(_gemm(mat, x), oracle.gemm_f64(x, w), f"M={M} {a_operand}")


@pytest.mark.parametrize("shape", [(1, 1), (1, 32), (129, 33), (300, 1000), (300, 1001), (130, 7000)])
@pytest.mark.parametrize("M", [1, 2, 5, 32])
def test_ragged_gemm(shape, M):
    from gpu_util import check_tolerance
    n, k = shape
    w = wl.heavy_tail_weights(n, k, seed=n + k)
    x = wl.activations(M, k, seed=n * k + M)
    check_tolerance(_gemm(W12Weight(w), x), oracle.gemm_f64(x, w), f"{shape} M={M}")


@pytest.mark.parametrize("frac", [0.02, 0.10, 1.0])
@pytest.mark.parametrize("M", [1, 2, 16])
def test_forced_escape_gemm(frac, M, a_operand):
    from gpu_util import check_tolerance
    w = wl.forced_escape_weights(256, 4096, frac, seed=int(frac * 1000) + M)
    # huge exponents overflow the sum; keep the weights finite and moderate
    e = (w >> 7) & 0xFF
    w = np.where((e > 140) | (e == 255), (w & 0x807F) | np.uint16(130 << 7), w).astype(np.uint16)
    x = wl.activations(M, 4096, seed=7 + M)
    check_tolerance(_gemm(W12Weight(w), x), oracle.gemm_f64(x, w), f"escapes {frac} M={M}")


def test_one_hot_is_exact(a_operand):
    from gpu_util import bits_to_f64
    w = wl.heavy_tail_weights(256, 1024, seed=11)
    ks = [0, 1, 31, 32, 500, 1023]
    x = np.zeros((len(ks), 1024), dtype=np.uint16)
    for i, k in enumerate(ks):
        x[i, k] = 0x3F80  # 1.0
    y = bits_to_f64(_gemm(W12Weight(w), x))
    for i, k in enumerate(ks):
        assert np.array_equal(y[i], bits_to_f64(w[:, k])), f"column {k}"


def test_small_integers_are_exact():
    from gpu_util import bits_to_f64
    rng = np.random.default_rng(12)
    wi = rng.integers(-8, 9, (256, 1536)).astype(np.float32)
    xi = rng.integers(-8, 9, (7, 1536)).astype(np.float32)
    y = bits_to_f64(_gemm(W12Weight(wl.to_bf16_bits(wi)), wl.to_bf16_bits(xi)))
    ref = (xi.astype(np.int64) @ wi.astype(np.int64).T).astype(np.float64)
    ref_bf16 = bits_to_f64(wl.to_bf16_bits(ref.astype(np.float32)))
    assert np.array_equal(y, ref_bf16)


def test_reproducible_and_workspace_restored():
    import torch
    from gpu_util import dev_to_bits, to_dev_bf16
    w = wl.gaussian_weights(1024, 17408, seed=13)
    x = to_dev_bf16(wl.activations(16, 17408, seed=14))
    mat = W12Weight(w)
    y1 = dev_to_bits(mat.gemm(x))
    ws = mat.workspace(16)
    w12.w12_check_status()
    tiles = int(mat.info.tiles)
    assert int(ws[: tiles * 4].view(torch.int32).abs().sum().item()) == 0, "split-K counters not reset"
    y2 = dev_to_bits(mat.gemm(x))
    w12.w12_check_status()
    assert np.array_equal(y1, y2)


def test_unaligned_x_is_handled():
    import torch
    from gpu_util import check_tolerance, dev_to_bits, to_dev_bf16
    w = wl.gaussian_weights(256, 1024, seed=15)
    x = wl.activations(3, 1024, seed=16)
    buf = torch.zeros(3 * 1024 + 1, dtype=torch.bfloat16, device="cuda")
    xv = buf[1:].view(3, 1024)
    xv.copy_(to_dev_bf16(x))
    mat = W12Weight(w)
    y = torch.empty((3, 256), dtype=torch.bfloat16, device="cuda")
    w12.w12_gemm(xv, mat.blob, mat.info, y, 3, mat.workspace(3))
    w12.w12_check_status()
    check_tolerance(dev_to_bits(y), oracle.gemm_f64(x, w), "unaligned x")


def test_argument_errors():
    import torch
    w = wl.gaussian_weights(128, 256, seed=17)
    mat = W12Weight(w)
    x = torch.zeros((33, 256), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((33, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(w12.W12Error) as ei:
        w12.w12_gemm(x, mat.blob, mat.info, y, 33, mat.workspace(1))
    assert ei.value.status == 1
    # workspace too small: rejected on the host before any launch
    big = W12Weight(wl.gaussian_weights(128, 8192, seed=18))
    xb = torch.zeros((1, 8192), dtype=torch.bfloat16, device="cuda")
    small = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert w12.w12_gemm_workspace_size(big.info, 1) > 256
    with pytest.raises(w12.W12Error) as ei:
        w12.w12_gemm(xb, big.blob, big.info, y[:1], 1, small)
    assert ei.value.status == 3
    bad_blob = torch.zeros(mat.blob.numel() + 16, dtype=torch.uint8, device="cuda")[16:]
    with pytest.raises(w12.W12Error) as ei:
        w12.w12_gemm(x[:1], bad_blob, mat.info, y[:1], 1, mat.workspace(1))
    assert ei.value.status == 4


def test_bounded_wait_reports_timeout():
    w12.w12_check_status()
    w12.w12_selftest_timeout(2000)
    with pytest.raises(w12.W12Error) as ei:
        w12.w12_check_status()
    assert ei.value.status == 8
    w12.w12_check_status()  # cleared; the context is still usable


@pytest.mark.parametrize("workload,Ms", [("layer", (1, 2, 4, 8, 16, 32)), ("heavy", (1, 16))])
def test_layer_shapes_sampled_rows(workload, Ms):
    """Every layer matrix at full size, in the launch configuration the
    benchmark uses; the oracle checks 512 seeded rows of y per matrix and M."""
    from gpu_util import check_tolerance
    rng = np.random.default_rng(19)
    for name, w in wl.layer_weights(workload):
        mat = W12Weight(w)
        rows = np.sort(rng.choice(w.shape[0], size=512, replace=False))
        for M in Ms:
            x = wl.activations(M, w.shape[1], seed=wl.activation_seed(workload, M))
            y = _gemm(mat, x)
            ref = oracle.gemm_f64(x, np.ascontiguousarray(w[rows]))
            check_tolerance(y[:, rows], ref, f"{workload} {name} M={M}")


@pytest.fixture(params=["gemv", "tc"])
def m1_path(request, w12_opts):
    w12_opts(gemv_max_m=2 if request.param == "gemv" else 0)
    return request.param


@pytest.mark.parametrize("case", ["gauss", "ragged", "forced2", "forced10", "forced100", "heavy_long"])
def test_one_token_paths(case, m1_path):
    """M = 1 runs on CUDA cores by default and on tensor cores on request;
    both must meet the tolerance, including ragged tiles and every escape
    regime (staged in SMEM, or read from global memory when a segment holds
    too many)."""
    from gpu_util import check_tolerance
    if case == "gauss":
        w = wl.gaussian_weights(512, 5120, seed=31)
    elif case == "ragged":
        w = wl.heavy_tail_weights(301, 1001, seed=32)
    elif case == "heavy_long":
        w = wl.heavy_tail_weights(256, 17408, seed=33)
    else:
        frac = {"forced2": 0.02, "forced10": 0.10, "forced100": 1.0}[case]
        w = wl.forced_escape_weights(256, 4096, frac, seed=34)
        e = (w >> 7) & 0xFF
        w = np.where((e > 140) | (e == 255), (w & 0x807F) | np.uint16(130 << 7), w).astype(np.uint16)
    x = wl.activations(1, w.shape[1], seed=35)
    mat = W12Weight(w)
    assert w12.w12_gemm_launch_info(mat.info, 1)["ntok"] == (1 if m1_path == "gemv" else 16)
    check_tolerance(_gemm(mat, x), oracle.gemm_f64(x, w), f"{case} {m1_path}")


def test_one_token_one_hot_exact(m1_path):
    from gpu_util import bits_to_f64
    w = wl.heavy_tail_weights(256, 1024, seed=36)
    for k in (0, 17, 1023):
        x = np.zeros((1, 1024), dtype=np.uint16)
        x[0, k] = 0x3F80
        y = bits_to_f64(_gemm(W12Weight(w), x))
        assert np.array_equal(y[0], bits_to_f64(w[:, k])), f"{m1_path} column {k}"


@pytest.fixture(params=["2", "1"])
def gemv_max_m(request, w12_opts):
    w12_opts(gemv_max_m=int(request.param))
    return int(request.param)


@pytest.mark.parametrize("M", [2, 3])
@pytest.mark.parametrize("case", ["gauss", "ragged", "forced10", "heavy_long"])
def test_two_token_paths(case, M, gemv_max_m):
    """Two tokens run on CUDA cores by default and on tensor cores when the
    CUDA-core limit is 1; three always on tensor cores; every path must meet
    the tolerance."""
    from gpu_util import check_tolerance
    if case == "gauss":
        w = wl.gaussian_weights(512, 5120, seed=41)
    elif case == "ragged":
        w = wl.heavy_tail_weights(301, 1001, seed=42)
    elif case == "heavy_long":
        w = wl.heavy_tail_weights(256, 17408, seed=43)
    else:
        w = wl.forced_escape_weights(256, 4096, 0.10, seed=44)
        e = (w >> 7) & 0xFF
        w = np.where((e > 140) | (e == 255), (w & 0x807F) | np.uint16(130 << 7), w).astype(np.uint16)
    x = wl.activations(M, w.shape[1], seed=45 + M)
    mat = W12Weight(w)
    ntok = w12.w12_gemm_launch_info(mat.info, M)["ntok"]
    assert ntok == (2 if M <= gemv_max_m else 16)
    check_tolerance(_gemm(mat, x), oracle.gemm_f64(x, w), f"{case} M={M} ntok={ntok}")


@pytest.mark.parametrize("M", [16, 32])
@pytest.mark.parametrize("kernel", ["tc", "gemv"])
def test_subnormal_weights_one_hot(M, kernel, w12_opts):
    """Weights with subnormal BF16 patterns (exponent 0, mantissa != 0, both
    signs) through a one-hot x: the product must return each weight bit for
    bit, so subnormal inputs are neither flushed by the tensor pipe nor by
    the CUDA-core multiply-add, and the fp32 accumulator keeps them."""
    if kernel == "gemv":
        M = 2
        w12_opts(gemv_max_m=2)
    rng = np.random.default_rng(50 + M)
    w = wl.gaussian_weights(256, 1024, seed=51)
    sub = rng.integers(1, 128, size=(256, 1024)).astype(np.uint16) | (rng.integers(0, 2, size=(256, 1024))
                                                                        .astype(np.uint16) << 15)
    pick = rng.random((256, 1024)) < 0.5
    w = np.where(pick, sub, w).astype(np.uint16)
    ks = np.sort(rng.choice(1024, size=M, replace=False))
    x = np.zeros((M, 1024), dtype=np.uint16)
    x[np.arange(M), ks] = 0x3F80  # 1.0
    mat = W12Weight(w)
    assert (w12.w12_gemm_launch_info(mat.info, M)["ntok"] <= 2) == (kernel == "gemv")
    y = _gemm(mat, x)
    for i, k in enumerate(ks):
        col = w[:, k]
        assert np.count_nonzero(((col >> 7) & 0xFF) == 0) > 50
        assert np.array_equal(y[i], col), f"column {k}: {np.count_nonzero(y[i] != col)} differ"
