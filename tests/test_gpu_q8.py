"""Q8 copy GEMM (w12_q8_gemm) on both tensor-core kernels (one CTA per SM with
stream-K ranges, and several CTAs per SM with fixed split-K) against the
oracle's fp64 product over its own Q8 copy (same quantizer, same fp32
decisions): tolerance on every output, bit-exact where the arithmetic is exact
(one-hot x), ranges across tiles, and full layer shapes on sampled rows."""
import numpy as np
import pytest

import oracle
from lossless_bit_weight_encode_gb300 import Q8Weight, w12
from lossless_bit_weight_encode_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from gpu_util import ensure_built
    ensure_built()


@pytest.fixture(params=[1, 0], ids=["tc_sm", "tc_multi"])
def q8_kernel(request, w12_opts):
    w12_opts(tc_sm=request.param)
    return request.param


def _gemm(mat, x_bits):
    import torch
    from gpu_util import dev_to_bits, to_dev_bf16
    y = mat.gemm(to_dev_bf16(x_bits))
    w12.w12_check_status()
    torch.cuda.synchronize()
    return dev_to_bits(y)


def test_q8_single_output_within_one_ulp():
    """A 1 x 1 product has one output: the relative Frobenius bound (written
    for many outputs) does not apply, the BF16 rounding does: at most one unit
    in the last place from the fp64 value."""
    for seed in range(20):
        w = wl.heavy_tail_weights(1, 1 + seed, seed=80 + seed)
        x = wl.activations(1, 1 + seed, seed=90 + seed)
        y = wl.bf16_bits_to_f32(_gemm(Q8Weight(w), x))[0, 0]
        ref = oracle.q8_gemm_f64(x, w)[0, 0]
        ulp = 2.0 ** (np.floor(np.log2(abs(ref))) - 7) if ref != 0 else 0.0
        assert abs(float(y) - ref) <= ulp, (seed, float(y), ref)


@pytest.mark.parametrize("shape", [(129, 33), (384, 2048), (300, 1001), (130, 7000)])
@pytest.mark.parametrize("M", [1, 2, 5, 16, 17, 32])
def test_q8_gemm_matches_oracle(shape, M, q8_kernel):
    from gpu_util import check_tolerance
    n, k = shape
    w = wl.heavy_tail_weights(n, k, seed=70 + n + k)
    x = wl.activations(M, k, seed=71 + M)
    check_tolerance(_gemm(Q8Weight(w), x), oracle.q8_gemm_f64(x, w), f"q8 {shape} M={M}")


def test_q8_one_hot_is_exact(q8_kernel):
    """x = e_k: the sum is q[n][k] exactly; y = BF16(fp32(s[n] * q[n][k]))."""
    w = wl.gaussian_weights(256, 512, seed=72)
    s, q = oracle.q8_decode(oracle.q8_encode(w), 256, 512)
    mat = Q8Weight(w)
    for kk in (0, 200, 511):
        x = np.zeros((3, 512), dtype=np.uint16)
        x[:, kk] = 0x3F80
        y = _gemm(mat, x)
        ref = wl.to_bf16_bits((s * q[:, kk].astype(np.float32)).astype(np.float32))
        assert np.array_equal(y[0], ref) and np.array_equal(y[2], ref), f"column {kk}"


def test_q8_layer_shapes_sampled_rows():
    from gpu_util import check_tolerance
    rng = np.random.default_rng(73)
    for name, w in wl.layer_weights("layer"):
        mat = Q8Weight(w)
        rows = np.sort(rng.choice(w.shape[0], size=256, replace=False))
        for M in (1, 16, 32):
            x = wl.activations(M, w.shape[1], seed=wl.activation_seed("layer", M))
            ref = oracle.q8_gemm_f64(x, np.ascontiguousarray(w[rows]))
            check_tolerance(_gemm(mat, x)[:, rows], ref, f"q8 {name} M={M}")


@pytest.mark.parametrize("M", [3, 16, 32])
def test_q8_stream_k_ranges(M):
    """Ranges that end inside a tile (12763 x 5020) and many short tiles
    (60000 x 64) on the one-CTA-per-SM kernel."""
    from gpu_util import check_tolerance
    for n, k in [(12763, 5020), (60000, 64)]:
        w = wl.heavy_tail_weights(n, k, seed=74 + n % 91)
        x = wl.activations(M, k, seed=75 + M)
        mat = Q8Weight(w)
        check_tolerance(_gemm(mat, x), oracle.q8_gemm_f64(x, w), f"q8 {n}x{k} M={M}")


@pytest.mark.parametrize("M", [1, 4, 16, 32])
def test_q8_group_matches_oracle(M, q8_kernel):
    """Q8 copies sharing K in one launch (ragged member heights, a tile that
    ends inside a member): every output within tolerance of the oracle's
    product over its own copy, each with its own row scales."""
    import torch
    from gpu_util import check_tolerance, dev_to_bits, to_dev_bf16
    from lossless_bit_weight_encode_gb300 import Q8Group
    k = 1000
    ws = [wl.heavy_tail_weights(n, k, seed=76 + n) for n in (300, 129, 640)]
    x = wl.activations(M, k, seed=77 + M)
    ys = Q8Group([Q8Weight(w) for w in ws]).gemm(to_dev_bf16(x))
    w12.w12_check_status()
    torch.cuda.synchronize()
    for i, (w, y) in enumerate(zip(ws, ys)):
        check_tolerance(dev_to_bits(y), oracle.q8_gemm_f64(x, w), f"q8 group member {i} M={M}")


def test_q8_layer_groups_sampled_rows():
    """The layer's q+k+v and gate+up groups at full size, sampled rows."""
    import torch
    from gpu_util import check_tolerance, dev_to_bits, to_dev_bf16
    from lossless_bit_weight_encode_gb300 import Q8Group
    rng = np.random.default_rng(78)
    ws = dict(wl.layer_weights("layer"))
    for names in (("q", "k", "v"), ("gate", "up")):
        grp = Q8Group([Q8Weight(ws[n]) for n in names])
        for M in (1, 16, 32):
            x = wl.activations(M, grp.K, seed=wl.activation_seed("layer", M))
            ys = grp.gemm(to_dev_bf16(x))
            w12.w12_check_status()
            torch.cuda.synchronize()
            for n, y in zip(names, ys):
                rows = np.sort(rng.choice(ws[n].shape[0], size=128, replace=False))
                ref = oracle.q8_gemm_f64(x, np.ascontiguousarray(ws[n][rows]))
                check_tolerance(dev_to_bits(y)[:, rows], ref, f"q8 {n} (group) M={M}")
