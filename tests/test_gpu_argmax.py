"""LM-head GEMM with the fused argmax (w12_gemm_argmax) against the oracle's
fp64 argmax.  The kernel ranks fp32 sums, so where two logits lie within the
fp32 accumulation error of each other either may win; the check is therefore:
the chosen row's exact logit is within that error of the exact maximum, the
reported value is within that error of the chosen row's exact logit, and a
winner whose margin exceeds the error is found exactly.  Exact cases (one-hot
x, identical rows) need no error term."""
import numpy as np
import pytest

import oracle
from lossless_bit_weight_encode_gb300 import W12Weight, w12
from lossless_bit_weight_encode_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from gpu_util import ensure_built
    ensure_built()


@pytest.fixture(params=["gemv", "tc"])
def m1_path(request, w12_opts):
    w12_opts(gemv_max_m=2 if request.param == "gemv" else 0)
    return request.param


def _run(mat, x_bits, logits=False):
    import torch
    from gpu_util import to_dev_bf16
    idx, val, y = mat.gemm_argmax(to_dev_bf16(x_bits), logits=logits)
    w12.w12_check_status()
    torch.cuda.synchronize()
    return idx.cpu().numpy(), val.cpu().numpy(), y


def _check(idx, val, x, w):
    ref, logits = oracle.argmax_f64(x, w)
    k = x.shape[1]
    xa = np.abs(wl.bf16_bits_to_f32(x).astype(np.float64))
    wa = np.abs(wl.bf16_bits_to_f32(w).astype(np.float64))
    # |fp32 sum - exact| <= (K + 2) u sum|x w| for any summation order (u = 2^-24)
    err = (k + 2) * 2.0 ** -24 * (xa @ wa.T)
    for m in range(x.shape[0]):
        i = int(idx[m])
        assert 0 <= i < w.shape[0], f"token {m}: index {i}"
        r = int(ref[m])
        assert logits[m, i] + err[m, i] >= logits[m, r] - err[m, r], f"token {m}: row {i} is not a near-maximum"
        assert abs(float(val[m]) - logits[m, i]) <= err[m, i] + 1e-30, f"token {m}: value"
        others = np.delete(logits[m] + err[m], r)
        if logits[m, r] - err[m, r] > others.max():
            assert i == r, f"token {m}: clear winner {r} missed (got {i})"


@pytest.mark.parametrize("M", [1, 2, 3, 16, 32])
def test_argmax_matches_oracle(M, m1_path):
    if M > 1 and m1_path == "tc":
        pytest.skip("the M = 1 path switch only matters at one token")
    w = wl.heavy_tail_weights(4099, 5120, seed=60)
    x = wl.activations(M, 5120, seed=61 + M)
    idx, val, _ = _run(W12Weight(w), x)
    _check(idx, val, x, w)


def test_logits_are_the_plain_gemm():
    from gpu_util import dev_to_bits, to_dev_bf16
    w = wl.gaussian_weights(3000, 2048, seed=62)
    mat = W12Weight(w)
    for M in (1, 7, 32):
        x = wl.activations(M, 2048, seed=63 + M)
        _, _, y = _run(mat, x, logits=True)
        ref = dev_to_bits(mat.gemm(to_dev_bf16(x)))
        w12.w12_check_status()
        assert np.array_equal(dev_to_bits(y), ref), f"M={M}"


@pytest.mark.parametrize("M", [1, 2, 4, 17])
def test_ties_go_to_the_lowest_row(M, m1_path):
    """Identical rows give identical fp32 sums; the lowest of them must win,
    also across tiles and with a NaN row present."""
    if M > 1 and m1_path == "tc":
        pytest.skip("the M = 1 path switch only matters at one token")
    rng = np.random.default_rng(64)
    k = 3072
    x = wl.activations(M, k, seed=65)
    w = wl.gaussian_weights(1000, k, seed=66)
    xs = wl.bf16_bits_to_f32(x[0])
    star = wl.to_bf16_bits(np.sign(xs) * 0.08)  # aligned with token 0: a large logit
    for r in (300, 5, 77, 900):                 # rows 5 and 77 share a tile, 300 and 900 do not
        w[r] = star
    w[2] = np.uint16(0x7FC0)                    # a NaN row never wins
    idx, val, _ = _run(W12Weight(w), x)
    assert idx[0] == 5
    ref, logits = oracle.argmax_f64(x, w)
    assert ref[0] == 5
    assert np.all(idx != 2)


def test_one_hot_is_exact(m1_path):
    """x = e_k: the logits are column k of W exactly, so the argmax and its
    value are exact (lowest row among equal maxima)."""
    w = wl.gaussian_weights(2500, 1024, seed=67)
    mat = W12Weight(w)
    for kk in (0, 511, 1023):
        x = np.zeros((1, 1024), dtype=np.uint16)
        x[0, kk] = 0x3F80
        idx, val, _ = _run(mat, x)
        col = wl.bf16_bits_to_f32(w[:, kk])
        assert idx[0] == int(np.argmax(col)) and val[0] == col.max()


@pytest.mark.parametrize("M", [1, 4])
def test_full_lm_head(M):
    name, n, k = wl.LMHEAD_SHAPE
    w = wl.gaussian_weights(n, k, seed=wl.weight_seed("lmhead", 0))
    x = wl.activations(M, k, seed=wl.activation_seed("lmhead", M))
    idx, val, _ = _run(W12Weight(w), x)
    _check(idx, val, x, w)
