"""Grouped launch (w12_gemm_group) of matrices that share x: every output
meets the tolerance against the fp64 oracle, equals w12_gemm bit for bit when
both use the same split count, and the argument checks hold."""
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


def _mats(k=2048):
    shapes = [(640, k), (128, k), (300, k)]  # q/k/v-like, one ragged
    ws = [wl.heavy_tail_weights(n, kk, seed=90 + i) for i, (n, kk) in enumerate(shapes)]
    return ws, [W12Weight(w) for w in ws]


@pytest.mark.parametrize("M", [1, 2, 5, 16, 32])
def test_group_matches_oracle(M):
    import torch
    from gpu_util import check_tolerance, dev_to_bits, to_dev_bf16
    ws, mats = _mats()
    x = wl.activations(M, 2048, seed=95 + M)
    ys = W12Group(mats).gemm(to_dev_bf16(x))
    w12.w12_check_status()
    torch.cuda.synchronize()
    for i, (w, y) in enumerate(zip(ws, ys)):
        check_tolerance(dev_to_bits(y), oracle.gemm_f64(x, w), f"member {i} M={M}")


@pytest.mark.parametrize("M", [1, 2, 16])
def test_group_equals_single_launches(M, w12_opts):
    from gpu_util import dev_to_bits, to_dev_bf16
    w12_opts(splits=4)  # same split count for the group and each matrix
    ws, mats = _mats()
    x = to_dev_bf16(wl.activations(M, 2048, seed=97 + M))
    ys = W12Group(mats).gemm(x)
    for i, m in enumerate(mats):
        ref = dev_to_bits(m.gemm(x))
        w12.w12_check_status()
        assert np.array_equal(dev_to_bits(ys[i]), ref), f"member {i} M={M}"


def test_layer_groups_sampled_rows():
    """q/k/v and gate/up of the layer as two groups, sampled rows, M = 1 and 16."""
    import torch
    from gpu_util import check_tolerance, dev_to_bits, to_dev_bf16
    layer = dict(wl.layer_weights("layer"))
    rng = np.random.default_rng(98)
    for names in (("q", "k", "v"), ("gate", "up")):
        mats = [W12Weight(layer[n]) for n in names]
        k = mats[0].K
        for M in (1, 16):
            x = wl.activations(M, k, seed=wl.activation_seed("layer", M))
            ys = W12Group(mats).gemm(to_dev_bf16(x))
            w12.w12_check_status()
            torch.cuda.synchronize()
            for n, y in zip(names, ys):
                rows = np.sort(rng.choice(layer[n].shape[0], size=256, replace=False))
                ref = oracle.gemm_f64(x, np.ascontiguousarray(layer[n][rows]))
                check_tolerance(dev_to_bits(y)[:, rows], ref, f"{n} M={M}")


def test_group_argument_errors():
    import torch
    _, mats = _mats()
    other = W12Weight(wl.gaussian_weights(128, 1024, seed=99))
    with pytest.raises(w12.W12Error) as ei:
        w12.w12_gemm_group_workspace_size([mats[0].info, other.info], 1)
    assert ei.value.status == 2  # K differs
    with pytest.raises(w12.W12Error) as ei:
        w12.w12_gemm_group_workspace_size([m.info for m in mats] * 2, 1)
    assert ei.value.status == 1  # more than 4
    x = torch.zeros((1, 2048), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    ys = [torch.empty((1, m.N), dtype=torch.bfloat16, device="cuda") for m in mats]
    with pytest.raises(w12.W12Error) as ei:
        w12.w12_gemm_group(x, [m.blob for m in mats], [m.info for m in mats], ys, 1, ws)
    assert ei.value.status == 3  # workspace too small
