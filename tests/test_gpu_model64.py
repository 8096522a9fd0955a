"""The 64-layer stream: 64 decoder layers of the 27B-class shapes (448
matrices, 21.8 G weights, 32.7 GB of W12 resident in HBM), encoded on the GPU
and run as one chained pass of 448 GEMMs in layer order at 16 and 32 tokens.
Every layer must decode bit-exactly to the weights it was built from; four
seeded layers are checked against the fp64 oracle (sampled rows of every
matrix) from the chained pass's own outputs."""
import numpy as np
import pytest

import oracle
from lossless_bit_weight_encode_gb300 import W12Weight, w12
from lossless_bit_weight_encode_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

LAYERS = wl.MODEL64_LAYERS
CHECKED_LAYERS = sorted(np.random.default_rng(51).choice(LAYERS, size=4, replace=False).tolist())
ROWS = 128


@pytest.fixture(scope="module")
def model():
    import torch
    from gpu_util import ensure_built
    ensure_built()
    mats, host_rows = [], {}
    rng = np.random.default_rng(52)
    for layer in range(LAYERS):
        for idx in range(len(wl.LAYER_SHAPES)):
            w = wl.model64_weight_dev(layer, idx)
            mat = W12Weight.from_device(w)
            back = mat.decode()
            w12.w12_check_status()
            assert torch.equal(back.view(torch.int16), w.view(torch.int16)), f"layer {layer} matrix {idx}"
            if layer in CHECKED_LAYERS:
                rows = np.sort(rng.choice(w.shape[0], size=ROWS, replace=False))
                sel = w[torch.from_numpy(rows).cuda()].view(torch.int16).cpu().numpy().view(np.uint16)
                host_rows[(layer, idx)] = (rows, sel)
            del w, back
            mats.append(mat)
    torch.cuda.synchronize()
    total = sum(int(m.info.total_bytes) for m in mats)
    assert 32.5e9 < total < 33.0e9, total
    yield mats, host_rows
    del mats
    torch.cuda.empty_cache()


@pytest.mark.parametrize("M", wl.MODEL64_M)
def test_chained_pass(model, M):
    import torch
    from gpu_util import check_tolerance, dev_to_bits, to_dev_bf16
    mats, host_rows = model
    xs_host = [wl.model64_activation(M, i) for i in range(len(wl.LAYER_SHAPES))]
    xs = [to_dev_bf16(x) for x in xs_host]
    keep = {}
    for i, mat in enumerate(mats):  # layer order, one stream
        layer, idx = divmod(i, len(wl.LAYER_SHAPES))
        y = mat.gemm(xs[idx])
        if layer in CHECKED_LAYERS:
            keep[(layer, idx)] = y
    w12.w12_check_status()
    torch.cuda.synchronize()
    for (layer, idx), y in keep.items():
        rows, wsel = host_rows[(layer, idx)]
        got = dev_to_bits(y)[:, rows]
        check_tolerance(got, oracle.gemm_f64(xs_host[idx], wsel), f"layer {layer} {wl.LAYER_SHAPES[idx][0]} M={M}")
