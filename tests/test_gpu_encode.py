"""GPU encoder (w12_encode_device) through the C ABI: the blob must be byte
for byte the oracle's encoding of the same weights (the format is canonical),
its size must match the oracle's, and a blob built on the GPU must drive the
GEMM exactly as the host-built one does.  Errors: a short buffer is refused
on the host or, for the escape plane, reported by the status word with no byte
written past the buffer."""
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


def _encode_dev(w_dev):
    import torch
    n, k = int(w_dev.shape[0]), int(w_dev.shape[1])
    ws = torch.empty(w12.w12_encode_workspace_size(n, k), dtype=torch.uint8, device="cuda")
    size = w12.w12_encoded_size_device(w_dev, ws)
    blob = torch.full((size,), 0xA5, dtype=torch.uint8, device="cuda")
    w12.w12_encode_device(w_dev, blob, ws)
    w12.w12_check_status()
    return size, blob.cpu().numpy()


def _check_equal(w, w_dev=None):
    from gpu_util import to_dev_bf16
    ref = oracle.encode(w)
    size, got = _encode_dev(to_dev_bf16(w) if w_dev is None else w_dev)
    assert size == ref.size == oracle.encoded_size(w)
    diff = np.flatnonzero(got != ref)
    assert diff.size == 0, f"{diff.size} bytes differ, first at offset {diff[0]}"


CASES = {
    "gauss": lambda: wl.gaussian_weights(512, 5120, seed=41),
    "heavy_ragged": lambda: wl.heavy_tail_weights(300, 1001, seed=42),
    "forced2": lambda: wl.forced_escape_weights(256, 4096, 0.02, seed=43),
    "forced10": lambda: wl.forced_escape_weights(256, 4096, 0.10, seed=44),
    "forced100": lambda: wl.forced_escape_weights(256, 4096, 1.0, seed=45),
    "all_patterns": lambda: wl.all_bf16_patterns(6),
    "table_rule": lambda: wl.table_rule_weights(46),
    "zeros": lambda: np.zeros((200, 700), dtype=np.uint16),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_encoder_matches_oracle(case):
    _check_equal(CASES[case]())


@pytest.mark.parametrize("shape", [(1, 1), (1, 32), (1, 33), (129, 33), (127, 255), (128, 256), (130, 7000),
                                   (257, 264), (1000, 1001)])
def test_ragged_shapes(shape):
    n, k = shape
    _check_equal(wl.heavy_tail_weights(n, k, seed=n * 7 + k))


def test_unaligned_rows_take_the_scalar_path():
    """Weights starting 2 bytes past a 16-byte boundary (rows not 16-byte
    aligned): the same bytes."""
    import torch
    from gpu_util import to_dev_bf16
    w = wl.heavy_tail_weights(384, 2048, seed=47)
    buf = torch.zeros(w.size + 8, dtype=torch.bfloat16, device="cuda")
    view = buf[1:1 + w.size].view(384, 2048)
    view.copy_(to_dev_bf16(w))
    _check_equal(w, view)


def test_layer_matrix_full_size():
    """The largest layer matrix (17408 x 5120), encoded on the GPU, is the
    oracle's blob."""
    name, n, k = wl.LAYER_SHAPES[4]
    _check_equal(wl.gaussian_weights(n, k, seed=wl.weight_seed("layer", 4)))


def test_device_blob_drives_the_gemm():
    import torch
    from gpu_util import dev_to_bits, to_dev_bf16
    w = wl.heavy_tail_weights(1000, 5120, seed=48)
    host = W12Weight(w)
    dev = W12Weight.from_device(to_dev_bf16(w))
    assert dev.info.as_dict() == host.info.as_dict()
    for M in (1, 7, 32):
        x = to_dev_bf16(wl.activations(M, 5120, seed=49 + M))
        a = dev_to_bits(host.gemm(x))
        b = dev_to_bits(dev.gemm(x))
        w12.w12_check_status()
        assert np.array_equal(a, b), f"M={M}"
    out = dev.decode()
    w12.w12_check_status()
    torch.cuda.synchronize()
    assert np.array_equal(dev_to_bits(out), w)


def test_short_buffers():
    import torch
    from gpu_util import to_dev_bf16
    w = wl.forced_escape_weights(256, 4096, 0.10, seed=50)
    wd = to_dev_bf16(w)
    ws = torch.empty(w12.w12_encode_workspace_size(256, 4096), dtype=torch.uint8, device="cuda")
    size = w12.w12_encoded_size_device(wd, ws)
    info = w12.w12_blob_info(oracle.encode(w))
    assert size == info.total_bytes and info.n_escapes > 1000
    # shorter than the packed planes: refused before any launch
    small = torch.zeros(int(info.off_escapes) - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(w12.W12Error) as ei:
        w12.w12_encode_device(wd, small, ws)
    assert ei.value.status == 3
    # room for the planes but not all escapes: found on the device, nothing
    # written past the buffer, no header
    cap = int(info.off_escapes) + 512
    buf = torch.full((size,), 0x5A, dtype=torch.uint8, device="cuda")
    w12.w12_encode_device(wd, buf, ws, nbytes=cap)
    with pytest.raises(w12.W12Error) as ei:
        w12.w12_check_status()
    assert ei.value.status == 3
    host = buf.cpu().numpy()
    assert (host[cap:] == 0x5A).all()
    assert (host[:4] == 0x5A).all(), "header must not be written"
    w12.w12_check_status()  # cleared
    # workspace too small
    with pytest.raises(w12.W12Error) as ei:
        w12.w12_encoded_size_device(wd, ws[:256])
    assert ei.value.status == 3
