"""GPU decode (W12 -> BF16) through the C ABI: bit-exact against the original
weights ("decodes bit-exactly": StargazerX0/SpecPilot, §What it is)."""
import numpy as np
import pytest

from lossless_bit_weight_encode_gb300 import W12Weight, w12
from lossless_bit_weight_encode_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from gpu_util import ensure_built
    ensure_built()


def _roundtrip(w):
    import torch
    from gpu_util import dev_to_bits
    mat = W12Weight(w)
    out = mat.decode()
    w12.w12_check_status()
    torch.cuda.synchronize()
    got = dev_to_bits(out)
    assert got.shape == w.shape
    diff = got != w
    assert not diff.any(), f"{int(diff.sum())} mismatches, first at {np.argwhere(diff)[0]}"


@pytest.mark.parametrize("shuffle", [None, 5])
def test_exhaustive_patterns(shuffle):
    _roundtrip(wl.all_bf16_patterns(shuffle))


@pytest.mark.parametrize("shape", [(1, 1), (1, 33), (127, 255), (129, 257), (300, 1000), (1000, 1001)])
def test_ragged_shapes(shape):
    _roundtrip(wl.gaussian_weights(*shape, seed=sum(shape)))


@pytest.mark.parametrize("frac", [0.02, 0.10, 1.0])
def test_forced_escapes(frac):
    _roundtrip(wl.forced_escape_weights(384, 2048, frac, seed=int(frac * 100)))


def test_special_values():
    v = np.array([0x0000, 0x8000, 0x0001, 0x807F, 0x7F80, 0xFF80, 0x7FC0, 0xFFFF, 0x7F81, 0x3F80],
                 dtype=np.uint16)
    _roundtrip(np.resize(v, 256 * 320).reshape(256, 320))


@pytest.mark.parametrize("workload", ["layer", "heavy"])
def test_layer_shapes_decode_exactly(workload):
    for name, w in wl.layer_weights(workload):
        _roundtrip(w)
