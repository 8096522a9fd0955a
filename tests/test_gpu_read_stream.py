"""The read-stream helper behind the bench's HBM read ceiling: it reads every
16-byte word it is given and writes its sink only when the fold of what it
read equals `never`."""
import numpy as np
import pytest

from lossless_bit_weight_encode_gb300 import w12

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from gpu_util import ensure_built
    ensure_built()


@pytest.mark.parametrize("nwords", [1, 7, 4096, 1 << 20, (1 << 20) + 3])
def test_read_stream_reads_every_word(nwords):
    import torch
    rng = np.random.default_rng(nwords)
    for pos in {0, nwords - 1, int(rng.integers(0, nwords))}:
        buf = torch.zeros(4 * nwords, dtype=torch.int32, device="cuda")
        buf[4 * pos + 2] = 0x5A5A5A5A  # the only nonzero word: one thread folds to it
        sink = torch.zeros(4, dtype=torch.int32, device="cuda")
        assert w12.w12_read_stream_ptr(buf.data_ptr(), 16 * nwords, sink.data_ptr(), 0x5A5A5A5A, None) == 0
        w12.w12_check_status()
        assert int(sink[0]) == 0x5A5A5A5A, (nwords, pos)
        sink.zero_()
        assert w12.w12_read_stream_ptr(buf.data_ptr(), 16 * nwords, sink.data_ptr(), 0x12345678, None) == 0
        w12.w12_check_status()
        assert int(sink[0]) == 0, (nwords, pos)
