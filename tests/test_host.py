"""Host side of the library on CPU: the C ABI loads and exports every symbol
include/w12.h declares; the library's encoder is byte-equal to the oracle's;
header parsing and blob validation accept good blobs and reject bad ones."""
import os
import re

import numpy as np
import pytest

import oracle
from lossless_bit_weight_encode_gb300 import build as libbuild
from lossless_bit_weight_encode_gb300 import w12
from lossless_bit_weight_encode_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    libbuild.build()
    oracle.build()


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "w12.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(w12_\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = w12.lib()
    declared = _declared_symbols()
    assert len(declared) >= 12
    for name in declared:
        assert hasattr(lib, name), name
    assert set(declared) == set(w12.EXPORTED)
    assert lib.w12_format_version() == 1
    for code, name in w12.STATUS_NAMES.items():
        assert lib.w12_status_string(code).decode() == name


CASES = {
    "exhaustive": lambda: wl.all_bf16_patterns(),
    "exhaustive_shuffled": lambda: wl.all_bf16_patterns(77),
    "single": lambda: wl.single_case()[0],
    "ragged_small": lambda: wl.gaussian_weights(1, 1, seed=1),
    "ragged": lambda: wl.gaussian_weights(333, 777, seed=2),
    "heavy": lambda: wl.heavy_tail_weights(384, 2048, seed=3),
    "forced2": lambda: wl.forced_escape_weights(256, 1024, 0.02, seed=4),
    "forced10": lambda: wl.forced_escape_weights(130, 1000, 0.10, seed=5),
    "forced100": lambda: wl.forced_escape_weights(128, 512, 1.0, seed=6),
    "zeros": lambda: np.zeros((200, 300), dtype=np.uint16),
    "big_exponents": lambda: (wl.gaussian_weights(256, 512, seed=7) | np.uint16(0x4000)),
    "table_rule": lambda: wl.table_rule_weights(8),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_encoder_is_byte_equal_to_oracle(case):
    w = CASES[case]()
    ref = oracle.encode(w)
    assert w12.w12_encoded_size_host(w) == ref.size
    blob = w12.w12_encode_host(w)
    assert blob.size == ref.size
    assert np.array_equal(blob, ref), f"first difference at byte {int(np.argmax(blob != ref))}"
    w12.w12_blob_validate(blob)
    assert np.array_equal(oracle.decode(blob), w)


def test_blob_info_fields():
    w = wl.heavy_tail_weights(300, 1000, seed=8)
    blob = w12.w12_encode_host(w)
    info = w12.w12_blob_info(blob)
    assert (info.N, info.K, info.N_pad, info.K_pad) == (300, 1000, 384, 1024)
    assert (info.tiles, info.chunks, info.segs) == (3, 32, 4)
    assert info.off_seghdr == 256 and info.bytes_seghdr == 32 * 12
    assert info.off_weights == 768 and info.bytes_weights == 6144 * 96  # 256 + 384 rounded up to 256
    assert info.off_escapes == 768 + 6144 * 96
    assert info.total_bytes == blob.size
    assert info.bytes_escapes == -(-info.n_escapes // 16) * 16
    assert abs(info.bits_per_weight - 8.0 * blob.size / (300 * 1000)) < 1e-12


def _expect(status, fn, *args):
    with pytest.raises(w12.W12Error) as ei:
        fn(*args)
    assert ei.value.status == status, str(ei.value)
    assert w12.w12_last_error() != ""


def test_rejects_bad_blobs():
    w = wl.forced_escape_weights(256, 600, 0.05, seed=9)
    blob = w12.w12_encode_host(w)
    _expect(3, w12.w12_blob_info, blob[:100])          # shorter than the header
    _expect(3, w12.w12_blob_info, blob[:-256])         # shorter than its total size
    bad = blob.copy(); bad[1] ^= 1
    _expect(5, w12.w12_blob_info, bad)                 # magic
    bad = blob.copy(); bad[4] = 2
    _expect(5, w12.w12_blob_info, bad)                 # version
    bad = blob.copy(); bad[0x48] ^= 1
    _expect(5, w12.w12_blob_info, bad)                 # chunk count
    seg0 = 256
    bad = blob.copy(); bad[seg0 + 15] = 3
    _expect(5, w12.w12_blob_validate, bad)             # escape slot must hold 0
    bad = blob.copy(); bad[seg0 + 0] ^= 0x80
    _expect(5, w12.w12_blob_validate, bad)             # paired slots on different top bits
    bad = blob.copy(); bad[seg0 + 32 + 16] ^= 1
    _expect(5, w12.w12_blob_validate, bad)             # second segment's escape offset
    bad = blob.copy(); bad[seg0 + 20] ^= 1
    _expect(5, w12.w12_blob_validate, bad)             # quarter count
    bad = blob.copy(); bad[seg0 + 28:seg0 + 32] = 0
    _expect(5, w12.w12_blob_validate, bad)             # mask disagrees with the counts


def test_host_argument_errors():
    lib = w12.lib()
    import ctypes
    out = ctypes.c_size_t()
    w = np.zeros((4, 4), dtype=np.uint16)
    assert lib.w12_encoded_size_host(None, 4, 4, ctypes.byref(out)) == 1
    assert lib.w12_encoded_size_host(w.ctypes.data, 0, 4, ctypes.byref(out)) == 2
    assert lib.w12_encoded_size_host(w.ctypes.data, 4, -1, ctypes.byref(out)) == 2
    size = w12.w12_encoded_size_host(w)
    buf = np.empty(size, dtype=np.uint8)
    assert lib.w12_encode_host(w.ctypes.data, 4, 4, buf.ctypes.data, size - 1) == 3
    assert lib.w12_encode_host(w.ctypes.data, 4, 4, buf.ctypes.data, size) == 0


Q8_CASES = {
    "gauss": lambda: wl.gaussian_weights(300, 1000, seed=20),
    "heavy": lambda: wl.heavy_tail_weights(129, 4099, seed=21),
    "tiny": lambda: wl.gaussian_weights(1, 1, seed=22),
    "zero_rows": lambda: np.where(np.arange(200)[:, None] % 3 == 0, np.uint16(0),
                                  wl.gaussian_weights(200, 70, seed=23)).astype(np.uint16),
    "ties": lambda: wl.to_bf16_bits(np.tile(np.array([127, 32.5, 33.5, -0.5, 1.5], np.float32) / 64, (3, 7))),
}


@pytest.mark.parametrize("case", sorted(Q8_CASES))
def test_q8_encoder_is_byte_equal_to_oracle(case):
    w = Q8_CASES[case]()
    ref = oracle.q8_encode(w)
    blob = w12.w12_q8_encode_host(w)
    assert np.array_equal(blob, ref), f"first difference at byte {int(np.argmax(blob != ref))}"
    info = w12.w12_q8_blob_info(blob)
    assert (info.N, info.K, info.total_bytes) == (w.shape[0], w.shape[1], ref.size)
    assert w12.w12_q8_blob_info(blob[:256], blob.size).as_dict() == info.as_dict()


def test_q8_rejects_bad_input():
    w = wl.gaussian_weights(10, 10, seed=24)
    w[4, 4] = np.uint16(0x7FC0)  # NaN
    with pytest.raises(w12.W12Error) as ei:
        w12.w12_q8_encode_host(w)
    assert ei.value.status == 1
    blob = w12.w12_q8_encode_host(wl.gaussian_weights(10, 10, seed=25))
    bad = blob.copy()
    bad[0x11] ^= 1  # N grows by 256: the padded geometry no longer matches
    with pytest.raises(w12.W12Error) as ei:
        w12.w12_q8_blob_info(bad)
    assert ei.value.status == 5
    with pytest.raises(w12.W12Error) as ei:
        w12.w12_q8_blob_info(oracle.encode(wl.gaussian_weights(10, 10, seed=26)))  # a W12 blob
    assert ei.value.status == 5


def test_gemm_argument_errors_before_any_device_work():
    """The GEMM entry points reject bad arguments with the documented codes
    before they touch a device (the pointers below are never dereferenced)."""
    import ctypes
    lib = w12.lib()
    a = 0x100000  # a 256-byte aligned stand-in for a device pointer
    info = w12.w12_blob_info(w12.w12_encode_host(wl.gaussian_weights(200, 300, seed=40)))
    other_k = w12.w12_blob_info(w12.w12_encode_host(wl.gaussian_weights(130, 64, seed=41)))
    INVALID, SHAPE, ALIGN = 1, 2, 4
    # w12_gemm: null pointers, token count, alignment
    assert w12.w12_gemm_ptr(0, a, info, a, 1, a, 1 << 20, None) == INVALID
    assert w12.w12_gemm_ptr(a, a, info, a, 0, a, 1 << 20, None) == INVALID
    assert w12.w12_gemm_ptr(a, a, info, a, 33, a, 1 << 20, None) == INVALID
    assert w12.w12_gemm_ptr(a, a + 16, info, a, 1, a, 1 << 20, None) == ALIGN
    assert w12.w12_gemm_ptr(a, a, info, a + 1, 1, a, 1 << 20, None) == ALIGN
    assert w12.w12_gemm_ptr(a, a, info, a, 1, a + 128, 1 << 20, None) == ALIGN
    out = (ctypes.c_int32 * 4)()
    assert lib.w12_gemm_launch_info(ctypes.byref(info), 0, out) == INVALID
    assert lib.w12_gemm_launch_info(ctypes.byref(info), 33, out) == INVALID
    # grouped launch: member count, shared K, null and misaligned members
    assert w12.w12_gemm_group_ptr(a, [], [], [], 1, a, 1 << 20, None) == INVALID
    five = [info] * (w12.MAX_GROUP + 1)
    assert w12.w12_gemm_group_ptr(a, [a] * 5, five, [a] * 5, 1, a, 1 << 20, None) == INVALID
    assert w12.w12_gemm_group_ptr(a, [a, a], [info, other_k], [a, a], 1, a, 1 << 20, None) == SHAPE
    assert w12.w12_gemm_group_ptr(a, [a, 0], [info, info], [a, a], 1, a, 1 << 20, None) == INVALID
    assert w12.w12_gemm_group_ptr(a, [a, a], [info, info], [a, a + 1], 1, a, 1 << 20, None) == ALIGN
    assert w12.w12_gemm_group_ptr(a, [a, a], [info, info], [a, a], 40, a, 1 << 20, None) == INVALID
    # fused argmax: index and value outputs are required and 4-byte aligned
    assert w12.w12_gemm_argmax_ptr(a, a, info, 1, None, 0, a, a, 1 << 20, None) == INVALID
    assert w12.w12_gemm_argmax_ptr(a, a, info, 1, None, a + 2, a, a, 1 << 20, None) == ALIGN
    # allocation-free entry point
    assert lib.w12_gemm_noalloc(a, a, ctypes.byref(info), None, 1, None) == INVALID
    assert lib.w12_gemm_noalloc(a, a, ctypes.byref(info), a, 0, None) == INVALID
    # Q8 copy
    q8 = w12.w12_q8_blob_info(w12.w12_q8_encode_host(wl.gaussian_weights(200, 300, seed=42)))
    assert w12.w12_q8_gemm_ptr(0, a, q8, a, 1, a, 1 << 20, None) == INVALID
    assert w12.w12_q8_gemm_ptr(a, a + 8, q8, a, 1, a, 1 << 20, None) == ALIGN
    # grouped Q8 launch: member count, shared K, a W12 info in place of a Q8
    # one, null and misaligned members
    q8_other_k = w12.w12_q8_blob_info(w12.w12_q8_encode_host(wl.gaussian_weights(130, 64, seed=43)))
    assert w12.w12_q8_gemm_group_ptr(a, [], [], [], 1, a, 1 << 20, None) == INVALID
    assert w12.w12_q8_gemm_group_ptr(a, [a] * 5, [q8] * 5, [a] * 5, 1, a, 1 << 20, None) == INVALID
    assert w12.w12_q8_gemm_group_ptr(a, [a, a], [q8, q8_other_k], [a, a], 1, a, 1 << 20, None) == SHAPE
    assert w12.w12_q8_gemm_group_ptr(a, [a, 0], [q8, q8], [a, a], 1, a, 1 << 20, None) == INVALID
    assert w12.w12_q8_gemm_group_ptr(a, [a, a + 64], [q8, q8], [a, a], 1, a, 1 << 20, None) == ALIGN
    assert w12.w12_q8_gemm_group_ptr(a, [a, a], [q8, q8], [a, a], 33, a, 1 << 20, None) == INVALID
    bad = w12.w12_q8_info()
    bad.N, bad.K = q8.N, q8.K  # geometry fields left at zero
    assert w12.w12_q8_gemm_group_ptr(a, [a], [bad], [a], 1, a, 1 << 20, None) != 0
    out5 = (ctypes.c_int32 * 5)()
    assert lib.w12_q8_gemm_group_launch_info(0, None, 1, out5) == INVALID
    # read-stream helper: null buffer or sink, misaligned buffer or size
    assert w12.w12_read_stream_ptr(0, 16, a, 0, None) == INVALID
    assert w12.w12_read_stream_ptr(a, 16, 0, 0, None) == INVALID
    assert w12.w12_read_stream_ptr(a + 8, 16, a, 0, None) == ALIGN
    assert w12.w12_read_stream_ptr(a, 24, a, 0, None) == ALIGN
    assert w12.w12_last_error() != ""


def test_launch_options_set_get_and_reject(monkeypatch):
    """Launch options come only from w12_set_option: unknown names and values
    out of range are refused (nothing changes), and an environment variable
    named like an option has no effect."""
    from lossless_bit_weight_encode_gb300 import w12
    defaults = {"gemv_max_m": 2, "token_tile": 0, "a_operand_smem": 0, "gemv_sm": -1, "stream_k": 1,
                "splits": 0, "pdl": 1, "timeout_ms": 4000, "tc_sm": 1}
    for name, v in defaults.items():
        assert w12.w12_get_option(name) == v, name
    monkeypatch.setenv("W12_NTOK", "16")
    monkeypatch.setenv("W12_GEMV_MAX_M", "1")
    assert w12.w12_get_option("token_tile") == 0 and w12.w12_get_option("gemv_max_m") == 2
    with w12.options(token_tile=16, gemv_sm=0, timeout_ms=25):
        assert w12.w12_get_option("token_tile") == 16
        assert w12.w12_get_option("gemv_sm") == 0 and w12.w12_get_option("timeout_ms") == 25
    for name, v in defaults.items():
        assert w12.w12_get_option(name) == v, name
    for name, bad in [("token_tile", 8), ("token_tile", 33), ("gemv_max_m", 3), ("gemv_sm", -2), ("pdl", 2),
                      ("timeout_ms", 0), ("no_such_option", 1)]:
        with pytest.raises(w12.W12Error) as e:
            w12.w12_set_option(name, bad)
        assert e.value.status == 1
    assert w12.w12_get_option("token_tile") == 0
    with pytest.raises(w12.W12Error):
        w12.w12_get_option("no_such_option")
