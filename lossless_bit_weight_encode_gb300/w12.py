"""Python binding of libw12.so (ctypes).  Argument marshalling only: every step
of the encode, decode and GEMM runs in the library; torch supplies device
memory and streams.  Function names match the C ABI in include/w12.h.

There is no fallback: if the library is missing or a call fails, an exception
is raised.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libw12.so")

W12_OK = 0
NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024  # W12_NOALLOC_SCRATCH_BYTES in include/w12.h
STATUS_NAMES = {
    0: "W12_OK", 1: "W12_ERR_INVALID_ARG", 2: "W12_ERR_SHAPE", 3: "W12_ERR_BUFFER_TOO_SMALL",
    4: "W12_ERR_ALIGNMENT", 5: "W12_ERR_CORRUPT_BLOB", 6: "W12_ERR_UNSUPPORTED_ARCH", 7: "W12_ERR_CUDA",
    8: "W12_ERR_TIMEOUT",
}
EXPORTED = (
    "w12_last_error", "w12_status_string", "w12_format_version", "w12_encoded_size_host", "w12_encode_host",
    "w12_blob_info", "w12_blob_validate", "w12_decode", "w12_gemm_workspace_size", "w12_gemm_launch_info",
    "w12_gemm", "w12_gemm_group_workspace_size", "w12_gemm_group", "w12_gemm_group_launch_info", "w12_gemm_argmax_workspace_size", "w12_gemm_argmax", "w12_gemm_noalloc", "w12_encode_workspace_size", "w12_encoded_size_device", "w12_encode_device",
    "w12_q8_encoded_size", "w12_q8_encode_host", "w12_q8_blob_info", "w12_q8_gemm_workspace_size", "w12_q8_gemm",
    "w12_q8_gemm_group_workspace_size", "w12_q8_gemm_group_launch_info", "w12_q8_gemm_group",
    "w12_read_stream", "w12_check_status", "w12_selftest_timeout", "w12_set_option", "w12_get_option",
)


class W12Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class w12_info(ctypes.Structure):
    _fields_ = [
        ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("N_pad", ctypes.c_int64), ("K_pad", ctypes.c_int64),
        ("tiles", ctypes.c_int64), ("chunks", ctypes.c_int64), ("segs", ctypes.c_int64),
        ("off_seghdr", ctypes.c_uint64), ("bytes_seghdr", ctypes.c_uint64),
        ("off_weights", ctypes.c_uint64), ("bytes_weights", ctypes.c_uint64),
        ("off_escapes", ctypes.c_uint64), ("bytes_escapes", ctypes.c_uint64),
        ("n_escapes", ctypes.c_uint64), ("total_bytes", ctypes.c_uint64),
        ("bits_per_weight", ctypes.c_double),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class w12_q8_info(ctypes.Structure):
    _fields_ = [
        ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("N_pad", ctypes.c_int64), ("K_pad", ctypes.c_int64),
        ("tiles", ctypes.c_int64), ("chunks", ctypes.c_int64), ("segs", ctypes.c_int64),
        ("off_scales", ctypes.c_uint64), ("bytes_scales", ctypes.c_uint64),
        ("off_q", ctypes.c_uint64), ("bytes_q", ctypes.c_uint64), ("total_bytes", ctypes.c_uint64),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"W12 library not built ({LIB_PATH} missing): run __graft_entry__.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, sz, i64, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int64, ctypes.c_int
    L.w12_last_error.restype = ctypes.c_char_p
    L.w12_last_error.argtypes = []
    L.w12_status_string.restype = ctypes.c_char_p
    L.w12_status_string.argtypes = [i32]
    L.w12_format_version.restype = i32
    L.w12_format_version.argtypes = []
    L.w12_encoded_size_host.argtypes = [vp, i64, i64, ctypes.POINTER(sz)]
    L.w12_encode_host.argtypes = [vp, i64, i64, vp, sz]
    L.w12_blob_info.argtypes = [vp, sz, ctypes.POINTER(w12_info)]
    L.w12_blob_validate.argtypes = [vp, sz]
    L.w12_decode.argtypes = [vp, ctypes.POINTER(w12_info), vp, vp]
    L.w12_gemm_workspace_size.argtypes = [ctypes.POINTER(w12_info), i32, ctypes.POINTER(sz)]
    L.w12_gemm_launch_info.argtypes = [ctypes.POINTER(w12_info), i32, ctypes.POINTER(ctypes.c_int32)]
    L.w12_gemm.argtypes = [vp, vp, ctypes.POINTER(w12_info), vp, i32, vp, sz, vp]
    L.w12_gemm_group_workspace_size.argtypes = [i32, ctypes.POINTER(w12_info), i32, ctypes.POINTER(sz)]
    L.w12_gemm_group_launch_info.argtypes = [i32, ctypes.POINTER(w12_info), i32, ctypes.POINTER(ctypes.c_int32)]
    L.w12_gemm_group.argtypes = [vp, i32, ctypes.POINTER(vp), ctypes.POINTER(w12_info), ctypes.POINTER(vp), i32, vp,
                                 sz, vp]
    L.w12_gemm_argmax_workspace_size.argtypes = [ctypes.POINTER(w12_info), i32, ctypes.POINTER(sz)]
    L.w12_gemm_argmax.argtypes = [vp, vp, ctypes.POINTER(w12_info), i32, vp, vp, vp, vp, sz, vp]
    L.w12_gemm_noalloc.argtypes = [vp, vp, ctypes.POINTER(w12_info), vp, i32, vp]
    L.w12_encode_workspace_size.argtypes = [i64, i64, ctypes.POINTER(sz)]
    L.w12_encoded_size_device.argtypes = [vp, i64, i64, vp, sz, ctypes.POINTER(sz), vp]
    L.w12_encode_device.argtypes = [vp, i64, i64, vp, sz, vp, sz, vp]
    L.w12_q8_encoded_size.argtypes = [i64, i64, ctypes.POINTER(sz)]
    L.w12_q8_encode_host.argtypes = [vp, i64, i64, vp, sz]
    L.w12_q8_blob_info.argtypes = [vp, sz, ctypes.POINTER(w12_q8_info)]
    L.w12_q8_gemm_workspace_size.argtypes = [ctypes.POINTER(w12_q8_info), i32, ctypes.POINTER(sz)]
    L.w12_q8_gemm.argtypes = [vp, vp, ctypes.POINTER(w12_q8_info), vp, i32, vp, sz, vp]
    L.w12_q8_gemm_group_workspace_size.argtypes = [i32, ctypes.POINTER(w12_q8_info), i32, ctypes.POINTER(sz)]
    L.w12_q8_gemm_group_launch_info.argtypes = [i32, ctypes.POINTER(w12_q8_info), i32,
                                                ctypes.POINTER(ctypes.c_int32)]
    L.w12_q8_gemm_group.argtypes = [vp, i32, ctypes.POINTER(vp), ctypes.POINTER(w12_q8_info), ctypes.POINTER(vp),
                                    i32, vp, sz, vp]
    L.w12_read_stream.argtypes = [vp, sz, vp, ctypes.c_uint32, vp]
    L.w12_check_status.argtypes = [vp]
    L.w12_selftest_timeout.argtypes = [ctypes.c_uint32, vp]
    L.w12_set_option.argtypes = [ctypes.c_char_p, i64]
    L.w12_get_option.argtypes = [ctypes.c_char_p, ctypes.POINTER(i64)]
    for name in EXPORTED[3:]:
        getattr(L, name).restype = i32
    _lib = L
    return L


def _check(rc: int) -> None:
    if rc != W12_OK:
        raise W12Error(rc, lib().w12_last_error().decode())


def _host_u16(w: np.ndarray) -> np.ndarray:
    w = np.ascontiguousarray(w)
    if w.dtype != np.uint16 or w.ndim != 2:
        raise TypeError("weights must be a 2-D uint16 array of BF16 bit patterns")
    return w


def _stream_handle(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---------------------------------------------------------------- host calls
def w12_encoded_size_host(w: np.ndarray) -> int:
    w = _host_u16(w)
    out = ctypes.c_size_t()
    _check(lib().w12_encoded_size_host(w.ctypes.data, w.shape[0], w.shape[1], ctypes.byref(out)))
    return out.value


def w12_encode_host(w: np.ndarray) -> np.ndarray:
    """Canonical W12 blob (uint8 array) of the N x K BF16 bit patterns `w`."""
    w = _host_u16(w)
    size = w12_encoded_size_host(w)
    blob = np.empty(size, dtype=np.uint8)
    _check(lib().w12_encode_host(w.ctypes.data, w.shape[0], w.shape[1], blob.ctypes.data, size))
    return blob


def w12_blob_info(blob: np.ndarray, blob_bytes: int | None = None) -> w12_info:
    """Header of a host blob; `blob` may be just the 256-byte header of a
    device blob when `blob_bytes` gives that blob's length."""
    blob = np.ascontiguousarray(blob, dtype=np.uint8)
    if blob_bytes is not None and blob.size < 256:
        raise ValueError("the header copy must hold 256 bytes")
    info = w12_info()
    _check(lib().w12_blob_info(blob.ctypes.data, blob.size if blob_bytes is None else int(blob_bytes),
                               ctypes.byref(info)))
    return info


def w12_blob_validate(blob: np.ndarray) -> None:
    blob = np.ascontiguousarray(blob, dtype=np.uint8)
    _check(lib().w12_blob_validate(blob.ctypes.data, blob.size))


# ---------------------------------------------------------------- device calls
def w12_decode(blob_dev, info: w12_info, out_dev, stream=None) -> None:
    """Decode a device blob (torch uint8 tensor) into out_dev (torch int16/bf16 [N, K])."""
    _check(lib().w12_decode(blob_dev.data_ptr(), ctypes.byref(info), out_dev.data_ptr(), _stream_handle(stream)))


def w12_gemm_workspace_size(info: w12_info, M: int) -> int:
    out = ctypes.c_size_t()
    _check(lib().w12_gemm_workspace_size(ctypes.byref(info), int(M), ctypes.byref(out)))
    return out.value


def w12_gemm_launch_info(info: w12_info, M: int) -> dict:
    out = (ctypes.c_int32 * 4)()
    _check(lib().w12_gemm_launch_info(ctypes.byref(info), int(M), out))
    return {"ntok": out[0], "splits": out[1], "ctas": out[2], "ctas_per_sm": out[3]}


def w12_gemm(x_dev, blob_dev, info: w12_info, y_dev, M: int, workspace, stream=None) -> None:
    """y_dev[M, N] = x_dev[M, K] . W^T on the device (torch tensors, BF16)."""
    _check(lib().w12_gemm(x_dev.data_ptr(), blob_dev.data_ptr(), ctypes.byref(info), y_dev.data_ptr(), int(M),
                          workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                          _stream_handle(stream)))


def w12_gemm_ptr(x_ptr: int, blob_ptr: int, info: w12_info, y_ptr: int, M: int, ws_ptr: int, ws_bytes: int,
                 stream_handle: int | None) -> int:
    """Raw-pointer form of w12_gemm that returns the status instead of raising
    (for timing loops that check once at the end)."""
    return lib().w12_gemm(x_ptr, blob_ptr, ctypes.byref(info), y_ptr, int(M), ws_ptr, ws_bytes, stream_handle)


MAX_GROUP = 4  # W12_MAX_GROUP in include/w12.h


def _infos(infos) -> ctypes.Array:
    return (w12_info * len(infos))(*infos)


def w12_gemm_group_workspace_size(infos, M: int) -> int:
    out = ctypes.c_size_t()
    _check(lib().w12_gemm_group_workspace_size(len(infos), _infos(infos), int(M), ctypes.byref(out)))
    return out.value


KERNEL_NAMES = {0: "w12_gemv_kernel", 1: "w12_gemv_sm_kernel", 2: "w12_gemm_tc_kernel", 3: "w12_gemm_tc_sm_kernel"}


def w12_gemm_group_launch_info(infos, M: int) -> dict:
    """Plan of a grouped launch (one info: a single w12_gemm), with the name
    of the kernel that runs it."""
    out = (ctypes.c_int32 * 5)()
    _check(lib().w12_gemm_group_launch_info(len(infos), _infos(infos), int(M), out))
    return {"ntok": out[0], "splits": out[1], "ctas": out[2], "ctas_per_sm": out[3], "kernel": out[4],
            "kernel_name": KERNEL_NAMES.get(out[4], str(out[4]))}


def w12_gemm_group_ptr(x_ptr: int, blob_ptrs, infos, y_ptrs, M: int, ws_ptr: int, ws_bytes: int,
                       stream_handle: int | None) -> int:
    """Raw-pointer form of w12_gemm_group that returns the status."""
    n = len(infos)
    return lib().w12_gemm_group(x_ptr, n, (ctypes.c_void_p * n)(*blob_ptrs), _infos(infos),
                                (ctypes.c_void_p * n)(*y_ptrs), int(M), ws_ptr, ws_bytes, stream_handle)


def w12_gemm_group(x_dev, blobs_dev, infos, ys_dev, M: int, workspace, stream=None) -> None:
    """ys_dev[i] = x_dev . W_i^T for matrices sharing K, in one launch."""
    _check(w12_gemm_group_ptr(x_dev.data_ptr(), [b.data_ptr() for b in blobs_dev], infos,
                              [y.data_ptr() for y in ys_dev], M, workspace.data_ptr(),
                              workspace.numel() * workspace.element_size(), _stream_handle(stream)))


def w12_gemm_argmax_ptr(x_ptr: int, blob_ptr: int, info: w12_info, M: int, y_ptr: int | None, idx_ptr: int,
                        val_ptr: int, ws_ptr: int, ws_bytes: int, stream_handle: int | None) -> int:
    """Raw-pointer form of w12_gemm_argmax that returns the status."""
    return lib().w12_gemm_argmax(x_ptr, blob_ptr, ctypes.byref(info), int(M), y_ptr, idx_ptr, val_ptr, ws_ptr,
                                 ws_bytes, stream_handle)


def w12_gemm_argmax_workspace_size(info: w12_info, M: int) -> int:
    out = ctypes.c_size_t()
    _check(lib().w12_gemm_argmax_workspace_size(ctypes.byref(info), int(M), ctypes.byref(out)))
    return out.value


def w12_gemm_argmax(x_dev, blob_dev, info: w12_info, M: int, y_dev, idx_dev, val_dev, workspace,
                    stream=None) -> None:
    """Argmax over rows of x . W^T per token (int32 idx_dev[M], float val_dev[M]);
    y_dev (BF16 [M, N]) may be None."""
    _check(lib().w12_gemm_argmax(x_dev.data_ptr(), blob_dev.data_ptr(), ctypes.byref(info), int(M),
                                 None if y_dev is None else y_dev.data_ptr(), idx_dev.data_ptr(),
                                 val_dev.data_ptr(), workspace.data_ptr(),
                                 workspace.numel() * workspace.element_size(), _stream_handle(stream)))


def w12_gemm_noalloc(x_dev, blob_dev, info: w12_info, y_dev, M: int, stream=None) -> None:
    """w12_gemm without a workspace argument: the library's fixed static
    scratch is used (see include/w12.h); nothing is allocated."""
    _check(lib().w12_gemm_noalloc(x_dev.data_ptr(), blob_dev.data_ptr(), ctypes.byref(info), y_dev.data_ptr(),
                                  int(M), _stream_handle(stream)))


def _dev_u16(w) -> tuple[int, int]:
    import torch
    if w.dim() != 2 or w.dtype not in (torch.bfloat16, torch.int16, torch.uint16) or not w.is_contiguous():
        raise TypeError("weights must be a contiguous 2-D BF16 (or 16-bit integer) device tensor")
    return int(w.shape[0]), int(w.shape[1])


def w12_encode_workspace_size(N: int, K: int) -> int:
    out = ctypes.c_size_t()
    _check(lib().w12_encode_workspace_size(int(N), int(K), ctypes.byref(out)))
    return out.value


def w12_encoded_size_device(w_dev, workspace, stream=None) -> int:
    """Exact blob size of the device weights `w_dev` (synchronises the stream)."""
    N, K = _dev_u16(w_dev)
    out = ctypes.c_size_t()
    _check(lib().w12_encoded_size_device(w_dev.data_ptr(), N, K, workspace.data_ptr(),
                                         workspace.numel() * workspace.element_size(), ctypes.byref(out),
                                         _stream_handle(stream)))
    return out.value


def w12_encode_device(w_dev, blob_dev, workspace, stream=None, nbytes: int | None = None) -> None:
    """Encode `w_dev` into the uint8 device tensor `blob_dev` (asynchronous;
    device-side errors surface through w12_check_status)."""
    N, K = _dev_u16(w_dev)
    cap = blob_dev.numel() if nbytes is None else int(nbytes)
    _check(lib().w12_encode_device(w_dev.data_ptr(), N, K, blob_dev.data_ptr(), cap, workspace.data_ptr(),
                                   workspace.numel() * workspace.element_size(), _stream_handle(stream)))


# ---------------------------------------------------------------- Q8 copy
def w12_q8_encode_host(w: np.ndarray) -> np.ndarray:
    """Q8 v1 blob (symmetric INT8 per row) of the N x K BF16 bit patterns."""
    w = _host_u16(w)
    size = ctypes.c_size_t()
    _check(lib().w12_q8_encoded_size(w.shape[0], w.shape[1], ctypes.byref(size)))
    blob = np.empty(size.value, dtype=np.uint8)
    _check(lib().w12_q8_encode_host(w.ctypes.data, w.shape[0], w.shape[1], blob.ctypes.data, size.value))
    return blob


def w12_q8_blob_info(blob: np.ndarray, blob_bytes: int | None = None) -> w12_q8_info:
    blob = np.ascontiguousarray(blob, dtype=np.uint8)
    info = w12_q8_info()
    _check(lib().w12_q8_blob_info(blob.ctypes.data, blob.size if blob_bytes is None else int(blob_bytes),
                                  ctypes.byref(info)))
    return info


def w12_q8_gemm_workspace_size(info: w12_q8_info, M: int) -> int:
    out = ctypes.c_size_t()
    _check(lib().w12_q8_gemm_workspace_size(ctypes.byref(info), int(M), ctypes.byref(out)))
    return out.value


def w12_q8_gemm(x_dev, blob_dev, info: w12_q8_info, y_dev, M: int, workspace, stream=None) -> None:
    _check(lib().w12_q8_gemm(x_dev.data_ptr(), blob_dev.data_ptr(), ctypes.byref(info), y_dev.data_ptr(), int(M),
                             workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                             _stream_handle(stream)))


def w12_q8_gemm_ptr(x_ptr: int, blob_ptr: int, info: w12_q8_info, y_ptr: int, M: int, ws_ptr: int, ws_bytes: int,
                    stream_handle: int | None) -> int:
    """Raw-pointer form of w12_q8_gemm that returns the status."""
    return lib().w12_q8_gemm(x_ptr, blob_ptr, ctypes.byref(info), y_ptr, int(M), ws_ptr, ws_bytes, stream_handle)


def _q8_infos(infos) -> ctypes.Array:
    return (w12_q8_info * len(infos))(*infos)


def w12_q8_gemm_group_workspace_size(infos, M: int) -> int:
    out = ctypes.c_size_t()
    _check(lib().w12_q8_gemm_group_workspace_size(len(infos), _q8_infos(infos), int(M), ctypes.byref(out)))
    return out.value


def w12_q8_gemm_group_launch_info(infos, M: int) -> dict:
    """Plan of a grouped Q8 launch (one info: a single w12_q8_gemm)."""
    out = (ctypes.c_int32 * 5)()
    _check(lib().w12_q8_gemm_group_launch_info(len(infos), _q8_infos(infos), int(M), out))
    return {"ntok": out[0], "splits": out[1], "ctas": out[2], "ctas_per_sm": out[3], "kernel": out[4],
            "kernel_name": KERNEL_NAMES.get(out[4], str(out[4]))}


def w12_q8_gemm_group_ptr(x_ptr: int, blob_ptrs, infos, y_ptrs, M: int, ws_ptr: int, ws_bytes: int,
                          stream_handle: int | None) -> int:
    """Raw-pointer form of w12_q8_gemm_group that returns the status."""
    n = len(infos)
    return lib().w12_q8_gemm_group(x_ptr, n, (ctypes.c_void_p * n)(*blob_ptrs), _q8_infos(infos),
                                   (ctypes.c_void_p * n)(*y_ptrs), int(M), ws_ptr, ws_bytes, stream_handle)


def w12_q8_gemm_group(x_dev, blobs_dev, infos, ys_dev, M: int, workspace, stream=None) -> None:
    """ys_dev[i] = the Q8 product of x_dev with copy i, for copies sharing K, in one launch."""
    _check(w12_q8_gemm_group_ptr(x_dev.data_ptr(), [b.data_ptr() for b in blobs_dev], infos,
                                 [y.data_ptr() for y in ys_dev], M, workspace.data_ptr(),
                                 workspace.numel() * workspace.element_size(), _stream_handle(stream)))


def w12_read_stream_ptr(buf_ptr: int, nbytes: int, sink_ptr: int, never: int, stream_handle: int | None) -> int:
    """Raw-pointer form of w12_read_stream (the HBM read ceiling) that returns the status."""
    return lib().w12_read_stream(buf_ptr, nbytes, sink_ptr, never, stream_handle)


def w12_check_status(stream=None) -> None:
    _check(lib().w12_check_status(_stream_handle(stream)))


def w12_set_option(name: str, value: int) -> None:
    _check(lib().w12_set_option(name.encode(), int(value)))


def w12_get_option(name: str) -> int:
    out = ctypes.c_int64()
    _check(lib().w12_get_option(name.encode(), ctypes.byref(out)))
    return out.value


class options:
    """Context manager: set launch options (w12_set_option) for a block and
    put the previous values back afterwards, e.g.
    ``with w12.options(token_tile=16, a_operand_smem=1): ...``."""

    def __init__(self, **values):
        self.values = values
        self.saved = {}

    def __enter__(self):
        for name, v in self.values.items():
            self.saved[name] = w12_get_option(name)
            w12_set_option(name, v)
        return self

    def __exit__(self, *exc):
        for name, v in self.saved.items():
            w12_set_option(name, v)
        return False


def w12_selftest_timeout(timeout_us: int, stream=None) -> None:
    _check(lib().w12_selftest_timeout(int(timeout_us), _stream_handle(stream)))


def w12_last_error() -> str:
    return lib().w12_last_error().decode()
