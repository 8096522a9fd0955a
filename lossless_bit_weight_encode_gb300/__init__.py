"""W12: lossless ~12-bit BF16 weights decoded inside the GEMM, for GB300 (sm_103a).

``w12`` is the ctypes binding of libw12.so (C ABI in include/w12.h);
``W12Weight`` is a small convenience holder built on it (torch provides the
device memory and the stream).  ``workloads`` draws the seeded synthetic inputs.
"""
from __future__ import annotations

import numpy as np

from . import w12
from .w12 import W12Error

__all__ = ["w12", "W12Error", "W12Weight", "W12Group", "Q8Weight", "Q8Group"]


class W12Weight:
    """A weight matrix held on the device in W12 form.

    ``W12Weight(bits)`` encodes the N x K BF16 bit patterns (numpy uint16) on
    the host with the library's encoder and copies the blob to the current CUDA
    device.  ``gemm(x)`` returns ``x . W^T`` (BF16) for x of shape [M, K],
    1 <= M <= 32; ``decode()`` returns W (BF16) bit-exactly.
    """

    def __init__(self, bits: np.ndarray, device=None):
        import torch

        self.blob_host = w12.w12_encode_host(bits)
        self.info = w12.w12_blob_info(self.blob_host)
        self.N, self.K = int(self.info.N), int(self.info.K)
        dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.blob = torch.from_numpy(self.blob_host).to(dev)
        self._ws = {}

    @classmethod
    def from_device(cls, w, stream=None) -> "W12Weight":
        """Encode a BF16 device tensor [N, K] on its GPU (same bytes as the
        host encoder); only the 256-byte header comes back to the host."""
        import torch

        N, K = int(w.shape[0]), int(w.shape[1])
        ws = torch.empty(w12.w12_encode_workspace_size(N, K), dtype=torch.uint8, device=w.device)
        size = w12.w12_encoded_size_device(w, ws, stream)
        blob = torch.empty(size, dtype=torch.uint8, device=w.device)
        w12.w12_encode_device(w, blob, ws, stream)
        w12.w12_check_status(stream)
        self = cls.__new__(cls)
        self.blob_host = None
        self.info = w12.w12_blob_info(blob[:256].cpu().numpy(), size)
        self.N, self.K = int(self.info.N), int(self.info.K)
        self.blob = blob
        self._ws = {}
        return self

    @property
    def bits_per_weight(self) -> float:
        return float(self.info.bits_per_weight)

    def workspace(self, M: int):
        import torch

        size = w12.w12_gemm_workspace_size(self.info, M)
        ws = self._ws.get(M)
        if ws is None or ws.numel() < size:
            ws = torch.zeros(max(size, 256), dtype=torch.uint8, device=self.blob.device)
            self._ws[M] = ws
        return ws

    def gemm(self, x, out=None, stream=None):
        import torch

        if x.dtype != torch.bfloat16 or x.dim() != 2 or x.shape[1] != self.K or not x.is_contiguous():
            raise ValueError("x must be a contiguous BF16 tensor of shape [M, K]")
        M = int(x.shape[0])
        if out is None:
            out = torch.empty((M, self.N), dtype=torch.bfloat16, device=x.device)
        w12.w12_gemm(x, self.blob, self.info, out, M, self.workspace(M), stream)
        return out

    def argmax_workspace(self, M: int):
        import torch

        size = w12.w12_gemm_argmax_workspace_size(self.info, M)
        key = ("argmax", M)
        ws = self._ws.get(key)
        if ws is None or ws.numel() < size:
            ws = torch.zeros(max(size, 256), dtype=torch.uint8, device=self.blob.device)
            self._ws[key] = ws
        return ws

    def gemm_argmax(self, x, logits: bool = False, stream=None):
        """Per token: (row index int32 [M], fp32 logit [M]) of the largest
        entry of x . W^T (ties to the lowest row), plus the BF16 logits
        [M, N] when `logits` is set (else None)."""
        import torch

        if x.dtype != torch.bfloat16 or x.dim() != 2 or x.shape[1] != self.K or not x.is_contiguous():
            raise ValueError("x must be a contiguous BF16 tensor of shape [M, K]")
        M = int(x.shape[0])
        idx = torch.empty(M, dtype=torch.int32, device=x.device)
        val = torch.empty(M, dtype=torch.float32, device=x.device)
        y = torch.empty((M, self.N), dtype=torch.bfloat16, device=x.device) if logits else None
        w12.w12_gemm_argmax(x, self.blob, self.info, M, y, idx, val, self.argmax_workspace(M), stream)
        return idx, val, y

    def decode(self, out=None, stream=None):
        import torch

        if out is None:
            out = torch.empty((self.N, self.K), dtype=torch.bfloat16, device=self.blob.device)
        w12.w12_decode(self.blob, self.info, out, stream)
        return out


class W12Group:
    """Matrices that multiply the same x (q/k/v, or gate/up), run as one
    launch: ``gemm(x)`` returns one BF16 output per matrix."""

    def __init__(self, mats):
        if not 1 <= len(mats) <= w12.MAX_GROUP or len({m.K for m in mats}) != 1:
            raise ValueError(f"1..{w12.MAX_GROUP} matrices with the same K")
        self.mats = list(mats)
        self.K = mats[0].K
        self.infos = [m.info for m in mats]
        self._ws = {}

    def workspace(self, M: int):
        import torch

        size = w12.w12_gemm_group_workspace_size(self.infos, M)
        ws = self._ws.get(M)
        if ws is None or ws.numel() < size:
            ws = torch.zeros(max(size, 256), dtype=torch.uint8, device=self.mats[0].blob.device)
            self._ws[M] = ws
        return ws

    def gemm(self, x, outs=None, stream=None):
        import torch

        if x.dtype != torch.bfloat16 or x.dim() != 2 or x.shape[1] != self.K or not x.is_contiguous():
            raise ValueError("x must be a contiguous BF16 tensor of shape [M, K]")
        M = int(x.shape[0])
        if outs is None:
            outs = [torch.empty((M, m.N), dtype=torch.bfloat16, device=x.device) for m in self.mats]
        w12.w12_gemm_group(x, [m.blob for m in self.mats], self.infos, outs, M, self.workspace(M), stream)
        return outs


class Q8Weight:
    """The 8-bit (symmetric INT8 per row) copy of a weight matrix on the
    device, for the first level of a two-level verification.  Lossy by design:
    ``gemm(x)`` returns ``x . (s * q)^T`` (BF16) for x [M, K], 1 <= M <= 32."""

    def __init__(self, bits: np.ndarray, device=None):
        import torch

        self.blob_host = w12.w12_q8_encode_host(bits)
        self.info = w12.w12_q8_blob_info(self.blob_host)
        self.N, self.K = int(self.info.N), int(self.info.K)
        dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.blob = torch.from_numpy(self.blob_host).to(dev)
        self._ws = {}

    def workspace(self, M: int):
        import torch

        size = w12.w12_q8_gemm_workspace_size(self.info, M)
        ws = self._ws.get(M)
        if ws is None or ws.numel() < size:
            ws = torch.zeros(max(size, 256), dtype=torch.uint8, device=self.blob.device)
            self._ws[M] = ws
        return ws

    def gemm(self, x, out=None, stream=None):
        import torch

        if x.dtype != torch.bfloat16 or x.dim() != 2 or x.shape[1] != self.K or not x.is_contiguous():
            raise ValueError("x must be a contiguous BF16 tensor of shape [M, K]")
        M = int(x.shape[0])
        if out is None:
            out = torch.empty((M, self.N), dtype=torch.bfloat16, device=x.device)
        w12.w12_q8_gemm(x, self.blob, self.info, out, M, self.workspace(M), stream)
        return out


class Q8Group:
    """Q8 copies that multiply the same x, run as one launch (as W12Group)."""

    def __init__(self, mats):
        if not 1 <= len(mats) <= w12.MAX_GROUP or len({m.K for m in mats}) != 1:
            raise ValueError(f"1..{w12.MAX_GROUP} matrices with the same K")
        self.mats = list(mats)
        self.K = mats[0].K
        self.infos = [m.info for m in mats]
        self._ws = {}

    def workspace(self, M: int):
        import torch

        size = w12.w12_q8_gemm_group_workspace_size(self.infos, M)
        ws = self._ws.get(M)
        if ws is None or ws.numel() < size:
            ws = torch.zeros(max(size, 256), dtype=torch.uint8, device=self.mats[0].blob.device)
            self._ws[M] = ws
        return ws

    def gemm(self, x, outs=None, stream=None):
        import torch

        if x.dtype != torch.bfloat16 or x.dim() != 2 or x.shape[1] != self.K or not x.is_contiguous():
            raise ValueError("x must be a contiguous BF16 tensor of shape [M, K]")
        M = int(x.shape[0])
        if outs is None:
            outs = [torch.empty((M, m.N), dtype=torch.bfloat16, device=x.device) for m in self.mats]
        w12.w12_q8_gemm_group(x, [m.blob for m in self.mats], self.infos, outs, M, self.workspace(M), stream)
        return outs
