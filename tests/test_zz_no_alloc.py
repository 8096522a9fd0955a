"""w12_gemm_noalloc: the GEMM for callers that cannot allocate device memory
(for example a serving engine whose allocator owns all free HBM, or a plug-in
that must not allocate behind its host framework).  Its scratch is a fixed
array in the library's static device memory; this checks, through the C ABI,
that two calls in a row give bit for bit the result of w12_gemm with a
caller workspace (the same plan and the same fixed split-K order, so a stale
partial sum or counter left in the shared array would show), that both meet
the GEMM tolerance against the fp64 oracle, and that a problem needing more
scratch than the fixed array is refused before anything runs.  Collected
last on purpose."""
import ctypes

import numpy as np
import pytest

from lossless_bit_weight_encode_gb300 import W12Weight, w12
from lossless_bit_weight_encode_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from gpu_util import ensure_built
    ensure_built()


def _noalloc_raw(x, mat, y, M):
    import torch
    lib = w12.lib()
    return lib.w12_gemm_noalloc(x.data_ptr(), mat.blob.data_ptr(), ctypes.byref(mat.info), y.data_ptr(), int(M),
                                torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("n,k,M", [(384, 2048, 1), (640, 3000, 2), (1000, 5120, 7), (6144, 5120, 16),
                                   (1024, 17408, 32)])
def test_noalloc_matches_workspace_gemm_twice(n, k, M):
    import torch
    import oracle
    from gpu_util import check_tolerance, dev_to_bits, to_dev_bf16
    w = wl.heavy_tail_weights(n, k, seed=n + M)
    xb = wl.activations(M, k, seed=k + M)
    x = to_dev_bf16(xb)
    mat = W12Weight(w)
    ref = dev_to_bits(mat.gemm(x))
    w12.w12_check_status()
    ref64 = oracle.gemm_f64(xb, w)
    check_tolerance(ref, ref64, f"w12_gemm {n}x{k} M={M}")
    for _ in range(2):  # two calls in a row share (and reuse) the one scratch array
        y = torch.full((M, n), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _noalloc_raw(x, mat, y, M) == 0, w12.w12_last_error()
        w12.w12_check_status()
        got = dev_to_bits(y)
        assert np.array_equal(got, ref), f"noalloc {n}x{k} M={M} differs from w12_gemm"
        check_tolerance(got, ref64, f"noalloc {n}x{k} M={M}")


def test_noalloc_rejects_oversized_problem():
    import torch
    from gpu_util import to_dev_bf16
    k = 262144
    mat = W12Weight(wl.gaussian_weights(128, k, seed=3))
    need = w12.w12_gemm_workspace_size(mat.info, 32)
    assert need > w12.NOALLOC_SCRATCH_BYTES
    x = torch.zeros((32, k), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((32, 128), dtype=torch.bfloat16, device="cuda")
    assert _noalloc_raw(x, mat, y, 32) == 3  # W12_ERR_BUFFER_TOO_SMALL, nothing launched
    assert "scratch" in w12.w12_last_error()
    # the same matrix at M = 1 fits and still agrees with w12_gemm
    x1 = to_dev_bf16(wl.activations(1, k, seed=4))
    y1 = torch.zeros((1, 128), dtype=torch.bfloat16, device="cuda")
    assert w12.w12_gemm_workspace_size(mat.info, 1) <= w12.NOALLOC_SCRATCH_BYTES
    assert _noalloc_raw(x1, mat, y1, 1) == 0, w12.w12_last_error()
    w12.w12_check_status()
    ref = mat.gemm(x1)
    w12.w12_check_status()
    assert np.array_equal(y1.view(torch.int16).cpu().numpy(), ref.view(torch.int16).cpu().numpy())
