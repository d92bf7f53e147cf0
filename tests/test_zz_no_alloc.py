"""w12_gemm_noalloc: the GEMM for callers that cannot pass a workspace.

Such callers (an engine that has already reserved all device memory, a plugin
interface with no workspace argument, a loop that must not call cudaMalloc)
use the library's fixed device scratch instead.  These tests call it through
the C ABI and check it against w12_gemm (which takes a caller workspace) on
two calls in a row: both run the same kernel with the same partition and the
same slot order, so the results must be bit-identical (a scratch-layout fault
that changed the reduction order would show); the GEMM tolerance the other
tests use (1e-4 x sum_k |x_k * w_k|) is checked as well.  A shape too large
for the fixed scratch, and a call with a bad argument, are refused.  This file is collected last so that a run stopping at
the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import synth
from tests._gpu_util import device_weights, f32_of_bf16, to_np16

pytestmark = pytest.mark.gpu
REL = 1e-4


@pytest.fixture(scope="module")
def w12():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import lossless_bit_weights_gb300 as m
    m.lib()
    return m


def call_noalloc(w12, x, A, y):
    """Raw C-ABI call of w12_gemm_noalloc on the current stream."""
    rc = w12.lib().w12_gemm_noalloc(ctypes.c_void_p(x.data_ptr()), x.shape[0], A.desc(),
                                    ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, w12.lib().w12_last_error()


@pytest.mark.parametrize("N,K,M", [(5120, 5120, 16), (300, 1001, 5), (7168, 5120, 32)])
def test_noalloc_matches_workspace_gemm_twice(w12, N, K, M):
    W = device_weights(0, 7, N + K, N, K)
    A = w12.encode(W)
    x = torch.empty((M, K), dtype=torch.int16, device="cuda")
    synth.activations_dev(1, 7, N + K, x)
    ref32 = w12.w12_gemm(x, A).cpu().numpy()
    ref = ref32.astype(np.float64)
    # bound sum_k |x_k w_k| from the decoded weights (fp64 on the host)
    wd = np.abs(f32_of_bf16(to_np16(w12.w12_decode(A))).astype(np.float64))
    xd = np.abs(f32_of_bf16(to_np16(x)).astype(np.float64))
    B = xd @ wd.T
    prev = None
    for _ in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        call_noalloc(w12, x, A, y)
        got32 = y.cpu().numpy()
        assert np.array_equal(got32, ref32)
        if prev is not None:
            assert np.array_equal(got32, prev)
        prev = got32
        assert np.all(np.abs(got32.astype(np.float64) - ref) <= REL * B)


def test_noalloc_refuses_shapes_beyond_its_scratch(w12):
    """An LM-head-sized matrix at 32 rows needs more scratch than the fixed
    array holds; the call fails before any device work."""
    lib = w12.lib()
    assert lib.w12_gemm_noalloc_max_scratch() == 16 << 20
    fake = w12.w12_matrix(151936, 5120, 4096, 4096, 4096, 4096, 4096, 4)   # never dereferenced
    y = ctypes.c_void_p(4096)
    rc = lib.w12_gemm_noalloc(ctypes.c_void_p(4096), 32, ctypes.byref(fake), y, None)
    assert rc == 2 and b"fixed scratch" in lib.w12_last_error()


def test_noalloc_refused_call_leaves_the_scratch_alone(w12):
    """A call refused by an argument check (null x, a misaligned plane) returns before the
    scratch is cleared: a result still being produced in it stays intact."""
    N, K, M = 1024, 512, 8
    A = w12.encode(device_weights(0, 8, 1, N, K))
    x = torch.empty((M, K), dtype=torch.int16, device="cuda")
    synth.activations_dev(1, 8, 1, x)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    call_noalloc(w12, x, A, y)
    lib = w12.lib()
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.w12_gemm_noalloc(None, M, A.desc(), ctypes.c_void_p(y.data_ptr()), s) == 1
    bad = w12.w12_matrix(N, K, A.hi.data_ptr() + 8, A.lo.data_ptr(), A.base.data_ptr(),
                         A.esc_tile_ptr.data_ptr(), A.esc.data_ptr(), A.n_esc)
    assert lib.w12_gemm_noalloc(ctypes.c_void_p(x.data_ptr()), M, ctypes.byref(bad),
                                ctypes.c_void_p(y.data_ptr()), s) == 1
    assert b"aligned" in lib.w12_last_error()
    y2 = torch.empty_like(y)
    call_noalloc(w12, x, A, y2)
    assert torch.equal(y, y2)
