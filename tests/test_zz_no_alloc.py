"""w12_gemm_noalloc: the GEMM for callers that cannot pass a workspace.

Such callers (an engine that has already reserved all device memory, a plugin
interface with no workspace argument, a loop that must not call cudaMalloc)
use the library's fixed device scratch instead.  These tests call it through
the C ABI and check it against w12_gemm (which takes a caller workspace) on
two calls in a row, within the GEMM tolerance the other tests use
(1e-4 x sum_k |x_k * w_k|), and check that a shape too large for the fixed
scratch is refused.  This file is collected last so that a run stopping at
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
    ref = w12.w12_gemm(x, A).cpu().numpy().astype(np.float64)
    # bound sum_k |x_k w_k| from the decoded weights (fp64 on the host)
    wd = np.abs(f32_of_bf16(to_np16(w12.w12_decode(A))).astype(np.float64))
    xd = np.abs(f32_of_bf16(to_np16(x)).astype(np.float64))
    B = xd @ wd.T
    for _ in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        call_noalloc(w12, x, A, y)
        got = y.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - ref) <= REL * B)


def test_noalloc_refuses_shapes_beyond_its_scratch(w12):
    """An LM-head-sized matrix at 32 rows needs more scratch than the fixed
    array holds; the call fails before any device work."""
    lib = w12.lib()
    assert lib.w12_gemm_noalloc_max_scratch() == 16 << 20
    fake = w12.w12_matrix(151936, 5120, 4096, 4096, 4096, 4096, 4096, 4)   # never dereferenced
    y = ctypes.c_void_p(4096)
    rc = lib.w12_gemm_noalloc(ctypes.c_void_p(4096), 32, ctypes.byref(fake), y, None)
    assert rc == 2 and b"fixed scratch" in lib.w12_last_error()
