"""Device-side error reporting of the verify GEMM and the index check.

- A wait that runs out: with the GEMM kernels' wait bound lowered far below a unit's
  latency (w12_set_wait_limit), every CTA gives up early, leaves nothing in flight and
  frees its tensor memory; w12_workspace_status then reports W12_ERR_TIMEOUT and clears
  the workspace, and the next call on the same workspace gives the full result, in every
  launch mode (two pipelines with their own ranges at 16 tokens, one pipeline at 192 tokens
  on a short matrix, row-block pairs at 64 and 192 tokens on tall ones, pairs summed after
  the launch at 100 tokens on long rows).  No GPU fault is
  involved: the kernels return normally.
- A damaged escape index: w12_validate reports W12_ERR_BOUNDS for index arrays corrupted
  on the host (copies of a valid matrix's); such a matrix is never given to a GEMM.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import synth
from tests._gpu_util import assert_gemm_close, device_weights, to_dev16

pytestmark = pytest.mark.gpu

W12_OK, W12_ERR_BOUNDS, W12_ERR_TIMEOUT = 0, 5, 6


@pytest.fixture(scope="module")
def w12():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import lossless_bit_weights_gb300 as m
    m.lib()
    return m


@pytest.mark.parametrize("M,N,K", [(16, 5120, 5120), (192, 2048, 5120), (64, 20480, 1024), (192, 20480, 1024),
                                   (100, 5120, 17408)])
def test_wait_timeout_is_reported_and_the_workspace_recovers(w12, M, N, K):
    layer = 11
    Wd = device_weights(0, layer, M, N, K)
    A = w12.encode(Wd)
    del Wd
    x_h = synth.activations(1, layer, M, M, K)
    x = to_dev16(x_h)
    ws = w12.Workspace()
    ref = w12.w12_gemm(x, A, ws=ws).clone()
    assert ws.status() == W12_OK
    w12.w12_set_wait_limit(64)
    try:
        y = torch.full_like(ref, float("nan"))
        w12.w12_gemm(x, A, y=y, ws=ws)
        torch.cuda.synchronize()
    finally:
        w12.w12_set_wait_limit(0)
    assert ws.status() == W12_ERR_TIMEOUT
    assert ws.status() == W12_OK                    # the query cleared the word
    again = w12.w12_gemm(x, A, ws=ws)
    assert ws.status() == W12_OK
    assert torch.equal(again, ref)
    rows = np.sort(np.random.default_rng(M).choice(N, 16, replace=False))
    y64, B = oracle.gemm(x_h, synth.weight_rows(0, layer, M, K, rows))
    assert_gemm_close(again.cpu().numpy()[:, rows], y64, B, 1e-4)


def _copy(w12, A, tp=None, esc=None, base=None):
    """A descriptor with A's planes and (possibly replaced) index arrays."""
    return w12.W12Matrix(A.N, A.K, A.hi, A.lo, A.base if base is None else base,
                         A.esc_tile_ptr if tp is None else tp, A.esc if esc is None else esc, A.n_esc)


def test_validate_accepts_encoded_matrices(w12):
    for N, K, seed in [(300, 700, 1), (512, 256, 2), (7168, 5120, 3)]:
        A = w12.encode(device_weights(0, 21, seed, N, K))
        assert int(w12.w12_validate(A).item()) == W12_OK


def test_validate_reports_damaged_indices(w12):
    N, K = 300, 700
    A = w12.encode(device_weights(0, 21, 9, N, K))
    tp = A.esc_tile_ptr.cpu().numpy().view(np.uint32).copy()
    esc = A.esc.cpu().numpy().view(np.uint32).copy()
    assert A.n_esc > 40 and tp[-1] == A.n_esc
    busy = int(np.argmax(np.diff(tp.astype(np.int64))))        # a tile with escapes
    e = int(tp[busy])

    def dev32(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).cuda()

    cases = {}
    t = tp.copy(); t[busy], t[busy + 1] = t[busy + 1], t[busy]
    cases["offsets fall"] = dict(tp=t)
    t = tp.copy(); t[-1] = A.n_esc + 4
    cases["last offset past the list"] = dict(tp=t)
    t = tp.copy(); t[0] = 1
    cases["first offset not zero"] = dict(tp=t)
    t = tp.copy(); t[busy + 1] = 0xFFFFFFF0
    cases["offset far past the list"] = dict(tp=t)
    x = esc.copy(); x[e] = (x[e] & 0xFFFF) | (4096 << 16)
    cases["slot outside the tile"] = dict(esc=x)
    x = esc.copy(); x[e] = x[e] | (1 << 16)
    cases["odd slot"] = dict(esc=x)
    if tp[busy + 1] - tp[busy] >= 2:
        x = esc.copy(); x[e], x[e + 1] = x[e + 1], x[e]
        cases["entries out of order"] = dict(esc=x)
    b = A.base.cpu().numpy().copy(); b[7] = 0
    cases["window base 0"] = dict(base=b)
    b = A.base.cpu().numpy().copy(); b[8] = 240
    cases["window base 240"] = dict(base=b)
    for name, kw in cases.items():
        args = {}
        if "tp" in kw:
            args["tp"] = dev32(kw["tp"])
        if "esc" in kw:
            args["esc"] = dev32(kw["esc"])
        if "base" in kw:
            args["base"] = torch.from_numpy(kw["base"]).cuda()
        st = int(w12.w12_validate(_copy(w12, A, **args)).item())
        assert st == W12_ERR_BOUNDS, name
    assert int(w12.w12_validate(A).item()) == W12_OK


def test_validate_reports_an_escape_past_the_matrix(w12):
    """A ragged matrix (N = 40, K = 70): an entry moved to channel 63 of the first row
    tile pair, or to column 10 of the last chunk (column 74 >= K), is out of range."""
    N, K = 40, 70
    W = synth.weights(0, 22, 1, N, K).copy()
    W[33, 66] = 0                                   # an escape in row tile 1, chunk 1
    A = w12.encode(to_dev16(W))
    tp = A.esc_tile_ptr.cpu().numpy().view(np.uint32)
    esc = A.esc.cpu().numpy().view(np.uint32).copy()
    KC = 2
    tile = (0 * KC + 1) * 4 + 1                     # row tile 1, chunk 1
    assert tp[tile + 1] > tp[tile]
    e = int(tp[tile])
    dev32 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).cuda()

    def slot(rr, kk):
        return rr * 128 + (((kk >> 3) ^ (rr & 7)) & 7) * 16 + (kk & 7) * 2

    bad_row = esc.copy(); bad_row[e] = (bad_row[e] & 0xFFFF) | (slot(31, 2) << 16)    # channel 63 >= N
    bad_col = esc.copy(); bad_col[e] = (bad_col[e] & 0xFFFF) | (slot(1, 10) << 16)    # column 74 >= K
    for x in (bad_row, bad_col):
        assert int(w12.w12_validate(_copy(w12, A, esc=dev32(x))).item()) == W12_ERR_BOUNDS
    assert int(w12.w12_validate(A).item()) == W12_OK
