"""Certified INT8 LM-head argmax on the GPU against the oracle.

The SpecPilot summary page (onedev.kr/papers/1654), section "What's different",
keeps the H100 build's LM head in INT8 and filters argmax candidates with a
Cauchy-Schwarz error bound before computing them exactly.  The encoder must give
the oracle's codes and scales bit for bit (bound factors within 2 ulp: both sum
squares in fp64, in different orders), and the certified argmax must equal the
argmax of the exact fp64 logits (the plain argmax, which pins it), top-2 gaps
under 1e-5 counting as ties.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests._gpu_util import f32_of_bf16, to_dev16

pytestmark = pytest.mark.gpu
TIE = 1e-5
HEAD = (151936, 5120)


@pytest.fixture(scope="module")
def w12():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import lossless_bit_weights_gb300 as m
    m.lib()
    return m


def untile_codes(code_plane, V, K):
    """Canonical [V, K] codes from the hi-plane tile layout of include/w12.h."""
    KC = (K + 63) // 64
    v = np.arange(V)[:, None]
    k = np.arange(K)[None, :]
    rt, r, kc, kk = v // 32, v % 32, k // 64, k % 64
    tile = ((rt >> 2) * KC + kc) * 4 + (rt & 3)
    q, g, t, j = r >> 3, r & 7, kk >> 4, kk & 15
    u = j & 3
    pos = (j & ~3) | np.where(u == 1, 2, np.where(u == 2, 1, u))
    return code_plane[tile * 2048 + q * 512 + (4 * g + t) * 16 + pos]


def special_rows(W):
    W = W.copy()
    if W.shape[0] > 3:
        W[1] = 0                                              # all-zero channel
        W[2] = (np.arange(W.shape[1]) % 127 + 1).astype(np.uint16)   # denormals only
        W[3, :] = 0
        W[3, 0] = 0x3F80                                     # a single 1.0
    return W


@pytest.mark.parametrize("V,K,outliers", [(1, 1, True), (33, 70, True), (100, 300, False), (257, 640, True),
                                          (64, 5120, False), (130, 1000, True)])
def test_i8_encode_matches_oracle(w12, V, K, outliers):
    W = special_rows(synth.weights(2, V, K, V, K, outliers=outliers))
    H = w12.i8_encode(to_dev16(W))
    code, scale, cb = oracle.i8_quantize(W)
    got = untile_codes(H.code.cpu().numpy(), V, K)
    assert np.array_equal(got, code)
    assert np.array_equal(H.scale.cpu().numpy(), scale)
    cg = H.cbound.cpu().numpy()
    assert (np.abs(cg.astype(np.float64) - cb) <= 2 * np.spacing(cb)).all()
    # padding codes are zero
    plane = H.code.cpu().numpy()
    mask = np.ones(plane.size, bool)
    KC = (K + 63) // 64
    v = np.arange(V)[:, None]
    k = np.arange(K)[None, :]
    rt, r, kc, kk = v // 32, v % 32, k // 64, k % 64
    j = kk & 15
    u = j & 3
    pos = (j & ~3) | np.where(u == 1, 2, np.where(u == 2, 1, u))
    mask[((((rt >> 2) * KC + kc) * 4 + (rt & 3)) * 2048 + (r >> 3) * 512 + (4 * (r & 7) + (kk >> 4)) * 16 + pos).ravel()] = False
    assert not plane[mask].any()


def peaked_rows(seed, V, K, M, W_rows_fn, beta, rng):
    t = rng.integers(0, V, M)
    return synth.peaked_activations(seed, 0, 101, W_rows_fn(t), beta), t


def check_tokens(tok, x, W):
    y64 = oracle.gemm(x, W, with_bound=False)
    idx, gap = oracle.argmax(y64)
    ties = 0
    for m in range(len(idx)):
        if tok[m] != idx[m]:
            assert y64[m, idx[m]] - y64[m, tok[m]] < TIE, (m, tok[m], idx[m], gap[m])
            ties += 1
    return ties


@pytest.mark.parametrize("M", [1, 7, 16, 40])
@pytest.mark.parametrize("peaked,outliers", [(True, False), (False, False), (True, True)])
def test_cert_argmax_small(w12, M, peaked, outliers):
    V, K = 700, 320
    W = synth.weights(3, M, K, V, K, outliers=outliers)
    rng = np.random.default_rng(M * 10 + peaked)
    if peaked:
        x, _ = peaked_rows(4, V, K, M, lambda t: W[t], 6.0, rng)
    else:
        x = synth.activations(4, M, 102, M, K)
    Wd = to_dev16(W)
    H = w12.i8_encode(Wd)
    A = w12.encode(Wd)
    tok, ncand = w12.w12_cert_head_argmax(to_dev16(x), H, A)
    tok, ncand = tok.cpu().numpy(), ncand.cpu().numpy()
    assert check_tokens(tok, x, W) == 0
    assert (ncand >= 1).all() and (ncand <= V).all()
    # the oracle's certified argmax (fp64 approximate logits) agrees
    code, scale, cb = oracle.i8_quantize(W)
    idx_o, ncand_o = oracle.cert_argmax(x, W, code, scale, cb)
    assert np.array_equal(idx_o, tok)
    if peaked and not outliers:
        assert ncand.mean() < V / 10


def test_cert_argmax_repeatable_and_equals_w12_head(w12):
    V, K, M = 3000, 512, 16
    W = synth.weights(5, 0, 9, V, K, outliers=False)
    rng = np.random.default_rng(7)
    x, _ = peaked_rows(6, V, K, M, lambda t: W[t], 8.0, rng)
    Wd = to_dev16(W)
    H, A = w12.i8_encode(Wd), w12.encode(Wd)
    xd = to_dev16(x)
    ws = w12.Workspace()
    t0, n0 = w12.w12_cert_head_argmax(xd, H, A, ws=ws)
    for _ in range(5):
        t1, n1 = w12.w12_cert_head_argmax(xd, H, A, ws=ws)
        assert torch.equal(t0, t1) and torch.equal(n0, n1)
    assert torch.equal(t0, w12.w12_lmhead_argmax(xd, A, ws=ws))


def test_cert_argmax_full_head_m16(w12):
    """151936 x 5120 head (the head recipe, no x2^9 outliers), 16 rows pointing at
    random tokens: the certified argmax equals the exact-logit argmax of every row."""
    V, K = HEAD
    M = 16
    Wd = torch.empty((V, K), dtype=torch.int16, device="cuda")
    synth.weights_dev(0, 0, 9, Wd, outliers=False)
    H, A = w12.i8_encode(Wd), w12.encode(Wd)
    del Wd
    torch.cuda.empty_cache()
    rng = np.random.default_rng(16)
    x, t = peaked_rows(1, V, K, M, lambda t: synth.weight_rows(0, 0, 9, K, t, outliers=False), 8.0, rng)
    tok, ncand = w12.w12_cert_head_argmax(to_dev16(x), H, A)
    tok, ncand = tok.cpu().numpy(), ncand.cpu().numpy()
    Wh = synth.weights(0, 0, 9, V, K, outliers=False)
    assert check_tokens(tok, x, Wh) == 0
    assert ncand.max() < 1000
