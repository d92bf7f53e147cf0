"""GPU W12 / Q8 GEMM against the fp64 oracle: |y - y64| <= 1e-4 * sum|x*w|, and
repeated calls bit-identical."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import synth
from tests._gpu_util import assert_gemm_close, device_weights, to_dev16, to_np16

pytestmark = pytest.mark.gpu

REL = 1e-4  # tolerance of the verify GEMM, in units of sum_k |x_k * w_k|


@pytest.fixture(scope="module")
def w12():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import lossless_bit_weights_gb300 as m
    m.lib()
    return m


def check(w12, W, x, q8=False, ws=None):
    A = w12.encode(to_dev16(W))
    enc = oracle.encode(W)
    Wq = oracle.decode_q8(enc) if q8 else oracle.decode(enc)
    y64, B = oracle.gemm(x, Wq)
    fn = w12.w12_gemm_q8 if q8 else w12.w12_gemm
    y = fn(to_dev16(x), A, ws=ws).cpu().numpy()
    return assert_gemm_close(y, y64, B, REL)


@pytest.mark.parametrize("M", [1, 8])
@pytest.mark.parametrize("q8", [False, True])
def test_tiny_config(w12, M, q8):
    W = synth.weights(0, 0, 0, 512, 256)
    x = synth.activations(1, 0, 100, 8, 256)[:M]
    check(w12, W, x, q8)


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 33, 65), (17, 100, 1000), (32, 64, 128), (33, 70, 190),
                                   (5, 7, 7), (16, 31, 63), (2, 257, 640), (40, 96, 320), (192, 64, 256),
                                   # 64..256 tokens: row-block pairs, odd row-block counts, stream-K splits
                                   (100, 640, 2048), (255, 384, 4160), (129, 1000, 700), (64, 1152, 5120),
                                   (70, 5248, 1024)])
@pytest.mark.parametrize("q8", [False, True])
def test_ragged_shapes(w12, M, N, K, q8):
    W = synth.weights(0, M, N * 7 + K, N, K)
    x = synth.activations(1, M, K, M, K)
    check(w12, W, x, q8)


@pytest.mark.parametrize("M,N,K,q8", [(16, 256, 17408, False), (16, 256, 17408, True), (32, 200, 12000, False),
                                      (192, 256, 17408, False)])
def test_many_parts_per_row_block(w12, M, N, K, q8):
    """Long rows over few row blocks: each row block is split over dozens of parts, so the
    last arrival adds more slots than a warp's share of shared memory holds (the register
    path) and most ranges start inside a row block (published early by their pipeline's
    publisher warp).  Repeats stay bit-identical."""
    W = synth.weights(3, M, N * 5 + K, N, K)
    x = synth.activations(2, M, K, M, K)
    ws = w12.Workspace()
    check(w12, W, x, q8, ws=ws)
    A = w12.encode(to_dev16(W))
    fn = w12.w12_gemm_q8 if q8 else w12.w12_gemm
    y0 = fn(to_dev16(x), A, ws=ws)
    y1 = fn(to_dev16(x), A, ws=ws)
    assert torch.equal(y0, y1)
    assert ws.status() == 0


@pytest.mark.parametrize("M,N,K,q8", [(65, 1100, 46789, False), (65, 1100, 46789, True), (150, 1300, 40000, False)])
def test_pairs_summed_after_the_launch(w12, M, N, K, q8):
    """64 to 192 tokens on a matrix with fewer row blocks than SMs and long rows: row-block
    pairs whose split rows are summed by a second kernel over every SM.  Odd row-block
    counts (the last pair has one row block), a ragged last row block, ragged K (x padded)
    and ragged tokens; every element against the oracle, and repeats bit-identical."""
    W = synth.weights(5, M, N * 3 + K, N, K)
    x = synth.activations(6, M, K, M, K)
    ws = w12.Workspace()
    check(w12, W, x, q8, ws=ws)
    A = w12.encode(to_dev16(W))
    fn = w12.w12_gemm_q8 if q8 else w12.w12_gemm
    y0 = fn(to_dev16(x), A, ws=ws)
    y1 = fn(to_dev16(x), A, ws=ws)
    assert torch.equal(y0, y1)
    assert ws.status() == 0


def test_exact_on_small_integers(w12):
    """Integer-valued weights and activations with small magnitudes: every
    partial sum is exact in fp32, so the GPU result equals the integer GEMM."""
    rng = np.random.default_rng(9)
    M, N, K = 16, 96, 512
    xi = rng.integers(-4, 5, (M, K)).astype(np.float32)
    wi = rng.integers(-4, 5, (N, K)).astype(np.float32)
    bf = lambda a: (a.view(np.uint32) >> 16).astype(np.uint16)
    A = w12.encode(to_dev16(bf(wi)))
    y = w12.w12_gemm(to_dev16(bf(xi)), A).cpu().numpy()
    assert np.array_equal(y, xi @ wi.T)


def test_deterministic_repeats(w12):
    W = device_weights(0, 0, 1, 5120, 5120)
    A = w12.encode(W)
    x = torch.empty((16, 5120), dtype=torch.int16, device="cuda")
    synth.activations_dev(1, 0, 1, x)
    ws = w12.Workspace()
    ref = w12.w12_gemm(x, A, ws=ws).clone()
    for _ in range(10):
        assert torch.equal(w12.w12_gemm(x, A, ws=ws), ref)
    refq = w12.w12_gemm_q8(x, A, ws=ws).clone()
    for _ in range(5):
        assert torch.equal(w12.w12_gemm_q8(x, A, ws=ws), refq)


@pytest.mark.parametrize("M", [32, 100, 192, 256])
def test_deterministic_repeats_wide(w12, M):
    """Back-to-back launches on a full-size gate/up matrix at 32, 100 and 192 tokens
    (row-block pairs) and 256 (one pipeline, shallow record rings): every
    launch gives the same bits (the stream-K sums run in a fixed order), and a sample of
    channels matches the oracle."""
    N, K = 34816, 5120
    W = device_weights(0, 0, 2, N, K)
    A = w12.encode(W)
    del W
    x_h = synth.activations(1, 0, 2, M, K)
    x = to_dev16(x_h)
    ws = w12.Workspace()
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ref = w12.w12_gemm(x, A, ws=ws).clone()
    for _ in range(40):
        w12.w12_gemm(x, A, y=y, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(y, ref)
    rows = np.sort(np.random.default_rng(M).choice(N, 16, replace=False))
    y64, B = oracle.gemm(x_h, synth.weight_rows(0, 0, 2, K, rows))
    assert_gemm_close(ref.cpu().numpy()[:, rows], y64, B, REL)


BLOCK = [(7168, 5120), (5120, 5120), (34816, 5120), (5120, 17408)]


def sampled_block_check(w12, layer, M, q8, n_rows=64, seed_rows=0):
    """Full-size block at M tokens in the bench's launch configuration; the
    oracle recomputes a random sample of output channels from host-generated rows."""
    rng = np.random.default_rng(seed_rows + layer)
    ws = w12.Workspace()
    worst = 0.0
    for tensor, (N, K) in enumerate(BLOCK):
        Wd = device_weights(0, layer, tensor, N, K)
        A = w12.encode(Wd)
        del Wd
        x_h = synth.activations(1, layer, tensor, M, K)
        y = (w12.w12_gemm_q8 if q8 else w12.w12_gemm)(to_dev16(x_h), A, ws=ws).cpu().numpy()
        rows = np.sort(rng.choice(N, n_rows, replace=False))
        Wr = synth.weight_rows(0, layer, tensor, K, rows)
        if q8:
            Wr = oracle.decode_q8(oracle.encode(Wr))
        y64, B = oracle.gemm(x_h, Wr)
        worst = max(worst, assert_gemm_close(y[:, rows], y64, B, REL))
        del A
        torch.cuda.empty_cache()
    return worst


def test_block_m16_sampled(w12):
    sampled_block_check(w12, layer=0, M=16, q8=False)


def test_block_m32_q8_sampled(w12):
    sampled_block_check(w12, layer=63, M=32, q8=True)


def test_block_m32_exact_sampled(w12):
    """The exact pass of the 64-layer stack at 32 tokens: all four full-size block
    matrices of one layer, in the launch configuration the stack uses."""
    sampled_block_check(w12, layer=5, M=32, q8=False)


def test_block_m192_sampled(w12):
    sampled_block_check(w12, layer=1, M=192, q8=False, n_rows=24)


def escape_dense_matrix(N, K, seed):
    """Weights of the usual recipe with escapes planted far above its rate: the first
    32x64 tile holds nothing but escapes (zeros of both signs, denormals, values 2^20
    above or 2^40 below the window), the next row tile's second chunk 8% escapes and
    the third row tile's third chunk 25%, so a row tile exceeds 32 escapes and a 128x64
    unit exceeds 128 (the escape list of a unit is then read partly from global memory).
    Every value stays finite."""
    W = synth.weights(0, 77, seed, N, K).copy()
    rng = np.random.default_rng(seed)

    def plant(rows, cols, frac):
        blk = W[rows, cols]
        pick = rng.random(blk.shape) < frac
        kind = rng.integers(0, 4, blk.shape)
        sign = (rng.integers(0, 2, blk.shape) << 15).astype(np.uint16)
        e = (blk >> 7) & 0xFF
        den = sign | rng.integers(1, 128, blk.shape).astype(np.uint16)
        up = np.where(e + 20 <= 254, (blk & 0x807F) | ((e + 20) << 7), blk).astype(np.uint16)
        dn = np.where(e >= 41, (blk & 0x807F) | ((e - 40) << 7), den).astype(np.uint16)
        new = np.choose(kind, [sign, den, up, dn]).astype(np.uint16)
        W[rows, cols] = np.where(pick, new, blk)

    plant(slice(0, 32), slice(0, 64), 1.0)
    plant(slice(32, 64), slice(64, 128), 0.08)
    plant(slice(64, 96), slice(128, 192), 0.25)
    return W


@pytest.mark.parametrize("M", [5, 16, 40, 192])
@pytest.mark.parametrize("q8", [False, True])
def test_escape_dense(w12, M, q8):
    """Escapes restored exactly, also where a tile or unit holds more than its stage keeps:
    the GEMM against the oracle, the codec bit-exact."""
    N, K = 300, 700
    W = escape_dense_matrix(N, K, 3)
    enc = oracle.encode(W)
    cols = enc.esc >> 16
    first_tile = sum(int((cols[enc.rowptr[r]:enc.rowptr[r + 1]] < 64).sum()) for r in range(32))
    assert first_tile == 2048          # the first tile is all escapes
    A = w12.encode(to_dev16(W))
    assert A.n_esc == enc.n_esc and enc.n_esc > 2048 + 200
    assert np.array_equal(to_np16(w12.w12_decode(A)), W)
    x = synth.activations(1, 77, M, M, K)
    Wq = oracle.decode_q8(enc) if q8 else oracle.decode(enc)
    y64, B = oracle.gemm(x, Wq)
    ws = w12.Workspace()
    y = (w12.w12_gemm_q8 if q8 else w12.w12_gemm)(to_dev16(x), A, ws=ws).cpu().numpy()
    assert_gemm_close(y, y64, B, REL)
    assert ws.status() == 0
