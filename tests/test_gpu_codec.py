"""GPU encoder / decoder / canonical export, bit-exact against the oracle."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import synth
from tests._gpu_util import assert_canonical_equal, device_weights, to_dev16, to_np16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w12():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import lossless_bit_weights_gb300 as m
    m.lib()
    return m


def roundtrip(w12, W: np.ndarray):
    A = w12.encode(to_dev16(W))
    enc = oracle.encode(W)
    assert_canonical_equal(A, enc)
    assert np.array_equal(to_np16(w12.w12_decode(A)), W)
    assert np.array_equal(to_np16(w12.w12_decode_q8(A)), oracle.decode_q8(enc))
    return A, enc


def test_tiny_config_matrix(w12):
    """512 x 256 layer and its 1024 x 256 head (seeds 0 and 1)."""
    roundtrip(w12, synth.weights(0, 0, 0, 512, 256))
    roundtrip(w12, synth.weights(1, 0, 9, 1024, 256))


@pytest.mark.parametrize("target_base", [1, 60, 112, 127, 239])
def test_every_bf16_pattern(w12, target_base):
    filler = []
    for E in range(target_base, target_base + 16):
        for i in range(600):
            filler.append(((i & 1) << 15) | (E << 7) | (i % 128))
    filler = np.array(filler, np.uint16)
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(16, 4096)
    W = np.concatenate([pats, np.broadcast_to(filler, (16, filler.size))], axis=1)
    A, enc = roundtrip(w12, W)
    assert np.all(enc.base == target_base)


@pytest.mark.parametrize("N,K", [(1, 1), (1, 7), (31, 63), (33, 65), (100, 130), (7, 1000), (64, 64), (65, 129),
                                 (3, 65535)])
def test_ragged_shapes(w12, N, K):
    roundtrip(w12, synth.weights(0, N, K, N, K))


def test_golden_rows(w12):
    from tests.test_oracle_pins import load_record_fixture
    rows, q8 = load_record_fixture()
    W = np.array([rows[r]["w"] for r in sorted(rows)], np.uint16)
    A, enc = roundtrip(w12, W)
    assert enc.base.tolist() == [rows[r]["base"] for r in sorted(rows)]


def test_device_generator_matches_host(w12):
    """The device generator writes the same bits as the host one (so full-size
    oracle checks may regenerate sampled rows on the host)."""
    W = device_weights(0, 5, 2, 96, 5120)
    host = synth.weights(0, 5, 2, 96, 5120)
    assert np.array_equal(to_np16(W), host)
    x = torch.empty((16, 5120), dtype=torch.int16, device="cuda")
    synth.activations_dev(1, 5, 2, x)
    assert np.array_equal(to_np16(x), synth.activations(1, 5, 2, 16, 5120))


def test_full_size_block_roundtrip(w12):
    """The 27B-class block matrices at full size: lossless decode on the GPU and
    canonical equality with the oracle on sampled channels."""
    rng = np.random.default_rng(0)
    for tensor, (N, K) in enumerate([(7168, 5120), (5120, 5120), (34816, 5120), (5120, 17408)]):
        Wd = device_weights(0, 0, tensor, N, K)
        A = w12.encode(Wd)
        dec = w12.w12_decode(A)
        assert torch.equal(dec.view(torch.int16), Wd), tensor
        rows = np.sort(rng.choice(N, 48, replace=False))
        host = synth.weight_rows(0, 0, tensor, K, rows)
        assert np.array_equal(to_np16(Wd[torch.from_numpy(rows).cuda()]), host)
        enc = oracle.encode(host)
        c = w12.w12_export_canonical(A)
        idx = torch.from_numpy(rows).cuda()
        assert np.array_equal(c["hi"][idx].cpu().numpy(), enc.hi)
        assert np.array_equal(c["lo"][idx].cpu().numpy(), enc.lo)
        assert np.array_equal(c["base"][idx].cpu().numpy(), enc.base)
        rp = c["rowptr"].cpu().numpy().view(np.uint32)
        esc = c["esc"].cpu().numpy().view(np.uint32)
        for i, r in enumerate(rows):
            assert np.array_equal(esc[rp[r]:rp[r + 1]], enc.esc[enc.rowptr[i]:enc.rowptr[i + 1]])
        del Wd, A, dec, c
        torch.cuda.empty_cache()


def test_save_and_load_round_trip(w12, tmp_path):
    """An encoded matrix written by w12_save and read back by w12_load has the same
    planes, bases, escape index and escapes, and gives the same GEMM bit for bit; a
    truncated file is refused."""
    import ctypes
    W = synth.weights(4, 0, 3, 700, 1000)
    A = w12.encode(to_dev16(W))
    path = tmp_path / "m.w12"
    w12.w12_save(A, str(path))
    B = w12.w12_load(str(path))
    assert (B.N, B.K, B.n_esc) == (A.N, A.K, A.n_esc)
    for name in ("hi", "lo", "base", "esc_tile_ptr"):
        assert torch.equal(getattr(A, name), getattr(B, name)), name
    assert torch.equal(A.esc[:A.n_esc], B.esc[:B.n_esc])
    x = to_dev16(synth.activations(5, 0, 7, 16, 1000))
    assert torch.equal(w12.w12_gemm(x, A), w12.w12_gemm(x, B))
    data = path.read_bytes()
    cut = tmp_path / "cut.w12"
    cut.write_bytes(data[:-5])
    assert w12.lib().w12_load(str(cut).encode(), B.desc(), None) == 7
