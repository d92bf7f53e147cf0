"""Two-level verification on the GPU against the oracle.

The splice (the Q pass's accepted path + bonus node + a subtree drafted again, renumbered
into the exact pass's tree) must match the oracle bit for bit; the full TLV step on the
tiny head (Q8 head argmax -> acceptance -> splice -> exact head argmax -> acceptance) must
give the oracle's path and bonus whenever no argmax on the way is a near-tie (oracle top-2
gap below 1e-5, reported as a tie as for the LM head)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import synth
from tests._gpu_util import to_dev16, to_np16

pytestmark = pytest.mark.gpu
TIE = 1e-5


@pytest.fixture(scope="module")
def w12():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import lossless_bit_weights_gb300 as m
    m.lib()
    return m


def i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()


def random_q_tree(rng, n_q, V, plant=0.6):
    parent = synth.tree(2, 70, n_q, n_q)
    tok = rng.integers(0, V, n_q).astype(np.int32)
    draft = rng.integers(0, V, n_q).astype(np.int32)
    for i in range(1, n_q):
        if rng.random() < plant:
            draft[i] = tok[parent[i]]
    return parent, tok, draft


def subtree(rng, n, V):
    sp = np.array([-1 if j == 0 or rng.random() < 0.3 else int(rng.integers(0, j)) for j in range(n - 2)], np.int32)
    sd = rng.integers(0, V, n - 2).astype(np.int32)
    return sp, sd


def test_splice_matches_oracle(w12):
    rng = np.random.default_rng(5)
    K = 72                      # not a multiple of 8 either way: both copy paths below
    for t in range(300):
        n_q = int(rng.integers(1, 40))
        n = int(rng.choice([2, 3, 8, 32, 33]))
        V = int(rng.integers(2, 5))
        parent, tok, draft = random_q_tree(rng, n_q, V)
        if t % 37 == 0:
            parent[0] = 0       # an invalid Q tree
        sp, sd = subtree(rng, n, V)
        if t % 41 == 0 and n > 4:
            sp[3] = 3           # an invalid subtree
        Kt = K if t % 2 else 64
        xq = rng.integers(0, 65536, (n_q, Kt)).astype(np.uint16)
        xs = rng.integers(0, 65536, (n - 1, Kt)).astype(np.uint16)
        pl, pn, bo = w12.tree_verify_tokens(i32(tok), i32(parent), i32(draft))
        par, dr, src, x = w12.tlv_splice(pl, pn, bo, i32(draft), to_dev16(xq), i32(sp), i32(sd), to_dev16(xs), n)
        L, path, bonus = oracle.accept(tok, parent, draft)
        ref = oracle.tlv_splice(L, path, bonus, draft, sp, sd, n)
        par, dr, src, x = par.cpu().numpy(), dr.cpu().numpy(), src.cpu().numpy(), to_np16(x)
        if ref is None:
            assert (par == -2).all() and (dr == -1).all() and (x == 0).all(), t
            continue
        assert np.array_equal(par, ref[0]) and np.array_equal(dr, ref[1]) and np.array_equal(src, ref[2]), t
        rows = np.where(ref[2][:, None] >= 0, xq[np.maximum(ref[2], 0)], xs[np.clip(-1 - ref[2], 0, n - 2)])
        assert np.array_equal(x, rows), t


def test_tlv_step_tiny_head(w12):
    """Config 0's 1024 x 256 head: a 16-node Q tree through the 8-bit view, splice into a
    32-node tree with a subtree drafted again, exact pass, acceptance."""
    V, K, n_q, n = 1024, 256, 16, 32
    Wh = synth.weights(1, 0, 9, V, K)
    A = w12.encode(to_dev16(Wh))
    enc = oracle.encode(Wh)
    Wq, We = oracle.decode_q8(enc), oracle.decode(enc)
    rng = np.random.default_rng(16)
    done = 0
    for trial in range(6):
        xq = synth.activations(1, trial, 200, n_q, K)
        xs = synth.activations(1, trial, 201, n - 1, K)
        yq = oracle.gemm(xq, Wq, with_bound=False)
        tq_ref, gq = oracle.argmax(yq)
        parent = synth.tree(2, 80 + trial, n_q, n_q)
        draft = synth.drafts(3, 80 + trial, n_q, n_q, V)
        for i in range(1, n_q):
            if rng.random() < 0.7:
                draft[i] = tq_ref[parent[i]]
        sp, sd = subtree(rng, n, V)
        # Q pass on the GPU (8-bit view head + acceptance), then the splice
        tq, pl, pn, bo = w12.w12_lmhead_verify(to_dev16(xq), A, i32(parent), i32(draft), q8=True)
        par, dr, src, x = w12.tlv_splice(pl, pn, bo, i32(draft), to_dev16(xq), i32(sp), i32(sd), to_dev16(xs), n)
        # exact pass on the spliced tree
        te, pl2, pn2, bo2 = w12.w12_lmhead_verify(x, A, par, dr, q8=False)
        if (gq < TIE).any():
            continue            # a near-tie in the Q pass: the GPU may pick the other token
        assert np.array_equal(tq.cpu().numpy(), tq_ref)
        L, path, bonus = oracle.accept(tq_ref, parent, draft)
        ref = oracle.tlv_splice(L, path, bonus, draft, sp, sd, n)
        assert ref is not None
        assert np.array_equal(par.cpu().numpy(), ref[0]) and np.array_equal(dr.cpu().numpy(), ref[1])
        xe = np.where(ref[2][:, None] >= 0, xq[np.maximum(ref[2], 0)], xs[np.clip(-1 - ref[2], 0, n - 2)])
        assert np.array_equal(to_np16(x), xe)
        ye = oracle.gemm(xe, We, with_bound=False)
        te_ref, ge = oracle.argmax(ye)
        if (ge < TIE).any():
            continue
        assert np.array_equal(te.cpu().numpy(), te_ref)
        L2, path2, bonus2 = oracle.accept(te_ref, ref[0], ref[1])
        assert int(pl2[0]) == L2 and int(bo2[0]) == bonus2
        assert pn2[:L2 + 1].cpu().tolist() == path2.tolist()
        assert L2 >= 0
        done += 1
    assert done >= 4
