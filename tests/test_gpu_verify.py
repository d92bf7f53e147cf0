"""GPU tree acceptance and LM-head argmax against the oracle.

Accepted paths and bonus tokens must be bit-exact; an argmax that differs
from the oracle's is accepted only when the oracle's top-2 logit gap is below
1e-5 (reported as a tie)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import synth
from tests._gpu_util import device_weights, to_dev16

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


def check_paths(path_len, path_nodes, bonus, tok, parent, draft, offsets):
    pl, pn, bo = path_len.cpu().numpy(), path_nodes.cpu().numpy(), bonus.cpu().numpy()
    for r, (L, path, b) in enumerate(oracle.accept_batched(tok, parent, draft, offsets)):
        assert pl[r] == L, r
        assert bo[r] == b, r
        if L >= 0:
            o = offsets[r]
            assert pn[o:o + L + 1].tolist() == path.tolist(), r


def test_golden_trees(w12):
    from tests.test_oracle_pins import load_tree_fixture
    for c in load_tree_fixture():
        n = len(c["parent"])
        pl, pn, bo = w12.tree_verify_tokens(i32(c["tok"]), i32(c["parent"]), i32(c["draft"]))
        assert int(pl[0]) == c["L"], c["name"]
        assert int(bo[0]) == c["bonus"], c["name"]
        if c["L"] >= 0:
            assert pn[: c["L"] + 1].cpu().tolist() == c["path"], c["name"]


@pytest.mark.parametrize("n_req,nodes", [(1, 8), (1, 32), (24, 8), (7, 1), (5, 300)])
def test_random_batched_trees(w12, n_req, nodes):
    rng = np.random.default_rng(n_req * 1000 + nodes)
    parents, toks, drafts = [], [], []
    for r in range(n_req):
        p = synth.tree(2, r, nodes, nodes)
        t = rng.integers(0, 4, nodes)
        d = rng.integers(0, 4, nodes)
        plant = rng.random(nodes) < 0.5
        for i in range(1, nodes):
            if plant[i]:
                d[i] = t[p[i]]
        parents.append(p), toks.append(t), drafts.append(d)
    parent, tok, draft = (np.concatenate(a).astype(np.int32) for a in (parents, toks, drafts))
    offsets = np.arange(0, n_req * nodes + 1, nodes, dtype=np.int32)
    pl, pn, bo = w12.tree_verify_tokens(i32(tok), i32(parent), i32(draft), i32(offsets))
    check_paths(pl, pn, bo, tok, parent, draft, offsets)


def test_invalid_trees_flagged(w12):
    parent = np.array([-1, 0, -1, 1, 5, 0], np.int32)   # request 1 has parent 5 >= index
    offsets = np.array([0, 2, 6], np.int32)
    tok = np.zeros(6, np.int32)
    pl, pn, bo = w12.tree_verify_tokens(i32(tok), i32(parent), i32(tok), i32(offsets))
    assert pl.cpu().tolist() == [1, -1] and bo.cpu().tolist()[1] == -1


def test_tree_verify_from_logits(w12):
    rng = np.random.default_rng(4)
    M, V = 32, 1000
    logits = rng.standard_normal((M, V)).astype(np.float32)
    logits[3, 10] = logits[3, 20] = logits[3].max() + 1.0        # exact tie -> lower index
    tok = np.argmax(logits, axis=1).astype(np.int32)
    parent = synth.tree(2, 9, 0, M)
    draft = synth.drafts(3, 9, 0, M, V)
    for i in range(1, M):
        if i % 2:
            draft[i] = tok[parent[i]]
    pl, pn, bo = w12.tree_verify(torch.from_numpy(logits).cuda(), i32(parent), i32(draft))
    check_paths(pl, pn, bo, tok, parent, draft, np.array([0, M]))


def argmax_check(tok_gpu, y64):
    idx, gap = oracle.argmax(y64)
    ties = 0
    for m in range(len(idx)):
        if tok_gpu[m] != idx[m]:
            assert y64[m, idx[m]] - y64[m, tok_gpu[m]] < TIE, (m, tok_gpu[m], idx[m], gap[m])
            ties += 1
    return ties


@pytest.mark.parametrize("q8", [False, True])
def test_lmhead_tiny(w12, q8):
    """Tiny config: 1024 x 256 head, M = 8, logits from x . W."""
    Wh = synth.weights(1, 0, 9, 1024, 256)
    x = synth.activations(1, 0, 100, 8, 256)
    A = w12.encode(to_dev16(Wh))
    enc = oracle.encode(Wh)
    y64 = oracle.gemm(x, oracle.decode_q8(enc) if q8 else oracle.decode(enc), with_bound=False)
    tok = w12.w12_lmhead_argmax(to_dev16(x), A, q8=q8).cpu().numpy()
    argmax_check(tok, y64)
    # fused path: same tokens, and acceptance of an 8-node tree on them
    parent = synth.tree(2, 0, 0, 8)
    draft = synth.drafts(3, 0, 0, 8, 1024)
    draft[2] = tok[parent[2]]
    t2, pl, pn, bo = w12.w12_lmhead_verify(to_dev16(x), A, i32(parent), i32(draft), q8=q8)
    assert np.array_equal(t2.cpu().numpy(), tok)
    check_paths(pl, pn, bo, tok, parent, draft, np.array([0, 8]))


def test_lmhead_full_size_m32(w12):
    """151936 x 5120 head at M = 32: full fp64 oracle logits on the host."""
    V, K, M = 151936, 5120, 32
    Wd = device_weights(0, 0, 9, V, K)
    A = w12.encode(Wd)
    del Wd
    x = synth.activations(1, 0, 9, M, K)
    tok = w12.w12_lmhead_argmax(to_dev16(x), A).cpu().numpy()
    Wh = synth.weights(0, 0, 9, V, K)
    y64 = oracle.gemm(x, Wh, with_bound=False)
    ties = argmax_check(tok, y64)
    assert ties <= 1
