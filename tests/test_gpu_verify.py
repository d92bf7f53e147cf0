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


@pytest.mark.parametrize("q8", [False, True])
def test_lmhead_short_long_rows(w12, q8):
    """A 1100 x 46789 head at 65 tokens: fewer row blocks than SMs, long rows and an odd
    row-block count, so the launch takes row-block pairs with the fused argmax (its split
    rows reduced in the kernel); tokens against the fp64 logits."""
    V, K, M = 1100, 46789, 65
    Wh = synth.weights(2, 0, 19, V, K)
    x = synth.activations(2, 0, 119, M, K)
    A = w12.encode(to_dev16(Wh))
    enc = oracle.encode(Wh)
    y64 = oracle.gemm(x, oracle.decode_q8(enc) if q8 else oracle.decode(enc), with_bound=False)
    tok = w12.w12_lmhead_argmax(to_dev16(x), A, q8=q8).cpu().numpy()
    argmax_check(tok, y64)


HEAD = (151936, 5120)   # the LM head of the 27B-class configs: vocab x hidden


@pytest.fixture(scope="module")
def head(w12):
    """The 151936 x 5120 head, W12-encoded on the device (seed 0, tensor 9)."""
    V, K = HEAD
    Wd = device_weights(0, 0, 9, V, K)
    A = w12.encode(Wd)
    del Wd
    torch.cuda.empty_cache()
    return A


@pytest.fixture(scope="module")
def head_host():
    """The same head's bf16 bits generated on the host, and its oracle encoding."""
    V, K = HEAD
    Wh = synth.weights(0, 0, 9, V, K)
    return Wh, oracle.encode(Wh)


def planted_tree(seed_layer, n, V, tok, rng, p_plant=0.5):
    """A random tree (parent of node i uniform over 0..i-1) with uniform drafts over
    the vocab, where each node's draft is set to its parent's target token with
    probability p_plant, so that acceptance is exercised."""
    parent = synth.tree(2, seed_layer, n, n)
    draft = synth.drafts(3, seed_layer, n, n, V)
    for i in range(1, n):
        if rng.random() < p_plant:
            draft[i] = tok[parent[i]]
    return parent, draft


def test_lmhead_full_size_m32(w12, head, head_host):
    """151936 x 5120 head at M = 32: fp64 oracle logits on the host for every row, then
    greedy acceptance on a 32-node tree from the fused verify call."""
    V, K = HEAD
    M = 32
    Wh, _ = head_host
    x = synth.activations(1, 0, 9, M, K)
    tok = w12.w12_lmhead_argmax(to_dev16(x), head).cpu().numpy()
    y64 = oracle.gemm(x, Wh, with_bound=False)
    ties = argmax_check(tok, y64)
    assert ties <= 1
    rng = np.random.default_rng(32)
    for plant in (0.0, 0.5, 1.0):   # the literal uniform drafts, then planted ones
        parent, draft = planted_tree(32, M, V, tok, rng, plant)
        t2, pl, pn, bo = w12.w12_lmhead_verify(to_dev16(x), head, i32(parent), i32(draft))
        assert np.array_equal(t2.cpu().numpy(), tok)
        check_paths(pl, pn, bo, tok, parent, draft, np.array([0, M]))


def test_lmhead_q8_full_size_m32_and_agreement(w12, head, head_host):
    """The 8-bit-view head at M = 32 against the oracle's Q8 logits, and the Q-vs-exact
    top-1 agreement: the rate the GPU reports equals the oracle's on the same rows
    (rows whose oracle top-2 gap is below the tie bound are left out of the comparison)."""
    V, K = HEAD
    M = 32
    Wh, enc = head_host
    x = synth.activations(1, 0, 9, M, K)
    xd = to_dev16(x)
    tq = w12.w12_lmhead_argmax(xd, head, q8=True).cpu().numpy()
    te = w12.w12_lmhead_argmax(xd, head).cpu().numpy()
    yq = oracle.gemm(x, oracle.decode_q8(enc), with_bound=False)
    ye = oracle.gemm(x, Wh, with_bound=False)
    assert argmax_check(tq, yq) <= 1
    iq, gq = oracle.argmax(yq)
    ie, ge = oracle.argmax(ye)
    clear = (gq >= TIE) & (ge >= TIE)
    assert clear.sum() >= M - 2
    assert np.array_equal((tq == te)[clear], (iq == ie)[clear])


def test_lmhead_m192_24_trees(w12, head, head_host):
    """24 requests x 8 tree nodes = 192 rows through the head in one call with per-request
    acceptance: the argmax of 16 sampled rows against fp64 oracle logits, and every
    request's path and bonus bit-exact against the oracle on the GPU's tokens."""
    V, K = HEAD
    M, n_req, nodes = 192, 24, 8
    Wh, _ = head_host
    x = synth.activations(1, 0, 10, M, K)
    tok = w12.w12_lmhead_argmax(to_dev16(x), head).cpu().numpy()
    rows = np.sort(np.random.default_rng(192).choice(M, 16, replace=False))
    y64 = oracle.gemm(x[rows], Wh, with_bound=False)
    assert argmax_check(tok[rows], y64) <= 1
    rng = np.random.default_rng(24)
    parents, drafts = [], []
    for r in range(n_req):
        p, d = planted_tree(100 + r, nodes, V, tok[r * nodes:(r + 1) * nodes], rng)
        parents.append(p), drafts.append(d)
    parent = np.concatenate(parents).astype(np.int32)
    draft = np.concatenate(drafts).astype(np.int32)
    offsets = np.arange(0, M + 1, nodes, dtype=np.int32)
    t2, pl, pn, bo = w12.w12_lmhead_verify(to_dev16(x), head, i32(parent), i32(draft), req_offsets=i32(offsets))
    assert np.array_equal(t2.cpu().numpy(), tok)
    check_paths(pl, pn, bo, tok, parent, draft, offsets)
    assert (pl.cpu().numpy() > 0).sum() >= 1   # the planted drafts accept somewhere


def test_tlv_step_full_head(w12, head, head_host):
    """The two-level verification step on the 151936 x 5120 head: a 32-node Q tree through
    the 8-bit view, splice into a 32-node exact tree (subtree drafted again, planted to the
    Q tokens half the time), exact pass; every argmax against fp64 oracle logits and the
    final path bit-exact on the GPU's tokens."""
    V, K = HEAD
    n = 32
    Wh, enc = head_host
    rng = np.random.default_rng(33)
    xq = synth.activations(1, 0, 12, n, K)
    xs = synth.activations(1, 0, 13, n - 1, K)
    tq = w12.w12_lmhead_argmax(to_dev16(xq), head, q8=True).cpu().numpy()
    parent, draft = planted_tree(33, n, V, tq, rng, 0.7)
    sp = np.array([-1 if j == 0 or rng.random() < 0.3 else int(rng.integers(0, j)) for j in range(n - 2)], np.int32)
    sd = synth.drafts(3, 1, 33, n - 2, V)
    t_q, pl, pn, bo = w12.w12_lmhead_verify(to_dev16(xq), head, i32(parent), i32(draft), q8=True)
    assert np.array_equal(t_q.cpu().numpy(), tq)
    assert argmax_check(tq, oracle.gemm(xq, oracle.decode_q8(enc), with_bound=False)) <= 1
    check_paths(pl, pn, bo, tq, parent, draft, np.array([0, n]))
    par, dr, src, x = w12.tlv_splice(pl, pn, bo, i32(draft), to_dev16(xq), i32(sp), i32(sd), to_dev16(xs), n)
    L, path, bonus = oracle.accept(tq, parent, draft)
    ref = oracle.tlv_splice(L, path, bonus, draft, sp, sd, n)
    assert ref is not None and np.array_equal(par.cpu().numpy(), ref[0]) and np.array_equal(dr.cpu().numpy(), ref[1])
    te, pl2, pn2, bo2 = w12.w12_lmhead_verify(x, head, par, dr)
    xe = np.where(ref[2][:, None] >= 0, xq[np.maximum(ref[2], 0)], xs[np.clip(-1 - ref[2], 0, n - 2)])
    te = te.cpu().numpy()
    assert argmax_check(te, oracle.gemm(xe, Wh, with_bound=False)) <= 1
    check_paths(pl2, pn2, bo2, te, ref[0], ref[1], np.array([0, n]))
    assert int(pl2[0]) >= 0
