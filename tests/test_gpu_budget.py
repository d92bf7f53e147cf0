"""Node budget shared across requests on the GPU, bit-exact against the oracle, and the
selected trees through the LM head and acceptance."""
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


def forest(rng, n_req, max_nodes):
    parents, confs, offs = [], [], [0]
    for r in range(n_req):
        n = int(rng.integers(1, max_nodes + 1))
        p = np.array([-1] + [int(rng.integers(0, i)) for i in range(1, n)], np.int32)
        c = rng.uniform(0.05, 1.0, n).astype(np.float32)
        c[rng.random(n) < 0.15] = 1.0
        parents.append(p), confs.append(c), offs.append(offs[-1] + n)
    return np.concatenate(parents), np.concatenate(confs), np.array(offs, np.int32)


@pytest.mark.parametrize("per_request", [False, True])
def test_budget_select_matches_oracle(w12, per_request):
    rng = np.random.default_rng(41 + per_request)
    for t in range(120):
        n_req = int(rng.choice([1, 3, 24, 100]))
        parent, conf, off = forest(rng, n_req, int(rng.choice([1, 8, 32])))
        if t % 29 == 0 and parent.size > 3:
            parent[off[-2]] = 0            # a request without a root
        C = int(off[-1])
        budget = int(rng.integers(1, 12)) if per_request else int(rng.integers(1, C + 3))
        draft = rng.integers(0, 1000, C).astype(np.int32)
        po, do, so, oo, nk = w12.tree_budget_select(i32(parent), torch.from_numpy(conf).cuda(), i32(draft), i32(off),
                                                    budget, per_request)
        ref = oracle.budget_select(parent, conf, draft, off, budget, per_request)
        k = int(nk[0])
        if ref is None:
            assert k == -1, t
            continue
        assert k == len(ref[0]), t
        assert po[:k].cpu().tolist() == ref[0].tolist(), t
        assert do[:k].cpu().tolist() == ref[1].tolist(), t
        assert so[:k].cpu().tolist() == ref[2].tolist(), t
        assert oo.cpu().tolist() == ref[3].tolist(), t


def test_gather_rows(w12):
    rng = np.random.default_rng(3)
    for K in (64, 72):
        x = rng.integers(0, 65536, (40, K)).astype(np.uint16)
        src = np.array([3, 0, 39, -1, 40, 7], np.int32)
        out = to_np16(w12.gather_rows(to_dev16(x), i32(src)))
        want = np.where(((src >= 0) & (src < 40))[:, None], x[np.clip(src, 0, 39)], 0)
        assert np.array_equal(out, want)


def test_budget_then_verify_tiny_head(w12):
    """24 requests x 12 candidate nodes, shared budget of 96 and per-request budget of 4:
    selection, row gather, the 1024 x 256 head and batched acceptance, against the oracle
    (argmax near-ties skipped)."""
    V, K, n_req, nodes = 1024, 256, 24, 12
    Wh = synth.weights(1, 0, 9, V, K)
    A = w12.encode(to_dev16(Wh))
    We = oracle.decode(oracle.encode(Wh))
    rng = np.random.default_rng(96)
    parent = np.concatenate([synth.tree(2, 300 + r, nodes, nodes) for r in range(n_req)]).astype(np.int32)
    off = np.arange(0, n_req * nodes + 1, nodes, dtype=np.int32)
    C = int(off[-1])
    conf = rng.uniform(0.1, 0.95, C).astype(np.float32)
    x = synth.activations(1, 0, 400, C, K)
    t_all, gaps = oracle.argmax(oracle.gemm(x, We, with_bound=False))
    draft = rng.integers(0, V, C).astype(np.int32)
    for i in range(C):
        r = i // nodes
        if parent[i] >= 0 and rng.random() < conf[i]:
            draft[i] = t_all[off[r] + parent[i]]
    for budget, per_request in ((96, False), (4, True)):
        po, do, so, oo, nk = w12.tree_budget_select(i32(parent), torch.from_numpy(conf).cuda(), i32(draft), i32(off),
                                                    budget, per_request)
        k = int(nk[0])
        assert k == 96
        xs = w12.gather_rows(to_dev16(x), so, k)
        tok, pl, pn, bo = w12.w12_lmhead_verify(xs, A, po[:k].contiguous(), do[:k].contiguous(), req_offsets=oo)
        ref = oracle.budget_select(parent, conf, draft, off, budget, per_request)
        src = ref[2]
        if (gaps[src] < TIE).any():
            continue
        assert np.array_equal(tok.cpu().numpy(), t_all[src])
        res = oracle.accept_batched(t_all[src], ref[0], ref[1], ref[3])
        got_len = pl.cpu().numpy()
        for r, (L, path, b) in enumerate(res):
            assert got_len[r] == L and int(bo[r]) == b
