"""Pins of the CPU oracle to facts fixed by the pages and by mathematics.

The W12 facts come from the SpecPilot summary page (onedev.kr/papers/1654),
section "What's different": lossless restoration of every value (zeros and
denormals included), the fullest 16-binade window per channel, 12 bits per
weight plus the escape overhead, the 8-bit front view used by the Q pass, and
greedy acceptance with a bonus token.  Each test below checks the oracle
against something other than its own formula: exhaustive round trips, brute
force, hand-worked fixtures, closed forms and library routines.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def f32_of_bf16(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_of_f32(f):
    """Round-to-nearest-even float32 -> bf16 bits (finite inputs)."""
    u = np.asarray(f, np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def exponent(bits):
    return (np.asarray(bits, np.uint16) >> 7) & 0xFF


# ----------------------------------------------------------------------------- round trip

@pytest.mark.parametrize("target_base", [1, 2, 60, 100, 112, 120, 127, 200, 239])
def test_roundtrip_every_bf16_pattern(target_base):
    """decode(encode(w)) == w bit for bit for all 65,536 bf16 patterns (±0,
    denormals, Inf and NaN payloads included), each row forced to a window
    base by a dominant block of filler values inside [base, base+15]."""
    filler = []
    for E in range(target_base, target_base + 16):
        for i in range(600):
            filler.append(((i & 1) << 15) | (E << 7) | (i % 128))
    filler = np.array(filler, np.uint16)
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(16, 4096)
    W = np.concatenate([pats, np.broadcast_to(filler, (16, filler.size))], axis=1)
    enc = oracle.encode(W)
    assert np.all(enc.base == target_base)
    dec = oracle.decode(enc)
    assert np.array_equal(dec, W)
    # every pattern outside the window (or E in {0, 255}) is an escape, and only those
    E = exponent(W)
    outside = (E == 0) | (E == 255) | (E < target_base) | (E > target_base + 15)
    assert enc.n_esc == int(outside.sum())
    cols = enc.esc >> 16
    raws = (enc.esc & 0xFFFF).astype(np.uint16)
    rows = np.repeat(np.arange(16), np.diff(enc.rowptr.astype(np.int64)))
    assert np.array_equal(W[rows, cols], raws)
    assert np.all(outside[rows, cols])


def test_roundtrip_generated_matrix():
    import synth
    W = synth.weights(0, 0, 0, 512, 256)
    enc = oracle.encode(W)
    assert np.array_equal(oracle.decode(enc), W)


# ----------------------------------------------------------------------------- window choice

def brute_force_base(row):
    """Count normal values in every legal window directly; fullest, lowest base."""
    E = exponent(row).astype(np.int64)
    normal = (E >= 1) & (E <= 254)
    best, best_b = -1, None
    for b in range(1, 240):
        c = int(np.sum(normal & (E >= b) & (E <= b + 15)))
        if c > best:
            best, best_b = c, b
    return best_b, best


def test_window_matches_brute_force_on_tiny_rows():
    rng = np.random.default_rng(1234)
    for trial in range(400):
        K = int(rng.integers(1, 65))
        centre = int(rng.integers(1, 255))
        spread = int(rng.integers(0, 60))
        E = np.clip(rng.integers(centre - spread, centre + spread + 1, K), 0, 255)
        if trial % 7 == 0:
            E[rng.random(K) < 0.3] = 0          # zeros / denormals
        if trial % 11 == 0:
            E[rng.random(K) < 0.2] = 255        # Inf / NaN
        row = ((rng.integers(0, 2, K) << 15) | (E << 7) | rng.integers(0, 128, K)).astype(np.uint16)
        b_ref, count = brute_force_base(row)
        b = oracle.base_of_row(row)
        assert b == b_ref, (trial, b, b_ref)
        enc = oracle.encode(row[None, :])
        assert K - enc.n_esc == count          # in-window values are exactly the fullest window's count


@pytest.mark.parametrize("E0,expect", [(127, 112), (5, 1), (1, 1), (16, 1), (17, 2), (254, 239), (200, 185)])
def test_window_single_binade(E0, expect):
    """All values share one exponent: every window holding it ties, the lowest wins."""
    row = np.array([(E0 << 7) | m for m in range(20)], np.uint16)
    assert oracle.base_of_row(row) == expect


def test_window_two_clusters():
    far = np.array([100 << 7] * 10 + [140 << 7] * 20, np.uint16)        # 40 binades apart: larger cluster wins
    assert oracle.base_of_row(far) == 125
    near = np.array([100 << 7] * 10 + [110 << 7] * 20, np.uint16)       # both fit: lowest window holding both
    assert oracle.base_of_row(near) == 95
    no_normal = np.array([0x0000, 0x8000, 0x0001, 0x807F], np.uint16)
    assert oracle.base_of_row(no_normal) == 1


# ----------------------------------------------------------------------------- golden fixtures

def _hex_list(s):
    return [int(t, 16) for t in s.split()] if s.strip() else []


def load_record_fixture():
    rows, q8 = {}, {}
    for line in open(os.path.join(GOLDEN, "w12_records.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        parts = [p.strip() for p in line.split("|")]
        if parts[0].startswith("q8"):
            q8[int(parts[0].split()[1])] = _hex_list(parts[1])
            continue
        esc = [(int(c), int(r, 16)) for c, r in (t.split(":") for t in parts[5].split())]
        rows[int(parts[0])] = dict(w=_hex_list(parts[1]), base=int(parts[2]), hi=_hex_list(parts[3]),
                                   lo=_hex_list(parts[4]), esc=esc)
    return rows, q8


def test_golden_records():
    rows, q8 = load_record_fixture()
    for r, case in rows.items():
        enc = oracle.encode(np.array([case["w"]], np.uint16))
        assert int(enc.base[0]) == case["base"], r
        assert enc.hi[0].tolist() == case["hi"], r
        assert enc.lo[0].tolist() == case["lo"], r
        got = [(int(e >> 16), int(e & 0xFFFF)) for e in enc.esc]
        assert got == case["esc"], r
        assert oracle.decode(enc)[0].tolist() == case["w"], r
        assert oracle.decode_q8(enc)[0].tolist() == q8[r], r


# ----------------------------------------------------------------------------- size

def test_bits_per_weight_is_12_plus_escape_overhead():
    import synth
    for (N, K) in [(512, 256), (64, 5120), (7, 33)]:
        W = synth.weights(0, 3, 1, N, K)
        enc = oracle.encode(W)
        # escapes counted independently of the encoder, from the chosen bases
        E = exponent(W).astype(np.int64)
        b = enc.base.astype(np.int64)[:, None]
        outside = (E == 0) | (E == 255) | (E < b) | (E > b + 15)
        assert enc.n_esc == int(outside.sum())
        bits = 12 * N * K + 32 * enc.n_esc + 32 * (N + 1) + 8 * N
        assert enc.storage_bits() == bits
        assert enc.hi.size == N * K and enc.lo.size == N * ((K + 1) // 2)


def test_bits_per_weight_on_gaussian_rows_is_in_the_pages_range():
    """Plain per-channel Gaussian weights (no injected outliers) land at
    12.01-12.02 bits/weight, the range the pages report for 8 dense models."""
    rng = np.random.default_rng(7)
    N, K = 256, 5120
    s = np.exp(rng.uniform(np.log(0.005), np.log(0.05), N)).astype(np.float32)
    W = bf16_of_f32(rng.standard_normal((N, K)).astype(np.float32) * s[:, None])
    enc = oracle.encode(W)
    bpw = enc.storage_bits() / (N * K)
    assert 12.005 < bpw < 12.02, bpw


# ----------------------------------------------------------------------------- Q8 view

def test_q8_closed_form():
    import synth
    W = synth.weights(0, 0, 1, 300, 200)
    enc = oracle.encode(W)
    q = oracle.decode_q8(enc)
    E = exponent(W).astype(np.int64)
    b = enc.base.astype(np.int64)[:, None]
    inwin = (E >= 1) & (E <= 254) & (E >= b) & (E <= b + 15)
    assert np.array_equal(q[inwin], W[inwin] & 0xFFF0)
    assert np.array_equal(q[~inwin], W[~inwin])
    wf, qf = np.abs(f32_of_bf16(W[inwin])).astype(np.float64), np.abs(f32_of_bf16(q[inwin])).astype(np.float64)
    assert np.all(qf <= wf)
    assert np.all((wf - qf) / wf < 2.0 ** -3)


# ----------------------------------------------------------------------------- GEMM

def test_gemm_one_hot_selects_a_column():
    import synth
    W = synth.weights(0, 0, 0, 64, 96)
    for k0 in [0, 17, 95]:
        x = np.zeros((1, 96), np.uint16)
        x[0, k0] = 0x3F80                       # 1.0
        y, B = oracle.gemm(x, W, threads=1)
        assert np.array_equal(y[0], f32_of_bf16(W[:, k0]).astype(np.float64))
        assert np.array_equal(B[0], np.abs(y[0]))


def test_gemm_exact_on_small_integers():
    rng = np.random.default_rng(3)
    M, N, K = 5, 37, 203
    xi = rng.integers(-8, 9, (M, K))
    wi = rng.integers(-8, 9, (N, K))
    y, B = oracle.gemm(bf16_of_f32(xi.astype(np.float32)), bf16_of_f32(wi.astype(np.float32)), threads=3)
    assert np.array_equal(y, (xi @ wi.T).astype(np.float64))
    assert np.array_equal(B, (np.abs(xi) @ np.abs(wi).T).astype(np.float64))


def test_gemm_matches_numpy_float64():
    import synth
    W = synth.weights(0, 1, 2, 70, 300)
    x = synth.activations(1, 1, 2, 6, 300)
    y, B = oracle.gemm(x, W, threads=4)
    xf, wf = f32_of_bf16(x).astype(np.float64), f32_of_bf16(W).astype(np.float64)
    assert np.allclose(y, xf @ wf.T, rtol=0, atol=1e-12 * B.max())
    assert np.allclose(B, np.abs(xf) @ np.abs(wf).T, rtol=1e-12)
    assert np.all(B >= np.abs(y))


# ----------------------------------------------------------------------------- argmax

def test_argmax_ties_lowest_index_and_gap():
    L = np.array([[1.0, 3.0, 3.0, 2.0],
                  [-0.0, 0.0, -1.0, -2.0],
                  [np.nan, -np.inf, -5.0, np.nan],
                  [7.0, np.nan, 7.5, 7.25]])
    idx, gap = oracle.argmax(L)
    assert idx.tolist() == [1, 0, 2, 2]
    assert gap[0] == 0.0 and gap[1] == 0.0 and gap[3] == 0.25


def test_argmax_matches_numpy():
    rng = np.random.default_rng(5)
    L = rng.standard_normal((9, 1000))
    idx, gap = oracle.argmax(L)
    assert np.array_equal(idx, np.argmax(L, axis=1))
    s = np.sort(L, axis=1)
    assert np.allclose(gap, s[:, -1] - s[:, -2])


# ----------------------------------------------------------------------------- acceptance

def brute_force_accept(tok, parent, draft):
    """Walk every root-to-leaf path while draft == target token at the parent;
    best = max by (depth, -node)."""
    n = len(parent)
    children = {i: [] for i in range(n)}
    for i in range(1, n):
        children[int(parent[i])].append(i)
    leaves = [i for i in range(n) if not children[i]]
    best = (0, 0)
    for leaf in leaves:
        path = [leaf]
        while path[-1] != 0:
            path.append(int(parent[path[-1]]))
        path = path[::-1]
        for d in range(1, len(path)):
            if draft[path[d]] != tok[path[d - 1]]:
                break
            if (d, -path[d]) > (best[0], -best[1]):
                best = (d, path[d])
    node = best[1]
    path = [node]
    while path[-1] != 0:
        path.append(int(parent[path[-1]]))
    return best[0], path[::-1], int(tok[node])


def load_tree_fixture():
    cases = []
    for line in open(os.path.join(GOLDEN, "tree_cases.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        p = [s.strip() for s in line.split("|")]
        ints = lambda s: [int(t) for t in s.split()] if s != "-" else []
        cases.append(dict(name=p[0], parent=ints(p[1]), tok=ints(p[2]), draft=ints(p[3]), L=int(p[4]),
                          path=ints(p[5]), bonus=int(p[6])))
    return cases


def test_golden_trees():
    for c in load_tree_fixture():
        L, path, bonus = oracle.accept(c["tok"], c["parent"], c["draft"])
        assert L == c["L"], c["name"]
        if L >= 0:
            assert path.tolist() == c["path"] and bonus == c["bonus"], c["name"]


def test_accept_matches_brute_force_on_random_trees():
    import synth
    rng = np.random.default_rng(11)
    for t in range(600):
        n = int(rng.integers(1, 40))
        V = int(rng.choice([2, 3, 4, 1024]))
        parent = synth.tree(2, t, 0, n)
        tok = rng.integers(0, V, n).astype(np.int32)
        draft = rng.integers(0, V, n).astype(np.int32)
        # plant: half the nodes copy the target token at their parent
        plant = rng.random(n) < 0.6
        for i in range(1, n):
            if plant[i]:
                draft[i] = tok[parent[i]]
        L, path, bonus = oracle.accept(tok, parent, draft)
        Lb, pathb, bonusb = brute_force_accept(tok, parent, draft)
        assert (L, path.tolist(), bonus) == (Lb, pathb, bonusb), t


def test_accept_chain_all_match_gives_full_depth():
    for n in [1, 2, 8, 33]:
        parent = np.arange(-1, n - 1, dtype=np.int32)
        tok = np.arange(100, 100 + n, dtype=np.int32)
        draft = np.concatenate([[0], tok[:-1]]).astype(np.int32)
        L, path, bonus = oracle.accept(tok, parent, draft)
        assert L == n - 1 and path.tolist() == list(range(n)) and bonus == tok[-1]


# ---------------------------------------------------------------- two-level verification splice

def load_tlv_fixture():
    cases = []
    for line in open(os.path.join(GOLDEN, "tlv_splice_cases.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        p = [t.strip() for t in line.split("|")]
        ints = lambda t: [int(v) for v in t.split()] if t != "-" else None
        cases.append(dict(name=p[0], L=int(p[1]), path=ints(p[2]) or [], bonus=int(p[3]), draft_q=ints(p[4]),
                          sub_parent=ints(p[5]), sub_draft=ints(p[6]), n=int(p[7]), parent=ints(p[8]),
                          draft=ints(p[9]), src=ints(p[10])))
    return cases


def test_golden_tlv_splices():
    for c in load_tlv_fixture():
        r = oracle.tlv_splice(c["L"], c["path"], c["bonus"], c["draft_q"], c["sub_parent"], c["sub_draft"], c["n"])
        if c["parent"] is None:
            assert r is None, c["name"]
            continue
        parent, draft, src = r
        assert parent.tolist() == c["parent"], c["name"]
        assert draft.tolist() == c["draft"], c["name"]
        assert src.tolist() == c["src"], c["name"]


def test_tlv_splice_keeps_the_q_path_accepted():
    """Property of the splice itself: when the exact pass reproduces the Q pass's target
    tokens on the reused rows, greedy acceptance on the spliced tree walks the whole Q
    path and then the bonus node (L_exact >= L_q + 1, path prefix 0..L_q+1), whatever the
    new rows' tokens.  Checked against the brute-force acceptance walk on random trees."""
    import synth
    rng = np.random.default_rng(21)
    checked = 0
    for t in range(400):
        n1 = int(rng.integers(1, 32))
        V = int(rng.integers(2, 6))
        p1 = synth.tree(2, 50, t, n1)
        tq = rng.integers(0, V, n1).astype(np.int32)
        d1 = rng.integers(0, V, n1).astype(np.int32)
        for i in range(1, n1):
            if rng.random() < 0.6:
                d1[i] = tq[p1[i]]
        L, path, bonus = oracle.accept(tq, p1, d1)
        n = 32
        sp = np.array([-1 if j == 0 or rng.random() < 0.3 else int(rng.integers(0, j)) for j in range(n)], np.int32)
        sd = rng.integers(0, V, n).astype(np.int32)
        r = oracle.tlv_splice(L, path, bonus, d1, sp, sd, n)
        if L + 2 > n:
            assert r is None
            continue
        parent, draft, src = r
        assert parent[0] == -1 and all(0 <= parent[i] < i for i in range(1, n))
        assert sorted(src[src >= 0].tolist()) == sorted(path.tolist())
        assert sorted((-1 - src[src < 0]).tolist()) == list(range(n - L - 1))
        te = np.where(src >= 0, tq[np.maximum(src, 0)], rng.integers(0, V, n)).astype(np.int32)
        L2, path2, _ = brute_force_accept(te, parent, draft)
        assert L2 >= L + 1 and path2[:L + 2] == list(range(L + 2)), (t, L, L2, path2)
        checked += 1
    assert checked > 300


def test_tlv_splice_rejects_invalid_input():
    assert oracle.tlv_splice(-1, [], -1, [0], [-1], [0], 4) is None          # Q tree was invalid
    assert oracle.tlv_splice(3, [0, 1, 2, 3], 5, [0, 1, 2, 3], [-1], [0], 4) is None   # no room for the bonus
    assert oracle.tlv_splice(0, [0], 5, [0], [-1, 1], [0, 0], 4) is None      # subtree parent not earlier


# ---------------------------------------------------------------- node budget shared across requests

def load_budget_fixture():
    cases = []
    for line in open(os.path.join(GOLDEN, "budget_cases.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        p = [t.strip() for t in line.split("|")]
        ints = lambda t: [int(v) for v in t.split()]
        cases.append(dict(name=p[0], off=ints(p[1]), parent=ints(p[2]), conf=[float(v) for v in p[3].split()],
                          budget=int(p[4]), per_request=bool(int(p[5])), parent_out=ints(p[6]), src_out=ints(p[7]),
                          off_out=ints(p[8])))
    return cases


def test_golden_budget_selections():
    for c in load_budget_fixture():
        draft = list(range(100, 100 + len(c["parent"])))
        po, do, so, oo = oracle.budget_select(c["parent"], np.array(c["conf"], np.float32), draft, c["off"],
                                              c["budget"], c["per_request"])
        assert po.tolist() == c["parent_out"], c["name"]
        assert so.tolist() == c["src_out"], c["name"]
        assert oo.tolist() == c["off_out"], c["name"]
        assert do.tolist() == [draft[i] for i in c["src_out"]], c["name"]


def random_forest(rng, n_req, max_nodes, one_prob=0.2):
    parents, confs, offs = [], [], [0]
    for r in range(n_req):
        n = int(rng.integers(1, max_nodes + 1))
        p = np.array([-1] + [int(rng.integers(0, i)) for i in range(1, n)], np.int32)
        c = rng.uniform(0.05, 1.0, n).astype(np.float32)
        c[rng.random(n) < one_prob] = 1.0       # ties: whole paths of equal score
        parents.append(p), confs.append(c), offs.append(offs[-1] + n)
    return np.concatenate(parents), np.concatenate(confs), np.array(offs, np.int32)


def path_scores(parent, conf, off):
    """float32 product of the confidences from the root, root first (written out here
    independently of the oracle)."""
    score = np.zeros(conf.size, np.float32)
    depth = np.zeros(conf.size, np.int32)
    for r in range(off.size - 1):
        for i in range(off[r], off[r + 1]):
            if i == off[r]:
                score[i], depth[i] = conf[i], 0
            else:
                p = off[r] + parent[i]
                score[i] = np.float32(score[p] * conf[i])
                depth[i] = depth[p] + 1
    return score, depth


def test_budget_is_the_best_ancestor_closed_set():
    """Brute force on tiny forests: the kept set is closed under ancestors, has
    min(budget, nodes) nodes, and its score sum is the largest over every ancestor-closed
    set of that size; kept parents are renumbered onto kept ancestors."""
    import itertools
    rng = np.random.default_rng(31)
    for t in range(250):
        parent, conf, off = random_forest(rng, int(rng.integers(1, 4)), 5)
        C = int(off[-1])
        budget = int(rng.integers(1, C + 2))
        draft = np.arange(C, dtype=np.int32)
        po, do, so, oo = oracle.budget_select(parent, conf, draft, off, budget)
        score, _ = path_scores(parent, conf, off)
        req = np.searchsorted(off, np.arange(C), side="right") - 1
        glob_parent = np.array([-1 if parent[i] < 0 else off[req[i]] + parent[i] for i in range(C)])
        kept = set(so.tolist())
        k = min(budget, C)
        assert len(kept) == k, t
        assert all(glob_parent[i] < 0 or glob_parent[i] in kept for i in kept), t
        best = -1.0
        for sub in itertools.combinations(range(C), k):
            ss = set(sub)
            if all(glob_parent[i] < 0 or glob_parent[i] in ss for i in sub):
                best = max(best, float(sum(np.float64(score[i]) for i in sub)))
        assert abs(float(sum(np.float64(score[i]) for i in kept)) - best) < 1e-12, t
        for r in range(off.size - 1):
            a, b = oo[r], oo[r + 1]
            for j in range(a, b):
                i = so[j]
                assert req[i] == r and (po[j] == -1) == (parent[i] < 0), t
                if po[j] >= 0:
                    assert so[a + po[j]] == glob_parent[i] and po[j] < j - a, t
        assert np.array_equal(do, draft[so]), t


def test_per_request_budget_is_the_shared_rule_on_each_request():
    rng = np.random.default_rng(32)
    for t in range(150):
        parent, conf, off = random_forest(rng, int(rng.integers(1, 6)), 12)
        k = int(rng.integers(1, 6))
        draft = np.arange(off[-1], dtype=np.int32)
        po, do, so, oo = oracle.budget_select(parent, conf, draft, off, k, per_request=True)
        for r in range(off.size - 1):
            a, b = off[r], off[r + 1]
            p1, d1, s1, o1 = oracle.budget_select(parent[a:b], conf[a:b], draft[a:b], np.array([0, b - a]), k)
            assert po[oo[r]:oo[r + 1]].tolist() == p1.tolist(), t
            assert (so[oo[r]:oo[r + 1]] - a).tolist() == s1.tolist(), t


def test_budget_rejects_invalid_trees():
    conf = np.ones(4, np.float32)
    assert oracle.budget_select([0, 0, 1, 2], conf, [0] * 4, [0, 4], 2) is None     # no root
    assert oracle.budget_select([-1, 1, 0, 0], conf, [0] * 4, [0, 4], 2) is None    # parent not earlier


# ----------------------------------------------------------------------------- certified INT8 head
# Same page and section: on H100 the LM head stays in INT8, a Cauchy-Schwarz error
# bound filters the candidates and those are computed exactly.  The pins: closed forms
# of the quantizer, the bound containing every exact logit (tight along the error
# direction), and the certified argmax equal to a brute-force argmax of the exact logits.

def i8_values(code):
    code = np.asarray(code)
    return np.where(code & 0x80, -(code & 0x7F).astype(np.int64), (code & 0x7F).astype(np.int64))


def test_i8_quantize_unit_scale_is_rint_ties_to_even():
    """A channel whose largest magnitude is 127 has scale exactly 1, so the codes are
    the weights rounded half to even, as sign-magnitude bytes."""
    W = bf16_of_f32([[127.0, 2.5, 3.5, -0.5, -2.5, 0.0, -127.0, 1.5, 0.25, -0.75, 126.5]])
    code, scale, _ = oracle.i8_quantize(W)
    assert scale[0] == 1.0
    assert code[0].tolist() == [127, 2, 4, 0, 0x82, 0, 0xFF, 2, 0, 0x81, 126]


def head_like_rows(rng, N, K):
    """bf16 rows with per-channel scales, a few zeros, denormals and, in some rows, outliers."""
    s = 0.005 * 10 ** rng.random(N)
    w = rng.standard_normal((N, K)) * s[:, None]
    w[rng.random((N, K)) < 0.002] = 0.0
    out = rng.random((N, K)) < 0.01
    w[out & (rng.random((N, 1)) < 0.3)] *= 512.0
    bits = bf16_of_f32(w.astype(np.float32))
    den = rng.random((N, K)) < 0.001
    bits[den] = (rng.integers(1, 128, den.sum()) | (rng.integers(0, 2, den.sum()) << 15)).astype(np.uint16)
    return bits


def test_i8_quantize_invariants():
    rng = np.random.default_rng(21)
    W = head_like_rows(rng, 60, 200)
    W[5] = 0                                   # an all-zero channel
    W[6] = (np.arange(200) % 127 + 1).astype(np.uint16)    # denormals only
    code, scale, cb = oracle.i8_quantize(W)
    w = f32_of_bf16(W).astype(np.float64)
    q = i8_values(code)
    s = scale.astype(np.float64)
    amax = np.abs(w).max(axis=1)
    assert (np.abs(q) <= 127).all() and (np.sign(q) * np.sign(w) >= 0).all()
    assert ((code & 0x80) == 0)[q == 0].all()           # no negative zero code
    for n in range(60):
        if amax[n] == 0:
            assert s[n] == 0 and (q[n] == 0).all() and cb[n] == 0
            continue
        assert abs(q[n, np.argmax(np.abs(w[n]))]) == 127
        assert abs(s[n] * 127 - amax[n]) <= amax[n] * 2.0 ** -23
        # every weight within half a step of its code
        assert (np.abs(w[n] - s[n] * q[n]) <= 0.5 * s[n] * (1 + 1e-12)).all()
        assert cb[n] >= np.sqrt(((w[n] - s[n] * q[n]) ** 2).sum())


def test_i8_bound_contains_exact_logits_and_is_tight_along_the_error():
    """|exact - approximate| <= ||x|| c for every channel and row; along the error
    direction the difference reaches ||x|| ||w - s q|| (Cauchy-Schwarz is an equality
    there), so the quantization term of c cannot be dropped or shrunk."""
    rng = np.random.default_rng(22)
    N, K = 48, 320
    W = head_like_rows(rng, N, K)
    code, scale, cb = oracle.i8_quantize(W)
    w = f32_of_bf16(W).astype(np.float64)
    q = i8_values(code).astype(np.float64)
    s = scale.astype(np.float64)
    x = f32_of_bf16(bf16_of_f32(rng.standard_normal((20, K)).astype(np.float32))).astype(np.float64)
    exact = x @ w.T
    approx = (x @ q.T) * s[None, :]
    B = np.sqrt((x * x).sum(1))[:, None] * cb[None, :].astype(np.float64)
    assert (np.abs(exact - approx) <= B).all()
    for n in range(N):
        err = w[n] - s[n] * q[n]
        if not err.any():
            continue
        xe = f32_of_bf16(bf16_of_f32((err / np.abs(err).max()).astype(np.float32))).astype(np.float64)
        gap = abs(xe @ w[n] - s[n] * (xe @ q[n]))
        nx = np.sqrt((xe * xe).sum())
        assert gap <= nx * cb[n]
        assert gap >= 0.99 * nx * np.sqrt((err * err).sum())


@pytest.mark.parametrize("peaked", [False, True])
def test_cert_argmax_equals_brute_force_argmax(peaked):
    rng = np.random.default_rng(23 + peaked)
    V, K, M = 400, 256, 24
    W = head_like_rows(rng, V, K)
    w = f32_of_bf16(W).astype(np.float64)
    z = rng.standard_normal((M, K))
    if peaked:
        t = rng.integers(0, V, M)
        z = z + 6.0 * w[t] / np.linalg.norm(w[t], axis=1, keepdims=True)
    x = bf16_of_f32(z.astype(np.float32))
    code, scale, cb = oracle.i8_quantize(W)
    idx, ncand = oracle.cert_argmax(x, W, code, scale, cb)
    exact = f32_of_bf16(x).astype(np.float64) @ w.T
    assert np.array_equal(idx, np.argmax(exact, axis=1))
    assert (ncand >= 1).all() and (ncand <= V).all()
    if peaked:
        assert ncand.mean() < V / 4


def test_cert_argmax_all_zero_head_and_single_channel():
    x = bf16_of_f32(np.ones((2, 8), np.float32))
    W = np.zeros((3, 8), np.uint16)
    code, scale, cb = oracle.i8_quantize(W)
    idx, ncand = oracle.cert_argmax(x, W, code, scale, cb)
    assert idx.tolist() == [0, 0] and ncand.tolist() == [3, 3]     # a three-way tie: lowest index
    W1 = bf16_of_f32(np.full((1, 8), -0.5, np.float32))
    code, scale, cb = oracle.i8_quantize(W1)
    idx, ncand = oracle.cert_argmax(x, W1, code, scale, cb)
    assert idx.tolist() == [0, 0] and ncand.tolist() == [1, 1]


# ----------------------------------------------------------------------------- GDN path verify
# Same page and section: for a hybrid target (most layers Gated DeltaNet) a path-verify
# kernel recomputes the recurrent state along each draft path, a commit kernel replays the
# accepted path, and the WY kernel holds the FP32 state in three BF16 pieces exactly.

def test_split3_is_exact_and_first_piece_is_bf16_rne():
    import torch
    rng = np.random.default_rng(31)
    e = rng.integers(-100, 127, 20000)
    m = rng.random(20000) + 1.0
    x = (np.sign(rng.random(20000) - 0.5) * m * 2.0 ** e).astype(np.float32)
    x = np.concatenate([x, np.float32([0.0, -0.0, 1.0, -2.5, 1 + 2 ** -23, 3.0e38, 2.0 ** -100])])
    s1, s2, s3 = oracle.split3(x)
    v = [f32_of_bf16(s).astype(np.float64) for s in (s1, s2, s3)]
    assert np.array_equal(v[0] + v[1] + v[2], x.astype(np.float64))
    # the first piece is the library's round-to-nearest-even bf16 conversion
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(s1, ref)
    # each further piece is at most half a unit in the last place of the one before
    nz = v[0] != 0
    assert (np.abs(v[1][nz]) <= np.abs(v[0][nz]) * 2.0 ** -8).all()
    # a value that is already bf16 has empty further pieces
    b = f32_of_bf16(s1)
    t1, t2, t3 = oracle.split3(b)
    assert np.array_equal(t1, s1) and not t2.any() and not t3.any()


def gdn_inputs(rng, n, H, dk, dv, unit_k=True):
    S0 = rng.standard_normal((H, dv, dk)).astype(np.float32) * 0.5
    q = bf16_of_f32((rng.standard_normal((n, H, dk)) / np.sqrt(dk)).astype(np.float32))
    kk = rng.standard_normal((n, H, dk))
    if unit_k:
        kk /= np.linalg.norm(kk, axis=2, keepdims=True)
    k = bf16_of_f32(kk.astype(np.float32))
    v = bf16_of_f32(rng.standard_normal((n, H, dv)).astype(np.float32))
    alpha = rng.uniform(0.85, 1.0, (n, H)).astype(np.float32)
    beta = rng.uniform(0.1, 0.9, (n, H)).astype(np.float32)
    return S0, q, k, v, alpha, beta


def random_tree(rng, n):
    return np.array([-1] + [int(rng.integers(0, i)) for i in range(1, n)], np.int32)


def depth_of(parent):
    d = np.zeros(len(parent), np.int64)
    for i in range(1, len(parent)):
        d[i] = d[parent[i]] + 1
    return d


def test_gdn_no_write_is_the_gated_decay_of_s0():
    """beta = 0: no rank-1 writes, so node i reads (product of alpha on its path) * S0 q_i;
    alpha = 1 as well leaves S0 q_i."""
    rng = np.random.default_rng(32)
    n, H, dk, dv = 12, 2, 16, 8
    S0, q, k, v, alpha, beta = gdn_inputs(rng, n, H, dk, dv)
    parent = random_tree(rng, n)
    beta[:] = 0
    O = oracle.gdn_tree(S0, q, k, v, alpha, beta, parent)
    qf = f32_of_bf16(q).astype(np.float64)
    base = np.einsum("hvk,nhk->nhv", S0.astype(np.float64), qf)
    decay = np.ones((n, H))
    for i in range(1, n):
        decay[i] = decay[parent[i]] * alpha[i].astype(np.float64)
    assert np.allclose(O, base * decay[:, :, None], rtol=1e-12, atol=1e-12)
    alpha[:] = 1
    assert np.allclose(oracle.gdn_tree(S0, q, k, v, alpha, beta, parent), base, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("a", [1.0, 0.75])
def test_gdn_delta_rule_overwrites_the_key_column(a):
    """k = e_j, beta = 1, alpha = a: the update erases the decayed column j and writes v
    there, so a query e_j reads v exactly and a query e_m (m != j) reads a * S0's
    column m."""
    rng = np.random.default_rng(33)
    H, dk, dv = 3, 8, 6
    S0, q, k, v, alpha, beta = gdn_inputs(rng, 2, H, dk, dv)
    parent = np.array([-1, 0], np.int32)
    alpha[:] = a
    beta[:] = 1
    j, mcol = 3, 5
    k[:] = 0
    k[1, :, j] = 0x3F80                   # e_j
    for col, expect in ((j, f32_of_bf16(v[1]).astype(np.float64)), (mcol, a * S0[:, :, mcol].astype(np.float64))):
        q[:] = 0
        q[1, :, col] = 0x3F80
        O = oracle.gdn_tree(S0, q, k, v, alpha, beta, parent)
        assert np.array_equal(O[1], expect)


def test_gdn_tree_node_equals_its_path_as_a_chain():
    rng = np.random.default_rng(34)
    n, H, dk, dv = 10, 2, 16, 16
    S0, q, k, v, alpha, beta = gdn_inputs(rng, n, H, dk, dv)
    parent = random_tree(rng, n)
    O = oracle.gdn_tree(S0, q, k, v, alpha, beta, parent)
    for i in range(n):
        path = []
        j = i
        while j >= 0:
            path.append(j)
            j = parent[j]
        path = path[::-1]                        # root .. i
        L = len(path)
        chain = np.arange(-1, L - 1, dtype=np.int32)
        Oc = oracle.gdn_tree(S0, q[path], k[path], v[path], alpha[path], beta[path], chain)
        assert np.array_equal(Oc[L - 1], O[i])


def test_gdn_commit_then_read_equals_the_tree_output():
    """Replaying a path into the state and then reading with node i's query gives node i's
    tree output; an empty commit leaves S0."""
    rng = np.random.default_rng(35)
    n, H, dk, dv = 9, 2, 16, 12
    S0, q, k, v, alpha, beta = gdn_inputs(rng, n, H, dk, dv)
    parent = random_tree(rng, n)
    O = oracle.gdn_tree(S0, q, k, v, alpha, beta, parent)
    i = int(np.argmax(depth_of(parent)))
    path = []
    j = i
    while j > 0:
        path.append(j)
        j = parent[j]
    S = oracle.gdn_commit(S0, k, v, alpha, beta, path[::-1])
    read = np.einsum("hvk,hk->hv", S, f32_of_bf16(q[i]).astype(np.float64))
    assert np.allclose(read, O[i], rtol=1e-12, atol=1e-12)
    assert np.array_equal(oracle.gdn_commit(S0, k, v, alpha, beta, []), S0.astype(np.float64))


def test_gdn_rejects_invalid_trees():
    rng = np.random.default_rng(36)
    S0, q, k, v, alpha, beta = gdn_inputs(rng, 3, 1, 4, 4)
    for bad in ([0, 0, 1], [-1, 1, 0], [-1, 0, 3]):
        assert oracle.gdn_tree(S0, q, k, v, alpha, beta, np.array(bad, np.int32)) is None
