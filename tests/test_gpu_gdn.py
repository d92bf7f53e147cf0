"""Recurrent-layer verification (gated delta rule) on the GPU against the oracle.

The SpecPilot summary page (onedev.kr/papers/1654), section "What's different":
path verify recomputes each draft node's recurrent state along its path, commit
replays the accepted path, and the FP32 state is held exactly in three BF16 pieces.
The split is compared bit for bit.  Outputs and states are float on the GPU and fp64
in the oracle: every value is a sum of at most dk products per step, at most depth+1
steps, so the float error stays below about (depth+1) * dk * 2^-24 of the values'
scale; the tests allow 2e-4 of each row's largest magnitude (plus 1e-6).
"""
import numpy as np
import pytest
import torch

import oracle
from tests._gpu_util import f32_of_bf16, to_dev16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w12():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import lossless_bit_weights_gb300 as m
    m.lib()
    return m


def bf16_bits(a):
    u = np.asarray(a, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def inputs(rng, n, H, dk, dv):
    S0 = (rng.standard_normal((H, dv, dk)) * 0.5).astype(np.float32)
    q = bf16_bits(rng.standard_normal((n, H, dk)) / np.sqrt(dk))
    kk = rng.standard_normal((n, H, dk))
    k = bf16_bits(kk / np.linalg.norm(kk, axis=2, keepdims=True))
    v = bf16_bits(rng.standard_normal((n, H, dv)))
    alpha = rng.uniform(0.85, 1.0, (n, H)).astype(np.float32)
    beta = rng.uniform(0.1, 0.9, (n, H)).astype(np.float32)
    return S0, q, k, v, alpha, beta


def tree(rng, n, chain=False):
    if chain:
        return np.arange(-1, n - 1, dtype=np.int32)
    return np.array([-1] + [int(rng.integers(max(0, i - 4), i)) for i in range(1, n)], np.int32)


def dev(a, dtype=None):
    if a.dtype == np.uint16:
        return to_dev16(a)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_close(got, ref):
    scale = np.abs(ref).max(axis=-1, keepdims=True)
    err = np.abs(got.astype(np.float64) - ref)
    assert (err <= 2e-4 * scale + 1e-6).all(), float((err / (scale + 1e-30)).max())


def test_split3_matches_oracle(w12):
    rng = np.random.default_rng(41)
    e = rng.integers(-100, 127, 100000)
    x = (np.sign(rng.random(100000) - 0.5) * (rng.random(100000) + 1.0) * 2.0 ** e).astype(np.float32)
    x = np.concatenate([x, np.float32([0.0, -0.0, 1.0, 3.0e38, 2.0 ** -100, 1 + 2 ** -23])])
    got = w12.gdn_split3(dev(x))
    ref = oracle.split3(x)
    for g, r in zip(got, ref):
        assert np.array_equal(g.cpu().numpy().view(np.uint16), r)
    assert np.array_equal(sum(f32_of_bf16(r).astype(np.float64) for r in ref), x.astype(np.float64))


@pytest.mark.parametrize("n,H,dk,dv,chain", [(1, 1, 16, 16, False), (5, 3, 64, 32, False), (32, 2, 128, 128, False),
                                             (12, 2, 48, 80, True), (40, 1, 96, 64, False), (9, 2, 64, 100, False),
                                             (7, 2, 128, 200, False), (6, 1, 128, 1, True)])
def test_path_verify_matches_oracle(w12, n, H, dk, dv, chain):
    rng = np.random.default_rng(n * 7 + H)
    S0, q, k, v, alpha, beta = inputs(rng, n, H, dk, dv)
    parent = tree(rng, n, chain)
    O, status = w12.gdn_path_verify(dev(S0), dev(q), dev(k), dev(v), dev(alpha), dev(beta), dev(parent))
    assert int(status.item()) == 0
    assert_close(O.cpu().numpy(), oracle.gdn_tree(S0, q, k, v, alpha, beta, parent))


def test_path_verify_full_size_tree(w12):
    """32-node tree, 32 heads of 128 x 128 state: the per-layer shape of the bench row."""
    rng = np.random.default_rng(42)
    n, H, dk, dv = 32, 32, 128, 128
    S0, q, k, v, alpha, beta = inputs(rng, n, H, dk, dv)
    parent = tree(rng, n)
    O, status = w12.gdn_path_verify(dev(S0), dev(q), dev(k), dev(v), dev(alpha), dev(beta), dev(parent))
    assert int(status.item()) == 0
    assert_close(O.cpu().numpy(), oracle.gdn_tree(S0, q, k, v, alpha, beta, parent))


def test_path_verify_flags_invalid_trees(w12):
    rng = np.random.default_rng(43)
    S0, q, k, v, alpha, beta = inputs(rng, 4, 1, 16, 16)
    for bad in ([0, 0, 1, 2], [-1, 0, 2, 1], [-1, 0, 5, 1]):
        _, status = w12.gdn_path_verify(dev(S0), dev(q), dev(k), dev(v), dev(alpha), dev(beta),
                                        dev(np.array(bad, np.int32)))
        assert int(status.item()) & 1


@pytest.mark.parametrize("L,dk,dv", [(0, 128, 64), (1, 128, 64), (3, 128, 64), (3, 64, 128), (2, 96, 40),
                                     (3, 128, 160)])
def test_commit_matches_oracle(w12, L, dk, dv):
    rng = np.random.default_rng(44 + L + dk + dv)
    n, H = 16, 4
    S0, q, k, v, alpha, beta = inputs(rng, n, H, dk, dv)
    nodes = [int(j) for j in rng.choice(np.arange(1, n), L, replace=False)]
    path_nodes = np.zeros(n, np.int32)
    path_nodes[1:L + 1] = nodes
    S = dev(S0.copy())
    status = w12.gdn_commit(S, dev(k), dev(v), dev(alpha), dev(beta), dev(np.int32([L])), dev(path_nodes))
    assert int(status.item()) == 0
    ref = oracle.gdn_commit(S0, k, v, alpha, beta, nodes)
    assert_close(S.cpu().numpy().reshape(H * dv, dk), ref.reshape(H * dv, dk))


def test_commit_rejects_bad_paths(w12):
    rng = np.random.default_rng(45)
    n, H, dk, dv = 6, 1, 16, 16
    S0, q, k, v, alpha, beta = inputs(rng, n, H, dk, dv)
    for L, nodes in ((6, [0, 1, 2, 3, 4, 5]), (2, [0, 1, 9, 0, 0, 0]), (1, [0, 0, 0, 0, 0, 0])):
        S = dev(S0.copy())
        status = w12.gdn_commit(S, dev(k), dev(v), dev(alpha), dev(beta), dev(np.int32([L])),
                                dev(np.array(nodes, np.int32)))
        assert int(status.item()) & 2
        assert torch.equal(S.cpu(), torch.from_numpy(S0))


def test_commit_after_acceptance(w12):
    """Commit the path the tree acceptance returns (device outputs fed straight in), then
    path-verify a one-node tree from the new state: it equals the accepted node's output."""
    rng = np.random.default_rng(46)
    n, H, dk, dv = 24, 2, 64, 64
    S0, q, k, v, alpha, beta = inputs(rng, n, H, dk, dv)
    parent = tree(rng, n)
    O, _ = w12.gdn_path_verify(dev(S0), dev(q), dev(k), dev(v), dev(alpha), dev(beta), dev(parent))
    tok = np.arange(n, dtype=np.int32) + 100
    draft = np.zeros(n, np.int32)
    for i in range(1, n):
        draft[i] = tok[parent[i]] if rng.random() < 0.7 else 7
    path_len, path_nodes, _ = w12.tree_verify_tokens(dev(tok), dev(parent), dev(draft))
    L = int(path_len[0].item())
    assert L >= 1
    S = dev(S0.copy())
    assert int(w12.gdn_commit(S, dev(k), dev(v), dev(alpha), dev(beta), path_len, path_nodes).item()) == 0
    last = int(path_nodes[L].item())
    # a one-node tree from the committed state reads S q with the last accepted node's query
    O1, _ = w12.gdn_path_verify(S, dev(q[last:last + 1]), dev(k[:1]), dev(v[:1]), dev(alpha[:1]), dev(beta[:1]),
                                dev(np.int32([-1])))
    assert_close(O1.cpu().numpy()[0], O.cpu().numpy()[last].astype(np.float64))


@pytest.mark.parametrize("n,H,dk,dv,chain", [(1, 1, 64, 16, False), (5, 3, 64, 32, False), (32, 2, 128, 128, False),
                                             (64, 2, 128, 100, False), (17, 1, 128, 1, True), (40, 2, 64, 200, False)])
def test_wy_verify_matches_oracle(w12, n, H, dk, dv, chain):
    rng = np.random.default_rng(n * 11 + dv)
    S0, q, k, v, alpha, beta = inputs(rng, n, H, dk, dv)
    parent = tree(rng, n, chain)
    O, status = w12.gdn_wy_verify(dev(S0), dev(q), dev(k), dev(v), dev(alpha), dev(beta), dev(parent))
    assert int(status.item()) == 0
    assert_close(O.cpu().numpy(), oracle.gdn_tree(S0, q, k, v, alpha, beta, parent))


def test_wy_verify_full_size_and_agrees_with_path_verify(w12):
    rng = np.random.default_rng(47)
    n, H, dk, dv = 32, 32, 128, 128
    S0, q, k, v, alpha, beta = inputs(rng, n, H, dk, dv)
    parent = tree(rng, n)
    args = [dev(a) for a in (S0, q, k, v, alpha, beta, parent)]
    O1, s1 = w12.gdn_wy_verify(*args)
    O2, s2 = w12.gdn_path_verify(*args)
    assert int(s1.item()) == 0 and int(s2.item()) == 0
    ref = oracle.gdn_tree(S0, q, k, v, alpha, beta, parent)
    assert_close(O1.cpu().numpy(), ref)
    assert_close(O2.cpu().numpy(), ref)


def test_wy_verify_flags_invalid_trees(w12):
    rng = np.random.default_rng(48)
    S0, q, k, v, alpha, beta = inputs(rng, 4, 1, 64, 16)
    for bad in ([0, 0, 1, 2], [-1, 0, 2, 1], [-1, 0, 5, 1]):
        _, status = w12.gdn_wy_verify(dev(S0), dev(q), dev(k), dev(v), dev(alpha), dev(beta),
                                      dev(np.array(bad, np.int32)))
        assert int(status.item()) & 1
