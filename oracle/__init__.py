"""Plain CPU oracle for the W12 verify path (ctypes wrapper around w12_oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg (and its ``--impl reference`` arm) are the only
callers.  The CUDA library never imports or links this package.

Every function cites the passage it follows: the SpecPilot summary page
(onedev.kr/papers/1654), section "What's different" (무엇과 다른가), for the W12
format, the 8-bit Q-pass view and greedy tree acceptance.  The readings taken
where that passage is silent are listed at the top of ``w12_oracle.c``.

Multi-core helpers split rows over Python threads; ctypes releases the GIL
during each foreign call, so the threads run the plain C loops in parallel.
The arithmetic in each thread is unchanged.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD = os.path.join(HERE, "_build")
SO = os.path.join(BUILD, "libw12oracle.so")
# A test may point this at a deliberately broken build of w12_oracle.c to check
# that the pins catch the mistake.
OVERRIDE_ENV = "W12_ORACLE_SO"

_lock = threading.Lock()
_lib = None


def build() -> str:
    os.makedirs(BUILD, exist_ok=True)
    src = os.path.join(HERE, "w12_oracle.c")
    if not os.path.exists(SO) or os.path.getmtime(src) > os.path.getmtime(SO):
        tmp = SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
                               "-o", tmp, src, "-lm"])
        os.replace(tmp, SO)
    return SO


def _L():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(os.environ.get(OVERRIDE_ENV) or build())
            p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
            lib.w12o_base.argtypes = [p, i64]
            lib.w12o_base.restype = ctypes.c_int
            lib.w12o_encode.argtypes = [p, i64, i64, p, p, p, p, p, i64]
            lib.w12o_encode.restype = i64
            lib.w12o_decode.argtypes = [i64, i64, p, p, p, p, p, p]
            lib.w12o_decode.restype = None
            lib.w12o_decode_q8.argtypes = [i64, i64, p, p, p, p, p]
            lib.w12o_decode_q8.restype = None
            lib.w12o_gemm.argtypes = [p, i64, i64, p, i64, p, i64, p]
            lib.w12o_gemm.restype = None
            lib.w12o_argmax.argtypes = [p, i64, i64, p, p]
            lib.w12o_argmax.restype = None
            lib.w12o_accept.argtypes = [p, p, p, i32, p, p]
            lib.w12o_accept.restype = i32
            lib.w12o_tlv_splice.argtypes = [i32, p, i32, p, p, p, i32, p, p, p]
            lib.w12o_tlv_splice.restype = i32
            lib.w12o_budget_select.argtypes = [p, p, p, p, i32, i32, i32, p, p, p, p]
            lib.w12o_budget_select.restype = i32
            lib.w12o_i8_quantize.argtypes = [p, i64, i64, p, p, p]
            lib.w12o_i8_quantize.restype = None
            lib.w12o_cert_argmax.argtypes = [p, i64, i64, p, i64, p, p, p, p, p]
            lib.w12o_cert_argmax.restype = i64
            lib.w12o_split3.argtypes = [p, i64, p, p, p]
            lib.w12o_split3.restype = None
            lib.w12o_gdn_tree.argtypes = [p, p, p, p, p, p, p, i64, i64, i64, i64, p]
            lib.w12o_gdn_tree.restype = ctypes.c_int
            lib.w12o_gdn_commit.argtypes = [p, p, p, p, p, p, i64, i64, i64, i64, p]
            lib.w12o_gdn_commit.restype = None
            _lib = lib
        return _lib


def _p(a: np.ndarray | None) -> int | None:
    return None if a is None else a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


class Encoded:
    """Canonical W12 encoding of an N x K matrix (the layout the oracle defines)."""

    def __init__(self, N, K, hi, lo, base, rowptr, esc):
        self.N, self.K = N, K
        self.hi, self.lo, self.base, self.rowptr, self.esc = hi, lo, base, rowptr, esc

    @property
    def n_esc(self) -> int:
        return int(self.esc.size)

    def storage_bits(self) -> int:
        """Bits stored: 12 per weight, 32 per escape, 32 per rowptr entry, 8 per base."""
        return self.hi.size * 8 + (self.N * self.K) * 4 + self.esc.size * 32 + self.rowptr.size * 32 + self.base.size * 8


def base_of_row(row) -> int:
    """Window base of one channel (fullest 16-binade window, lowest base on ties)."""
    row = _c(row, np.uint16)
    return int(_L().w12o_base(_p(row), row.size))


def encode(W) -> Encoded:
    """Encode an N x K bf16 (uint16 bits) matrix into the canonical W12 planes."""
    W = _c(W, np.uint16)
    N, K = W.shape
    lib = _L()
    n_esc = int(lib.w12o_encode(_p(W), N, K, None, None, None, None, None, 0))
    hi = np.empty((N, K), np.uint8)
    lo = np.empty((N, (K + 1) // 2), np.uint8)
    base = np.empty(N, np.uint8)
    rowptr = np.empty(N + 1, np.uint32)
    esc = np.empty(max(n_esc, 1), np.uint32)
    got = int(lib.w12o_encode(_p(W), N, K, _p(hi), _p(lo), _p(base), _p(rowptr), _p(esc), n_esc))
    assert got == n_esc
    return Encoded(N, K, hi, lo, base, rowptr, esc[:n_esc].copy())


def decode(enc: Encoded) -> np.ndarray:
    out = np.empty((enc.N, enc.K), np.uint16)
    esc = enc.esc if enc.esc.size else np.zeros(1, np.uint32)
    _L().w12o_decode(enc.N, enc.K, _p(enc.hi), _p(enc.lo), _p(enc.base), _p(enc.rowptr), _p(esc), _p(out))
    return out


def decode_q8(enc: Encoded) -> np.ndarray:
    out = np.empty((enc.N, enc.K), np.uint16)
    esc = enc.esc if enc.esc.size else np.zeros(1, np.uint32)
    _L().w12o_decode_q8(enc.N, enc.K, _p(enc.hi), _p(enc.base), _p(enc.rowptr), _p(esc), _p(out))
    return out


def gemm(x, W, threads: int | None = None, with_bound: bool = True):
    """fp64 y[M,N] = x[M,K] . W[N,K]^T (k increasing) and B = sum |x*w|.

    W holds bf16 bits of the decoded weights.  Rows of W are split over threads."""
    x = _c(x, np.uint16)
    W = _c(W, np.uint16)
    M, K = x.shape
    N = W.shape[0]
    y = np.empty((M, N), np.float64)
    B = np.empty((M, N), np.float64) if with_bound else None
    lib = _L()
    nt = max(1, min(threads or (os.cpu_count() or 1), N))
    bounds = [(N * i) // nt for i in range(nt + 1)]

    def run(i):
        a, b = bounds[i], bounds[i + 1]
        if b > a:
            lib.w12o_gemm(_p(x), M, K, W.ctypes.data + a * K * 2, b - a, y.ctypes.data + a * 8, N,
                          None if B is None else B.ctypes.data + a * 8)

    if nt == 1:
        run(0)
    else:
        with ThreadPoolExecutor(nt) as ex:
            list(ex.map(run, range(nt)))
    return (y, B) if with_bound else y


def argmax(logits):
    """Row argmax (lowest index on ties, NaN below all) and the top-1 minus top-2 gap."""
    logits = _c(logits, np.float64)
    M, V = logits.shape
    idx = np.empty(M, np.int32)
    gap = np.empty(M, np.float64)
    _L().w12o_argmax(_p(logits), M, V, _p(idx), _p(gap))
    return idx, gap


def accept(tok, parent, draft):
    """Greedy acceptance on one tree: (L, path nodes root..a*, bonus); L = -1 if invalid."""
    tok = _c(tok, np.int32)
    parent = _c(parent, np.int32)
    draft = _c(draft, np.int32)
    n = parent.size
    path = np.full(max(n, 1), -1, np.int32)
    bonus = np.zeros(1, np.int32)
    L = int(_L().w12o_accept(_p(tok), _p(parent), _p(draft), n, _p(path), _p(bonus)))
    if L < 0:
        return -1, np.zeros(0, np.int32), -1
    return L, path[: L + 1].copy(), int(bonus[0])


def accept_batched(tok, parent, draft, offsets):
    """Acceptance for several trees concatenated; offsets[r]..offsets[r+1] is request r."""
    res = []
    for r in range(len(offsets) - 1):
        a, b = int(offsets[r]), int(offsets[r + 1])
        res.append(accept(tok[a:b], parent[a:b], draft[a:b]))
    return res


def tlv_splice(L, path, bonus, draft_q, sub_parent, sub_draft, n):
    """The two-level-verification splice: the Q pass's accepted path (L, path, bonus)
    on a tree with drafts draft_q, plus a subtree (sub_parent relative, -1 = under the
    bonus node) cut to fill n nodes.  Returns (parent, draft, src) of the n-node tree,
    src[i] = Q-pass row reused by node i, or -1 - r for new row r; None if invalid."""
    path = _c(np.asarray(path if L >= 0 else [0]), np.int32)
    draft_q = _c(draft_q, np.int32)
    sub_parent = _c(np.asarray(sub_parent) if len(sub_parent) else np.zeros(1), np.int32)
    sub_draft = _c(np.asarray(sub_draft) if len(sub_draft) else np.zeros(1), np.int32)
    parent = np.empty(max(n, 1), np.int32)
    draft = np.empty(max(n, 1), np.int32)
    src = np.empty(max(n, 1), np.int32)
    rc = int(_L().w12o_tlv_splice(int(L), _p(path), int(bonus), _p(draft_q), _p(sub_parent), _p(sub_draft), int(n),
                                  _p(parent), _p(draft), _p(src)))
    if rc != 0:
        return None
    return parent[:n].copy(), draft[:n].copy(), src[:n].copy()


def budget_select(parent, conf, draft, offsets, budget, per_request=False):
    """Node budget over several candidate trees (parent relative to its request, conf a
    float32 confidence per node): keeps the top `budget` nodes by path score (over all
    requests, or per request).  Returns (parent, draft, src, offsets) of the kept trees,
    or None for an invalid candidate tree."""
    parent = _c(parent, np.int32)
    conf = _c(conf, np.float32)
    draft = _c(draft, np.int32)
    offsets = _c(offsets, np.int32)
    n_req = offsets.size - 1
    C = int(offsets[-1])
    po = np.empty(max(C, 1), np.int32)
    do = np.empty(max(C, 1), np.int32)
    so = np.empty(max(C, 1), np.int32)
    oo = np.empty(n_req + 1, np.int32)
    k = int(_L().w12o_budget_select(_p(parent), _p(conf), _p(draft), _p(offsets), n_req, int(budget), int(per_request),
                                    _p(po), _p(do), _p(so), _p(oo)))
    if k < 0:
        return None
    return po[:k].copy(), do[:k].copy(), so[:k].copy(), oo.copy()


def i8_quantize(W, threads: int | None = None):
    """INT8 head of the certified LM-head argmax (same page and section: on H100 the LM
    head stays in INT8 and a Cauchy-Schwarz bound filters candidates that are then
    computed exactly).  W holds bf16 bits [N, K].  Returns code [N, K] (sign<<7 | |q|),
    scale [N] float32 and cbound [N] float32 (the bound's per-channel factor)."""
    W = _c(W, np.uint16)
    N, K = W.shape
    code = np.empty((N, K), np.uint8)
    scale = np.empty(N, np.float32)
    cbound = np.empty(N, np.float32)
    lib = _L()
    nt = max(1, min(threads or (os.cpu_count() or 1), N))
    bounds = [(N * i) // nt for i in range(nt + 1)]

    def run(i):
        a, b = bounds[i], bounds[i + 1]
        if b > a:
            lib.w12o_i8_quantize(W.ctypes.data + a * K * 2, b - a, K, code.ctypes.data + a * K,
                                 scale.ctypes.data + a * 4, cbound.ctypes.data + a * 4)

    if nt == 1:
        run(0)
    else:
        with ThreadPoolExecutor(nt) as ex:
            list(ex.map(run, range(nt)))
    return code, scale, cbound


def cert_argmax(x, W, code, scale, cbound, threads: int | None = None):
    """Argmax of the exact logits x . W^T for each row of x, through the certified
    candidates of the INT8 head (code, scale, cbound from i8_quantize).  Returns
    (idx [M] int32, ncand [M] int32).  Rows of x are split over threads."""
    x = _c(x, np.uint16)
    W = _c(W, np.uint16)
    code = _c(code, np.uint8)
    scale = _c(scale, np.float32)
    cbound = _c(cbound, np.float32)
    M, K = x.shape
    V = W.shape[0]
    idx = np.empty(M, np.int32)
    ncand = np.empty(M, np.int32)
    lib = _L()
    nt = max(1, min(threads or (os.cpu_count() or 1), M))
    bounds = [(M * i) // nt for i in range(nt + 1)]

    def run(i):
        a, b = bounds[i], bounds[i + 1]
        if b > a:
            lib.w12o_cert_argmax(x.ctypes.data + a * K * 2, b - a, K, _p(W), V, _p(code), _p(scale), _p(cbound),
                                 idx.ctypes.data + a * 4, ncand.ctypes.data + a * 4)

    if nt == 1:
        run(0)
    else:
        with ThreadPoolExecutor(nt) as ex:
            list(ex.map(run, range(nt)))
    return idx, ncand


def split3(x):
    """Three bf16 pieces of each float (same page and section: the WY kernel holds the
    FP32 state's 24-bit significand exactly in three BF16 pieces).  Returns bf16 bits
    (s1, s2, s3), each the shape of x."""
    x = _c(x, np.float32)
    s1, s2, s3 = (np.empty(x.shape, np.uint16) for _ in range(3))
    _L().w12o_split3(_p(x), x.size, _p(s1), _p(s2), _p(s3))
    return s1, s2, s3


def gdn_tree(S0, q, k, v, alpha, beta, parent):
    """Gated-delta-rule outputs of every node of a draft tree (same page and section:
    the path-verify kernel recomputes the recurrent state along each path).
    S0 [H, dv, dk] float32; q, k [n, H, dk], v [n, H, dv] bf16 bits; alpha, beta [n, H]
    float32; parent [n].  Returns O [n, H, dv] fp64, or None for an invalid tree."""
    S0 = _c(S0, np.float32)
    q, k, v = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    alpha, beta, parent = _c(alpha, np.float32), _c(beta, np.float32), _c(parent, np.int32)
    H, dv, dk = S0.shape
    n = parent.size
    O = np.empty((n, H, dv), np.float64)
    rc = _L().w12o_gdn_tree(_p(S0), _p(q), _p(k), _p(v), _p(alpha), _p(beta), _p(parent), n, H, dk, dv, _p(O))
    return None if rc != 0 else O


def gdn_commit(S0, k, v, alpha, beta, nodes):
    """State after replaying the accepted nodes (path order, root excluded) into S0
    (same page and section: the commit kernel).  Returns S [H, dv, dk] fp64."""
    S0 = _c(S0, np.float32)
    k, v = _c(k, np.uint16), _c(v, np.uint16)
    alpha, beta = _c(alpha, np.float32), _c(beta, np.float32)
    L = len(nodes)
    nodes = _c(np.asarray(nodes if L else [0]), np.int32)
    H, dv, dk = S0.shape
    S = np.empty((H, dv, dk), np.float64)
    _L().w12o_gdn_commit(_p(S0), _p(k), _p(v), _p(alpha), _p(beta), _p(nodes), L, H, dk, dv, _p(S))
    return S
