"""Python binding of libw12 (the W12 verify-path C ABI in include/w12.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch supplies device memory and streams.  There is no CPU
fallback: if libw12.so cannot be built or loaded, every call raises.

The names mirror the C functions: ``w12_encode_plan``/``w12_encode`` (wrapped
together by :func:`encode`), :func:`w12_decode`, :func:`w12_decode_q8`,
:func:`w12_gemm`, :func:`w12_gemm_q8`, :func:`w12_lmhead_argmax`,
:func:`w12_lmhead_verify`, :func:`tree_verify_tokens`, :func:`tree_verify` and
:func:`w12_export_canonical`.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

_lock = threading.Lock()
_lib = None

W12_OK = 0
STATUS_NAMES = {0: "W12_OK", 1: "W12_ERR_INVALID_ARG", 2: "W12_ERR_SHAPE", 3: "W12_ERR_BUFFER_TOO_SMALL",
                4: "W12_ERR_CUDA", 5: "W12_ERR_BOUNDS", 6: "W12_ERR_TIMEOUT"}


class W12Error(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class w12_matrix(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int64), ("K", ctypes.c_int64), ("hi", ctypes.c_void_p), ("lo", ctypes.c_void_p),
                ("base", ctypes.c_void_p), ("esc_tile_ptr", ctypes.c_void_p), ("esc", ctypes.c_void_p),
                ("n_esc", ctypes.c_int64)]


class w12_i8_head(ctypes.Structure):
    _fields_ = [("V", ctypes.c_int64), ("K", ctypes.c_int64), ("code", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("cbound", ctypes.c_void_p)]


# (name, restype, argtypes) of every exported symbol, in include/w12.h order.
_P, _I64, _I32, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
_MP = ctypes.POINTER(w12_matrix)
SIGNATURES = [
    ("w12_last_error", ctypes.c_char_p, []),
    ("w12_status_string", ctypes.c_char_p, [ctypes.c_int]),
    ("w12_abi_version", ctypes.c_int, []),
    ("w12_hi_bytes", _I64, [_I64, _I64]),
    ("w12_lo_bytes", _I64, [_I64, _I64]),
    ("w12_tile_count", _I64, [_I64, _I64]),
    ("w12_encode_plan", ctypes.c_int, [_P, _I64, _I64, _P, _P, ctypes.POINTER(_I64), _P]),
    ("w12_encode", ctypes.c_int, [_P, _MP, _P]),
    ("w12_decode", ctypes.c_int, [_MP, _P, _P]),
    ("w12_decode_q8", ctypes.c_int, [_MP, _P, _P]),
    ("w12_export_canonical", ctypes.c_int, [_MP, _P, _P, _P, _P, _P]),
    ("w12_save", ctypes.c_int, [_MP, ctypes.c_char_p, _P]),
    ("w12_load_info", ctypes.c_int, [ctypes.c_char_p, ctypes.POINTER(_I64), ctypes.POINTER(_I64),
                                     ctypes.POINTER(_I64)]),
    ("w12_load", ctypes.c_int, [ctypes.c_char_p, _MP, _P]),
    ("w12_gemm_workspace_size", _SZ, [_I64, _I64, _I64]),
    ("w12_gemm_counter_bytes", _SZ, [_I64]),
    ("w12_gemm", ctypes.c_int, [_P, _I64, _MP, _P, _P, _SZ, _P]),
    ("w12_gemm_q8", ctypes.c_int, [_P, _I64, _MP, _P, _P, _SZ, _P]),
    ("w12_workspace_status", ctypes.c_int, [_P, _SZ, ctypes.POINTER(_I32), _P]),
    ("w12_set_wait_limit", ctypes.c_int, [_I64]),
    ("w12_validate", ctypes.c_int, [_MP, _P, _P]),
    ("w12_gemm_noalloc_max_scratch", _SZ, []),
    ("w12_gemm_noalloc", ctypes.c_int, [_P, _I64, _MP, _P, _P]),
    ("w12_lmhead_workspace_size", _SZ, [_I64, _I64, _I64]),
    ("w12_lmhead_argmax", ctypes.c_int, [_P, _I64, _MP, _P, _P, _SZ, _P]),
    ("w12_lmhead_argmax_q8", ctypes.c_int, [_P, _I64, _MP, _P, _P, _SZ, _P]),
    ("w12_lmhead_verify", ctypes.c_int, [_P, _I64, _MP, ctypes.c_int, _P, _P, _P, _I32, _P, _P, _P, _P, _P, _SZ, _P]),
    ("tree_verify_tokens", ctypes.c_int, [_P, _P, _P, _P, _I32, _I64, _P, _P, _P, _P]),
    ("tree_verify_workspace_size", _SZ, [_I64]),
    ("tree_verify", ctypes.c_int, [_P, _I64, _I64, _P, _P, _P, _I32, _P, _P, _P, _P, _SZ, _P]),
    ("tlv_splice", ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _P, _P, _P, _I64, _I64, _P, _P, _P, _P, _P]),
    ("tree_budget_select", ctypes.c_int, [_P, _P, _P, _P, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P]),
    ("gather_rows", ctypes.c_int, [_P, _I64, _P, _I64, _I64, _P, _P]),
    ("w12_i8_code_bytes", _I64, [_I64, _I64]),
    ("w12_i8_encode", ctypes.c_int, [_P, ctypes.POINTER(w12_i8_head), _P]),
    ("w12_cert_head_workspace_size", _SZ, [_I64, _I64, _I64]),
    ("w12_cert_head_argmax", ctypes.c_int, [_P, _I64, ctypes.POINTER(w12_i8_head), _MP, _P, _P, _P, _SZ, _P]),
    ("gdn_split3", ctypes.c_int, [_P, _I64, _P, _P, _P, _P]),
    ("gdn_path_verify", ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _P, _P, _P]),
    ("gdn_wy_verify", ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _P, _P, _P]),
    ("gdn_commit", ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _P, _P]),
]


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load (building first if the sources changed) libw12.so.  Raises on failure."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"libw12.so missing at {path}")
            L = ctypes.CDLL(path)
            for name, res, args in SIGNATURES:
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
        return _lib


def _check(status: int) -> None:
    if status != W12_OK:
        raise W12Error(status, lib().w12_last_error().decode(errors="replace"))


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _bits16(t: torch.Tensor) -> torch.Tensor:
    if t.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError(f"expected bf16 bits (bfloat16/int16/uint16), got {t.dtype}")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("expected a contiguous CUDA tensor")
    return t


def _i32(t: torch.Tensor) -> torch.Tensor:
    if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
        raise ValueError("expected a contiguous int32 CUDA tensor")
    return t


class W12Matrix:
    """Device buffers of one W12-encoded matrix (layout of include/w12.h)."""

    def __init__(self, N, K, hi, lo, base, esc_tile_ptr, esc, n_esc):
        self.N, self.K = int(N), int(K)
        self.hi, self.lo, self.base, self.esc_tile_ptr, self.esc = hi, lo, base, esc_tile_ptr, esc
        self.n_esc = int(n_esc)
        self._desc = w12_matrix(self.N, self.K, _ptr(hi), _ptr(lo), _ptr(base), _ptr(esc_tile_ptr),
                                _ptr(esc) if self.n_esc else None, self.n_esc)

    def desc(self):
        return ctypes.byref(self._desc)

    @property
    def device(self):
        return self.hi.device

    def stored_bytes(self) -> int:
        """Bytes this matrix occupies on the device (planes, bases, escape index and escapes)."""
        return (self.hi.numel() + self.lo.numel() + self.base.numel() + 4 * self.esc_tile_ptr.numel()
                + 4 * self.n_esc)

    def stream_bytes(self, q8: bool = False) -> int:
        """Bytes one GEMM pass must read: records (1.5 or 1 B/weight on the tiled planes),
        escapes (4 B each), the escape index and the bases."""
        rec = self.hi.numel() + (0 if q8 else self.lo.numel())
        return rec + 4 * self.n_esc + 4 * self.esc_tile_ptr.numel() + self.base.numel()


def esc_alloc_entries(n_esc: int) -> int:
    """Entries to allocate for an escape list: a multiple of 4 (the GEMM stages
    escapes in 16-byte runs), at least 4."""
    return max(4, (n_esc + 3) // 4 * 4)


def tile_count(N: int, K: int) -> int:
    return int(lib().w12_tile_count(N, K))


def encode(W: torch.Tensor, stream=None) -> W12Matrix:
    """w12_encode_plan + w12_encode of an N x K bf16 matrix (synchronises the stream once)."""
    W = _bits16(W)
    N, K = W.shape
    L = lib()
    dev = W.device
    T = int(L.w12_tile_count(N, K))
    if T < 0:
        raise W12Error(2, f"shape {N}x{K} out of range")
    base = torch.empty(N, dtype=torch.uint8, device=dev)
    tp = torch.empty(T + 1, dtype=torch.int32, device=dev)
    n_esc = ctypes.c_int64(0)
    s = _stream(stream)
    _check(L.w12_encode_plan(_ptr(W), N, K, _ptr(base), _ptr(tp), ctypes.byref(n_esc), s))
    hi = torch.empty(int(L.w12_hi_bytes(N, K)), dtype=torch.uint8, device=dev)
    lo = torch.empty(int(L.w12_lo_bytes(N, K)), dtype=torch.uint8, device=dev)
    esc = torch.empty(esc_alloc_entries(int(n_esc.value)), dtype=torch.int32, device=dev)
    A = W12Matrix(N, K, hi, lo, base, tp, esc, n_esc.value)
    _check(L.w12_encode(_ptr(W), A.desc(), s))
    return A


def w12_save(A: W12Matrix, path: str, stream=None) -> None:
    """Writes the encoded matrix to a file (w12_save)."""
    _check(lib().w12_save(A.desc(), os.fsencode(path), _stream(stream)))


def w12_load(path: str, device=None, stream=None) -> W12Matrix:
    """A matrix that w12_save wrote, in new device buffers (w12_load_info, then w12_load)."""
    L = lib()
    N, K, n_esc = ctypes.c_int64(0), ctypes.c_int64(0), ctypes.c_int64(0)
    _check(L.w12_load_info(os.fsencode(path), ctypes.byref(N), ctypes.byref(K), ctypes.byref(n_esc)))
    N, K, n_esc = N.value, K.value, n_esc.value
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    hi = torch.empty(int(L.w12_hi_bytes(N, K)), dtype=torch.uint8, device=dev)
    lo = torch.empty(int(L.w12_lo_bytes(N, K)), dtype=torch.uint8, device=dev)
    base = torch.empty(N, dtype=torch.uint8, device=dev)
    tp = torch.empty(int(L.w12_tile_count(N, K)) + 1, dtype=torch.int32, device=dev)
    esc = torch.empty(esc_alloc_entries(n_esc), dtype=torch.int32, device=dev)
    A = W12Matrix(N, K, hi, lo, base, tp, esc, n_esc)
    _check(L.w12_load(os.fsencode(path), A.desc(), _stream(stream)))
    return A


def w12_decode(A: W12Matrix, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    out = torch.empty((A.N, A.K), dtype=torch.bfloat16, device=A.device) if out is None else _bits16(out)
    _check(lib().w12_decode(A.desc(), _ptr(out), _stream(stream)))
    return out


def w12_decode_q8(A: W12Matrix, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    out = torch.empty((A.N, A.K), dtype=torch.bfloat16, device=A.device) if out is None else _bits16(out)
    _check(lib().w12_decode_q8(A.desc(), _ptr(out), _stream(stream)))
    return out


def w12_export_canonical(A: W12Matrix, stream=None) -> dict:
    """Canonical planes: hi [N,K] u8, lo [N,ceil(K/2)] u8, rowptr [N+1] i32, esc [n_esc] i32."""
    dev = A.device
    hi = torch.empty((A.N, A.K), dtype=torch.uint8, device=dev)
    lo = torch.empty((A.N, (A.K + 1) // 2), dtype=torch.uint8, device=dev)
    rowptr = torch.empty(A.N + 1, dtype=torch.int32, device=dev)
    esc = torch.empty(max(A.n_esc, 1), dtype=torch.int32, device=dev)
    _check(lib().w12_export_canonical(A.desc(), _ptr(hi), _ptr(lo), _ptr(rowptr), _ptr(esc), _stream(stream)))
    return dict(hi=hi, lo=lo, rowptr=rowptr, esc=esc[: A.n_esc], base=A.base)


class Workspace:
    """A zero-initialised device workspace that grows on demand (counters start at zero)."""

    def __init__(self, device=None):
        self.device = device or torch.device("cuda")
        self.buf = torch.zeros(256, dtype=torch.uint8, device=self.device)

    def get(self, nbytes: int) -> torch.Tensor:
        if nbytes > self.buf.numel():
            self.buf = torch.zeros(int(nbytes), dtype=torch.uint8, device=self.device)
        return self.buf

    def status(self, stream=None) -> int:
        """w12_workspace_status: W12_OK, W12_ERR_TIMEOUT or W12_ERR_BOUNDS for the calls made
        on this workspace since the last query (synchronises the stream; clears the
        workspace after an error)."""
        st = ctypes.c_int32(-1)
        _check(lib().w12_workspace_status(_ptr(self.buf), self.buf.numel(), ctypes.byref(st), _stream(stream)))
        return int(st.value)

    def check(self, stream=None) -> None:
        """Raises W12Error if a GEMM call on this workspace met a device error."""
        st = self.status(stream)
        if st != W12_OK:
            raise W12Error(st, "a GEMM kernel reported a device error on this workspace")


def w12_set_wait_limit(cycles: int) -> None:
    """Diagnostic: bound of the GEMM kernels' waits for another warp (0 = default)."""
    _check(lib().w12_set_wait_limit(int(cycles)))


def w12_validate(A: "W12Matrix", status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Checks A's escape index and window bases on the device; returns a device int32
    tensor holding W12_OK or W12_ERR_BOUNDS."""
    status = torch.empty(1, dtype=torch.int32, device=A.device) if status is None else _i32(status)
    _check(lib().w12_validate(A.desc(), _ptr(status), _stream(stream)))
    return status


def gemm_workspace_size(M: int, N: int, K: int) -> int:
    return int(lib().w12_gemm_workspace_size(M, N, K))


def lmhead_workspace_size(M: int, V: int, K: int) -> int:
    return int(lib().w12_lmhead_workspace_size(M, V, K))


def _gemm(fn, x, A, y, ws, stream):
    x = _bits16(x)
    M = x.shape[0]
    if x.shape[1] != A.K:
        raise ValueError(f"x has {x.shape[1]} columns, matrix has K={A.K}")
    y = torch.empty((M, A.N), dtype=torch.float32, device=x.device) if y is None else y
    ws = ws or Workspace(x.device)
    need = gemm_workspace_size(M, A.N, A.K)
    buf = ws.get(need)
    _check(fn(_ptr(x), M, A.desc(), _ptr(y), _ptr(buf), buf.numel(), _stream(stream)))
    return y


def w12_gemm(x: torch.Tensor, A: W12Matrix, y: torch.Tensor | None = None, ws: Workspace | None = None,
             stream=None) -> torch.Tensor:
    """y[M,N] fp32 = x[M,K] bf16 . decode(A)^T."""
    return _gemm(lib().w12_gemm, x, A, y, ws, stream)


def w12_gemm_q8(x: torch.Tensor, A: W12Matrix, y: torch.Tensor | None = None, ws: Workspace | None = None,
                stream=None) -> torch.Tensor:
    """Same with the 8-bit view of the weights (Q pass)."""
    return _gemm(lib().w12_gemm_q8, x, A, y, ws, stream)


def w12_gemm_noalloc(x: torch.Tensor, A: W12Matrix, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """w12_gemm using the library's own fixed scratch instead of a workspace (see include/w12.h)."""
    x = _bits16(x)
    M = x.shape[0]
    y = torch.empty((M, A.N), dtype=torch.float32, device=x.device) if y is None else y
    _check(lib().w12_gemm_noalloc(_ptr(x), M, A.desc(), _ptr(y), _stream(stream)))
    return y


def w12_lmhead_argmax(x: torch.Tensor, head: W12Matrix, q8: bool = False, tok: torch.Tensor | None = None,
                      ws: Workspace | None = None, stream=None) -> torch.Tensor:
    x = _bits16(x)
    M = x.shape[0]
    tok = torch.empty(M, dtype=torch.int32, device=x.device) if tok is None else tok
    ws = ws or Workspace(x.device)
    buf = ws.get(lmhead_workspace_size(M, head.N, head.K))
    fn = lib().w12_lmhead_argmax_q8 if q8 else lib().w12_lmhead_argmax
    _check(fn(_ptr(x), M, head.desc(), _ptr(tok), _ptr(buf), buf.numel(), _stream(stream)))
    return tok


def _tree_out(M, n_req, device):
    return (torch.empty(n_req, dtype=torch.int32, device=device), torch.empty(M, dtype=torch.int32, device=device),
            torch.empty(n_req, dtype=torch.int32, device=device))


def w12_lmhead_verify(x, head: W12Matrix, parent, draft, req_offsets=None, q8: bool = False,
                      ws: Workspace | None = None, stream=None):
    """LM-head argmax + acceptance: returns (tok, path_len, path_nodes, bonus)."""
    x = _bits16(x)
    M = x.shape[0]
    n_req = 1 if req_offsets is None else req_offsets.numel() - 1
    tok = torch.empty(M, dtype=torch.int32, device=x.device)
    path_len, path_nodes, bonus = _tree_out(M, n_req, x.device)
    ws = ws or Workspace(x.device)
    buf = ws.get(lmhead_workspace_size(M, head.N, head.K))
    _check(lib().w12_lmhead_verify(_ptr(x), M, head.desc(), int(q8), _ptr(_i32(parent)), _ptr(_i32(draft)),
                                   _ptr(req_offsets), n_req, _ptr(tok), _ptr(path_len), _ptr(path_nodes),
                                   _ptr(bonus), _ptr(buf), buf.numel(), _stream(stream)))
    return tok, path_len, path_nodes, bonus


def tree_verify_tokens(tok, parent, draft, req_offsets=None, stream=None):
    """Greedy acceptance from target tokens: returns (path_len, path_nodes, bonus)."""
    M = tok.numel()
    n_req = 1 if req_offsets is None else req_offsets.numel() - 1
    path_len, path_nodes, bonus = _tree_out(M, n_req, tok.device)
    _check(lib().tree_verify_tokens(_ptr(_i32(tok)), _ptr(_i32(parent)), _ptr(_i32(draft)),
                                    _ptr(None if req_offsets is None else _i32(req_offsets)), n_req, M,
                                    _ptr(path_len), _ptr(path_nodes), _ptr(bonus), _stream(stream)))
    return path_len, path_nodes, bonus


def tree_verify(logits, parent, draft, req_offsets=None, stream=None):
    """Greedy acceptance from fp32 logits [M, V]: returns (path_len, path_nodes, bonus)."""
    if logits.dtype != torch.float32 or not logits.is_cuda or not logits.is_contiguous():
        raise ValueError("logits must be a contiguous float32 CUDA tensor")
    M, V = logits.shape
    n_req = 1 if req_offsets is None else req_offsets.numel() - 1
    path_len, path_nodes, bonus = _tree_out(M, n_req, logits.device)
    ws = torch.empty(int(lib().tree_verify_workspace_size(M)), dtype=torch.uint8, device=logits.device)
    _check(lib().tree_verify(_ptr(logits), M, V, _ptr(_i32(parent)), _ptr(_i32(draft)),
                             _ptr(None if req_offsets is None else _i32(req_offsets)), n_req, _ptr(path_len),
                             _ptr(path_nodes), _ptr(bonus), _ptr(ws), ws.numel(), _stream(stream)))
    return path_len, path_nodes, bonus


def tlv_splice(path_len, path_nodes, bonus, draft_q, x_q, sub_parent, sub_draft, x_sub, n: int, stream=None):
    """Two-level-verification splice: the Q pass's accepted path (path_len, path_nodes,
    bonus of one request, as tree_verify returns them) on a tree with drafts draft_q and
    activation rows x_q [n_q, K], plus a subtree (sub_parent relative, -1 = under the bonus
    node; sub_draft) with rows x_sub [n-1, K] (row 0 for the bonus node).  Returns
    (parent, draft, src, x) of the n-node tree for the exact pass."""
    x_q, x_sub = _bits16(x_q), _bits16(x_sub)
    n_q, K = x_q.shape
    if x_sub.shape != (n - 1, K):
        raise ValueError(f"x_sub must be [{n - 1}, {K}]")
    dev = x_q.device
    parent = torch.empty(n, dtype=torch.int32, device=dev)
    draft = torch.empty(n, dtype=torch.int32, device=dev)
    src = torch.empty(n, dtype=torch.int32, device=dev)
    x = torch.empty((n, K), dtype=x_q.dtype, device=dev)
    sp = _i32(sub_parent) if n > 2 else None
    sd = _i32(sub_draft) if n > 2 else None
    _check(lib().tlv_splice(_ptr(_i32(path_len)), _ptr(_i32(path_nodes)), _ptr(_i32(bonus)), _ptr(_i32(draft_q)),
                            _ptr(x_q), n_q, _ptr(sp), _ptr(sd), _ptr(x_sub), n, K, _ptr(parent), _ptr(draft),
                            _ptr(src), _ptr(x), _stream(stream)))
    return parent, draft, src, x


def tree_budget_select(parent, conf, draft, req_offsets, budget: int, per_request: bool = False, stream=None):
    """Node budget over candidate trees (see include/w12.h): returns (parent, draft, src,
    offsets, n_kept) as device tensors; the first n_kept entries of parent/draft/src are
    the kept trees (n_kept = -1 for an invalid candidate tree)."""
    if conf.dtype != torch.float32 or not conf.is_cuda or not conf.is_contiguous():
        raise ValueError("conf must be a contiguous float32 CUDA tensor")
    C = conf.numel()
    n_req = req_offsets.numel() - 1
    dev = conf.device
    po = torch.empty(C, dtype=torch.int32, device=dev)
    do = torch.empty(C, dtype=torch.int32, device=dev)
    so = torch.empty(C, dtype=torch.int32, device=dev)
    oo = torch.empty(n_req + 1, dtype=torch.int32, device=dev)
    nk = torch.empty(1, dtype=torch.int32, device=dev)
    _check(lib().tree_budget_select(_ptr(_i32(parent)), _ptr(conf), _ptr(_i32(draft)), _ptr(_i32(req_offsets)), n_req,
                                    C, int(budget), int(per_request), _ptr(po), _ptr(do), _ptr(so), _ptr(oo), _ptr(nk),
                                    _stream(stream)))
    return po, do, so, oo, nk


def gather_rows(x, src, n: int | None = None, stream=None):
    """out[i] = x[src[i]] (zero rows for indices outside x) for the first n entries of src."""
    x = _bits16(x)
    n_src, K = x.shape
    n = src.numel() if n is None else n
    out = torch.empty((n, K), dtype=x.dtype, device=x.device)
    _check(lib().gather_rows(_ptr(x), n_src, _ptr(_i32(src)), n, K, _ptr(out), _stream(stream)))
    return out


# ---------------------------------------------------------------- certified INT8 head

class I8Head:
    """Device buffers of an INT8 head (include/w12.h, w12_i8_head): codes in the W12
    hi-plane layout, per-channel scale and bound factor."""

    def __init__(self, V, K, code, scale, cbound):
        self.V, self.K = int(V), int(K)
        self.code, self.scale, self.cbound = code, scale, cbound
        self._desc = w12_i8_head(self.V, self.K, _ptr(code), _ptr(scale), _ptr(cbound))

    def desc(self):
        return ctypes.byref(self._desc)

    def stream_bytes(self) -> int:
        """Bytes the approximate-logit GEMM reads: one code byte per (padded) weight and the scales."""
        return self.code.numel() + 4 * self.V


def i8_encode(W: torch.Tensor, stream=None) -> I8Head:
    """INT8 head of a V x K bf16 head (certified argmax: SpecPilot page, "What's different")."""
    W = _bits16(W)
    V, K = W.shape
    L = lib()
    dev = W.device
    code = torch.empty(int(L.w12_i8_code_bytes(V, K)), dtype=torch.uint8, device=dev)
    scale = torch.empty(V, dtype=torch.float32, device=dev)
    cbound = torch.empty(V, dtype=torch.float32, device=dev)
    H = I8Head(V, K, code, scale, cbound)
    _check(L.w12_i8_encode(_ptr(W), H.desc(), _stream(stream)))
    return H


def cert_head_workspace_size(M: int, V: int, K: int) -> int:
    return int(lib().w12_cert_head_workspace_size(M, V, K))


def w12_cert_head_argmax(x: torch.Tensor, H: I8Head, exact: W12Matrix, tok: torch.Tensor | None = None,
                         ncand: torch.Tensor | None = None, ws: Workspace | None = None, stream=None):
    """Exact-logit argmax of x . W^T through the INT8 head's certified candidates; the
    exact logits of the candidates come from `exact` (the W12 form of the same head).
    Returns (tok [M] int32, ncand [M] int32)."""
    x = _bits16(x)
    M = x.shape[0]
    if x.shape[1] != H.K:
        raise ValueError(f"x has {x.shape[1]} columns, head has K={H.K}")
    tok = torch.empty(M, dtype=torch.int32, device=x.device) if tok is None else _i32(tok)
    ncand = torch.empty(M, dtype=torch.int32, device=x.device) if ncand is None else _i32(ncand)
    ws = ws or Workspace(x.device)
    buf = ws.get(cert_head_workspace_size(M, H.V, H.K))
    _check(lib().w12_cert_head_argmax(_ptr(x), M, H.desc(), exact.desc(), _ptr(tok), _ptr(ncand), _ptr(buf),
                                      buf.numel(), _stream(stream)))
    return tok, ncand


# ---------------------------------------------------------------- recurrent layers (gated delta rule)

def _f32(t: torch.Tensor) -> torch.Tensor:
    if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
        raise ValueError("expected a contiguous float32 CUDA tensor")
    return t


def gdn_split3(x: torch.Tensor, stream=None):
    """Three bf16 pieces (bits as int16) of each float of x: s1 + s2 + s3 == x."""
    x = _f32(x)
    s = [torch.empty(x.shape, dtype=torch.int16, device=x.device) for _ in range(3)]
    _check(lib().gdn_split3(_ptr(x), x.numel(), _ptr(s[0]), _ptr(s[1]), _ptr(s[2]), _stream(stream)))
    return tuple(s)


def gdn_path_verify(S0, q, k, v, alpha, beta, parent, O=None, status=None, stream=None):
    """Outputs O [n, H, dv] of every node of a draft tree under the gated delta rule
    (state recomputed along each path).  S0 [H, dv, dk] float32; q, k [n, H, dk], v [n, H, dv]
    bf16 bits; alpha, beta [n, H] float32; parent [n] int32.  Returns (O, status)."""
    S0, alpha, beta = _f32(S0), _f32(alpha), _f32(beta)
    q, k, v, parent = _bits16(q), _bits16(k), _bits16(v), _i32(parent)
    H, dv, dk = S0.shape
    n = parent.numel()
    O = torch.empty((n, H, dv), dtype=torch.float32, device=S0.device) if O is None else _f32(O)
    status = torch.zeros(1, dtype=torch.int32, device=S0.device) if status is None else _i32(status)
    _check(lib().gdn_path_verify(_ptr(S0), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(parent), n, H, dk,
                                 dv, _ptr(O), _ptr(status), _stream(stream)))
    return O, status


def gdn_wy_verify(S0, q, k, v, alpha, beta, parent, O=None, status=None, stream=None):
    """gdn_path_verify's outputs in the WY form (every node once); dk 64 or 128, n <= 64."""
    S0, alpha, beta = _f32(S0), _f32(alpha), _f32(beta)
    q, k, v, parent = _bits16(q), _bits16(k), _bits16(v), _i32(parent)
    H, dv, dk = S0.shape
    n = parent.numel()
    O = torch.empty((n, H, dv), dtype=torch.float32, device=S0.device) if O is None else _f32(O)
    status = torch.zeros(1, dtype=torch.int32, device=S0.device) if status is None else _i32(status)
    _check(lib().gdn_wy_verify(_ptr(S0), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(parent), n, H, dk,
                               dv, _ptr(O), _ptr(status), _stream(stream)))
    return O, status


def gdn_commit(S, k, v, alpha, beta, path_len, path_nodes, status=None, stream=None):
    """S [H, dv, dk] float32, in place: advanced by the accepted nodes path_nodes[1..path_len]
    (device int32 tensors as w12_lmhead_verify returns them).  Returns status."""
    S, alpha, beta = _f32(S), _f32(alpha), _f32(beta)
    k, v = _bits16(k), _bits16(v)
    path_len, path_nodes = _i32(path_len), _i32(path_nodes)
    H, dv, dk = S.shape
    n = alpha.shape[0]
    status = torch.zeros(1, dtype=torch.int32, device=S.device) if status is None else _i32(status)
    _check(lib().gdn_commit(_ptr(S), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(path_len), _ptr(path_nodes), n, H,
                            dk, dv, _ptr(status), _stream(stream)))
    return status
