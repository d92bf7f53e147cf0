"""Seeded synthetic inputs for the W12 verify path (host and device).

This package makes inputs only; it holds none of the W12 arithmetic.  The C
sources in this folder define every value as a pure function of
(seed, layer, tensor id, element index), so the host library (gcc) and the
device library (nvcc) give identical bf16 bits.  ``build()`` compiles both.
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
HOST_SO = os.path.join(BUILD, "libsynth_host.so")
DEV_SO = os.path.join(BUILD, "libsynth_dev.so")

_lock = threading.Lock()
_host = None
_dev = None


def _stale(out: str, srcs) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(os.path.join(HERE, s)) > t for s in srcs)


def build_host() -> str:
    os.makedirs(BUILD, exist_ok=True)
    if _stale(HOST_SO, ["synth.h", "synth_host.c"]):
        tmp = HOST_SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
                               "-fno-math-errno", "-o", tmp, os.path.join(HERE, "synth_host.c"), "-lm"])
        os.replace(tmp, HOST_SO)
    return HOST_SO


def build_dev() -> str:
    os.makedirs(BUILD, exist_ok=True)
    if _stale(DEV_SO, ["synth.h", "synth_dev.cu"]):
        tmp = DEV_SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["nvcc", "-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
                               "-Xcompiler", "-fPIC", "-shared", "-cudart", "static", "-o", tmp,
                               os.path.join(HERE, "synth_dev.cu")])
        os.replace(tmp, DEV_SO)
    return DEV_SO


def build() -> None:
    build_host()
    build_dev()


def _h():
    global _host
    with _lock:
        if _host is None:
            lib = ctypes.CDLL(build_host())
            u64, i64, p = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
            lib.syn_weights_rows.argtypes = [u64, u64, u64, i64, i64, i64, p]
            lib.syn_weights_rows_ex.argtypes = [u64, u64, u64, i64, i64, i64, ctypes.c_int, p]
            lib.syn_weights_rows_ex.restype = None
            lib.syn_channel_scales.argtypes = [u64, u64, u64, i64, i64, p]
            lib.syn_activations.argtypes = [u64, u64, u64, i64, i64, p]
            lib.syn_tree.argtypes = [u64, u64, u64, i64, p]
            lib.syn_drafts.argtypes = [u64, u64, u64, i64, i64, p]
            lib.syn_u64.argtypes = [u64, u64, u64, i64, i64, p]
            for f in (lib.syn_weights_rows, lib.syn_channel_scales, lib.syn_activations, lib.syn_tree,
                      lib.syn_drafts, lib.syn_u64):
                f.restype = None
            _host = lib
        return _host


def _d():
    global _dev
    with _lock:
        if _dev is None:
            lib = ctypes.CDLL(build_dev())
            u64, i64, p = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
            lib.syn_weights_dev.argtypes = [u64, u64, u64, i64, i64, p, p]
            lib.syn_weights_dev_ex.argtypes = [u64, u64, u64, i64, i64, ctypes.c_int, p, p]
            lib.syn_weights_dev_ex.restype = ctypes.c_int
            lib.syn_activations_dev.argtypes = [u64, u64, u64, i64, p, p]
            lib.syn_weights_dev.restype = ctypes.c_int
            lib.syn_activations_dev.restype = ctypes.c_int
            _dev = lib
        return _dev


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _threads(n_items: int, threads: int | None) -> int:
    t = threads or (os.cpu_count() or 1)
    return max(1, min(t, n_items))


def weights(seed: int, layer: int, tensor: int, N: int, K: int, row0: int = 0, nrows: int | None = None,
            threads: int | None = None, outliers: bool = True) -> np.ndarray:
    """bf16 bits (uint16) of rows [row0, row0+nrows) of the N x K weight matrix
    (outliers=False: the head recipe, without the x2^9 outliers)."""
    nrows = N - row0 if nrows is None else nrows
    out = np.empty((nrows, K), dtype=np.uint16)
    if nrows == 0 or K == 0:
        return out
    lib = _h()
    nt = _threads(nrows, threads)
    bounds = [row0 + (nrows * i) // nt for i in range(nt + 1)]

    def run(i):
        a, b = bounds[i], bounds[i + 1]
        if b > a:
            lib.syn_weights_rows_ex(seed, layer, tensor, K, a, b - a, int(outliers), _ptr(out) + (a - row0) * K * 2)

    if nt == 1:
        run(0)
    else:
        with ThreadPoolExecutor(nt) as ex:
            list(ex.map(run, range(nt)))
    return out


def weight_rows(seed: int, layer: int, tensor: int, K: int, rows, outliers: bool = True) -> np.ndarray:
    """bf16 bits of an arbitrary list of rows (any order) of a weight matrix."""
    rows = np.asarray(rows, dtype=np.int64)
    out = np.empty((len(rows), K), dtype=np.uint16)
    lib = _h()
    for i, r in enumerate(rows):
        lib.syn_weights_rows_ex(seed, layer, tensor, K, int(r), 1, int(outliers), _ptr(out) + i * K * 2)
    return out


def channel_scales(seed: int, layer: int, tensor: int, N: int) -> np.ndarray:
    out = np.empty(N, dtype=np.float32)
    _h().syn_channel_scales(seed, layer, tensor, 0, N, _ptr(out))
    return out


def activations(seed: int, layer: int, tensor: int, M: int, K: int) -> np.ndarray:
    """bf16 bits of an M x K activation matrix (element index m*K + k)."""
    out = np.empty((M, K), dtype=np.uint16)
    if M * K:
        _h().syn_activations(seed, layer, tensor, 0, M * K, _ptr(out))
    return out


def tree(seed: int, layer: int, tensor: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    if n:
        _h().syn_tree(seed, layer, tensor, n, _ptr(out))
    return out


def drafts(seed: int, layer: int, tensor: int, n: int, V: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    if n:
        _h().syn_drafts(seed, layer, tensor, n, V, _ptr(out))
    return out


def u64(seed: int, layer: int, tensor: int, count: int, i0: int = 0) -> np.ndarray:
    out = np.empty(count, dtype=np.uint64)
    if count:
        _h().syn_u64(seed, layer, tensor, i0, count, _ptr(out))
    return out


# ----------------------------------------------------------------------------------------------
# device generation (torch is used only for the buffers and the stream)

def weights_dev(seed: int, layer: int, tensor: int, out, stream=None, outliers: bool = True) -> None:
    """Fill a contiguous torch.uint16/int16 CUDA tensor of shape (N, K) with the weight matrix."""
    import torch
    N, K = out.shape
    s = stream if stream is not None else torch.cuda.current_stream()
    rc = _d().syn_weights_dev_ex(seed, layer, tensor, N, K, int(outliers), out.data_ptr(), s.cuda_stream)
    if rc:
        raise RuntimeError(f"syn_weights_dev failed with CUDA error {rc}")


def activations_dev(seed: int, layer: int, tensor: int, out, stream=None) -> None:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    rc = _d().syn_activations_dev(seed, layer, tensor, out.numel(), out.data_ptr(), s.cuda_stream)
    if rc:
        raise RuntimeError(f"syn_activations_dev failed with CUDA error {rc}")


def peaked_activations(seed: int, layer: int, tensor: int, head_rows, beta: float) -> np.ndarray:
    """bf16 bits of M hidden-state rows that point at given head rows:
    x_m = bf16(z_m + beta * w_m / ||w_m||), z_m the N(0,1) activation rows (seed, layer,
    tensor) and w_m = head_rows[m] (bf16 bits, M x K).  A verify pass's final hidden
    state points at the token it predicts; plain N(0,1) rows leave no top logit."""
    head_rows = np.asarray(head_rows, np.uint16)
    M, K = head_rows.shape
    z = (activations(seed, layer, tensor, M, K).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    w = (head_rows.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    nrm = np.sqrt((w * w).sum(axis=1, keepdims=True))
    nrm[nrm == 0] = 1.0
    f = (z + beta * w / nrm).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
