"""libw12.so builds, loads without a GPU and exports every symbol include/w12.h
declares; the pure host size queries answer without touching CUDA."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "w12.h")).read()
    return set(re.findall(r"^W12_API [^(]*?\b(\w+)\(", text, flags=re.M))


def test_header_and_binding_agree():
    import lossless_bit_weights_gb300 as w12
    names = {n for n, _, _ in w12.SIGNATURES}
    assert declared_symbols() == names


def test_library_exports_every_declared_symbol():
    import lossless_bit_weights_gb300 as w12
    lib = w12.lib()
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert lib.w12_abi_version() == 1


def test_host_size_queries():
    import lossless_bit_weights_gb300 as w12
    lib = w12.lib()
    assert lib.w12_tile_count(32, 64) == 4       # one row block of 4 row tiles
    assert lib.w12_tile_count(129, 65) == 16     # two row blocks, two chunks
    assert lib.w12_hi_bytes(5120, 5120) == 160 * 80 * 2048
    assert lib.w12_lo_bytes(5120, 5120) == 160 * 80 * 1024
    assert lib.w12_hi_bytes(1, 65536) == -1
    assert lib.w12_tile_count(0, 5) == -1
    assert lib.w12_status_string(2) == b"W12_ERR_SHAPE"


def test_argument_errors_are_reported_without_device_work():
    """Null pointers and bad shapes fail host-side checks before any CUDA call."""
    import ctypes
    import lossless_bit_weights_gb300 as w12
    lib = w12.lib()
    n = ctypes.c_int64(0)
    assert lib.w12_encode_plan(None, 4, 4, None, None, ctypes.byref(n), None) == 1
    assert b"null" in lib.w12_last_error()
    assert lib.w12_encode_plan(ctypes.c_void_p(256), 4, 70000, ctypes.c_void_p(256), ctypes.c_void_p(256),
                               ctypes.byref(n), None) == 2
    bad = w12.w12_matrix(0, 5, 256, 256, 256, 256, 0, 0)
    assert lib.w12_decode(ctypes.byref(bad), ctypes.c_void_p(256), None) == 2
    good_shape_null_plane = w12.w12_matrix(4, 5, None, 256, 256, 256, 0, 0)
    assert lib.w12_decode(ctypes.byref(good_shape_null_plane), ctypes.c_void_p(256), None) == 1
    assert lib.tree_verify_tokens(None, None, None, None, 1, 4, None, None, None, None) == 1
    p = ctypes.c_void_p(256)
    assert lib.tree_verify_tokens(p, p, p, None, 2, 4, p, p, p, None) == 1   # several requests need offsets


def test_certified_head_and_recurrent_argument_errors():
    """The INT8 head and recurrent-layer calls check shapes and pointers on the host."""
    import ctypes
    import lossless_bit_weights_gb300 as w12
    lib = w12.lib()
    p = ctypes.c_void_p(256)
    assert lib.w12_i8_code_bytes(5120, 5120) == lib.w12_hi_bytes(5120, 5120)
    assert lib.w12_cert_head_workspace_size(0, 10, 10) == 0
    assert lib.w12_cert_head_workspace_size(16, 151936, 5120) > 16 * 151936 * 8
    H = w12.w12_i8_head(0, 5120, 256, 256, 256)
    assert lib.w12_i8_encode(p, ctypes.byref(H), None) == 2                      # V = 0
    H = w12.w12_i8_head(8, 64, 264, 256, 256)
    assert lib.w12_i8_encode(p, ctypes.byref(H), None) == 1                      # misaligned codes
    assert b"aligned" in lib.w12_last_error()
    H = w12.w12_i8_head(8, 64, 256, 256, 256)
    A = w12.w12_matrix(8, 32, 256, 256, 256, 256, 0, 0)                          # K differs
    assert lib.w12_cert_head_argmax(p, 4, ctypes.byref(H), ctypes.byref(A), p, None, p, 1 << 30, None) == 2
    A = w12.w12_matrix(8, 64, 256, 256, 256, 256, 0, 0)
    assert lib.w12_cert_head_argmax(p, 4, ctypes.byref(H), ctypes.byref(A), p, None, p, 16, None) == 3
    # recurrent layers: dims, tree size, pointers
    assert lib.gdn_split3(None, 0, None, None, None, None) == 0                  # nothing to do
    assert lib.gdn_split3(None, 4, None, None, None, None) == 1
    assert lib.gdn_path_verify(p, p, p, p, p, p, p, 4, 2, 256, 256, p, p, None) == 2   # state too large
    assert b"shared memory" in lib.w12_last_error()
    assert lib.gdn_path_verify(p, p, p, p, p, p, p, 5000, 2, 128, 128, p, p, None) == 2  # too many nodes
    assert lib.gdn_path_verify(p, p, p, p, p, p, None, 4, 2, 128, 128, p, p, None) == 1
    assert lib.gdn_commit(p, p, p, p, p, p, p, 0, 2, 128, 128, p, None) == 2
    assert lib.gdn_commit(p, p, p, p, p, None, p, 4, 2, 128, 128, p, None) == 1


def test_error_queries_and_noalloc_check_arguments_before_any_cuda_call():
    """w12_workspace_status, w12_validate and w12_gemm_noalloc refuse bad arguments on the
    host: on a machine without a GPU the answer is the argument error, not a CUDA error,
    so no device work (and for w12_gemm_noalloc no clearing of its scratch) came first."""
    import ctypes
    import lossless_bit_weights_gb300 as w12
    lib = w12.lib()
    st = ctypes.c_int32(-1)
    p = ctypes.c_void_p(256)
    assert lib.w12_workspace_status(None, 4096, ctypes.byref(st), None) == 1
    assert lib.w12_workspace_status(p, 4096, None, None) == 1
    assert lib.w12_workspace_status(p, 128, ctypes.byref(st), None) == 3
    A = w12.w12_matrix(64, 64, 256, 256, 256, 256, 256, 4)
    assert lib.w12_validate(ctypes.byref(A), None, None) == 1
    assert lib.w12_validate(None, p, None) == 1
    assert lib.w12_gemm_noalloc(None, 4, ctypes.byref(A), p, None) == 1
    mis = w12.w12_matrix(64, 64, 264, 256, 256, 256, 256, 4)
    assert lib.w12_gemm_noalloc(p, 4, ctypes.byref(mis), p, None) == 1
    assert b"aligned" in lib.w12_last_error()
    assert lib.w12_gemm_noalloc(p, 0, ctypes.byref(A), p, None) == 2
    assert lib.w12_gemm_counter_bytes(5120) == 256 + 768       # error word, then 40 x 4 counters


def test_storage_header_checks_without_a_gpu(tmp_path):
    """w12_load_info / w12_load read and check a file's header on the host: a missing
    file, a file of another kind, a truncated header or sizes that do not fit the shape
    are W12_ERR_IO; a descriptor that differs from the file is W12_ERR_SHAPE, before
    any CUDA call."""
    import ctypes
    import struct
    import lossless_bit_weights_gb300 as w12
    lib = w12.lib()
    N_, K_, E_ = ctypes.c_int64(0), ctypes.c_int64(0), ctypes.c_int64(0)
    info = lambda p: lib.w12_load_info(str(p).encode(), ctypes.byref(N_), ctypes.byref(K_), ctypes.byref(E_))
    assert lib.w12_status_string(7) == b"W12_ERR_IO"
    assert info(tmp_path / "missing.w12") == 7
    other = tmp_path / "other.bin"
    other.write_bytes(b"not a matrix file" * 8)
    assert info(other) == 7
    assert b"not a W12" in lib.w12_last_error()
    N, K, n_esc = 100, 300, 7
    sizes = [lib.w12_hi_bytes(N, K), lib.w12_lo_bytes(N, K), N, (lib.w12_tile_count(N, K) + 1) * 4, n_esc * 4]
    header = b"W12M" + struct.pack("<I3q5q", 1, N, K, n_esc, *sizes)
    assert len(header) == 72
    good = tmp_path / "good.w12"
    good.write_bytes(header)
    assert info(good) == 0 and (N_.value, K_.value, E_.value) == (N, K, n_esc)
    (tmp_path / "short.w12").write_bytes(header[:40])
    assert info(tmp_path / "short.w12") == 7
    bad = tmp_path / "bad.w12"
    bad.write_bytes(b"W12M" + struct.pack("<I3q5q", 1, N, K, n_esc, sizes[0] + 1, *sizes[1:]))
    assert info(bad) == 7
    p = ctypes.c_void_p(256)
    A = w12.w12_matrix(N, K + 1, 256, 256, 256, 256, 256, n_esc)   # K differs from the file's
    assert lib.w12_load(str(good).encode(), ctypes.byref(A), None) == 2
    assert lib.w12_load(None, ctypes.byref(A), None) == 1
    assert lib.w12_save(None, str(good).encode(), None) == 1
