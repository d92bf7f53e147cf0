// w12_api.cu - status reporting and size queries of the C ABI.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "w12_internal.cuh"

namespace w12 {

static thread_local char g_err[512] = "";

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return status;
}

int cuda_fail(cudaError_t e, const char* what) {
  set_error("%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
  return W12_ERR_CUDA;
}

int check_matrix(const w12_matrix* A, bool need_lo, const char* fn) {
  if (!A) return fail(W12_ERR_INVALID_ARG, "%s: null matrix descriptor", fn);
  if (A->N < 1 || A->K < 1 || A->K > kMaxK)
    return fail(W12_ERR_SHAPE, "%s: shape N=%lld K=%lld out of range (1<=N, 1<=K<=65535)", fn, (long long)A->N,
                (long long)A->K);
  if (!A->hi || !A->base || !A->esc_tile_ptr || (need_lo && !A->lo))
    return fail(W12_ERR_INVALID_ARG, "%s: null plane pointer in descriptor", fn);
  if (A->n_esc < 0 || A->n_esc > 0xFFFFFFFFll)
    return fail(W12_ERR_INVALID_ARG, "%s: n_esc=%lld out of range", fn, (long long)A->n_esc);
  if (A->n_esc > 0 && !A->esc) return fail(W12_ERR_INVALID_ARG, "%s: esc is null but n_esc=%lld", fn, (long long)A->n_esc);
  return W12_OK;
}

}  // namespace w12

using namespace w12;

extern "C" {

const char* w12_last_error(void) { return g_err; }

const char* w12_status_string(int s) {
  switch (s) {
    case W12_OK: return "W12_OK";
    case W12_ERR_INVALID_ARG: return "W12_ERR_INVALID_ARG";
    case W12_ERR_SHAPE: return "W12_ERR_SHAPE";
    case W12_ERR_BUFFER_TOO_SMALL: return "W12_ERR_BUFFER_TOO_SMALL";
    case W12_ERR_CUDA: return "W12_ERR_CUDA";
    case W12_ERR_BOUNDS: return "W12_ERR_BOUNDS";
    case W12_ERR_TIMEOUT: return "W12_ERR_TIMEOUT";
    case W12_ERR_IO: return "W12_ERR_IO";
    default: return "W12_ERR_UNKNOWN";
  }
}

int w12_abi_version(void) { return W12_ABI_VERSION; }

static bool shape_ok(int64_t N, int64_t K) { return N >= 1 && K >= 1 && K <= kMaxK; }

int64_t w12_hi_bytes(int64_t N, int64_t K) {
  return shape_ok(N, K) ? row_tiles(N) * k_chunks(K) * kHiTileBytes : -1;
}

int64_t w12_lo_bytes(int64_t N, int64_t K) {
  return shape_ok(N, K) ? row_tiles(N) * k_chunks(K) * kLoTileBytes : -1;
}

int64_t w12_tile_count(int64_t N, int64_t K) { return shape_ok(N, K) ? row_tiles(N) * k_chunks(K) : -1; }

}  // extern "C"
