// w12_io.cu - storage of encoded matrices: the device planes of a W12 matrix to a file
// and back, so that a model is converted once.
//
// The SpecPilot summary page (onedev.kr/papers/1654), section "What's different", stores
// the converted layers.  The file is a 72-byte little-endian header (magic "W12M", format
// version, N, K, n_esc, then the byte counts of the five arrays) followed by the hi plane,
// the lo plane, base[N], esc_tile_ptr[tile_count + 1] and esc[n_esc], as the device
// format of include/w12.h lays them out.  Copies go through a bounded host buffer, so a
// large head needs no host copy of the whole matrix.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <vector>

#include "w12_internal.cuh"

namespace w12 {
namespace {

constexpr char kMagic[4] = {'W', '1', '2', 'M'};
constexpr uint32_t kFormat = 1;
constexpr size_t kChunk = size_t(64) << 20;  // host staging buffer

struct Header {
  char magic[4];
  uint32_t format;
  int64_t N, K, n_esc;
  int64_t bytes[5];  // hi, lo, base, esc_tile_ptr, esc
};
static_assert(sizeof(Header) == 72, "header layout");

void array_bytes(int64_t N, int64_t K, int64_t n_esc, int64_t out[5]) {
  out[0] = w12_hi_bytes(N, K);
  out[1] = w12_lo_bytes(N, K);
  out[2] = N;
  out[3] = (w12_tile_count(N, K) + 1) * 4;
  out[4] = n_esc * 4;
}

struct File {
  FILE* f = nullptr;
  ~File() {
    if (f) fclose(f);
  }
};

int read_header(FILE* f, Header* h, const char* fn, const char* path) {
  if (fread(h, sizeof(Header), 1, f) != 1) return fail(W12_ERR_IO, "%s: %s: truncated header", fn, path);
  if (memcmp(h->magic, kMagic, 4) != 0) return fail(W12_ERR_IO, "%s: %s is not a W12 matrix file", fn, path);
  if (h->format != kFormat)
    return fail(W12_ERR_IO, "%s: %s has format %u (this library reads %u)", fn, path, h->format, kFormat);
  if (h->N < 1 || h->K < 1 || h->K > kMaxK || h->n_esc < 0 || h->n_esc > 0xFFFFFFFFll)
    return fail(W12_ERR_IO, "%s: %s: header sizes out of range", fn, path);
  int64_t want[5];
  array_bytes(h->N, h->K, h->n_esc, want);
  for (int i = 0; i < 5; ++i)
    if (h->bytes[i] != want[i]) return fail(W12_ERR_IO, "%s: %s: array %d has %lld bytes, %lld expected", fn, path, i,
                                            (long long)h->bytes[i], (long long)want[i]);
  return W12_OK;
}

}  // namespace
}  // namespace w12

using namespace w12;

extern "C" {

int w12_save(const w12_matrix* A, const char* path, void* stream) {
  const char* fn = "w12_save";
  int st = check_matrix(A, true, fn);
  if (st) return st;
  if (!path) return fail(W12_ERR_INVALID_ARG, "%s: null path", fn);
  Header h{};
  memcpy(h.magic, kMagic, 4);
  h.format = kFormat;
  h.N = A->N;
  h.K = A->K;
  h.n_esc = A->n_esc;
  array_bytes(A->N, A->K, A->n_esc, h.bytes);
  const void* src[5] = {A->hi, A->lo, A->base, A->esc_tile_ptr, A->esc};
  File out;
  out.f = fopen(path, "wb");
  if (!out.f) return fail(W12_ERR_IO, "%s: cannot open %s for writing", fn, path);
  if (fwrite(&h, sizeof(h), 1, out.f) != 1) return fail(W12_ERR_IO, "%s: write to %s failed", fn, path);
  cudaStream_t s = (cudaStream_t)stream;
  std::vector<uint8_t> buf;
  for (int i = 0; i < 5; ++i) {
    for (int64_t off = 0; off < h.bytes[i]; off += (int64_t)kChunk) {
      const size_t n = (size_t)std::min<int64_t>((int64_t)kChunk, h.bytes[i] - off);
      if (buf.size() < n) buf.resize(n);
      W12_CUDA_TRY(cudaMemcpyAsync(buf.data(), static_cast<const uint8_t*>(src[i]) + off, n, cudaMemcpyDeviceToHost, s));
      W12_CUDA_TRY(cudaStreamSynchronize(s));
      if (fwrite(buf.data(), 1, n, out.f) != n) return fail(W12_ERR_IO, "%s: write to %s failed", fn, path);
    }
  }
  if (fclose(out.f) != 0) {
    out.f = nullptr;
    return fail(W12_ERR_IO, "%s: closing %s failed", fn, path);
  }
  out.f = nullptr;
  return W12_OK;
}

int w12_load_info(const char* path, int64_t* N, int64_t* K, int64_t* n_esc) {
  const char* fn = "w12_load_info";
  if (!path || !N || !K || !n_esc) return fail(W12_ERR_INVALID_ARG, "%s: null pointer", fn);
  File in;
  in.f = fopen(path, "rb");
  if (!in.f) return fail(W12_ERR_IO, "%s: cannot open %s", fn, path);
  Header h{};
  int st = read_header(in.f, &h, fn, path);
  if (st) return st;
  *N = h.N;
  *K = h.K;
  *n_esc = h.n_esc;
  return W12_OK;
}

int w12_load(const char* path, const w12_matrix* A, void* stream) {
  const char* fn = "w12_load";
  if (!path) return fail(W12_ERR_INVALID_ARG, "%s: null path", fn);
  int st = check_matrix(A, true, fn);
  if (st) return st;
  File in;
  in.f = fopen(path, "rb");
  if (!in.f) return fail(W12_ERR_IO, "%s: cannot open %s", fn, path);
  Header h{};
  if ((st = read_header(in.f, &h, fn, path))) return st;
  if (h.N != A->N || h.K != A->K || h.n_esc != A->n_esc)
    return fail(W12_ERR_SHAPE, "%s: %s holds %lld x %lld with %lld escapes, the descriptor %lld x %lld with %lld", fn,
                path, (long long)h.N, (long long)h.K, (long long)h.n_esc, (long long)A->N, (long long)A->K,
                (long long)A->n_esc);
  void* dst[5] = {A->hi, A->lo, A->base, A->esc_tile_ptr, A->esc};
  cudaStream_t s = (cudaStream_t)stream;
  std::vector<uint8_t> buf;
  for (int i = 0; i < 5; ++i) {
    for (int64_t off = 0; off < h.bytes[i]; off += (int64_t)kChunk) {
      const size_t n = (size_t)std::min<int64_t>((int64_t)kChunk, h.bytes[i] - off);
      if (buf.size() < n) buf.resize(n);
      if (fread(buf.data(), 1, n, in.f) != n) return fail(W12_ERR_IO, "%s: %s is truncated", fn, path);
      W12_CUDA_TRY(cudaMemcpyAsync(static_cast<uint8_t*>(dst[i]) + off, buf.data(), n, cudaMemcpyHostToDevice, s));
      W12_CUDA_TRY(cudaStreamSynchronize(s));  // the staging buffer is reused
    }
  }
  return W12_OK;
}

}  // extern "C"
