// w12_cert.cu - certified LM-head argmax over an INT8 head.
//
// The SpecPilot summary page (onedev.kr/papers/1654), section "What's
// different", keeps the LM head of its H100 build in INT8 and filters the
// argmax candidates with a Cauchy-Schwarz error bound, computing only those
// exactly; on an RTX PRO 6000 that was slower than a W12 head.  Here:
//   - each output channel v gets a symmetric INT8 code q (scale s_v =
//     max|w|/127, q = rint(w/s_v)), stored in the W12 hi-plane layout so the
//     tcgen05 GEMM streams it like the 8-bit view; the GEMM gives s_v * x.q_v;
//   - |x.w_v - s_v x.q_v| <= ||x|| c_v with c_v = ||w_v - s_v q_v|| +
//     gamma * s_v * ||q_v||, gamma = (K + 16) * 2^-21 covering the float
//     accumulation of x.q_v (its products are exact);
//   - candidates are the channels whose approximate logit plus bound reaches
//     the row's largest approximate logit minus bound; every bound and
//     comparison is rounded outward, so the exact argmax is always among them;
//   - each candidate's exact logit is recomputed in fp64 from the lossless W12
//     form of the same head (decode of one channel), and the largest wins,
//     ties to the lowest index.
#include <cstdint>

#include "w12_internal.cuh"

namespace w12 {

int i8_gemm_impl(const uint16_t* x, int64_t M, const uint8_t* codes, const float* scale, int64_t V, int64_t K,
                 float* y, void* ws, size_t ws_bytes, cudaStream_t s, const char* fn);

namespace {

constexpr int kExactBlocks = 16;  // blocks per row of the exact recompute
constexpr int kExactWarps = 8;

inline size_t al256(size_t b) { return (b + 255) & ~(size_t)255; }

double i8_gamma(int64_t K) { return (double)(K + 16) * 4.76837158203125e-07; /* 2^-21 */ }

__device__ __forceinline__ float bf16f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// Block-wide reductions over blockDim.x threads (a multiple of 32, at most 1024), in a
// fixed tree order.
__device__ double block_sum(double v, double* sh) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sh[w] = v;
  __syncthreads();
  double t = 0.0;
  if (threadIdx.x < 32) {
    t = (int)threadIdx.x < nw ? sh[threadIdx.x] : 0.0;
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, o);
  }
  return t;  // valid in thread 0
}

__device__ float block_max(float v, float* sh) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sh[w] = v;
  __syncthreads();
  float t = -INFINITY;
  if (threadIdx.x < 32) {
    t = (int)threadIdx.x < nw ? sh[threadIdx.x] : -INFINITY;
    for (int o = 16; o > 0; o >>= 1) t = fmaxf(t, __shfl_xor_sync(0xFFFFFFFFu, t, o));
  }
  return t;  // valid in thread 0
}

// One block per channel.  code must be zero beforehand (padding rows and columns).
__global__ void __launch_bounds__(256) k_i8_encode(const uint16_t* __restrict__ W, int64_t K, int64_t KC,
                                                   uint8_t* __restrict__ code, float* __restrict__ scale,
                                                   float* __restrict__ cbound, double gamma) {
  __shared__ double shd[32];
  __shared__ float shf[32];
  __shared__ float s_sh;
  const int64_t v = blockIdx.x;
  const uint16_t* row = W + v * K;
  float amax = 0.f;
  for (int64_t k = threadIdx.x; k < K; k += blockDim.x) amax = fmaxf(amax, fabsf(bf16f(row[k])));
  amax = block_max(amax, shf);
  if (threadIdx.x == 0) s_sh = amax / 127.0f;
  __syncthreads();
  const float s = s_sh;
  const int64_t rt = v / kTileRows;
  const int r = (int)(v % kTileRows);
  double e2 = 0.0, q2 = 0.0;
  for (int64_t k = threadIdx.x; k < K; k += blockDim.x) {
    const double w = (double)bf16f(row[k]);
    double q = 0.0;
    if (s > 0.f) q = fmin(127.0, fmax(-127.0, rint(w / (double)s)));
    const int iq = (int)q;
    const int64_t kc = k / kTileK;
    code[tile_index(rt, kc, KC) * kHiTileBytes + hi_offset(r, (int)(k - kc * kTileK))] =
        (uint8_t)(iq < 0 ? (0x80 | -iq) : iq);
    const double d = w - (double)s * q;
    e2 += d * d;
    q2 += q * q;
  }
  e2 = block_sum(e2, shd);
  q2 = block_sum(q2, shd);
  if (threadIdx.x == 0) {
    scale[v] = s;
    cbound[v] = __double2float_ru(__dadd_ru(__dsqrt_ru(e2), __dmul_ru(__dmul_ru(gamma, (double)s), __dsqrt_ru(q2))));
  }
}

// nx[m] >= ||x_m||, rounded up to float.
__global__ void __launch_bounds__(256) k_rownorm(const uint16_t* __restrict__ x, int64_t K, float* __restrict__ nx) {
  __shared__ double shd[32];
  const uint16_t* xr = x + (int64_t)blockIdx.x * K;
  double a = 0.0;
  for (int64_t k = threadIdx.x; k < K; k += blockDim.x) {
    const double f = (double)bf16f(xr[k]);
    a += f * f;
  }
  a = block_sum(a, shd);
  if (threadIdx.x == 0) nx[blockIdx.x] = __double2float_ru(__dsqrt_ru(a));
}

// thr[m] = max_v (approx[m,v] - bound[m,v]), every step rounded down.
__global__ void __launch_bounds__(1024) k_cert_thr(const float* __restrict__ lh, int64_t V, const float* __restrict__ nx,
                                                   const float* __restrict__ cb, float* __restrict__ thr) {
  __shared__ float shf[32];
  const int64_t m = blockIdx.x;
  const float n = nx[m];
  float t = -INFINITY;
  for (int64_t v = threadIdx.x; v < V; v += blockDim.x) t = fmaxf(t, __fsub_rd(lh[m * V + v], __fmul_ru(n, cb[v])));
  t = block_max(t, shf);
  if (threadIdx.x == 0) thr[m] = t;
}

// Candidates: approx + bound (rounded up) >= thr.
__global__ void __launch_bounds__(1024) k_cert_cand(const float* __restrict__ lh, int64_t V, const float* __restrict__ nx,
                                                    const float* __restrict__ cb, const float* __restrict__ thr,
                                                    int32_t* __restrict__ count, int32_t* __restrict__ cand) {
  const int64_t m = blockIdx.y, v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (v >= V) return;
  if (__fadd_ru(lh[m * V + v], __fmul_ru(nx[m], cb[v])) >= thr[m]) {
    const int pos = atomicAdd(count + m, 1);
    cand[m * V + pos] = (int32_t)v;
  }
}

struct Best {
  double val;
  int32_t idx;  // -1: none
};

__device__ __forceinline__ bool beats(double a, int32_t ia, double b, int32_t ib) {
  if (ia < 0) return false;
  if (ib < 0) return true;
  return a > b || (a == b && ia < ib);
}

// Exact logits of the candidates in fp64 from the W12 head: warp w of block b takes
// candidates b*8 + w, stepping by 16 blocks x 8 warps.  Lane 4*c8 + t decodes the 16
// columns 16t.. of chunk kc0 + c8 (the same decode as the GEMM), patches the channel's
// escapes in them and multiplies by x.
__global__ void __launch_bounds__(kExactWarps * 32)
    k_cert_exact(const uint16_t* __restrict__ x, int64_t K, int64_t KC, const uint8_t* __restrict__ hi,
                 const uint8_t* __restrict__ lo, const uint8_t* __restrict__ base, const uint32_t* __restrict__ tile_ptr,
                 const uint32_t* __restrict__ esc, const int32_t* __restrict__ count, const int32_t* __restrict__ cand,
                 int64_t V, DecodeMul mul, Best* __restrict__ part) {
  __shared__ Best sh[kExactWarps];
  const int64_t m = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c8 = lane >> 2, t = lane & 3;
  const int n_c = count[m];
  const uint16_t* xr = x + m * K;
  Best best{0.0, -1};
  for (int i = blockIdx.x * kExactWarps + warp; i < n_c; i += kExactBlocks * kExactWarps) {
    const int64_t v = cand[m * V + i];
    const int64_t rt = v / kTileRows;
    const int r = (int)(v % kTileRows), q = r >> 3, g = r & 7;
    const uint32_t bb = base[v];
    const uint32_t base2 = (bb << 7) | (bb << 23);
    double acc = 0.0;
    for (int64_t kc0 = 0; kc0 < KC; kc0 += 8) {
      const int64_t kc = kc0 + c8;
      if (kc >= KC) continue;
      const int64_t tile = tile_index(rt, kc, KC);
      const uint4 hq = *reinterpret_cast<const uint4*>(hi + tile * kHiTileBytes + q * 512 + (4 * g + t) * 16);
      const uint2 lq = *reinterpret_cast<const uint2*>(lo + tile * kLoTileBytes + q * 256 + (4 * g + t) * 8);
      uint32_t pr[8];
      decode16<false>(hq, lq, base2, mul, pr);
      uint16_t w[16];
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        w[2 * p] = (uint16_t)(pr[p] & 0xFFFFu);
        w[2 * p + 1] = (uint16_t)(pr[p] >> 16);
      }
      for (uint32_t e = tile_ptr[tile]; e < tile_ptr[tile + 1]; ++e) {
        const uint32_t ent = esc[e];
        const int c = esc_col(ent);
        if (esc_row(ent) == r && (c >> 4) == t) {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (j == (c & 15)) w[j] = (uint16_t)esc_raw(ent);
        }
      }
      const int64_t k0 = kc * kTileK + 16 * t;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (k0 + j < K) acc += (double)bf16f(xr[k0 + j]) * (double)bf16f(w[j]);
    }
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    if (beats(acc, (int32_t)v, best.val, best.idx)) best = Best{acc, (int32_t)v};
  }
  if (lane == 0) sh[warp] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    Best b = sh[0];
    for (int w = 1; w < kExactWarps; ++w)
      if (beats(sh[w].val, sh[w].idx, b.val, b.idx)) b = sh[w];
    part[m * kExactBlocks + blockIdx.x] = b;
  }
}

__global__ void k_cert_final(const Best* __restrict__ part, const int32_t* __restrict__ count, int32_t* __restrict__ tok,
                             int32_t* __restrict__ ncand) {
  const int64_t m = blockIdx.x;
  if (threadIdx.x != 0) return;
  Best b = part[m * kExactBlocks];
  for (int i = 1; i < kExactBlocks; ++i) {
    const Best c = part[m * kExactBlocks + i];
    if (beats(c.val, c.idx, b.val, b.idx)) b = c;
  }
  tok[m] = b.idx;
  if (ncand) ncand[m] = count[m];
}

struct CertWs {
  size_t gemm, lh, nx, thr, count, cand, part, total;
};

CertWs cert_ws(int64_t M, int64_t V, int64_t K) {
  CertWs L{};
  L.gemm = 0;
  size_t off = al256(w12_gemm_workspace_size(M, V, K));
  L.lh = off;
  off = al256(off + (size_t)M * (size_t)V * 4);
  L.nx = off;
  off = al256(off + (size_t)M * 4);
  L.thr = off;
  off = al256(off + (size_t)M * 4);
  L.count = off;
  off = al256(off + (size_t)M * 4);
  L.cand = off;
  off = al256(off + (size_t)M * (size_t)V * 4);
  L.part = off;
  off = al256(off + (size_t)M * kExactBlocks * sizeof(Best));
  L.total = off;
  return L;
}

int check_head(const w12_i8_head* H, const char* fn) {
  if (!H) return fail(W12_ERR_INVALID_ARG, "%s: null head", fn);
  if (H->V < 1 || H->K < 1 || H->K > kMaxK)
    return fail(W12_ERR_SHAPE, "%s: V=%lld K=%lld out of range", fn, (long long)H->V, (long long)H->K);
  if (!H->code || !H->scale || !H->cbound) return fail(W12_ERR_INVALID_ARG, "%s: null head buffer", fn);
  if (((uintptr_t)H->code & 15u) != 0) return fail(W12_ERR_INVALID_ARG, "%s: code must be 16-byte aligned", fn);
  return W12_OK;
}

}  // namespace
}  // namespace w12

using namespace w12;

extern "C" {

int64_t w12_i8_code_bytes(int64_t V, int64_t K) { return w12_hi_bytes(V, K); }

int w12_i8_encode(const uint16_t* W, const w12_i8_head* H, void* stream) {
  const char* fn = "w12_i8_encode";
  int st = check_head(H, fn);
  if (st) return st;
  if (!W) return fail(W12_ERR_INVALID_ARG, "%s: null W", fn);
  cudaStream_t s = (cudaStream_t)stream;
  const int64_t KC = k_chunks(H->K);
  W12_CUDA_TRY(cudaMemsetAsync(H->code, 0, (size_t)w12_hi_bytes(H->V, H->K), s));
  k_i8_encode<<<(unsigned)H->V, 256, 0, s>>>(W, H->K, KC, H->code, H->scale, H->cbound, i8_gamma(H->K));
  W12_LAUNCH_CHECK("w12_i8_encode");
  return W12_OK;
}

size_t w12_cert_head_workspace_size(int64_t M, int64_t V, int64_t K) {
  if (M < 1 || V < 1 || K < 1) return 0;
  return cert_ws(M, V, K).total;
}

int w12_cert_head_argmax(const uint16_t* x, int64_t M, const w12_i8_head* H, const w12_matrix* exact, int32_t* tok,
                         int32_t* ncand, void* ws, size_t ws_bytes, void* stream) {
  const char* fn = "w12_cert_head_argmax";
  int st = check_head(H, fn);
  if (st) return st;
  if ((st = check_matrix(exact, true, fn))) return st;
  if (exact->N != H->V || exact->K != H->K)
    return fail(W12_ERR_SHAPE, "%s: exact head is %lld x %lld, INT8 head %lld x %lld", fn, (long long)exact->N,
                (long long)exact->K, (long long)H->V, (long long)H->K);
  if (!x || !tok) return fail(W12_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (M < 1 || M > (1 << 20)) return fail(W12_ERR_SHAPE, "%s: M=%lld out of range (1..2^20)", fn, (long long)M);
  if (!ws) return fail(W12_ERR_INVALID_ARG, "%s: null workspace", fn);
  const int64_t V = H->V, K = H->K, KC = k_chunks(K);
  const CertWs L = cert_ws(M, V, K);
  if (ws_bytes < L.total)
    return fail(W12_ERR_BUFFER_TOO_SMALL, "%s: workspace %zu bytes < %zu required", fn, ws_bytes, L.total);
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* lh = reinterpret_cast<float*>(w + L.lh);
  float* nx = reinterpret_cast<float*>(w + L.nx);
  float* thr = reinterpret_cast<float*>(w + L.thr);
  int32_t* count = reinterpret_cast<int32_t*>(w + L.count);
  int32_t* cand = reinterpret_cast<int32_t*>(w + L.cand);
  Best* part = reinterpret_cast<Best*>(w + L.part);
  // approximate logits s_v * x.q_v
  if ((st = i8_gemm_impl(x, M, H->code, H->scale, V, K, lh, w + L.gemm, L.lh, s, fn))) return st;
  k_rownorm<<<(unsigned)M, 256, 0, s>>>(x, K, nx);
  W12_LAUNCH_CHECK("w12_cert_head_argmax: row norms");
  k_cert_thr<<<(unsigned)M, 1024, 0, s>>>(lh, V, nx, H->cbound, thr);
  W12_LAUNCH_CHECK("w12_cert_head_argmax: threshold");
  W12_CUDA_TRY(cudaMemsetAsync(count, 0, (size_t)M * 4, s));
  k_cert_cand<<<dim3((unsigned)((V + 1023) / 1024), (unsigned)M), 1024, 0, s>>>(lh, V, nx, H->cbound, thr, count, cand);
  W12_LAUNCH_CHECK("w12_cert_head_argmax: candidates");
  k_cert_exact<<<dim3(kExactBlocks, (unsigned)M), kExactWarps * 32, 0, s>>>(
      x, K, KC, exact->hi, exact->lo, exact->base, exact->esc_tile_ptr, exact->esc, count, cand, V, W12_DECODE_MUL,
      part);
  W12_LAUNCH_CHECK("w12_cert_head_argmax: exact logits");
  k_cert_final<<<(unsigned)M, 32, 0, s>>>(part, count, tok, ncand);
  W12_LAUNCH_CHECK("w12_cert_head_argmax: final");
  return W12_OK;
}

}  // extern "C"
