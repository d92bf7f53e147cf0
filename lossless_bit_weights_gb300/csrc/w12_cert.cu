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
//   - each candidate's exact logit is recomputed from the lossless W12 form of
//     the same head (decode of one channel; exact products, a float-pair sum),
//     and the largest wins, ties to the lowest index.
#include <cstdint>

#include "w12_internal.cuh"

namespace w12 {

int i8_gemm_impl(const uint16_t* x, int64_t M, const uint8_t* codes, const float* scale, int64_t V, int64_t K,
                 const float* nx, const float* cb, uint32_t* thr_key, uint32_t* sup_count, uint2* sup,
                 int64_t ldsup, void* ws, size_t ws_bytes, cudaStream_t s, const char* fn);

namespace {

constexpr int kFilterBlocks = 16;  // blocks per row of the candidate filter
constexpr int kExactPerSM = 12;    // blocks per SM of the exact recompute
constexpr int kExactWarps = 5;     // 5 x 8 chunks a round: K = 5120 in two

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

// nx[m] >= ||x_m||: every square and every addition rounds
// up, so the sum (and its square root, rounded up) bound the norm from above.  Also zeroes
// the row's threshold key and counters for the GEMM's epilogue and the exact recompute.
__global__ void __launch_bounds__(256) k_cert_prep(const uint16_t* __restrict__ x, int64_t K, float* __restrict__ nx,
                                                   uint32_t* __restrict__ thr_key, int32_t* __restrict__ count,
                                                   uint32_t* __restrict__ sup_count, uint32_t* __restrict__ n_list) {
  // the GEMM that follows may start streaming its weights; it reads nothing of ours
  // before its griddepcontrol.wait
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ float shf[32];
  const uint16_t* xr = x + (int64_t)blockIdx.x * K;
  float a = 0.f;
  for (int64_t k = threadIdx.x; k < K; k += blockDim.x) {
    const float f = bf16f(xr[k]);
    a = __fadd_ru(a, __fmul_ru(f, f));
  }
  for (int o = 16; o > 0; o >>= 1) a = __fadd_ru(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
  if ((threadIdx.x & 31) == 0) shf[threadIdx.x >> 5] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t = __fadd_ru(t, shf[w]);
    nx[blockIdx.x] = __fsqrt_ru(t);
    thr_key[blockIdx.x] = 0u;
    count[blockIdx.x] = 0;
    sup_count[blockIdx.x] = 0u;
    if (blockIdx.x == 0) *n_list = 0u;
  }
}

// Inverse of the GEMM epilogue's order-preserving key (larger float, larger key).
__device__ __forceinline__ float fkey_inv(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

struct Best {
  double val;
  int32_t idx;  // -1: none
};

// Error-free float addition (Knuth's TwoSum): s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// (hi, lo) += p with the rounding error of the high part carried in lo.
__device__ __forceinline__ void acc2(float& hi, float& lo, float p) {
  float e;
  two_sum(hi, p, hi, e);
  lo = __fadd_rn(lo, e);
}

__device__ __forceinline__ bool beats(double a, int32_t ia, double b, int32_t ib) {
  if (ia < 0) return false;
  if (ib < 0) return true;
  return a > b || (a == b && ia < ib);
}

// Candidates: the superset entries of row m whose upper bound reaches the row's final
// threshold, appended to one list over all rows (entry: row, channel; the order varies
// from call to call, the set does not).  count[m] and *n_list are zero beforehand.
__global__ void __launch_bounds__(256) k_cert_filter(const uint32_t* __restrict__ thr_key,
                                                     const uint32_t* __restrict__ sup_count,
                                                     const uint2* __restrict__ sup, int64_t ldsup,
                                                     int32_t* __restrict__ count, uint2* __restrict__ list,
                                                     uint32_t* __restrict__ n_list) {
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the INT8 GEMM has completed
  const int64_t m = blockIdx.y;
  const int lane = threadIdx.x & 31;
  const uint32_t n_sup = min(sup_count[m], (uint32_t)ldsup);
  const float thr = fkey_inv(thr_key[m]);
  for (uint32_t e0 = blockIdx.x * blockDim.x; e0 < n_sup; e0 += gridDim.x * blockDim.x) {
    const uint32_t e = e0 + threadIdx.x;
    bool keep = false;
    uint32_t v = 0u;
    if (e < n_sup) {
      const uint2 ent = sup[m * ldsup + e];
      keep = fkey_inv(ent.y) >= thr;
      v = ent.x;
    }
    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, keep);
    if (bal) {
      uint32_t p0 = 0u;
      if (lane == 0) {
        p0 = atomicAdd(n_list, (uint32_t)__popc(bal));
        atomicAdd(count + m, __popc(bal));
      }
      p0 = __shfl_sync(0xFFFFFFFFu, p0, 0);
      if (keep) list[p0 + (uint32_t)__popc(bal & ((1u << lane) - 1u))] = make_uint2((uint32_t)m, v);
    }
  }
}

// Exact logits of the listed candidates from the W12 head, val[i] for list entry i.  The
// blocks take the entries i = b, b + gridDim.x, ... (a grid of a few blocks per SM keeps
// every SM busy whatever the rows' candidate counts); the whole block computes one
// candidate: lane 4*c8 + t of warp w decodes the 16 columns 16t.. of chunks w*8 + c8 + 40i
// (the same decode as the GEMM) and patches the channel's escapes in them.  A product of
// two bf16 values is exact in float; the sum is a float pair (TwoSum), whose error is near
// 2^-48 of sum|x*w|, far inside the argmax's tie tolerance and on the full-rate float pipe
// (float64 runs at a small fraction of it on this GPU).
__global__ void __launch_bounds__(kExactWarps * 32)
    k_cert_exact(const uint16_t* __restrict__ x, int64_t K, int64_t KC, const uint8_t* __restrict__ hi,
                 const uint8_t* __restrict__ lo, const uint8_t* __restrict__ base, const uint32_t* __restrict__ tile_ptr,
                 const uint32_t* __restrict__ esc, const uint2* __restrict__ list, const uint32_t* __restrict__ n_list,
                 uint32_t cap, DecodeMul mul, double* __restrict__ val) {
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the candidate list is complete
  __shared__ float shh[kExactWarps], shl[kExactWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c8 = lane >> 2, t = lane & 3;
  const uint32_t n = min(*n_list, cap);
  for (uint32_t i = blockIdx.x; i < n; i += gridDim.x) {
    const uint2 ent = list[i];
    const int64_t m = ent.x, v = ent.y;
    const uint16_t* xr = x + m * K;
    const int64_t rt = v / kTileRows;
    const int r = (int)(v % kTileRows), q = r >> 3, g = r & 7;
    const uint32_t bb = base[v];
    const uint32_t base2 = (bb << 7) | (bb << 23);
    float ah = 0.f, al = 0.f;
    for (int64_t kc = warp * 8 + c8; kc < KC; kc += kExactWarps * 8) {
      const int64_t tile = tile_index(rt, kc, KC);
      const uint4 hq = *reinterpret_cast<const uint4*>(hi + tile * kHiTileBytes + q * 512 + (4 * g + t) * 16);
      const uint2 lq = *reinterpret_cast<const uint2*>(lo + tile * kLoTileBytes + q * 256 + (4 * g + t) * 8);
      const uint32_t e0 = tile_ptr[tile], e1 = tile_ptr[tile + 1];
      uint32_t pr[8];
      decode16<false>(hq, lq, base2, mul, pr);
      uint16_t w[16];
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        w[2 * p] = (uint16_t)(pr[p] & 0xFFFFu);
        w[2 * p + 1] = (uint16_t)(pr[p] >> 16);
      }
      // the tile's escapes, four independent loads at a time
      for (uint32_t e = e0; e < e1; e += 4) {
        uint32_t ent4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) ent4[u] = e + u < e1 ? esc[e + u] : 0xFFFFFFFFu;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = esc_col(ent4[u]);
          if (ent4[u] != 0xFFFFFFFFu && esc_row(ent4[u]) == r && (c >> 4) == t) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (j == (c & 15)) w[j] = (uint16_t)esc_raw(ent4[u]);
          }
        }
      }
      const int64_t k0 = kc * kTileK + 16 * t;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (k0 + j < K) acc2(ah, al, __fmul_rn(bf16f(xr[k0 + j]), bf16f(w[j])));
    }
    for (int o = 16; o > 0; o >>= 1) {
      const float oh = __shfl_xor_sync(0xFFFFFFFFu, ah, o), ol = __shfl_xor_sync(0xFFFFFFFFu, al, o);
      acc2(ah, al, oh);
      al = __fadd_rn(al, ol);
    }
    if (lane == 0) {
      shh[warp] = ah;
      shl[warp] = al;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      float h = shh[0], l = shl[0];
      for (int w2 = 1; w2 < kExactWarps; ++w2) {
        acc2(h, l, shh[w2]);
        l = __fadd_rn(l, shl[w2]);
      }
      val[i] = (double)h + (double)l;
    }
    __syncthreads();
  }
}

// One block of 256 per row: its threads scan the candidate list for the row's entries and
// keep the largest exact logit (lowest channel on ties), then the warps and the block
// merge; the result does not depend on the list's order.
__global__ void __launch_bounds__(256) k_cert_final(const uint2* __restrict__ list, const double* __restrict__ val,
                                                    const uint32_t* __restrict__ n_list, uint32_t cap,
                                                    const int32_t* __restrict__ count, int32_t* __restrict__ tok,
                                                    int32_t* __restrict__ ncand) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the exact recompute has completed
  __shared__ Best sh[8];
  const uint32_t m = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t n = min(*n_list, cap);
  Best b{0.0, -1};
  for (uint32_t i = threadIdx.x; i < n; i += 256) {
    const uint2 ent = list[i];
    if (ent.x == m && beats(val[i], (int32_t)ent.y, b.val, b.idx)) b = Best{val[i], (int32_t)ent.y};
  }
  for (int o = 16; o > 0; o >>= 1) {
    const double ov = __shfl_xor_sync(0xFFFFFFFFu, b.val, o);
    const int32_t oi = __shfl_xor_sync(0xFFFFFFFFu, b.idx, o);
    if (beats(ov, oi, b.val, b.idx)) b = Best{ov, oi};
  }
  if (lane == 0) sh[warp] = b;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < 8; ++w)
      if (beats(sh[w].val, sh[w].idx, b.val, b.idx)) b = sh[w];
    tok[m] = b.idx;
    if (ncand) ncand[m] = count[m];
  }
}

struct CertWs {
  size_t gemm, nx, thr, count, sup_count, n_list, sup, list, val, total;
};

// A row's candidate superset, and the candidate list over all rows, hold at most one entry
// per channel and row: M x V entries each.
CertWs cert_ws(int64_t M, int64_t V, int64_t K) {
  CertWs L{};
  L.gemm = 0;
  size_t off = al256(w12_gemm_workspace_size(M, V, K));
  L.nx = off;
  off = al256(off + (size_t)M * 4);
  L.thr = off;
  off = al256(off + (size_t)M * 4);
  L.count = off;
  off = al256(off + (size_t)M * 4);
  L.sup_count = off;
  off = al256(off + (size_t)M * 4);
  L.n_list = off;
  off = al256(off + 4);
  L.sup = off;
  off = al256(off + (size_t)M * (size_t)V * 8);
  L.list = off;
  off = al256(off + (size_t)M * (size_t)V * 8);
  L.val = off;
  off = al256(off + (size_t)M * (size_t)V * 8);
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
  float* nx = reinterpret_cast<float*>(w + L.nx);
  uint32_t* thr = reinterpret_cast<uint32_t*>(w + L.thr);
  int32_t* count = reinterpret_cast<int32_t*>(w + L.count);
  uint32_t* sup_count = reinterpret_cast<uint32_t*>(w + L.sup_count);
  uint32_t* n_list = reinterpret_cast<uint32_t*>(w + L.n_list);
  uint2* sup = reinterpret_cast<uint2*>(w + L.sup);
  uint2* list = reinterpret_cast<uint2*>(w + L.list);
  double* val = reinterpret_cast<double*>(w + L.val);
  const uint32_t cap = (uint32_t)std::min<int64_t>(M * V, 0xFFFFFFFFll);
  static int sms_of[64] = {0};
  int dev = 0;
  W12_CUDA_TRY(cudaGetDevice(&dev));
  int sms = dev < 64 ? sms_of[dev] : 0;
  if (sms == 0) {
    W12_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    if (dev < 64) sms_of[dev] = sms;
  }
  // row norms; zero thresholds and counters
  k_cert_prep<<<(unsigned)M, 256, 0, s>>>(x, K, nx, thr, count, sup_count, n_list);
  W12_LAUNCH_CHECK("w12_cert_head_argmax: row norms");
  // approximate logits s_v * x.q_v -> thresholds and the candidate superset
  if ((st = i8_gemm_impl(x, M, H->code, H->scale, V, K, nx, H->cbound, thr, sup_count, sup, V, w + L.gemm, L.nx, s,
                         fn)))
    return st;
  // The filter is launched plainly: launched early, its blocks would wait beside the GEMM's
  // CTAs and slow them.  The two kernels after it start early (programmatic dependent
  // launch) and wait for their predecessor's grid before reading its results.
  k_cert_filter<<<dim3(kFilterBlocks, (unsigned)M), 256, 0, s>>>(thr, sup_count, sup, (int64_t)V, count, list, n_list);
  W12_LAUNCH_CHECK("w12_cert_head_argmax: candidates");
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3((unsigned)(kExactPerSM * sms));
  cfg.blockDim = dim3(kExactWarps * 32);
  W12_CUDA_TRY(cudaLaunchKernelEx(&cfg, k_cert_exact, x, K, KC, (const uint8_t*)exact->hi, (const uint8_t*)exact->lo,
                                  (const uint8_t*)exact->base, (const uint32_t*)exact->esc_tile_ptr,
                                  (const uint32_t*)exact->esc, (const uint2*)list, (const uint32_t*)n_list, cap,
                                  W12_DECODE_MUL, val));
  W12_LAUNCH_CHECK("w12_cert_head_argmax: exact logits");
  cfg.gridDim = dim3((unsigned)M);
  cfg.blockDim = dim3(256);
  W12_CUDA_TRY(cudaLaunchKernelEx(&cfg, k_cert_final, (const uint2*)list, (const double*)val, (const uint32_t*)n_list,
                                  cap, (const int32_t*)count, tok, ncand));
  W12_LAUNCH_CHECK("w12_cert_head_argmax: final");
  return W12_OK;
}

}  // extern "C"
