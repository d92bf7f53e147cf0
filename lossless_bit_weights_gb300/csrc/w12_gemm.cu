// w12_gemm.cu - decode-fused weight-streaming GEMM for few rows (M <= 32 per
// launch), its 8-bit-view variant, and the LM-head argmax epilogue.
//
// The SpecPilot summary page (onedev.kr/papers/1654), section "What's
// different", describes a GEMM that decodes the 12-bit records in registers,
// hides the decode behind the memory stream and stays deterministic with
// stream-K.  This kernel:
//  - streams each warp's contiguous run of 32x64 weight tiles (2 KB of the
//    front-byte plane + 1 KB of nibbles) with 16-byte L1-bypassing loads,
//    prefetched two tiles ahead;
//  - decodes 16 weights per thread in registers to bf16 (sign, base+offset,
//    mantissa: a shift, two masks, one add, one or), stores them to a
//    swizzled shared tile, and writes the tile's escapes over their slots;
//  - feeds mma.sync m16n8k16 with the weights as the 16-row A operand
//    (ldmatrix) and up to 32 tokens as 8-column B blocks ("swap-AB");
//  - splits the flat list of (row tile, column chunk) iterations evenly over
//    all warps (stream-K).  A warp that owns only part of a row tile writes
//    its partial sums to a fixed slot; the last of that tile's warps to
//    arrive (atomic counter, no waiting) adds the slots in slot order.  The
//    partition depends only on the shape and the device's warp count, so
//    repeated calls give identical bits.
#include <algorithm>
#include <cstdint>
#include <mutex>

#include "w12_internal.cuh"

namespace w12 {
namespace {

constexpr int kWarps = 4;                   // warps per block
constexpr int kWarpSmem = kTileRows * 128;  // decoded 32x64 bf16 tile per warp
constexpr int kMinIters = 6;                // fewest tile iterations per warp
constexpr int kMaxTokens = 32;              // tokens per launch

enum Epi { EPI_STORE = 0, EPI_ARGMAX = 1 };

struct GemmArgs {
  const uint8_t* hi;
  const uint8_t* lo;
  const uint8_t* base;
  const uint32_t* tile_ptr;
  const uint32_t* esc;
  int64_t N, KC, T, W;
  const uint16_t* x;   // [M][ldx] bf16, ldx even, zero past K
  int64_t ldx;
  int M;               // tokens of this launch (<= 8*NB)
  float* y;            // EPI_STORE: y[m*ldy + n]
  int64_t ldy;
  unsigned long long* pbest;  // EPI_ARGMAX: pbest[rt*ldp + tok0 + m]
  int64_t ldp;
  int tok0;
  float* slots;
  uint32_t* counters;
};

struct Stage {
  uint4 h[4];
  uint2 l[4];
  uint32_t ent;
  uint32_t e0, cnt;
};

__device__ __forceinline__ int64_t warp_of_iter(int64_t i, int64_t W, int64_t T) { return ((i + 1) * W - 1) / T; }

template <bool Q8>
__device__ __forceinline__ void issue(Stage& st, const GemmArgs& a, int64_t c, int lane, uint64_t pol,
                                      uint32_t& tp_cur, uint32_t& tp_nxt) {
  const uint8_t* hp = a.hi + c * kHiTileBytes + lane * 16;
#pragma unroll
  for (int q = 0; q < 4; ++q) st.h[q] = ldg_stream16(hp + q * 512, pol);
  if (!Q8) {
    const uint8_t* lp = a.lo + c * kLoTileBytes + lane * 8;
#pragma unroll
    for (int q = 0; q < 4; ++q) st.l[q] = ldg_stream8(lp + q * 256, pol);
  }
  st.e0 = tp_cur;
  st.cnt = tp_nxt - tp_cur;
  st.ent = lane < (int)st.cnt ? __ldg(a.esc + tp_cur + lane) : 0u;
  tp_cur = tp_nxt;
  tp_nxt = (c + 2 <= a.T) ? __ldg(a.tile_ptr + c + 2) : tp_nxt;
}

template <int NB, bool Q8>
__device__ __forceinline__ void compute(Stage& st, const GemmArgs& a, int64_t c, int64_t kx, int64_t seg_end,
                                        int lane, uint32_t sm, const uint32_t base2[4], float acc[2][NB][4],
                                        uint64_t pol, uint32_t& tp_cur, uint32_t& tp_nxt) {
  const int g = lane >> 2, t = lane & 3;
  // B fragments (tokens) for the chunk: b0 = x[tok][k 16s+2t..+1], b1 = +8
  uint32_t bf[4][NB][2];
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    const int tok = nb * 8 + g;
    const uint32_t* xr = reinterpret_cast<const uint32_t*>(a.x + (int64_t)tok * a.ldx + kx) + t;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      bf[s][nb][0] = tok < a.M ? __ldg(xr + 8 * s) : 0u;
      bf[s][nb][1] = tok < a.M ? __ldg(xr + 8 * s + 4) : 0u;
    }
  }
  // decode the four channel groups this thread holds into the shared tile
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t pr[8];
    decode16<Q8>(st.h[q], st.l[q], base2[q], pr);
    const int r = 8 * q + g;
    const uint32_t row = sm + r * 128;
    sts128(row + (((2 * t) ^ g) << 4), pr[0], pr[1], pr[2], pr[3]);
    sts128(row + (((2 * t + 1) ^ g) << 4), pr[4], pr[5], pr[6], pr[7]);
  }
  __syncwarp();
  // escapes overwrite their slots with the exact bf16 value
  if (lane < (int)st.cnt) {
    const uint32_t e = st.ent;
    const int rr = esc_row(e), kk = esc_col(e);
    sts16(sm + rr * 128 + ((((kk >> 3) ^ (rr & 7))) << 4) + (kk & 7) * 2, (uint16_t)esc_raw(e));
  }
  for (uint32_t extra = 32; extra < st.cnt; extra += 32) {
    if (extra + lane < st.cnt) {
      const uint32_t e = __ldg(a.esc + st.e0 + extra + lane);
      const int rr = esc_row(e), kk = esc_col(e);
      sts16(sm + rr * 128 + ((((kk >> 3) ^ (rr & 7))) << 4) + (kk & 7) * 2, (uint16_t)esc_raw(e));
    }
  }
  __syncwarp();
  if (c + 2 < seg_end) issue<Q8>(st, a, c + 2, lane, pol, tp_cur, tp_nxt);
  // tensor-core products: A = weights (ldmatrix), B = tokens
  const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = 16 * h + (mi & 1) * 8 + rr;
      const int chunk = 2 * s + (mi >> 1);
      uint32_t a0, a1, a2, a3;
      ldsm_x4(sm + row * 128 + ((chunk ^ rr) << 4), a0, a1, a2, a3);
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) mma_bf16_16816(acc[h][nb], a0, a1, a2, a3, bf[s][nb][0], bf[s][nb][1]);
    }
  }
  __syncwarp();
}

template <int NB, bool Q8, int EPI>
__global__ void __launch_bounds__(kWarps * 32, 3) k_gemm(const GemmArgs a) {
  __shared__ __align__(128) uint8_t smem[kWarps * kWarpSmem];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t w = (int64_t)blockIdx.x * kWarps + warp;
  if (w >= a.W) return;
  const uint32_t sm = smem_u32(smem + warp * kWarpSmem);
  const uint64_t pol = policy_evict_first();
  const int g = lane >> 2, t = lane & 3;
  const int64_t it1 = (w + 1) * a.T / a.W;
  int64_t it = w * a.T / a.W;

  while (it < it1) {
    const int64_t rt = it / a.KC;
    const int64_t kc0 = it - rt * a.KC;
    const int64_t seg_end = it1 < (rt + 1) * a.KC ? it1 : (rt + 1) * a.KC;
    uint32_t base2[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int64_t n = rt * kTileRows + 8 * q + g;
      const uint32_t b = n < a.N ? (uint32_t)__ldg(a.base + n) : 1u;
      base2[q] = (b << 7) | (b << 23);
    }
    float acc[2][NB][4];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[h][nb][i] = 0.f;

    uint32_t tp_cur = __ldg(a.tile_ptr + it), tp_nxt = __ldg(a.tile_ptr + it + 1);
    Stage sa, sb;
    issue<Q8>(sa, a, it, lane, pol, tp_cur, tp_nxt);
    if (it + 1 < seg_end) issue<Q8>(sb, a, it + 1, lane, pol, tp_cur, tp_nxt);
    for (int64_t c = it; c < seg_end; c += 2) {
      compute<NB, Q8>(sa, a, c, (c - rt * a.KC) * kTileK, seg_end, lane, sm, base2, acc, pol, tp_cur, tp_nxt);
      if (c + 1 < seg_end)
        compute<NB, Q8>(sb, a, c + 1, (c + 1 - rt * a.KC) * kTileK, seg_end, lane, sm, base2, acc, pol, tp_cur,
                        tp_nxt);
    }

    // ---- combine partial row tiles (fixed slot order)
    const bool whole = (kc0 == 0) && (seg_end == (rt + 1) * a.KC);
    bool emit = true;
    if (!whole) {
      const int64_t wf = warp_of_iter(rt * a.KC, a.W, a.T);
      const int64_t wl = warp_of_iter((rt + 1) * a.KC - 1, a.W, a.T);
      const int64_t ncov = wl - wf + 1;
      constexpr int kSlot = 2 * NB * 4 * 32;  // floats per slot
      float4* slot = reinterpret_cast<float4*>(a.slots + (wf + rt + (w - wf)) * kSlot);
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
          slot[(h * NB + nb) * 32 + lane] = make_float4(acc[h][nb][0], acc[h][nb][1], acc[h][nb][2], acc[h][nb][3]);
      __threadfence();
      __syncwarp();
      uint32_t old = 0;
      if (lane == 0) old = atomicAdd(a.counters + rt, 1u);
      old = __shfl_sync(0xFFFFFFFFu, old, 0);
      emit = (int64_t)old == ncov - 1;
      if (emit) {
        __threadfence();
        if (lane == 0) a.counters[rt] = 0u;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[h][nb][i] = 0.f;
        for (int64_t j = 0; j < ncov; ++j) {
          const float4* sj = reinterpret_cast<const float4*>(a.slots + (wf + rt + j) * kSlot);
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
              const float4 v = __ldcg(sj + (h * NB + nb) * 32 + lane);
              acc[h][nb][0] += v.x;
              acc[h][nb][1] += v.y;
              acc[h][nb][2] += v.z;
              acc[h][nb][3] += v.w;
            }
        }
      }
    }

    if (emit) {
      if (EPI == EPI_STORE) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int64_t n = rt * kTileRows + 16 * h + g + 8 * (i >> 1);
              const int tok = nb * 8 + 2 * t + (i & 1);
              if (n < a.N && tok < a.M) a.y[(int64_t)tok * a.ldy + n] = acc[h][nb][i];
            }
      } else {
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            unsigned long long best = 0ull;
            // rows in increasing order: g, g+8, g+16, g+24
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const int64_t n = rt * kTileRows + 16 * h + 8 * hh + g;
                if (n < a.N) {
                  const uint32_t key = (uint32_t)order_key(acc[h][nb][2 * hh + e]) ^ 0x80000000u;
                  const unsigned long long cand =
                      ((unsigned long long)key << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)n);
                  best = cand > best ? cand : best;
                }
              }
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
              const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, best, o);
              best = other > best ? other : best;
            }
            const int tok = nb * 8 + 2 * t + e;
            if (g == 0 && tok < a.M) a.pbest[rt * a.ldp + a.tok0 + tok] = best;
          }
      }
    }
    it = seg_end;
  }
}

// Zero-padded copy of x: xp[m][ldx] with ldx = KC*64.
__global__ void k_pad_x(const uint16_t* __restrict__ x, int64_t M, int64_t K, int64_t ldx, uint16_t* __restrict__ xp) {
  const int64_t total = M * ldx;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = i / ldx, k = i - m * ldx;
    xp[i] = k < K ? x[m * K + k] : (uint16_t)0;
  }
}

// Final argmax over row tiles: one block per token.
__global__ void __launch_bounds__(256) k_argmax_final(const unsigned long long* __restrict__ pbest, int64_t RT,
                                                      int64_t ldp, int32_t* __restrict__ tok) {
  __shared__ unsigned long long red[8];
  const int64_t m = blockIdx.x;
  unsigned long long best = 0ull;
  for (int64_t r = threadIdx.x; r < RT; r += 256) {
    const unsigned long long v = pbest[r * ldp + m];
    best = v > best ? v : best;
  }
  for (int o = 16; o; o >>= 1) {
    const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, best, o);
    best = other > best ? other : best;
  }
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    best = red[0];
    for (int i = 1; i < 8; ++i) best = red[i] > best ? red[i] : best;
    tok[m] = best ? (int32_t)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull)) : -1;
  }
}

// ---------------------------------------------------------------- host side

int device_sms(int* sms) {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lk(mu);
  if (dev < 64 && cached[dev]) {
    *sms = cached[dev];
    return W12_OK;
  }
  int v = 0;
  e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
  if (dev < 64) cached[dev] = v;
  *sms = v;
  return W12_OK;
}

// Warps of the stream-K partition for a T-iteration problem.
int64_t partition_warps(int64_t T, int sms) {
  const int64_t resident = (int64_t)sms * 3 * kWarps;  // 3 blocks of kWarps per SM (launch bounds)
  int64_t w = (T + kMinIters - 1) / kMinIters;
  return std::max<int64_t>(1, std::min(w, resident));
}

inline size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

struct WsLayout {
  size_t counters, slots, xpad, pbest, total;
};

WsLayout ws_layout(int64_t M, int64_t N, int64_t K, bool argmax, int sms) {
  const int64_t RT = row_tiles(N), KC = k_chunks(K), T = RT * KC;
  const int64_t W = partition_warps(T, sms);
  const int64_t Mg = std::min<int64_t>(M, kMaxTokens);
  const int64_t nb = Mg <= 8 ? 1 : Mg <= 16 ? 2 : 4;
  WsLayout L{};
  L.counters = 0;
  size_t off = align256((size_t)RT * 4);
  L.slots = off;
  off = align256(off + (size_t)(RT + W) * (size_t)(2 * nb * 4 * 32) * 4);
  L.xpad = off;
  off = align256(off + (size_t)M * (size_t)(KC * kTileK) * 2);
  L.pbest = off;
  if (argmax) off = align256(off + (size_t)RT * (size_t)M * 8);
  L.total = off;
  return L;
}

template <int NB, bool Q8, int EPI>
int launch_one(const GemmArgs& a, cudaStream_t s) {
  const unsigned blocks = (unsigned)((a.W + kWarps - 1) / kWarps);
  k_gemm<NB, Q8, EPI><<<blocks, kWarps * 32, 0, s>>>(a);
  W12_LAUNCH_CHECK("w12 gemm kernel");
  return W12_OK;
}

template <bool Q8, int EPI>
int launch_nb(int nb, const GemmArgs& a, cudaStream_t s) {
  switch (nb) {
    case 1: return launch_one<1, Q8, EPI>(a, s);
    case 2: return launch_one<2, Q8, EPI>(a, s);
    default: return launch_one<4, Q8, EPI>(a, s);
  }
}

int run_gemm(const uint16_t* x, int64_t M, const w12_matrix* A, float* y, int32_t* tok, bool q8, bool argmax,
             void* ws, size_t ws_bytes, cudaStream_t s, const char* fn) {
  int st = check_matrix(A, !q8, fn);
  if (st) return st;
  if (!x || (!argmax && !y) || (argmax && !tok)) return fail(W12_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (M < 1 || M > (1 << 20)) return fail(W12_ERR_SHAPE, "%s: M=%lld out of range (1..2^20)", fn, (long long)M);
  if (!ws) return fail(W12_ERR_INVALID_ARG, "%s: null workspace", fn);
  int sms = 0;
  if ((st = device_sms(&sms))) return st;
  const WsLayout L = ws_layout(M, A->N, A->K, argmax, sms);
  if (ws_bytes < L.total)
    return fail(W12_ERR_BUFFER_TOO_SMALL, "%s: workspace %zu bytes < %zu required", fn, ws_bytes, L.total);
  const int64_t RT = row_tiles(A->N), KC = k_chunks(A->K), T = RT * KC;
  uint8_t* wsb = static_cast<uint8_t*>(ws);

  const uint16_t* xs = x;
  int64_t ldx = A->K;
  const bool direct = (A->K % kTileK == 0) && (((uintptr_t)x & 3u) == 0);
  if (!direct) {
    ldx = KC * kTileK;
    uint16_t* xp = reinterpret_cast<uint16_t*>(wsb + L.xpad);
    const int64_t total = M * ldx;
    const unsigned blocks = (unsigned)std::min<int64_t>((total + 255) / 256, 4096);
    k_pad_x<<<blocks, 256, 0, s>>>(x, M, A->K, ldx, xp);
    W12_LAUNCH_CHECK("w12 gemm: pad x");
    xs = xp;
  }

  GemmArgs a{};
  a.hi = A->hi;
  a.lo = A->lo;
  a.base = A->base;
  a.tile_ptr = A->esc_tile_ptr;
  a.esc = A->esc;
  a.N = A->N;
  a.KC = KC;
  a.T = T;
  a.W = partition_warps(T, sms);
  a.ldx = ldx;
  a.ldy = A->N;
  a.slots = reinterpret_cast<float*>(wsb + L.slots);
  a.counters = reinterpret_cast<uint32_t*>(wsb + L.counters);
  a.pbest = reinterpret_cast<unsigned long long*>(wsb + L.pbest);
  a.ldp = M;
  for (int64_t m0 = 0; m0 < M; m0 += kMaxTokens) {
    const int Mg = (int)std::min<int64_t>(kMaxTokens, M - m0);
    const int nb = Mg <= 8 ? 1 : Mg <= 16 ? 2 : 4;
    a.x = xs + m0 * ldx;
    a.M = Mg;
    a.tok0 = (int)m0;
    if (!argmax) {
      a.y = y + m0 * A->N;
      st = q8 ? launch_nb<true, EPI_STORE>(nb, a, s) : launch_nb<false, EPI_STORE>(nb, a, s);
    } else {
      st = q8 ? launch_nb<true, EPI_ARGMAX>(nb, a, s) : launch_nb<false, EPI_ARGMAX>(nb, a, s);
    }
    if (st) return st;
  }
  if (argmax) {
    k_argmax_final<<<(unsigned)M, 256, 0, s>>>(a.pbest, RT, M, tok);
    W12_LAUNCH_CHECK("w12 lmhead: final argmax");
  }
  return W12_OK;
}

}  // namespace

// used by w12_verify.cu
int lmhead_argmax_impl(const uint16_t* x, int64_t M, const w12_matrix* head, int32_t* tok, bool q8, void* ws,
                       size_t ws_bytes, cudaStream_t s, const char* fn) {
  return run_gemm(x, M, head, nullptr, tok, q8, true, ws, ws_bytes, s, fn);
}

size_t lmhead_ws_bytes(int64_t M, int64_t V, int64_t K) {
  int sms = 0;
  if (device_sms(&sms)) return 0;
  return ws_layout(M, V, K, true, sms).total;
}

}  // namespace w12

using namespace w12;

extern "C" {

size_t w12_gemm_counter_bytes(int64_t N) { return N >= 1 ? align256((size_t)row_tiles(N) * 4) : 0; }

size_t w12_gemm_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M < 1 || N < 1 || K < 1 || K > kMaxK) return 0;
  int sms = 0;
  if (device_sms(&sms)) return 0;
  return ws_layout(M, N, K, false, sms).total;
}

size_t w12_lmhead_workspace_size(int64_t M, int64_t V, int64_t K) {
  if (M < 1 || V < 1 || K < 1 || K > kMaxK) return 0;
  return lmhead_ws_bytes(M, V, K);
}

int w12_gemm(const uint16_t* x, int64_t M, const w12_matrix* A, float* y, void* ws, size_t ws_bytes, void* stream) {
  return run_gemm(x, M, A, y, nullptr, false, false, ws, ws_bytes, (cudaStream_t)stream, "w12_gemm");
}

int w12_gemm_q8(const uint16_t* x, int64_t M, const w12_matrix* A, float* y, void* ws, size_t ws_bytes,
                void* stream) {
  return run_gemm(x, M, A, y, nullptr, true, false, ws, ws_bytes, (cudaStream_t)stream, "w12_gemm_q8");
}

int w12_lmhead_argmax(const uint16_t* x, int64_t M, const w12_matrix* head, int32_t* tok, void* ws, size_t ws_bytes,
                      void* stream) {
  return run_gemm(x, M, head, nullptr, tok, false, true, ws, ws_bytes, (cudaStream_t)stream, "w12_lmhead_argmax");
}

int w12_lmhead_argmax_q8(const uint16_t* x, int64_t M, const w12_matrix* head, int32_t* tok, void* ws,
                         size_t ws_bytes, void* stream) {
  return run_gemm(x, M, head, nullptr, tok, true, true, ws, ws_bytes, (cudaStream_t)stream, "w12_lmhead_argmax_q8");
}

}  // extern "C"
