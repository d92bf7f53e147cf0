// w12_codec.cu - W12 encoder, decoders and canonical export (device side).
//
// W12 as the SpecPilot summary page (onedev.kr/papers/1654), section "What's
// different", defines it: per channel the 16-binade window holding the most
// weights; in-window values as 1 sign / 4 exponent-offset / 7 mantissa bits;
// everything else (out-of-window, zeros, denormals) exact in a per-channel
// escape list.  The device layout (tiles of 32 channels x 64 columns) is the
// one include/w12.h documents.
#include <algorithm>
#include <cstdint>

#include "w12_internal.cuh"

namespace w12 {
namespace {

__device__ __forceinline__ int expo(uint32_t w) { return (int)((w >> 7) & 0xFFu); }

__device__ __forceinline__ bool in_window(uint32_t w, int base) {
  int E = expo(w);
  return E >= 1 && E <= 254 && E >= base && E <= base + 15;
}

// ---------------------------------------------------------------- window choice

// One block per channel: exponent histogram over normal values, then the first
// base in 1..239 with the largest count of exponents in [base, base+15].
__global__ void __launch_bounds__(256) k_window(const uint16_t* __restrict__ W, int64_t N, int64_t K, bool vec,
                                                uint8_t* __restrict__ base) {
  __shared__ uint32_t hist[8][256];
  __shared__ unsigned long long best[8];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t n = blockIdx.x;
  for (int i = tid; i < 8 * 256; i += 256) (&hist[0][0])[i] = 0;
  __syncthreads();
  const uint16_t* row = W + n * K;
  if (vec) {
    const uint4* r4 = reinterpret_cast<const uint4*>(row);
    for (int64_t i = tid; i < K / 8; i += 256) {
      uint4 v = r4[i];
      uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        int e0 = expo(u[h] & 0xFFFFu), e1 = expo(u[h] >> 16);
        if (e0 >= 1 && e0 <= 254) atomicAdd(&hist[warp][e0], 1u);
        if (e1 >= 1 && e1 <= 254) atomicAdd(&hist[warp][e1], 1u);
      }
    }
  } else {
    for (int64_t k = tid; k < K; k += 256) {
      int e = expo(row[k]);
      if (e >= 1 && e <= 254) atomicAdd(&hist[warp][e], 1u);
    }
  }
  __syncthreads();
  {
    uint32_t s = 0;
    for (int w = 0; w < 8; ++w) s += hist[w][tid];
    __syncthreads();
    hist[0][tid] = s;
  }
  __syncthreads();
  unsigned long long key = 0;
  if (tid >= 1 && tid <= 239) {
    uint32_t c = 0;
    for (int E = tid; E <= tid + 15; ++E) c += hist[0][E];
    key = ((unsigned long long)c << 32) | (0xFFFFFFFFu - (uint32_t)tid);  // more values, then lower base
  }
  for (int o = 16; o; o >>= 1) {
    unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, key, o);
    key = other > key ? other : key;
  }
  if (lane == 0) best[warp] = key;
  __syncthreads();
  if (tid == 0) {
    unsigned long long k = best[0];
    for (int w = 1; w < 8; ++w) k = best[w] > k ? best[w] : k;
    base[n] = (uint8_t)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFu));
  }
}

// Loads the 64 values of channel n in column chunk kc (zeros past K).
__device__ __forceinline__ void load_chunk(const uint16_t* __restrict__ W, int64_t N, int64_t K, bool vec, int64_t n,
                                           int64_t kc, uint32_t v[32]) {
  const int64_t k0 = kc * kTileK;
  if (n >= N) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0;
    return;
  }
  const uint16_t* row = W + n * K;
  if (vec && k0 + kTileK <= K) {
    const uint4* r4 = reinterpret_cast<const uint4*>(row + k0);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint4 q = r4[i];
      v[4 * i] = q.x;
      v[4 * i + 1] = q.y;
      v[4 * i + 2] = q.z;
      v[4 * i + 3] = q.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      int64_t k = k0 + 2 * i;
      uint32_t a = k < K ? row[k] : 0u, b = k + 1 < K ? row[k + 1] : 0u;
      v[i] = a | (b << 16);
    }
  }
}

// ---------------------------------------------------------------- escape counts per tile

__global__ void __launch_bounds__(256) k_tile_count(const uint16_t* __restrict__ W, int64_t N, int64_t K, bool vec,
                                                    const uint8_t* __restrict__ base, int64_t KC, int64_t T,
                                                    uint32_t* __restrict__ tile_ptr) {
  const int lane = threadIdx.x & 31;
  const int64_t tile = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (blockIdx.x == 0 && threadIdx.x == 0) tile_ptr[T] = 0;
  if (tile >= T) return;
  int64_t rt, kc;
  tile_coords(tile, KC, rt, kc);
  const int64_t n = rt * kTileRows + lane;
  uint32_t v[32];
  load_chunk(W, N, K, vec, n, kc, v);
  uint32_t c = 0;
  if (n < N) {
    const int b = base[n];
    const int64_t k0 = kc * kTileK;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (k0 + 2 * i < K && !in_window(v[i] & 0xFFFFu, b)) ++c;
      if (k0 + 2 * i + 1 < K && !in_window(v[i] >> 16, b)) ++c;
    }
  }
  for (int o = 16; o; o >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
  if (lane == 0) tile_ptr[tile] = c;
}

// ---------------------------------------------------------------- exclusive scan (one block)

__global__ void __launch_bounds__(1024) k_exclusive_scan(uint32_t* __restrict__ a, int64_t n) {
  __shared__ uint32_t warp_tot[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t per = (n + 1023) / 1024;
  const int64_t lo = tid * per, hi = lo + per < n ? lo + per : n;
  uint32_t s = 0;
  for (int64_t i = lo; i < hi; ++i) s += a[i];
  uint32_t incl = s;
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = warp_tot[lane];
    uint32_t wi = w;
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t t = __shfl_up_sync(0xFFFFFFFFu, wi, o);
      if (lane >= o) wi += t;
    }
    warp_tot[lane] = wi - w;
  }
  __syncthreads();
  uint32_t run = warp_tot[warp] + incl - s;
  for (int64_t i = lo; i < hi; ++i) {
    uint32_t x = a[i];
    a[i] = run;
    run += x;
  }
}

// ---------------------------------------------------------------- pack records and escapes

__global__ void __launch_bounds__(256) k_pack(const uint16_t* __restrict__ W, int64_t N, int64_t K, bool vec,
                                              const uint8_t* __restrict__ base, int64_t KC, int64_t T,
                                              const uint32_t* __restrict__ tile_ptr, uint8_t* __restrict__ hi,
                                              uint8_t* __restrict__ lo, uint32_t* __restrict__ esc) {
  const int lane = threadIdx.x & 31;
  const int64_t tile = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (tile >= T) return;
  int64_t rt, kc;
  tile_coords(tile, KC, rt, kc);
  const int64_t n = rt * kTileRows + lane;
  const int64_t k0 = kc * kTileK;
  uint32_t v[32];
  load_chunk(W, N, K, vec, n, kc, v);
  const int b = n < N ? base[n] : 1;
  // records and escape flags, column order
  uint32_t rec[32];        // two 12-bit records per word
  uint64_t escmask = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    uint32_t r2 = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t w = h ? (v[i] >> 16) : (v[i] & 0xFFFFu);
      const bool valid = n < N && k0 + 2 * i + h < K;
      uint32_t r = 0;
      if (valid) {
        if (in_window(w, b)) {
          r = (((w >> 15) & 1u) << 11) | ((uint32_t)(expo(w) - b) << 7) | (w & 0x7Fu);
        } else {
          escmask |= 1ull << (2 * i + h);
        }
      }
      r2 |= r << (16 * h);
    }
    rec[i] = r2;
  }
  const int q = lane >> 3, g = lane & 7;
  uint8_t* htile = hi + tile * kHiTileBytes;
  uint8_t* ltile = lo + tile * kLoTileBytes;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    uint32_t hw[4] = {0, 0, 0, 0};
    uint32_t lw[2] = {0, 0};
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int kk = 16 * t + j;
      const uint32_t r = (rec[kk >> 1] >> (16 * (kk & 1))) & 0xFFFu;
      const int u = j & 3;
      const int pos = (j & ~3) | (u == 1 ? 2 : u == 2 ? 1 : u);
      hw[pos >> 2] |= (r >> 4) << (8 * (pos & 3));
      const int p = 2 * (j >> 2) + ((j & 3) >> 1);
      const int bit = 4 * (p & 3) + 16 * (j & 1);
      lw[p >> 2] |= (r & 0xFu) << bit;
    }
    *reinterpret_cast<uint4*>(htile + q * 512 + (4 * g + t) * 16) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint2*>(ltile + q * 256 + (4 * g + t) * 8) = make_uint2(lw[0], lw[1]);
  }
  // escapes: tile-contiguous, ordered by (channel, column)
  const uint32_t cnt = (uint32_t)__popcll(escmask);
  uint32_t incl = cnt;
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  uint32_t off = tile_ptr[tile] + incl - cnt;
  while (escmask) {
    const int kk = __ffsll((long long)escmask) - 1;
    escmask &= escmask - 1;
    const uint32_t w = (v[kk >> 1] >> (16 * (kk & 1))) & 0xFFFFu;
    esc[off++] = esc_entry(lane, kk, w);
  }
}

// ---------------------------------------------------------------- decode

template <bool Q8>
__global__ void __launch_bounds__(256) k_decode(const uint8_t* __restrict__ hi, const uint8_t* __restrict__ lo,
                                                const uint8_t* __restrict__ base, const uint32_t* __restrict__ tile_ptr,
                                                const uint32_t* __restrict__ esc, int64_t N, int64_t K, int64_t KC,
                                                int64_t T, bool vec, uint16_t* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int64_t tile = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (tile >= T) return;
  int64_t rt, kc;
  tile_coords(tile, KC, rt, kc);
  const int64_t n = rt * kTileRows + lane;
  const int64_t k0 = kc * kTileK;
  const int q = lane >> 3, g = lane & 7;
  if (n < N) {
    const uint32_t b = base[n];
    const uint32_t base2 = (b << 7) | (b << 23);
    uint16_t* row = out + n * K;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint4 h = *reinterpret_cast<const uint4*>(hi + tile * kHiTileBytes + q * 512 + (4 * g + t) * 16);
      uint2 l = make_uint2(0, 0);
      if (!Q8) l = *reinterpret_cast<const uint2*>(lo + tile * kLoTileBytes + q * 256 + (4 * g + t) * 8);
      uint32_t pr[8];
      decode16<Q8>(h, l, base2, W12_DECODE_MUL, pr);
      const int64_t kb = k0 + 16 * t;
      if (vec && kb + 16 <= K) {
        uint4* dst = reinterpret_cast<uint4*>(row + kb);
        dst[0] = make_uint4(pr[0], pr[1], pr[2], pr[3]);
        dst[1] = make_uint4(pr[4], pr[5], pr[6], pr[7]);
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (kb + j < K) row[kb + j] = (uint16_t)(pr[j >> 1] >> (16 * (j & 1)));
      }
    }
  }
  __syncwarp();
  const uint32_t e0 = tile_ptr[tile], e1 = tile_ptr[tile + 1];
  for (uint32_t e = e0 + lane; e < e1; e += 32) {
    const uint32_t ent = esc[e];
    const int64_t nn = rt * kTileRows + esc_row(ent);
    const int64_t kk = k0 + esc_col(ent);
    if (nn < N && kk < K) out[nn * K + kk] = (uint16_t)esc_raw(ent);
  }
}

// ---------------------------------------------------------------- canonical export

__global__ void __launch_bounds__(256) k_export_planes(const uint8_t* __restrict__ hi, const uint8_t* __restrict__ lo,
                                                       int64_t N, int64_t K, int64_t KC, int64_t T,
                                                       uint8_t* __restrict__ hi_out, uint8_t* __restrict__ lo_out) {
  const int lane = threadIdx.x & 31;
  const int64_t tile = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (tile >= T) return;
  int64_t rt, kc;
  tile_coords(tile, KC, rt, kc);
  const int64_t n = rt * kTileRows + lane;
  if (n >= N) return;
  const int64_t lo_row = (K + 1) / 2;
  const uint8_t* ht = hi + tile * kHiTileBytes;
  const uint8_t* lt = lo + tile * kLoTileBytes;
  for (int kk = 0; kk < kTileK; kk += 2) {
    const int64_t k = kc * kTileK + kk;
    if (k >= K) break;
    uint8_t byte = 0;
    for (int h = 0; h < 2 && k + h < K; ++h) {
      hi_out[n * K + k + h] = ht[hi_offset(lane, kk + h)];
      const int bit = lo_bit(lane, kk + h);
      const uint32_t nib = (lt[bit >> 3] >> (bit & 7)) & 0xFu;
      byte |= (uint8_t)(nib << (4 * h));
    }
    lo_out[n * lo_row + k / 2] = byte;
  }
}

// One warp per row tile; lane = channel.  pass 0 counts escapes per channel
// into rowptr[n]; pass 1 writes them in column order at rowptr[n].
__global__ void __launch_bounds__(256) k_export_esc(const uint32_t* __restrict__ tile_ptr,
                                                    const uint32_t* __restrict__ esc, int64_t N, int64_t RT, int64_t KC,
                                                    int pass, uint32_t* __restrict__ rowptr, uint32_t* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int64_t rt = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (blockIdx.x == 0 && threadIdx.x == 0 && pass == 0) rowptr[N] = 0;
  if (rt >= RT) return;
  const int64_t n = rt * kTileRows + lane;
  uint32_t off = (pass == 1 && n < N) ? rowptr[n] : 0;
  uint32_t cnt = 0;
  for (int64_t kc = 0; kc < KC; ++kc) {
    const int64_t tile = tile_index(rt, kc, KC);
    const uint32_t e0 = tile_ptr[tile], e1 = tile_ptr[tile + 1];
    for (uint32_t e = e0; e < e1; ++e) {
      const uint32_t ent = esc[e];
      if (esc_row(ent) != lane) continue;
      if (pass == 1) out[off++] = ((uint32_t)(kc * kTileK + esc_col(ent)) << 16) | esc_raw(ent);
      ++cnt;
    }
  }
  if (pass == 0 && n < N) rowptr[n] = cnt;
}

// ---------------------------------------------------------------- index validation

// One thread per tile, then one per channel.  A tile's escape offsets must rise, start at
// 0 and end at n_esc; each entry must lie within the list, name an even byte slot of the
// 32x64 tile image, a real weight (channel < N, column < K), and come after the previous
// entry of its tile in (channel, column) order.  Every window base must be in 1..239.  Any
// violation sets *status to W12_ERR_BOUNDS; only offsets within 0..n_esc are dereferenced.
__global__ void __launch_bounds__(256) k_validate(const uint32_t* __restrict__ tile_ptr, const uint32_t* __restrict__ esc,
                                                  const uint8_t* __restrict__ base, int64_t N, int64_t K, int64_t KC,
                                                  int64_t T, uint32_t n_esc, int32_t* __restrict__ status) {
  bool bad = false;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < T; t += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t e0 = tile_ptr[t], e1 = tile_ptr[t + 1];
    if ((t == 0 && e0 != 0u) || (t == T - 1 && e1 != n_esc) || e1 < e0 || e1 > n_esc) {
      bad = true;
      continue;
    }
    int64_t rt, kc;
    tile_coords(t, KC, rt, kc);
    int prev = -1;
    for (uint32_t e = e0; e < e1; ++e) {
      const uint32_t ent = esc[e], slot = esc_slot(ent);
      const int rr = esc_row(ent), kk = esc_col(ent), key = rr * kTileK + kk;
      if ((slot & 1u) || slot >= 4096u || rt * kTileRows + rr >= N || kc * kTileK + kk >= K || key <= prev) {
        bad = true;
        break;
      }
      prev = key;
    }
  }
  for (int64_t n = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; n < N; n += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t b = base[n];
    if (b < 1u || b > 239u) bad = true;
  }
  if (bad) *status = W12_ERR_BOUNDS;
}

inline unsigned blocks_for(int64_t warps) { return (unsigned)((warps + 7) / 8); }

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace
}  // namespace w12

using namespace w12;

extern "C" {

int w12_encode_plan(const uint16_t* W, int64_t N, int64_t K, uint8_t* base, uint32_t* esc_tile_ptr, int64_t* n_esc,
                    void* stream) {
  if (!W || !base || !esc_tile_ptr || !n_esc) return fail(W12_ERR_INVALID_ARG, "w12_encode_plan: null pointer");
  if (N < 1 || K < 1 || K > kMaxK || (uint64_t)N * (uint64_t)K > 0xFFFFFFFFull)
    return fail(W12_ERR_SHAPE, "w12_encode_plan: N=%lld K=%lld out of range (1<=K<=65535, N*K<2^32)", (long long)N,
                (long long)K);
  cudaStream_t s = (cudaStream_t)stream;
  const bool vec = (K % 8 == 0) && aligned16(W);
  const int64_t KC = k_chunks(K), T = row_tiles(N) * KC;
  k_window<<<(unsigned)N, 256, 0, s>>>(W, N, K, vec, base);
  W12_LAUNCH_CHECK("w12_encode_plan: window kernel");
  k_tile_count<<<blocks_for(T), 256, 0, s>>>(W, N, K, vec, base, KC, T, esc_tile_ptr);
  W12_LAUNCH_CHECK("w12_encode_plan: count kernel");
  k_exclusive_scan<<<1, 1024, 0, s>>>(esc_tile_ptr, T + 1);
  W12_LAUNCH_CHECK("w12_encode_plan: scan kernel");
  uint32_t total = 0;
  W12_CUDA_TRY(cudaMemcpyAsync(&total, esc_tile_ptr + T, sizeof(uint32_t), cudaMemcpyDeviceToHost, s));
  W12_CUDA_TRY(cudaStreamSynchronize(s));
  *n_esc = (int64_t)total;
  return W12_OK;
}

int w12_encode(const uint16_t* W, const w12_matrix* A, void* stream) {
  if (!W) return fail(W12_ERR_INVALID_ARG, "w12_encode: null W");
  int st = check_matrix(A, true, "w12_encode");
  if (st) return st;
  if ((uint64_t)A->N * (uint64_t)A->K > 0xFFFFFFFFull) return fail(W12_ERR_SHAPE, "w12_encode: N*K >= 2^32");
  cudaStream_t s = (cudaStream_t)stream;
  const bool vec = (A->K % 8 == 0) && aligned16(W);
  const int64_t KC = k_chunks(A->K), T = row_tiles(A->N) * KC;
  k_pack<<<blocks_for(T), 256, 0, s>>>(W, A->N, A->K, vec, A->base, KC, T, A->esc_tile_ptr, A->hi, A->lo, A->esc);
  W12_LAUNCH_CHECK("w12_encode: pack kernel");
  return W12_OK;
}

static int decode_common(const w12_matrix* A, uint16_t* out, void* stream, bool q8, const char* fn) {
  if (!out) return fail(W12_ERR_INVALID_ARG, "%s: null output", fn);
  int st = check_matrix(A, !q8, fn);
  if (st) return st;
  cudaStream_t s = (cudaStream_t)stream;
  const bool vec = (A->K % 8 == 0) && aligned16(out);
  const int64_t KC = k_chunks(A->K), T = row_tiles(A->N) * KC;
  if (q8)
    k_decode<true><<<blocks_for(T), 256, 0, s>>>(A->hi, A->lo, A->base, A->esc_tile_ptr, A->esc, A->N, A->K, KC, T, vec,
                                                 out);
  else
    k_decode<false><<<blocks_for(T), 256, 0, s>>>(A->hi, A->lo, A->base, A->esc_tile_ptr, A->esc, A->N, A->K, KC, T,
                                                  vec, out);
  W12_LAUNCH_CHECK(fn);
  return W12_OK;
}

int w12_decode(const w12_matrix* A, uint16_t* W_out, void* stream) {
  return decode_common(A, W_out, stream, false, "w12_decode");
}

int w12_decode_q8(const w12_matrix* A, uint16_t* W_out, void* stream) {
  return decode_common(A, W_out, stream, true, "w12_decode_q8");
}

int w12_export_canonical(const w12_matrix* A, uint8_t* hi_out, uint8_t* lo_out, uint32_t* rowptr_out,
                         uint32_t* esc_out, void* stream) {
  int st = check_matrix(A, true, "w12_export_canonical");
  if (st) return st;
  if (!hi_out || !lo_out || !rowptr_out || (A->n_esc > 0 && !esc_out))
    return fail(W12_ERR_INVALID_ARG, "w12_export_canonical: null output");
  cudaStream_t s = (cudaStream_t)stream;
  const int64_t RT = row_tiles(A->N), KC = k_chunks(A->K), T = RT * KC;
  k_export_planes<<<blocks_for(T), 256, 0, s>>>(A->hi, A->lo, A->N, A->K, KC, T, hi_out, lo_out);
  W12_LAUNCH_CHECK("w12_export_canonical: planes");
  k_export_esc<<<blocks_for(RT), 256, 0, s>>>(A->esc_tile_ptr, A->esc, A->N, RT, KC, 0, rowptr_out, esc_out);
  W12_LAUNCH_CHECK("w12_export_canonical: count");
  k_exclusive_scan<<<1, 1024, 0, s>>>(rowptr_out, A->N + 1);
  W12_LAUNCH_CHECK("w12_export_canonical: scan");
  if (A->n_esc > 0) {
    k_export_esc<<<blocks_for(RT), 256, 0, s>>>(A->esc_tile_ptr, A->esc, A->N, RT, KC, 1, rowptr_out, esc_out);
    W12_LAUNCH_CHECK("w12_export_canonical: fill");
  }
  return W12_OK;
}

int w12_validate(const w12_matrix* A, int32_t* status, void* stream) {
  const char* fn = "w12_validate";
  int st = check_matrix(A, false, fn);
  if (st) return st;
  if (!status) return fail(W12_ERR_INVALID_ARG, "%s: null status", fn);
  cudaStream_t s = (cudaStream_t)stream;
  const int64_t KC = k_chunks(A->K), T = row_tiles(A->N) * KC;
  W12_CUDA_TRY(cudaMemsetAsync(status, 0, sizeof(int32_t), s));
  const int64_t work = T > A->N ? T : A->N;
  const unsigned blocks = (unsigned)std::min<int64_t>((work + 255) / 256, 4096);
  k_validate<<<blocks, 256, 0, s>>>(A->esc_tile_ptr, A->esc, A->base, A->N, A->K, KC, T, (uint32_t)A->n_esc, status);
  W12_LAUNCH_CHECK(fn);
  return W12_OK;
}

}  // extern "C"
