// w12_internal.cuh - layout constants, status plumbing and PTX helpers shared by
// the library's translation units.  See include/w12.h for the device layout.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdarg>
#include <cstdio>

#include "../../include/w12.h"

namespace w12 {

constexpr int kTileRows = 32;        // channels per tile
constexpr int kTileK = 64;           // columns per tile
constexpr int kHiTileBytes = 2048;   // 32 x 64 bytes
constexpr int kLoTileBytes = 1024;   // 32 x 64 nibbles
constexpr int64_t kMaxK = 65535;

__host__ __device__ inline int64_t row_tiles(int64_t N) { return (N + kTileRows - 1) / kTileRows; }
__host__ __device__ inline int64_t k_chunks(int64_t K) { return (K + kTileK - 1) / kTileK; }

// Byte offset inside a hi tile of channel r (0..31) and column kk (0..63).
__host__ __device__ inline int hi_offset(int r, int kk) {
  int q = r >> 3, g = r & 7, t = kk >> 4, j = kk & 15, u = j & 3;
  int pos = (j & ~3) | (u == 1 ? 2 : u == 2 ? 1 : u);
  return q * 512 + (4 * g + t) * 16 + pos;
}

// Bit offset inside a lo tile of channel r and column kk.
__host__ __device__ inline int lo_bit(int r, int kk) {
  int q = r >> 3, g = r & 7, t = kk >> 4, j = kk & 15;
  int p = 2 * (j >> 2) + ((j & 3) >> 1);
  return (q * 256 + (4 * g + t) * 8) * 8 + 32 * (p >> 2) + 4 * (p & 3) + 16 * (j & 1);
}

// Escape entry of the device layout.
__host__ __device__ inline uint32_t esc_entry(int rr, int kk, uint32_t raw) {
  return raw | ((uint32_t)kk << 16) | ((uint32_t)rr << 22);
}
__host__ __device__ inline int esc_row(uint32_t e) { return (int)(e >> 22); }
__host__ __device__ inline int esc_col(uint32_t e) { return (int)((e >> 16) & 63u); }
__host__ __device__ inline uint32_t esc_raw(uint32_t e) { return e & 0xFFFFu; }

// ---------------------------------------------------------------- status

void set_error(const char* fmt, ...);
int fail(int status, const char* fmt, ...);
int cuda_fail(cudaError_t e, const char* what);
int check_matrix(const w12_matrix* A, bool need_lo, const char* fn);

#define W12_CUDA_TRY(expr)                           \
  do {                                               \
    cudaError_t _e = (expr);                         \
    if (_e != cudaSuccess) return cuda_fail(_e, #expr); \
  } while (0)

#define W12_LAUNCH_CHECK(what)                       \
  do {                                               \
    cudaError_t _e = cudaGetLastError();             \
    if (_e != cudaSuccess) return cuda_fail(_e, what); \
  } while (0)

// ---------------------------------------------------------------- device helpers

// Decode 16 weights of one channel (one 16-byte hi slice, one 8-byte lo
// slice) into 8 bf16 pairs in column order: out[p] holds columns 2p (low half)
// and 2p+1 (high half).  base2 = base<<7 | base<<23.  With Q8 the low nibbles
// read as zero.
template <bool Q8>
__device__ __forceinline__ void decode16(uint4 h, uint2 l, uint32_t base2, uint32_t out[8]) {
  const uint32_t H[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const uint32_t Hs = H[p >> 1];
    const uint32_t Q = (p & 1) ? Hs : (Hs << 8);      // front bytes at bits 8..15 / 24..31
    const uint32_t R = (Q >> 4) & 0x07F007F0u;          // exponent offset and mantissa 6..4
    const uint32_t S = Q & 0x80008000u;                 // sign
    uint32_t v = R + S + base2;                         // exponent = base + offset
    if (!Q8) {
      const uint32_t L = (p < 4) ? l.x : l.y;
      v |= (L >> (4 * (p & 3))) & 0x000F000Fu;          // mantissa 3..0
    }
    out[p] = v;
  }
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint4 ldg_stream16(const void* p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}

__device__ __forceinline__ uint2 ldg_stream8(const void* p, uint64_t policy) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v2.u32 {%0,%1}, [%2], %3;"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p), "l"(policy));
  return v;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ void sts16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& a0, uint32_t& a1, uint32_t& a2, uint32_t& a3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void mma_bf16_16816(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Total order used by every argmax: larger key = larger value; NaN lowest;
// -0 and +0 equal.
__device__ __forceinline__ int32_t order_key(float f) {
  if (f != f) return INT32_MIN;
  if (f == 0.0f) f = 0.0f;
  int32_t s = __float_as_int(f);
  return s >= 0 ? s : (s ^ 0x7FFFFFFF);
}

}  // namespace w12
