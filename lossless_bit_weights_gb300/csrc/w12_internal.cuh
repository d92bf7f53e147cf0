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
constexpr int kBlockTiles = 4;       // row tiles per row block (128 channels)
constexpr int kHiTileBytes = 2048;   // 32 x 64 bytes
constexpr int kLoTileBytes = 1024;   // 32 x 64 nibbles
constexpr int64_t kMaxK = 65535;

// Row blocks of 128 channels; row tiles (4 per block, the last block padded).
__host__ __device__ inline int64_t row_blocks(int64_t N) { return (N + kTileRows * kBlockTiles - 1) / (kTileRows * kBlockTiles); }
__host__ __device__ inline int64_t row_tiles(int64_t N) { return row_blocks(N) * kBlockTiles; }
__host__ __device__ inline int64_t k_chunks(int64_t K) { return (K + kTileK - 1) / kTileK; }

// Tile order: the four row tiles of a row block at one column chunk are
// adjacent, so tile (rt, kc) has index ((rt/4)*KC + kc)*4 + rt%4.
__host__ __device__ inline int64_t tile_index(int64_t rt, int64_t kc, int64_t KC) {
  return ((rt >> 2) * KC + kc) * kBlockTiles + (rt & 3);
}
__host__ __device__ inline void tile_coords(int64_t i, int64_t KC, int64_t& rt, int64_t& kc) {
  const int64_t bk = i >> 2;
  const int64_t rb = bk / KC;
  kc = bk - rb * KC;
  rt = rb * kBlockTiles + (i & 3);
}

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

// Escape entry of the device layout: raw bf16 | slot << 16, where slot is the
// byte offset of (channel-in-tile rr, column-in-chunk kk) in the tile's decoded
// 32x64 bf16 image with the 128-byte swizzle the GEMM's A operand uses: row rr
// at rr*128, 16-byte chunk kk/8 stored at chunk (kk/8) ^ (rr%8).  The GEMM
// patches an escape with one 2-byte store at that offset.
__host__ __device__ inline uint32_t esc_slot_of(int rr, int kk) {
  return (uint32_t)(rr * 128 + ((((kk >> 3) ^ (rr & 7)) & 7) << 4) + (kk & 7) * 2);
}
__host__ __device__ inline uint32_t esc_entry(int rr, int kk, uint32_t raw) { return raw | (esc_slot_of(rr, kk) << 16); }
__host__ __device__ inline uint32_t esc_slot(uint32_t e) { return e >> 16; }
__host__ __device__ inline int esc_row(uint32_t e) { return (int)(e >> 23); }
__host__ __device__ inline int esc_col(uint32_t e) {
  const uint32_t off = e >> 16, rr = off >> 7;
  return (int)(((((off >> 4) & 7u) ^ (rr & 7u)) << 3) | ((off >> 1) & 7u));
}
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
//
// Word H_s of the hi slice holds the front bytes of columns 4s, 4s+2, 4s+1,
// 4s+3 (bytes 0..3), so bytes 0,2 give pair 2s and bytes 1,3 give pair 2s+1.
// A lane's bf16 is s<<15 | (base + eo)<<7 | m6..4<<4 | m3..0 from a front byte
// f = s<<7 | eo<<3 | m6..4 and a nibble.  The nibbles of pair p sit in lo word
// p/4 at bits 4(p%4) and 16+4(p%4).
//
// The work is split between the two integer pipes: masks and merges on the
// logic pipe, every shift on the multiply-add pipe (x*16 and x*256 move bytes
// left; the high word of x*2^(32-k) is x>>k, and mad.hi adds it to the partly
// built pair in the same instruction, which is exact because the target bits
// are still zero).  Per 16 weights that is 24 logic and 18 multiply-add
// instructions.
__device__ __forceinline__ uint32_t mul_hi_add(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("mad.hi.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// The multipliers come in as run-time values (16, 256 and 2^(32-k) for k = 4,
// 8, 12) so that the compiler keeps them as integer multiply-adds instead of
// logic-pipe shifts.
struct DecodeMul {
  uint32_t m16, m256, m2p28, m2p24, m2p20;
};
#define W12_DECODE_MUL DecodeMul{16u, 256u, 1u << 28, 1u << 24, 1u << 20}

// nibbles k*4 and 16+k*4 of L added at bits 0 and 16 of v (k = 0..3)
template <int K>
__device__ __forceinline__ uint32_t add_nibbles(uint32_t v, uint32_t L, const DecodeMul& m) {
  if (K == 0) return (L & 0x000F000Fu) | v;
  const uint32_t mul = K == 1 ? m.m2p28 : K == 2 ? m.m2p24 : m.m2p20;
  return mul_hi_add(L & (0x000F000Fu << (4 * K)), mul, v);
}

template <bool Q8>
__device__ __forceinline__ void decode16(uint4 h, uint2 l, uint32_t base2, const DecodeMul& k, uint32_t out[8]) {
  const uint32_t H[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const uint32_t Hs = H[s];
    const uint32_t L = (s < 2) ? l.x : l.y;
    // pair 2s: bytes 0 and 2 -> (f & 0x7F) * 16 + base<<7, sign * 256
    const uint32_t e7 = Hs & 0x007F007Fu;
    const uint32_t es = Hs & 0x00800080u;
    uint32_t ve = es * k.m256 + (e7 * k.m16 + base2);
    // pair 2s+1: bytes 1 and 3 -> (f & 0x7F00) >> 4 via the high product, sign already at bit 15
    const uint32_t o7 = Hs & 0x7F007F00u;
    uint32_t vo = mul_hi_add(o7, k.m2p28, base2) | (Hs & 0x80008000u);
    if (!Q8) {
      // pair 2s has p%4 = 2s%4 in {0, 2}; pair 2s+1 has p%4 in {1, 3}
      if ((s & 1) == 0) {
        ve = add_nibbles<0>(ve, L, k);
        vo = add_nibbles<1>(vo, L, k);
      } else {
        ve = add_nibbles<2>(ve, L, k);
        vo = add_nibbles<3>(vo, L, k);
      }
    }
    out[2 * s] = ve;
    out[2 * s + 1] = vo;
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

// ---- mbarrier / bulk-copy (TMA) helpers

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Default bound of every device-side wait, in SM clock cycles: about a second.
constexpr long long kWaitCycles = 1ll << 31;

// Slow path of mbar_wait_bounded: try_wait (the thread may be suspended in
// hardware until the phase completes) until `limit` clock cycles have passed.
// Returns false when the limit ran out.
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, long long limit) {
  const long long start = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - start > limit) return false;
  }
  return true;
}

// Waits for the barrier phase with parity `parity`, bounded; one non-blocking
// test first, so a phase that has already completed costs two instructions.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, long long limit = kWaitCycles) {
  if (mbar_test_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, limit);
}

// The same wait without a function call in the slow path: a noinline call would make the
// caller keep its live registers across the call.  The first try_wait lets the hardware
// suspend the thread until the phase completes (or a short while passes).
__device__ __forceinline__ bool mbar_wait_inline(uint32_t bar, uint32_t parity, long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long start = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - start > limit) return false;
  }
  return true;
}

// Global -> shared bulk copy completing on an mbarrier (size multiple of 16, both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}

// Warm L2 with a global range (size multiple of 16, 16-byte aligned).
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& a0, uint32_t& a1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(a0), "=r"(a1) : "r"(addr) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// ---- tcgen05 (5th-generation tensor core) helpers

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B, both K-major, M = 128,
// N = n (16..256, a multiple of 16).
__host__ __device__ __forceinline__ constexpr uint32_t umma_idesc_n(uint32_t n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}
template <int NT>
__device__ __forceinline__ constexpr uint32_t umma_idesc() {
  return umma_idesc_n((uint32_t)NT);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 lanes x 16 fp32 columns of the accumulator (this warp's lane quarter).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float v[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  // the registers are operands of the wait, so no use of them is scheduled before it
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
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
