// w12_gemm.cu - decode-fused weight-streaming GEMM for few rows (up to 256
// tokens per launch), its 8-bit-view variant, and the LM-head argmax epilogue.
//
// The SpecPilot summary page (onedev.kr/papers/1654), section "What's
// different", describes a GEMM that decodes the 12-bit records in registers,
// hides the decode behind the memory stream and stays deterministic with
// stream-K.  This kernel is built for sm_103a:
//  - a unit of work is a row block (128 channels = 4 row tiles) x one
//    64-column chunk; the flat list of units is split evenly over the CTAs
//    (stream-K);
//  - one producer warp fills a shared-memory ring with bulk copies (TMA): the
//    block's 8 KB of front bytes and 4 KB of nibbles (adjacent in the device
//    tile order) and its escape run; another warp streams the chunk of x
//    through a 2-D tensor map (128-byte swizzle; rows past M and columns past
//    K read as zero);
//  - two groups of four decode warps take alternate units; each warp decodes
//    its 32x64 tile in registers to bf16 (sign, base+offset, mantissa), stores
//    it to a swizzled A buffer (the buffers rotate over the units) and writes
//    the tile's escapes over their slots;
//  - one thread issues tcgen05.mma (M = 128 channels, N = 16..256 tokens,
//    swap-AB: weights on the M side) with the fp32 accumulator in tensor
//    memory (two, alternating by row block, for the 12-bit pass up to 32
//    tokens); at the end of a row block the group that decoded its last unit
//    reads the accumulator back;
//  - a part of the partition that covers only some of a row block writes
//    partial sums to a fixed slot and publishes each row tile with an atomic
//    counter; the last part to arrive (no waiting) adds the slots in part
//    order, so results are bit-identical from call to call.  At a range's end
//    it fetches them by bulk copy into the consumed ring; a range's first row,
//    drained early, is published by a publisher warp while the decode goes on
//    (with one or two own ranges per CTA);
//  - launches use programmatic dependent launch: a GEMM starts streaming its
//    weights while the previous kernel on the stream drains, and waits for
//    that kernel only before it reads x.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "w12_internal.cuh"

namespace w12 {
namespace {

constexpr int kEscRun = 128;  // escape entries a record stage holds
constexpr int kMinIters = 4;  // fewest units per CTA

// Bits of the workspace's error word (its first 4 bytes), set by a CTA that gave up or
// met a bad escape index, read and cleared by w12_workspace_status.
constexpr uint32_t kErrTimeout = 1u;  // a wait for another warp's work ran out
constexpr uint32_t kErrBounds = 2u;   // an escape offset lay outside the escape list

// Bound of the kernel's waits for another warp's work (records landed, a stage or buffer
// released, an accumulator ready), in SM clock cycles.  w12_set_wait_limit lowers it to
// exercise the timeout path.  Waits for a warp's own copies and MMAs in flight keep the
// default bound, so a CTA that gives up still leaves with nothing in flight.
__constant__ long long c_wait_limit = kWaitCycles;

// EPI_I8: the weights are INT8 codes (sign<<7 | |q|, in the hi-plane layout; no lo plane,
// window bases or escapes); the approximate logit of token m and channel n is
// scale[n] * acc, and the epilogue feeds the certified argmax (CertEpi) instead of
// storing it.
enum Epi { EPI_STORE = 0, EPI_ARGMAX = 1, EPI_I8 = 2 };

// The certified argmax's use of the approximate logits a (EPI_I8).  With the bound
// b = nx[m] * cb[n] (rounded up), the threshold of token m is max_n (a - b) rounded down,
// kept as an order-preserving key in thr_key[m] (atomicMax; zero beforehand); a channel is
// a candidate when a + b (rounded up) reaches the final threshold.  Each warp appends to
// sup[m*ldsup ..] (count in sup_count[m], zero beforehand) every channel whose a + b reaches
// the largest threshold known to it (its own channels' and the running value): a superset
// of the candidates, since every known value is at most the final threshold.  An entry is
// (channel, key of a + b).
struct CertEpi {
  const float* nx;
  const float* cb;
  uint32_t* thr_key;
  uint32_t* sup_count;
  uint2* sup;
  int64_t ldsup;
};

struct GemmArgs {
  const uint8_t* hi;
  const uint8_t* lo;
  const uint8_t* base;
  const uint32_t* tile_ptr;
  const uint32_t* esc;
  int64_t N, KC, T, G;  // T = units of the partition, G = its places (pipelines or CTAs)
  int M;                // tokens of this launch (<= NT)
  int tok0;             // first token of this launch (x tensor-map row)
  float* y;             // EPI_STORE: y[m*ldy + n] (already offset to tok0)
  int64_t ldy;
  unsigned long long* pbest;  // EPI_ARGMAX: pbest[rt*ldp + tok0 + m]
  int64_t ldp;
  float* slots;
  uint32_t* counters;
  uint32_t* error;
  DecodeMul mul;
  // Last: with the ring at 64..256 tokens decode-issue bound, inserting a field above
  // measured 6% slower (only the offsets of the members after it changed).
  int64_t RB;  // row blocks of the matrix
  const float* scale;  // EPI_I8: per-channel scale
  uint32_t n_esc;      // escape entries; escape offsets are clamped to it
  CertEpi cert;        // EPI_I8
};

// Order-preserving map of floats to unsigned keys (larger float, larger key; key 0 is
// below every float).
__device__ __forceinline__ uint32_t order_key32(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float order_key32_inv(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__device__ __forceinline__ int64_t cta_of_unit(int64_t i, int64_t G, int64_t T) { return ((i + 1) * G - 1) / T; }

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tma_x(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], "
      "[%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "l"(pol)
      : "memory");
}

// ===========================================================================
// tcgen05 variant: decode warps unpack into shared memory; one thread issues
// the MMAs (5th-generation tensor core, fp32 accumulator in tensor memory).
//   warps 0..4G-1  decode, G groups of four: group g takes the units j with
//                  j % G == g, warp w of a group the row tile w % 4 (32 rows).
//                  The group that decodes a row block's last unit drains the
//                  accumulator (warp w reads TMEM lanes 32(w%4)..32(w%4)+31).
//   warp 4G        TMA producer of the weight records (hi, lo, escape run)
//   warp 4G+1      lane 0 issues tcgen05.mma (M=128 channels, N=NT tokens, K=16)
//   warp 4G+2      lane 0 streams x through the tensor map on its own ring
// A record stage goes back to the producer as soon as its group holds the
// unit in registers; x stages and A buffers go back on the MMA commit.  With
// four groups a group has four unit-times for its own unit, so a record stage
// is taken as soon as it lands and the whole shared memory of the SM serves
// one deep ring.
constexpr int kABuf = kBlockTiles * kTileRows * 128;  // decoded 128x64 bf16 block (16 KB, swizzled)

// Launch modes.  A pipeline is a producer warp, two decode groups, an MMA issuer and an x
// warp, with its own shared memory, barriers and TMEM columns.
//  kModeOwn  (NT <= 32 on matrices with fewer row blocks than SMs): two pipelines per CTA,
//            one CTA per SM, each pipeline with its own unit range (units = row block x 64
//            columns).  As two CTAs on an SM, the older one's warps were favoured by the
//            scheduler and it finished its equal share ~6 us sooner on gate/up (a launch
//            ends with the slower one); as two pipelines of one CTA they finish together.
//  kModeOne  (NT >= 64 on short matrices, and 256): one pipeline per CTA; its x chunks are
//            large.  At NT = 192 the rows split between CTAs are summed after the launch
//            (k_slot_sum).
//  kModePair (up to 192 tokens on matrices with a row block per SM or more): two pipelines
//            share one range of row-block pairs x 64 columns, pipeline p on row block
//            2*pair + p, and one x warp and ring (each stage freed by both MMA issuers).
//            Against kModeOne: twice the decode warps per SM; against kModeOwn: one x
//            stream for both pipelines and deeper record rings.  Stream-K splits run over
//            twice as many CTAs per (longer) row, so it pays on tall matrices only.
//  kModePairSum (64 to 192 tokens on shorter matrices with long rows): kModePair's CTA, but
//            the rows split between CTAs are summed after the launch over every SM
//            (k_slot_sum), not by each row's last part.
enum { kModeOwn = 0, kModeOne = 1, kModePair = 2, kModePairSum = 3 };

template <int NT, bool Q8, int MODE>
struct TcPlan {
  static constexpr bool kWide = MODE == kModePair || MODE == kModePairSum;
  static constexpr int kPipes = MODE == kModeOne ? 1 : 2;
  static constexpr int kParts = MODE == kModeOwn ? 2 : 1;     // places in the partition per CTA
  static constexpr int kGroups = 2;
  static constexpr int kDecoders = kGroups * kBlockTiles;
  // producer, MMA issuer (, publisher, x loader; the wide CTA's x loader is shared, after
  // the pipelines).  A publisher measured faster with one or two own ranges per CTA; with
  // row-block pairs the decode loop's register allocation moved and it lost.
  static constexpr bool kHasPub = !kWide;
  static constexpr int kRoles = kWide ? 2 : 4;
  static constexpr int kProducer = kDecoders, kMma = kDecoders + 1, kPub = kDecoders + 2;
  static constexpr int kXWarp = kWide ? kDecoders + 2 : kDecoders + 3;
  static constexpr int kThreads = (kDecoders + kRoles) * 32;  // one pipeline
  static constexpr int kCtaThreads = kPipes * kThreads + (kWide ? 32 : 0);
  static constexpr int kCtasPerSM = 1;
  // Warps are spread over the SM's four sub-partitions (16K registers each); a 21- to
  // 24-warp CTA puts six on one, so 80 registers a thread is the most that launches.
  static constexpr int kBoundThreads = kPipes == 1 ? kCtaThreads : kCtaThreads > 704 ? kCtaThreads : 704;
  static constexpr int kX = NT * 128;                         // swizzled x chunk, 1 KB multiple
  // x stages: at 192 tokens with row-block pairs a third 24 KB stage (shared by both
  // pipelines) measured better than a fourth record stage per pipeline
  static constexpr int kXStages = NT <= 16 ? 4 : NT <= 64 ? 3 : (kWide && NT == 192) ? 3 : 2;
  // A buffers (decoded 128x64 tiles) in rotation over the pipeline's units: with more than
  // one per decode group, a group stores a unit while the MMA of the unit before its previous
  // one may still run.  At 16 tokens with own ranges a fifth record stage measured better
  // than a third A buffer.
  static constexpr int kABufs = MODE == kModeOwn ? (NT <= 16 ? 2 : 3) : MODE == kModeOne ? 4 : 2;
  // shared x region (wide): x stages, then x_full[SX] x_empty[SX]
  static constexpr int kXRegion = kWide ? (kXStages * kX + 2 * kXStages * 8 + 1023) / 1024 * 1024 : 0;
  static constexpr int kOffXBar = kXStages * kX;
  static constexpr int kHi = kBlockTiles * kHiTileBytes;
  static constexpr int kLo = Q8 ? 0 : kBlockTiles * kLoTileBytes;
  static constexpr int kOffLo = kHi;
  static constexpr int kOffEsc = kHi + kLo;
  static constexpr int kOffHdr = kOffEsc + kEscRun * 4;       // tile_ptr[4u..4u+4], run start
  static constexpr int kRec = kOffHdr + 32;
  static constexpr int kOffA = kWide ? 0 : kXStages * kX;
  static constexpr int kOffRec = kOffA + kABufs * kABuf;
  static constexpr int kBudget =
      kWide ? ((227 * 1024 - kXRegion) / 2) / 1024 * 1024 : (MODE == kModeOne ? 224 : 112) * 1024;
  static constexpr int kStagesRaw = (kBudget - kOffRec - 64 * 8 - 64) / kRec;
  static constexpr int kStages = kStagesRaw > 16 ? 16 : kStagesRaw;
  static constexpr int kOffBar = kOffRec + kStages * kRec;
  // rec_full[S] rec_empty[S] (x_full[SX] x_empty[SX]) a_full[AB] a_empty[AB] epi[2] acc_full
  // acc_empty mma_done (pub); epi: the second accumulator's full and drained barriers; pub:
  // a range's first row drained, for the publisher
  static constexpr int kNumBars = 2 * kStages + (kWide ? 0 : 2 * kXStages) + 2 * kABufs + kGroups + 3 + (kHasPub ? 1 : 0);
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 64;
  static constexpr int kPipeBytes = (kBytes + 1023) / 1024 * 1024;
  static constexpr int kCtaBytes = kPipes == 1 ? kBytes : kXRegion + kPipes * kPipeBytes;
  static constexpr int kTmemCols = NT <= 32 ? 32 : NT <= 64 ? 64 : NT <= 128 ? 128 : 256;
  // accumulators per pipeline: with two, the MMAs of a row block's first unit do not wait
  // for the drain of the row block before (segments alternate between them).  Measured
  // faster for the 12-bit pass at 16 tokens; the 8-bit view and larger token tiles keep one.
  static constexpr int kAccBufs = !Q8 && NT <= 32 ? 2 : 1;
  static_assert(kStages >= 3 && kStages > kGroups, "record ring too shallow");
  static_assert(kABufs >= kGroups, "an A buffer per decode group at least");
  static_assert(kCtaBytes <= 227 * 1024, "shared memory plan too large");
  static_assert(MODE != kModeOwn || NT <= 32, "launch mode does not fit the token tile");
  static_assert(kPipes * kAccBufs * kTmemCols <= 512, "tensor memory plan too large");
};

// 16 INT8 codes (sign<<7 | |q|, in the hi-plane byte order) -> 8 exact bf16 pairs.  A byte
// permute places each code in the low byte of a 16-bit lane and its sign across the high
// byte; masking in 0x4300 gives the bf16 +-(128 + |q|), and subtracting +-128 (same sign)
// leaves +-|q| exactly.
__device__ __forceinline__ uint32_t i8_pair(uint32_t t) {
  const uint32_t v = (t & 0x807F807Fu) | 0x43004300u, w = (t & 0x80008000u) | 0x43004300u;
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(v), "r"(w));
  return d;
}

// prmt in its default mode: selector nibble bits 2..0 pick a byte, bit 3 fills the result
// byte with the picked byte's sign bit.
__device__ __forceinline__ uint32_t prmt_sign(uint32_t a, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(d) : "r"(a), "r"(sel));
  return d;
}

__device__ __forceinline__ void decode16_i8(uint4 h, uint32_t out[8]) {
  const uint32_t H[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    // pair 2s = bytes 0 and 2 (columns 4s, 4s+1); pair 2s+1 = bytes 1 and 3
    out[2 * s] = i8_pair(prmt_sign(H[s], 0xA280u));
    out[2 * s + 1] = i8_pair(prmt_sign(H[s], 0xB391u));
  }
}

// Wait for another warp's work on a barrier phase, bounded by c_wait_limit.
__device__ __forceinline__ bool peer_wait(uint32_t bar, uint32_t parity) {
  return mbar_wait_inline(bar, parity, c_wait_limit);
}

// Bounded barrier wait whose outcome is the same in every lane of the warp.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
  return __all_sync(0xFFFFFFFFu, peer_wait(bar, parity));
}

__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Waits (bounded, warp-uniform) until a shared-memory counter reaches target.
__device__ __forceinline__ bool wait_count(const uint32_t* c, uint32_t target) {
  bool ok = true;
  if (*reinterpret_cast<const volatile uint32_t*>(c) < target) {
    const long long start = clock64();
    while (*reinterpret_cast<const volatile uint32_t*>(c) < target) {
      __nanosleep(64);
      if (clock64() - start > c_wait_limit) {
        ok = false;
        break;
      }
    }
  }
  return __all_sync(0xFFFFFFFFu, ok);
}


// Output of 16 token columns [c0, c0+16) for this warp's 32 rows (row tile rt).
template <int EPI>
__device__ __forceinline__ void emit_cols(const GemmArgs& a, int64_t rt, int lane, int c0, const float v[16]) {
  const int64_t n = rt * kTileRows + lane;
  if (EPI == EPI_STORE) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int tok = c0 + i;
      if (tok < a.M && n < a.N) a.y[(int64_t)tok * a.ldy + n] = v[i];
    }
  } else if (EPI == EPI_I8) {
    const bool ch = n < a.N;
    const float sc = ch ? a.scale[n] : 0.f, cbn = ch ? a.cert.cb[n] : 0.f;
    // lane i < 16: token c0 + i's row norm and the running threshold (any stale value is a
    // lower bound of the final one)
    const int tl16 = c0 + (lane & 15);
    const bool tv = lane < 16 && tl16 < a.M;
    const int64_t mrow = (int64_t)a.tok0 + tl16;
    const float nxl = tv ? a.cert.nx[mrow] : 0.f;
    const uint32_t runl = tv ? *reinterpret_cast<const volatile uint32_t*>(a.cert.thr_key + mrow) : 0u;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int tok = c0 + i;
      if (tok >= a.M) break;  // warp-uniform
      const float nt = __shfl_sync(0xFFFFFFFFu, nxl, i);
      const uint32_t run = __shfl_sync(0xFFFFFFFFu, runl, i);
      const float lh = v[i] * sc;
      const float bnd = __fmul_ru(nt, cbn);
      const float up = __fadd_ru(lh, bnd);
      const float down = __fsub_rd(lh, bnd);
      uint32_t lo = (ch && down == down) ? order_key32(down) : 0u;  // a NaN is never the threshold
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) lo = max(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, o));
      const int64_t m = (int64_t)a.tok0 + tok;
      if (lane == 0 && lo > run) atomicMax(a.cert.thr_key + m, lo);
      const uint32_t known = max(lo, run);
      const bool keep = ch && known != 0u && up >= order_key32_inv(known);
      const uint32_t bal = __ballot_sync(0xFFFFFFFFu, keep);
      if (bal) {
        uint32_t b0 = 0u;
        if (lane == 0) b0 = atomicAdd(a.cert.sup_count + m, (uint32_t)__popc(bal));
        b0 = __shfl_sync(0xFFFFFFFFu, b0, 0);
        if (keep)
          a.cert.sup[m * a.cert.ldsup + b0 + (uint32_t)__popc(bal & ((1u << lane) - 1u))] =
              make_uint2((uint32_t)n, order_key32(up));
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int tok = c0 + i;
      unsigned long long best = 0ull;
      if (n < a.N) {
        const uint32_t key = (uint32_t)order_key(v[i]) ^ 0x80000000u;
        best = ((unsigned long long)key << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)n);
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, best, o);
        best = other > best ? other : best;
      }
      if (lane == 0 && tok < a.M) a.pbest[rt * a.ldp + a.tok0 + tok] = best;
    }
  }
}

template <int NT, bool Q8, int MODE, int EPI>
__global__ void __launch_bounds__(TcPlan<NT, Q8, MODE>::kBoundThreads, TcPlan<NT, Q8, MODE>::kCtasPerSM)
    k_gemm_tc(const __grid_constant__ CUtensorMap xmap, const GemmArgs a) {
  using P = TcPlan<NT, Q8, MODE>;
  constexpr bool I8 = EPI == EPI_I8;  // INT8 codes: no window bases, escapes or lo plane
  static_assert(!I8 || Q8, "INT8 codes use the 8-bit record plan");
  constexpr int S = P::kStages, SX = P::kXStages, kTcGroups = P::kGroups, AB = P::kABufs;
  constexpr int kTcProducer = P::kProducer, kTcMma = P::kMma, kTcPub = P::kPub, kTcX = P::kXWarp;
  // storing y with pairs summed after, or one pipeline per CTA at 192 tokens (96 KB slots):
  // a row block split between CTAs is summed after the launch (k_slot_sum, over every SM)
  // instead of by its last part alone.  With one pipeline at 64 and 128 tokens the extra
  // launch cost more than the fix-up it saves.
  constexpr bool kDefer = EPI == EPI_STORE && ((MODE == kModeOne && NT == 192) || MODE == kModePairSum);
  extern __shared__ __align__(1024) uint8_t smem_cta[];
  const int lane = threadIdx.x & 31, gwarp = threadIdx.x >> 5;
  // pipeline and the warp's role index inside it: the decode warps of pipeline p are
  // warps 8p..8p+7 (groups stay aligned to TMEM lane quarters), then each pipeline's
  // producer and MMA issuer (and x loader); the shared x loader of a wide CTA comes last
  constexpr int nd = P::kDecoders, nr = P::kRoles, np = P::kPipes;
  int pipe = 0, warp = kTcX;
  if (gwarp < np * nd) {
    pipe = gwarp / nd;
    warp = gwarp % nd;
  } else if (gwarp < np * (nd + nr)) {
    pipe = (gwarp - np * nd) / nr;
    warp = nd + (gwarp - np * nd) % nr;
  }
  // place in the partition: each pipeline has one (kModeOwn), or the CTA has one
  const int64_t b = (int64_t)blockIdx.x * P::kParts + (P::kParts == 2 ? pipe : 0);
  const bool active = b < a.G;
  uint8_t* smem = smem_cta + P::kXRegion + pipe * P::kPipeBytes;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t xbase = P::kWide ? smem_u32(smem_cta) : sbase;  // x stage 0
  const uint32_t bar0 = sbase + P::kOffBar;
  const uint32_t rec_full0 = bar0, rec_empty0 = bar0 + 8 * S;
  const uint32_t x_full0 = P::kWide ? xbase + P::kOffXBar : bar0 + 16 * S, x_empty0 = x_full0 + 8 * SX;
  const uint32_t a_full0 = bar0 + 16 * S + (P::kWide ? 0 : 16 * SX), a_empty0 = a_full0 + 8 * AB;
  const uint32_t epi0 = a_empty0 + 8 * AB;
  const uint32_t acc_full = epi0 + 8 * kTcGroups, acc_empty = acc_full + 8, mma_done = acc_empty + 8, pub = mma_done + 8;
  // misc: [0] TMEM address, [4..11] bulk fix-up barriers, [15] drains finished (four per segment)
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + P::kOffMisc);
  const int64_t u0 = active ? b * a.T / a.G : 0, u1 = active ? (b + 1) * a.T / a.G : 0;
  const int nun = (int)(u1 - u0);
  // units this pipeline decodes: with an odd number of row blocks, the last pair of a
  // wide launch has no second row block
  int nunp = nun;
  if (P::kWide && pipe == 1 && (a.RB & 1)) {
    const int64_t lim = (a.T / a.KC - 1) * a.KC;
    nunp = (int)(lim < u0 ? 0 : (lim < u1 ? lim - u0 : nun));
  }

  // The next kernel on the stream may start as this one's CTAs retire (programmatic
  // dependent launch): its weight stream does not depend on this kernel's output.
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (warp == 0 && lane == 0) {
    misc[15] = 0u;
    for (int i = 0; i < S; ++i) {
      mbar_init(rec_full0 + 8 * i, 1);
      mbar_init(rec_empty0 + 8 * i, kBlockTiles * 32);
    }
    if (!P::kWide || pipe == 0)
      for (int i = 0; i < SX; ++i) {
        mbar_init(x_full0 + 8 * i, 1);
        mbar_init(x_empty0 + 8 * i, P::kWide ? 2 : 1);  // wide: freed by both MMA issuers
      }
    for (int i = 0; i < AB; ++i) {
      mbar_init(a_full0 + 8 * i, kBlockTiles * 32);
      mbar_init(a_empty0 + 8 * i, 1);
    }
    mbar_init(epi0, 1);                        // second accumulator full
    mbar_init(epi0 + 8, kBlockTiles * 32);     // second accumulator drained
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, kBlockTiles * 32);
    mbar_init(mma_done, 1);
    if (P::kHasPub) mbar_init(pub, kBlockTiles * 32);
    mbar_init_fence();
  }
  // one warp allocates the TMEM columns of every pipeline (address in pipeline 0's misc[0])
  uint32_t* misc0 = reinterpret_cast<uint32_t*>(smem_cta + P::kXRegion + P::kOffMisc);
  if (warp == kTcMma && pipe == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(misc0)),
                 "n"(P::kPipes * P::kAccBufs * P::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem0 = misc0[0];  // kept in a register: the teardown frees exactly this
  const uint32_t tmem = tmem0 + (uint32_t)(pipe * P::kAccBufs * P::kTmemCols);
  bool bail = false, bad_index = false;

  if (!active) {
    // a pipeline with no place in the partition goes straight to the teardown
  } else if (warp == kTcProducer) {
    // ---------------------------------------------------------------- weight records
    const uint64_t pol_w = policy_evict_first();
    const int KC = (int)a.KC;
    const int64_t TR = a.RB * a.KC;  // record units (tile_ptr has 4 TR + 1 entries)
    int kc = P::kWide ? (int)(u0 % a.KC) : 0;
    // record unit (row block x 64 columns) of the pipeline's first unit
    int64_t ru = P::kWide ? (2 * (u0 / a.KC) + pipe) * a.KC + kc : u0;
    // tile_ptr[4ru + wo ..] in a window of 96 entries held across the lanes in three
    // registers; the third is loaded 8 units before any shuffle reads it.  A wide
    // pipeline skips the other pipeline's row block at each pair boundary and reloads.
    const uint32_t* tpw = nullptr;
    int64_t TT = 0;  // entries left from tpw on
    int wo = 0;
    uint32_t w0 = 0u, w1 = 0u, w2 = 0u;
    auto window = [&](int64_t r) {
      tpw = a.tile_ptr + 4 * r;
      TT = 4 * (TR - r);
      wo = 0;
      w0 = lane <= TT ? __ldg(tpw + lane) : 0u;
      w1 = 32 + lane <= TT ? __ldg(tpw + 32 + lane) : 0u;
      w2 = 64 + lane <= TT ? __ldg(tpw + 64 + lane) : 0u;
    };
    if constexpr (!I8) window(ru);
    const uint8_t* hp = a.hi + ru * P::kHi;
    const uint8_t* lp = a.lo + ru * (kBlockTiles * kLoTileBytes);
    int issued = 0, s = 0;
    uint32_t ph = 0;  // parity of the empty phase to wait for, once the ring has wrapped
    for (int j = 0; j < nunp; ++j) {
      if (j >= S && !warp_wait(rec_empty0 + 8 * s, ph)) {
        bail = true;
        break;
      }
      uint32_t esc_bytes = 0u, e0 = 0u;
      if constexpr (!I8) {
        if (wo >= 32) {
          w0 = w1;
          w1 = w2;
          tpw += 32;
          TT -= 32;
          wo -= 32;
          w2 = 64 + lane <= TT ? __ldg(tpw + 64 + lane) : 0u;
        }
        const int src = wo + (lane < 5 ? lane : 0);  // lane i < 5 gets tile_ptr[4ru + i]
        const uint32_t v0 = __shfl_sync(0xFFFFFFFFu, w0, src & 31);
        const uint32_t v1 = __shfl_sync(0xFFFFFFFFu, w1, src & 31);
        const uint32_t tpv = src < 32 ? v0 : v1;
        uint32_t t_first = __shfl_sync(0xFFFFFFFFu, tpv, 0), t_last = __shfl_sync(0xFFFFFFFFu, tpv, 4);
        // offsets past the escape list (a damaged index) are clamped and reported
        if (t_last > a.n_esc || t_first > t_last) {
          bad_index = true;
          t_last = min(t_last, a.n_esc);
          t_first = min(t_first, t_last);
        }
        e0 = t_first & ~3u;
        uint32_t e1 = (t_last + 3u) & ~3u;
        if (e1 > e0 + kEscRun) e1 = e0 + kEscRun;
        esc_bytes = t_last > t_first ? (e1 - e0) * 4u : 0u;
        uint8_t* rec = smem + P::kOffRec + s * P::kRec;
        if (lane < 6) reinterpret_cast<uint32_t*>(rec + P::kOffHdr)[lane] = lane < 5 ? tpv : e0;
        __syncwarp();
      }
      if (lane == 0) {
        const uint32_t full = rec_full0 + 8 * s;
        const uint32_t recs = sbase + P::kOffRec + s * P::kRec;
        mbar_arrive_expect_tx(full, P::kHi + P::kLo + esc_bytes);
        bulk_g2s(recs, hp, P::kHi, full, pol_w);
        if (!Q8) bulk_g2s(recs + P::kOffLo, lp, P::kLo, full, pol_w);
        if (esc_bytes) bulk_g2s(recs + P::kOffEsc, a.esc + e0, esc_bytes, full, pol_w);
      }
      hp += P::kHi;
      lp += kBlockTiles * kLoTileBytes;
      wo += 4;
      issued = j + 1;
      if (++s == S) {
        s = 0;
        if (j >= S) ph ^= 1u;
      }
      if constexpr (P::kWide) {
        ++ru;
        if (++kc == KC) {
          kc = 0;
          if (j + 1 < nunp) {
            ru += a.KC;
            hp += (int64_t)KC * P::kHi;
            lp += (int64_t)KC * (kBlockTiles * kLoTileBytes);
            if constexpr (!I8) window(ru);
          }
        }
      }
    }
    // copies still in flight land before the CTA leaves (they have, unless a wait gave up)
    if (lane == 0)
      for (int j = std::max(0, issued - S); j < issued; ++j)
        mbar_wait_bounded(rec_full0 + 8 * (j % S), (uint32_t)((j / S) & 1));
    __syncwarp();
  } else if (warp == kTcX) {
    // ---------------------------------------------------------------- x chunks
    if (lane == 0) {
      // x may be the previous kernel's output: wait for that grid to complete and its
      // writes to be visible.  Every store of this kernel (y, slots, counters) follows an
      // MMA that reads x, so it also comes after the previous grid has finished.
      asm volatile("griddepcontrol.wait;" ::: "memory");
      const uint64_t pol_x = policy_evict_last();
      int64_t kc = u0 % a.KC;
      int issued = 0;
      for (int j = 0; j < nun; ++j) {
        const int s = j % SX;
        if (j >= SX && !peer_wait(x_empty0 + 8 * s, (uint32_t)(((j / SX) - 1) & 1))) {
          bail = true;
          break;
        }
        const uint32_t xfull = x_full0 + 8 * s;
        mbar_arrive_expect_tx(xfull, P::kX);
        tma_x(xbase + s * P::kX, &xmap, (int)(kc * kTileK), a.tok0, xfull, pol_x);
        issued = j + 1;
        if (++kc == a.KC) kc = 0;
      }
      for (int j = std::max(0, issued - SX); j < issued; ++j)
        mbar_wait_bounded(x_full0 + 8 * (j % SX), (uint32_t)((j / SX) & 1));
    }
    __syncwarp();
  } else if (warp == kTcMma) {
    // ---------------------------------------------------------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc<NT>();
      // Descriptors are built once: a K step of 16 adds 32 bytes (2 in the 16-byte address
      // field) and an x stage adds kX bytes.  Shared addresses stay below 2^18, so the
      // address field never carries into the neighbouring bits.
      const uint64_t ad0 = umma_desc(sbase + P::kOffA), xd0 = umma_desc(xbase);
      const int KC = (int)a.KC;
      int kc = (int)(u0 % a.KC);
      int seg = 0, s = 0, ab = 0;
      uint32_t xph = 0, aph = 0;
      for (int j = 0; j < nunp; ++j) {
        const bool first = (j == 0) || (kc == 0);
        const int abuf = P::kAccBufs == 2 ? (seg & 1) : 0;
        // a segment's first MMAs wait for the drain of the accumulator's previous segment
        if (first && seg >= P::kAccBufs &&
            !peer_wait(abuf ? epi0 + 8 : acc_empty, (uint32_t)((seg / P::kAccBufs - 1) & 1))) {
          bail = true;
          break;
        }
        if (!peer_wait(a_full0 + 8 * ab, aph) || !peer_wait(x_full0 + 8 * s, xph)) {
          bail = true;
          break;
        }
        tc_fence_after();
        const uint64_t ad = ad0 + (uint64_t)((ab * kABuf) >> 4), xd = xd0 + (uint64_t)((s * P::kX) >> 4);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_bf16(tmem + (uint32_t)(abuf * P::kTmemCols), ad + 2 * ks, xd + 2 * ks, idesc, (first && ks == 0) ? 0u : 1u);
        umma_commit(a_empty0 + 8 * ab);
        umma_commit(x_empty0 + 8 * s);
        if (kc + 1 == KC || j + 1 == nunp) {
          umma_commit(abuf ? epi0 : acc_full);
          ++seg;
        }
        if (++kc == KC) kc = 0;
        if (++s == SX) {
          s = 0;
          xph ^= 1u;
        }
        if (++ab == AB) {
          ab = 0;
          aph ^= 1u;
        }
      }
      // a wide pipeline past its last row block still frees the shared x stages it skips
      for (int j = nunp; j < nun && !bail; ++j) {
        if (!peer_wait(x_full0 + 8 * s, xph)) {
          bail = true;
          break;
        }
        mbar_arrive(x_empty0 + 8 * s);
        if (++s == SX) {
          s = 0;
          xph ^= 1u;
        }
      }
      // every MMA issued here has finished before TMEM is released
      if (nunp > 0) {
        umma_commit(mma_done);
        mbar_wait_bounded(mma_done, 0u);
      }
    }
    __syncwarp();
  } else if (P::kHasPub && warp == kTcPub) {
    // ---------------------------------------------------------------- publisher
    // A range that starts inside a row block and goes on past it drains that row early:
    // its group signals here instead of publishing, and this warp publishes the row's four
    // tiles and, when it is their last arrival, adds the parts' slots.
    const int KC = (int)a.KC, U0 = (int)u0;
    const int srb0 = U0 / KC;
    if (!kDefer && nunp > 0 && (U0 % KC) != 0 && (U0 + nunp - 1) / KC > srb0) {
      if (!warp_wait(pub, 0u)) {
        bail = true;
      } else {
        const int rb = P::kWide ? 2 * srb0 + pipe : srb0;
        const int64_t cf = cta_of_unit((int64_t)srb0 * KC, a.G, a.T);
        const int64_t cl = cta_of_unit((int64_t)(srb0 + 1) * KC - 1, a.G, a.T);
        const int64_t ncov = cl - cf + 1;
        constexpr int kWarpSlot = NT * 32;
        // lane t < 4 publishes row tile t: the barrier's acquire, then this release
        uint32_t arrived = 0u;
        if (lane < kBlockTiles) arrived = atom_add_acq_rel(a.counters + rb * kBlockTiles + lane, 1u);
        const uint32_t last = __ballot_sync(0xFFFFFFFFu, lane < kBlockTiles && (int64_t)arrived == ncov - 1);
        __syncwarp();  // the lanes' reads below follow the acquiring lane's increment
#pragma unroll 1
        for (int t = 0; t < kBlockTiles; ++t) {
          if (!((last >> t) & 1u)) continue;
          if (lane == 0) a.counters[rb * kBlockTiles + t] = 0u;
          const int64_t rt = (int64_t)rb * kBlockTiles + t;
#pragma unroll 1
          for (int c0 = 0; c0 < NT; c0 += 16) {
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = 0.f;
            for (int64_t jj = 0; jj < ncov; ++jj) {
              const int64_t slot = P::kWide ? 2 * (cf + jj + srb0) + pipe : cf + jj + srb0;
              const float4* sj = reinterpret_cast<const float4*>(a.slots + (slot * kBlockTiles + t) * kWarpSlot);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float4 q4 = __ldcg(sj + (c0 / 4 + i) * 32 + lane);
                v[4 * i] += q4.x;
                v[4 * i + 1] += q4.y;
                v[4 * i + 2] += q4.z;
                v[4 * i + 3] += q4.w;
              }
            }
            emit_cols<EPI>(a, rt, lane, c0, v);
          }
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- decode warps
    // Group gi visits only its own units j = gi, gi+G, ...; row block, chunk,
    // ring stage and phase advance by G units per step.  Unit indices fit in
    // 32 bits (the host caps T).
    const int gi = warp >> 2, tl = warp & 3;  // group, row tile inside the block
    const int g = lane >> 2, t = lane & 3;
    // unit j decodes into A buffer j % AB; au counts the buffer's earlier uses (its phase)
    uint8_t* const abase = smem + P::kOffA + tl * (kTileRows * 128);
    int ab = gi % AB;
    uint32_t au = (uint32_t)(gi / AB);
    const int KC = (int)a.KC, U0 = (int)u0;
    const int srb0 = U0 / KC;
    int j = gi;
    int srb = (U0 + j) / KC, kc = (U0 + j) - srb * KC;  // partition row (row block or pair) and chunk
    int s = j % S;
    uint32_t ph = (uint32_t)((j / S) & 1);
    int cur_rb = -1;
    uint32_t base2[4];
    for (; j < nunp; j += kTcGroups) {
      const int rb = P::kWide ? 2 * srb + pipe : srb;
      if (!I8 && rb != cur_rb) {  // this unit starts a new row block for the group: its rows' bases
        cur_rb = rb;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int64_t n = ((int64_t)rb * kBlockTiles + tl) * kTileRows + 8 * q + g;
          const uint32_t bb = n < a.N ? (uint32_t)__ldg(a.base + n) : 1u;
          base2[q] = (bb << 7) | (bb << 23);
        }
      }
      // The full barrier's parity wait is exact only while this stage's previous unit
      // (j - S) has already been consumed.  That holds when it is this group's own unit (S
      // even) or AB + 2 or more back: this group's previous unit waited for the MMA of unit
      // j - 2 - AB, which followed the decode of every unit up to it.  A shorter odd ring
      // (three stages with two A buffers) waits for the release of unit j - S first.
      if (S % 2 == 1 && S < AB + 2 && j >= S && !warp_wait(rec_empty0 + 8 * s, ph ^ 1u)) {
        bail = true;
        break;
      }
      if (!warp_wait(rec_full0 + 8 * s, ph)) {
        bail = true;
        break;
      }
      {
        const uint8_t* rec = smem + P::kOffRec + s * P::kRec;
        uint4 hq[4];
        uint2 lq[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          hq[q] = *reinterpret_cast<const uint4*>(rec + tl * kHiTileBytes + q * 512 + lane * 16);
          lq[q] = Q8 ? make_uint2(0u, 0u)
                     : *reinterpret_cast<const uint2*>(rec + P::kOffLo + tl * kLoTileBytes + q * 256 + lane * 8);
        }
        // this row tile's escapes: entry ta + lane into a register (the rare tail past 32 stays in memory)
        const uint32_t* hdr = reinterpret_cast<const uint32_t*>(rec + P::kOffHdr);
        // the tile's escape range, clamped to the escape list (the producer reports a bad index)
        const uint32_t tb = I8 ? 0u : min(hdr[tl + 1], a.n_esc), ta = I8 ? 0u : min(hdr[tl], tb);
        const uint32_t e0 = I8 ? 0u : hdr[5];
        const uint32_t cnt = tb - ta;
        uint32_t ent = 0u;
        if ((uint32_t)lane < cnt) {
          const uint32_t e = ta + lane;
          ent = e - e0 < (uint32_t)kEscRun ? reinterpret_cast<const uint32_t*>(rec + P::kOffEsc)[e - e0]
                                           : __ldg(a.esc + e);
        }
        // the record stage can be refilled now (every thread arrives once its own loads are done)
        mbar_arrive(rec_empty0 + 8 * s);
        // the A buffer is free once the MMA of its previous unit (j - AB) has finished.  The
        // parity wait is exact: that MMA's phase is the buffer's latest unless the one before
        // (unit j - 2 AB) is still open, and it is not: this group waited for unit j - 2 - AB
        // before its previous unit, and MMAs complete in issue order.
        uint8_t* const atp = abase + ab * kABuf;
        if (au > 0 && !warp_wait(a_empty0 + 8 * ab, (au - 1) & 1u)) {
          bail = true;
          break;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t pr[8];
          if constexpr (I8)
            decode16_i8(hq[q], pr);
          else
            decode16<Q8>(hq[q], lq[q], base2[q], a.mul, pr);
          uint8_t* row = atp + (8 * q + g) * 128;
          *reinterpret_cast<uint4*>(row + (((2 * t) ^ g) << 4)) = make_uint4(pr[0], pr[1], pr[2], pr[3]);
          *reinterpret_cast<uint4*>(row + (((2 * t + 1) ^ g) << 4)) = make_uint4(pr[4], pr[5], pr[6], pr[7]);
        }
        __syncwarp();  // the decoded stores of all lanes land before any escape overwrites a slot
        // a slot is an even byte offset below 4096 (32 rows of 128 bytes): the mask keeps a
        // damaged entry inside this warp's tile
        if ((uint32_t)lane < cnt) *reinterpret_cast<uint16_t*>(atp + (esc_slot(ent) & 0xFFEu)) = (uint16_t)esc_raw(ent);
        if (cnt > 32u) {
          for (uint32_t e = ta + 32 + lane; e < tb; e += 32) {
            const uint32_t en = __ldg(a.esc + e);
            *reinterpret_cast<uint16_t*>(atp + (esc_slot(en) & 0xFFEu)) = (uint16_t)esc_raw(en);
          }
        }
        fence_proxy_async_smem();  // this thread's generic-proxy stores -> tensor-core reads
        mbar_arrive(a_full0 + 8 * ab);
      }
      if (kc == KC - 1 || j == nunp - 1) {
        // ---- this unit ends a row block (or the CTA's share of one): the accumulator
        // from TMEM.  seg counts the segments of this CTA before this one.  The drains of
        // the earlier segments (by any group) end first; after them the accumulator
        // barrier is at most one phase from this segment's, so its parity wait is exact.
        const int seg = srb - srb0;
        if (seg > 0 && !wait_count(misc + 15, 4u * (uint32_t)seg)) {
          bail = true;
          break;
        }
        const int abuf = P::kAccBufs == 2 ? (seg & 1) : 0;
        if (!warp_wait(abuf ? epi0 : acc_full, (uint32_t)((seg / P::kAccBufs) & 1))) {
          bail = true;
          break;
        }
        tc_fence_after();
        const int64_t rt = (int64_t)rb * kBlockTiles + tl;
        const bool whole = U0 <= srb * KC && kc == KC - 1;
        const uint32_t trow = tmem + (uint32_t)(abuf * P::kTmemCols) + ((uint32_t)(tl * 32) << 16);
        if (whole) {
#pragma unroll 1
          for (int c0 = 0; c0 < NT; c0 += 16) {
            float v[16];
            tmem_ld16(trow + c0, v);
            emit_cols<EPI>(a, rt, lane, c0, v);
          }
          tc_fence_before();
          mbar_arrive(abuf ? epi0 + 8 : acc_empty);
          if (lane == 0) atomicAdd(misc + 15, 1u);
        } else {
          const int64_t cf = cta_of_unit((int64_t)srb * KC, a.G, a.T);
          const int64_t cl = cta_of_unit((int64_t)(srb + 1) * KC - 1, a.G, a.T);
          const int64_t ncov = cl - cf + 1;
          constexpr int kWarpSlot = NT * 32;  // floats per warp in a slot
          // slot of (part c, row srb): c + srb is unique among the parts covering a row;
          // a wide launch keeps one per pipeline
          auto slot_of = [&](int64_t c) { return P::kWide ? 2 * (c + srb) + pipe : c + srb; };
          float4* slot = reinterpret_cast<float4*>(a.slots + (slot_of(b) * kBlockTiles + tl) * kWarpSlot);
#pragma unroll 1
          for (int c0 = 0; c0 < NT; c0 += 16) {
            float v[16];
            tmem_ld16(trow + c0, v);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              __stcg(slot + (c0 / 4 + i) * 32 + lane, make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
          }
          tc_fence_before();
          mbar_arrive(abuf ? epi0 + 8 : acc_empty);
          if (lane == 0) atomicAdd(misc + 15, 1u);
          if (kDefer) {
            // the parts' slots are added after the launch
          } else if (P::kHasPub && j != nunp - 1) {
            // A partial row that ends before the range does is the range's first: the
            // publisher warp publishes it, and this group goes on decoding.  The barrier's
            // release orders each thread's slot stores before the publisher's increment.
            mbar_arrive(pub);
          } else {
            // Each warp publishes its own row tile: the warp barrier orders its lanes' slot
            // stores before lane 0's acquire-release increment of the tile's counter, which
            // publishes them at GPU scope; the last arriver's increment acquires every other
            // part's, and the second barrier orders the lanes' reads after it.
            __syncwarp();
            uint32_t arrived = 0u;
            if (lane == 0) arrived = atom_add_acq_rel(a.counters + rb * kBlockTiles + tl, 1u);
            arrived = __shfl_sync(0xFFFFFFFFu, arrived, 0);
            __syncwarp();
            const bool emit = (int64_t)arrived == ncov - 1;
            // At the pipeline's last unit every record stage and A buffer has been consumed
            // (the accumulator barrier follows every MMA, and each MMA follows its unit's
            // decode): each warp of the group then takes a quarter of that space and fetches
            // the parts' slots with bulk copies, all in flight at once, where the fallback
            // below waits for one L2 round trip per slot.  Both add the slots in part order.
            constexpr int kPiece = 16 * 32 * 4;  // 16 token columns of one warp's slot
            constexpr int kQuarter = ((P::kOffBar - P::kOffA) / 4) & ~(kPiece - 1);
            const int per = kQuarter / (kPiece * (int)ncov);  // column chunks per batch
            if (emit && j == nunp - 1 && per >= 1) {
              if (lane == 0) a.counters[rb * kBlockTiles + tl] = 0u;
              const uint32_t sc = sbase + P::kOffA + tl * kQuarter;
              const uint32_t fb = smem_u32(misc + 4 + 2 * tl);
              if (lane == 0) {
                mbar_init(fb, 1);
                mbar_init_fence();
                fence_proxy_async_smem();    // earlier generic accesses of the space -> the copies
                fence_proxy_async_global();  // the other parts' slots, acquired above -> the copies
              }
              __syncwarp();
              const uint64_t pol_s = policy_evict_first();
              uint32_t fph = 0;
#pragma unroll 1
              for (int c = 0; c < NT / 16 && !bail; c += per) {
                const int nb = min(per, NT / 16 - c);
                if (lane == 0) {
                  mbar_arrive_expect_tx(fb, (uint32_t)(nb * ncov * kPiece));
                  for (int cc = 0; cc < nb; ++cc)
                    for (int64_t jj = 0; jj < ncov; ++jj)
                      bulk_g2s(sc + (uint32_t)((cc * ncov + jj) * kPiece),
                               a.slots + (slot_of(cf + jj) * kBlockTiles + tl) * kWarpSlot + (c + cc) * 16 * 32, kPiece,
                               fb, pol_s);
                }
                if (!warp_wait(fb, fph)) {
                  if (lane == 0) mbar_wait_bounded(fb, fph);  // copies in flight land before the CTA leaves
                  bail = true;
                  break;
                }
                fph ^= 1u;
#pragma unroll 1
                for (int cc = 0; cc < nb; ++cc) {
                  float v[16];
#pragma unroll
                  for (int i = 0; i < 16; ++i) v[i] = 0.f;
                  for (int64_t jj = 0; jj < ncov; ++jj) {
                    const uint32_t pc = sc + (uint32_t)((cc * ncov + jj) * kPiece) + (uint32_t)lane * 16u;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                      const uint4 q4 = lds128(pc + (uint32_t)i * 512u);
                      v[4 * i] += __uint_as_float(q4.x);
                      v[4 * i + 1] += __uint_as_float(q4.y);
                      v[4 * i + 2] += __uint_as_float(q4.z);
                      v[4 * i + 3] += __uint_as_float(q4.w);
                    }
                  }
                  emit_cols<EPI>(a, rt, lane, (c + cc) * 16, v);
                }
                __syncwarp();  // every lane has read the batch before the next one lands
              }
              if (bail) break;
            } else if (emit) {
              if (lane == 0) a.counters[rb * kBlockTiles + tl] = 0u;
#pragma unroll 1
              for (int c0 = 0; c0 < NT; c0 += 16) {
                float v[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = 0.f;
                for (int64_t jj = 0; jj < ncov; ++jj) {
                  const float4* sj =
                      reinterpret_cast<const float4*>(a.slots + (slot_of(cf + jj) * kBlockTiles + tl) * kWarpSlot);
#pragma unroll
                  for (int i = 0; i < 4; ++i) {
                    const float4 q4 = __ldcg(sj + (c0 / 4 + i) * 32 + lane);
                    v[4 * i] += q4.x;
                    v[4 * i + 1] += q4.y;
                    v[4 * i + 2] += q4.z;
                    v[4 * i + 3] += q4.w;
                  }
                }
                emit_cols<EPI>(a, rt, lane, c0, v);
              }
            }
          }
        }
      }
      // G units on (S > G and AB >= G, so the ring and the buffers wrap at most once)
      ab += kTcGroups;
      if (ab >= AB) {
        ab -= AB;
        ++au;
      }
      s += kTcGroups;
      if (s >= S) {
        s -= S;
        ph ^= 1u;
      }
      kc += kTcGroups;
      while (kc >= KC) {
        kc -= KC;
        ++srb;
      }
    }
  }

  // ---- teardown: every warp reaches this point, TMEM is always freed
  if (lane == 0 && (bail || bad_index)) atomicOr(a.error, (bail ? kErrTimeout : 0u) | (bad_index ? kErrBounds : 0u));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kTcMma && pipe == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem0),
                 "n"(P::kPipes * P::kAccBufs * P::kTmemCols)
                 : "memory");
}

// Copy of x with row pitch ldx (a multiple of 8 elements), zero past K.
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

// Launch shape for M tokens on an N x K matrix: tokens per launch (the MMA's N), launch
// mode and places in the partition per SM.
struct LaunchShape {
  int nt, mode, parts;
};
LaunchShape launch_shape(int64_t M, int64_t N, int64_t K, int sms) {
  const int nt = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : M <= 192 ? 192 : 256;
  const int64_t RB = row_blocks(N);
  // up to 32 tokens: row-block pairs on tall matrices (a row block per SM or more), else two
  // pipelines with their own ranges
  if (nt <= 32) return RB >= sms ? LaunchShape{nt, kModePair, 1} : LaunchShape{nt, kModeOwn, 2};
  // row-block pairs: on matrices with a row block per SM or more, up to 192 tokens (at 256
  // a pipeline's record ring would drop to three stages)
  if (nt <= 192 && RB >= sms) return {nt, kModePair, 1};
  // shorter matrices: pairs summed after the launch where a CTA still gets 24 pair units or
  // more (long rows), else one pipeline per CTA
  if (nt <= 192 && ((RB + 1) / 2) * k_chunks(K) >= 24 * (int64_t)sms) return {nt, kModePairSum, 1};
  return {nt, kModeOne, 1};
}

// Units of the partition: row block x 64 columns, or row-block pair x 64 columns.
int64_t partition_units(int64_t N, int64_t K, int mode) {
  const int64_t RB = row_blocks(N), KC = k_chunks(K);
  return (mode == kModePair || mode == kModePairSum ? (RB + 1) / 2 : RB) * KC;
}

// CTAs of the stream-K partition for a T-unit problem.
int64_t partition_ctas(int64_t T, int sms, int bpsm) {
  const int64_t resident = (int64_t)sms * bpsm;
  const int64_t g = (T + kMinIters - 1) / kMinIters;
  return std::max<int64_t>(1, std::min(g, resident));
}

inline size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

// Workspace: the error word (first 256 bytes), the tile counters, then scratch that every
// call writes before reading.  The error word and counters start at zero.
struct WsLayout {
  size_t error, counters, slots, xpad, pbest, total;
};

WsLayout ws_layout(int64_t M, int64_t N, int64_t K, bool argmax, int sms) {
  const int64_t RB = row_blocks(N), RT = row_tiles(N), KC = k_chunks(K), T = RB * KC;
  const LaunchShape ls = launch_shape(M, N, K, sms);
  const int64_t TP = partition_units(N, K, ls.mode);
  const int64_t G = partition_ctas(TP, sms, ls.parts);
  const int64_t n_slots = ls.mode == kModePair || ls.mode == kModePairSum ? 2 * ((RB + 1) / 2 + G) : RB + G;
  WsLayout L{};
  L.error = 0;
  L.counters = 256;
  size_t off = 256 + align256((size_t)RB * kBlockTiles * 4);
  L.slots = off;  // one slot of 128 channels x nt tokens per (partition part, row block) pair
  off = align256(off + (size_t)n_slots * (size_t)(kBlockTiles * kTileRows) * (size_t)ls.nt * 4);
  L.xpad = off;
  off = align256(off + (size_t)M * (size_t)(KC * kTileK) * 2);
  L.pbest = off;
  if (argmax) off = align256(off + (size_t)RT * (size_t)M * 8);
  L.total = off;
  return L;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D tensor map over x[M][ldx] bf16: box of 64 columns x rows tokens, 128-byte swizzle.
int make_x_map(CUtensorMap* map, const uint16_t* x, int64_t M, int64_t K, int64_t ldx, int rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return fail(W12_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
  cuuint64_t strides[1] = {(cuuint64_t)ldx * 2};
  cuuint32_t box[2] = {(cuuint32_t)kTileK, (cuuint32_t)rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(W12_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return W12_OK;
}

template <int NT, bool Q8, int MODE, int EPI>
int launch_tc(const CUtensorMap& map, const GemmArgs& a, cudaStream_t s) {
  using P = TcPlan<NT, Q8, MODE>;
  constexpr int smem = P::kCtaBytes;
  static int configured_for_device[64] = {0};
  int dev = 0;
  W12_CUDA_TRY(cudaGetDevice(&dev));
  if (dev >= 64 || !configured_for_device[dev]) {
    W12_CUDA_TRY(cudaFuncSetAttribute(k_gemm_tc<NT, Q8, MODE, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    if (dev < 64) configured_for_device[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((a.G + P::kParts - 1) / P::kParts));
  cfg.blockDim = dim3(P::kCtaThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  W12_CUDA_TRY(cudaLaunchKernelEx(&cfg, k_gemm_tc<NT, Q8, MODE, EPI>, map, a));
  W12_LAUNCH_CHECK("w12 gemm kernel (tcgen05)");
  return W12_OK;
}

template <bool Q8, int EPI>
int launch_nt(const LaunchShape& ls, const CUtensorMap& map, const GemmArgs& a, cudaStream_t s) {
  // pairs summed after the launch store y; for the other outputs they are plain pairs
  const bool pair = ls.mode == kModePair || (ls.mode == kModePairSum && EPI != EPI_STORE);
  if constexpr (EPI == EPI_STORE) {
    if (ls.mode == kModePairSum) {
      if (ls.nt == 64) return launch_tc<64, Q8, kModePairSum, EPI>(map, a, s);
      if (ls.nt == 128) return launch_tc<128, Q8, kModePairSum, EPI>(map, a, s);
      return launch_tc<192, Q8, kModePairSum, EPI>(map, a, s);
    }
  }
  switch (ls.nt) {
    case 16: return pair ? launch_tc<16, Q8, kModePair, EPI>(map, a, s) : launch_tc<16, Q8, kModeOwn, EPI>(map, a, s);
    case 32: return pair ? launch_tc<32, Q8, kModePair, EPI>(map, a, s) : launch_tc<32, Q8, kModeOwn, EPI>(map, a, s);
    case 64: return pair ? launch_tc<64, Q8, kModePair, EPI>(map, a, s) : launch_tc<64, Q8, kModeOne, EPI>(map, a, s);
    case 128:
      return pair ? launch_tc<128, Q8, kModePair, EPI>(map, a, s) : launch_tc<128, Q8, kModeOne, EPI>(map, a, s);
    case 192:
      return pair ? launch_tc<192, Q8, kModePair, EPI>(map, a, s) : launch_tc<192, Q8, kModeOne, EPI>(map, a, s);
    default: return launch_tc<256, Q8, kModeOne, EPI>(map, a, s);
  }
}

// y of the rows that a launch split between CTAs: the parts' slots added in part order from
// zero, as the in-kernel fix-up adds them.  Block (row tile, group of 8 token quads); thread
// (lane = channel of the row tile, quad).  Row blocks held by one part were stored by the GEMM.
__global__ void __launch_bounds__(256) k_slot_sum(const float* __restrict__ slots, float* __restrict__ y,
                                                  int64_t ldy, int64_t N, int M, int nt, int64_t KC, int64_t G,
                                                  int64_t T, bool wide) {
  // the next GEMM may start streaming its weights; it reads x only after this grid completes
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ int64_t parts[2];
  const int64_t rt = blockIdx.x, rb = rt / kBlockTiles;
  const int tl = (int)(rt % kBlockTiles);
  // row of the partition: the row block, or with row-block pairs the pair (pipeline rb & 1)
  const int64_t srb = wide ? rb >> 1 : rb;
  if (threadIdx.x == 0) {
    parts[0] = cta_of_unit(srb * KC, G, T);
    parts[1] = cta_of_unit((srb + 1) * KC - 1, G, T);
  }
  __syncthreads();
  const int64_t cf = parts[0], cl = parts[1];
  const int lane = threadIdx.x & 31, q = (int)blockIdx.y * 8 + (threadIdx.x >> 5), tok = 4 * q;
  const int64_t n = rt * kTileRows + lane;
  if (cf == cl || tok >= M || n >= N) return;
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t c = cf; c <= cl; ++c) {
    // slot of (part c, row block rb): [row tile][token quad][lane] float4
    const int64_t slot = wide ? 2 * (c + srb) + (rb & 1) : c + srb;
    const float4 p =
        __ldcg(reinterpret_cast<const float4*>(slots + (slot * kBlockTiles + tl) * (int64_t)nt * 32) + q * 32 + lane);
    v.x += p.x;
    v.y += p.y;
    v.z += p.z;
    v.w += p.w;
  }
  float* yo = y + (int64_t)tok * ldy + n;
  yo[0] = v.x;
  if (tok + 1 < M) yo[ldy] = v.y;
  if (tok + 2 < M) yo[2 * ldy] = v.z;
  if (tok + 3 < M) yo[3 * ldy] = v.w;
}

// Host-side checks of a GEMM call's arguments (everything but the workspace); a call that
// fails them touches no memory.
int check_gemm_args(const uint16_t* x, int64_t M, const w12_matrix* A, const float* y, const int32_t* tok, bool q8,
                    bool argmax, bool i8, const char* fn) {
  // i8: A->hi holds INT8 codes (the caller has checked A's shape and pointers)
  int st = i8 ? W12_OK : check_matrix(A, !q8, fn);
  if (st) return st;
  if (!x || (!argmax && !i8 && !y) || (argmax && !tok)) return fail(W12_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (M < 1 || M > (1 << 20)) return fail(W12_ERR_SHAPE, "%s: M=%lld out of range (1..2^20)", fn, (long long)M);
  if ((((uintptr_t)A->hi | (uintptr_t)A->lo | (uintptr_t)A->esc) & 15u) != 0)
    return fail(W12_ERR_INVALID_ARG, "%s: hi, lo and esc must be 16-byte aligned", fn);
  const int64_t T = row_blocks(A->N) * k_chunks(A->K);
  if (T >= (int64_t(1) << 30))
    return fail(W12_ERR_SHAPE, "%s: %lld row blocks x %lld column chunks exceed 2^30 units", fn,
                (long long)row_blocks(A->N), (long long)k_chunks(A->K));
  return W12_OK;
}

int run_gemm(const uint16_t* x, int64_t M, const w12_matrix* A, float* y, int32_t* tok, bool q8, bool argmax,
             void* ws, size_t ws_bytes, cudaStream_t s, const char* fn, const float* i8_scale = nullptr,
             const CertEpi* cert = nullptr) {
  int st = check_gemm_args(x, M, A, y, tok, q8, argmax, i8_scale != nullptr, fn);
  if (st) return st;
  if (!ws) return fail(W12_ERR_INVALID_ARG, "%s: null workspace", fn);
  int sms = 0;
  if ((st = device_sms(&sms))) return st;
  const WsLayout L = ws_layout(M, A->N, A->K, argmax, sms);
  if (ws_bytes < L.total)
    return fail(W12_ERR_BUFFER_TOO_SMALL, "%s: workspace %zu bytes < %zu required", fn, ws_bytes, L.total);
  const int64_t RB = row_blocks(A->N), RT = row_tiles(A->N), KC = k_chunks(A->K);
  uint8_t* wsb = static_cast<uint8_t*>(ws);

  // x through a tensor map needs a 16-byte aligned base and a row pitch that is a multiple of 16 bytes
  const uint16_t* xs = x;
  int64_t ldx = A->K;
  if ((A->K % 8) != 0 || ((uintptr_t)x & 15u) != 0) {
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
  a.RB = RB;
  const LaunchShape ls = launch_shape(M, A->N, A->K, sms);
  a.T = partition_units(A->N, A->K, ls.mode);
  a.G = partition_ctas(a.T, sms, ls.parts);
  a.ldy = A->N;
  a.slots = reinterpret_cast<float*>(wsb + L.slots);
  a.counters = reinterpret_cast<uint32_t*>(wsb + L.counters);
  a.error = reinterpret_cast<uint32_t*>(wsb + L.error);
  a.pbest = reinterpret_cast<unsigned long long*>(wsb + L.pbest);
  a.ldp = M;
  a.mul = W12_DECODE_MUL;
  a.scale = i8_scale;
  a.n_esc = i8_scale ? 0u : (uint32_t)A->n_esc;
  if (cert) a.cert = *cert;
  CUtensorMap map;
  if ((st = make_x_map(&map, xs, M, A->K, ldx, ls.nt))) return st;
  for (int64_t m0 = 0; m0 < M; m0 += ls.nt) {
    const int Mg = (int)std::min<int64_t>(ls.nt, M - m0);
    a.M = Mg;
    a.tok0 = (int)m0;
    if (i8_scale) {
      st = launch_nt<true, EPI_I8>(ls, map, a, s);
    } else if (!argmax) {
      a.y = y + m0 * A->N;
      st = q8 ? launch_nt<true, EPI_STORE>(ls, map, a, s) : launch_nt<false, EPI_STORE>(ls, map, a, s);
      if (!st && ((ls.mode == kModeOne && ls.nt == 192) || ls.mode == kModePairSum)) {
        // plain launch: it starts when the GEMM's grid has completed
        // 8 token quads per block (nt is a multiple of 32 here); fewer than 2^31 row tiles
        const dim3 grid((unsigned)(RB * kBlockTiles), (unsigned)(ls.nt / 32));
        k_slot_sum<<<grid, 256, 0, s>>>(a.slots, a.y, a.ldy, A->N, Mg, ls.nt, KC, a.G, a.T, ls.mode == kModePairSum);
        W12_LAUNCH_CHECK("w12 gemm: split row blocks");
      }
    } else {
      st = q8 ? launch_nt<true, EPI_ARGMAX>(ls, map, a, s) : launch_nt<false, EPI_ARGMAX>(ls, map, a, s);
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

// used by w12_cert.cu: the approximate logits scale[v] * (x . codes^T) of an INT8 head whose
// code plane (hi-plane layout) is codes, fed to the certified argmax's threshold and
// candidate superset (CertEpi); ws as for w12_gemm.
int i8_gemm_impl(const uint16_t* x, int64_t M, const uint8_t* codes, const float* scale, int64_t V, int64_t K,
                 const float* nx, const float* cb, uint32_t* thr_key, uint32_t* sup_count, uint2* sup,
                 int64_t ldsup, void* ws, size_t ws_bytes, cudaStream_t s, const char* fn) {
  w12_matrix A{};
  A.N = V;
  A.K = K;
  A.hi = const_cast<uint8_t*>(codes);
  const CertEpi cert{nx, cb, thr_key, sup_count, sup, ldsup};
  return run_gemm(x, M, &A, nullptr, nullptr, true, false, ws, ws_bytes, s, fn, scale, &cert);
}

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

size_t w12_gemm_counter_bytes(int64_t N) {
  return N >= 1 ? 256 + align256((size_t)row_blocks(N) * kBlockTiles * 4) : 0;
}

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

int w12_workspace_status(void* ws, size_t ws_bytes, int32_t* status, void* stream) {
  const char* fn = "w12_workspace_status";
  if (!ws || !status) return fail(W12_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (ws_bytes < 256) return fail(W12_ERR_BUFFER_TOO_SMALL, "%s: a workspace holds at least 256 bytes", fn);
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t word = 0;
  W12_CUDA_TRY(cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, s));
  W12_CUDA_TRY(cudaStreamSynchronize(s));
  *status = (word & kErrTimeout) ? W12_ERR_TIMEOUT : (word & kErrBounds) ? W12_ERR_BOUNDS : W12_OK;
  // a CTA that gave up may have left tile counters raised: start the next call clean
  if (word) W12_CUDA_TRY(cudaMemsetAsync(ws, 0, ws_bytes, s));
  return W12_OK;
}

int w12_set_wait_limit(int64_t cycles) {
  const long long v = cycles > 0 ? (long long)cycles : kWaitCycles;
  W12_CUDA_TRY(cudaMemcpyToSymbol(c_wait_limit, &v, sizeof(v)));
  return W12_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// w12_gemm without a caller workspace.
//
// Some callers cannot give this library a workspace: an inference engine
// whose memory planner has already handed out the whole device, a plugin or
// callback interface whose signature has no workspace argument, or a
// latency-critical loop that must not call cudaMalloc (it can synchronise the
// device).  For them the GEMM's scratch (stream-K tile counters, the error
// word, partial-sum slots and, for unaligned x, a padded copy of x) lives in
// one file-scope device array.  Every GPU that loads the library keeps this
// array until the process exits.  The array's name is only a host-side stand-in;
// its device address comes from cudaGetSymbolAddress, looked up once per
// device with that device current, on the first call.
namespace w12 {

constexpr size_t kFixedScratchBytes = size_t(16) << 20;  // 16 MiB
static __device__ __align__(256) uint8_t g_fixed_scratch[kFixedScratchBytes];

static int fixed_scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "w12_gemm_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(W12_ERR_INVALID_ARG, "w12_gemm_noalloc: device %d out of range", dev);
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_fixed_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "w12_gemm_noalloc: cudaGetSymbolAddress");
    addr[dev] = p;
  }
  *out = addr[dev];
  return W12_OK;
}

}  // namespace w12

extern "C" {

size_t w12_gemm_noalloc_max_scratch(void) { return w12::kFixedScratchBytes; }

int w12_gemm_noalloc(const uint16_t* x, int64_t M, const w12_matrix* A, float* y, void* stream) {
  using namespace w12;
  const char* fn = "w12_gemm_noalloc";
  // every argument check comes before the scratch is touched: a refused call leaves it alone
  int st = check_gemm_args(x, M, A, y, nullptr, false, false, false, fn);
  if (st) return st;
  int sms = 0;
  if ((st = device_sms(&sms))) return st;
  const WsLayout L = ws_layout(M, A->N, A->K, false, sms);
  if (L.total > kFixedScratchBytes)
    return fail(W12_ERR_SHAPE,
                "%s: M=%lld N=%lld K=%lld needs %zu bytes of scratch; the fixed scratch holds %zu "
                "(use w12_gemm with a workspace)",
                fn, (long long)M, (long long)A->N, (long long)A->K, L.total, kFixedScratchBytes);
  void* scratch = nullptr;
  if ((st = fixed_scratch_address(&scratch))) return st;
  cudaStream_t s = (cudaStream_t)stream;
  // the error word and the tile counters must start at zero on every call
  W12_CUDA_TRY(cudaMemsetAsync(scratch, 0, L.slots, s));
  return run_gemm(x, M, A, y, nullptr, false, false, scratch, kFixedScratchBytes, s, fn);
}

}  // extern "C"
