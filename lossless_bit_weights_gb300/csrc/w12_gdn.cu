// w12_gdn.cu - recurrent-layer verification for a hybrid target.
//
// The SpecPilot summary page (onedev.kr/papers/1654), section "What's
// different", verifies a draft tree on a target whose layers are mostly Gated
// DeltaNet with a path-verify kernel that recomputes the recurrent state along
// each path instead of snapshotting it per node, a commit kernel that replays
// the accepted path into the layers' states, and a WY kernel that keeps the
// FP32 state as three BF16 pieces holding its 24-bit significand exactly.
// The recurrence is the gated delta rule on a dv x dk state per head:
//     S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
//     o_t = S_t q_t,
// so one step is a row dot u = S k and a rank-1 write
//     S <- alpha S + (beta v - alpha beta u) k^T.
#include <cstdint>
#include <mutex>

#include "w12_internal.cuh"

namespace w12 {
namespace {

constexpr int64_t kGdnMaxNodes = 4096;  // tree size a path-verify launch accepts
constexpr int64_t kGdnMaxDim = 256;     // dk, dv

__device__ __forceinline__ float bf16v(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

__device__ __forceinline__ uint16_t bf16_rne(float f) {
  uint32_t u = __float_as_uint(f);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

__global__ void k_split3(const float* __restrict__ x, int64_t n, uint16_t* __restrict__ s1, uint16_t* __restrict__ s2,
                         uint16_t* __restrict__ s3) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const float a = x[i];
    const uint16_t p1 = bf16_rne(a);
    const float r1 = __fsub_rn(a, bf16v(p1));
    const uint16_t p2 = bf16_rne(r1);
    const float r2 = __fsub_rn(r1, bf16v(p2));
    s1[i] = p1;
    s2[i] = p2;
    s3[i] = bf16_rne(r2);
  }
}

// The head's state lives in shared memory row-major with a row stride of dk + 4 floats;
// four threads share row r = t/4, thread part p = t%4 holding columns p, p+4, p+8, ...
// (the stride puts the 32 threads of a warp on 32 distinct banks).  kv holds the step's
// k (dk floats) then v (dv floats).
__device__ __forceinline__ int64_t srow(int64_t dk) { return dk + 4; }

// State copies in 32-bit index arithmetic (dv * dk <= 65536), four floats at a time when
// the rows allow it (dk % 4 == 0: rows and the 16-byte-aligned head stay aligned).
__device__ __forceinline__ void gdn_load(const float* __restrict__ S0, int64_t dk, int64_t dv, float* S) {
  const uint32_t K = (uint32_t)dk, R = (uint32_t)srow(dk);
  if ((K & 3u) == 0 && (((uintptr_t)S0) & 15u) == 0) {
    const uint32_t K4 = K >> 2, n4 = (uint32_t)dv * K4;
    for (uint32_t e = threadIdx.x; e < n4; e += blockDim.x) {
      const uint32_t r = e / K4, c = (e - r * K4) << 2;
      *reinterpret_cast<float4*>(S + r * R + c) = reinterpret_cast<const float4*>(S0)[e];
    }
  } else {
    for (uint32_t e = threadIdx.x; e < (uint32_t)dv * K; e += blockDim.x) {
      const uint32_t r = e / K, c = e - r * K;
      S[r * R + c] = S0[e];
    }
  }
}

__device__ __forceinline__ void gdn_store(float* __restrict__ S_out, int64_t dk, int64_t dv, const float* S) {
  const uint32_t K = (uint32_t)dk, R = (uint32_t)srow(dk);
  if ((K & 3u) == 0 && (((uintptr_t)S_out) & 15u) == 0) {
    const uint32_t K4 = K >> 2, n4 = (uint32_t)dv * K4;
    for (uint32_t e = threadIdx.x; e < n4; e += blockDim.x) {
      const uint32_t r = e / K4, c = (e - r * K4) << 2;
      reinterpret_cast<float4*>(S_out)[e] = *reinterpret_cast<const float4*>(S + r * R + c);
    }
  } else {
    for (uint32_t e = threadIdx.x; e < (uint32_t)dv * K; e += blockDim.x) {
      const uint32_t r = e / K, c = e - r * K;
      S_out[e] = S[r * R + c];
    }
  }
}

// Inputs of one step, one element of k and of v per thread (blockDim >= dk, dv), fetched a
// step ahead so that their loads overlap the step before.
struct StepIn {
  float k, v, alpha, beta;
};

__device__ __forceinline__ StepIn fetch_step(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                                             const float* __restrict__ alpha, const float* __restrict__ beta,
                                             int64_t j, int64_t h, int64_t H, int64_t dk, int64_t dv) {
  StepIn in;
  const int64_t t = threadIdx.x;
  in.k = t < dk ? bf16v(k[(j * H + h) * dk + t]) : 0.f;
  in.v = t < dv ? bf16v(v[(j * H + h) * dv + t]) : 0.f;
  in.alpha = alpha[j * H + h];
  in.beta = beta[j * H + h];
  return in;
}

// Row dot of this thread's row with a dk-vector in shared memory, summed over the row's
// four threads (two shuffles); every thread of the row gets the sum.
__device__ __forceinline__ float row_dot(const float* Srow, const float* vec, int64_t dk, int p) {
  float a0 = 0.f, a1 = 0.f;
  int64_t c = p;
  for (; c + 4 < dk; c += 8) {
    a0 = fmaf(Srow[c], vec[c], a0);
    a1 = fmaf(Srow[c + 4], vec[c + 4], a1);
  }
  if (c < dk) a0 = fmaf(Srow[c], vec[c], a0);
  float u = a0 + a1;
  u += __shfl_xor_sync(0xFFFFFFFFu, u, 1);
  u += __shfl_xor_sync(0xFFFFFFFFu, u, 2);
  return u;
}

// One gated delta step (all threads of the block) with this thread's prefetched inputs.
__device__ __forceinline__ void gdn_step(float* S, float* kv, int64_t dk, int64_t dv, const StepIn& in) {
  __syncthreads();  // the previous step's reads of kv are done
  if (threadIdx.x < dk) kv[threadIdx.x] = in.k;
  if (threadIdx.x < dv) kv[dk + threadIdx.x] = in.v;
  __syncthreads();
  const int64_t r = threadIdx.x >> 2;
  const int p = threadIdx.x & 3;
  float* Srow = S + r * srow(dk);
  const float u = row_dot(Srow, kv, dk, p);  // all four threads of a row, rows past dv included
  if (r < dv) {
    const float coef = in.beta * kv[dk + r] - in.alpha * in.beta * u;
    for (int64_t c = p; c < dk; c += 4) Srow[c] = fmaf(in.alpha, Srow[c], coef * kv[c]);
  }
}

// One block per (node i = blockIdx.x, head h = blockIdx.y).
__global__ void k_gdn_path_verify(const float* __restrict__ S0, const uint16_t* __restrict__ q,
                                  const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                                  const float* __restrict__ alpha, const float* __restrict__ beta,
                                  const int32_t* __restrict__ parent, int64_t n, int64_t H, int64_t dk, int64_t dv,
                                  float* __restrict__ O, int32_t* __restrict__ status) {
  extern __shared__ float gsm[];
  __shared__ int32_t path[kGdnMaxNodes];
  __shared__ int32_t plen;
  const int64_t i = blockIdx.x, h = blockIdx.y;
  float* S = gsm;
  float* kv = gsm + (int64_t)(blockDim.x >> 2) * srow(dk);  // a row per four threads, rows past dv spare
  if (threadIdx.x == 0) {
    // node i up to the first draft node; a parent that is not an earlier node stops the walk
    int32_t L = 0;
    bool ok = parent[0] == -1;
    for (int64_t j = i; ok && j > 0;) {
      const int32_t p = parent[j];
      if (p < 0 || p >= j) {
        ok = false;
        break;
      }
      path[L++] = (int32_t)j;
      j = p;
    }
    if (!ok) {
      atomicOr(status, 1);
      L = -1;
    }
    plen = L;
  }
  gdn_load(S0 + h * dv * dk, dk, dv, S);
  __syncthreads();
  const int32_t L = plen;
  if (L < 0) return;
  StepIn in{};
  if (L > 0) in = fetch_step(k, v, alpha, beta, path[L - 1], h, H, dk, dv);
  const float qx = threadIdx.x < dk ? bf16v(q[(i * H + h) * dk + threadIdx.x]) : 0.f;
  for (int32_t t = L - 1; t >= 0; --t) {
    const StepIn cur = in;
    if (t > 0) in = fetch_step(k, v, alpha, beta, path[t - 1], h, H, dk, dv);
    gdn_step(S, kv, dk, dv, cur);
  }
  __syncthreads();
  if (threadIdx.x < dk) kv[threadIdx.x] = qx;
  __syncthreads();
  const int64_t r = threadIdx.x >> 2;
  const float o = row_dot(S + r * srow(dk), kv, dk, threadIdx.x & 3);
  if (r < dv && (threadIdx.x & 3) == 0) O[(i * H + h) * dv + r] = o;
}

// One block per head: S <- the state after the accepted nodes path_nodes[1 .. *path_len]
// (path_nodes[0] is the root, whose update is already in S).  A path length below zero
// (an invalid tree in the acceptance call) commits nothing.
__global__ void k_gdn_commit(float* __restrict__ S_io, const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                             const float* __restrict__ alpha, const float* __restrict__ beta,
                             const int32_t* __restrict__ path_len, const int32_t* __restrict__ path_nodes, int64_t n,
                             int64_t H, int64_t dk, int64_t dv, int32_t* __restrict__ status) {
  extern __shared__ float gsm[];
  const int64_t h = blockIdx.x;
  float* S = gsm;
  float* kv = gsm + (int64_t)(blockDim.x >> 2) * srow(dk);
  const int32_t L = *path_len;
  if (L <= 0) return;
  if (L >= n) {
    if (threadIdx.x == 0) atomicOr(status, 2);
    return;
  }
  for (int32_t t = 1; t <= L; ++t) {  // every node checked before the state is touched
    const int32_t j = path_nodes[t];
    if (j <= 0 || j >= n) {  // block-uniform: every thread reads the same entries
      if (threadIdx.x == 0) atomicOr(status, 2);
      return;
    }
  }
  gdn_load(S_io + h * dv * dk, dk, dv, S);
  StepIn in = fetch_step(k, v, alpha, beta, path_nodes[1], h, H, dk, dv);
  for (int32_t t = 1; t <= L; ++t) {
    const StepIn cur = in;
    if (t < L) in = fetch_step(k, v, alpha, beta, path_nodes[t + 1], h, H, dk, dv);
    gdn_step(S, kv, dk, dv, cur);
  }
  __syncthreads();
  gdn_store(S_io + h * dv * dk, dk, dv, S);
}

// ---- register-resident state for dk = 64 and 128.  The rows of a state evolve
// independently (they share only k and v), so a block takes 32 rows: thread
// (r = t/4, p = t%4) of the 128 keeps columns [p*Q, p*Q + Q) of row r0 + r in registers
// (Q = DK/4); k, v and q go through shared memory with each quarter of k padded by 4
// floats (the four quarters on distinct banks).
constexpr int kRegRows = 32;
constexpr int kRegThreads = 4 * kRegRows;

template <int DK>
struct RegState {
  static constexpr int Q = DK / 4;
  float s[Q];
};

template <int DK>
__device__ __forceinline__ void reg_load(RegState<DK>& S, const float* __restrict__ src, int64_t rows) {
  const int64_t r = threadIdx.x >> 2;
  const int p = threadIdx.x & 3;
  if (r < rows) {
    const float4* g = reinterpret_cast<const float4*>(src + r * DK + p * RegState<DK>::Q);
#pragma unroll
    for (int m = 0; m < RegState<DK>::Q / 4; ++m) {
      const float4 f = g[m];
      S.s[4 * m] = f.x;
      S.s[4 * m + 1] = f.y;
      S.s[4 * m + 2] = f.z;
      S.s[4 * m + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int m = 0; m < RegState<DK>::Q; ++m) S.s[m] = 0.f;
  }
}

template <int DK>
__device__ __forceinline__ void reg_store(const RegState<DK>& S, float* __restrict__ dst, int64_t rows) {
  const int64_t r = threadIdx.x >> 2;
  const int p = threadIdx.x & 3;
  if (r < rows) {
    float4* g = reinterpret_cast<float4*>(dst + r * DK + p * RegState<DK>::Q);
#pragma unroll
    for (int m = 0; m < RegState<DK>::Q / 4; ++m)
      g[m] = make_float4(S.s[4 * m], S.s[4 * m + 1], S.s[4 * m + 2], S.s[4 * m + 3]);
  }
}

// padded position of element c of k (or q) in shared memory
template <int DK>
__device__ __forceinline__ int vpos(int c) {
  return c + (c / RegState<DK>::Q) * 4;
}

template <int DK>
__device__ __forceinline__ float reg_dot(const RegState<DK>& S, const float* vec) {
  constexpr int Q = RegState<DK>::Q;
  const float4* v4 = reinterpret_cast<const float4*>(vec + (threadIdx.x & 3) * (Q + 4));
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int m = 0; m < Q / 4; ++m) {
    const float4 f = v4[m];
    a0 = fmaf(S.s[4 * m], f.x, a0);
    a1 = fmaf(S.s[4 * m + 1], f.y, a1);
    a0 = fmaf(S.s[4 * m + 2], f.z, a0);
    a1 = fmaf(S.s[4 * m + 3], f.w, a1);
  }
  float u = a0 + a1;
  u += __shfl_xor_sync(0xFFFFFFFFu, u, 1);
  u += __shfl_xor_sync(0xFFFFFFFFu, u, 2);
  return u;
}

// One step's inputs: k element t (t < DK), v of row r0 + t (t < 32), alpha, beta.
template <int DK>
__device__ __forceinline__ StepIn fetch_rows(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                                             const float* __restrict__ alpha, const float* __restrict__ beta,
                                             int64_t j, int64_t h, int64_t H, int64_t dv, int64_t r0) {
  StepIn in;
  const int64_t t = threadIdx.x;
  in.k = t < DK ? bf16v(k[(j * H + h) * DK + t]) : 0.f;
  in.v = t < kRegRows && r0 + t < dv ? bf16v(v[(j * H + h) * dv + r0 + t]) : 0.f;
  in.alpha = alpha[j * H + h];
  in.beta = beta[j * H + h];
  return in;
}

// kv: k (padded, 4*(Q+4) floats) then the block's 32 v values
template <int DK>
__device__ __forceinline__ void reg_step(RegState<DK>& S, float* kv, const StepIn& in) {
  constexpr int Q = RegState<DK>::Q;
  __syncthreads();  // the previous step's reads of kv are done
  if (threadIdx.x < DK) kv[vpos<DK>(threadIdx.x)] = in.k;
  if (threadIdx.x < kRegRows) kv[4 * (Q + 4) + threadIdx.x] = in.v;
  __syncthreads();
  const float u = reg_dot<DK>(S, kv);
  const float coef = in.beta * kv[4 * (Q + 4) + (threadIdx.x >> 2)] - in.alpha * in.beta * u;
  const float4* k4 = reinterpret_cast<const float4*>(kv + (threadIdx.x & 3) * (Q + 4));
#pragma unroll
  for (int m = 0; m < Q / 4; ++m) {
    const float4 f = k4[m];
    S.s[4 * m] = fmaf(in.alpha, S.s[4 * m], coef * f.x);
    S.s[4 * m + 1] = fmaf(in.alpha, S.s[4 * m + 1], coef * f.y);
    S.s[4 * m + 2] = fmaf(in.alpha, S.s[4 * m + 2], coef * f.z);
    S.s[4 * m + 3] = fmaf(in.alpha, S.s[4 * m + 3], coef * f.w);
  }
}

// grid (node, head, row block of 32)
template <int DK>
__global__ void __launch_bounds__(kRegThreads) k_gdn_path_verify_reg(
    const float* __restrict__ S0, const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
    const uint16_t* __restrict__ v, const float* __restrict__ alpha, const float* __restrict__ beta,
    const int32_t* __restrict__ parent, int64_t n, int64_t H, int64_t dv, float* __restrict__ O,
    int32_t* __restrict__ status) {
  constexpr int Q = RegState<DK>::Q;
  __shared__ __align__(16) float kv[4 * (Q + 4) + kRegRows];
  __shared__ int32_t path[kGdnMaxNodes];
  __shared__ int32_t plen;
  const int64_t i = blockIdx.x, h = blockIdx.y, r0 = (int64_t)blockIdx.z * kRegRows;
  // the next kernel on the stream may start now (programmatic dependent launch); the state
  // is read before this one waits for the previous kernel, the node inputs after
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  RegState<DK> S;
  reg_load<DK>(S, S0 + (h * dv + r0) * DK, dv - r0);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) {
    int32_t L = 0;
    bool ok = parent[0] == -1;
    for (int64_t j = i; ok && j > 0;) {
      const int32_t p = parent[j];
      if (p < 0 || p >= j) {
        ok = false;
        break;
      }
      path[L++] = (int32_t)j;
      j = p;
    }
    if (!ok) {
      if (blockIdx.z == 0) atomicOr(status, 1);
      L = -1;
    }
    plen = L;
  }
  __syncthreads();
  const int32_t L = plen;
  if (L < 0) return;
  StepIn in{};
  if (L > 0) in = fetch_rows<DK>(k, v, alpha, beta, path[L - 1], h, H, dv, r0);
  const float qx = threadIdx.x < DK ? bf16v(q[(i * H + h) * DK + threadIdx.x]) : 0.f;
  for (int32_t t = L - 1; t >= 0; --t) {
    const StepIn cur = in;
    if (t > 0) in = fetch_rows<DK>(k, v, alpha, beta, path[t - 1], h, H, dv, r0);
    reg_step<DK>(S, kv, cur);
  }
  __syncthreads();
  if (threadIdx.x < DK) kv[vpos<DK>(threadIdx.x)] = qx;
  __syncthreads();
  const float o = reg_dot<DK>(S, kv);
  const int64_t r = r0 + (threadIdx.x >> 2);
  if (r < dv && (threadIdx.x & 3) == 0) O[(i * H + h) * dv + r] = o;
}

// grid (head, row block of 32)
template <int DK>
__global__ void __launch_bounds__(kRegThreads) k_gdn_commit_reg(
    float* __restrict__ S_io, const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
    const float* __restrict__ alpha, const float* __restrict__ beta, const int32_t* __restrict__ path_len,
    const int32_t* __restrict__ path_nodes, int64_t n, int64_t H, int64_t dv, int32_t* __restrict__ status) {
  constexpr int Q = RegState<DK>::Q;
  __shared__ __align__(16) float kv[4 * (Q + 4) + kRegRows];
  const int64_t h = blockIdx.x, r0 = (int64_t)blockIdx.y * kRegRows;
  // launched early behind a kernel that signals early, it waits for that kernel before it
  // reads anything; it never signals early itself, since it writes the state
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int32_t L = *path_len;
  if (L <= 0) return;
  if (L >= n) {
    if (threadIdx.x == 0 && blockIdx.y == 0) atomicOr(status, 2);
    return;
  }
  for (int32_t t = 1; t <= L; ++t) {
    const int32_t j = path_nodes[t];
    if (j <= 0 || j >= n) {
      if (threadIdx.x == 0 && blockIdx.y == 0) atomicOr(status, 2);
      return;
    }
  }
  RegState<DK> S;
  float* base = S_io + (h * dv + r0) * DK;
  reg_load<DK>(S, base, dv - r0);
  StepIn in = fetch_rows<DK>(k, v, alpha, beta, path_nodes[1], h, H, dv, r0);
  for (int32_t t = 1; t <= L; ++t) {
    const StepIn cur = in;
    if (t < L) in = fetch_rows<DK>(k, v, alpha, beta, path_nodes[t + 1], h, H, dv, r0);
    reg_step<DK>(S, kv, cur);
  }
  reg_store<DK>(S, base, dv - r0);
}

// ---- WY form on the tensor core: every node of the tree at once.  With gamma_t the
// product of alpha along t's path, node t's state is
//     S_t = gamma_t S0 + sum_{j on path(t)} (gamma_t/gamma_j) d_j k_j^T,
// whose pseudo-values d_j solve, in node order (ancestors come first),
//     d_t = beta_t (v_t - gamma_t S0 k_t - sum_{j ancestor of t} (gamma_t/gamma_j) (k_j.k_t) d_j),
// and o_t = gamma_t S0 q_t + sum_{j on path(t)} (gamma_t/gamma_j) (k_j.q_t) d_j.  The state
// enters only through the products S0 [k_0 .. k_{n-1} q_0 .. q_{n-1}], one matrix product
// per head.  It runs on the tensor core in bf16 with the float state held exactly as three
// bf16 pieces, S0 = s1 + s2 + s3 (gdn_split3's split): the pieces are the A operand (128
// state rows x 3 dk columns), the node vectors the B operand (each repeated for the three
// pieces), so every product of a piece and a k or q element is exact and the tensor core
// accumulates them in fp32.  A second product gives the node tables k_t.k_j and q_t.k_j.
// The per-row substitution over the tree then runs on the CUDA cores, one thread per row.
//
// One CTA per (head, 128 state rows): the rows arrive by one bulk copy, 16 warps split them
// into the three pieces in the operands' 128-byte-swizzled layout, one thread issues the
// MMAs (accumulators in tensor memory), four warps read the state products back (lane =
// state row) and four the node tables, and four warps run the substitution and the outputs
// with each row's pseudo-values in registers.
constexpr int kWyMaxNodes = 64;
constexpr int kWyRows = 128;                 // state rows per CTA: the MMA's M
constexpr int kWyThreads = 512;
constexpr int kWyTile = kWyRows * 128;       // one operand tile: 128 rows x 64 bf16 (16 KB)

template <int DK>
struct WyPlan {
  static constexpr int KB = DK / 64;                       // 64-column blocks of a vector
  static constexpr int kPieces = 0;                        // 3*KB tiles: piece p, block kb
  static constexpr int kNodes = 3 * KB * kWyTile;          // KB tiles: k rows, then q rows
  static constexpr int kStage = 4 * KB * kWyTile;          // the float rows as copied in
  static constexpr int kRegion = 4 * KB * kWyTile + kWyRows * DK * 4;
  // after the MMAs (the operands and staging are dead): per-row values, node tables
  static constexpr int kA = 0;                             // v_t - gamma_t (S0 k_t), [node][row]
  static constexpr int kB = kWyMaxNodes * kWyRows * 4;     // S0 q_t
  static constexpr int kG = 3 * kWyMaxNodes * kWyRows * 4; // (gamma_t/gamma_j) k_j.k_t, [t][j]
  static constexpr int kHq = kG + kWyMaxNodes * kWyMaxNodes * 4;  // (gamma_t/gamma_j) k_j.q_t
  static constexpr int kTablesEnd = kHq + kWyMaxNodes * kWyMaxNodes * 4;
  static constexpr int kMisc = kRegion > kTablesEnd ? kRegion : kTablesEnd;
  // misc: each node's path as a bit mask over the nodes (t and its ancestors below the
  // root), gamma, beta, alpha, parents, two barriers, the tensor-memory address, a flag
  static constexpr int kPath = kMisc;
  static constexpr int kGam = kPath + kWyMaxNodes * 8;
  static constexpr int kBet = kGam + kWyMaxNodes * 4;
  static constexpr int kAlp = kBet + kWyMaxNodes * 4;
  static constexpr int kPar = kAlp + kWyMaxNodes * 4;
  static constexpr int kBar = kPar + kWyMaxNodes * 4;      // staging barrier, MMA barrier
  static constexpr int kTmem = kBar + 16;
  static constexpr int kFlag = kTmem + 4;
  static constexpr int kVs = kFlag + 12;                   // v of the CTA's rows, bf16 [node][row]
  static constexpr int kBytes = kVs + kWyMaxNodes * kWyRows * 2;
  static_assert(kA + 3 * kWyMaxNodes * kWyRows * 4 <= kG, "per-row values overlap the tables");
  static_assert(kBytes <= 227 * 1024, "shared memory plan too large");
};

__device__ __forceinline__ uint32_t pack_bf16(uint16_t lo, uint16_t hi) { return (uint32_t)lo | ((uint32_t)hi << 16); }

template <int DK>
__global__ void __launch_bounds__(kWyThreads, 1) k_gdn_wy_verify_tc(
    const float* __restrict__ S0, const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
    const uint16_t* __restrict__ v, const float* __restrict__ alpha, const float* __restrict__ beta,
    const int32_t* __restrict__ parent, int n, int64_t H, int64_t dv, float* __restrict__ O,
    int32_t* __restrict__ status) {
  using P = WyPlan<DK>;
  constexpr int KB = P::KB;
  extern __shared__ __align__(1024) uint8_t wsm_tc[];
  uint8_t* sm = wsm_tc;
  const uint32_t sbase = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t h = blockIdx.x, r0 = (int64_t)blockIdx.y * kWyRows;
  const int rows = (int)(dv - r0 < kWyRows ? dv - r0 : kWyRows);
  const int n16 = (n + 15) & ~15;
  unsigned long long* pmask = reinterpret_cast<unsigned long long*>(sm + P::kPath);
  float* gam = reinterpret_cast<float*>(sm + P::kGam);
  float* bet = reinterpret_cast<float*>(sm + P::kBet);
  float* alp = reinterpret_cast<float*>(sm + P::kAlp);
  int32_t* par = reinterpret_cast<int32_t*>(sm + P::kPar);
  const uint32_t bar_stage = sbase + P::kBar, bar_mma = bar_stage + 8;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + P::kTmem);
  int32_t* flag = reinterpret_cast<int32_t*>(sm + P::kFlag);

  // ---- inputs: the head's state rows by one bulk copy, node scalars, node vectors.  The
  // next kernel on the stream may start now (programmatic dependent launch); this one reads
  // the state before it waits for the previous kernel, everything else after.
  if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    *flag = 0;
    mbar_init(bar_stage, 1);
    mbar_init(bar_mma, 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (tid == 0) {
    const uint32_t bytes = (uint32_t)rows * DK * 4;
    const uint64_t pol = policy_evict_first();
    mbar_arrive_expect_tx(bar_stage, bytes);
    const uint8_t* src = reinterpret_cast<const uint8_t*>(S0 + (h * dv + r0) * DK);
    for (uint32_t off = 0; off < bytes; off += 16384u)
      bulk_g2s(sbase + P::kStage + off, src + off, bytes - off < 16384u ? bytes - off : 16384u, bar_stage, pol);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the node inputs may be the previous kernel's
  // Warps 0-3 stage v of their state rows for every node; warps 4-5 read the tree and build
  // each node's path mask and gamma; warps 6-15 zero the rows past dv and fill the node
  // tiles.  The state rows land meanwhile.
  uint16_t* vs = reinterpret_cast<uint16_t*>(sm + P::kVs);
  if (warp < 4) {
    const int R = tid;
#pragma unroll 8
    for (int t = 0; t < n; ++t) vs[t * kWyRows + R] = R < rows ? v[((int64_t)t * H + h) * dv + r0 + R] : (uint16_t)0;
  } else if (warp < 6) {
    // ---- the tree: parents checked, each node's path as a mask, gamma (root side first:
    // a parent's index is below its child's, so rising bit order walks the path from the root)
    const int t = tid - 128;
    if (t < n) {
      par[t] = parent[t];
      alp[t] = alpha[(int64_t)t * H + h];
      bet[t] = beta[(int64_t)t * H + h];
    }
    asm volatile("bar.sync 1, 64;" ::: "memory");  // warps 4 and 5
    if (t < n) {
      bool ok = t == 0 ? par[0] == -1 : (par[t] >= 0 && par[t] < t);
      unsigned long long m = 0ull;
      if (ok)
        for (int j = t; j > 0; j = par[j]) {
          if (par[j] < 0 || par[j] >= j) {  // an ancestor's bad parent (also flagged by that node)
            ok = false;
            break;
          }
          m |= 1ull << j;
        }
      if (!ok) atomicOr(flag, 1);
      pmask[t] = m;
      float g = 1.f;
      for (unsigned long long r = m; r; r &= r - 1) g = alp[__ffsll((long long)r) - 1] * g;
      gam[t] = g;
    }
  } else {
    const int w6 = tid - 192, nw6 = kWyThreads - 192;
    // rows past dv read as zero (their lanes are never stored)
    for (int e = rows * DK + w6; e < kWyRows * DK; e += nw6) reinterpret_cast<float*>(sm + P::kStage)[e] = 0.f;
    // node tiles: rows 0..n16-1 hold k_t, rows n16..2*n16-1 q_t, the rest zero
    for (int u = w6; u < KB * kWyRows * 8; u += nw6) {
      const int kb = u / (kWyRows * 8), R = (u / 8) % kWyRows, c8 = u & 7;
      const uint16_t* src = nullptr;
      if (R < n16) {
        if (R < n) src = k + ((int64_t)R * H + h) * DK;
      } else if (R < 2 * n16 && R - n16 < n) {
        src = q + ((int64_t)(R - n16) * H + h) * DK;
      }
      uint32_t w[4] = {0u, 0u, 0u, 0u};
      if (src) {
        src += kb * 64 + c8 * 8;
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = pack_bf16(src[2 * i], src[2 * i + 1]);
      }
      sts128(sbase + P::kNodes + kb * kWyTile + R * 128 + ((c8 ^ (R & 7)) << 4), w[0], w[1], w[2], w[3]);
    }
  }
  const bool landed = mbar_wait_bounded(bar_stage, 0u);
  if (!landed) atomicOr(flag, 4);
  __syncthreads();
  if (*flag) {
    if (tid == 0) {
      if (blockIdx.y == 0 && (*flag & 1)) atomicOr(status, 1);
      if (*flag & 4) atomicOr(status, 4);
    }
    return;  // no tensor memory held yet; a copy that did not land in a second is abandoned
  }
  // ---- the three pieces of every state element, in the A operand's swizzled layout
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(smem_u32(tslot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  {
    const float* st = reinterpret_cast<const float*>(sm + P::kStage);
    for (int u = tid; u < KB * kWyRows * 8; u += kWyThreads) {
      const int R = u / (KB * 8), kb = (u / 8) % KB, c8 = u & 7;
      const float4 f0 = *reinterpret_cast<const float4*>(st + R * DK + kb * 64 + c8 * 8);
      const float4 f1 = *reinterpret_cast<const float4*>(st + R * DK + kb * 64 + c8 * 8 + 4);
      const float f[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
      uint16_t p1[8], p2[8], p3[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        p1[i] = bf16_rne(f[i]);
        const float e1 = __fsub_rn(f[i], bf16v(p1[i]));
        p2[i] = bf16_rne(e1);
        p3[i] = bf16_rne(__fsub_rn(e1, bf16v(p2[i])));
      }
      const uint32_t off = R * 128 + ((c8 ^ (R & 7)) << 4);
      const uint32_t a0 = sbase + P::kPieces + kb * kWyTile + off;
      sts128(a0, pack_bf16(p1[0], p1[1]), pack_bf16(p1[2], p1[3]), pack_bf16(p1[4], p1[5]), pack_bf16(p1[6], p1[7]));
      sts128(a0 + KB * kWyTile, pack_bf16(p2[0], p2[1]), pack_bf16(p2[2], p2[3]), pack_bf16(p2[4], p2[5]),
             pack_bf16(p2[6], p2[7]));
      sts128(a0 + 2 * KB * kWyTile, pack_bf16(p3[0], p3[1]), pack_bf16(p3[2], p3[3]), pack_bf16(p3[4], p3[5]),
             pack_bf16(p3[6], p3[7]));
    }
  }
  fence_proxy_async_smem();  // the generic-proxy operand stores -> the tensor core's reads
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  // ---- D1[row][c] = pieces . [k | q]^T (columns 0..2*n16), D2[i][j] = [k | q]_i . k_j
  if (tid == 0) {
    const uint32_t id1 = umma_idesc_n((uint32_t)(2 * n16)), id2 = umma_idesc_n((uint32_t)n16);
    for (int p = 0; p < 3; ++p)
      for (int kb = 0; kb < KB; ++kb) {
        const uint64_t ad = umma_desc(sbase + P::kPieces + (p * KB + kb) * kWyTile);
        const uint64_t bd = umma_desc(sbase + P::kNodes + kb * kWyTile);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) umma_bf16(tmem, ad + 2 * ks, bd + 2 * ks, id1, (p | kb | ks) ? 1u : 0u);
      }
    for (int kb = 0; kb < KB; ++kb) {
      const uint64_t nd = umma_desc(sbase + P::kNodes + kb * kWyTile);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) umma_bf16(tmem + 128, nd + 2 * ks, nd + 2 * ks, id2, (kb | ks) ? 1u : 0u);
    }
    umma_commit(bar_mma);
  }
  const int Rw = (warp & 3) * 32 + lane;
  const bool done = mbar_wait_bounded(bar_mma, 0u);
  tc_fence_after();
  if (!done) atomicOr(flag, 4);
  // ---- read back: warps 0-3 the state products (lane = state row), warps 4-7 the node
  // tables, kept only on each node's path (zero elsewhere, so the solve below runs dense)
  float* A_s = reinterpret_cast<float*>(sm + P::kA);
  float* B_s = reinterpret_cast<float*>(sm + P::kB);
  float* G = reinterpret_cast<float*>(sm + P::kG);
  float* Hq = reinterpret_cast<float*>(sm + P::kHq);
  if (done && warp < 4) {
    const uint32_t lanes = (uint32_t)(warp * 32) << 16;
#pragma unroll
    for (int c0 = 0; c0 < kWyMaxNodes; c0 += 16) {
      if (c0 < n16) {
        float val[16];
        tmem_ld16(tmem + lanes + (uint32_t)c0, val);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int c = c0 + i;
          if (c < n) A_s[c * kWyRows + Rw] = bf16v(vs[c * kWyRows + Rw]) - gam[c] * val[i];
        }
      }
    }
    for (int c0 = 0; c0 < n16; c0 += 16) {
      float val[16];
      tmem_ld16(tmem + lanes + (uint32_t)(n16 + c0), val);
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (c0 + i < n) B_s[(c0 + i) * kWyRows + Rw] = val[i];
    }
  } else if (done && warp < 8) {
    const int i = (warp - 4) * 32 + lane;  // D2 lane: k row i (i < n16) or q row i - n16
    const bool isk = i < n16;
    const int t = isk ? i : i - n16;
    const bool use = t < n && i < 2 * n16;
    const unsigned long long m = use ? pmask[t] : 0ull;
    for (int c0 = 0; c0 < n16; c0 += 16) {
      float val[16];
      tmem_ld16(tmem + 128 + ((uint32_t)((warp - 4) * 32) << 16) + (uint32_t)c0, val);
#pragma unroll
      for (int x = 0; x < 16; ++x) {
        const int j = c0 + x;
        // k rows: the ancestors of t below the root; q rows: t and those ancestors
        const bool on = ((m >> j) & 1ull) && (!isk || j != t);
        if (use && j < n) (isk ? G : Hq)[t * kWyMaxNodes + j] = on ? (gam[t] / gam[j]) * val[x] : 0.f;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(tmem) : "memory");
  if (!done) {
    if (tid == 0) atomicOr(status, 4);
    return;
  }
  // ---- pseudo-values and outputs, node order, one thread per state row, the pseudo-values
  // in registers.  The tables are zero off each node's path, so the sums run over every
  // earlier node without indirection; each node's output follows its pseudo-value and fills
  // the latency of the next one's chain.
  if (tid < kWyRows) {
    const int R = tid;
    const bool live = R < rows;
    float d[kWyMaxNodes];
    d[0] = 0.f;  // the root has no update here
    if (live) O[(int64_t)h * dv + r0 + R] = gam[0] * B_s[R];
#pragma unroll
    for (int t = 1; t < kWyMaxNodes; ++t) {
      if (t >= n) break;
      const float* Gt = G + t * kWyMaxNodes;
      float s0 = A_s[t * kWyRows + R], s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
      for (int j = 1; j < t; ++j) {
        float& acc = (j & 3) == 0 ? s0 : (j & 3) == 1 ? s1 : (j & 3) == 2 ? s2 : s3;
        acc = fmaf(-Gt[j], d[j], acc);
      }
      d[t] = bet[t] * ((s0 + s1) + (s2 + s3));
      const float* Ht = Hq + t * kWyMaxNodes;
      float o0 = gam[t] * B_s[t * kWyRows + R], o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll
      for (int j = 1; j <= t; ++j) {
        float& acc = (j & 3) == 0 ? o0 : (j & 3) == 1 ? o1 : (j & 3) == 2 ? o2 : o3;
        acc = fmaf(Ht[j], d[j], acc);
      }
      if (live) O[((int64_t)t * H + h) * dv + r0 + R] = (o0 + o1) + (o2 + o3);
    }
  }
}

template <int DK>
size_t wy_tc_smem() {
  return (size_t)WyPlan<DK>::kBytes;
}

// four threads per state row and a thread per element of k, whole warps
int gdn_threads(int64_t dk, int64_t dv) {
  const int64_t t = 4 * dv > dk ? 4 * dv : dk;
  return (int)((t + 31) / 32 * 32);
}

// a state row per four threads (rows past dv are read and unused), then k and v
size_t gdn_smem(int64_t dk, int64_t dv) { return (size_t)((gdn_threads(dk, dv) / 4) * (dk + 4) + dk + dv) * 4; }

// The state and the step vectors in dynamic shared memory, beside 16 KB of path list.
constexpr size_t kGdnMaxSmem = 200 * 1024;

int check_gdn_dims(int64_t H, int64_t dk, int64_t dv, const char* fn) {
  if (H < 1 || H > 65535 || dk < 1 || dv < 1 || dk > kGdnMaxDim || dv > kGdnMaxDim)
    return fail(W12_ERR_SHAPE, "%s: H=%lld dk=%lld dv=%lld out of range (dk, dv in 1..%lld)", fn, (long long)H,
                (long long)dk, (long long)dv, (long long)kGdnMaxDim);
  if (gdn_smem(dk, dv) > kGdnMaxSmem)
    return fail(W12_ERR_SHAPE, "%s: a %lld x %lld state does not fit in shared memory", fn, (long long)dv,
                (long long)dk);
  return W12_OK;
}

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current device, once per
// (kernel, device) unless a larger size is asked for later.
int set_gdn_smem(const void* kernel, size_t bytes) {
  struct Entry {
    const void* k;
    int dev;
    size_t bytes;
  };
  static std::mutex mu;
  static Entry done[32];
  static int n_done = 0;
  int dev = 0;
  W12_CUDA_TRY(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lk(mu);
  for (int i = 0; i < n_done; ++i)
    if (done[i].k == kernel && done[i].dev == dev && done[i].bytes >= bytes) return W12_OK;
  W12_CUDA_TRY(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes));
  for (int i = 0; i < n_done; ++i)
    if (done[i].k == kernel && done[i].dev == dev) {
      done[i].bytes = bytes;
      return W12_OK;
    }
  if (n_done < 32) done[n_done++] = Entry{kernel, dev, bytes};
  return W12_OK;
}

// Launch configuration with programmatic dependent launch: the kernel may start while the
// previous kernel on the stream drains (if that kernel signals early) and waits for it with
// griddepcontrol.wait before reading that kernel's outputs.
cudaLaunchConfig_t pdl_config(dim3 grid, int threads, void* stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3((unsigned)threads);
  cfg.stream = (cudaStream_t)stream;
  return cfg;
}

void pdl_attr(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr) {
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
}

}  // namespace
}  // namespace w12

using namespace w12;

extern "C" {

int gdn_split3(const float* x, int64_t n, uint16_t* s1, uint16_t* s2, uint16_t* s3, void* stream) {
  const char* fn = "gdn_split3";
  if (n < 0) return fail(W12_ERR_SHAPE, "%s: n=%lld", fn, (long long)n);
  if (n == 0) return W12_OK;
  if (!x || !s1 || !s2 || !s3) return fail(W12_ERR_INVALID_ARG, "%s: null pointer", fn);
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, 4096);
  k_split3<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(x, n, s1, s2, s3);
  W12_LAUNCH_CHECK(fn);
  return W12_OK;
}

int gdn_path_verify(const float* S0, const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* alpha,
                    const float* beta, const int32_t* parent, int64_t n, int64_t H, int64_t dk, int64_t dv, float* O,
                    int32_t* status, void* stream) {
  const char* fn = "gdn_path_verify";
  int st = check_gdn_dims(H, dk, dv, fn);
  if (st) return st;
  if (n < 1 || n > kGdnMaxNodes)
    return fail(W12_ERR_SHAPE, "%s: n=%lld out of range (1..%lld)", fn, (long long)n, (long long)kGdnMaxNodes);
  if (!S0 || !q || !k || !v || !alpha || !beta || !parent || !O || !status)
    return fail(W12_ERR_INVALID_ARG, "%s: null pointer", fn);
  const bool aligned = (((uintptr_t)S0) & 15u) == 0;
  if (aligned && (dk == 128 || dk == 64)) {  // state in registers, 32 rows a block
    cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)n, (unsigned)H, (unsigned)((dv + kRegRows - 1) / kRegRows)),
                                         kRegThreads, stream);
    cudaLaunchAttribute attr[1];
    pdl_attr(cfg, attr);
    if (dk == 128)
      W12_CUDA_TRY(cudaLaunchKernelEx(&cfg, k_gdn_path_verify_reg<128>, S0, q, k, v, alpha, beta, parent, n, H, dv, O,
                                      status));
    else
      W12_CUDA_TRY(cudaLaunchKernelEx(&cfg, k_gdn_path_verify_reg<64>, S0, q, k, v, alpha, beta, parent, n, H, dv, O,
                                      status));
    W12_LAUNCH_CHECK(fn);
    return W12_OK;
  }
  const size_t smem = gdn_smem(dk, dv);
  if ((st = set_gdn_smem((const void*)k_gdn_path_verify, smem))) return st;
  k_gdn_path_verify<<<dim3((unsigned)n, (unsigned)H), gdn_threads(dk, dv), smem, (cudaStream_t)stream>>>(
      S0, q, k, v, alpha, beta, parent, n, H, dk, dv, O, status);
  W12_LAUNCH_CHECK(fn);
  return W12_OK;
}

int gdn_wy_verify(const float* S0, const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* alpha,
                  const float* beta, const int32_t* parent, int64_t n, int64_t H, int64_t dk, int64_t dv, float* O,
                  int32_t* status, void* stream) {
  const char* fn = "gdn_wy_verify";
  int st = check_gdn_dims(H, dk, dv, fn);
  if (st) return st;
  if (dk != 64 && dk != 128) return fail(W12_ERR_SHAPE, "%s: dk=%lld (64 or 128)", fn, (long long)dk);
  if (n < 1 || n > kWyMaxNodes)
    return fail(W12_ERR_SHAPE, "%s: n=%lld out of range (1..%d)", fn, (long long)n, kWyMaxNodes);
  if (dv > 65535 * (int64_t)kWyRows) return fail(W12_ERR_SHAPE, "%s: dv=%lld", fn, (long long)dv);
  if (!S0 || !q || !k || !v || !alpha || !beta || !parent || !O || !status)
    return fail(W12_ERR_INVALID_ARG, "%s: null pointer", fn);
  if ((((uintptr_t)S0) & 15u) != 0) return fail(W12_ERR_INVALID_ARG, "%s: S0 must be 16-byte aligned", fn);
  cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)H, (unsigned)((dv + kWyRows - 1) / kWyRows)), kWyThreads, stream);
  cudaLaunchAttribute attr[1];
  pdl_attr(cfg, attr);
  if (dk == 128) {
    if ((st = set_gdn_smem((const void*)k_gdn_wy_verify_tc<128>, wy_tc_smem<128>()))) return st;
    cfg.dynamicSmemBytes = wy_tc_smem<128>();
    W12_CUDA_TRY(cudaLaunchKernelEx(&cfg, k_gdn_wy_verify_tc<128>, S0, q, k, v, alpha, beta, parent, (int)n, H, dv, O,
                                    status));
  } else {
    if ((st = set_gdn_smem((const void*)k_gdn_wy_verify_tc<64>, wy_tc_smem<64>()))) return st;
    cfg.dynamicSmemBytes = wy_tc_smem<64>();
    W12_CUDA_TRY(cudaLaunchKernelEx(&cfg, k_gdn_wy_verify_tc<64>, S0, q, k, v, alpha, beta, parent, (int)n, H, dv, O,
                                    status));
  }
  W12_LAUNCH_CHECK(fn);
  return W12_OK;
}

int gdn_commit(float* S, const uint16_t* k, const uint16_t* v, const float* alpha, const float* beta,
               const int32_t* path_len, const int32_t* path_nodes, int64_t n, int64_t H, int64_t dk, int64_t dv,
               int32_t* status, void* stream) {
  const char* fn = "gdn_commit";
  int st = check_gdn_dims(H, dk, dv, fn);
  if (st) return st;
  if (n < 1) return fail(W12_ERR_SHAPE, "%s: n=%lld", fn, (long long)n);
  if (!S || !k || !v || !alpha || !beta || !path_len || !path_nodes || !status)
    return fail(W12_ERR_INVALID_ARG, "%s: null pointer", fn);
  if ((((uintptr_t)S) & 15u) == 0 && (dk == 128 || dk == 64)) {  // state in registers, 32 rows a block
    cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)H, (unsigned)((dv + kRegRows - 1) / kRegRows)), kRegThreads,
                                         stream);
    cudaLaunchAttribute attr[1];
    pdl_attr(cfg, attr);
    if (dk == 128)
      W12_CUDA_TRY(cudaLaunchKernelEx(&cfg, k_gdn_commit_reg<128>, S, k, v, alpha, beta, path_len, path_nodes, n, H, dv,
                                      status));
    else
      W12_CUDA_TRY(cudaLaunchKernelEx(&cfg, k_gdn_commit_reg<64>, S, k, v, alpha, beta, path_len, path_nodes, n, H, dv,
                                      status));
    W12_LAUNCH_CHECK(fn);
    return W12_OK;
  }
  const size_t smem = gdn_smem(dk, dv);
  if ((st = set_gdn_smem((const void*)k_gdn_commit, smem))) return st;
  k_gdn_commit<<<(unsigned)H, gdn_threads(dk, dv), smem, (cudaStream_t)stream>>>(S, k, v, alpha, beta, path_len,
                                                                              path_nodes, n, H, dk, dv, status);
  W12_LAUNCH_CHECK(fn);
  return W12_OK;
}

}  // extern "C"
