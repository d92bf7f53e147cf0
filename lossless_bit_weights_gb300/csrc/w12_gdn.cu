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
  RegState<DK> S;
  reg_load<DK>(S, S0 + (h * dv + r0) * DK, dv - r0);
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

// ---- WY form: every node of the tree at once.  With gamma_t the product of alpha along
// t's path, node t's state is S_t = gamma_t S0 + sum_{j on path(t)} (gamma_t/gamma_j) d_j k_j^T,
// whose pseudo-values d_j solve, in node order (ancestors come first),
//     d_t = beta_t (v_t - gamma_t S0 k_t - sum_{j ancestor of t} (gamma_t/gamma_j) (k_j.k_t) d_j),
// and o_t = gamma_t S0 q_t + sum_{j on path(t)} (gamma_t/gamma_j) (k_j.q_t) d_j.  The state
// enters only through S0 k_t and S0 q_t (all nodes in one pass over the state, rows in
// registers); the rest is node-by-node scalars and a substitution per state row.  Rows are
// independent, so a block takes (head, 32 rows).
constexpr int kWyMaxNodes = 64;

template <int DK>
struct WyLayout {  // dynamic shared memory, in floats
  static constexpr int P = 4 * (RegState<DK>::Q + 4);  // one padded vector
  int n;
  __device__ int kpad() const { return 0; }
  __device__ int qpad() const { return n * P; }
  __device__ int a() const { return 2 * n * P; }                       // S0 k_t, [n][32]
  __device__ int b() const { return 2 * n * P + n * kRegRows; }        // S0 q_t
  __device__ int d() const { return 2 * n * P + 2 * n * kRegRows; }    // pseudo-values
  __device__ int vv() const { return 2 * n * P + 3 * n * kRegRows; }   // v of the block's rows
  __device__ int kk() const { return 2 * n * P + 4 * n * kRegRows; }   // k_j.k_t, [n][n]
  __device__ int kq() const { return kk() + n * n; }                   // k_j.q_t
  __device__ int gam() const { return kq() + n * n; }
  __device__ int bet() const { return gam() + n; }
  __device__ int total() const { return bet() + n; }
};

size_t wy_smem(int64_t dk, int64_t n) {
  const int64_t P = 4 * (dk / 4 + 4);
  return (size_t)(2 * n * P + 4 * n * kRegRows + 2 * n * n + 2 * n) * 4 + (size_t)n * 4;
}

template <int DK>
__global__ void __launch_bounds__(kRegThreads) k_gdn_wy_verify(
    const float* __restrict__ S0, const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
    const uint16_t* __restrict__ v, const float* __restrict__ alpha, const float* __restrict__ beta,
    const int32_t* __restrict__ parent, int64_t n64, int64_t H, int64_t dv, float* __restrict__ O,
    int32_t* __restrict__ status) {
  extern __shared__ __align__(16) float wsm[];
  __shared__ int32_t ok_sh;
  const int n = (int)n64;
  const WyLayout<DK> Lw{n};
  int32_t* par = reinterpret_cast<int32_t*>(wsm + Lw.total());
  const int64_t h = blockIdx.x, r0 = (int64_t)blockIdx.y * kRegRows;
  const int tid = threadIdx.x, p = tid & 3;
  const int r = tid >> 2;
  for (int t = tid; t < n; t += blockDim.x) par[t] = parent[t];
  if (tid == 0) ok_sh = 1;
  __syncthreads();
  if (tid == 0) {
    bool ok = par[0] == -1;
    for (int t = 1; ok && t < n; ++t) ok = par[t] >= 0 && par[t] < t;
    if (!ok) {
      if (blockIdx.y == 0) atomicOr(status, 1);
      ok_sh = 0;
    } else {
      float* g = wsm + Lw.gam();
      g[0] = 1.f;  // the committed root: its update is already in S0
      for (int t = 1; t < n; ++t) g[t] = alpha[(int64_t)t * H + h] * g[par[t]];
    }
  }
  // node vectors (padded so the four quarters of k and q sit on distinct banks), v, beta
  for (int e = tid; e < n * DK; e += blockDim.x) {
    const int t = e / DK, c = e - t * DK;
    wsm[Lw.kpad() + t * WyLayout<DK>::P + vpos<DK>(c)] = bf16v(k[((int64_t)t * H + h) * DK + c]);
    wsm[Lw.qpad() + t * WyLayout<DK>::P + vpos<DK>(c)] = bf16v(q[((int64_t)t * H + h) * DK + c]);
  }
  for (int e = tid; e < n * kRegRows; e += blockDim.x) {
    const int t = e / kRegRows, rr = e - t * kRegRows;
    wsm[Lw.vv() + e] = r0 + rr < dv ? bf16v(v[((int64_t)t * H + h) * dv + r0 + rr]) : 0.f;
  }
  for (int t = tid; t < n; t += blockDim.x) wsm[Lw.bet() + t] = beta[(int64_t)t * H + h];
  RegState<DK> S;
  reg_load<DK>(S, S0 + (h * dv + r0) * DK, dv - r0);
  __syncthreads();
  if (!ok_sh) return;
  // S0 k_t and S0 q_t of this block's rows, every node
  for (int t = 0; t < n; ++t) {
    const float at = reg_dot<DK>(S, wsm + Lw.kpad() + t * WyLayout<DK>::P);
    const float bt = reg_dot<DK>(S, wsm + Lw.qpad() + t * WyLayout<DK>::P);
    if (p == 0) {
      wsm[Lw.a() + t * kRegRows + r] = at;
      wsm[Lw.b() + t * kRegRows + r] = bt;
    }
  }
  // (gamma_t/gamma_j) k_j.k_t and (gamma_t/gamma_j) k_j.q_t for j <= t (the four quarters
  // of each padded vector, skipping the padding)
  {
    const float* gm = wsm + Lw.gam();
    constexpr int Q = RegState<DK>::Q;
    for (int e = tid; e < n * n; e += blockDim.x) {
      const int t = e / n, j = e - t * n;
      if (j > t) continue;
      const float* kj = wsm + Lw.kpad() + j * WyLayout<DK>::P;
      const float* kt = wsm + Lw.kpad() + t * WyLayout<DK>::P;
      const float* qt = wsm + Lw.qpad() + t * WyLayout<DK>::P;
      float g0 = 0.f, g1 = 0.f;
#pragma unroll
      for (int qq = 0; qq < 4; ++qq)
        for (int m = 0; m < Q; ++m) {
          const int c = qq * (Q + 4) + m;
          g0 = fmaf(kj[c], kt[c], g0);
          g1 = fmaf(kj[c], qt[c], g1);
        }
      const float ratio = gm[t] / gm[j];
      wsm[Lw.kk() + t * n + j] = ratio * g0;
      wsm[Lw.kq() + t * n + j] = ratio * g1;
    }
  }
  __syncthreads();
  // pseudo-values, node order, one thread per row
  const float* gam = wsm + Lw.gam();
  if (p == 0) {
    float* d = wsm + Lw.d();
    d[r] = 0.f;  // the root has no update here
    for (int t = 1; t < n; ++t) {
      float acc = wsm[Lw.vv() + t * kRegRows + r] - gam[t] * wsm[Lw.a() + t * kRegRows + r];
      for (int j = par[t]; j > 0; j = par[j]) acc = fmaf(-wsm[Lw.kk() + t * n + j], d[j * kRegRows + r], acc);
      d[t * kRegRows + r] = wsm[Lw.bet() + t] * acc;
    }
  }
  __syncthreads();
  // outputs: the four threads of a row split the nodes
  const int64_t row = r0 + r;
  for (int t = p; t < n; t += 4) {
    float o = gam[t] * wsm[Lw.b() + t * kRegRows + r];
    for (int j = t; j > 0; j = par[j]) o = fmaf(wsm[Lw.kq() + t * n + j], wsm[Lw.d() + j * kRegRows + r], o);
    if (row < dv) O[((int64_t)t * H + h) * dv + row] = o;
  }
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

int set_gdn_smem(const void* kernel, size_t bytes) {
  W12_CUDA_TRY(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes));
  return W12_OK;
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
    const dim3 grid((unsigned)n, (unsigned)H, (unsigned)((dv + kRegRows - 1) / kRegRows));
    const int threads = kRegThreads;
    if (dk == 128)
      k_gdn_path_verify_reg<128><<<grid, threads, 0, (cudaStream_t)stream>>>(S0, q, k, v, alpha, beta, parent, n, H,
                                                                             dv, O, status);
    else
      k_gdn_path_verify_reg<64><<<grid, threads, 0, (cudaStream_t)stream>>>(S0, q, k, v, alpha, beta, parent, n, H,
                                                                            dv, O, status);
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
  if (dv > 65535 * (int64_t)kRegRows) return fail(W12_ERR_SHAPE, "%s: dv=%lld", fn, (long long)dv);
  if (!S0 || !q || !k || !v || !alpha || !beta || !parent || !O || !status)
    return fail(W12_ERR_INVALID_ARG, "%s: null pointer", fn);
  if ((((uintptr_t)S0) & 15u) != 0) return fail(W12_ERR_INVALID_ARG, "%s: S0 must be 16-byte aligned", fn);
  const size_t smem = wy_smem(dk, n);
  const dim3 grid((unsigned)H, (unsigned)((dv + kRegRows - 1) / kRegRows));
  if (dk == 128) {
    if ((st = set_gdn_smem((const void*)k_gdn_wy_verify<128>, smem))) return st;
    k_gdn_wy_verify<128><<<grid, kRegThreads, smem, (cudaStream_t)stream>>>(S0, q, k, v, alpha, beta, parent, n, H,
                                                                           dv, O, status);
  } else {
    if ((st = set_gdn_smem((const void*)k_gdn_wy_verify<64>, smem))) return st;
    k_gdn_wy_verify<64><<<grid, kRegThreads, smem, (cudaStream_t)stream>>>(S0, q, k, v, alpha, beta, parent, n, H, dv,
                                                                          O, status);
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
    const dim3 grid((unsigned)H, (unsigned)((dv + kRegRows - 1) / kRegRows));
    if (dk == 128)
      k_gdn_commit_reg<128><<<grid, kRegThreads, 0, (cudaStream_t)stream>>>(S, k, v, alpha, beta, path_len, path_nodes,
                                                                           n, H, dv, status);
    else
      k_gdn_commit_reg<64><<<grid, kRegThreads, 0, (cudaStream_t)stream>>>(S, k, v, alpha, beta, path_len, path_nodes,
                                                                          n, H, dv, status);
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
