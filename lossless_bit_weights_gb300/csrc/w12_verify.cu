// w12_verify.cu - greedy draft-tree acceptance, row argmax and the two-level
// verification splice.
//
// The SpecPilot summary page (onedev.kr/papers/1654), section "What's
// different", verifies a draft tree by taking the path whose tokens match the
// target and a bonus token (the two-level verification paragraph; the batched
// case gives every request its own tree).  Node i is accepted when its parent
// is accepted and its drafted token equals the target's greedy token at the
// parent; the deepest accepted node wins, the lowest index among equals.
#include <cstdint>

#include "w12_internal.cuh"

namespace w12 {

int lmhead_argmax_impl(const uint16_t* x, int64_t M, const w12_matrix* head, int32_t* tok, bool q8, void* ws,
                       size_t ws_bytes, cudaStream_t s, const char* fn);

namespace {

// One thread per request.  path_nodes[off .. off+m) doubles as the depth
// scratch (-1 = not accepted) before it receives the path.
__device__ void accept_one(const int32_t* __restrict__ tok, const int32_t* __restrict__ parent,
                           const int32_t* __restrict__ draft, int64_t off, int64_t m, int64_t M, int32_t* path_len,
                           int32_t* __restrict__ path_nodes, int32_t* bonus, int r) {
  if (off < 0 || m < 1 || off + m > M || parent[off] != -1) {
    path_len[r] = -1;
    bonus[r] = -1;
    return;
  }
  int32_t* depth = path_nodes + off;
  depth[0] = 0;
  int64_t best = 0;
  int32_t best_d = 0;
  for (int64_t i = 1; i < m; ++i) {
    const int32_t p = parent[off + i];
    if (p < 0 || p >= i) {
      path_len[r] = -1;
      bonus[r] = -1;
      return;
    }
    const int32_t dp = depth[p];
    const int32_t d = (dp >= 0 && draft[off + i] == tok[off + p]) ? dp + 1 : -1;
    depth[i] = d;
    if (d > best_d) {
      best_d = d;
      best = i;
    }
  }
  int64_t v = best;
  for (int32_t j = best_d; j >= 0; --j) {
    path_nodes[off + j] = (int32_t)v;
    v = parent[off + v];
  }
  path_len[r] = best_d;
  bonus[r] = tok[off + best];
}

__global__ void k_accept(const int32_t* __restrict__ tok, const int32_t* __restrict__ parent,
                         const int32_t* __restrict__ draft, const int32_t* __restrict__ offsets, int32_t n_req, int64_t M,
                         int32_t* path_len, int32_t* path_nodes, int32_t* bonus) {
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < n_req; r += gridDim.x * blockDim.x) {
    const int64_t off = offsets ? offsets[r] : 0;
    const int64_t end = offsets ? offsets[r + 1] : M;
    accept_one(tok, parent, draft, off, end - off, M, path_len, path_nodes, bonus, r);
  }
}

// Row argmax of fp32 logits, one block per row (ties -> lowest index, NaN lowest).
__global__ void __launch_bounds__(256) k_row_argmax(const float* __restrict__ logits, int64_t V, int32_t* tok) {
  __shared__ unsigned long long red[8];
  const int64_t m = blockIdx.x;
  const float* row = logits + m * V;
  unsigned long long best = 0ull;
  for (int64_t v = threadIdx.x; v < V; v += 256) {
    const uint32_t key = (uint32_t)order_key(row[v]) ^ 0x80000000u;
    const unsigned long long c = ((unsigned long long)key << 32) | (0xFFFFFFFFu - (uint32_t)v);
    best = c > best ? c : best;
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
    tok[m] = (int32_t)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull));
  }
}

int check_tree_args(const void* tok, const int32_t* parent, const int32_t* draft, int32_t n_req, int64_t M,
                    const int32_t* path_len, const int32_t* path_nodes, const int32_t* bonus, const int32_t* offsets,
                    const char* fn) {
  if (!tok || !parent || !draft || !path_len || !path_nodes || !bonus)
    return fail(W12_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (M < 1 || M > 0x7FFFFFFF) return fail(W12_ERR_SHAPE, "%s: M=%lld out of range", fn, (long long)M);
  if (n_req < 1) return fail(W12_ERR_SHAPE, "%s: n_req=%d must be >= 1", fn, n_req);
  if (!offsets && n_req != 1) return fail(W12_ERR_INVALID_ARG, "%s: req_offsets is null but n_req=%d", fn, n_req);
  return W12_OK;
}

int launch_accept(const int32_t* tok, const int32_t* parent, const int32_t* draft, const int32_t* offsets,
                  int32_t n_req, int64_t M, int32_t* path_len, int32_t* path_nodes, int32_t* bonus, cudaStream_t s) {
  const int threads = 128;
  const int blocks = (n_req + threads - 1) / threads;
  k_accept<<<blocks < 1024 ? blocks : 1024, threads, 0, s>>>(tok, parent, draft, offsets, n_req, M, path_len,
                                                            path_nodes, bonus);
  W12_LAUNCH_CHECK("tree acceptance kernel");
  return W12_OK;
}

// Two-level verification splice, one block per node of the n-node output tree.  Every
// block checks the inputs (O(n)), then fills its node: path nodes 0..L keep the Q pass's
// path in order and reuse its rows, node L+1 is the bonus node, subtree node j is node
// L+2+j.  An invalid Q result, a path with no room for the bonus node, a path node outside
// the Q tree or a subtree parent that is not an earlier subtree node gives parent -2 on
// every node (acceptance then reports the tree invalid) and zero rows.
__global__ void __launch_bounds__(256) k_tlv_splice(const int32_t* __restrict__ path_len,
                                                    const int32_t* __restrict__ path_nodes,
                                                    const int32_t* __restrict__ bonus,
                                                    const int32_t* __restrict__ draft_q,
                                                    const uint16_t* __restrict__ x_q, int64_t n_q,
                                                    const int32_t* __restrict__ sub_parent,
                                                    const int32_t* __restrict__ sub_draft,
                                                    const uint16_t* __restrict__ x_sub, int64_t n, int64_t K,
                                                    int32_t* parent_out, int32_t* draft_out, int32_t* src_out,
                                                    uint16_t* __restrict__ x_out) {
  __shared__ int32_t s_src;
  const int64_t i = blockIdx.x;
  const int32_t L = *path_len;
  bool ok = L >= 0 && (int64_t)L + 2 <= n;
  if (ok) {  // the checks are spread over the block
    for (int64_t k = threadIdx.x; k <= L; k += blockDim.x) ok = ok && path_nodes[k] >= 0 && path_nodes[k] < n_q;
    for (int64_t j = threadIdx.x; j < n - L - 2; j += blockDim.x) ok = ok && sub_parent[j] < j;
  }
  ok = __syncthreads_and(ok) != 0;
  if (threadIdx.x == 0) {
    int32_t par = -2, dr = -1, src = -1 - (int32_t)n;  // invalid: no row
    if (ok) {
      if (i <= L) {
        par = (int32_t)i - 1;
        dr = draft_q[path_nodes[i]];
        src = path_nodes[i];
      } else if (i == L + 1) {
        par = L;
        dr = *bonus;
        src = -1;
      } else {
        const int64_t j = i - L - 2;
        par = sub_parent[j] < 0 ? L + 1 : L + 2 + sub_parent[j];
        dr = sub_draft[j];
        src = -1 - (int32_t)(j + 1);
      }
    }
    parent_out[i] = par;
    draft_out[i] = dr;
    src_out[i] = src;
    s_src = src;
  }
  __syncthreads();
  const int32_t src = s_src;
  const uint16_t* row = src >= 0 ? x_q + (int64_t)src * K : (-1 - src < n ? x_sub + (int64_t)(-1 - src) * K : nullptr);
  uint16_t* out = x_out + i * K;
  const bool vec = (K % 8) == 0 && (((uintptr_t)x_q | (uintptr_t)x_sub | (uintptr_t)x_out) & 15u) == 0;
  if (vec) {
    for (int64_t k = threadIdx.x; k < K / 8; k += blockDim.x)
      reinterpret_cast<uint4*>(out)[k] = row ? reinterpret_cast<const uint4*>(row)[k] : make_uint4(0, 0, 0, 0);
  } else {
    for (int64_t k = threadIdx.x; k < K; k += blockDim.x) out[k] = row ? row[k] : (uint16_t)0;
  }
}

}  // namespace
}  // namespace w12

using namespace w12;

extern "C" {

int tree_verify_tokens(const int32_t* tok, const int32_t* parent, const int32_t* draft, const int32_t* req_offsets,
                       int32_t n_req, int64_t M, int32_t* path_len, int32_t* path_nodes, int32_t* bonus, void* stream) {
  int st = check_tree_args(tok, parent, draft, n_req, M, path_len, path_nodes, bonus, req_offsets, "tree_verify_tokens");
  if (st) return st;
  return launch_accept(tok, parent, draft, req_offsets, n_req, M, path_len, path_nodes, bonus, (cudaStream_t)stream);
}

size_t tree_verify_workspace_size(int64_t M) { return M >= 1 ? (size_t)((M * 4 + 255) & ~(int64_t)255) : 0; }

int tree_verify(const float* logits, int64_t M, int64_t V, const int32_t* parent, const int32_t* draft,
                const int32_t* req_offsets, int32_t n_req, int32_t* path_len, int32_t* path_nodes, int32_t* bonus,
                void* ws, size_t ws_bytes, void* stream) {
  int st = check_tree_args(logits, parent, draft, n_req, M, path_len, path_nodes, bonus, req_offsets, "tree_verify");
  if (st) return st;
  if (V < 1 || V > 0x7FFFFFFF) return fail(W12_ERR_SHAPE, "tree_verify: V=%lld out of range", (long long)V);
  if (!ws) return fail(W12_ERR_INVALID_ARG, "tree_verify: null workspace");
  if (ws_bytes < tree_verify_workspace_size(M))
    return fail(W12_ERR_BUFFER_TOO_SMALL, "tree_verify: workspace %zu < %zu", ws_bytes, tree_verify_workspace_size(M));
  cudaStream_t s = (cudaStream_t)stream;
  int32_t* tok = static_cast<int32_t*>(ws);
  k_row_argmax<<<(unsigned)M, 256, 0, s>>>(logits, V, tok);
  W12_LAUNCH_CHECK("tree_verify: row argmax");
  return launch_accept(tok, parent, draft, req_offsets, n_req, M, path_len, path_nodes, bonus, s);
}

int w12_lmhead_verify(const uint16_t* x, int64_t M, const w12_matrix* head, int q8, const int32_t* parent,
                      const int32_t* draft, const int32_t* req_offsets, int32_t n_req, int32_t* tok, int32_t* path_len,
                      int32_t* path_nodes, int32_t* bonus, void* ws, size_t ws_bytes, void* stream) {
  int st = check_tree_args(tok, parent, draft, n_req, M, path_len, path_nodes, bonus, req_offsets, "w12_lmhead_verify");
  if (st) return st;
  cudaStream_t s = (cudaStream_t)stream;
  st = lmhead_argmax_impl(x, M, head, tok, q8 != 0, ws, ws_bytes, s, "w12_lmhead_verify");
  if (st) return st;
  return launch_accept(tok, parent, draft, req_offsets, n_req, M, path_len, path_nodes, bonus, s);
}

int tlv_splice(const int32_t* path_len, const int32_t* path_nodes, const int32_t* bonus, const int32_t* draft_q,
               const uint16_t* x_q, int64_t n_q, const int32_t* sub_parent, const int32_t* sub_draft,
               const uint16_t* x_sub, int64_t n, int64_t K, int32_t* parent_out, int32_t* draft_out, int32_t* src_out,
               uint16_t* x_out, void* stream) {
  if (!path_len || !path_nodes || !bonus || !draft_q || !x_q || !x_sub || !parent_out || !draft_out || !src_out ||
      !x_out || (n > 2 && (!sub_parent || !sub_draft)))
    return fail(W12_ERR_INVALID_ARG, "tlv_splice: null pointer");
  if (n < 2 || n > (1 << 20) || n_q < 1 || n_q > 0x7FFFFFFF || K < 1 || K > kMaxK)
    return fail(W12_ERR_SHAPE, "tlv_splice: n=%lld (2..2^20), n_q=%lld, K=%lld out of range", (long long)n,
                (long long)n_q, (long long)K);
  k_tlv_splice<<<(unsigned)n, 256, 0, (cudaStream_t)stream>>>(path_len, path_nodes, bonus, draft_q, x_q, n_q, sub_parent,
                                                              sub_draft, x_sub, n, K, parent_out, draft_out, src_out,
                                                              x_out);
  W12_LAUNCH_CHECK("tlv_splice kernel");
  return W12_OK;
}

}  // extern "C"
