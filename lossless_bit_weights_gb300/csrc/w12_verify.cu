// w12_verify.cu - greedy draft-tree acceptance, row argmax, the two-level
// verification splice and the node budget shared across requests.
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

// ---- programmatic dependent launch: a kernel launched with launch_pdl may start while the
// previous kernel on the stream drains (when that kernel signals early); it calls pdl_wait()
// before it reads anything the previous kernel wrote.  pdl_signal() lets the next kernel
// start early.  Used only behind small kernels: a waiting block that shares an SM with a
// long kernel slows it (an LM head's final argmax launched this way cost the head 13 %).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_signal() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}


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
  if (threadIdx.x == 0) pdl_signal();
  pdl_wait();  // the tokens may be the previous kernel's
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
  W12_CUDA_TRY(launch_pdl(k_accept, dim3(blocks < 1024 ? blocks : 1024), dim3(threads), 0, s, tok, parent, draft,
                          offsets, n_req, M, path_len, path_nodes, bonus));
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
  if (threadIdx.x == 0) pdl_signal();
  pdl_wait();  // the acceptance results may be the previous kernel's
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

// Node budget over several candidate trees, one block.  Scores are the float products of
// the draft confidences from each root (root first, rounded multiplies), ranked by (score
// descending, depth ascending, index ascending); the first `budget` are kept over all
// requests, or within each request when per_request is set.  A child never outranks its
// parent, so the kept set is closed under ancestors.  Kept nodes are renumbered per
// request in their original order.  An invalid candidate tree sets *n_kept = -1.
constexpr int kBudgetMaxNodes = 4096;
constexpr int kBudgetThreads = 1024;

__global__ void __launch_bounds__(kBudgetThreads) k_budget_select(const int32_t* __restrict__ parent,
                                                                  const float* __restrict__ conf,
                                                                  const int32_t* __restrict__ draft,
                                                                  const int32_t* __restrict__ off, int32_t n_req,
                                                                  int32_t C, int32_t budget, int32_t per_request,
                                                                  int32_t* parent_out, int32_t* draft_out,
                                                                  int32_t* src_out, int32_t* off_out, int32_t* n_kept) {
  if (threadIdx.x == 0) pdl_signal();  // the row gather that follows starts early
  extern __shared__ uint8_t sm[];
  float* score = reinterpret_cast<float*>(sm);
  int32_t* depth = reinterpret_cast<int32_t*>(score + C);
  int32_t* req = depth + C;
  int32_t* idx = req + C;  // rank < budget ? new index : -1
  __shared__ int32_t s_bad;
  __shared__ int32_t s_cnt[kBudgetThreads];
  if (threadIdx.x == 0) s_bad = (off[0] != 0 || off[n_req] != C) ? 1 : 0;  // requests tile 0..C-1
  __syncthreads();
  if (s_bad) {
    if (threadIdx.x == 0) *n_kept = -1;
    return;
  }
  // scores and depths, one request per thread, nodes in order (parents come first)
  for (int32_t r = threadIdx.x; r < n_req; r += blockDim.x) {
    const int32_t a = off[r], e = off[r + 1];
    bool ok = e > a && a >= 0 && e <= C && parent[a] == -1;
    for (int32_t i = a; ok && i < e; ++i) {
      req[i] = r;
      if (i == a) {
        score[i] = conf[i];
        depth[i] = 0;
      } else {
        const int32_t p = parent[i];
        ok = p >= 0 && p < i - a;
        if (ok) {
          score[i] = __fmul_rn(score[a + p], conf[i]);
          depth[i] = depth[a + p] + 1;
        }
      }
    }
    if (!ok) s_bad = 1;
  }
  __syncthreads();
  if (s_bad) {
    if (threadIdx.x == 0) *n_kept = -1;
    return;
  }
  // rank = number of nodes before this one in the order (all, or the node's request's)
  for (int32_t i = threadIdx.x; i < C; i += blockDim.x) {
    const float si = score[i];
    const int32_t di = depth[i];
    int32_t j0 = 0, j1 = C;
    if (per_request) {
      j0 = off[req[i]];
      j1 = off[req[i] + 1];
    }
    int32_t rank = 0;
    for (int32_t j = j0; j < j1; ++j) {
      const float sj = score[j];
      rank += (sj > si || (sj == si && (depth[j] < di || (depth[j] == di && j < i)))) ? 1 : 0;
    }
    idx[i] = rank < budget ? 0 : -1;
  }
  __syncthreads();
  // per request: new indices in original order, then the request's place in the output
  for (int32_t r = threadIdx.x; r < n_req; r += blockDim.x) {
    int32_t n = 0;
    for (int32_t i = off[r]; i < off[r + 1]; ++i)
      if (idx[i] >= 0) idx[i] = n++;
    s_cnt[r % kBudgetThreads] = n;  // n_req <= kBudgetThreads (host check)
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t acc = 0;
    for (int32_t r = 0; r < n_req; ++r) {
      const int32_t n = s_cnt[r];
      s_cnt[r] = acc;
      off_out[r] = acc;
      acc += n;
    }
    off_out[n_req] = acc;
    *n_kept = acc;
  }
  __syncthreads();
  for (int32_t r = threadIdx.x; r < n_req; r += blockDim.x) {
    const int32_t a = off[r], base = s_cnt[r];
    for (int32_t i = a; i < off[r + 1]; ++i) {
      if (idx[i] < 0) continue;
      const int32_t o = base + idx[i];
      parent_out[o] = i == a ? -1 : idx[a + parent[i]];
      draft_out[o] = draft[i];
      src_out[o] = i;
    }
  }
}

// out[i] = x[src[i]] (zero rows where src[i] is outside 0..n_src-1), one block per row.
__global__ void __launch_bounds__(256) k_gather_rows(const uint16_t* __restrict__ x, int64_t n_src,
                                                     const int32_t* __restrict__ src, int64_t K,
                                                     uint16_t* __restrict__ out) {
  if (threadIdx.x == 0) pdl_signal();
  pdl_wait();  // the source rows may be the previous kernel's
  const int64_t i = blockIdx.x;
  const int32_t s = src[i];
  const uint16_t* row = (s >= 0 && s < n_src) ? x + (int64_t)s * K : nullptr;
  uint16_t* o = out + i * K;
  if ((K % 8) == 0 && (((uintptr_t)x | (uintptr_t)out) & 15u) == 0) {
    for (int64_t k = threadIdx.x; k < K / 8; k += blockDim.x)
      reinterpret_cast<uint4*>(o)[k] = row ? reinterpret_cast<const uint4*>(row)[k] : make_uint4(0, 0, 0, 0);
  } else {
    for (int64_t k = threadIdx.x; k < K; k += blockDim.x) o[k] = row ? row[k] : (uint16_t)0;
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
  W12_CUDA_TRY(launch_pdl(k_tlv_splice, dim3((unsigned)n), dim3(256), 0, (cudaStream_t)stream, path_len, path_nodes,
                          bonus, draft_q, x_q, n_q, sub_parent, sub_draft, x_sub, n, K, parent_out, draft_out, src_out,
                          x_out));
  W12_LAUNCH_CHECK("tlv_splice kernel");
  return W12_OK;
}

int tree_budget_select(const int32_t* parent, const float* conf, const int32_t* draft, const int32_t* req_offsets,
                       int32_t n_req, int32_t C, int32_t budget, int32_t per_request, int32_t* parent_out,
                       int32_t* draft_out, int32_t* src_out, int32_t* offsets_out, int32_t* n_kept, void* stream) {
  if (!parent || !conf || !draft || !req_offsets || !parent_out || !draft_out || !src_out || !offsets_out || !n_kept)
    return fail(W12_ERR_INVALID_ARG, "tree_budget_select: null pointer");
  if (n_req < 1 || n_req > kBudgetThreads || C < 1 || C > kBudgetMaxNodes || budget < 1)
    return fail(W12_ERR_SHAPE, "tree_budget_select: n_req=%d (1..%d), C=%d (1..%d), budget=%d (>= 1)", n_req,
                kBudgetThreads, C, kBudgetMaxNodes, budget);
  const size_t smem = (size_t)C * 16;
  static int configured[64] = {0};
  int dev = 0;
  W12_CUDA_TRY(cudaGetDevice(&dev));
  if (dev >= 64 || !configured[dev]) {
    W12_CUDA_TRY(cudaFuncSetAttribute(k_budget_select, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      kBudgetMaxNodes * 16));
    if (dev < 64) configured[dev] = 1;
  }
  k_budget_select<<<1, kBudgetThreads, smem, (cudaStream_t)stream>>>(parent, conf, draft, req_offsets, n_req, C, budget,
                                                                    per_request, parent_out, draft_out, src_out,
                                                                    offsets_out, n_kept);
  W12_LAUNCH_CHECK("tree_budget_select kernel");
  return W12_OK;
}

int gather_rows(const uint16_t* x, int64_t n_src, const int32_t* src, int64_t n, int64_t K, uint16_t* out,
                void* stream) {
  if (!x || !src || !out) return fail(W12_ERR_INVALID_ARG, "gather_rows: null pointer");
  if (n < 1 || n > 0x7FFFFFFF || n_src < 1 || K < 1 || K > kMaxK)
    return fail(W12_ERR_SHAPE, "gather_rows: n=%lld, n_src=%lld, K=%lld out of range", (long long)n, (long long)n_src,
                (long long)K);
  W12_CUDA_TRY(launch_pdl(k_gather_rows, dim3((unsigned)n), dim3(256), 0, (cudaStream_t)stream, x, n_src, src, K, out));
  W12_LAUNCH_CHECK("gather_rows kernel");
  return W12_OK;
}

}  // extern "C"
