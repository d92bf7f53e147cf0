/*
 * w12_oracle.c - plain CPU oracle for the W12 verify path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant generator with the CUDA library, and the CUDA
 * library never calls it.
 *
 * Source of every definition below: the SpecPilot summary page
 * (onedev.kr/papers/1654), section "What's different" (무엇과 다른가), which
 * describes W12 as: per channel, pick the 16-binade interval in which the
 * weights cluster; store sign 1 bit, exponent offset 4 bits and mantissa
 * 7 bits in 12 bits; restore values outside the interval, zeros and denormals
 * exactly from a per-channel sparse escape list; the two-level verification
 * Q pass reads an 8-bit view of the front of the W12 record; acceptance is
 * greedy along the draft tree with a bonus token.  Where that paragraph is
 * silent this file takes the plainest reading:
 *   - record r = s<<11 | (E-base)<<7 | m   (s: sign bit, E: 8-bit exponent
 *     field, m: 7-bit mantissa of the bf16 value);
 *   - stored as a hi plane (r >> 4, one byte per weight: the 8-bit front view)
 *     and a lo plane (r & 0xF, two weights per byte, even k in the low nibble);
 *   - the window is [base, base+15] with base in 1..239 (normal exponents
 *     only); the fullest window wins, ties go to the lowest base, and a row
 *     with no normal value gets base 1;
 *   - E = 0 (zeros, denormals) and E = 255 (Inf, NaN) are always escapes;
 *   - an escape entry is one u32: col<<16 | raw bf16 bits, entries of a row
 *     sorted by col, rows delimited by rowptr[N+1]; the record slot of an
 *     escaped weight holds r = 0;
 *   - the 8-bit view truncates: the low 4 mantissa bits read as zero;
 *     escapes stay exact in that view.
 * Arithmetic is fp64 with sums taken in increasing k.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static int exponent_field(uint16_t w) { return (w >> 7) & 0xFF; }

/* Window choice for one channel: hist[E] over normal values, then the first
 * base with the strictly largest count of E in [base, base+15]. */
int w12o_base(const uint16_t* row, int64_t K) {
  int64_t hist[256];
  memset(hist, 0, sizeof(hist));
  for (int64_t k = 0; k < K; ++k) {
    int E = exponent_field(row[k]);
    if (E >= 1 && E <= 254) hist[E] += 1;
  }
  int best_base = 1;
  int64_t best_count = -1;
  for (int b = 1; b <= 239; ++b) {
    int64_t count = 0;
    for (int E = b; E <= b + 15; ++E) count += hist[E];
    if (count > best_count) {
      best_count = count;
      best_base = b;
    }
  }
  return best_base;
}

/* True when weight w is stored as a 12-bit record under window base. */
static int in_window(uint16_t w, int base) {
  int E = exponent_field(w);
  return E >= 1 && E <= 254 && E >= base && E <= base + 15;
}

/* Encode an N x K bf16 matrix.  hi[N*K], lo[N*ceil(K/2)], base[N], rowptr[N+1];
 * esc may be NULL (count only).  Returns the number of escapes, or -1 when
 * esc_cap is too small. */
int64_t w12o_encode(const uint16_t* W, int64_t N, int64_t K, uint8_t* hi, uint8_t* lo, uint8_t* base,
                    uint32_t* rowptr, uint32_t* esc, int64_t esc_cap) {
  int64_t lo_row = (K + 1) / 2;
  int64_t n_esc = 0;
  for (int64_t n = 0; n < N; ++n) {
    const uint16_t* row = W + n * K;
    int b = w12o_base(row, K);
    if (base) base[n] = (uint8_t)b;
    if (rowptr) rowptr[n] = (uint32_t)n_esc;
    if (lo) memset(lo + n * lo_row, 0, (size_t)lo_row);
    for (int64_t k = 0; k < K; ++k) {
      uint16_t w = row[k];
      uint32_t r;
      if (in_window(w, b)) {
        uint32_t s = (w >> 15) & 1u;
        uint32_t eo = (uint32_t)(exponent_field(w) - b);
        uint32_t m = w & 0x7Fu;
        r = (s << 11) | (eo << 7) | m;
      } else {
        r = 0;
        if (esc) {
          if (n_esc >= esc_cap) return -1;
          esc[n_esc] = ((uint32_t)k << 16) | w;
        }
        n_esc += 1;
      }
      if (hi) hi[n * K + k] = (uint8_t)(r >> 4);
      if (lo) lo[n * lo_row + k / 2] |= (uint8_t)((r & 0xFu) << ((k & 1) ? 4 : 0));
    }
  }
  if (rowptr) rowptr[N] = (uint32_t)n_esc;
  return n_esc;
}

/* Record of weight (n, k) from the two planes. */
static uint32_t record_at(const uint8_t* hi, const uint8_t* lo, int64_t K, int64_t n, int64_t k) {
  int64_t lo_row = (K + 1) / 2;
  uint32_t h = hi[n * K + k];
  uint32_t l = (lo[n * lo_row + k / 2] >> ((k & 1) ? 4 : 0)) & 0xFu;
  return (h << 4) | l;
}

/* Decode: in-window weights from their record and the channel base, escaped
 * weights from the escape list.  q8 != 0 gives the 8-bit front view. */
static void decode_impl(int64_t N, int64_t K, const uint8_t* hi, const uint8_t* lo, const uint8_t* base,
                        const uint32_t* rowptr, const uint32_t* esc, uint16_t* out, int q8) {
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t k = 0; k < K; ++k) {
      uint32_t r = q8 ? ((uint32_t)hi[n * K + k] << 4) : record_at(hi, lo, K, n, k);
      uint32_t s = (r >> 11) & 1u;
      uint32_t eo = (r >> 7) & 0xFu;
      uint32_t m = r & 0x7Fu;
      out[n * K + k] = (uint16_t)((s << 15) | ((base[n] + eo) << 7) | m);
    }
    for (uint32_t e = rowptr[n]; e < rowptr[n + 1]; ++e) {
      int64_t col = esc[e] >> 16;
      out[n * K + col] = (uint16_t)(esc[e] & 0xFFFFu);
    }
  }
}

void w12o_decode(int64_t N, int64_t K, const uint8_t* hi, const uint8_t* lo, const uint8_t* base,
                 const uint32_t* rowptr, const uint32_t* esc, uint16_t* out) {
  decode_impl(N, K, hi, lo, base, rowptr, esc, out, 0);
}

void w12o_decode_q8(int64_t N, int64_t K, const uint8_t* hi, const uint8_t* base, const uint32_t* rowptr,
                    const uint32_t* esc, uint16_t* out) {
  decode_impl(N, K, hi, NULL, base, rowptr, esc, out, 1);
}

static double bf16_value(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* y[m*ldy + n] = sum_k x[m,k] * W[n,k] in fp64, k increasing; bound[m*ldy + n]
 * = sum_k |x[m,k] * W[n,k]| (may be NULL).  W holds N rows of K bf16 values. */
void w12o_gemm(const uint16_t* x, int64_t M, int64_t K, const uint16_t* W, int64_t N, double* y, int64_t ldy,
               double* bound) {
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0, mag = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        double p = bf16_value(x[m * K + k]) * bf16_value(W[n * K + k]);
        acc += p;
        mag += p < 0 ? -p : p;
      }
      y[m * ldy + n] = acc;
      if (bound) bound[m * ldy + n] = mag;
    }
  }
}

/* Ordering used by argmax: NaN ranks below every number, -0 equals +0. */
static int better(double a, double b) {
  if (a != a) return 0;
  if (b != b) return 1;
  return a > b;
}

/* Row-wise argmax of an M x V matrix; ties go to the lowest index.  gap[m] =
 * value at the argmax minus the largest value at any other index (+inf when
 * V == 1); may be NULL. */
void w12o_argmax(const double* logits, int64_t M, int64_t V, int32_t* idx, double* gap) {
  for (int64_t m = 0; m < M; ++m) {
    const double* row = logits + m * V;
    int64_t best = 0;
    for (int64_t v = 1; v < V; ++v)
      if (better(row[v], row[best])) best = v;
    idx[m] = (int32_t)best;
    if (gap) {
      int64_t second = -1;
      for (int64_t v = 0; v < V; ++v) {
        if (v == best) continue;
        if (second < 0 || better(row[v], row[second])) second = v;
      }
      gap[m] = second < 0 ? 1.0 / 0.0 : row[best] - row[second];
    }
  }
}

/* Greedy acceptance on one draft tree of n nodes (node 0 = root, parent[0] =
 * -1, parent[i] < i).  tok[i] is the target's greedy token after node i;
 * draft[i] is node i's drafted token (draft[0] unused).  Node i is accepted
 * when its parent is accepted and draft[i] == tok[parent[i]].  The answer is
 * the deepest accepted node (lowest index among equals), the root-to-node
 * path, and the bonus token tok[node].  Writes the path (root first) to
 * path_nodes[0..L] and returns L, the number of accepted draft tokens; returns
 * -1 for an invalid tree. */
int32_t w12o_accept(const int32_t* tok, const int32_t* parent, const int32_t* draft, int32_t n, int32_t* path_nodes,
                    int32_t* bonus) {
  if (n < 1 || parent[0] != -1) return -1;
  int32_t* acc = (int32_t*)malloc(sizeof(int32_t) * (size_t)n);
  int32_t* depth = (int32_t*)malloc(sizeof(int32_t) * (size_t)n);
  acc[0] = 1;
  depth[0] = 0;
  int32_t best = 0;
  for (int32_t i = 1; i < n; ++i) {
    int32_t p = parent[i];
    if (p < 0 || p >= i) {
      free(acc);
      free(depth);
      return -1;
    }
    acc[i] = acc[p] && draft[i] == tok[p];
    depth[i] = depth[p] + 1;
    if (acc[i] && depth[i] > depth[best]) best = i;
  }
  int32_t L = depth[best];
  int32_t v = best;
  for (int32_t j = L; j >= 0; --j) {
    path_nodes[j] = v;
    v = parent[v];
  }
  *bonus = tok[best];
  free(acc);
  free(depth);
  return L;
}

/* Two-level verification splice (same page and section, TLV sentence: the Q
 * pass over the 8-bit view finds the matching path and the bonus token in the
 * draft tree; a subtree drafted again at its end is attached, and the 32-node
 * tree is checked by one exact pass).  The page gives no numbering; the
 * plainest one is used:
 *   node 0..L      the Q pass's accepted path, in path order (node 0 = root);
 *                  node i's parent is i-1 and its draft is draft_q[path[i]];
 *   node L+1       the bonus node: parent L, draft = the Q pass's bonus token;
 *   node L+2+j     subtree node j (j < n - L - 2): parent L+1 when
 *                  sub_parent[j] < 0, else L+2+sub_parent[j]; draft sub_draft[j].
 * src[i] is the Q-pass row node i reuses (path[i] for i <= L) or -1 - r for
 * new row r (the bonus node takes new row 0, subtree node j new row j+1).
 * Returns 0; returns -1 (and fills nothing) when the Q result is invalid
 * (L < 0) or the path leaves no room for the bonus node (L + 2 > n), or when
 * a subtree parent is not an earlier subtree node. */
int32_t w12o_tlv_splice(int32_t L, const int32_t* path, int32_t bonus, const int32_t* draft_q,
                        const int32_t* sub_parent, const int32_t* sub_draft, int32_t n, int32_t* parent,
                        int32_t* draft, int32_t* src) {
  if (L < 0 || L + 2 > n) return -1;
  for (int32_t j = 0; j < n - L - 2; ++j)
    if (sub_parent[j] >= j) return -1;
  for (int32_t i = 0; i <= L; ++i) {
    parent[i] = i - 1;
    draft[i] = draft_q[path[i]];
    src[i] = path[i];
  }
  parent[L + 1] = L;
  draft[L + 1] = bonus;
  src[L + 1] = -1;
  for (int32_t j = 0; j < n - L - 2; ++j) {
    const int32_t i = L + 2 + j;
    parent[i] = sub_parent[j] < 0 ? L + 1 : L + 2 + sub_parent[j];
    draft[i] = sub_draft[j];
    src[i] = -1 - (j + 1);
  }
  return 0;
}

/* Node budget shared across requests (same page and section: for batching, one node
 * budget shared by all requests, 192 nodes for 24 requests).  The page gives no
 * selection rule; the plainest one is used.  Request r owns candidate nodes
 * off[r]..off[r+1]-1 (parent relative to the request, -1 for its root, parent < index);
 * node i has a draft confidence conf[i] in (0, 1].  Its path score is the float product
 * of the confidences from the root to i, taken root first (score of a root = its own
 * confidence).  Nodes are ranked by (score descending, depth ascending, index
 * ascending) and the first `budget` are kept: over all requests when per_request is 0,
 * within each request (budget nodes each) otherwise.  A child never outranks its parent,
 * so the kept set is closed under ancestors, and when conf is a calibrated acceptance
 * probability it maximises the expected number of accepted nodes.  The kept nodes of a
 * request are renumbered in their original order; outputs are parent_out, draft_out and
 * src_out (the candidate index) per kept node, requests one after another, and
 * off_out[n_req+1].  Returns the number kept, or -1 for an invalid candidate tree. */
int32_t w12o_budget_select(const int32_t* parent, const float* conf, const int32_t* draft, const int32_t* off,
                           int32_t n_req, int32_t budget, int32_t per_request, int32_t* parent_out,
                           int32_t* draft_out, int32_t* src_out, int32_t* off_out) {
  const int32_t C = off[n_req];
  float* score = (float*)malloc(sizeof(float) * (size_t)(C > 0 ? C : 1));
  int32_t* depth = (int32_t*)malloc(sizeof(int32_t) * (size_t)(C > 0 ? C : 1));
  int32_t* req = (int32_t*)malloc(sizeof(int32_t) * (size_t)(C > 0 ? C : 1));
  int32_t* keep = (int32_t*)malloc(sizeof(int32_t) * (size_t)(C > 0 ? C : 1));
  int32_t* newidx = (int32_t*)malloc(sizeof(int32_t) * (size_t)(C > 0 ? C : 1));
  int32_t kept = 0;
  for (int32_t r = 0; r < n_req && kept >= 0; ++r) {
    if (off[r + 1] <= off[r] || parent[off[r]] != -1) kept = -1;
    for (int32_t i = off[r]; i < off[r + 1] && kept >= 0; ++i) {
      const int32_t p = parent[i];
      req[i] = r;
      if (i == off[r]) {
        score[i] = conf[i];
        depth[i] = 0;
      } else if (p < 0 || p >= i - off[r]) {
        kept = -1;
      } else {
        score[i] = score[off[r] + p] * conf[i];
        depth[i] = depth[off[r] + p] + 1;
      }
    }
  }
  if (kept == 0) {
    /* rank of node i = number of nodes that come before it in the order (among all
     * nodes, or among its request's) */
    for (int32_t i = 0; i < C; ++i) {
      int32_t rank = 0;
      for (int32_t j = 0; j < C; ++j) {
        if (j == i || (per_request && req[j] != req[i])) continue;
        const int before = score[j] > score[i] ||
                           (score[j] == score[i] && (depth[j] < depth[i] || (depth[j] == depth[i] && j < i)));
        rank += before;
      }
      keep[i] = rank < budget;
    }
    for (int32_t r = 0; r < n_req; ++r) {
      off_out[r] = kept;
      int32_t n = 0;
      for (int32_t i = off[r]; i < off[r + 1]; ++i) {
        if (!keep[i]) continue;
        newidx[i] = n;
        parent_out[kept + n] = i == off[r] ? -1 : newidx[off[r] + parent[i]];
        draft_out[kept + n] = draft[i];
        src_out[kept + n] = i;
        ++n;
      }
      kept += n;
    }
    off_out[n_req] = kept;
  }
  free(score);
  free(depth);
  free(req);
  free(keep);
  free(newidx);
  return kept;
}

/* ---------------------------------------------------------------------------
 * Certified LM-head argmax (same page and section: on H100 the LM head stays
 * in INT8 and a Cauchy-Schwarz error bound filters the candidates, which are
 * then computed exactly; on an RTX PRO 6000 that was slower than a W12 head).
 * Readings where the sentence is silent:
 *   - INT8 is symmetric per output channel: s = (float)(max_k |w| / 127)
 *     (s = 0 for an all-zero row), q = rint(w / s) in [-127, 127] (ties to
 *     even), stored as the byte sign<<7 | |q|; weights are finite;
 *   - the approximate logit of channel v is s_v * sum_k x_k q_k.  Its distance
 *     to the exact logit sum_k x_k w_k is at most
 *         ||x|| * ( ||w_v - s_v q_v|| + gamma * s_v * ||q_v|| )
 *     by Cauchy-Schwarz: the first term is the quantization error, the second
 *     (gamma = (K + 16) * 2^-21) covers a float accumulation of the
 *     approximate sum, where the products are exact;
 *     c_v = ||w_v - s_v q_v|| + gamma * s_v * ||q_v|| is kept per channel,
 *     rounded up to float;
 *   - candidates are the channels whose approximate logit plus bound reaches
 *     the largest approximate logit minus bound; their exact logits decide,
 *     ties to the lowest index, as in w12o_argmax.
 */
#include <math.h>

static float round_up_float(double d) {
  float f = (float)d;
  if ((double)f < d) f = nextafterf(f, INFINITY);
  return f;
}

static double i8_gamma(int64_t K) { return (double)(K + 16) * ldexp(1.0, -21); }

/* code[N*K] (sign<<7 | |q|), scale[N], cbound[N]. */
void w12o_i8_quantize(const uint16_t* W, int64_t N, int64_t K, uint8_t* code, float* scale, float* cbound) {
  const double gamma = i8_gamma(K);
  for (int64_t n = 0; n < N; ++n) {
    const uint16_t* row = W + n * K;
    float amax = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
      float a = (float)fabs(bf16_value(row[k]));
      if (a > amax) amax = a;
    }
    const float s = amax / 127.0f;
    double e2 = 0.0, q2 = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      const double w = bf16_value(row[k]);
      double q = 0.0;
      if (s > 0.0f) {
        q = rint(w / (double)s);
        if (q > 127.0) q = 127.0;
        if (q < -127.0) q = -127.0;
      }
      const int iq = (int)q;
      code[n * K + k] = (uint8_t)((iq < 0 ? 0x80 : 0x00) | (iq < 0 ? -iq : iq));
      const double d = w - (double)s * q;
      e2 += d * d;
      q2 += q * q;
    }
    scale[n] = s;
    cbound[n] = round_up_float(sqrt(e2) + gamma * (double)s * sqrt(q2));
  }
}

static double i8_value(uint8_t c) { return (c & 0x80) ? -(double)(c & 0x7F) : (double)(c & 0x7F); }

/* For each of the M rows of x: the argmax over V channels of the exact logits,
 * found through the certified candidates.  idx[m], ncand[m] (candidates of row
 * m); returns the total number of candidates. */
int64_t w12o_cert_argmax(const uint16_t* x, int64_t M, int64_t K, const uint16_t* W, int64_t V, const uint8_t* code,
                         const float* scale, const float* cbound, int32_t* idx, int32_t* ncand) {
  int64_t total = 0;
  double* lo = (double*)malloc(sizeof(double) * (size_t)V);
  double* hi = (double*)malloc(sizeof(double) * (size_t)V);
  for (int64_t m = 0; m < M; ++m) {
    const uint16_t* xr = x + m * K;
    double nx2 = 0.0;
    for (int64_t k = 0; k < K; ++k) nx2 += bf16_value(xr[k]) * bf16_value(xr[k]);
    const double nx = sqrt(nx2);
    double thr = -INFINITY;
    for (int64_t v = 0; v < V; ++v) {
      double a = 0.0;
      for (int64_t k = 0; k < K; ++k) a += bf16_value(xr[k]) * i8_value(code[v * K + k]);
      const double approx = (double)scale[v] * a, b = nx * (double)cbound[v];
      lo[v] = approx - b;
      hi[v] = approx + b;
      if (lo[v] > thr) thr = lo[v];
    }
    int64_t best = -1, count = 0;
    double best_val = 0.0;
    for (int64_t v = 0; v < V; ++v) {
      if (hi[v] < thr) continue;
      ++count;
      double L = 0.0;
      for (int64_t k = 0; k < K; ++k) L += bf16_value(xr[k]) * bf16_value(W[v * K + k]);
      if (best < 0 || better(L, best_val)) {
        best = v;
        best_val = L;
      }
    }
    idx[m] = (int32_t)best;
    ncand[m] = (int32_t)count;
    total += count;
  }
  free(lo);
  free(hi);
  return total;
}

/* ---------------------------------------------------------------------------
 * Hybrid-target recurrent verification (same page and section: for a target
 * whose layers are mostly Gated DeltaNet, a path-verify kernel recomputes the
 * recurrent state along each path instead of snapshotting it per node, a
 * commit kernel replays the accepted path into the layers' states, and the
 * WY kernel keeps the FP32 state as three BF16 pieces that hold its 24-bit
 * significand exactly).  Readings where the sentence is silent:
 *   - the recurrence is the gated delta rule on a d_v x d_k state:
 *       S_t = alpha_t * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *       o_t = S_t q_t,
 *     per head, with q, k, v bf16 and alpha, beta float;
 *   - a tree node's state is the root state S0 advanced by the updates of
 *     every node on its path from the first draft node down to itself (node 0
 *     is the committed root: its update is already in S0);
 *   - the split of a float x is s1 = bf16_rne(x), s2 = bf16_rne(x - s1),
 *     s3 = bf16_rne(x - s1 - s2), the differences taken in float.
 * Arithmetic is fp64 (the split is float, as the reading states).
 */
static uint16_t bf16_rne_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static float bf16_float(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

void w12o_split3(const float* x, int64_t n, uint16_t* s1, uint16_t* s2, uint16_t* s3) {
  for (int64_t i = 0; i < n; ++i) {
    const float a = x[i];
    s1[i] = bf16_rne_bits(a);
    const float r1 = a - bf16_float(s1[i]);
    s2[i] = bf16_rne_bits(r1);
    const float r2 = r1 - bf16_float(s2[i]);
    s3[i] = bf16_rne_bits(r2);
  }
}

/* One gated delta update of a dv x dk state (row-major S[v*dk + k]). */
static void gdn_step(double* S, int64_t dk, int64_t dv, const uint16_t* k, const uint16_t* v, double alpha,
                     double beta) {
  for (int64_t r = 0; r < dv; ++r) {
    double u = 0.0;
    for (int64_t c = 0; c < dk; ++c) u += S[r * dk + c] * bf16_value(k[c]);
    const double coef = beta * bf16_value(v[r]) - alpha * beta * u;
    for (int64_t c = 0; c < dk; ++c) S[r * dk + c] = alpha * S[r * dk + c] + coef * bf16_value(k[c]);
  }
}

/* Outputs of every node of a tree of n nodes for H heads.  S0[h*dv*dk] (float),
 * q, k [n*H*dk], v [n*H*dv] (bf16), alpha, beta [n*H], parent[n] (parent[0] = -1,
 * parent[i] < i).  O[(i*H + h)*dv + r] = (S_i q_i)[r].  Returns 0, or -1 for an
 * invalid tree. */
int w12o_gdn_tree(const float* S0, const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* alpha,
                  const float* beta, const int32_t* parent, int64_t n, int64_t H, int64_t dk, int64_t dv, double* O) {
  if (n < 1 || parent[0] != -1) return -1;
  for (int64_t i = 1; i < n; ++i)
    if (parent[i] < 0 || parent[i] >= i) return -1;
  double* S = (double*)malloc(sizeof(double) * (size_t)(dv * dk));
  int64_t* path = (int64_t*)malloc(sizeof(int64_t) * (size_t)n);
  for (int64_t i = 0; i < n; ++i) {
    int64_t L = 0;
    for (int64_t j = i; j > 0; j = parent[j]) path[L++] = j;  /* node i up to the first draft node */
    for (int64_t h = 0; h < H; ++h) {
      for (int64_t e = 0; e < dv * dk; ++e) S[e] = (double)S0[h * dv * dk + e];
      for (int64_t t = L - 1; t >= 0; --t) {
        const int64_t j = path[t];
        gdn_step(S, dk, dv, k + (j * H + h) * dk, v + (j * H + h) * dv, (double)alpha[j * H + h],
                 (double)beta[j * H + h]);
      }
      for (int64_t r = 0; r < dv; ++r) {
        double o = 0.0;
        for (int64_t c = 0; c < dk; ++c) o += S[r * dk + c] * bf16_value(q[(i * H + h) * dk + c]);
        O[(i * H + h) * dv + r] = o;
      }
    }
  }
  free(S);
  free(path);
  return 0;
}

/* Commit: the states after the accepted nodes nodes[0..L) (in path order, root
 * excluded) are applied to S0 -> S_out[h*dv*dk], fp64. */
void w12o_gdn_commit(const float* S0, const uint16_t* k, const uint16_t* v, const float* alpha, const float* beta,
                     const int32_t* nodes, int64_t L, int64_t H, int64_t dk, int64_t dv, double* S_out) {
  for (int64_t h = 0; h < H; ++h) {
    double* S = S_out + h * dv * dk;
    for (int64_t e = 0; e < dv * dk; ++e) S[e] = (double)S0[h * dv * dk + e];
    for (int64_t t = 0; t < L; ++t) {
      const int64_t j = nodes[t];
      gdn_step(S, dk, dv, k + (j * H + h) * dk, v + (j * H + h) * dv, (double)alpha[j * H + h],
               (double)beta[j * H + h]);
    }
  }
}
