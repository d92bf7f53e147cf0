/*
 * w12.h - C ABI of the W12 verify-path library (libw12.so, sm_103a).
 *
 * W12 is the lossless 12-bit weight format of the SpecPilot summary page
 * (onedev.kr/papers/1654), section "What's different" (무엇과 다른가): for
 * each output channel the 16-binade exponent window holding the most weights
 * is chosen; an in-window bf16 weight is stored as sign 1 bit, exponent
 * offset 4 bits and mantissa 7 bits; values outside the window, zeros and
 * denormals are restored exactly from a per-channel sparse escape list.  The
 * same paragraph describes the GEMM that decodes the 12-bit records in
 * registers behind the weight stream and stays deterministic with stream-K,
 * the two-level verification Q pass over an 8-bit view of the front of the
 * record, and the greedy acceptance of a draft tree plus a bonus token.  The
 * page's "What it is" (무엇인가) section gives why this path matters: every
 * tree node of a verify step reads the full target weights (80% of a 23.61 ms
 * step).
 *
 * Record (canonical): r = s<<11 | (E-base)<<7 | m for a bf16 value with sign s,
 * exponent field E and mantissa m; base is in 1..239; E = 0 (zeros,
 * denormals) and E = 255 (Inf, NaN) always escape; the 8-bit view is r >> 4
 * and reads the low 4 mantissa bits as zero (escapes stay exact).
 *
 * ---------------------------------------------------------------------------
 * Conventions for every call
 *  - Status: each call returns W12_OK (0) or one of the W12_ERR_* codes; the
 *    thread-local w12_last_error() then holds a one-line reason.  Nothing is
 *    thrown across the ABI.  Argument checks happen on the host before any
 *    launch; a call that fails them touches no memory.
 *  - Memory: every pointer argument is device memory owned by the caller,
 *    except where a parameter says "host".  No call allocates device memory;
 *    calls that need scratch take a caller-owned workspace whose size is given
 *    by the matching *_workspace_size query.
 *  - Streams: `stream` is a cudaStream_t (NULL = legacy default stream).  All
 *    device work is enqueued on it asynchronously; only w12_encode_plan
 *    synchronises it (it returns the escape count to the host).
 *  - The GEMM kernels (w12_gemm*, the LM-head calls, w12_cert_head_argmax)
 *    are launched with programmatic dependent launch: they may start while
 *    the previous kernel on the stream finishes and begin reading the
 *    matrix before it has completed; x, the workspace and the outputs are
 *    touched only after it completes.  A kernel that signals early
 *    (griddepcontrol.launch_dependents) must therefore not write the matrix
 *    a following GEMM reads.  Kernels that do not signal, such as the
 *    encoders here, complete before the GEMM starts.  From 64 tokens on, a
 *    call that stores y may add a second kernel, launched plainly after the
 *    GEMM's grid, that adds the rows the GEMM split between CTAs; it signals
 *    early too and writes only y.
 *  - bf16 tensors are passed as uint16_t bit patterns.
 *  - Shapes: 1 <= N, 1 <= K <= 65535 (the escape entry keeps the column in 16
 *    bits and reserves the all-ones column), 1 <= M.
 *
 * Device layout of a W12 matrix (what w12_encode writes and the kernels read)
 *  The matrix is cut into tiles of 32 channels x 64 columns.  Channels come
 *  in row blocks of 128 (RB = ceil(N/128), RT = 4*RB row tiles) and columns in
 *  KC = ceil(K/64) chunks.  The four row tiles of a block at one chunk are
 *  adjacent: tile (rt, kc) has index ((rt/4)*KC + kc)*4 + rt%4, so one row
 *  block's chunk is a single 8 KB run of the hi plane and 4 KB of the lo plane.
 *  Rows and columns past N and K hold record 0 and never escape.
 *  - hi:  RT*KC tiles of 2048 bytes, the 8-bit front view (r >> 4) of each
 *         weight.  In a tile, channel 8q+g and column 16t+j sit at byte
 *         q*512 + (4g+t)*16 + 4*(j/4) + {0,2,1,3}[j%4].
 *  - lo:  RT*KC tiles of 1024 bytes, the low nibble (r & 0xF).  Channel 8q+g,
 *         column 16t+j sits in the 8-byte group at q*256 + (4g+t)*8, at bit
 *         32*(p/4) + 4*(p%4) + 16*(j%2) of that group, p = 2*(j/4) + (j%4)/2.
 *  - base: N bytes, the window base of each channel.
 *  - esc_tile_ptr: RT*KC+1 u32, exclusive prefix of escape counts per tile.
 *  - esc: n_esc u32 entries, grouped by tile and sorted by (channel, column)
 *         within a tile: raw bf16 | slot << 16, where slot is the byte offset of
 *         (channel-in-tile r, column-in-chunk c) in the tile's decoded 32x64 bf16
 *         image with a 128-byte swizzle: r*128 + ((c/8 XOR r%8) * 16) + (c%8)*2.
 *         The allocation holds ceil(n_esc/4)*4 entries (at least 4): the GEMM
 *         copies escapes in aligned 16-byte runs.
 *  hi, lo and esc must be 16-byte aligned (cudaMalloc gives 256).
 *  w12_export_canonical converts to the canonical planes for comparison.
 */
#ifndef W12_H
#define W12_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define W12_ABI_VERSION 1

#if defined(__GNUC__)
#define W12_API __attribute__((visibility("default")))
#else
#define W12_API
#endif

typedef enum w12_status {
  W12_OK = 0,
  W12_ERR_INVALID_ARG = 1,      /* null pointer, negative count, bad stream use */
  W12_ERR_SHAPE = 2,            /* N, K or M out of range */
  W12_ERR_BUFFER_TOO_SMALL = 3, /* workspace smaller than the size query says */
  W12_ERR_CUDA = 4,             /* a CUDA runtime call or launch failed */
  W12_ERR_BOUNDS = 5,           /* device data inconsistent with the descriptor (w12_validate,
                                   w12_workspace_status) */
  W12_ERR_TIMEOUT = 6,          /* a GEMM kernel's device-side wait ran out (w12_workspace_status) */
  W12_ERR_IO = 7                /* a file could not be read or written, or is not a W12 matrix file */
} w12_status;

/* A W12 matrix in device memory (layout above).  The struct itself lives in
 * host memory; the library reads it during the call and keeps no reference. */
typedef struct w12_matrix {
  int64_t N, K;
  uint8_t* hi;
  uint8_t* lo;
  uint8_t* base;
  uint32_t* esc_tile_ptr;
  uint32_t* esc;
  int64_t n_esc;
} w12_matrix;

/* One-line reason for the last non-OK status on this host thread. */
W12_API const char* w12_last_error(void);
/* Name of a status code. */
W12_API const char* w12_status_string(int status);
/* W12_ABI_VERSION of the loaded library. */
W12_API int w12_abi_version(void);

/* ---- sizes (pure host functions, no CUDA calls) ------------------------- */

/* Bytes of the hi plane, the lo plane, and tiles (4*ceil(N/128)*ceil(K/64)) of
 * an N x K matrix; -1 for an invalid shape. */
W12_API int64_t w12_hi_bytes(int64_t N, int64_t K);
W12_API int64_t w12_lo_bytes(int64_t N, int64_t K);
W12_API int64_t w12_tile_count(int64_t N, int64_t K);

/* ---- storage (pages: "What's different": the converted layers are stored) */

/* Writes the device matrix A to the file `path`: a 72-byte little-endian header
 * (magic "W12M", format 1, N, K, n_esc and the byte counts of the five arrays)
 * followed by the hi plane, the lo plane, base[N], esc_tile_ptr[tile_count+1]
 * and esc[n_esc], as laid out on the device.  Copies through a bounded host
 * buffer and synchronises `stream`.  Errors: W12_ERR_INVALID_ARG (null
 * pointers), W12_ERR_SHAPE, W12_ERR_IO (the file cannot be written),
 * W12_ERR_CUDA. */
W12_API int w12_save(const w12_matrix* A, const char* path, void* stream);

/* N, K and n_esc (host pointers) of a file w12_save wrote, so that the caller can
 * allocate the planes (w12_hi_bytes, w12_lo_bytes, N bytes of bases,
 * w12_tile_count+1 offsets, n_esc escapes rounded up to a multiple of 4).
 * Errors: W12_ERR_INVALID_ARG, W12_ERR_IO (no such file, not a W12 matrix file,
 * a truncated header or sizes that do not match the shape). */
W12_API int w12_load_info(const char* path, int64_t* N, int64_t* K, int64_t* n_esc);

/* Copies the arrays of the file into the device buffers A describes (A->N,
 * A->K and A->n_esc must equal the file's); synchronises `stream`.  Errors:
 * W12_ERR_INVALID_ARG, W12_ERR_SHAPE (the descriptor's sizes differ from the
 * file's), W12_ERR_IO (unreadable, not a W12 matrix file or truncated),
 * W12_ERR_CUDA. */
W12_API int w12_load(const char* path, const w12_matrix* A, void* stream);

/* ---- encode (pages: "What's different", W12 conversion) ----------------- */

/* Step 1 of 2.  Reads W[N*K] (bf16, row-major, channel n = row n), writes the
 * window base of every channel to base[N] and the tile escape offsets to
 * esc_tile_ptr[tile_count+1], and stores the total escape count in *n_esc
 * (host pointer).  Synchronises `stream` to return the count. */
W12_API int w12_encode_plan(const uint16_t* W, int64_t N, int64_t K, uint8_t* base, uint32_t* esc_tile_ptr,
                    int64_t* n_esc, void* stream);

/* Step 2 of 2.  A->base and A->esc_tile_ptr must hold step 1's output for the
 * same W; A->hi, A->lo and A->esc (A->n_esc entries, may be NULL when 0) are
 * written.  Asynchronous. */
W12_API int w12_encode(const uint16_t* W, const w12_matrix* A, void* stream);

/* ---- decode ------------------------------------------------------------- */

/* Exact inverse of encode: W_out[N*K] bf16 row-major. */
W12_API int w12_decode(const w12_matrix* A, uint16_t* W_out, void* stream);
/* The 8-bit view: in-window weights with the low 4 mantissa bits cleared,
 * escapes exact.  Reads only hi, base and the escapes. */
W12_API int w12_decode_q8(const w12_matrix* A, uint16_t* W_out, void* stream);

/* Canonical planes: hi_out[N*K] = r >> 4; lo_out[N*ceil(K/2)] with even
 * columns in the low nibble; rowptr_out[N+1]; esc_out[n_esc] = col<<16 | raw,
 * sorted by column within each channel.  Asynchronous. */
W12_API int w12_export_canonical(const w12_matrix* A, uint8_t* hi_out, uint8_t* lo_out, uint32_t* rowptr_out,
                         uint32_t* esc_out, void* stream);

/* ---- verify GEMM (pages: "What's different", decode-fused stream-K GEMM) -- */

/* Workspace bytes for w12_gemm / w12_gemm_q8 with these shapes on the current
 * device.  The workspace's first w12_gemm_counter_bytes(N) bytes (an error word
 * in the first 256 bytes, then one tile counter per row tile: four per 128-row
 * block) must be zero
 * before the first call; every call that completes without a device error
 * leaves them zero again, and w12_workspace_status clears them after one. */
W12_API size_t w12_gemm_workspace_size(int64_t M, int64_t N, int64_t K);
W12_API size_t w12_gemm_counter_bytes(int64_t N);

/* y[M*N] (fp32, row-major, token m = row m) = x[M*K] (bf16, row-major) times
 * decode(A)^T, fp32 accumulation.  The K range is split over warps by a fixed
 * partition and partial sums are added in a fixed order, so repeated calls
 * give identical bits.  Asynchronous. */
W12_API int w12_gemm(const uint16_t* x, int64_t M, const w12_matrix* A, float* y, void* ws, size_t ws_bytes, void* stream);

/* Same, with the 8-bit view of the weights (the two-level verification Q
 * pass).  Reads only hi, base and the escapes. */
W12_API int w12_gemm_q8(const uint16_t* x, int64_t M, const w12_matrix* A, float* y, void* ws, size_t ws_bytes,
                void* stream);

/* ---- device errors of the GEMM kernels -------------------------------------
 * Every wait of a GEMM kernel (for records to land, a buffer to be released, an
 * accumulator to be ready) is bounded.  A CTA whose wait runs out stops its work,
 * waits for its own copies and MMAs in flight, frees its tensor memory and sets
 * a bit in the workspace's error word; the launch then ends normally and the call
 * returned W12_OK, but its outputs are incomplete.  A CTA that meets an escape
 * offset beyond the matrix's escape list clamps it and sets another bit.  The
 * word covers w12_gemm, w12_gemm_q8, the LM-head calls and w12_cert_head_argmax
 * (whose workspaces start with the GEMM's). */

/* Synchronises `stream`, then stores in *status (host) W12_ERR_TIMEOUT if a wait
 * of a call on this workspace ran out since the last query, else W12_ERR_BOUNDS if
 * an escape offset was out of range, else W12_OK.  After an error it zeroes the
 * whole workspace (ws_bytes), so that tile counters left raised by a CTA that gave
 * up do not disturb the next call.  Returns W12_OK, or W12_ERR_INVALID_ARG /
 * W12_ERR_BUFFER_TOO_SMALL (ws_bytes < 256) / W12_ERR_CUDA. */
W12_API int w12_workspace_status(void* ws, size_t ws_bytes, int32_t* status, void* stream);

/* Diagnostic for tests of the path above: bounds the GEMM kernels' waits for another
 * warp's work at `cycles` SM clock cycles on the current device (cycles <= 0
 * restores the default, 2^31, about a second).  Waits for a CTA's own copies and
 * MMAs keep the default.  Synchronous; kernels launched after it returns see it. */
W12_API int w12_set_wait_limit(int64_t cycles);

/* Checks the index arrays of A against its descriptor without touching the planes
 * (the GEMM trusts them): esc_tile_ptr rises from 0 to n_esc; every entry of a
 * tile's run is an even slot of the 32x64 tile image, names a channel < N and a
 * column < K, and follows the previous entry of the tile in (channel, column)
 * order; every window base is in 1..239.  Writes W12_OK or W12_ERR_BOUNDS to
 * *status (device int32).  Reads esc only at offsets below n_esc.  Asynchronous.
 * Errors: W12_ERR_INVALID_ARG, W12_ERR_SHAPE. */
W12_API int w12_validate(const w12_matrix* A, int32_t* status, void* stream);

/* ---- verify GEMM without a caller workspace ------------------------------
 * Not part of the method: the pages have no counterpart.  It is w12_gemm for
 * callers that cannot give the library a workspace: an engine whose memory
 * planner has already reserved the whole device, a plugin or callback
 * interface with no workspace argument, or a latency-critical loop that must
 * not call cudaMalloc (which can synchronise the device).
 *  - Scratch is one library-owned device array of w12_gemm_noalloc_max_scratch()
 *    bytes (16 MiB).  Every GPU that loads libw12.so holds it until the process
 *    exits.  Nothing is allocated per call.
 *  - The first call on a device looks up the array's device address with that
 *    device current.  Make that first call before any stream capture.
 *  - Each call clears the array's error word and counters on `stream` before the
 *    GEMM; a call refused by an argument check touches nothing.
 *  - All calls share the one array: calls that can overlap on the GPU (other
 *    streams, other host threads on the same device) race and corrupt each
 *    other's results.  Serialise them.
 *  - Shapes needing more scratch than the array holds fail with W12_ERR_SHAPE
 *    (for example M <= 32 covers N up to ~34K at K = 5120; larger M or N needs
 *    w12_gemm).  Same result as w12_gemm otherwise.  Asynchronous. */
W12_API size_t w12_gemm_noalloc_max_scratch(void);
W12_API int w12_gemm_noalloc(const uint16_t* x, int64_t M, const w12_matrix* A, float* y, void* stream);

/* ---- LM head with fused argmax ----------------------------------------- */

/* Workspace bytes for the LM-head calls (same counter rule as w12_gemm). */
W12_API size_t w12_lmhead_workspace_size(int64_t M, int64_t V, int64_t K);

/* tok[M] = argmax over v of (x . decode(head)^T)[m, v]; the logits are never
 * written to memory.  Ties go to the lowest v; NaN ranks below every number.
 * head has N = V channels.  Asynchronous. */
W12_API int w12_lmhead_argmax(const uint16_t* x, int64_t M, const w12_matrix* head, int32_t* tok, void* ws,
                      size_t ws_bytes, void* stream);
W12_API int w12_lmhead_argmax_q8(const uint16_t* x, int64_t M, const w12_matrix* head, int32_t* tok, void* ws,
                         size_t ws_bytes, void* stream);

/* LM-head argmax followed by tree acceptance (tree_verify_tokens semantics)
 * in the same stream without a host round trip; tok[M] is also written. */
W12_API int w12_lmhead_verify(const uint16_t* x, int64_t M, const w12_matrix* head, int q8, const int32_t* parent,
                      const int32_t* draft, const int32_t* req_offsets, int32_t n_req, int32_t* tok,
                      int32_t* path_len, int32_t* path_nodes, int32_t* bonus, void* ws, size_t ws_bytes,
                      void* stream);

/* ---- tree acceptance (pages: "What's different", greedy path + bonus) ---- */

/* M tree nodes of n_req requests, request r owning nodes
 * [req_offsets[r], req_offsets[r+1]) (req_offsets = NULL: one request of M
 * nodes).  Node indices in parent[] and path_nodes[] are local to the
 * request; parent[first] = -1 and 0 <= parent[i] < i otherwise.  tok[i] is
 * the target's greedy token after node i, draft[i] node i's drafted token.
 * Node i is accepted when its parent is and draft[i] == tok[parent[i]]; the
 * deepest accepted node a* wins (lowest index among equals).  Outputs per
 * request: path_len[r] = depth of a*, path_nodes[off_r .. off_r+L] = the
 * root-to-a* path, bonus[r] = tok[a*].  An invalid tree or offset range gives
 * path_len[r] = -1 and bonus[r] = -1.  path_nodes[off_r ..) beyond the path
 * is scratch.  Asynchronous. */
W12_API int tree_verify_tokens(const int32_t* tok, const int32_t* parent, const int32_t* draft,
                       const int32_t* req_offsets, int32_t n_req, int64_t M, int32_t* path_len,
                       int32_t* path_nodes, int32_t* bonus, void* stream);

/* Same from fp32 logits[M*V]: the row argmax (same tie rule) gives tok;
 * workspace >= tree_verify_workspace_size(M) bytes. */
W12_API size_t tree_verify_workspace_size(int64_t M);
W12_API int tree_verify(const float* logits, int64_t M, int64_t V, const int32_t* parent, const int32_t* draft,
                const int32_t* req_offsets, int32_t n_req, int32_t* path_len, int32_t* path_nodes,
                int32_t* bonus, void* ws, size_t ws_bytes, void* stream);

/* Two-level verification splice.  SpecPilot summary page (onedev.kr/papers/1654),
 * section "What's different", TLV sentence: the Q pass over the 8-bit view finds the
 * matching path and the bonus token in the draft tree; a subtree drafted again at the
 * end of that path is attached and the resulting tree (32 nodes there) goes through one
 * exact pass.  The page gives no numbering; this call uses:
 *   node 0..L     the Q pass's accepted path in order: parent i-1, draft
 *                 draft_q[path_nodes[i]], activation row x_q[path_nodes[i]];
 *   node L+1      the bonus node: parent L, draft = *bonus, row x_sub[0];
 *   node L+2+j    subtree node j (j < n-L-2): parent L+1 when sub_parent[j] < 0, else
 *                 L+2+sub_parent[j]; draft sub_draft[j]; row x_sub[j+1].
 * Inputs (device): path_len[1], path_nodes[>= L+1], bonus[1] as tree_verify writes them
 * for one request; draft_q[n_q]; x_q[n_q*K] bf16 rows of the Q pass; sub_parent[n-2],
 * sub_draft[n-2]; x_sub[(n-1)*K].  Outputs (device): parent_out[n], draft_out[n],
 * src_out[n] (Q row reused by the node, or -1-r for x_sub row r), x_out[n*K], the exact
 * pass's rows.  When the Q result is invalid (L < 0), the path leaves no room for the
 * bonus node (L+2 > n), a path node is outside 0..n_q-1 or a subtree parent is not an
 * earlier subtree node, every parent_out is -2 (tree_verify then reports the tree
 * invalid), draft_out is -1 and x_out is zero.  The caller owns every buffer; the call is
 * asynchronous on `stream` and allocates nothing.  Errors: W12_ERR_INVALID_ARG (null
 * pointer), W12_ERR_SHAPE (n outside 2..2^20, K outside 1..65535). */
W12_API int tlv_splice(const int32_t* path_len, const int32_t* path_nodes, const int32_t* bonus,
                       const int32_t* draft_q, const uint16_t* x_q, int64_t n_q, const int32_t* sub_parent,
                       const int32_t* sub_draft, const uint16_t* x_sub, int64_t n, int64_t K, int32_t* parent_out,
                       int32_t* draft_out, int32_t* src_out, uint16_t* x_out, void* stream);

/* Node budget shared across requests.  SpecPilot summary page (onedev.kr/papers/1654),
 * section "What's different": for batching, one node budget shared by all requests (192
 * nodes for 24 requests).  The page gives no selection rule; this call uses: request r
 * owns candidate nodes req_offsets[r]..req_offsets[r+1]-1 (parent relative to the request,
 * -1 for its root, parent < index); conf[i] in (0, 1] is node i's draft confidence; the
 * path score is the float product of the confidences from the root (root first, each
 * multiply rounded); nodes are ranked by (score descending, depth ascending, index
 * ascending) and the first `budget` are kept over all requests (per_request = 0) or within
 * each request (per_request != 0).  A child never outranks its parent, so the kept set is
 * closed under ancestors; with calibrated confidences it maximises the expected number
 * of accepted nodes.  Kept nodes are renumbered per request in their original order.
 * Inputs (device): parent[C], conf[C] (fp32), draft[C], req_offsets[n_req+1] with
 * req_offsets[n_req] = C.  Outputs (device, C entries each suffice): parent_out[k],
 * draft_out[k], src_out[k] (candidate index of each kept node), offsets_out[n_req+1],
 * n_kept[1] = k, or -1 for an invalid candidate tree.  One block; asynchronous on
 * `stream`; allocates nothing.  Errors: W12_ERR_INVALID_ARG (null pointer),
 * W12_ERR_SHAPE (n_req outside 1..1024, C outside 1..4096, budget < 1). */
W12_API int tree_budget_select(const int32_t* parent, const float* conf, const int32_t* draft,
                               const int32_t* req_offsets, int32_t n_req, int32_t C, int32_t budget,
                               int32_t per_request, int32_t* parent_out, int32_t* draft_out, int32_t* src_out,
                               int32_t* offsets_out, int32_t* n_kept, void* stream);

/* Row gather for the verify pass of selected or spliced nodes (no counterpart in the
 * pages: a helper of the two calls above): out[i*K..] = x[src[i]*K..] for i < n, zero
 * rows where src[i] is outside 0..n_src-1.  x[n_src*K], src[n], out[n*K] are device
 * buffers owned by the caller; asynchronous on `stream`.  Errors: W12_ERR_INVALID_ARG,
 * W12_ERR_SHAPE (n < 1, n_src < 1, K outside 1..65535). */
W12_API int gather_rows(const uint16_t* x, int64_t n_src, const int32_t* src, int64_t n, int64_t K, uint16_t* out,
                        void* stream);

/* ---------------------------------------------------------------------------
 * Certified LM-head argmax over an INT8 head.  The SpecPilot summary page,
 * section "What's different", keeps the LM head of its H100 build in INT8 and
 * filters the argmax candidates with a Cauchy-Schwarz error bound, computing
 * only those exactly (878 -> 482 us there; on an RTX PRO 6000 it was slower
 * than a W12 head).
 *
 * INT8 head of a V x K bf16 head W (finite values), per output channel v:
 *   scale[v]  = (float)(max_k |w| / 127)   (0 for an all-zero channel)
 *   q         = rint(w / scale[v]) in [-127, 127], ties to even
 *   code      = sign<<7 | |q|, one byte per weight, in the W12 hi-plane layout
 *               (tiles of 32 channels x 64 columns, byte position as for hi;
 *               w12_i8_code_bytes(V, K) bytes, padding 0)
 *   cbound[v] = ||w_v - scale[v] q_v|| + (K + 16) 2^-21 scale[v] ||q_v||,
 *               rounded up: |x.w_v - scale[v] x.q_v| <= ||x|| cbound[v] for
 *               every x (Cauchy-Schwarz), the second term covering a float
 *               accumulation of x.q_v.
 */
typedef struct w12_i8_head {
  int64_t V, K;
  uint8_t* code;   /* 16-byte aligned */
  float* scale;    /* V */
  float* cbound;   /* V */
} w12_i8_head;

W12_API int64_t w12_i8_code_bytes(int64_t V, int64_t K);

/* Fill H (caller-allocated, H->V x H->K) from the bf16 head W[V*K].
 * Errors: W12_ERR_INVALID_ARG (null or misaligned buffer), W12_ERR_SHAPE. */
W12_API int w12_i8_encode(const uint16_t* W, const w12_i8_head* H, void* stream);

W12_API size_t w12_cert_head_workspace_size(int64_t M, int64_t V, int64_t K);

/* tok[m] = argmax_v x_m . w_v of the exact logits (lowest index on ties), for
 * the M rows of x[M*K] bf16.  The approximate logits come from H, the bound
 * selects candidates (every channel whose approximate logit plus bound reaches
 * the row's largest approximate logit minus bound, rounded outward), and the
 * candidates' logits are recomputed from `exact`, the W12 form of the same head
 * (exact bf16 products, a float-pair sum whose error is near 2^-48 sum|x*w|).  ncand[m] (may be NULL) receives the candidate count.
 * The approximate logits are never stored: the INT8 GEMM's epilogue keeps each
 * row's threshold and a superset of its candidates, which the recompute filters.
 * Workspace >= w12_cert_head_workspace_size(M, V, K) bytes, first
 * w12_gemm_counter_bytes(V) bytes zero before first use (as for w12_gemm).
 * Errors: W12_ERR_INVALID_ARG, W12_ERR_SHAPE (shapes of H and exact differ,
 * M out of 1..2^20), W12_ERR_BUFFER_TOO_SMALL. */
W12_API int w12_cert_head_argmax(const uint16_t* x, int64_t M, const w12_i8_head* H, const w12_matrix* exact,
                                 int32_t* tok, int32_t* ncand, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Recurrent layers of a hybrid target.  The SpecPilot summary page, section
 * "What's different", verifies a draft tree on a target whose layers are
 * mostly Gated DeltaNet with a path-verify kernel (the recurrent state is
 * recomputed along each path instead of snapshotted per node), a commit kernel
 * (the accepted path is replayed into the state) and FP32 state held exactly
 * as three BF16 pieces.  Recurrence per head, state S (dv x dk, row-major
 * float), q, k (dk) and v (dv) bf16, alpha and beta float:
 *     S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *     o_t = S_t q_t.
 * dk, dv <= 256 with (dk * (dv + 1) + dk + dv) * 4 <= 200 KB (W12_ERR_SHAPE
 * otherwise).
 * The three calls use programmatic dependent launch: gdn_path_verify and
 * gdn_wy_verify let the next kernel on the stream start early and read S0
 * before they wait for the previous kernel (their other inputs after it), so
 * S0 must not be written by the kernel just before them unless that kernel
 * never signals early (gdn_commit does not); gdn_commit waits for the previous
 * kernel before it reads anything.
 */

/* s1 = bf16_rne(x), s2 = bf16_rne(x - s1), s3 = bf16_rne(x - s1 - s2) (float
 * differences) for n floats; s1 + s2 + s3 == x exactly when no piece overflows
 * bf16 and |x| >= 2^-110 (or x = 0). */
W12_API int gdn_split3(const float* x, int64_t n, uint16_t* s1, uint16_t* s2, uint16_t* s3, void* stream);

/* Outputs of every node of an n-node draft tree (parent[0] = -1, parent[i] <
 * i; node 0 is the committed root, whose update is already in S0):
 * O[(i*H + h)*dv + r] = (S_i q_i)[r], S_i = S0[h] advanced by the updates of
 * the nodes on i's path below the root, root side first.  q, k [n*H*dk], v
 * [n*H*dv], alpha, beta [n*H], S0 [H*dv*dk].  A malformed tree sets bit 0 of
 * *status (device int32, zeroed by the caller) and leaves O unwritten.
 * n in 1..4096. */
W12_API int gdn_path_verify(const float* S0, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                            const float* alpha, const float* beta, const int32_t* parent, int64_t n, int64_t H,
                            int64_t dk, int64_t dv, float* O, int32_t* status, void* stream);

/* The same outputs as gdn_path_verify in the WY form: node t's state is
 * gamma_t S0 + sum_{j on path(t)} (gamma_t/gamma_j) d_j k_j^T (gamma: product of
 * alpha along the path), whose pseudo-values d_j solve a triangular system over
 * the tree; the state enters only through S0 k_t and S0 q_t, so every node is
 * computed once instead of once per path that reaches it.  Those products run on
 * the tensor core as bf16 MMAs with fp32 accumulation over the float state split
 * exactly into three bf16 pieces (gdn_split3's split), so every product of a state
 * element and a k or q element is exact.  One CTA per (head, 128 state rows).
 * dk = 64 or 128, n in 1..64, S0 16-byte aligned; other arguments, errors and
 * *status as for gdn_path_verify; a device wait that runs out (about a second)
 * sets bit 2 of *status. */
W12_API int gdn_wy_verify(const float* S0, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                          const float* alpha, const float* beta, const int32_t* parent, int64_t n, int64_t H,
                          int64_t dk, int64_t dv, float* O, int32_t* status, void* stream);

/* S[h] <- S[h] advanced by the accepted nodes path_nodes[1 .. *path_len] (device
 * values, as w12_lmhead_verify writes them: path_nodes[0] is the root), in
 * order; node inputs as for gdn_path_verify.  *path_len <= 0 commits nothing;
 * a length >= n or a node outside 1..n-1 sets bit 1 of *status and leaves S. */
W12_API int gdn_commit(float* S, const uint16_t* k, const uint16_t* v, const float* alpha, const float* beta,
                       const int32_t* path_len, const int32_t* path_nodes, int64_t n, int64_t H, int64_t dk,
                       int64_t dv, int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* W12_H */
