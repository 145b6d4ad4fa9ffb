/*
 * svp.h -- C ABI of the packed speculative-verification library (GB300, sm_103a).
 *
 * One step of block-diffusion speculative verification, as described in
 * "DScale: Scaling Block-Diffusion Speculative Decoding with Adaptive Verification"
 * (SIII-B tile routing, SIII-C Flat-buffer packer, SIII-D graph integration and Prefix
 * verifier) and the DFlash-Mini-Lab README (anchor + draft suffix, accept the exact
 * prefix, top-1/top-2 draft-logit margin):
 *
 *   N live requests; request i owns packed rows cu_slots[i] .. cu_slots[i+1]-1 of every
 *   per-row buffer; row cu_slots[i] + j holds candidate j (j = 0 is the anchor), and its
 *   target logits predict candidate j + 1.  k_i = cu_slots[i+1] - cu_slots[i] lies in
 *   [0, w] (0 = inactive).  Row j of request i attends to the request's ctx_len[i]
 *   context tokens and then to its own candidates 0..j (request-local causal mask).
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is DEVICE memory owned by the caller, unless it is marked
 *     "host".  The library never allocates, frees or synchronises; each call is
 *     enqueued on `stream` (a cudaStream_t; NULL = legacy default stream) and reads no
 *     device value back to the host, so it can be captured in a CUDA graph.
 *   - Metadata arrays (cu_slots, ctx_len, cu_ctx, block_table, cu_seqlens) are read on
 *     the device only.  Values that break the contract (cu_slots not non-decreasing,
 *     k_i > w, cu_slots[n] > m_cap, a context beyond its storage) never cause an
 *     out-of-bounds access: the affected request is skipped and a bit is set in the
 *     workspace status word (see svp_read_status).
 *   - Host-checkable errors (null pointers, head counts, unsupported head_dim or dtype,
 *     workspace too small, failed launch) are returned synchronously as svp_status and
 *     nothing is enqueued.
 *   - Workspaces: query the size, allocate it once, zero it once with
 *     svp_workspace_init, then reuse it for later calls of the same entry point.  The
 *     number of requests, m_cap and w may change from call to call (re-query the size:
 *     it grows with n); the attention workspace is tied to one head_dim and tile mode
 *     (a mismatch is reported as SVP_DEV_WORKSPACE and nothing is computed).  Kernels
 *     leave their counters and per-call scratch at zero when they finish (the attention
 *     kernel's partial slots sit at size-independent offsets before its counters), so a
 *     workspace serves later calls of any size.  Calls that share one workspace
 *     must not overlap on the GPU.  After SVP_DEV_TIMEOUT, zero the workspace again:
 *     until then an attention call on it computes nothing and reports SVP_DEV_WORKSPACE
 *     (its split-KV tickets may have been left mid-count).
 *   - Rows of out/lse that belong to no request (rows >= cu_slots[n], padding) are
 *     never written.
 *   - Kernels never trap.  Every wait inside a kernel is bounded; on expiry the kernel
 *     sets SVP_DEV_TIMEOUT in the status word and returns.
 *   - The DVL allocator, the row gathers, the verification attention, the margin /
 *     accept calls and the stochastic verifier's second pass are launched as
 *     programmatic dependents of the previous kernel on their stream: they may be
 *     scheduled while it finishes, but read nothing before it has completed, so the
 *     results are those of plain stream order (also inside a captured CUDA graph).
 */
#ifndef SVP_H_
#define SVP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SVP_VERSION 1

typedef enum {
    SVP_OK = 0,
    SVP_EINVAL = 1,          /* null pointer, negative size, hq % hkv != 0, ...        */
    SVP_EUNSUPPORTED = 2,    /* head_dim, dtype, page size or tile mode not supported  */
    SVP_EWORKSPACE = 3,      /* workspace missing or smaller than the queried size     */
    SVP_ECUDA = 4            /* a CUDA call or kernel launch failed                    */
} svp_status;

/* Bits of the device status word (svp_read_status). */
#define SVP_DEV_BAD_SLOTS   0x1   /* cu_slots decreasing, k_i > w, or cu_slots[n] > m_cap */
#define SVP_DEV_BAD_CONTEXT 0x2   /* ctx_len < 0 or a context beyond its storage          */
#define SVP_DEV_TIMEOUT     0x4   /* a bounded in-kernel wait expired                    */
#define SVP_DEV_WORKSPACE   0x8   /* workspace last used with another head_dim or tile mode:
                                     nothing was computed; run svp_workspace_init first     */

typedef enum { SVP_F32 = 0, SVP_BF16 = 1 } svp_dtype;

/* Query-row tile of the verification attention (DScale SIII-B, path-aware tile router). */
typedef enum {
    SVP_TILE_AUTO = 0,      /* w <= 16: SHORT, otherwise WIDE                                */
    SVP_TILE_SHORT = 1,     /* candidate-width tile: the G query heads sharing one KV head
                               are packed into one tile of G*min(w, 128/G) rows; split-KV   */
    SVP_TILE_FIXED128 = 2,  /* contrast: one query head per 128-row tile, one block per
                               (request, head), no split (the prior-art native tile)       */
    SVP_TILE_WIDE = 3,      /* prefill-style 128-row tile of one head, split-KV            */
    SVP_TILE_SHORT_UNPACKED = 4  /* contrast: the candidate-width tile without GQA packing:
                               one query head per tile of min(w, 128) rows (96 at d = 256),
                               so each KV head is streamed once per query head; split-KV;
                               d = 128 or 256                                              */
} svp_tile_mode;

/* GQA head layout.  Query head h reads KV head h / (hq / hkv). */
typedef struct {
    int32_t hq;       /* query heads                                              */
    int32_t hkv;      /* key/value heads; hq % hkv == 0                           */
    int32_t d;        /* head_dim: 64, 128 or 256                                  */
    float scale;      /* softmax scale; 0 selects 1/sqrt(d)                       */
} svp_heads;

/* Committed-context KV storage of the requests (DScale SIII-D: historyKV). */
typedef struct {
    int32_t paged;              /* 0: contiguous varlen, 1: paged                          */
    const void *k;              /* contiguous: [total_tokens, hkv, d]; paged: page pool   */
    const void *v;              /* same layout as k                                        */
    const int64_t *cu_ctx;      /* contiguous: [n] first token row of request i            */
    int64_t total_tokens;       /* contiguous: rows in k/v (a host-known allocation size) */
    const int32_t *block_table; /* paged: [n, max_pages] page ids, row-major              */
    int32_t max_pages;          /* paged: columns of block_table                          */
    int32_t page_size;          /* paged: tokens per page; must be 16                      */
    int64_t num_pages;          /* paged: pages in the pool                                */
    int64_t stride_page;        /* paged: element strides of the pool; the last dim (d)   */
    int64_t stride_head;        /*   is contiguous.  [pages][hkv][16][d] and              */
    int64_t stride_tok;         /*   [pages][16][hkv][d] are both expressible.            */
} svp_kv;

/* Library version and status text. */
int32_t svp_version(void);
const char *svp_status_string(svp_status s);

/* Zero a workspace (once, after allocating it).  Enqueued on `stream`. */
svp_status svp_workspace_init(void *ws, size_t ws_bytes, void *stream);

/* Copy the device status word of a workspace into *status (host) and clear it.
 * This is the one call that synchronises `stream`. */
svp_status svp_read_status(void *ws, void *stream, int32_t *status);

/* ---------------------------------------------------------------------------------- */
/* Verification attention over packed, ragged candidate prefixes.                      */
/* DScale SIII-B (short verify tile sized to the candidate width; grid over requests,   */
/* heads and query tiles), SIII-C (packed rows, offsets), SIII-D (rows read             */
/* offset_i + j with request-local causal masking over the supplied KV refs).           */

/* Workspace bytes for svp_verify_attn_packed(_ex) with these sizes (host). */
svp_status svp_verify_attn_workspace_size(int32_t n, int32_t m_cap, int32_t w,
                                          const svp_heads *heads, svp_dtype dtype,
                                          int32_t tile_mode, size_t *bytes);

/*
 * q      [m_cap, hq, d]   queries of the packed candidate rows
 * k_new  [m_cap, hkv, d]  keys of the packed candidate rows (same row map as q)
 * v_new  [m_cap, hkv, d]  values of the packed candidate rows
 * kv     host struct describing the committed context (contiguous or paged)
 * ctx_len  [n] int32      context tokens of each request
 * cu_slots [n+1] int32    packed row offsets (exclusive prefix sums of k_i)
 * n, m_cap, w             requests, packed row capacity, largest allowed k_i (host)
 * heads, dtype            host; q/k/v/kv/out share dtype (SVP_F32 or SVP_BF16)
 * out    [m_cap, hq, d]   softmax(scale q K^T) V per row, in dtype
 * lse    [m_cap, hq] fp32 natural-log softmax normaliser per row (may be NULL)
 * ws     workspace of at least svp_verify_attn_workspace_size bytes
 * dtype SVP_F32 runs an fp32 FFMA kernel; SVP_BF16 runs the tcgen05/TMA kernel with
 * fp32 accumulation.  All of q, k_new, v_new, kv->k, kv->v, out must be 16-byte aligned.
 */
svp_status svp_verify_attn_packed(const void *q, const void *k_new, const void *v_new,
                                  const svp_kv *kv, const int32_t *ctx_len,
                                  const int32_t *cu_slots, int32_t n, int32_t m_cap,
                                  int32_t w, const svp_heads *heads, svp_dtype dtype,
                                  void *out, float *lse, void *ws, size_t ws_bytes,
                                  void *stream);

/* As svp_verify_attn_packed, with an explicit svp_tile_mode (SVP_BF16 only for modes
 * other than AUTO). */
svp_status svp_verify_attn_packed_ex(const void *q, const void *k_new, const void *v_new,
                                     const svp_kv *kv, const int32_t *ctx_len,
                                     const int32_t *cu_slots, int32_t n, int32_t m_cap,
                                     int32_t w, const svp_heads *heads, svp_dtype dtype,
                                     int32_t tile_mode, void *out, float *lse, void *ws,
                                     size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------------- */
/* Wide-tile causal prefill attention (the contrast path of DScale SIII-B: prefill keeps */
/* the hardware-selected 128-row tile for KV reuse).                                    */

svp_status svp_prefill_attn_workspace_size(int32_t n, int32_t max_s,
                                           const svp_heads *heads, svp_dtype dtype,
                                           size_t *bytes);

/*
 * q [total_s, hq, d], k, v [total_s, hkv, d]  sequences packed by cu_seqlens
 * cu_seqlens [n+1] int32 (device)  row offsets; sequence lengths <= max_s (host bound)
 * causal   must be 1 (SVP_EUNSUPPORTED otherwise)
 * out [total_s, hq, d] (dtype), lse [total_s, hq] fp32 (may be NULL)
 * SVP_BF16 only; 0 <= total_s < 2^31 (SVP_EINVAL otherwise).
 * Routing: d = 128 with an even number of query heads per KV head, 1 <= n <= 16 and
 *   max_s <= 32768 run the dedicated kernel (q, k, v, out 16-byte aligned, else
 *   SVP_EINVAL; it uses only the workspace header); every other shape runs the general
 *   128-row attention kernel.  A sequence whose offsets run backwards, leave the buffer or
 *   exceed max_s is skipped and sets SVP_DEV_BAD_SLOTS in the workspace status word.
 */
svp_status svp_prefill_attn(const void *q, const void *k, const void *v,
                            const int32_t *cu_seqlens, int32_t n, int32_t max_s,
                            int64_t total_s, int32_t causal, const svp_heads *heads,
                            svp_dtype dtype, void *out, float *lse, void *ws,
                            size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------------- */
/* Row top-1 / top-2 / margin over vocabulary logits (DFlash-Mini-Lab, DFlash7-ACT     */
/* margin; DScale SII-B, Fig. 4 Top1-Top2 logit gap).                                  */
/*   top1_idx = smallest index of the row maximum; top1 = the maximum;                  */
/*   top2 = second element of the row sorted descending as a multiset (a repeated       */
/*   maximum gives top2 == top1); margin = top1 - top2 in fp32.  NaN is not supported.   */

svp_status svp_draft_margin_workspace_size(int32_t rows, int32_t vocab, size_t *bytes);

/*
 * logits [rows, row_stride] (dtype), vocab <= row_stride, vocab >= 2; rows may be 0.
 * Outputs [rows] each; any output pointer may be NULL.
 */
svp_status svp_draft_margin(const void *logits, int64_t row_stride, int32_t rows,
                            int32_t vocab, svp_dtype dtype, int32_t *top1_idx,
                            float *top1, float *top2, float *margin, void *ws,
                            size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------------- */
/* Greedy prefix acceptance (DScale SIII-D, Prefix verifier at temperature 0;           */
/* DFlash-Mini-Lab "accept exact prefix").                                              */
/*   a_i = largest a <= k_i - 1 with tokens[off_i + j] == target_argmax[off_i + j - 1]   */
/*   for all 1 <= j <= a; accept_len[i] = 1 + a_i (the anchor counts);                   */
/*   next_token[i] = target_argmax[off_i + a_i] (row off_i + a_i supplies the successor).*/
/*   k_i = 0: accept_len = 0, next_token = -1.                                          */

/*
 * target_argmax [m_cap] int32, tokens [m_cap] int32 (row off_i = anchor, off_i + j =
 * draft j), cu_slots [n+1]; outputs accept_len [n], next_token [n].  No workspace.
 */
svp_status svp_greedy_accept(const int32_t *target_argmax, const int32_t *tokens,
                             const int32_t *cu_slots, int32_t n, int32_t m_cap,
                             int32_t *accept_len, int32_t *next_token, void *stream);

/* Fused: svp_draft_margin over the packed target-logit rows, then svp_greedy_accept,
 * in one launch.  Rows >= cu_slots[n] are not read.  m_cap rows of logits. */
svp_status svp_margin_accept_workspace_size(int32_t n, int32_t m_cap, int32_t vocab,
                                            size_t *bytes);

/*
 * logits [m_cap, row_stride] (dtype F32 or BF16, else SVP_EUNSUPPORTED): packed target
 * rows, row off_i + j the target distribution after slot j of request i; 2 <= vocab <=
 * row_stride.  tokens [m_cap] int32 (row off_i = anchor, off_i + j = draft j) and
 * cu_slots [n+1] as for svp_greedy_accept.  Outputs: top1_idx / top1 / top2 / margin
 * [m_cap] as svp_draft_margin for the live rows r < cu_slots[n] (other rows are neither
 * read nor written; any of the four pointers may be NULL); accept_len / next_token [n]
 * as svp_greedy_accept (required).  ws: at least svp_margin_accept_workspace_size bytes,
 * zeroed once by svp_workspace_init; every call leaves it zeroed.  A NULL cu_slots,
 * tokens, accept_len or next_token, n < 0, vocab < 2 or row_stride < vocab returns
 * SVP_EINVAL; a missing or small workspace SVP_EWORKSPACE; nothing is enqueued then.
 * cu_slots that break the contract on the device (not starting at 0, decreasing, or
 * cu_slots[n] > m_cap): no logit is read, no output is written and SVP_DEV_BAD_SLOTS is
 * set in the status word.
 */
svp_status svp_margin_accept(const void *logits, int64_t row_stride, int32_t m_cap,
                             int32_t vocab, svp_dtype dtype, const int32_t *tokens,
                             const int32_t *cu_slots, int32_t n, int32_t *top1_idx,
                             float *top1, float *top2, float *margin, int32_t *accept_len,
                             int32_t *next_token, void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------------- */
/* Allocation-free variant of svp_margin_accept.  The pages describe no such call; it   */
/* exists for callers that cannot allocate device memory: code running inside a memory  */
/* pool or host framework that owns every device allocation, and paths where a          */
/* cudaMalloc (and the synchronisation it may cause) is not acceptable.                 */
/*                                                                                      */
/* Arguments, outputs and results are those of svp_margin_accept, without the workspace.*/
/* The scratch is a fixed 2 MiB array inside the library, held by every GPU that loads  */
/* the library until the process exits; sizes whose workspace                           */
/* (svp_margin_accept_workspace_size) exceeds 2 MiB return SVP_EWORKSPACE and nothing   */
/* is enqueued.  The first call on each device (with that device current) looks up the  */
/* array's device address and clears it once on `stream`, waiting for that stream       */
/* (cudaGetSymbolAddress, cudaMemsetAsync, cudaStreamSynchronize; no allocation), so    */
/* make that first call before capturing any stream.  All calls share                   */
/* the one array: calls that overlap on the GPU (other streams, other host threads)     */
/* race and must be serialised by the caller.  The kernel leaves the array zeroed.      */
/* Device-side metadata errors are not reported through a status word in this variant:  */
/* invalid cu_slots leave every row and request unwritten.  Allocates nothing.          */
svp_status svp_margin_accept_noalloc(const void *logits, int64_t row_stride, int32_t m_cap,
                                     int32_t vocab, svp_dtype dtype, const int32_t *tokens,
                                     const int32_t *cu_slots, int32_t n, int32_t *top1_idx,
                                     float *top1, float *top2, float *margin,
                                     int32_t *accept_len, int32_t *next_token, void *stream);

/* ---------------------------------------------------------------------------------- */
/* DVL budget allocator and flat-buffer packer (DScale SIII-C, Budget allocator and     */
/* Flat-buffer packer, Algorithm 1, Fig. 6), one thread block, no host round trip.       */
/*   q[i,0] = 1 (anchor); q[i,j] = min(q[i,j-1], scores[i,j-1]) for j = 1..w-1.          */
/*   k0_i = clip(rint(sum_{j=1}^{w-1} q[i,j]), 1, w) for live requests (the sum in fp32, */
/*   positions in order; rint = nearest, ties to even), 0 for the others.               */
/*   budget = budget_per_req * n_live; delta = budget - sum(k0).  delta > 0: the delta   */
/*   best next slots q[i,k_i] are added (a request grows up to w); delta < 0: the -delta  */
/*   worst last slots q[i,k_i-1] are removed (never the anchor).  Ties go to the lowest   */
/*   request index.  This equals the page's one-slot-at-a-time loop because q is         */
/*   non-increasing along a request.  Growing stops when all live requests reach w,      */
/*   shrinking when all are at 1.                                                       */
/*   cu_slots = exclusive prefix sums of k (inactive requests: k = 0, offset = the end). */
/*   Packed row cu_slots[i] + j of tokens / positions / kv_refs = field[i, j] for j < k_i;*/
/*   rows cu_slots[n_bs] .. m_cap-1 hold fill_token / fill_pos / fill_ref.               */

/*
 * scores [n_bs, w-1] fp32: acceptance scores of draft positions 1..w-1 (finite; NaN not
 * supported).  n_live: device int32 scalar (requests 0..n_live-1 are live), or NULL for
 * all n_bs.  tokens / positions / kv_refs [n_bs, w] int32, each may be NULL (then the
 * matching packed output is all fill, or not written if its pointer is NULL too).
 * Outputs: k_init [n_bs] (may be NULL), k_out [n_bs], cu_slots [n_bs + 1],
 * tokens_packed / pos_packed / ref_packed [m_cap] (each may be NULL), n_adjust (device
 * int32 scalar, slots added or removed; may be NULL).  ws: at least 256 bytes, zeroed
 * once (svp_workspace_init); n_live outside [0, n_bs] or budget > m_cap sets
 * SVP_DEV_BAD_SLOTS and treats every request as inactive.
 * Limits: 1 <= n_bs <= 2048, 2 <= w <= 16, 1 <= budget_per_req <= w, m_cap >= 1
 * (SVP_EINVAL / SVP_EUNSUPPORTED otherwise).
 */
svp_status svp_dvl_allocate_pack(const float *scores, int32_t n_bs, int32_t w,
                                 const int32_t *n_live, int32_t budget_per_req,
                                 const int32_t *tokens, const int32_t *positions,
                                 const int32_t *kv_refs, int32_t m_cap, int32_t fill_token,
                                 int32_t fill_pos, int32_t fill_ref, int32_t *k_init,
                                 int32_t *k_out, int32_t *cu_slots, int32_t *tokens_packed,
                                 int32_t *pos_packed, int32_t *ref_packed, int32_t *n_adjust,
                                 void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------------- */
/* Row-mapped packing of a wide per-row field (DScale SIII-C, Flat-buffer packer: every  */
/* field is packed with the same row mapping; SIII-D, fixed-address workspace).          */
/*   dst row r = src row idx[r] for 0 <= idx[r] < src_rows, else zeros; r < rows.       */

/*
 * src [src_rows, row_bytes] and dst [rows, row_bytes] device buffers, 16-byte aligned,
 * row_bytes >= 16 (SVP_EINVAL otherwise, as for NULL pointers or negative counts) and a
 * multiple of 16 (SVP_EUNSUPPORTED otherwise, as for unaligned buffers); idx [rows] int32
 * (e.g. the packed KV references of svp_dvl_allocate_pack).  No workspace.
 */
svp_status svp_gather_rows(const void *src, int64_t src_rows, int64_t row_bytes,
                           const int32_t *idx, int32_t rows, void *dst, void *stream);

/*
 * The same for up to SVP_GATHER_MAX_FIELDS fields that share one row map, in one launch
 * (a step packs its query, key, value and logit rows together).  fields: a HOST array of
 * n_fields descriptors (1 <= n_fields <= SVP_GATHER_MAX_FIELDS), read during the call and
 * not retained, SVP_EINVAL for a count outside that range; each src / dst pair follows
 * the rules of svp_gather_rows (16-byte aligned, row_bytes >= 16 and a multiple of 16);
 * dst of field f holds [rows, row_bytes_f].  idx [rows] int32, shared.  No workspace.
 */
#define SVP_GATHER_MAX_FIELDS 8
typedef struct {
    const void *src;    /* [src_rows, row_bytes] */
    int64_t src_rows;
    int64_t row_bytes;
    void *dst;          /* [rows, row_bytes] */
} svp_gather_field;

svp_status svp_gather_rows_multi(const svp_gather_field *fields, int32_t n_fields,
                                 const int32_t *idx, int32_t rows, void *stream);

/* ---------------------------------------------------------------------------------- */
/* Stochastic prefix verifier, temperature T > 0 (DScale SIII-D, Prefix verifier).       */
/*   P_r = softmax(logits[r] / T).  Candidate j of request i (tokens[off_i + j],          */
/*   1 <= j < k_i) is accepted iff u_accept[off_i + j] < P_{off_i+j-1}(candidate), in     */
/*   order; the first rejection ends the prefix.  a_i = accepted candidates;              */
/*   accept_len[i] = 1 + a_i.  The successor next_token[i] is the smallest token y with   */
/*   sum_{y' <= y} w(y') > u_next[i] * sum w, over row off_i + a_i with weights          */
/*   w = P_{off_i+a_i}, the rejected candidate's weight set to 0 (none removed when every */
/*   candidate passed).  k_i = 0: accept_len 0, next_token -1.  The row softmax is       */
/*   evaluated in fp32 (exp2 of scaled differences), so a draw within rounding of a      */
/*   boundary may fall on either side.                                                    */

svp_status svp_stochastic_accept_workspace_size(int32_t m_cap, int32_t vocab, size_t *bytes);

/*
 * logits [m_cap, row_stride] (dtype), vocab <= row_stride; tokens [m_cap] int32;
 * cu_slots [n+1]; u_accept [m_cap] fp32 and u_next [n] fp32, uniform draws in [0, 1)
 * supplied by the caller; outputs accept_len [n], next_token [n] int32 and p_draft [m_cap]
 * (the acceptance probability of each tested candidate; may be NULL).  Rows >=
 * cu_slots[n] are not read.  Invalid cu_slots (cu_slots[0] != 0, a decrease, or
 * cu_slots[n] > m_cap) set SVP_DEV_BAD_SLOTS: no row is read and every request gets
 * accept_len 0 and next_token -1.  ws zeroed once (svp_workspace_init); the kernels leave
 * it zeroed (tickets, row and chunk statistics), so it can serve later calls with other
 * m_cap and vocabularies.
 */
svp_status svp_stochastic_accept(const void *logits, int64_t row_stride, int32_t m_cap,
                                 int32_t vocab, svp_dtype dtype, const int32_t *tokens,
                                 const int32_t *cu_slots, int32_t n, float temperature,
                                 const float *u_accept, const float *u_next,
                                 int32_t *accept_len, int32_t *next_token, float *p_draft,
                                 void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------------- */
/* Draft-signal features (DScale SIII-C, Acceptance predictor).  For every row of draft  */
/* logits, 18 fp32 values: [0] the highest logit; [1..15] its gaps to ranks 2..16 (rank r */
/* = r-th element of the row sorted descending as a multiset, gap = top1 - rank_r in     */
/* fp32); [16] the top token's log-probability (top1 - log-sum-exp of the row); [17] the  */
/* entropy -sum p ln p of softmax(row).  Sums are fp32.                                    */

svp_status svp_draft_features_workspace_size(int32_t rows, int32_t vocab, size_t *bytes);

/*
 * logits [rows, row_stride] (dtype), 16 <= vocab <= row_stride; features [rows, 18] fp32.
 * ws zeroed once (svp_workspace_init); the kernel leaves it zeroed (tickets and partial
 * lists), so it can serve later calls with other row counts and vocabularies.
 */
svp_status svp_draft_features(const void *logits, int64_t row_stride, int32_t rows,
                              int32_t vocab, svp_dtype dtype, float *features, void *ws,
                              size_t ws_bytes, void *stream);

/* ACT truncation (DFlash-Mini-Lab README, DFlash7-ACT): the draft suffix of request i is  */
/* cut before its first position j (1 <= j < w) whose margin is below `threshold`;       */
/* k_out[i] = 1 + the number of positions kept (threshold 0 keeps the full block w).      */
/* margins: element ((i * (w-1) + j - 1) * stride) is the margin of position j of request */
/* i (stride = 1 for svp_draft_margin's margin array, 18 with features + 1).  No         */
/* workspace.                                                                             */
svp_status svp_act_truncate(const float *margins, int64_t stride, int32_t n, int32_t w,
                            float threshold, int32_t *k_out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SVP_H_ */
