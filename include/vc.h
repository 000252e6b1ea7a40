/*
 * vc.h -- C ABI of the VeriCache attention-step library (libvc.so, sm_103a).
 *
 * VeriCache ("VeriCache: Making Lossy KV Compression Exact", section "The
 * Core Idea") drafts x tokens autoregressively with a lossy compressed KV
 * cache (KV_comp), checks them in ONE pass over the full cache (KV_full)
 * that yields x + 1 greedy predictions, and emits the longest matching
 * prefix plus the verifier's correction (or bonus) token, so the output is
 * identical to greedy decoding with the full cache.  This library holds the
 * four data-parallel operations of that attention step:
 *
 *   vc_compress     KV_full -> KV_comp: gather by a kept-index list and/or
 *                   asymmetric 2/3/4-bit group quantisation ("VeriCache
 *                   Guide", "The Uniform Compressor Interface": token
 *                   eviction and low-bit quantisation behind one compress()).
 *   vc_draft_attn   one decode query per request over KV_comp (the drafting
 *                   step, "The Core Idea" items 1-2; memory-bandwidth bound,
 *                   "Verifying Without Giving Back the Speedup").
 *   vc_verify_attn  the drafted block's queries over KV_full, causal inside
 *                   the block ("The Core Idea" items 3-5).
 *   vc_accept       LM-head argmax over the verifier's rows, longest
 *                   matching prefix + correction / bonus (the accept step
 *                   and its worked example in "The Core Idea").
 * plus the host-to-device staging of KV_full on a side stream ("VeriCache
 * Guide", the dual-stream engine and "Best Practice 2: pinned memory") and a
 * single launch mixing drafting and verifying requests (cross-resource
 * staggering, "Verifying Without Giving Back the Speedup", Figure 2).
 *
 * Conventions
 *  - Every pointer argument named as "device" must point to device memory of
 *    the current device; "host" pointers to host memory.  The caller owns and
 *    allocates every buffer, including workspaces (sizes from the
 *    vc_*_workspace_bytes queries).  The library allocates nothing.
 *  - Every compute call is asynchronous on `stream` (a cudaStream_t; NULL is
 *    the legacy default stream).  Argument errors are returned synchronously
 *    (nothing is launched); a failed launch returns VC_ERR_CUDA.  Errors in
 *    device-resident data (a page id or kept index out of range, a wait that
 *    timed out) are written to the optional device word `dev_status` (first
 *    error wins; the caller zeroes it and reads it after synchronising); the
 *    offending element is skipped, never read or written out of bounds.
 *  - A call with batch 0 (for vc_compress also one with max_kept 0) checks
 *    its formats and sizes, launches nothing and returns VC_OK.  Pointers to
 *    per-request data (queries, outputs, pools, block tables, lengths, kept
 *    lists, hidden rows, drafts, uniforms) may then be NULL, as the data
 *    pointer of a zero-size tensor is.
 *  - No C++ exception crosses this interface.
 *
 * Paged KV layout (page = 16 tokens, separate K and V pools)
 *  - A pool is an array of pages; page p starts at byte p * vc_page_bytes().
 *    Inside a page, kv head h owns a contiguous block of vc_head_block_bytes()
 *    bytes starting at h * vc_head_block_bytes(); token slot s = position % 16.
 *  - bits == 16 (bf16, KV_full or token-drop KV_comp):
 *      block = bf16 [16][head_dim]                              (32 * D bytes)
 *  - bits in {2, 3, 4} (quantised KV_comp), D = head_dim (64, 128 or 256),
 *    G = D / 32 groups.  A head block holds, per token slot s (0..15) and
 *    32-channel group, the codes of the slot's D channels and an fp16 scale
 *    and zero (2 * D * (bits + 1) bytes in all).
 *    Logical content (what vc_comp_block_decode returns and the quantiser
 *    defines):
 *      codes  uint8 [16][D * bits / 8]   slot s, channel i at bits
 *                                        [bits*i, bits*i + bits) of the slot's
 *                                        little-endian byte string
 *      scales fp16  [16][G]              per slot and 32-channel group
 *      zeros  fp16  [16][G]
 *    Stored order (what the pools hold; chosen so that the draft kernel turns
 *    packed words into mma.sync fragments with one mask, sometimes one
 *    shift, per operand register):
 *      bytes [0, 16 D bits / 8)       the code region; K and V blocks place
 *                                     codes differently (below)
 *      then fp16 scales, then fp16 zeros, 16 G values each:
 *        K block: [16 slots][G], as in the logical content
 *        V block: [4][G][4], entry [t][g][i] = slot 2t + (i & 1) + 8 (i >> 1)
 *    Code bit offsets from the start of the code region (channel c, slot s;
 *    for bits 3 "low" = the code's low two bits, "high" = its top bit; every
 *    field lies inside one little-endian 32-bit word):
 *      K: ks = c / 16, t = (c / 4) % 4, e = c % 4, r = 2 ks + e / 2, h = e % 2
 *        bits 2: s 2D + t D/2 + 32 (r / 8) + 16 h + 2 (r % 8)
 *        bits 4: s 4D + t D   + 32 (r / 4) + 16 h + 4 (r % 4)
 *        bits 3 low:  s 3D + t D/2 + 32 (r / 8) + 16 h + 2 (r % 8)
 *        bits 3 high: with u = r / 8, j = r % 8, S = 2 (u % 2) + j / 4,
 *          beta = 2 (j % 4) + {0, 1, 8, 9}[S]:
 *          D = 64: s 3D + 2D + 16 t + 8 h + beta;
 *          else:   s 3D + 2D + t D/4 + 32 (u / 2) + 16 h + beta
 *      V: g = c % 8, w = (c / 8) % 2, m = c / 16, t = (s / 2) % 4,
 *         hi = s / 8, h = s % 2, R = 4 g + t
 *        bits 4: 32 (R D/16 + m) + 16 h + 8 w + 4 hi
 *        bits 2 and bits 3 low, with u = m / 2, n = m % 2:
 *                32 (R D/32 + u) + 16 h + 8 n + 4 w + 2 hi
 *        bits 3 high: j = 2 w + hi, S = 2 (u % 2) + n,
 *                32 D + 32 (R D/64 + u / 2) + 16 h + 2 j + {0, 1, 8, 9}[S]
 *    vc_comp_block_decode / vc_comp_block_encode (host functions, below)
 *    convert one stored head block to and from the logical content.
 *    Quantisation of one group x[0..31] (bf16 values, fp32 arithmetic, every
 *    operation rounded to nearest even, no contraction):
 *      mn = min x (a -0 minimum is stored as +0), mx = max x
 *      scale = fp16(sat((mx - mn) / (2^bits - 1))), zero = fp16(sat(mn))
 *      code_i = 0 if scale == 0 else clamp(rint((x_i - zero) / scale), 0, 2^bits-1)
 *    where sat() clamps to [-65504, 65504].  Dequantised value: scale * code + zero.
 *  - block_table: device int32 [batch][max_blocks]; entry j of row b is the
 *    page holding positions [16 j, 16 j + 16) of request b.
 *  - seq_lens: device int32 [batch]; tokens present for each request.
 */
#ifndef VC_H
#define VC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define VC_API __attribute__((visibility("default")))
#else
#define VC_API
#endif

#define VC_PAGE_TOKENS 16
#define VC_GROUP 32
#define VC_MAX_HEAD_DIM 256
#define VC_MAX_GQA_GROUP 8
#define VC_MAX_VERIFY_QUERIES 64
#define VC_STATIC_SCRATCH_BYTES (8u << 20)

typedef enum {
    VC_OK = 0,
    VC_ERR_INVALID_ARG = 1, /* null pointer, negative size, mismatched formats  */
    VC_ERR_UNSUPPORTED = 2, /* bits / head_dim / GQA group outside the support  */
    VC_ERR_BAD_INDEX = 3,   /* (device status) page id or kept index out of range */
    VC_ERR_CUDA = 4,        /* a CUDA launch or copy failed                       */
    VC_ERR_STAGING = 5,     /* staging source not in page-locked host memory      */
    VC_ERR_TIMEOUT = 6,     /* (device status) a bounded wait gave up             */
    VC_ERR_WORKSPACE = 7    /* workspace null or smaller than the size query      */
} vc_status;

typedef void *vc_stream_t; /* cudaStream_t */
typedef void *vc_event_t;  /* cudaEvent_t  */

typedef struct {
    int32_t num_kv_heads; /* >= 1                                   */
    int32_t head_dim;     /* multiple of 32, 32..256 (draft / verify: 64 or 128) */
    int32_t bits;         /* 16 (bf16), 4, 3 or 2                    */
} vc_kv_format;

typedef struct {
    void *k_pages;               /* device: K page pool                       */
    void *v_pages;               /* device: V page pool                       */
    int64_t num_pages;           /* pages in each pool (page ids < this)      */
    const int32_t *block_table;  /* device int32 [batch][max_blocks]          */
    const int32_t *seq_lens;     /* device int32 [batch]                      */
    int32_t batch;
    int32_t max_blocks;
    vc_kv_format fmt;
} vc_paged_kv;

/* Bytes of one page (all kv heads) and of one kv head's block in a page. */
VC_API size_t vc_page_bytes(const vc_kv_format *fmt);
VC_API size_t vc_head_block_bytes(const vc_kv_format *fmt);

/*
 * vc_comp_block_decode / vc_comp_block_encode -- host conversions of one
 * quantised KV_comp head block (vc_head_block_bytes(fmt) bytes, bits 2, 3 or
 * 4) between its stored order and the logical content described in the
 * layout notes above.  kind: 0 = a block of the K pool, 1 = of the V pool
 * (they order codes and parameters differently).  All pointers are host
 * memory owned by the caller: codes uint8 [16][D * bits / 8] (little-endian
 * bit string per slot), scales and zeros fp16 bits [16][D / 32].  encode
 * writes every byte of the block; bytes of a code's unused bit positions
 * are 0.  VC_ERR_INVALID_ARG for a null pointer, another kind or a format
 * other than bits 2 / 3 / 4 with head_dim 64, 128 or 256.  No CUDA call.
 */
VC_API vc_status vc_comp_block_decode(const vc_kv_format *fmt, int32_t kind, const void *block, uint8_t *codes,
                                      uint16_t *scales, uint16_t *zeros);
VC_API vc_status vc_comp_block_encode(const vc_kv_format *fmt, int32_t kind, const uint8_t *codes,
                                      const uint16_t *scales, const uint16_t *zeros, void *block);

/*
 * vc_select_kept -- the kept-index list of a token-drop KV_comp ("VeriCache
 * Guide", the compressor class of "Implementing VeriCache in Python and
 * PyTorch": tokens ranked by the norm of their key over head_dim averaged
 * over the heads, the top ones kept in position order).
 *  full          bits == 16 cache; seq_lens[b] = n_b positions of request b.
 *  scores        device fp32 [batch][score_stride] importance per position,
 *                or NULL: computed from full's K pages (head_dim 64 or 128)
 *                as, per kv head, sqrt of the sum of squares (one fused
 *                multiply-add per channel in increasing order, correctly
 *                rounded square root), added over heads in increasing order
 *                and divided by the head count.  Positions >= score_stride
 *                are not considered (n_b is capped to it).
 *  kept_offsets  device int32 [batch + 1]: request b's list goes to
 *                kept_idx[kept_offsets[b] .. kept_offsets[b + 1]); its
 *                length keep_b must equal s + r + top with s = min(sink, n),
 *                r = min(recent, n - s), top = min(n - s - r, keep_b - s - r)
 *                (else VC_ERR_INVALID_ARG in dev_status, nothing written).
 *  sink, recent  host: positions [0, s) and [n - r, n) are always kept.
 *  kept_idx      device int32 out: ascending positions; the middle positions
 *                are the `top` of highest score, equal scores by lower
 *                position.
 *  workspace     device, vc_select_workspace_bytes(batch, score_stride)
 *                bytes when scores == NULL (may be NULL otherwise).
 */
VC_API size_t vc_select_workspace_bytes(int32_t batch, int32_t score_stride);
VC_API vc_status vc_select_kept(const vc_paged_kv *full, const float *scores, int32_t score_stride,
                                const int32_t *kept_offsets, int32_t sink, int32_t recent, int32_t *kept_idx,
                                void *workspace, size_t workspace_bytes, int32_t *dev_status,
                                vc_stream_t stream);

/*
 * vc_compress -- KV_comp entries from KV_full ("VeriCache Guide", "The
 * Uniform Compressor Interface"; the guide's compressor gathers K and V with
 * one sorted index list shared by all heads).
 *  full          bits == 16 cache; positions read must be < full->seq_lens[b].
 *  kept_offsets  device int32 [batch + 1], CSR offsets into kept_idx.
 *  kept_idx      device int32 positions in KV_full, in the order they are
 *                stored (ascending for a token-drop list).
 *  comp_start    device int32 [batch] or NULL (= 0): slot of KV_comp where
 *                request b's first kept entry goes.  Appending the drafted
 *                tokens' K/V passes the current KV_comp length here.
 *  max_kept      host: upper bound of any request's kept count (grid size).
 *  comp          bits in {2, 3, 4, 16}; same num_kv_heads / head_dim as full;
 *                slots comp_start[b] + j must be covered by its block table.
 *                comp->seq_lens is not read or written (the caller sets it).
 * Entry (b, j) is written for every kv head: bits 16 copies the bf16 rows,
 * bits < 16 quantises K and V rows with the rule in the layout notes above.
 */
VC_API vc_status vc_compress(const vc_paged_kv *full, const int32_t *kept_offsets,
                      const int32_t *kept_idx, const int32_t *comp_start, int32_t max_kept,
                      const vc_paged_kv *comp, int32_t *dev_status, vc_stream_t stream);

/*
 * vc_draft_attn -- one decode query per query head over KV_comp:
 *   out[b][h] = sum_t softmax_t(scale * <q[b][h], k_t>) v_t
 * over the comp->seq_lens[b] entries of request b, k_t / v_t the dequantised
 * rows of kv head h / (num_q_heads / num_kv_heads).  Split over context
 * chunks (partials in `workspace`), then combined by a second launch.
 *  q            device bf16 [batch][num_q_heads][head_dim]
 *  out          device fp32 [batch][num_q_heads][head_dim]
 *  max_seq_len  host: bound of every comp->seq_lens[b] (grid size)
 *  workspace    device, >= vc_draft_workspace_bytes(comp, num_q_heads,
 *               max_seq_len) bytes (0 when the format is unsupported)
 * Requires num_q_heads / num_kv_heads <= 8, head_dim in {64, 128}.  A request
 * with seq_len 0 gets zeros.  q must be finite and, for bits < 16, within the
 * fp16 range (|q| <= 65504).  A block-table entry out of range is reported
 * (VC_ERR_BAD_INDEX in dev_status); that request's output is then finite but
 * void.
 */
VC_API size_t vc_draft_workspace_bytes(const vc_paged_kv *comp, int32_t num_q_heads,
                                int32_t max_seq_len);
VC_API vc_status vc_draft_attn(const void *q, int32_t num_q_heads, const vc_paged_kv *comp,
                        float softmax_scale, float *out, int32_t max_seq_len, void *workspace,
                        size_t workspace_bytes, int32_t *dev_status, vc_stream_t stream);

/*
 * vc_draft_step -- one drafting step: each request's new entry (the K and V
 * rows of the token just produced, "The Core Idea" item 2: each drafted
 * token's state is appended to KV_comp) is written into KV_comp at position
 * slot[b] in comp's format (quantised exactly as vc_compress would, or
 * copied for bits == 16), then the draft attention of vc_draft_attn runs
 * over the comp->seq_lens[b] entries, which should include slot[b].  One
 * launch: the block that reads slot[b]'s page writes the entry first.
 *  k_new, v_new  device bf16 [batch][num_kv_heads][head_dim]
 *  slot          device int32 [batch]; 0 <= slot[b] < seq_lens[b] (else
 *                VC_ERR_INVALID_ARG in dev_status and nothing written for b)
 * Other arguments and the workspace are vc_draft_attn's.  The KV_comp bytes
 * equal those of vc_compress appending the same rows at the same position.
 */
VC_API vc_status vc_draft_step(const void *q, int32_t num_q_heads, const vc_paged_kv *comp, const void *k_new,
                               const void *v_new, const int32_t *slot, float softmax_scale, float *out,
                               int32_t max_seq_len, void *workspace, size_t workspace_bytes, int32_t *dev_status,
                               vc_stream_t stream);

/*
 * vc_draft_attn_static -- vc_draft_attn without a caller workspace.
 * The pages have no counterpart of this entry point.  It is for callers that
 * cannot allocate device memory where they call the library: a plugin run by
 * a host engine that owns every device allocation and hands out no scratch
 * buffer, or a latency-critical path that must not call cudaMalloc (which can
 * synchronise the device).  Arguments and result are those of vc_draft_attn
 * without the workspace; the caller still passes q, the cache and out.
 * The split partials go to one fixed array of VC_STATIC_SCRATCH_BYTES (8 MiB)
 * inside the library, held on every GPU that loads the library until the
 * process exits.  The first call on a device looks up that array's device
 * address (a one-time set-up per device); make that first call before any
 * stream capture.  The address is cached per device together with the
 * device's current context: after cudaDeviceReset the next call looks it up
 * again (make that call before any capture too).  A call with batch 0 checks
 * the format and returns VC_OK before looking at any pointer, as
 * vc_draft_attn does.  All calls share the array and it keeps the last call's
 * contents: calls that overlap on the GPU (several streams or threads) race,
 * so the caller must serialise them.  Nothing in it needs clearing: a call
 * writes every partial before it reads it.  A call that would need more
 * than the array (vc_draft_workspace_bytes(comp, num_q_heads, max_seq_len) >
 * VC_STATIC_SCRATCH_BYTES) returns VC_ERR_WORKSPACE and launches nothing.
 * No cudaMalloc, cudaFree or allocating library routine is called.
 */
VC_API vc_status vc_draft_attn_static(const void *q, int32_t num_q_heads, const vc_paged_kv *comp,
                                      float softmax_scale, float *out, int32_t max_seq_len,
                                      int32_t *dev_status, vc_stream_t stream);
VC_API size_t vc_static_scratch_bytes(void);

/*
 * vc_verify_attn -- the verification pass over KV_full.  Request b holds
 * L = full->seq_lens[b] tokens, the last n_q of which form the block being
 * verified; query i sits at position L - n_q + i and attends to positions
 * 0 .. L - n_q + i (causal inside the block).
 *  q    device bf16 [batch][n_q][num_q_heads][head_dim]
 *  out  device fp32 [batch][n_q][num_q_heads][head_dim]
 * 1 <= n_q <= 64, num_q_heads / num_kv_heads <= 8, head_dim in {64, 128},
 * full->fmt.bits == 16, L >= n_q (a request with L < n_q gets
 * VC_ERR_BAD_INDEX in dev_status and zero output).  The split over context
 * chunks is fixed by position (3648 keys), so a query's result does not
 * depend on n_q, its place in the block, or the batch.
 */
VC_API size_t vc_verify_workspace_bytes(const vc_paged_kv *full, int32_t n_q, int32_t num_q_heads,
                                 int32_t max_seq_len);
VC_API vc_status vc_verify_attn(const void *q, int32_t n_q, int32_t num_q_heads,
                         const vc_paged_kv *full, float softmax_scale, float *out,
                         int32_t max_seq_len, void *workspace, size_t workspace_bytes,
                         int32_t *dev_status, vc_stream_t stream);

/*
 * vc_accept -- greedy acceptance ("The Core Idea": compare left to right;
 * at the first mismatch emit the verified prefix and the verifier's token;
 * if all x drafts match emit them plus the bonus prediction).
 *  hidden        device fp32 [batch][n_pred][hidden_group][d]; prediction
 *                i's hidden vector is the mean of its hidden_group vectors
 *                ((fp32 sum in index order) / hidden_group; 1 = as given).
 *  lm_head       device fp32 [d][vocab].
 *  logits        fp32, one fused multiply-add per term in increasing k
 *                (the same value for a row whatever batch / n_pred).
 *  drafts        device int32 [batch][x]
 *  verified      device int32 [batch][n_pred]: argmax, lowest id on ties
 *  accept_len    device int32 [batch]: a = first i < x with a mismatch, else x
 *  emitted       device int32 [batch][x + 1]: drafts[0:a] then verified[a]
 *                when a < n_pred; remaining slots -1.
 * n_pred is x + 1 (bonus available) or x (no bonus); 1 <= n_pred.
 */
VC_API size_t vc_accept_workspace_bytes(int32_t batch, int32_t n_pred, int32_t vocab, int32_t d);
VC_API vc_status vc_accept(const float *hidden, int32_t batch, int32_t n_pred, int32_t hidden_group,
                    const float *lm_head, int32_t d, int32_t vocab, const int32_t *drafts,
                    int32_t x, int32_t *verified, int32_t *accept_len, int32_t *emitted,
                    void *workspace, size_t workspace_bytes, vc_stream_t stream);

/*
 * vc_accept_sampled -- acceptance for sampling at temperature tau > 0
 * ("VeriCache Guide", "Mathematical Guarantee of Lossless Correctness"):
 * draft i is kept while u[b][i] < min(1, p_target_i(d_i) / p_draft_i(d_i));
 * at the first rejection a token is drawn from the normalised residual
 * max(0, p_target_i - p_draft_i) by inverse CDF with v[b][i] and the round
 * ends; when all x drafts are kept a bonus is drawn from p_target_x with
 * v[b][x].  p = softmax(logits / tau), logits as in vc_accept (group mean of
 * the hidden rows, fp32, one fused multiply-add per hidden index in
 * increasing order); the softmax sums and the inverse CDF run in fp32.
 *  target_hidden device fp32 [batch][x + 1][hidden_group][d]  (verifier rows)
 *  draft_hidden  device fp32 [batch][x][hidden_group][d]      (drafter rows)
 *  drafts        device int32 [batch][x]; an id outside [0, vocab) is rejected.
 *  u, v          device fp32 [batch][x] and [batch][x + 1], uniform in [0, 1):
 *                the caller's random numbers (the library draws none).
 *  accept_len    device int32 [batch]; emitted device int32 [batch][x + 1]
 *                (a kept drafts, then the drawn token; -1 after).
 *  workspace     vc_accept_sampled_workspace_bytes(batch, x, vocab, d).
 */
VC_API size_t vc_accept_sampled_workspace_bytes(int32_t batch, int32_t x, int32_t vocab, int32_t d);
VC_API vc_status vc_accept_sampled(const float *target_hidden, const float *draft_hidden, int32_t batch, int32_t x,
                                   int32_t hidden_group, const float *lm_head, int32_t d, int32_t vocab,
                                   float temperature, const int32_t *drafts, const float *u, const float *v,
                                   int32_t *accept_len, int32_t *emitted, void *workspace, size_t workspace_bytes,
                                   vc_stream_t stream);

/*
 * vc_stage_async -- copy `bytes` from page-locked host memory to device
 * memory on the side stream `side` and record `done` (may be NULL) after it,
 * so a verify launch on another stream can wait for the staged KV_full
 * ("VeriCache Guide": full KV reloaded on a swap stream while drafting
 * continues; pinned memory for full DMA bandwidth).  Returns VC_ERR_STAGING
 * when src is not page-locked (or registered) host memory.
 */
VC_API vc_status vc_stage_async(void *dev_dst, const void *pinned_src, size_t bytes,
                         vc_stream_t side, vc_event_t done);

/*
 * A slower link emulated on one machine (remote prefix caching: "VeriCache:
 * Making Lossy KV Compression Exact", the two serving settings -- the
 * compressed cache of a stored prefix is sent to the serving GPU, the full
 * cache stays reachable for verification; study notes "VeriCache: Turning
 * Lossy KV Cache into Lossless LLM Inference", case 3 -- KV_comp over the slow
 * link to the drafter, KV_full over a fast link to the verifier).
 *  vc_link_clock         writes the device global timer (ns) to *origin_ns
 *                        (device int64) on `stream`: the link's time origin.
 *  vc_stage_paced_async  the copy of vc_stage_async in chunks of chunk_bytes;
 *                        chunk k (bytes [k c, min((k+1) c, bytes))) is issued on
 *                        `side` only after the timer has reached
 *                        *origin_ns + (link_offset_bytes + end of chunk k) /
 *                        bytes_per_ns, so data arrive no faster than a link of
 *                        bytes_per_ns that had already carried
 *                        link_offset_bytes since the origin.  The origin must be
 *                        written (vc_link_clock, ordered before on `side`)
 *                        first.  VC_ERR_INVALID_ARG for a null pointer, chunk 0,
 *                        a rate <= 0 or a span over 60 s of link time;
 *                        VC_ERR_STAGING when src is not page-locked.  Each wait
 *                        is a one-thread kernel that ends at its deadline (and
 *                        in any case within 60 s).
 */
VC_API vc_status vc_link_clock(int64_t *origin_ns, vc_stream_t stream);
VC_API vc_status vc_stage_paced_async(void *dev_dst, const void *pinned_src, size_t bytes, size_t chunk_bytes,
                                      double bytes_per_ns, const int64_t *origin_ns, size_t link_offset_bytes,
                                      vc_stream_t side, vc_event_t done);

/*
 * vc_mixed_attn -- one launch in which requests with role[b] == 0 run the
 * draft attention over `comp` and requests with role[b] == 1 run the
 * verification attention of an n_q block over `full` (cross-resource
 * staggering: some requests draft while others verify).  Arguments are
 * those of vc_draft_attn / vc_verify_attn; both caches describe the same
 * batch; role is device int32 [batch].  Outputs of a request are written
 * only to the buffer of its role; a request whose role is neither 0 nor 1 is
 * skipped (idle this launch: its block-table rows in either cache are not
 * read).  Workspace: vc_mixed_workspace_bytes.
 */
VC_API size_t vc_mixed_workspace_bytes(const vc_paged_kv *comp, const vc_paged_kv *full, int32_t n_q,
                                int32_t num_q_heads, int32_t max_seq_len);
VC_API vc_status vc_mixed_attn(const int32_t *role, const void *q_draft, const vc_paged_kv *comp,
                        float *out_draft, const void *q_verify, int32_t n_q,
                        const vc_paged_kv *full, float *out_verify, int32_t num_q_heads,
                        float softmax_scale, int32_t max_seq_len, void *workspace,
                        size_t workspace_bytes, int32_t *dev_status, vc_stream_t stream);

/*
 * Staggering scheduler (host code; no device pointers, no CUDA calls).
 *
 * "VeriCache: Making Lossy KV Compression Exact", "Verifying Without Giving
 * Back the Speedup" and Figure 2 (verifications spread over time so one
 * request's full-cache transfer overlaps the others' drafting); study notes
 * "VeriCache: Turning Lossy KV Cache into Lossless LLM Inference", case 2
 * (stagger who verifies so few full caches cross the link at once);
 * "VeriCache Guide", "The Amortized Drafting Horizon" (swap cost per token
 * T_swap / L) and "Best Practice 1" (size the horizon to hide the swap).
 *
 * Model: request r cycles through P = x + 1 ticks, verifying at the ticks t
 * with t mod P == phase[r] and drafting one token at every other tick.  A tick
 * runs all n_layers layers; its compute time is tick_ns plus, over its
 * drafting requests, draft_ns[r] and, over its verifying requests,
 * verify_ns[r] (each for all layers, split evenly over the layers).  The
 * verifying requests of a tick form one staging job: their stage_bytes
 * (KV_full, all layers) cross the link at link_bytes_per_ns, layer by layer,
 * into one of n_slots staging buffers.  Jobs run in tick order; a job starts
 * when the previous one is done and its slot's previous job's tick has ended.
 * Layer l of a verifying tick waits for layer l of its job; waiting is stall.
 */
typedef struct {
    int32_t n_requests;
    const int64_t *stage_bytes; /* host [n]: KV_full bytes staged per verification   */
    const double *draft_ns;     /* host [n]: one draft step, all layers (ns)          */
    const double *verify_ns;    /* host [n]: one verification, all layers (ns)        */
    double tick_ns;             /* fixed cost of a tick (launch latencies), >= 0      */
    double link_bytes_per_ns;   /* staging bandwidth, > 0                             */
    int32_t n_slots;            /* staging buffers, >= 1                              */
    int32_t n_layers;           /* >= 1                                               */
} vc_stagger_model;

typedef struct {             /* steady state: the last of the simulated cycles */
    double cycle_ns;         /* wall time of one cycle (P ticks)                  */
    double compute_ns;       /* sum of the cycle's tick compute times             */
    double stall_ns;         /* time ticks waited for staged layers               */
    double stage_ns;         /* link time of the cycle's staged bytes (T_swap sum) */
    double overlap;          /* 1 - stall / stage, in [0, 1] (1 when nothing staged) */
    int64_t peak_stage_bytes;       /* n_slots x the largest job                   */
    int64_t draft_tokens_per_cycle; /* n_requests x (P - 1)                        */
} vc_stagger_result;

/*
 * vc_stagger_plan -- assign each of n requests a phase in [0, n_phases).
 * (1) Longest processing time first into G = min(n, n_phases) groups:
 * requests in decreasing stage_bytes order (ties: lower index first), each to
 * the group with the fewest bytes so far (ties: lower group).  (2) Groups in
 * decreasing byte order (ties: lower group), interleaved largest, smallest,
 * second largest, ...  (3) The k-th group of that sequence verifies at phase
 * floor(k * n_phases / G), so groups are evenly spaced over the cycle and a
 * large staging job follows a small one.  phase: host int32 [n];
 * phase_bytes: host int64 [n_phases] or NULL (bytes verified per phase).
 * VC_ERR_INVALID_ARG on a negative size or a null array.
 */
VC_API vc_status vc_stagger_plan(const int64_t *stage_bytes, int32_t n, int32_t n_phases, int32_t *phase,
                                 int64_t *phase_bytes);
/*
 * vc_stagger_simulate -- run the model above for n_cycles cycles of n_phases
 * ticks from a cold start (staging begins at time 0) and report the last
 * cycle.  VC_ERR_INVALID_ARG on a bad model or a phase out of range.
 */
VC_API vc_status vc_stagger_simulate(const vc_stagger_model *m, int32_t n_phases, const int32_t *phase,
                                     int32_t n_cycles, vc_stagger_result *out);
/*
 * vc_stagger_horizon -- the smallest draft horizon x in [x_lo, x_hi] whose
 * balanced plan (P = x + 1 phases) has no steady-state stall, else x_hi; writes
 * x, its plan (phase: host int32 [n]) and its simulated result.
 */
VC_API vc_status vc_stagger_horizon(const vc_stagger_model *m, int32_t x_lo, int32_t x_hi, int32_t n_cycles,
                                    int32_t *x_out, int32_t *phase, vc_stagger_result *out);

/*
 * Decoder-layer operations for the end-to-end greedy loop (prefill, draft
 * steps, verification pass).  "VeriCache: Making Lossy KV Compression
 * Exact", "The Core Idea": drafter and verifier run the same model and
 * weights, only the KV cache differs.  Every operation computes each row from
 * that row alone with a fixed reduction order, so a token's results are the
 * same bits whether it is processed alone, in a verification block or in a
 * prefill chunk (this is what makes the loop reproduce full-cache greedy
 * decoding exactly).  All pointers are device pointers; rows are m.
 *  vc_embed          out[r] = table[ids[r]]  (fp32 [vocab][d]; a bad id gives
 *                    zeros and VC_ERR_BAD_INDEX in dev_status)
 *  vc_rmsnorm        out[r] = x[r] / sqrt(mean(x[r]^2) + eps) * weight (fp32)
 *  vc_linear         out[r][n] (+)= sum_k bf16(x[r][k]) * W[k][n]: x fp32 [m][k]
 *                    rounded to bf16 on load (activations are stored as bf16
 *                    between layers), W bf16 [k][n], fp32 FMAs in increasing k;
 *                    accumulate != 0 adds to out (residual connection).  Up to
 *                    16 rows run on a small-row kernel, more on a tiled one:
 *                    the same FMA chain, so the same bits either way
 *  vc_swiglu         out[r][c] = silu(gu[r][c]) * gu[r][f + c]  (fp32 [m][2f] -> [m][f])
 *  vc_rope_kv_write  qkv fp32 [m][(Hq + 2 Hkv) D] -> q bf16 [m][Hq][D] after a
 *                    rotary embedding (channel i pairs with i + D/2, angle
 *                    pos * theta^(-2i/D)), and the row's rotated K and its V
 *                    written as bf16 into `full` at (row_req[r], row_pos[r]).
 */
VC_API vc_status vc_embed(const int32_t *ids, int32_t m, const float *table, int32_t d, int32_t vocab,
                          float *out, int32_t *dev_status, vc_stream_t stream);
VC_API vc_status vc_rmsnorm(const float *x, int32_t m, int32_t d, const float *weight, float eps, float *out,
                            vc_stream_t stream);
VC_API vc_status vc_linear(const float *x, const void *w_bf16, float *out, int32_t m, int32_t k, int32_t n,
                           int32_t accumulate, vc_stream_t stream);
VC_API vc_status vc_swiglu(const float *gu, int32_t m, int32_t f, float *out, vc_stream_t stream);
VC_API vc_status vc_rope_kv_write(const float *qkv, int32_t m, const int32_t *row_req, const int32_t *row_pos,
                                  int32_t num_q_heads, float rope_theta, void *q_out, const vc_paged_kv *full,
                                  int32_t *dev_status, vc_stream_t stream);

/*
 * vc_debug_set_wait_fault -- fault injection for tests of the bounded device
 * waits (host-side switch, process-wide, off by default; not for production
 * use).  Every wait of a kernel on a copy or on another warp gives up after
 * a time limit, reports VC_ERR_TIMEOUT in dev_status and lets the block
 * drain and exit (no GPU hang on a lost copy).  This sets that limit for the
 * draft, draft-step, verification and mixed launches made after the call:
 * wait_limit_ns in (0, 2e9], or 0 for the default of 2 s.  skip_copies != 0
 * makes those kernels issue none of their KV page copies (and signal none),
 * so every wait on a copy runs into the limit: outputs are then zeros and
 * nothing of the cache is read.  Calls racing with launches on other threads
 * see either setting.  VC_ERR_INVALID_ARG for a limit out of range.
 */
VC_API vc_status vc_debug_set_wait_fault(int64_t wait_limit_ns, int32_t skip_copies);

VC_API const char *vc_status_string(vc_status s);
VC_API const char *vc_version(void);

#ifdef __cplusplus
}
#endif
#endif /* VC_H */
