// Host side of the C ABI declared in include/vc.h: argument validation,
// workspace queries, launches, KV_full staging and status strings.  Nothing
// here allocates device or host memory.
#include <cstring>

#include "vc_internal.cuh"

namespace vc {
vc_status compress(const vc_paged_kv *full, const int32_t *kept_offsets, const int32_t *kept_idx,
                   const int32_t *comp_start, int32_t max_kept, const vc_paged_kv *comp,
                   int32_t *dev_status, cudaStream_t st);
bool draft_supported(const vc_kv_format &f, int hq);
size_t draft_workspace(const vc_paged_kv &c, int hq, int max_seq_len);
cudaError_t draft_launch(const void *q, int hq, const vc_paged_kv &c, float scale, float *out,
                         int max_seq_len, void *ws, int32_t *status, cudaStream_t st,
                         const void *k_new = nullptr, const void *v_new = nullptr, const int32_t *slot = nullptr);
bool verify_supported(const vc_kv_format &f, int hq, int n_q);
size_t verify_workspace(const vc_paged_kv &f, int n_q, int hq, int max_seq_len);
cudaError_t verify_launch(const void *q, int n_q, int hq, const vc_paged_kv &f, float scale, float *out,
                          int max_seq_len, void *ws, int32_t *status, cudaStream_t st);
size_t accept_workspace(int batch, int n_pred, int vocab, int d);
size_t select_workspace(int batch, int max_seq_len);
size_t accept_sampled_workspace(int batch, int x, int vocab, int d);
cudaError_t accept_sampled_launch(const float *target_hidden, const float *draft_hidden, int batch, int x, int hg,
                                  const float *w, int d, int vocab, float tau, const int32_t *drafts,
                                  const float *u, const float *v, int32_t *accept_len, int32_t *emitted, void *ws,
                                  cudaStream_t st);
vc_status select_kept(const vc_paged_kv *full, const float *scores, int32_t score_stride,
                      const int32_t *kept_offsets, int32_t sink, int32_t recent, int32_t *kept_idx, void *ws,
                      size_t ws_bytes, int32_t *dev_status, cudaStream_t st);
cudaError_t accept_launch(const float *hidden, int batch, int n_pred, int hg, const float *w, int d,
                          int vocab, const int32_t *drafts, int x, int32_t *verified, int32_t *accept_len,
                          int32_t *emitted, void *ws, cudaStream_t st);
size_t mixed_workspace(const vc_paged_kv &comp, const vc_paged_kv &full, int n_q, int hq, int max_seq_len);
cudaError_t mixed_launch(const int32_t *role, const void *q_draft, const vc_paged_kv &comp, float *out_draft,
                         const void *q_verify, int n_q, const vc_paged_kv &full, float *out_verify, int hq,
                         float scale, int max_seq_len, void *ws, int32_t *status, cudaStream_t st);

namespace {
WaitFault g_wait_fault;
}  // namespace
WaitFault wait_fault() { return g_wait_fault; }

namespace {
// The format and batch of a paged cache (all an empty batch needs).
bool paged_fmt_ok(const vc_paged_kv *p) {
    return p && p->batch >= 0 && p->fmt.num_kv_heads >= 1 && p->fmt.head_dim >= 32 && p->fmt.head_dim % 32 == 0 &&
           p->fmt.head_dim <= VC_MAX_HEAD_DIM;
}
// ... and its pools, table and lengths, for a batch with requests.
bool paged_ok(const vc_paged_kv *p) {
    return paged_fmt_ok(p) && p->k_pages && p->v_pages && p->block_table && p->seq_lens && p->max_blocks >= 1 &&
           p->num_pages >= 1;
}
bool bits_ok(int b) { return b == 2 || b == 3 || b == 4 || b == 16; }
vc_status from_cuda(cudaError_t e) { return e == cudaSuccess ? VC_OK : VC_ERR_CUDA; }
}  // namespace
}  // namespace vc

using namespace vc;

extern "C" {

size_t vc_head_block_bytes(const vc_kv_format *f) {
    if (!f || !bits_ok(f->bits) || f->head_dim < 32 || f->head_dim % 32) return 0;
    if (f->bits != 16 && f->head_dim % 64) return 0;  // quantised formats: head_dim a multiple of 64
    return (size_t)head_block_bytes(f->bits, f->head_dim);
}

size_t vc_page_bytes(const vc_kv_format *f) {
    if (!f || f->num_kv_heads < 1) return 0;
    return vc_head_block_bytes(f) * (size_t)f->num_kv_heads;
}

vc_status vc_compress(const vc_paged_kv *full, const int32_t *kept_offsets, const int32_t *kept_idx,
                      const int32_t *comp_start, int32_t max_kept, const vc_paged_kv *comp,
                      int32_t *dev_status, vc_stream_t stream) {
    if (!paged_fmt_ok(full) || !comp) return VC_ERR_INVALID_ARG;
    if (full->batch > 0 && max_kept > 0 &&
        (!paged_ok(full) || !comp->k_pages || !comp->v_pages || !comp->block_table || comp->num_pages < 1 ||
         comp->max_blocks < 1))
        return VC_ERR_INVALID_ARG;
    return compress(full, kept_offsets, kept_idx, comp_start, max_kept, comp, dev_status,
                    (cudaStream_t)stream);
}

size_t vc_select_workspace_bytes(int32_t batch, int32_t score_stride) {
    if (batch < 0 || score_stride < 1) return 0;
    return select_workspace(batch, score_stride);
}

vc_status vc_select_kept(const vc_paged_kv *full, const float *scores, int32_t score_stride,
                         const int32_t *kept_offsets, int32_t sink, int32_t recent, int32_t *kept_idx,
                         void *workspace, size_t workspace_bytes, int32_t *dev_status, vc_stream_t stream) {
    if (!full || full->batch < 0 || sink < 0 || recent < 0 || score_stride < 1) return VC_ERR_INVALID_ARG;
    if (full->batch == 0) return VC_OK;
    if (!full->seq_lens || !kept_offsets || !kept_idx) return VC_ERR_INVALID_ARG;
    if (!scores && (!paged_ok(full) || !full->k_pages)) return VC_ERR_INVALID_ARG;
    return select_kept(full, scores, score_stride, kept_offsets, sink, recent, kept_idx, workspace, workspace_bytes,
                       dev_status, (cudaStream_t)stream);
}

size_t vc_draft_workspace_bytes(const vc_paged_kv *comp, int32_t num_q_heads, int32_t max_seq_len) {
    if (!comp || !draft_supported(comp->fmt, num_q_heads) || comp->batch < 0) return 0;
    return draft_workspace(*comp, num_q_heads, max_seq_len);
}

vc_status vc_draft_attn(const void *q, int32_t num_q_heads, const vc_paged_kv *comp, float softmax_scale,
                        float *out, int32_t max_seq_len, void *workspace, size_t workspace_bytes,
                        int32_t *dev_status, vc_stream_t stream) {
    if (!paged_fmt_ok(comp) || max_seq_len < 0) return VC_ERR_INVALID_ARG;
    if (!bits_ok(comp->fmt.bits) || !draft_supported(comp->fmt, num_q_heads)) return VC_ERR_UNSUPPORTED;
    if (comp->batch == 0) return VC_OK;
    if (!q || !out || !paged_ok(comp)) return VC_ERR_INVALID_ARG;
    const size_t need = draft_workspace(*comp, num_q_heads, max_seq_len > 0 ? max_seq_len : 1);
    if (!workspace || workspace_bytes < need) return VC_ERR_WORKSPACE;
    return from_cuda(draft_launch(q, num_q_heads, *comp, softmax_scale, out, max_seq_len > 0 ? max_seq_len : 1,
                                  workspace, dev_status, (cudaStream_t)stream));
}

vc_status vc_draft_step(const void *q, int32_t num_q_heads, const vc_paged_kv *comp, const void *k_new,
                        const void *v_new, const int32_t *slot, float softmax_scale, float *out,
                        int32_t max_seq_len, void *workspace, size_t workspace_bytes, int32_t *dev_status,
                        vc_stream_t stream) {
    if (!paged_fmt_ok(comp) || max_seq_len < 0) return VC_ERR_INVALID_ARG;
    if (!bits_ok(comp->fmt.bits) || !draft_supported(comp->fmt, num_q_heads)) return VC_ERR_UNSUPPORTED;
    if (comp->batch == 0) return VC_OK;
    if (!q || !out || !k_new || !v_new || !slot || !paged_ok(comp)) return VC_ERR_INVALID_ARG;
    const size_t need = draft_workspace(*comp, num_q_heads, max_seq_len > 0 ? max_seq_len : 1);
    if (!workspace || workspace_bytes < need) return VC_ERR_WORKSPACE;
    return from_cuda(draft_launch(q, num_q_heads, *comp, softmax_scale, out, max_seq_len > 0 ? max_seq_len : 1,
                                  workspace, dev_status, (cudaStream_t)stream, k_new, v_new, slot));
}

size_t vc_verify_workspace_bytes(const vc_paged_kv *full, int32_t n_q, int32_t num_q_heads,
                                 int32_t max_seq_len) {
    if (!full || !verify_supported(full->fmt, num_q_heads, n_q) || full->batch < 0) return 0;
    return verify_workspace(*full, n_q, num_q_heads, max_seq_len);
}

vc_status vc_verify_attn(const void *q, int32_t n_q, int32_t num_q_heads, const vc_paged_kv *full,
                         float softmax_scale, float *out, int32_t max_seq_len, void *workspace,
                         size_t workspace_bytes, int32_t *dev_status, vc_stream_t stream) {
    if (!paged_fmt_ok(full) || max_seq_len < 0 || n_q < 1) return VC_ERR_INVALID_ARG;
    if (!verify_supported(full->fmt, num_q_heads, n_q)) return VC_ERR_UNSUPPORTED;
    if (full->batch == 0) return VC_OK;
    if (!q || !out || !paged_ok(full)) return VC_ERR_INVALID_ARG;
    const int msl = max_seq_len > 0 ? max_seq_len : 1;
    if (!workspace || workspace_bytes < verify_workspace(*full, n_q, num_q_heads, msl)) return VC_ERR_WORKSPACE;
    return from_cuda(verify_launch(q, n_q, num_q_heads, *full, softmax_scale, out, msl, workspace, dev_status,
                                   (cudaStream_t)stream));
}

size_t vc_accept_workspace_bytes(int32_t batch, int32_t n_pred, int32_t vocab, int32_t d) {
    if (batch < 0 || n_pred < 1 || vocab < 1 || d < 1) return 0;
    return accept_workspace(batch, n_pred, vocab, d);
}

vc_status vc_accept(const float *hidden, int32_t batch, int32_t n_pred, int32_t hidden_group,
                    const float *lm_head, int32_t d, int32_t vocab, const int32_t *drafts, int32_t x,
                    int32_t *verified, int32_t *accept_len, int32_t *emitted, void *workspace,
                    size_t workspace_bytes, vc_stream_t stream) {
    if (!lm_head || batch < 0 || n_pred < 1 || hidden_group < 1 || d < 1 || vocab < 1 || x < 0)
        return VC_ERR_INVALID_ARG;
    if (n_pred != x && n_pred != x + 1) return VC_ERR_INVALID_ARG;
    if (batch == 0) return VC_OK;
    if (!hidden || !verified || !accept_len || !emitted || (x > 0 && !drafts)) return VC_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < accept_workspace(batch, n_pred, vocab, d)) return VC_ERR_WORKSPACE;
    return from_cuda(accept_launch(hidden, batch, n_pred, hidden_group, lm_head, d, vocab, drafts, x, verified,
                                   accept_len, emitted, workspace, (cudaStream_t)stream));
}

size_t vc_accept_sampled_workspace_bytes(int32_t batch, int32_t x, int32_t vocab, int32_t d) {
    if (batch < 0 || x < 0 || vocab < 1 || d < 1) return 0;
    return accept_sampled_workspace(batch, x, vocab, d);
}

vc_status vc_accept_sampled(const float *target_hidden, const float *draft_hidden, int32_t batch, int32_t x,
                            int32_t hidden_group, const float *lm_head, int32_t d, int32_t vocab, float temperature,
                            const int32_t *drafts, const float *u, const float *v, int32_t *accept_len,
                            int32_t *emitted, void *workspace, size_t workspace_bytes, vc_stream_t stream) {
    if (!lm_head || batch < 0 || x < 0 || hidden_group < 1 || d < 1 || vocab < 1 || !(temperature > 0.0f))
        return VC_ERR_INVALID_ARG;
    if (batch == 0) return VC_OK;
    if (!target_hidden || !accept_len || !emitted || !v || (x > 0 && (!draft_hidden || !drafts || !u)))
        return VC_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < accept_sampled_workspace(batch, x, vocab, d)) return VC_ERR_WORKSPACE;
    return from_cuda(accept_sampled_launch(target_hidden, draft_hidden, batch, x, hidden_group, lm_head, d, vocab,
                                           temperature, drafts, u, v, accept_len, emitted, workspace,
                                           (cudaStream_t)stream));
}

vc_status vc_stage_async(void *dev_dst, const void *pinned_src, size_t bytes, vc_stream_t side,
                         vc_event_t done) {
    if (!dev_dst || !pinned_src) return VC_ERR_INVALID_ARG;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, pinned_src) != cudaSuccess) {
        cudaGetLastError();
        return VC_ERR_STAGING;
    }
    if (at.type != cudaMemoryTypeHost) return VC_ERR_STAGING;
    if (bytes && cudaMemcpyAsync(dev_dst, pinned_src, bytes, cudaMemcpyHostToDevice, (cudaStream_t)side) !=
                     cudaSuccess)
        return VC_ERR_CUDA;
    if (done && cudaEventRecord((cudaEvent_t)done, (cudaStream_t)side) != cudaSuccess) return VC_ERR_CUDA;
    return VC_OK;
}

size_t vc_mixed_workspace_bytes(const vc_paged_kv *comp, const vc_paged_kv *full, int32_t n_q,
                                int32_t num_q_heads, int32_t max_seq_len) {
    if (!comp || !full || !draft_supported(comp->fmt, num_q_heads) ||
        !verify_supported(full->fmt, num_q_heads, n_q))
        return 0;
    return mixed_workspace(*comp, *full, n_q, num_q_heads, max_seq_len);
}

vc_status vc_mixed_attn(const int32_t *role, const void *q_draft, const vc_paged_kv *comp, float *out_draft,
                        const void *q_verify, int32_t n_q, const vc_paged_kv *full, float *out_verify,
                        int32_t num_q_heads, float softmax_scale, int32_t max_seq_len, void *workspace,
                        size_t workspace_bytes, int32_t *dev_status, vc_stream_t stream) {
    if (!paged_fmt_ok(comp) || !paged_fmt_ok(full) || max_seq_len < 0 || n_q < 1 || comp->batch != full->batch)
        return VC_ERR_INVALID_ARG;
    if (comp->fmt.num_kv_heads != full->fmt.num_kv_heads || comp->fmt.head_dim != full->fmt.head_dim)
        return VC_ERR_INVALID_ARG;
    if (!draft_supported(comp->fmt, num_q_heads) || !verify_supported(full->fmt, num_q_heads, n_q))
        return VC_ERR_UNSUPPORTED;
    if (comp->batch == 0) return VC_OK;
    if (!role || !q_draft || !q_verify || !out_draft || !out_verify || !paged_ok(comp) || !paged_ok(full))
        return VC_ERR_INVALID_ARG;
    const int msl = max_seq_len > 0 ? max_seq_len : 1;
    if (!workspace || workspace_bytes < mixed_workspace(*comp, *full, n_q, num_q_heads, msl))
        return VC_ERR_WORKSPACE;
    return from_cuda(mixed_launch(role, q_draft, *comp, out_draft, q_verify, n_q, *full, out_verify, num_q_heads,
                                  softmax_scale, msl, workspace, dev_status, (cudaStream_t)stream));
}

vc_status vc_debug_set_wait_fault(int64_t wait_limit_ns, int32_t skip_copies) {
    if (wait_limit_ns < 0 || wait_limit_ns > (int64_t)kWaitNs) return VC_ERR_INVALID_ARG;
    g_wait_fault.wait_ns = wait_limit_ns == 0 ? kWaitNs : (uint64_t)wait_limit_ns;
    g_wait_fault.skip_copies = skip_copies != 0;
    return VC_OK;
}

const char *vc_status_string(vc_status s) {
    switch (s) {
        case VC_OK: return "ok";
        case VC_ERR_INVALID_ARG: return "invalid argument";
        case VC_ERR_UNSUPPORTED: return "unsupported format or shape";
        case VC_ERR_BAD_INDEX: return "page id or index out of range";
        case VC_ERR_CUDA: return "CUDA launch or copy failed";
        case VC_ERR_STAGING: return "staging source is not page-locked host memory";
        case VC_ERR_TIMEOUT: return "bounded device wait timed out";
        case VC_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

const char *vc_version(void) { return "vericache-gb300 0.1 (sm_103a)"; }

}  // extern "C"
