// vc_select_kept: the kept-index list of a token-drop KV_comp, on the GPU.
//
// "VeriCache Guide", the compressor class of "Implementing VeriCache in
// Python and PyTorch": a token's importance is the norm of its key over the
// head dimension averaged over the heads; the top tokens are kept, in
// position order, and K and V are gathered with that one list (vc_compress).
// The workloads add a sink window and a recent window that are always kept.
//
// Kernel 1 (only without caller scores): one thread per token, per kv head
// the sum of squares with one fused multiply-add per channel in increasing
// channel order, a correctly rounded square root, the heads' norms added in
// increasing order, divided by the head count -- every step fixed, so the
// list is the same bit for bit wherever it is computed.
// Kernel 2: one CTA per request.  A 4-pass 8-bit radix select over the
// middle positions' order-preserving score keys finds the score of the
// top-th best position and how many positions tied at that score to take
// (the lowest positions first); one ordered pass then writes sink, chosen
// middle and recent positions in ascending order.
#include "vc_internal.cuh"

namespace vc {
namespace {

constexpr int kSelThreads = 1024;

__device__ inline uint32_t order_key(float f) {  // larger float <=> larger key
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

template <int D>
__global__ void keynorm_kernel(const uint8_t *kp, int64_t n_pages, const int32_t *table, const int32_t *lens,
                               int maxb, int hkv, float *scores, int stride, int32_t *status) {
    pdl_begin();
    const int b = blockIdx.y;
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= lens[b] || t >= stride) return;
    const int pi = t / kPage;
    const int page = pi < maxb ? table[(int64_t)b * maxb + pi] : -1;
    if (page < 0 || page >= n_pages) {
        report(status, VC_ERR_BAD_INDEX);
        return;
    }
    float tot = 0.0f;
    for (int h = 0; h < hkv; ++h) {
        const uint4 *row = reinterpret_cast<const uint4 *>(kp + (((int64_t)page * hkv + h) * kPage + t % kPage) * D * 2);
        float ss = 0.0f;
#pragma unroll 4
        for (int i = 0; i < D / 8; ++i) {
            const uint4 u = row[i];
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xFFFF0000u);
                ss = __fmaf_rn(lo, lo, ss);
                ss = __fmaf_rn(hi, hi, ss);
            }
        }
        tot = __fadd_rn(tot, __fsqrt_rn(ss));
    }
    scores[(int64_t)b * stride + t] = __fdiv_rn(tot, (float)hkv);
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(const float *scores, int stride, const int32_t *lens,
                                                             const int32_t *offs, int sink_in, int recent_in,
                                                             int32_t *idx, int32_t *status) {
    pdl_begin();
    __shared__ unsigned int hist[256];
    __shared__ unsigned int wsum[2][kSelThreads / 32];
    __shared__ uint32_t s_prefix, s_mask;
    __shared__ int s_need;
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = max(0, min(lens[b], stride));
    const int keep = offs[b + 1] - offs[b];
    const int sink = min(sink_in, n);
    const int recent = min(recent_in, n - sink);
    const int m = n - sink - recent;
    const int top = max(0, min(m, keep - sink - recent));
    if (sink + recent + top != keep) {  // the caller's slot count does not match the rule
        if (tid == 0) report(status, VC_ERR_INVALID_ARG);
        return;
    }
    const float *sc = scores + (int64_t)b * stride;
    // ---- radix select: the key of the top-th best middle position ----
    if (tid == 0) {
        s_prefix = 0u;
        s_mask = 0u;
        s_need = top;
    }
    if (top > 0 && top < m) {
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int i = tid; i < 256; i += kSelThreads) hist[i] = 0u;
            __syncthreads();
            const uint32_t prefix = s_prefix, mask = s_mask;
            for (int j = tid; j < m; j += kSelThreads) {
                const uint32_t k = order_key(sc[sink + j]);
                if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
            }
            __syncthreads();
            if (tid == 0) {
                int need = s_need;
                unsigned int above = 0;
                int dsel = 0;
                for (int d = 255; d >= 0; --d) {
                    if ((int)(above + hist[d]) >= need) {
                        dsel = d;
                        break;
                    }
                    above += hist[d];
                }
                s_need = need - (int)above;
                s_prefix = prefix | ((uint32_t)dsel << shift);
                s_mask = mask | (255u << shift);
            }
            __syncthreads();
        }
    }
    __syncthreads();
    const uint32_t thr = s_prefix;        // key of the last position taken
    const int ties_wanted = s_need;       // positions at exactly that key to take
    const bool all_mid = top >= m, no_mid = top <= 0;
    // ---- ordered pass: flags, block prefix sums, writes ----
    int base_out = 0, base_tie = 0;
    int32_t *out = idx + offs[b];
    for (int c0 = 0; c0 < n; c0 += kSelThreads) {
        const int t = c0 + tid;
        bool in = false, tie = false;
        uint32_t k = 0;
        if (t < n) {
            if (t < sink || t >= n - recent) {
                in = true;
            } else if (all_mid) {
                in = true;
            } else if (!no_mid) {
                k = order_key(sc[t]);
                in = k > thr;
                tie = k == thr;
            }
        }
        // exclusive counts of ties and of kept positions before t in the chunk
        const unsigned int bt = __ballot_sync(0xffffffffu, tie);
        if (lane == 0) wsum[0][warp] = __popc(bt);
        __syncthreads();
        int tie_before = base_tie + __popc(bt & ((1u << lane) - 1u));
        for (int w = 0; w < warp; ++w) tie_before += wsum[0][w];
        if (tie && tie_before < ties_wanted) in = true;
        const unsigned int bk = __ballot_sync(0xffffffffu, in);
        if (lane == 0) wsum[1][warp] = __popc(bk);
        __syncthreads();
        int pos = base_out + __popc(bk & ((1u << lane) - 1u));
        for (int w = 0; w < warp; ++w) pos += wsum[1][w];
        if (in) out[pos] = t;
        int tot_t = 0, tot_k = 0;
        for (int w = 0; w < kSelThreads / 32; ++w) {
            tot_t += wsum[0][w];
            tot_k += wsum[1][w];
        }
        base_tie += tot_t;
        base_out += tot_k;
        __syncthreads();
    }
}

}  // namespace

size_t select_workspace(int batch, int max_seq_len) { return (size_t)batch * max(max_seq_len, 1) * sizeof(float); }

vc_status select_kept(const vc_paged_kv *full, const float *scores, int32_t score_stride,
                      const int32_t *kept_offsets, int32_t sink, int32_t recent, int32_t *kept_idx, void *ws,
                      size_t ws_bytes, int32_t *dev_status, cudaStream_t st) {
    const int batch = full->batch;
    if (batch == 0) return VC_OK;
    const float *sc = scores;
    int stride = score_stride;
    if (!sc) {
        const int d = full->fmt.head_dim;
        if (full->fmt.bits != 16 || !(d == 64 || d == 128)) return VC_ERR_UNSUPPORTED;
        if (score_stride < 1) return VC_ERR_INVALID_ARG;
        if (!ws || ws_bytes < select_workspace(batch, score_stride)) return VC_ERR_WORKSPACE;
        float *w = reinterpret_cast<float *>(ws);
        dim3 grid(ceil_div(score_stride, 256), batch);
        if (d == 64)
            launch_pdl(keynorm_kernel<64>, grid, 256, 0, st, (const uint8_t *)full->k_pages, full->num_pages,
                       full->block_table, full->seq_lens, full->max_blocks,
                       full->fmt.num_kv_heads, w, score_stride, dev_status);
        else
            launch_pdl(keynorm_kernel<128>, grid, 256, 0, st, (const uint8_t *)full->k_pages, full->num_pages,
                       full->block_table, full->seq_lens, full->max_blocks,
                       full->fmt.num_kv_heads, w, score_stride, dev_status);
        if (cudaGetLastError() != cudaSuccess) return VC_ERR_CUDA;
        sc = w;
    }
    launch_pdl(select_kernel, batch, kSelThreads, 0, st, sc, stride, full->seq_lens, kept_offsets, sink, recent,
               kept_idx, dev_status);
    return cudaGetLastError() == cudaSuccess ? VC_OK : VC_ERR_CUDA;
}

}  // namespace vc
