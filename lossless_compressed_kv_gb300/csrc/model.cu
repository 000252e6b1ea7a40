// Decoder-layer kernels around the attention step, used by the end-to-end
// greedy loop (draft steps, verification pass, prefill).  "VeriCache: Making
// Lossy KV Compression Exact", section "The Core Idea": the drafter and the
// verifier are the same model with the same weights; only the cache differs.
//
// Every kernel computes each output row from that row alone with a fixed
// reduction order, so a token's hidden state, K/V and logits are the same
// bits whether it is processed alone (one decode step), in a verification
// block of x + 1 tokens, or in a prefill chunk.  That row invariance is what
// lets the draft/verify loop reproduce full-cache greedy decoding exactly.
#include "vc_internal.cuh"

namespace vc {
namespace {

__global__ void embed_kernel(const int32_t *ids, int m, const float *table, int d, int vocab, float *out,
                             int32_t *status) {
    pdl_begin();
    const int r = blockIdx.x;
    const int id = ids[r];
    const bool ok = id >= 0 && id < vocab;
    if (!ok && threadIdx.x == 0) report(status, VC_ERR_BAD_INDEX);
    for (int c = threadIdx.x; c < d; c += blockDim.x) out[(int64_t)r * d + c] = ok ? table[(int64_t)id * d + c] : 0.0f;
}

// y = x / sqrt(mean(x^2) + eps) * w; per-thread strided sums, then a fixed
// shuffle / shared-memory tree.
__global__ void rmsnorm_kernel(const float *x, int d, const float *w, float eps, float *out) {
    pdl_begin();
    __shared__ float part[32];
    const int64_t r = blockIdx.x;
    const float *xr = x + r * d;
    float s = 0.0f;
    for (int c = threadIdx.x; c < d; c += blockDim.x) s = fmaf(xr[c], xr[c], s);
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = threadIdx.x < (blockDim.x >> 5) ? part[threadIdx.x] : 0.0f;
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (threadIdx.x == 0) part[0] = v;
    }
    __syncthreads();
    const float inv = rsqrtf(part[0] / (float)d + eps);
    for (int c = threadIdx.x; c < d; c += blockDim.x) out[r * d + c] = xr[c] * inv * w[c];
}

// out[m][n] (+)= sum_k bf16(x[m][k]) * W[k][n]: fp32 FMAs in increasing k.
// Tile 64 x 128 x 32, 256 threads, 4 x 8 outputs per thread.
constexpr int TM = 64, TN = 128, TK = 32;
__global__ void __launch_bounds__(256) linear_kernel(const float *x, const uint16_t *w, float *out, int m, int k,
                                                     int n, int accumulate) {
    pdl_begin();
    __shared__ float As[TK][TM + 4];
    __shared__ float Bs[TK][TN];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
    float acc[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;
    for (int k0 = 0; k0 < k; k0 += TK) {
        __syncthreads();
        for (int e = threadIdx.x; e < TM * TK; e += 256) {
            const int r = e / TK, kk = e % TK;
            float v = 0.0f;
            if (m0 + r < m && k0 + kk < k) {
                // activations are stored as bf16 between layers: round on load
                v = __bfloat162float(__float2bfloat16_rn(x[(int64_t)(m0 + r) * k + k0 + kk]));
            }
            As[kk][r] = v;
        }
        for (int e = threadIdx.x; e < TK * TN; e += 256) {
            const int kk = e / TN, c = e % TN;
            Bs[kk][c] = (k0 + kk < k && n0 + c < n) ? bf16_bits_to_f32(w[(int64_t)(k0 + kk) * n + n0 + c]) : 0.0f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < TK; ++kk) {
            float a[4], bv[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 8; ++j) bv[j] = Bs[kk][tx * 8 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], bv[j], acc[i][j]);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = m0 + ty * 4 + i;
        if (r >= m) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int c = n0 + tx * 8 + j;
            if (c >= n) continue;
            float *o = out + (int64_t)r * n + c;
            *o = accumulate ? (*o + acc[i][j]) : acc[i][j];
        }
    }
}

// The same products for up to MR rows (decode and draft steps): one output
// column per thread and every row's fp32 FMA chain in increasing k, exactly
// the tiled kernel's arithmetic (k padded with zeros to a multiple of TK), so
// a row's bits do not depend on which kernel computed it.  A 64 x 128 tile
// for a handful of rows wasted most of its work and gave the narrow
// projections a few CTAs; here one warp owns 32 columns, and its W tile
// (kChunk rows x 32 columns) is brought into shared memory by asynchronous
// 16-byte copies one chunk ahead, so enough bytes are in flight per warp
// (a column read straight from global memory leaves each warp a few
// hundred bytes in flight: the kernel then ran at ~100 GB/s).
constexpr int kSmallRows = 16;
constexpr int kSmallCols = 32;  // threads (= columns) per CTA
constexpr int kChunk = 256;     // k per W tile
__device__ inline void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
template <int MR>
__global__ void __launch_bounds__(kSmallCols) linear_rows_kernel(const float *x, const uint16_t *w, float *out,
                                                                 int m, int k, int n, int accumulate) {
    pdl_begin();
    __shared__ __align__(16) float xs[kChunk][MR];                // bf16-rounded activations, k-major
    __shared__ __align__(16) uint16_t ws[2][kChunk][kSmallCols];  // W tiles, double-buffered
    const int lane = threadIdx.x;
    const int c0 = blockIdx.x * kSmallCols, c = c0 + lane;
    const int kp = ceil_div(k, TK) * TK;  // the tiled kernel's zero-padded k
    const int nchunk = ceil_div(kp, kChunk);
    // 16-byte copies need whole 8-column groups at 16-byte aligned addresses
    const bool vec = (n % 8 == 0) && ((reinterpret_cast<uintptr_t>(w) & 15) == 0);
    auto load_w = [&](int buf, int k0) {  // rows [k0, k0 + kChunk), columns [c0, c0 + 32)
        for (int e = lane; e < kChunk * (kSmallCols / 8); e += kSmallCols) {
            const int kk = e / (kSmallCols / 8), q = e % (kSmallCols / 8);
            const int kr = k0 + kk, cq = c0 + 8 * q;
            uint16_t *dst = &ws[buf][kk][8 * q];
            if (vec && kr < k && cq + 8 <= n) {
                cp_async16(dst, w + (int64_t)kr * n + cq);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) dst[j] = (kr < k && cq + j < n) ? w[(int64_t)kr * n + cq + j] : 0;
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    float acc[MR];
#pragma unroll
    for (int r = 0; r < MR; ++r) acc[r] = 0.0f;
    load_w(0, 0);
    for (int i = 0; i < nchunk; ++i) {
        const int k0 = i * kChunk, kn = min(kChunk, kp - k0);
        if (i + 1 < nchunk) load_w((i + 1) & 1, k0 + kChunk);
        for (int e = lane; e < kn * MR; e += kSmallCols) {
            const int kk = e / MR, r = e % MR;
            float v = 0.0f;
            if (r < m && k0 + kk < k) v = __bfloat162float(__float2bfloat16_rn(x[(int64_t)r * k + k0 + kk]));
            xs[kk][r] = v;
        }
        if (i + 1 < nchunk)
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        else
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();
        const uint16_t(*wt)[kSmallCols] = ws[i & 1];
#pragma unroll 8
        for (int kk = 0; kk < kn; ++kk) {
            const float bv = bf16_bits_to_f32(wt[kk][lane]);
#pragma unroll
            for (int r = 0; r < MR; ++r) acc[r] = fmaf(xs[kk][r], bv, acc[r]);
        }
        __syncthreads();  // the tiles and xs are rewritten next
    }
    if (c >= n) return;
#pragma unroll
    for (int r = 0; r < MR; ++r) {
        if (r >= m) break;
        float *o = out + (int64_t)r * n + c;
        *o = accumulate ? (*o + acc[r]) : acc[r];
    }
}

// silu(g) * u, g = gu[:, :f], u = gu[:, f:]
__global__ void swiglu_kernel(const float *gu, int m, int f, float *out) {
    pdl_begin();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)m * f) return;
    const int64_t r = i / f, c = i % f;
    const float g = gu[r * 2 * f + c], u = gu[r * 2 * f + f + c];
    out[i] = g / (1.0f + expf(-g)) * u;
}

// Split qkv rows into heads, rotate q and k (rotate-half convention: channel
// i pairs with i + D/2, angle = pos * theta^(-2i/D)), write q (bf16) and the
// row's K and V (bf16) into the paged full cache at (request, position).
__global__ void rope_kv_kernel(const float *qkv, const int32_t *row_req, const int32_t *row_pos, int hq, int hkv,
                               int d, float theta, uint16_t *q_out, uint8_t *kp, uint8_t *vp, int64_t n_pages,
                               const int32_t *table, int maxb, int batch, int32_t *status) {
    pdl_begin();
    const int r = blockIdx.x;
    const int b = row_req[r], pos = row_pos[r];
    const bool req_ok = b >= 0 && b < batch;
    const int nh = hq + 2 * hkv;
    const float *x = qkv + (int64_t)r * nh * d;
    const int half = d / 2;
    const int blk = pos / kPage;
    const int page = (req_ok && pos >= 0 && blk < maxb) ? table[(int64_t)b * maxb + blk] : -1;
    const bool page_ok = page >= 0 && page < n_pages;
    if (!page_ok && threadIdx.x == 0) report(status, VC_ERR_BAD_INDEX);
    for (int e = threadIdx.x; e < nh * half; e += blockDim.x) {
        const int h = e / half, i = e % half;
        const float x0 = x[h * d + i], x1 = x[h * d + i + half];
        float y0 = x0, y1 = x1;
        if (h < hq + hkv) {
            const float inv_freq = powf(theta, -2.0f * (float)i / (float)d);
            float sn, cs;
            sincosf((float)pos * inv_freq, &sn, &cs);
            y0 = x0 * cs - x1 * sn;
            y1 = x1 * cs + x0 * sn;
        }
        const uint16_t b0 = __bfloat16_as_ushort(__float2bfloat16_rn(y0));
        const uint16_t b1 = __bfloat16_as_ushort(__float2bfloat16_rn(y1));
        if (h < hq) {
            q_out[((int64_t)r * hq + h) * d + i] = b0;
            q_out[((int64_t)r * hq + h) * d + i + half] = b1;
        } else if (page_ok) {
            const int kvh = h < hq + hkv ? h - hq : h - hq - hkv;
            uint8_t *pool = h < hq + hkv ? kp : vp;
            uint16_t *row = reinterpret_cast<uint16_t *>(pool + ((int64_t)page * hkv + kvh) * kPage * d * 2) +
                            (pos % kPage) * d;
            row[i] = b0;
            row[i + half] = b1;
        }
    }
}

}  // namespace
}  // namespace vc

using namespace vc;

extern "C" {

vc_status vc_embed(const int32_t *ids, int32_t m, const float *table, int32_t d, int32_t vocab, float *out,
                   int32_t *dev_status, vc_stream_t stream) {
    if (!ids || !table || !out || m < 0 || d < 1 || vocab < 1) return VC_ERR_INVALID_ARG;
    if (m == 0) return VC_OK;
    launch_pdl(embed_kernel, m, 256, 0, (cudaStream_t)stream, ids, m, table, d, vocab, out, dev_status);
    return cudaGetLastError() == cudaSuccess ? VC_OK : VC_ERR_CUDA;
}

vc_status vc_rmsnorm(const float *x, int32_t m, int32_t d, const float *weight, float eps, float *out,
                     vc_stream_t stream) {
    if (!x || !weight || !out || m < 0 || d < 1) return VC_ERR_INVALID_ARG;
    if (m == 0) return VC_OK;
    launch_pdl(rmsnorm_kernel, m, 256, 0, (cudaStream_t)stream, x, d, weight, eps, out);
    return cudaGetLastError() == cudaSuccess ? VC_OK : VC_ERR_CUDA;
}

vc_status vc_linear(const float *x, const void *w_bf16, float *out, int32_t m, int32_t k, int32_t n,
                    int32_t accumulate, vc_stream_t stream) {
    if (!x || !w_bf16 || !out || m < 0 || k < 1 || n < 1) return VC_ERR_INVALID_ARG;
    if (m == 0) return VC_OK;
    const uint16_t *w = (const uint16_t *)w_bf16;
    const cudaStream_t st = (cudaStream_t)stream;
    if (m <= kSmallRows) {
        const dim3 grid(ceil_div(n, kSmallCols));
        if (m <= 4)
            launch_pdl(linear_rows_kernel<4>, grid, kSmallCols, 0, st, x, w, out, m, k, n, accumulate);
        else if (m <= 8)
            launch_pdl(linear_rows_kernel<8>, grid, kSmallCols, 0, st, x, w, out, m, k, n, accumulate);
        else
            launch_pdl(linear_rows_kernel<16>, grid, kSmallCols, 0, st, x, w, out, m, k, n, accumulate);
    } else {
        dim3 grid(ceil_div(n, TN), ceil_div(m, TM));
        launch_pdl(linear_kernel, grid, 256, 0, st, x, w, out, m, k, n, accumulate);
    }
    return cudaGetLastError() == cudaSuccess ? VC_OK : VC_ERR_CUDA;
}

vc_status vc_swiglu(const float *gu, int32_t m, int32_t f, float *out, vc_stream_t stream) {
    if (!gu || !out || m < 0 || f < 1) return VC_ERR_INVALID_ARG;
    if (m == 0) return VC_OK;
    const int64_t n = (int64_t)m * f;
    launch_pdl(swiglu_kernel, (unsigned)((n + 255) / 256), 256, 0, (cudaStream_t)stream, gu, m, f, out);
    return cudaGetLastError() == cudaSuccess ? VC_OK : VC_ERR_CUDA;
}

vc_status vc_rope_kv_write(const float *qkv, int32_t m, const int32_t *row_req, const int32_t *row_pos,
                           int32_t num_q_heads, float rope_theta, void *q_out, const vc_paged_kv *full,
                           int32_t *dev_status, vc_stream_t stream) {
    if (!qkv || !row_req || !row_pos || !q_out || !full || !full->k_pages || !full->v_pages ||
        !full->block_table || m < 0 || num_q_heads < 1 || full->fmt.bits != 16 || full->fmt.head_dim % 2)
        return VC_ERR_INVALID_ARG;
    if (m == 0) return VC_OK;
    launch_pdl(rope_kv_kernel, m, 256, 0, (cudaStream_t)stream,
               qkv, row_req, row_pos, num_q_heads, full->fmt.num_kv_heads, full->fmt.head_dim, rope_theta,
               (uint16_t *)q_out, (uint8_t *)full->k_pages, (uint8_t *)full->v_pages, full->num_pages,
               full->block_table, full->max_blocks, full->batch, dev_status);
    return cudaGetLastError() == cudaSuccess ? VC_OK : VC_ERR_CUDA;
}

}  // extern "C"
