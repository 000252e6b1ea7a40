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

// The same products for up to 16 rows (decode and draft steps), with every
// (row, column) fp32 FMA chain in increasing k, exactly the tiled kernel's
// arithmetic (k padded with zeros to a multiple of TK; the further zero
// products of a chunk's tail leave a sum unchanged, as a sum that starts at
// +0 is never -0), so a row's bits do not depend on which kernel computed
// it.  Such a chain is k dependent FMAs long, which bounds the time from
// below (about 4 cycles per k); with a handful of rows a 64 x 128 tile
// wastes most of its work and gives the narrow projections a few CTAs.
// Here a CTA owns 32 columns and has one warp per kRowsPerWarp rows, each
// thread carrying those rows' chains of one column, fed by one W value; the
// CTA's warps share the W tile (kChunk x 32 columns) and the x tile (rows
// x kChunk), both requested by asynchronous 16-byte copies
// kStages - 1 chunks ahead and x rounded to bf16 in place once per chunk.
// A chunk is summed as straight-line code that asks for the next 16 k's
// operands before the current 16 k's FMAs.  Measured at 4 rows, k = 1024:
// ~15 cycles per k against the chain's ~4, most of it waiting on
// fixed-latency and shared-memory dependencies (the compiler keeps few
// operands in flight); one warp carrying all rows of a column spent ~40.
constexpr int kSmallRows = 16;
constexpr int kSmallCols = 32;  // columns per CTA (= lanes of a warp)
constexpr int kChunk = 256;     // k per tile
constexpr int kStages = 4;      // tiles in the ring
// rows (chains) per thread, one W value feeding them all: one up to 8 rows,
// two above (4 rows, k = 1024: 8.3 us against 14.0 with two; 16 rows: 16.4
// against 14.0)
inline int small_rows_per_warp(int m) { return m <= 8 ? 1 : 2; }
inline int small_rows_smem(int m, int R) {  // x tiles padded to whole warps with zero rows
    return kStages * (kChunk * kSmallCols * 2 + ceil_div(m, R) * R * kChunk * 4);
}
__device__ inline void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
template <int kRowsPerWarp>
__global__ void __launch_bounds__(kSmallCols *kSmallRows) linear_rows_kernel(const float *x, const uint16_t *w,
                                                                            float *out, int m, int k, int n,
                                                                            int accumulate) {
    pdl_begin();
    extern __shared__ __align__(16) uint8_t dsm[];
    uint16_t(*ws)[kChunk][kSmallCols] = reinterpret_cast<uint16_t(*)[kChunk][kSmallCols]>(dsm);
    const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, r0 = (tid >> 5) * kRowsPerWarp;
    const int mp = (nt >> 5) * kRowsPerWarp;  // x tile rows; rows from m on are zeros
    float *xs = reinterpret_cast<float *>(dsm + kStages * kChunk * kSmallCols * 2);  // stage s: [mp][kChunk]
    const int c0 = blockIdx.x * kSmallCols, c = c0 + lane;
    const int kp = ceil_div(k, TK) * TK;  // the tiled kernel's zero-padded k
    const int nchunk = ceil_div(kp, kChunk);
    // 16-byte copies need whole 8-column (W) or 4-element (x) groups at 16-byte aligned addresses
    const bool wvec = (n % 8 == 0) && ((reinterpret_cast<uintptr_t>(w) & 15) == 0);
    const bool xvec = (k % 4 == 0) && ((reinterpret_cast<uintptr_t>(x) & 15) == 0);
    auto load = [&](int i) {  // chunk i: k in [i kChunk, (i + 1) kChunk), zeros from k on
        if (i < nchunk) {
            const int k0 = i * kChunk;
            float *xd = xs + (i % kStages) * mp * kChunk;
            for (int e = tid; e < mp * (kChunk / 4); e += nt) {
                const int rr = e / (kChunk / 4), kk = 4 * (e % (kChunk / 4)), kr = k0 + kk;
                float *d = xd + rr * kChunk + kk;
                const float *src = x + (int64_t)rr * k + kr;
                if (xvec && rr < m && kr + 4 <= k) {
                    cp_async16(d, src);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) d[j] = (rr < m && kr + j < k) ? src[j] : 0.0f;
                }
            }
            uint16_t(*wd)[kSmallCols] = ws[i % kStages];
            for (int e = tid; e < kChunk * (kSmallCols / 8); e += nt) {
                const int kk = e / (kSmallCols / 8), q = e % (kSmallCols / 8);
                const int kr = k0 + kk, cq = c0 + 8 * q;
                if (wvec && kr < k && cq + 8 <= n) {
                    cp_async16(&wd[kk][8 * q], w + (int64_t)kr * n + cq);
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        wd[kk][8 * q + j] = (kr < k && cq + j < n) ? w[(int64_t)kr * n + cq + j] : 0;
                }
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");  // one group per chunk slot, empty past the end
    };
    float acc[kRowsPerWarp] = {};
    for (int i = 0; i < kStages - 1; ++i) load(i);
    for (int i = 0; i < nchunk; ++i) {
        load(i + kStages - 1);
        asm volatile("cp.async.wait_group %0;" ::"n"(kStages - 1) : "memory");  // chunk i has landed
        __syncthreads();
        float *xt = xs + (i % kStages) * mp * kChunk;
        for (int e = tid; e < mp * kChunk; e += nt) xt[e] = __bfloat162float(__float2bfloat16_rn(xt[e]));
        __syncthreads();
        const float *xr = xt + r0 * kChunk;
        const uint16_t(*wt)[kSmallCols] = ws[i % kStages];
        // register double buffer: sub-block b + 1's operands are loaded
        // before sub-block b's FMAs, so the loads' latency overlaps the chain
        constexpr int SB = 16;
        float4 xv[2][kRowsPerWarp][SB / 4];
        uint16_t wv[2][SB];
#pragma unroll
        for (int j = 0; j < SB; ++j) wv[0][j] = wt[j][lane];
#pragma unroll
        for (int q = 0; q < kRowsPerWarp; ++q)
#pragma unroll
            for (int j = 0; j < SB / 4; ++j) xv[0][q][j] = *reinterpret_cast<const float4 *>(xr + q * kChunk + 4 * j);
#pragma unroll
        for (int b = 0; b < kChunk / SB; ++b) {
            const int cur = b & 1, nxt = cur ^ 1;
            if (b + 1 < kChunk / SB) {
#pragma unroll
                for (int j = 0; j < SB; ++j) wv[nxt][j] = wt[(b + 1) * SB + j][lane];
#pragma unroll
                for (int q = 0; q < kRowsPerWarp; ++q)
#pragma unroll
                    for (int j = 0; j < SB / 4; ++j)
                        xv[nxt][q][j] = *reinterpret_cast<const float4 *>(xr + q * kChunk + (b + 1) * SB + 4 * j);
            }
#pragma unroll
            for (int j = 0; j < SB / 4; ++j) {
                const float w0 = bf16_bits_to_f32(wv[cur][4 * j]), w1 = bf16_bits_to_f32(wv[cur][4 * j + 1]);
                const float w2 = bf16_bits_to_f32(wv[cur][4 * j + 2]), w3 = bf16_bits_to_f32(wv[cur][4 * j + 3]);
#pragma unroll
                for (int q = 0; q < kRowsPerWarp; ++q) {
                    acc[q] = fmaf(xv[cur][q][j].x, w0, acc[q]);
                    acc[q] = fmaf(xv[cur][q][j].y, w1, acc[q]);
                    acc[q] = fmaf(xv[cur][q][j].z, w2, acc[q]);
                    acc[q] = fmaf(xv[cur][q][j].w, w3, acc[q]);
                }
            }
        }
        __syncthreads();  // the stage is refilled next
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    if (c < n) {
#pragma unroll
        for (int q = 0; q < kRowsPerWarp; ++q) {
            if (r0 + q >= m) break;
            float *o = out + (int64_t)(r0 + q) * n + c;
            *o = accumulate ? (*o + acc[q]) : acc[q];
        }
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
        const int R = small_rows_per_warp(m);
        // the largest tile set of each variant
        const cudaError_t e = R == 1 ? set_smem_limit((const void *)linear_rows_kernel<1>, small_rows_smem(8, 1))
                                     : set_smem_limit((const void *)linear_rows_kernel<2>,
                                                      small_rows_smem(kSmallRows, 2));
        if (e != cudaSuccess) return VC_ERR_CUDA;
        const dim3 grid(ceil_div(n, kSmallCols)), block(kSmallCols * ceil_div(m, R));
        if (R == 1)
            launch_pdl(linear_rows_kernel<1>, grid, block, small_rows_smem(m, 1), st, x, w, out, m, k, n, accumulate);
        else
            launch_pdl(linear_rows_kernel<2>, grid, block, small_rows_smem(m, 2), st, x, w, out, m, k, n, accumulate);
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
