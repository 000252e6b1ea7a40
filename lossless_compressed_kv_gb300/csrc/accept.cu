// vc_accept: greedy acceptance of one verification round.
//
// "VeriCache: Making Lossy KV Compression Exact", section "The Core Idea":
// the verifier's predictions are compared with the drafts left to right; at
// the first mismatch the matched prefix and the verifier's own token are
// emitted (the rest of the draft is discarded); when every draft matches
// the draft is emitted together with the verifier's extra (bonus) token.
//
// Kernel 1: logits of a tile of prediction rows x a tile of the vocabulary,
// one column per thread, fp32 with one fused multiply-add per term in
// increasing k (so a row's logits are the same bits whatever the batch or
// the number of rows), then the tile's argmax (ties -> lowest id).
// Kernel 2: per request, argmax over the vocabulary tiles and the prefix
// rule.
#include "vc_internal.cuh"

namespace vc {
namespace {

constexpr int kCols = 256;  // vocabulary columns per CTA (one per thread)
constexpr int kRowsT = 16;  // prediction rows per CTA
constexpr int kKT = 64;     // hidden dims staged per step

struct Best {
    float v;
    int i;
};
__device__ inline Best better(Best a, Best b) {  // larger value, lower id on ties
    if (b.v > a.v || (b.v == a.v && b.i < a.i)) return b;
    return a;
}

// h[r][k] = (sum_j hidden[r][j][k], in increasing j) / hg, once per row.
__global__ void group_mean_kernel(const float *hidden, int rows, int hg, int d, float *h) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)rows * d) return;
    const int64_t r = i / d, k = i % d;
    const float *hp = hidden + (r * hg) * d + k;
    float s = 0.0f;
    for (int j = 0; j < hg; ++j) s = __fadd_rn(s, hp[(int64_t)j * d]);
    h[i] = __fdiv_rn(s, (float)hg);
}

__global__ void __launch_bounds__(kCols) logits_argmax_kernel(const float *h, int rows, const float *w, int d,
                                                             int vocab, float *part_v, int *part_i, int ntiles) {
    __shared__ float hs[kRowsT][kKT];
    __shared__ Best red[kRowsT][kCols / 32];
    const int vt = blockIdx.x, r0 = blockIdx.y * kRowsT;
    const int v = vt * kCols + threadIdx.x;
    const bool vok = v < vocab;
    float acc[kRowsT];
#pragma unroll
    for (int r = 0; r < kRowsT; ++r) acc[r] = 0.0f;
    for (int k0 = 0; k0 < d; k0 += kKT) {
        __syncthreads();
        for (int e = threadIdx.x; e < kRowsT * kKT; e += kCols) {
            const int r = e / kKT, k = k0 + e % kKT;
            hs[r][e % kKT] = (r0 + r < rows && k < d) ? h[(int64_t)(r0 + r) * d + k] : 0.0f;
        }
        __syncthreads();
        if (vok) {
            const int kn = min(kKT, d - k0);
            for (int kk = 0; kk < kn; ++kk) {
                const float wv = w[(int64_t)(k0 + kk) * vocab + v];
#pragma unroll
                for (int r = 0; r < kRowsT; ++r) acc[r] = __fmaf_rn(hs[r][kk], wv, acc[r]);
            }
        }
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int r = 0; r < kRowsT; ++r) {
        Best bb = {vok ? acc[r] : -INFINITY, vok ? v : 0x7fffffff};
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            Best o;
            o.v = __shfl_xor_sync(0xffffffffu, bb.v, off);
            o.i = __shfl_xor_sync(0xffffffffu, bb.i, off);
            bb = better(bb, o);
        }
        if (lane == 0) red[r][warp] = bb;
    }
    __syncthreads();
    if (threadIdx.x < kRowsT && r0 + threadIdx.x < rows) {
        Best bb = red[threadIdx.x][0];
        for (int w2 = 1; w2 < kCols / 32; ++w2) bb = better(bb, red[threadIdx.x][w2]);
        const int64_t o = (int64_t)(r0 + threadIdx.x) * ntiles + vt;
        part_v[o] = bb.v;
        part_i[o] = bb.i;
    }
}

__global__ void accept_finalize_kernel(const float *part_v, const int *part_i, int ntiles, int n_pred,
                                       const int32_t *drafts, int x, int32_t *verified,
                                       int32_t *accept_len, int32_t *emitted) {
    extern __shared__ int32_t ver[];  // [n_pred]
    const int b = blockIdx.x;
    for (int i = threadIdx.x; i < n_pred; i += blockDim.x) {
        const int64_t r = (int64_t)b * n_pred + i;
        Best bb = {part_v[r * ntiles], part_i[r * ntiles]};
        for (int tt = 1; tt < ntiles; ++tt) bb = better(bb, Best{part_v[r * ntiles + tt], part_i[r * ntiles + tt]});
        ver[i] = bb.i;
        verified[r] = bb.i;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const int32_t *dr = drafts + (int64_t)b * x;
        int a = 0;
        while (a < x && a < n_pred && dr[a] == ver[a]) ++a;
        accept_len[b] = a;
        int32_t *em = emitted + (int64_t)b * (x + 1);
        int ne = 0;
        for (int j = 0; j < a; ++j) em[ne++] = dr[j];
        if (a < n_pred) em[ne++] = ver[a];
        for (int j = ne; j < x + 1; ++j) em[j] = -1;
    }
}

}  // namespace

size_t accept_workspace(int batch, int n_pred, int vocab, int d) {
    const int ntiles = ceil_div(vocab, kCols);
    return (size_t)batch * n_pred * ntiles * (sizeof(float) + sizeof(int)) + (size_t)batch * n_pred * d * sizeof(float);
}

cudaError_t accept_launch(const float *hidden, int batch, int n_pred, int hg, const float *w, int d,
                          int vocab, const int32_t *drafts, int x, int32_t *verified, int32_t *accept_len,
                          int32_t *emitted, void *ws, cudaStream_t st) {
    const int ntiles = ceil_div(vocab, kCols);
    const int rows = batch * n_pred;
    float *pv = (float *)ws;
    int *pi = (int *)(pv + (size_t)rows * ntiles);
    float *h = reinterpret_cast<float *>(pi + (size_t)rows * ntiles);
    const int64_t nh = (int64_t)rows * d;
    group_mean_kernel<<<(unsigned)((nh + 255) / 256), 256, 0, st>>>(hidden, rows, hg, d, h);
    dim3 grid(ntiles, ceil_div(rows, kRowsT));
    logits_argmax_kernel<<<grid, kCols, 0, st>>>(h, rows, w, d, vocab, pv, pi, ntiles);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    accept_finalize_kernel<<<batch, 128, n_pred * sizeof(int32_t), st>>>(pv, pi, ntiles, n_pred, drafts, x,
                                                                         verified, accept_len, emitted);
    return cudaGetLastError();
}

}  // namespace vc
