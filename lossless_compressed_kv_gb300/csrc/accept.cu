// vc_accept: greedy acceptance of one verification round.
//
// "VeriCache: Making Lossy KV Compression Exact", section "The Core Idea":
// the verifier's predictions are compared with the drafts left to right; at
// the first mismatch the matched prefix and the verifier's own token are
// emitted (the rest of the draft is discarded); when every draft matches
// the draft is emitted together with the verifier's extra (bonus) token.
//
// Kernel 1 (prepass): the mean of each row's hidden group, and the row's
// argmax key reset.  Kernel 2: logits of 16 prediction rows x 512
// vocabulary columns per CTA (a 16 x 4 register tile per thread, the row
// values of one hidden dimension read as four 16-byte shared loads), each
// logit fp32 with one fused multiply-add per term in increasing k (so a
// row's logits are the same bits whatever the batch or the number of rows);
// the tile's best column per row goes into the row's 64-bit key with
// atomicMax (larger value wins, lower id on ties).  Kernel 3: per request,
// the prefix rule.
#include "vc_internal.cuh"

namespace vc {
namespace {

constexpr int kThreadsL = 128;        // logits CTA
constexpr int kColsT = 4;             // vocabulary columns per thread
constexpr int kCols = kThreadsL * kColsT;
constexpr int kRowsT = 16;            // prediction rows per CTA
constexpr int kKT = 128;              // hidden dims staged per step
constexpr int kKU = 8;                // hidden dims whose W loads are in flight together

// Order-preserving key: value bits mapped to an unsigned order in the high
// word (-0 folded onto +0 first), the complement of the id in the low word.
__device__ inline unsigned long long argmax_key(float v, int id) {
    uint32_t b = __float_as_uint(v + 0.0f);
    b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return ((unsigned long long)b << 32) | (uint32_t)(~(uint32_t)id);
}

// h[r][k] = (sum_j hidden[r][j][k], in increasing j) / hg, once per row.
__global__ void group_mean_kernel(const float *hidden, int rows, int hg, int d, float *h,
                                  unsigned long long *keys) {
    pdl_begin();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (keys && i < rows) keys[i] = 0ull;
    if (i >= (int64_t)rows * d) return;
    const int64_t r = i / d, k = i % d;
    const float *hp = hidden + (r * hg) * d + k;
    float s = 0.0f;
    for (int j = 0; j < hg; ++j) s = __fadd_rn(s, hp[(int64_t)j * d]);
    h[i] = __fdiv_rn(s, (float)hg);
}

// Two rows' terms of one column in one packed instruction: lane i computes
// fma(h_i, w, acc_i) rounded to nearest, the same as two scalar fmaf.
__device__ __forceinline__ void fma_rows2(float &a0, float &a1, float h0, float h1, float w) {
    asm("{\n\t.reg .b64 ra, rh, rw;\n\t"
        "mov.b64 ra, {%0, %1};\n\t"
        "mov.b64 rh, {%2, %3};\n\t"
        "mov.b64 rw, {%4, %4};\n\t"
        "fma.rn.f32x2 ra, rh, rw, ra;\n\t"
        "mov.b64 {%0, %1}, ra;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(h0), "f"(h1), "f"(w));
}

// STORE: write the logits [rows][vocab] instead of the argmax keys.
template <bool STORE>
__global__ void __launch_bounds__(kThreadsL) logits_argmax_kernel(const float *h, int rows, const float *w, int d,
                                                                 int vocab, unsigned long long *keys,
                                                                 float *logits) {
    pdl_begin();
    __shared__ __align__(16) float hs[kKT][kRowsT];  // k-major: one k's 16 row values contiguous
    const int r0 = blockIdx.y * kRowsT;
    const int v0 = blockIdx.x * kCols + threadIdx.x * kColsT;
    const bool vec = (vocab % 4 == 0) && ((reinterpret_cast<uintptr_t>(w) & 15) == 0);
    float acc[kRowsT][kColsT];
#pragma unroll
    for (int r = 0; r < kRowsT; ++r)
#pragma unroll
        for (int c = 0; c < kColsT; ++c) acc[r][c] = 0.0f;
    for (int k0 = 0; k0 < d; k0 += kKT) {
        const int kn = min(kKT, d - k0);
        __syncthreads();
        for (int e = threadIdx.x; e < kRowsT * kKT; e += kThreadsL) {
            const int r = e / kKT, k = e % kKT;
            hs[k][r] = (r0 + r < rows && k < kn) ? h[(int64_t)(r0 + r) * d + k0 + k] : 0.0f;
        }
        __syncthreads();
        // kKU hidden dims per step: the W loads of all of them issued first
        // (enough loads in flight to cover the L2 latency)
        for (int kk = 0; kk < kn; kk += kKU) {
            float wv[kKU][kColsT];
#pragma unroll
            for (int u = 0; u < kKU; ++u) {
                const float *wp = w + (int64_t)(k0 + kk + u) * vocab + v0;
                if (kk + u < kn && vec && v0 + kColsT <= vocab) {
                    const float4 q4 = *reinterpret_cast<const float4 *>(wp);
                    wv[u][0] = q4.x; wv[u][1] = q4.y; wv[u][2] = q4.z; wv[u][3] = q4.w;
                } else {
#pragma unroll
                    for (int c = 0; c < kColsT; ++c) wv[u][c] = (kk + u < kn && v0 + c < vocab) ? wp[c] : 0.0f;
                }
            }
#pragma unroll
            for (int u = 0; u < kKU; ++u) {
                if (kk + u >= kn) break;
                float hv[kRowsT];
#pragma unroll
                for (int i = 0; i < kRowsT / 4; ++i) {
                    const float4 q4 = reinterpret_cast<const float4 *>(hs[kk + u])[i];
                    hv[4 * i] = q4.x; hv[4 * i + 1] = q4.y; hv[4 * i + 2] = q4.z; hv[4 * i + 3] = q4.w;
                }
#pragma unroll
                for (int r = 0; r < kRowsT; r += 2)
#pragma unroll
                    for (int c = 0; c < kColsT; ++c) fma_rows2(acc[r][c], acc[r + 1][c], hv[r], hv[r + 1], wv[u][c]);
            }
        }
    }
    if constexpr (STORE) {
#pragma unroll
        for (int r = 0; r < kRowsT; ++r)
            if (r0 + r < rows)
#pragma unroll
                for (int c = 0; c < kColsT; ++c)
                    if (v0 + c < vocab) logits[(int64_t)(r0 + r) * vocab + v0 + c] = acc[r][c];
        return;
    }
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int r = 0; r < kRowsT; ++r) {
        unsigned long long best = 0ull;
#pragma unroll
        for (int c = 0; c < kColsT; ++c)
            if (v0 + c < vocab) {
                const unsigned long long kc = argmax_key(acc[r][c], v0 + c);
                best = kc > best ? kc : best;
            }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
            best = o > best ? o : best;
        }
        if (lane == 0 && r0 + r < rows && best) atomicMax(&keys[r0 + r], best);
    }
}

// The same logits for up to MR rows (decode and draft steps of a small
// batch): one vocabulary column per thread, each row's fp32 FMA chain in
// increasing k as in the tiled kernel (bit-identical logits), one warp per
// 32 columns with its W tile (kLK rows x 32 columns, fp32) staged in shared
// memory by asynchronous 16-byte copies one chunk ahead.  The tiled kernel
// spends a 16-row tile on a handful of rows and keeps few bytes in flight.
constexpr int kLRows = 16;
constexpr int kLCols = 32;
constexpr int kLK = 128;
__device__ inline void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
template <int MR, bool STORE>
__global__ void __launch_bounds__(kLCols) logits_rows_kernel(const float *h, int rows, const float *w, int d,
                                                            int vocab, unsigned long long *keys, float *logits) {
    pdl_begin();
    __shared__ __align__(16) float hs[kLK][MR];
    __shared__ __align__(16) float ws[2][kLK][kLCols];
    const int lane = threadIdx.x;
    const int c0 = blockIdx.x * kLCols, c = c0 + lane;
    const int nchunk = ceil_div(d, kLK);
    const bool vec = (vocab % 4 == 0) && ((reinterpret_cast<uintptr_t>(w) & 15) == 0);
    auto load_w = [&](int buf, int k0) {
        for (int e = lane; e < kLK * (kLCols / 4); e += kLCols) {
            const int kk = e / (kLCols / 4), q = e % (kLCols / 4);
            const int kr = k0 + kk, cq = c0 + 4 * q;
            float *dst = &ws[buf][kk][4 * q];
            if (vec && kr < d && cq + 4 <= vocab) {
                cp_async16(dst, w + (int64_t)kr * vocab + cq);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) dst[j] = (kr < d && cq + j < vocab) ? w[(int64_t)kr * vocab + cq + j] : 0.0f;
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    float acc[MR];
#pragma unroll
    for (int r = 0; r < MR; ++r) acc[r] = 0.0f;
    load_w(0, 0);
    for (int i = 0; i < nchunk; ++i) {
        const int k0 = i * kLK, kn = min(kLK, d - k0);
        if (i + 1 < nchunk) load_w((i + 1) & 1, k0 + kLK);
        for (int e = lane; e < kn * MR; e += kLCols) {
            const int kk = e / MR, r = e % MR;
            hs[kk][r] = r < rows ? h[(int64_t)r * d + k0 + kk] : 0.0f;
        }
        if (i + 1 < nchunk)
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        else
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();
        const float(*wt)[kLCols] = ws[i & 1];
#pragma unroll 8
        for (int kk = 0; kk < kn; ++kk) {
            const float wv = wt[kk][lane];
#pragma unroll
            for (int r = 0; r < MR; ++r) acc[r] = fmaf(hs[kk][r], wv, acc[r]);
        }
        __syncthreads();
    }
    if constexpr (STORE) {
        if (c < vocab)
#pragma unroll
            for (int r = 0; r < MR; ++r)
                if (r < rows) logits[(int64_t)r * vocab + c] = acc[r];
        return;
    }
#pragma unroll
    for (int r = 0; r < MR; ++r) {
        if (r >= rows) break;
        unsigned long long best = c < vocab ? argmax_key(acc[r], c) : 0ull;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
            best = o > best ? o : best;
        }
        if (lane == 0 && best) atomicMax(&keys[r], best);
    }
}

// Logits (argmax keys, or stored) of `rows` prediction rows.
template <bool STORE>
void launch_logits(const float *h, int rows, const float *w, int d, int vocab, unsigned long long *keys,
                   float *logits, cudaStream_t st) {
    if (rows <= kLRows) {
        const dim3 grid(ceil_div(vocab, kLCols));
        if (rows <= 4)
            launch_pdl(logits_rows_kernel<4, STORE>, grid, kLCols, 0, st, h, rows, w, d, vocab, keys, logits);
        else if (rows <= 8)
            launch_pdl(logits_rows_kernel<8, STORE>, grid, kLCols, 0, st, h, rows, w, d, vocab, keys, logits);
        else
            launch_pdl(logits_rows_kernel<16, STORE>, grid, kLCols, 0, st, h, rows, w, d, vocab, keys, logits);
        return;
    }
    dim3 grid(ceil_div(vocab, kCols), ceil_div(rows, kRowsT));
    launch_pdl(logits_argmax_kernel<STORE>, grid, kThreadsL, 0, st, h, rows, w, d, vocab, keys, logits);
}

__global__ void accept_finalize_kernel(const unsigned long long *keys, int n_pred, const int32_t *drafts, int x,
                                       int32_t *verified, int32_t *accept_len, int32_t *emitted) {
    pdl_begin();
    extern __shared__ int32_t ver[];  // [n_pred]
    const int b = blockIdx.x;
    for (int i = threadIdx.x; i < n_pred; i += blockDim.x) {
        const int64_t r = (int64_t)b * n_pred + i;
        const int32_t id = (int32_t)~(uint32_t)(keys[r] & 0xffffffffull);
        ver[i] = id;
        verified[r] = id;
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

// ---------------------------------------------------------------------------
// Rejection-sampling acceptance ("VeriCache Guide", "Mathematical Guarantee
// of Lossless Correctness"): one CTA per request walks its drafts in order;
// softmax(logits / tau) statistics by block reductions in fp32; a rejected
// draft (or the bonus) is drawn by an inverse CDF over the residual (or the
// target) distribution: per-thread contiguous chunks, a block scan of the
// chunk sums, then the owning thread walks its chunk.
// ---------------------------------------------------------------------------
constexpr int kSampThreads = 512;

__device__ float block_reduce(float x, bool is_max, float *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, x, off);
        x = is_max ? fmaxf(x, o) : x + o;
    }
    __syncthreads();
    if (lane == 0) red[warp] = x;
    __syncthreads();
    if (warp == 0) {
        x = lane < kSampThreads / 32 ? red[lane] : (is_max ? -INFINITY : 0.0f);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float o = __shfl_xor_sync(0xffffffffu, x, off);
            x = is_max ? fmaxf(x, o) : x + o;
        }
        if (lane == 0) red[32] = x;
    }
    __syncthreads();
    return red[32];
}

struct RowStats {
    float m, z;  // max of logits / tau, sum of exp(logits / tau - m)
};

__device__ RowStats row_stats(const float *l, int vocab, float tau, float *red) {
    float mx = -INFINITY;
    for (int j = threadIdx.x; j < vocab; j += kSampThreads) mx = fmaxf(mx, __fdiv_rn(l[j], tau));
    RowStats r;
    r.m = block_reduce(mx, true, red);
    float z = 0.0f;
    for (int j = threadIdx.x; j < vocab; j += kSampThreads) z += __expf(__fdiv_rn(l[j], tau) - r.m);
    r.z = block_reduce(z, false, red);
    return r;
}

__device__ inline float prob(const float *l, int j, float tau, RowStats s) {
    return __expf(__fdiv_rn(l[j], tau) - s.m) / s.z;
}

// Inverse CDF over weights w(j) >= 0: the first j whose cumulative weight
// exceeds u * total (the last positive weight if rounding leaves none).
template <class W>
__device__ int draw(W w, int vocab, float u, float *red, float *scan, int *pick) {
    const int chunk = (vocab + kSampThreads - 1) / kSampThreads;
    const int c0 = min(vocab, threadIdx.x * chunk), c1 = min(vocab, c0 + chunk);
    float cs = 0.0f;
    int lastpos = -1;
    for (int j = c0; j < c1; ++j) {
        const float x = w(j);
        if (x > 0.0f) {
            cs += x;
            lastpos = j;
        }
    }
    scan[threadIdx.x] = cs;
    if (threadIdx.x == 0) {
        pick[0] = vocab;
        pick[1] = -1;
    }
    __syncthreads();
    if (threadIdx.x == 0) {  // exclusive prefix of the chunk sums, in thread order
        float run = 0.0f;
        for (int i = 0; i < kSampThreads; ++i) {
            const float c = scan[i];
            scan[i] = run;
            run += c;
        }
        red[33] = run;
    }
    __syncthreads();
    atomicMax(&pick[1], lastpos);
    const float thr = u * red[33];
    float cum = scan[threadIdx.x];
    if (cs > 0.0f && cum <= thr && thr < cum + cs) {
        for (int j = c0; j < c1; ++j) {
            const float x = w(j);
            if (x > 0.0f) {
                cum += x;
                if (cum > thr) {
                    atomicMin(&pick[0], j);
                    break;
                }
            }
        }
    }
    __syncthreads();
    const int r = pick[0] < vocab ? pick[0] : max(pick[1], 0);
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kSampThreads) accept_sample_kernel(const float *tl, const float *dl, int vocab,
                                                                    float tau, const int32_t *drafts, int x,
                                                                    const float *u, const float *v,
                                                                    int32_t *accept_len, int32_t *emitted) {
    pdl_begin();
    __shared__ float red[34];
    __shared__ float scan[kSampThreads];
    __shared__ int pick[2];
    const int b = blockIdx.x;
    const float *T = tl + (int64_t)b * (x + 1) * vocab;
    const float *Dl = dl + (int64_t)b * x * vocab;
    int32_t *em = emitted + (int64_t)b * (x + 1);
    int a = 0, ne = 0;
    for (; a < x; ++a) {
        const float *lt = T + (int64_t)a * vocab, *ld = Dl + (int64_t)a * vocab;
        const RowStats st = row_stats(lt, vocab, tau, red), sd = row_stats(ld, vocab, tau, red);
        const int d = drafts[(int64_t)b * x + a];
        float alpha = 0.0f;  // an out-of-range draft id is rejected
        if (d >= 0 && d < vocab) {
            const float pt = prob(lt, d, tau, st), pd = prob(ld, d, tau, sd);
            alpha = pd > 0.0f ? fminf(1.0f, pt / pd) : 1.0f;
        }
        if (u[(int64_t)b * x + a] < alpha) {
            if (threadIdx.x == 0) em[ne] = d;
            ++ne;
            continue;
        }
        const int t = draw([&](int j) { return fmaxf(0.0f, prob(lt, j, tau, st) - prob(ld, j, tau, sd)); },
                           vocab, v[(int64_t)b * (x + 1) + a], red, scan, pick);
        if (threadIdx.x == 0) em[ne] = t;
        ++ne;
        break;
    }
    if (a == x) {
        const float *lt = T + (int64_t)x * vocab;
        const RowStats st = row_stats(lt, vocab, tau, red);
        const int t = draw([&](int j) { return prob(lt, j, tau, st); }, vocab, v[(int64_t)b * (x + 1) + x], red,
                           scan, pick);
        if (threadIdx.x == 0) em[ne] = t;
        ++ne;
    }
    if (threadIdx.x == 0) {
        accept_len[b] = a;
        for (int j = ne; j < x + 1; ++j) em[j] = -1;
    }
}

}  // namespace

size_t accept_workspace(int batch, int n_pred, int vocab, int d) {
    (void)vocab;
    const size_t rows = (size_t)batch * n_pred;
    return rows * sizeof(unsigned long long) + rows * d * sizeof(float);
}

cudaError_t accept_launch(const float *hidden, int batch, int n_pred, int hg, const float *w, int d,
                          int vocab, const int32_t *drafts, int x, int32_t *verified, int32_t *accept_len,
                          int32_t *emitted, void *ws, cudaStream_t st) {
    const int rows = batch * n_pred;
    unsigned long long *keys = reinterpret_cast<unsigned long long *>(ws);
    float *h = reinterpret_cast<float *>(keys + rows);
    const int64_t nh = (int64_t)rows * d;
    launch_pdl(group_mean_kernel, (unsigned)((nh + 255) / 256), 256, 0, st, hidden, rows, hg, d, h, keys);
    launch_logits<false>(h, rows, w, d, vocab, keys, nullptr, st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    launch_pdl(accept_finalize_kernel, batch, 128, n_pred * sizeof(int32_t), st, keys, n_pred, drafts, x, verified,
               accept_len, emitted);
    return cudaGetLastError();
}

}  // namespace vc

namespace vc {

size_t accept_sampled_workspace(int batch, int x, int vocab, int d) {
    const size_t rt = (size_t)batch * (x + 1), rd = (size_t)batch * x;
    return (rt + rd) * (size_t)d * sizeof(float) + (rt + rd) * (size_t)vocab * sizeof(float);
}

cudaError_t accept_sampled_launch(const float *target_hidden, const float *draft_hidden, int batch, int x, int hg,
                                  const float *w, int d, int vocab, float tau, const int32_t *drafts,
                                  const float *u, const float *v, int32_t *accept_len, int32_t *emitted, void *ws,
                                  cudaStream_t st) {
    const int rt = batch * (x + 1), rd = batch * x;
    float *ht = reinterpret_cast<float *>(ws);
    float *hd = ht + (size_t)rt * d;
    float *lt = hd + (size_t)rd * d;
    float *ld = lt + (size_t)rt * vocab;
    launch_pdl(group_mean_kernel, (unsigned)(((int64_t)rt * d + 255) / 256), 256, 0, st, target_hidden, rt, hg, d,
               ht, nullptr);
    launch_logits<true>(ht, rt, w, d, vocab, nullptr, lt, st);
    if (rd > 0) {
        launch_pdl(group_mean_kernel, (unsigned)(((int64_t)rd * d + 255) / 256), 256, 0, st, draft_hidden, rd, hg,
                   d, hd, nullptr);
        launch_logits<true>(hd, rd, w, d, vocab, nullptr, ld, st);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    launch_pdl(accept_sample_kernel, batch, kSampThreads, 0, st, lt, ld, vocab, tau, drafts, x, u, v, accept_len,
               emitted);
    return cudaGetLastError();
}

}  // namespace vc
