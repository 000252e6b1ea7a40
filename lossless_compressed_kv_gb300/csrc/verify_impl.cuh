// Device body of the verification attention (shared by the verify launch
// and the mixed draft/verify launch).  See verify_attn.cu for the design.
#pragma once

#include "vc_internal.cuh"

namespace vc {
namespace verify {


constexpr int kWarps = 8;               // warps per CTA in the mixed launch
constexpr int kRows = kWarps * 16;      // rows per CTA in the mixed launch
constexpr int kMaxWarps = 16;           // standalone launch: one warp per m16 row tile
constexpr int kSplitPages = 256;        // 4096 keys per split (fixed)
constexpr int kStages = 4;

struct VerifyArgs {
    const uint16_t *q;  // [B][n_q][Hq][D]
    const uint8_t *kp, *vp;
    int64_t n_pages;
    const int32_t *table, *lens;
    int maxb;
    int n_q, hq, hkv, grp;
    float scale_log2;
    int n_splits;
    float *ws_o;   // [B][n_q][Hq][n_splits][D]
    float *ws_ml;  // [B][n_q][Hq][n_splits][2]
    int32_t *status;
};

template <int D>
struct VCfg {
    static constexpr int TILE = kPage * D * 2;      // one K or V head block
    static constexpr int STAGE = 2 * TILE;
    static constexpr int CHUNKS = D / 8;            // 16-byte chunks per row
    static constexpr int SMEM = kStages * STAGE;
};

// swizzled byte offset of (row, 16-byte chunk) inside a [16][D] bf16 tile
template <int D>
__device__ inline int swz(int row, int chunk) {
    return row * D * 2 + ((chunk ^ (row & 7)) << 4);
}

template <int D>
__device__ __forceinline__ void verify_block(const VerifyArgs &a, int split, int rb, int bk, uint8_t *smem) {
    using C = VCfg<D>;
    constexpr int NT = D / 16;  // k-steps of QK
    constexpr int NO = D / 8;   // n-tiles of PV output
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int b = bk / a.hkv, kvh = bk % a.hkv;
    const int len = a.lens[b];
    const int nrows = a.n_q * a.grp;
    const int nthreads = blockDim.x;
    const int row0 = rb * (nthreads / 32) * 16 + warp * 16;
    const bool len_ok = len >= a.n_q;
    if (!len_ok && threadIdx.x == 0 && split == 0 && rb == 0 && kvh == 0) report(a.status, VC_ERR_BAD_INDEX);
    const int npages = len_ok ? ceil_div(len, kPage) : 0;
    const int p0 = split * kSplitPages;
    const int p1 = min(p0 + kSplitPages, npages);
    const int np = max(0, p1 - p0);
    const int32_t *trow = a.table + (int64_t)b * a.maxb;

    // rows g and g+8 of this warp's tile
    int qpos[2];
    bool rvalid[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int r = row0 + g + 8 * h;
        rvalid[h] = r < nrows;
        const int i = rvalid[h] ? r / a.grp : 0;
        qpos[h] = len - a.n_q + i;
    }
    // Q fragments (A operand), row r = (query i, head n) with r = i * grp + n
    uint32_t qa[NT][4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int r = row0 + g + 8 * h;
        const uint16_t *qr = nullptr;
        if (rvalid[h]) {
            const int i = r / a.grp, n = r % a.grp;
            qr = a.q + (((int64_t)b * a.n_q + i) * a.hq + kvh * a.grp + n) * D;
        }
#pragma unroll
        for (int ks = 0; ks < NT; ++ks) {
            qa[ks][h] = qr ? *reinterpret_cast<const uint32_t *>(qr + 16 * ks + 2 * t) : 0u;
            qa[ks][h + 2] = qr ? *reinterpret_cast<const uint32_t *>(qr + 16 * ks + 2 * t + 8) : 0u;
        }
    }

    auto load_page = [&](int k) {  // all threads: page p0 + k into stage k % kStages
        uint8_t *st = smem + (k % kStages) * C::STAGE;
        const int pg = p0 + k;
        const int id = pg < a.maxb ? trow[pg] : -1;
        const bool ok = id >= 0 && id < a.n_pages;
        if (!ok && threadIdx.x == 0) report(a.status, VC_ERR_BAD_INDEX);
        const int64_t off = ((int64_t)(ok ? id : 0) * a.hkv + kvh) * C::TILE;
        for (int c = threadIdx.x; c < 2 * kPage * C::CHUNKS; c += nthreads) {
            const int kv = c / (kPage * C::CHUNKS);
            const int rem = c % (kPage * C::CHUNKS);
            const int row = rem / C::CHUNKS, ch = rem % C::CHUNKS;
            const uint8_t *src = (kv ? a.vp : a.kp) + off + row * D * 2 + ch * 16;
            uint8_t *dst = st + kv * C::TILE + swz<D>(row, ch);
            // slots past the request length are zero-filled: their bytes may be
            // anything (even NaN patterns) and 0 * NaN would leak into P V
            if (ok && pg * kPage + row < len) cp_async16(dst, src); else cp_async_zero16(dst, src);
        }
    };

    float o[NO][4];
#pragma unroll
    for (int i = 0; i < NO; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.0f, 0.0f};

#pragma unroll
    for (int k = 0; k < kStages - 1; ++k) {
        if (k < np) load_page(k);
        cp_async_commit();
    }
    for (int k = 0; k < np; ++k) {
        cp_async_wait<kStages - 2>();
        __syncthreads();
        if (k + kStages - 1 < np) load_page(k + kStages - 1);
        cp_async_commit();
        const uint8_t *kt = smem + (k % kStages) * C::STAGE;
        const uint8_t *vt = kt + C::TILE;
        const int kbase = (p0 + k) * kPage;
        // ---- S = Q K^T (16 rows x 16 keys) ----
        float s[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.0f;
        {
            const int mi = lane >> 3, r = lane & 7;
            const int key = (mi >> 1) * 8 + r;
#pragma unroll
            for (int ks = 0; ks < NT; ++ks) {
                uint32_t bk[4];
                ldsm_x4(bk, kt + swz<D>(key, 2 * ks + (mi & 1)));
                mma_bf16(s[0], qa[ks], bk[0], bk[1]);
                mma_bf16(s[1], qa[ks], bk[2], bk[3]);
            }
        }
        // ---- scale, causal / length mask, online softmax per row ----
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int h = e >> 1;
                const int key = kbase + 8 * j + 2 * t + (e & 1);
                float v = s[j][e] * a.scale_log2;
                if (!rvalid[h] || key > qpos[h] || key >= len) v = -INFINITY;
                s[j][e] = v;
                mx[h] = fmaxf(mx[h], v);
            }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
        }
        const float mn0 = fmaxf(m[0], mx[0]), mn1 = fmaxf(m[1], mx[1]);
        if (__any_sync(0xffffffffu, mn0 > m[0] || mn1 > m[1])) {
            const float al0 = mn0 == -INFINITY ? 1.0f : ex2(m[0] - mn0);
            const float al1 = mn1 == -INFINITY ? 1.0f : ex2(m[1] - mn1);
#pragma unroll
            for (int i = 0; i < NO; ++i) {
                o[i][0] *= al0; o[i][1] *= al0;
                o[i][2] *= al1; o[i][3] *= al1;
            }
            l[0] *= al0;
            l[1] *= al1;
            m[0] = mn0;
            m[1] = mn1;
        }
        const float ms[2] = {m[0] == -INFINITY ? 0.0f : m[0], m[1] == -INFINITY ? 0.0f : m[1]};
        uint32_t pa[4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const float p0v = ex2(s[j][0] - ms[0]), p1v = ex2(s[j][1] - ms[0]);
            const float p2v = ex2(s[j][2] - ms[1]), p3v = ex2(s[j][3] - ms[1]);
            l[0] += p0v + p1v;
            l[1] += p2v + p3v;
            pa[2 * j] = pack_bf16(p0v, p1v);      // row g,   keys 8j + 2t, +1
            pa[2 * j + 1] = pack_bf16(p2v, p3v);  // row g+8
        }
        // ---- O += P V ----
        {
            const uint32_t af[4] = {pa[0], pa[1], pa[2], pa[3]};
            const int mi = lane >> 3, r = lane & 7;
            const int key = (mi & 1) * 8 + r;
#pragma unroll
            for (int jj = 0; jj < NO / 2; ++jj) {
                uint32_t bv[4];
                ldsm_x4_t(bv, vt + swz<D>(key, 2 * jj + (mi >> 1)));
                mma_bf16(o[2 * jj], af, bv[0], bv[1]);
                mma_bf16(o[2 * jj + 1], af, bv[2], bv[3]);
            }
        }
    }
    cp_async_wait<0>();

    // ---- write this split's partial rows ----
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float lt = l[h];
        lt += __shfl_xor_sync(0xffffffffu, lt, 1);
        lt += __shfl_xor_sync(0xffffffffu, lt, 2);
        const int r = row0 + g + 8 * h;
        if (!rvalid[h]) continue;
        const int i = r / a.grp, n = r % a.grp;
        const int64_t row = (((int64_t)b * a.n_q + i) * a.hq + kvh * a.grp + n) * a.n_splits + split;
        float *dst = a.ws_o + row * D;
#pragma unroll
        for (int j = 0; j < NO; ++j)
            *reinterpret_cast<float2 *>(dst + 8 * j + 2 * t) = make_float2(o[j][2 * h], o[j][2 * h + 1]);
        if (t == 0) {
            a.ws_ml[row * 2] = m[h];
            a.ws_ml[row * 2 + 1] = lt;
        }
    }
}

// Combine the splits of one row in split order.
template <int D>
__device__ __forceinline__ void reduce_row(const float *ws_o, const float *ws_ml, int n_splits, int64_t row,
                                           float *out, int tid, int nthreads) {
    const float *ml = ws_ml + row * n_splits * 2;
    float M = -INFINITY;
    for (int s = 0; s < n_splits; ++s) M = fmaxf(M, ml[2 * s]);
    for (int c = tid; c < D; c += nthreads) {
        float acc = 0.0f, L = 0.0f;
        if (M != -INFINITY) {
            for (int s = 0; s < n_splits; ++s) {
                const float f = ex2(ml[2 * s] - M);
                acc += f * ws_o[(row * n_splits + s) * D + c];
                L += f * ml[2 * s + 1];
            }
        }
        out[row * D + c] = L > 0.0f ? acc / L : 0.0f;
    }
}

}  // namespace verify
}  // namespace vc
