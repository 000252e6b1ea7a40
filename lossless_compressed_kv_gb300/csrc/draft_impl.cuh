// Device body of the draft attention (shared by the draft launch and the
// mixed draft/verify launch).  See draft_attn.cu for the design notes.
#pragma once

#include "vc_internal.cuh"

namespace vc {
namespace draft {


struct DraftArgs {
    const uint16_t *q;  // [B][Hq][D] bf16
    const uint8_t *kp, *vp;
    int64_t n_pages;
    const int32_t *table, *lens;
    int maxb;
    int hq, hkv, grp;
    float scale_log2;
    int chunk_pages, n_splits;
    float *ws_o;   // [B][Hq][n_splits][D]
    float *ws_ml;  // [B][Hq][n_splits][2]
    int32_t *status;
};

template <int BITS, int D, int NW>
struct Cfg {
    static constexpr int NT = D / 16;
    static constexpr int NG = D / 32;
    static constexpr int HB = BITS == 16 ? kPage * D * 2 : 2 * D * (BITS + 1);
    static constexpr int CB = BITS == 16 ? D * 2 : D * BITS / 8;  // bytes per token row
    static constexpr int WPR = CB / 4;                            // 32-bit words per row
    static constexpr int NSTAGE = BITS == 16 ? 3 : 4;
    static constexpr int STAGE = 2 * HB;
    static constexpr int RING = NW * NSTAGE * STAGE;
    static constexpr int COMBINE = NW * 8 * (D + 2) * 4;
    static constexpr int BARS = NW * NSTAGE * 8;
    static constexpr int QS = 8 * D * 2 + 8 * NG * 4;  // q of the group (bf16) + its group sums
    static constexpr int SMEM = (RING > COMBINE ? RING : COMBINE) + BARS + QS;
};

// Load one token row of packed codes (CB bytes) as 32-bit words.
template <int CB>
__device__ inline void load_row(uint32_t (&w)[CB / 4], const uint8_t *p) {
    if constexpr (CB % 16 == 0) {
#pragma unroll
        for (int i = 0; i < CB / 16; ++i) {
            uint4 u = reinterpret_cast<const uint4 *>(p)[i];
            w[4 * i] = u.x; w[4 * i + 1] = u.y; w[4 * i + 2] = u.z; w[4 * i + 3] = u.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < CB / 8; ++i) {
            uint2 u = reinterpret_cast<const uint2 *>(p)[i];
            w[2 * i] = u.x; w[2 * i + 1] = u.y;
        }
    }
}

// 3-bit: the 48 bits of channels [16 j, 16 j + 16) of a row, right-aligned.
template <int WPR>
__device__ inline uint64_t win3(const uint32_t (&w)[WPR], int j) {
    const int wi = (3 * j) >> 1;
    uint64_t x = ((uint64_t)w[wi + 1] << 32) | w[wi];
    return (j & 1) ? (x >> 16) : x;
}

// Codes enter the MMA as f16 subnormals: a code c masked in place at bit p
// of a 16-bit half is the f16 value c * 2^(p - 24), exact (the tensor cores
// do not flush subnormal operands).  The query operand of those k-slots is
// pre-scaled by 2^-p, so every product is c * q * 2^-24 and the group scale
// carries the 2^24.  Per-thread shift s and in-half positions (pl for
// k-slots 2t, 2t+1; ph for 2t+8, 2t+9) keep every masked code below 2^10.
template <int BITS>
struct KPos {
    int s, pl, ph;
    __device__ explicit KPos(int t) {
        if constexpr (BITS == 2) {
            s = t < 2 ? 0 : (t == 2 ? 2 : 6);
            pl = 4 * t - s;
            ph = pl + 2;
        } else if constexpr (BITS == 4) {
            s = t < 2 ? 0 : 4 * t - 4;
            pl = ph = 4 * t - s;
        } else {
            s = 0;
            pl = ph = 0;
        }
    }
};

// K operand (A, rows = tokens) for k-step ks from one token row's words; the
// k-slot -> channel map of each bit width is mirrored by q_channel().
template <int BITS, int WPR>
__device__ inline void k_pair(const uint32_t (&w)[WPR], int ks, int t, const KPos<BITS> &kp, uint32_t &lo,
                              uint32_t &hi) {
    if constexpr (BITS == 2) {
        const uint32_t y = w[ks] >> kp.s;  // channels (2t, 2t+8) at pl, (2t+1, 2t+9) at ph
        lo = y & (0x00030003u << kp.pl);
        hi = y & (0x00030003u << kp.ph);
    } else if constexpr (BITS == 4) {
        lo = (w[2 * ks] >> kp.s) & (0x000F000Fu << kp.pl);      // channels (t, t+4)
        hi = (w[2 * ks + 1] >> kp.s) & (0x000F000Fu << kp.pl);  // channels (8+t, 12+t)
    } else {  // 3
        const uint64_t x = win3<WPR>(w, ks);
        lo = (uint32_t)((x >> (6 * t)) & 7u) | ((uint32_t)((x >> (6 * t + 24)) & 7u) << 16);
        hi = (uint32_t)((x >> (6 * t + 3)) & 7u) | ((uint32_t)((x >> (6 * t + 27)) & 7u) << 16);
    }
}

// Channel read by k-slot `slot` (0..15) of k-step ks.
template <int BITS>
__device__ inline int q_channel(int ks, int slot) {
    const int t = (slot & 7) >> 1, odd = slot & 1, upper = slot >> 3;
    if constexpr (BITS == 4) {
        // slots (2t, 2t+1) -> (t, t+4); (2t+8, 2t+9) -> (8+t, 12+t)
        return 16 * ks + (upper ? 8 : 0) + t + (odd ? 4 : 0);
    } else if constexpr (BITS == 16) {
        // per pair of k-steps, thread t holds channels 8t..8t+7 of a 32-block
        const int kk = ks >> 1, second = ks & 1;
        return 32 * kk + 8 * t + 4 * second + 2 * upper + odd;
    } else {
        // 2 and 3 bits: (2t, 2t+1) -> (2t, 2t+8); (2t+8, 2t+9) -> (2t+1, 2t+9)
        return 16 * ks + 2 * t + upper + (odd ? 8 : 0);
    }
}

// V operand (A, rows = channels of m-tile mt, k-slot pair = tokens (a, b)):
// row_lo -> channel 16 mt + g, row_hi -> channel 16 mt + 8 + g.  A byte
// permute brings the byte holding channel g of both tokens into the two
// halves, a mask keeps the code in place (f16 subnormal c * 2^(vp - 24),
// vp = v_pos(g)); the thread's output rows are rescaled by 2^(24 - vp).
template <int BITS>
__device__ inline int v_pos(int g) {
    return BITS == 2 ? 2 * (g & 3) : BITS == 4 ? 4 * (g & 1) : 0;
}
template <int BITS, int WPR>
__device__ inline void v_pair(const uint32_t (&wa)[WPR], const uint32_t (&wb)[WPR], int mt, int g,
                              uint32_t &row_lo, uint32_t &row_hi) {
    if constexpr (BITS == 2) {
        const uint32_t bi = g >> 2, bh = bi + 2;
        const uint32_t sl = bi | (bi << 4) | ((4 + bi) << 8) | ((4 + bi) << 12);
        const uint32_t sh = bh | (bh << 4) | ((4 + bh) << 8) | ((4 + bh) << 12);
        const uint32_t m = 0x00030003u << (2 * (g & 3));
        row_lo = __byte_perm(wa[mt], wb[mt], sl) & m;
        row_hi = __byte_perm(wa[mt], wb[mt], sh) & m;
    } else if constexpr (BITS == 4) {
        const uint32_t bi = g >> 1;
        const uint32_t sl = bi | (bi << 4) | ((4 + bi) << 8) | ((4 + bi) << 12);
        const uint32_t m = 0x000F000Fu << (4 * (g & 1));
        row_lo = __byte_perm(wa[2 * mt], wb[2 * mt], sl) & m;
        row_hi = __byte_perm(wa[2 * mt + 1], wb[2 * mt + 1], sl) & m;
    } else {
        const uint64_t xa = win3<WPR>(wa, mt), xb = win3<WPR>(wb, mt);
        row_lo = (uint32_t)((xa >> (3 * g)) & 7u) | ((uint32_t)((xb >> (3 * g)) & 7u) << 16);
        row_hi = (uint32_t)((xa >> (24 + 3 * g)) & 7u) | ((uint32_t)((xb >> (24 + 3 * g)) & 7u) << 16);
    }
}

// NG fp16 values (one token's scales or zeros) as floats.
template <int NG>
__device__ inline void load_halves(const __half *p, float (&f)[NG]) {
    if constexpr (NG == 4) {
        const uint2 u = *reinterpret_cast<const uint2 *>(p);
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
        f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    } else if constexpr (NG == 2) {
        const uint32_t u = *reinterpret_cast<const uint32_t *>(p);
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&u));
        f[0] = a.x; f[1] = a.y;
    } else {
#pragma unroll
        for (int i = 0; i < NG; ++i) f[i] = __half2float(p[i]);
    }
}

template <int BITS, int D, int NW>
__device__ __forceinline__ void draft_block(const DraftArgs &a, int split, int kvh, int b, uint8_t *smem) {
    using C = Cfg<BITS, D, NW>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int len = a.lens[b];
    const int npages = ceil_div(len, kPage);
    const int p0 = split * a.chunk_pages;
    const int p1 = min(p0 + a.chunk_pages, npages);
    uint8_t *ring = smem + warp * C::NSTAGE * C::STAGE;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (C::RING > C::COMBINE ? C::RING : C::COMBINE)) +
                     warp * C::NSTAGE;
    // pages of this warp: p0 + warp + 4 k
    const int nw = p1 > p0 + warp ? ceil_div(p1 - (p0 + warp), NW) : 0;
    const int32_t *trow = a.table + (int64_t)b * a.maxb;

    auto page_id = [&](int k) -> int {
        const int pg = p0 + warp + NW * k;
        const int id = pg < a.maxb ? trow[pg] : -1;
        return (id >= 0 && id < a.n_pages) ? id : -1;
    };
    auto issue = [&](int k) {  // lane 0 only
        const int st = k % C::NSTAGE;
        const int id = page_id(k);
        if (id < 0) {
            report(a.status, VC_ERR_BAD_INDEX);
            mbar_arrive(&bars[st]);
            return;
        }
        const int64_t off = ((int64_t)id * a.hkv + kvh) * C::HB;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive_expect_tx(&bars[st], 2 * C::HB);
        bulk_g2s(ring + st * C::STAGE, a.kp + off, C::HB, &bars[st]);
        bulk_g2s(ring + st * C::STAGE + C::HB, a.vp + off, C::HB, &bars[st]);
    };

    if (lane == 0) {
        for (int s = 0; s < C::NSTAGE; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (lane == 0)
        for (int k = 0; k < min(nw, C::NSTAGE); ++k) issue(k);

    // ---- the group's queries, staged once per CTA in shared memory ----
    uint16_t *qs = reinterpret_cast<uint16_t *>(smem + (C::RING > C::COMBINE ? C::RING : C::COMBINE) + C::BARS);
    float *qsum = reinterpret_cast<float *>(qs + 8 * D);  // [8 heads][NG] group sums, pre-scaled
    {
        const uint32_t *src = reinterpret_cast<const uint32_t *>(a.q + ((int64_t)b * a.hq + kvh * a.grp) * D);
        uint32_t *dst = reinterpret_cast<uint32_t *>(qs);
        for (int e = threadIdx.x; e < 8 * D / 2; e += NW * 32) dst[e] = e < a.grp * D / 2 ? src[e] : 0u;
        __syncthreads();
        if constexpr (BITS != 16) {
            for (int e = threadIdx.x; e < 8 * C::NG; e += NW * 32) {
                const int n = e / C::NG, gr = e % C::NG;
                float sum = 0.0f;
                for (int i = 0; i < kGroup; ++i) sum += bf16_bits_to_f32(qs[n * D + gr * kGroup + i]);
                qsum[e] = sum * a.scale_log2;
            }
            __syncthreads();
        }
    }
    // ---- query fragments (B operand of S^T = K Q^T), column n = head g ----
    const KPos<BITS> kpos(t);
    uint32_t bq[C::NT][2];
#pragma unroll
    for (int ks = 0; ks < C::NT; ++ks) {
        float v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int slot = (j & 1) + 2 * t + 8 * (j >> 1);
            v[j] = bf16_bits_to_f32(qs[g * D + q_channel<BITS>(ks, slot)]);
        }
        if constexpr (BITS == 16) {
            bq[ks][0] = pack_bf16(v[0], v[1]);
            bq[ks][1] = pack_bf16(v[2], v[3]);
        } else {
            const float fl = __uint_as_float((uint32_t)(127 - kpos.pl) << 23);  // 2^-pl
            const float fh = __uint_as_float((uint32_t)(127 - kpos.ph) << 23);
            bq[ks][0] = pack_f16(v[0] * fl, v[1] * fl);
            bq[ks][1] = pack_f16(v[2] * fh, v[3] * fh);
        }
    }
    // per-group query sums of the two head columns this thread accumulates
    float qg[C::NG][2];
    if constexpr (BITS != 16) {
#pragma unroll
        for (int gr = 0; gr < C::NG; ++gr) {
            qg[gr][0] = qsum[(2 * t) * C::NG + gr];
            qg[gr][1] = qsum[(2 * t + 1) * C::NG + gr];
        }
    }

    float o[C::NT][4];
#pragma unroll
    for (int i = 0; i < C::NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
    float zacc[C::NG][2];
#pragma unroll
    for (int i = 0; i < C::NG; ++i) zacc[i][0] = zacc[i][1] = 0.0f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.0f, 0.0f};
    const int src0 = t * 4 + (g >> 1), src1 = (t + 4) * 4 + (g >> 1);
    const bool odd_head = g & 1;

    for (int k = 0; k < nw; ++k) {
        const int st = k % C::NSTAGE;
        if (!mbar_wait(&bars[st], (k / C::NSTAGE) & 1, a.status)) break;
        const uint8_t *kb = ring + st * C::STAGE;
        uint8_t *vb = ring + st * C::STAGE + C::HB;
        const int pg = p0 + warp + NW * k;
        if (page_id(k) < 0) {  // reported at issue time; nothing landed in this stage
            __syncwarp();
            if (lane == 0 && k + C::NSTAGE < nw) issue(k + C::NSTAGE);
            continue;
        }
        const int slot0 = 2 * g, slot1 = 2 * g + 1;
        const int pos0 = pg * kPage + slot0;
        const bool valid0 = pos0 < len, valid1 = pos0 + 1 < len;
        float s[4];  // (slot0, head 2t), (slot0, 2t+1), (slot1, 2t), (slot1, 2t+1)
        if constexpr (BITS == 16) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < C::NT / 2; ++kk) {
                const uint4 u0 = *reinterpret_cast<const uint4 *>(kb + slot0 * D * 2 + (32 * kk + 8 * t) * 2);
                const uint4 u1 = *reinterpret_cast<const uint4 *>(kb + slot1 * D * 2 + (32 * kk + 8 * t) * 2);
                const uint32_t a0[4] = {u0.x, u1.x, u0.y, u1.y};
                const uint32_t a1[4] = {u0.z, u1.z, u0.w, u1.w};
                mma_bf16(acc, a0, bq[2 * kk][0], bq[2 * kk][1]);
                mma_bf16(acc, a1, bq[2 * kk + 1][0], bq[2 * kk + 1][1]);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) s[j] = acc[j] * a.scale_log2;
        } else {
            uint32_t w0[C::WPR], w1[C::WPR];
            load_row<C::CB>(w0, kb + slot0 * C::CB);
            load_row<C::CB>(w1, kb + slot1 * C::CB);
            const __half *scl = reinterpret_cast<const __half *>(kb + kPage * C::CB);
            const __half *zer = scl + kPage * C::NG;
            float sc0[C::NG], sc1[C::NG], zr0[C::NG], zr1[C::NG];
            load_halves<C::NG>(scl + slot0 * C::NG, sc0);
            load_halves<C::NG>(scl + slot1 * C::NG, sc1);
            load_halves<C::NG>(zer + slot0 * C::NG, zr0);
            load_halves<C::NG>(zer + slot1 * C::NG, zr1);
            const float kscale = a.scale_log2 * 16777216.0f;  // products carry 2^-24
            s[0] = s[1] = s[2] = s[3] = 0.0f;
#pragma unroll
            for (int gr = 0; gr < C::NG; ++gr) {
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int ks = 2 * gr + h2;
                    uint32_t af[4];
                    k_pair<BITS, C::WPR>(w0, ks, t, kpos, af[0], af[2]);
                    k_pair<BITS, C::WPR>(w1, ks, t, kpos, af[1], af[3]);
                    mma_f16(acc, af, bq[ks][0], bq[ks][1]);
                }
                const float f0 = sc0[gr] * kscale, f1 = sc1[gr] * kscale;
                s[0] = fmaf(f0, acc[0], fmaf(zr0[gr], qg[gr][0], s[0]));
                s[1] = fmaf(f0, acc[1], fmaf(zr0[gr], qg[gr][1], s[1]));
                s[2] = fmaf(f1, acc[2], fmaf(zr1[gr], qg[gr][0], s[2]));
                s[3] = fmaf(f1, acc[3], fmaf(zr1[gr], qg[gr][1], s[3]));
            }
        }
        // mask positions past the request length (their slots may hold garbage)
        if (!valid0) s[0] = s[1] = -INFINITY;
        if (!valid1) s[2] = s[3] = -INFINITY;

        // ---- online softmax over the page (per head column) ----
        float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
        if (__any_sync(0xffffffffu, mn0 > m[0] || mn1 > m[1])) {
            const float al0 = mn0 == -INFINITY ? 1.0f : ex2(m[0] - mn0);
            const float al1 = mn1 == -INFINITY ? 1.0f : ex2(m[1] - mn1);
#pragma unroll
            for (int i = 0; i < C::NT; ++i) {
                o[i][0] *= al0; o[i][2] *= al0;
                o[i][1] *= al1; o[i][3] *= al1;
            }
#pragma unroll
            for (int i = 0; i < C::NG; ++i) { zacc[i][0] *= al0; zacc[i][1] *= al1; }
            l[0] *= al0;
            l[1] *= al1;
            m[0] = mn0;
            m[1] = mn1;
        }
        const float ms0 = m[0] == -INFINITY ? 0.0f : m[0], ms1 = m[1] == -INFINITY ? 0.0f : m[1];
        const float p[4] = {ex2(s[0] - ms0), ex2(s[1] - ms1), ex2(s[2] - ms0), ex2(s[3] - ms1)};
        l[0] += p[0] + p[2];
        l[1] += p[1] + p[3];

        // ---- O^T += V^T P^T ----
        if constexpr (BITS == 16) {
            const int nvalid = len - pg * kPage;  // slots >= nvalid are past the end
            if (nvalid < kPage) {
                for (int c = lane; c < (kPage - nvalid) * D / 8; c += 32)
                    reinterpret_cast<uint4 *>(vb + nvalid * D * 2)[c] = make_uint4(0, 0, 0, 0);
                __syncwarp();
            }
            const uint32_t e = pack_bf16(p[0], p[2]), od = pack_bf16(p[1], p[3]);
            const uint32_t e0 = __shfl_sync(0xffffffffu, e, src0), o0 = __shfl_sync(0xffffffffu, od, src0);
            const uint32_t e1 = __shfl_sync(0xffffffffu, e, src1), o1 = __shfl_sync(0xffffffffu, od, src1);
            const uint32_t b0 = odd_head ? o0 : e0, b1 = odd_head ? o1 : e1;
            const int mi = lane >> 3, r = lane & 7;
            const uint8_t *vrow = vb + ((mi >> 1) * 8 + r) * D * 2 + (8 * (mi & 1)) * 2;
#pragma unroll
            for (int mt = 0; mt < C::NT; ++mt) {
                uint32_t af[4];
                ldsm_x4_t(af, vrow + 16 * mt * 2);
                mma_bf16(o[mt], af, b0, b1);
            }
        } else {
            uint32_t wa[C::WPR], wb[C::WPR], wc[C::WPR], wd[C::WPR];
            load_row<C::CB>(wa, vb + (2 * t) * C::CB);
            load_row<C::CB>(wb, vb + (2 * t + 1) * C::CB);
            load_row<C::CB>(wc, vb + (2 * t + 8) * C::CB);
            load_row<C::CB>(wd, vb + (2 * t + 9) * C::CB);
            const __half *vscl = reinterpret_cast<const __half *>(vb + kPage * C::CB);
            const __half *vzer = vscl + kPage * C::NG;
            // V scale / zero of this thread's tokens (slot0, slot1); slots past
            // the end contribute exactly nothing, whatever their bytes hold
            float vsc0[C::NG], vsc1[C::NG], vze0[C::NG], vze1[C::NG];
            load_halves<C::NG>(vscl + slot0 * C::NG, vsc0);
            load_halves<C::NG>(vscl + slot1 * C::NG, vsc1);
            load_halves<C::NG>(vzer + slot0 * C::NG, vze0);
            load_halves<C::NG>(vzer + slot1 * C::NG, vze1);
#pragma unroll
            for (int gr = 0; gr < C::NG; ++gr) {
                const float vs0 = valid0 ? vsc0[gr] : 0.0f, vs1 = valid1 ? vsc1[gr] : 0.0f;
                const float vz0 = valid0 ? vze0[gr] : 0.0f, vz1 = valid1 ? vze1[gr] : 0.0f;
                zacc[gr][0] = fmaf(p[0], vz0, fmaf(p[2], vz1, zacc[gr][0]));
                zacc[gr][1] = fmaf(p[1], vz0, fmaf(p[3], vz1, zacc[gr][1]));
                const uint32_t e = pack_f16(p[0] * vs0, p[2] * vs1), od = pack_f16(p[1] * vs0, p[3] * vs1);
                const uint32_t e0 = __shfl_sync(0xffffffffu, e, src0), o0 = __shfl_sync(0xffffffffu, od, src0);
                const uint32_t e1 = __shfl_sync(0xffffffffu, e, src1), o1 = __shfl_sync(0xffffffffu, od, src1);
                const uint32_t b0 = odd_head ? o0 : e0, b1 = odd_head ? o1 : e1;
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int mt = 2 * gr + h2;
                    uint32_t af[4];
                    v_pair<BITS, C::WPR>(wa, wb, mt, g, af[0], af[1]);
                    v_pair<BITS, C::WPR>(wc, wd, mt, g, af[2], af[3]);
                    mma_f16(o[mt], af, b0, b1);
                }
            }
        }
        __syncwarp();
        if (lane == 0 && k + C::NSTAGE < nw) issue(k + C::NSTAGE);
    }

    // ---- warp epilogue: finish l and the zero terms ----
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l[0] += __shfl_xor_sync(0xffffffffu, l[0], off);
        l[1] += __shfl_xor_sync(0xffffffffu, l[1], off);
    }
    if constexpr (BITS != 16) {
#pragma unroll
        for (int gr = 0; gr < C::NG; ++gr) {
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                zacc[gr][0] += __shfl_xor_sync(0xffffffffu, zacc[gr][0], off);
                zacc[gr][1] += __shfl_xor_sync(0xffffffffu, zacc[gr][1], off);
            }
        }
        const float osc = __uint_as_float((uint32_t)(127 + 24 - v_pos<BITS>(g)) << 23);  // 2^(24 - vp)
#pragma unroll
        for (int mt = 0; mt < C::NT; ++mt) {
            const int gr = mt / 2;
            o[mt][0] = fmaf(o[mt][0], osc, zacc[gr][0]);
            o[mt][2] = fmaf(o[mt][2], osc, zacc[gr][0]);
            o[mt][1] = fmaf(o[mt][1], osc, zacc[gr][1]);
            o[mt][3] = fmaf(o[mt][3], osc, zacc[gr][1]);
        }
    }
    // ---- combine the 4 warps of the CTA in shared memory ----
    __syncthreads();  // every warp is done with its ring
    float *cm = reinterpret_cast<float *>(smem);   // [warp][8] m
    float *cl = cm + NW * 8;                    // [warp][8] l
    float *co = cl + NW * 8;                    // [warp][8][D]
    if (g == 0) {
        cm[warp * 8 + 2 * t] = m[0]; cm[warp * 8 + 2 * t + 1] = m[1];
        cl[warp * 8 + 2 * t] = l[0]; cl[warp * 8 + 2 * t + 1] = l[1];
    }
#pragma unroll
    for (int mt = 0; mt < C::NT; ++mt) {
        float *base = co + warp * 8 * D;
        base[(2 * t) * D + 16 * mt + g] = o[mt][0];
        base[(2 * t + 1) * D + 16 * mt + g] = o[mt][1];
        base[(2 * t) * D + 16 * mt + 8 + g] = o[mt][2];
        base[(2 * t + 1) * D + 16 * mt + 8 + g] = o[mt][3];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < a.grp * D; e += NW * 32) {
        const int n = e / D, c = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, cm[w * 8 + n]);
        float acc = 0.0f, L = 0.0f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float f = ex2(cm[w * 8 + n] - M);
                acc += f * co[(w * 8 + n) * D + c];
                L += f * cl[w * 8 + n];
            }
        }
        const int64_t row = ((int64_t)b * a.hq + kvh * a.grp + n) * a.n_splits + split;
        a.ws_o[row * D + c] = acc;
        if (c == 0) {
            a.ws_ml[row * 2] = M;
            a.ws_ml[row * 2 + 1] = L;
        }
    }
}

// Combine the chunk partials of one (request, head) row.
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

}  // namespace draft
}  // namespace vc
