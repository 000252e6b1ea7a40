// Quantisation of one token row and the append of one (token, kv head)
// entry to a KV_comp page, shared by vc_compress (token-parallel appends)
// and vc_draft_step (the draft kernel appends the step's new token before
// it attends).  The format is the one vc.h states; the code placement is
// comp_layout.cuh's.
#pragma once

#include "comp_layout.cuh"
#include "vc_internal.cuh"

namespace vc {
namespace qrow {

__device__ inline uint16_t f16_store(float f) {  // saturate to +-65504, round to nearest even
    f = fminf(fmaxf(f, -65504.0f), 65504.0f);
    return __half_as_ushort(__float2half_rn(f));
}

// Quantise one row (D channels, CPL = D/32 consecutive ones per lane):
// codes of the lane's channels, and the fp16 scale / zero of its group.
template <int BITS, int D>
__device__ void quantize_row(const uint16_t (&x)[D / 32], uint8_t (&code)[D / 32], uint16_t &sh, uint16_t &zh) {
    constexpr int CPL = D / 32;             // channels per lane
    constexpr int LPG = kGroup / CPL;       // lanes per group
    constexpr int QMAX = (1 << BITS) - 1;
    float v[CPL];
    float mn, mx;
#pragma unroll
    for (int i = 0; i < CPL; ++i) v[i] = bf16_bits_to_f32(x[i]);
    mn = v[0];
    mx = v[0];
#pragma unroll
    for (int i = 1; i < CPL; ++i) {
        mn = fminf(mn, v[i]);
        mx = fmaxf(mx, v[i]);
    }
#pragma unroll
    for (int o = 1; o < LPG; o <<= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    mn = __fadd_rn(mn, 0.0f);  // -0 -> +0
    const float range = __fsub_rn(mx, mn);
    const float sdot = __fdiv_rn(range, (float)QMAX);
    sh = f16_store(sdot);
    zh = f16_store(mn);
    const float s = __half2float(__ushort_as_half(sh));
    const float z = __half2float(__ushort_as_half(zh));
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
        int c = 0;
        if (s != 0.0f) {
            float t = __fdiv_rn(__fsub_rn(v[i], z), s);
            float r = rintf(t);
            r = fminf(fmaxf(r, 0.0f), (float)QMAX);
            c = (int)r;
        }
        code[i] = (uint8_t)c;
    }
}

// Load the bf16 row a lane quantises: D/32 consecutive channels per lane.
template <int D>
__device__ inline void load_lane_row(const uint8_t *src, int lane, uint16_t (&x)[D / 32]) {
    constexpr int CPL = D / 32;
    if constexpr (CPL == 4) {
        uint2 u = reinterpret_cast<const uint2 *>(src)[lane];
        x[0] = u.x & 0xffff; x[1] = u.x >> 16; x[2] = u.y & 0xffff; x[3] = u.y >> 16;
    } else if constexpr (CPL == 2) {
        uint32_t u = reinterpret_cast<const uint32_t *>(src)[lane];
        x[0] = u & 0xffff; x[1] = u >> 16;
    } else {
#pragma unroll
        for (int i = 0; i < CPL; ++i) x[i] = reinterpret_cast<const uint16_t *>(src)[lane * CPL + i];
    }
}

// One warp appends one (token, kv head) entry: bf16 rows k_row / v_row
// (D channels) into token slot `slot` of the page's K / V head blocks gk /
// gv.  The K row and the fp16 parameters belong to the slot alone and are
// stored directly (the K row is assembled in `krow`, a per-warp shared
// buffer of D * BITS / 32 words); V codes share 32-bit words with the page's
// other tokens and are merged with global AND / OR reductions.  bits == 16:
// the rows are copied.
template <int BITS, int D>
__device__ void append_entry(const uint8_t *k_row, const uint8_t *v_row, uint8_t *gk, uint8_t *gv, int slot,
                             int lane, uint32_t *krow) {
    constexpr int CPL = D / 32;
    if constexpr (BITS == 16) {
        uint16_t xk[CPL], xv[CPL];
        load_lane_row<D>(k_row, lane, xk);
        load_lane_row<D>(v_row, lane, xv);
        uint16_t *dk = reinterpret_cast<uint16_t *>(gk + slot * D * 2);
        uint16_t *dv = reinterpret_cast<uint16_t *>(gv + slot * D * 2);
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
            dk[lane * CPL + i] = xk[i];
            dv[lane * CPL + i] = xv[i];
        }
    } else {
        constexpr int LPG = kGroup / CPL, G = D / kGroup;
        constexpr int CR = kPage * D * BITS / 8, RW = D * BITS / 32;  // K row words
        uint16_t xk[CPL], xv[CPL];
        load_lane_row<D>(k_row, lane, xk);
        load_lane_row<D>(v_row, lane, xv);
        for (int i = lane; i < RW; i += 32) krow[i] = 0u;
        __syncwarp();
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
            uint8_t code[CPL];
            uint16_t sh, zh;
            quantize_row<BITS, D>(kv ? xv : xk, code, sh, zh);
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                const int ch = lane * CPL + i;
#pragma unroll
                for (int pl = 0; pl < (BITS == 3 ? 2 : 1); ++pl) {
                    const int w = BITS == 3 ? (pl ? 1 : 2) : BITS;
                    const uint32_t v = BITS == 3 ? (pl ? code[i] >> 2 : code[i] & 3u) : code[i];
                    if (kv == 0) {  // K: the token's own row, built in shared memory
                        const int o = layout::k_bit(BITS, D, slot, ch, pl) - slot * D * BITS;
                        atomicOr(&krow[o >> 5], v << (o & 31));
                    } else {  // V: words shared with the page's other tokens
                        const int o = layout::v_bit(BITS, D, slot, ch, pl);
                        const uint32_t m = ((1u << w) - 1u) << (o & 31);
                        uint32_t *word = reinterpret_cast<uint32_t *>(gv) + (o >> 5);
                        atomicAnd(word, ~m);
                        atomicOr(word, (v << (o & 31)) & m);
                    }
                }
            }
            if (lane % LPG == 0) {
                const int gr = lane / LPG;
                const int e = kv ? layout::v_param(G, slot, gr) : slot * G + gr;
                uint16_t *par = reinterpret_cast<uint16_t *>((kv ? gv : gk) + CR);
                par[e] = sh;
                par[kPage * G + e] = zh;
            }
        }
        __syncwarp();
        uint32_t *kd = reinterpret_cast<uint32_t *>(gk + slot * (D * BITS / 8));
        for (int i = lane; i < RW; i += 32) kd[i] = krow[i];
    }
}

}  // namespace qrow
}  // namespace vc
