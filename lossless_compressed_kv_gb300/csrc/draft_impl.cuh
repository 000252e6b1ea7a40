// Device body of the draft attention (shared by the draft launch and the
// mixed draft/verify launch).  See draft_attn.cu for the design notes and
// comp_layout.cuh for the code placement this body reads.
#pragma once

#include <type_traits>

#include "quant_row.cuh"
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
    int chunk_pages, n_splits;  // pages per chunk; chunk slots per row of the workspace
    // the draft launch's first lo_units units (request x kv head) take n_lo
    // chunks of chunk_pages, the others n_hi chunks of chunk_hi pages
    int lo_units = 0, chunk_hi = 0, n_hi = 0, n_lo = 0;
    float *ws_o;   // [B][Hq][n_splits][D]
    float *ws_ml;  // [B][Hq][n_splits][2]
    int32_t *status;
    uint64_t wait_ns = kWaitNs;  // bounded-wait limit
    int skip_copies = 0;         // fault injection: issue no copy (every wait then times out)
    // vc_draft_step: the step's new entry of every request (bf16 K and V
    // rows, [B][Hkv][D]) is written to KV_comp position slot[b] before the
    // attention; null for a plain draft call
    const uint16_t *k_new = nullptr, *v_new = nullptr;
    const int32_t *slot = nullptr;
};

// Online softmax with a lazy reference: when a score beats the running
// reference, the reference moves kLazyRef (log2 units) above the new
// maximum, so that later, slightly larger scores do not rescale again.
// Probabilities stay <= 2^-kLazyRef <= 1 (their f16 / bf16 operands cannot
// overflow), and the partials carry the reference as their m.
constexpr float kLazyRef = 3.0f;

template <int BITS, int D, int NW>
struct Cfg {
    static constexpr int NT = D / 16;  // k-steps of QK^T, m-tiles of PV
    static constexpr int NG = D / 32;  // quantisation groups
    static constexpr int HB = BITS == 16 ? kPage * D * 2 : 2 * D * (BITS + 1);
    static constexpr int CR = kPage * D * (BITS == 16 ? 16 : BITS) / 8;  // code region bytes
    // ring stages per warp: a bf16 page-head is 8 KB (K and V), so two
    // stages keep three CTAs per SM (three stages held two: the 70B-shaped
    // draft took 120.7 us against 110.8 with two)
    static constexpr int NSTAGE = BITS == 16 ? 2 : 4;
    static constexpr int STAGE = 2 * HB;
    static constexpr int RING = NW * NSTAGE * STAGE;
    static constexpr int COMBINE = NW * 8 * (D + 2) * 4;
    static constexpr int BARS = NW * NSTAGE * 8 + NW * NSTAGE * 4;  // mbarriers + per-stage page-valid flags
    // q of the group (bf16) + its group sums + the quantised path's packed
    // query fragments ([NT/2][32 lanes][4 words])
    static constexpr int QS = 8 * D * 2 + 8 * NG * 4 + (BITS == 16 ? 0 : NT / 2 * 32 * 16);
    static constexpr int SMEM = (RING > COMBINE ? RING : COMBINE) + BARS + QS;
};

// ---------------------------------------------------------------------------
// packed f32x2 arithmetic (one instruction for two lanes of fp32)
// ---------------------------------------------------------------------------
struct f2 {
    float x, y;
};
__device__ inline f2 fma2(f2 a, f2 b, f2 c) {
    unsigned long long ua, ub, uc, ud;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ua) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(ub) : "f"(b.x), "f"(b.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(uc) : "f"(c.x), "f"(c.y));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(ud) : "l"(ua), "l"(ub), "l"(uc));
    f2 d;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(ud));
    return d;
}
__device__ inline f2 mul2(f2 a, f2 b) {
    unsigned long long ua, ub, ud;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ua) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(ub) : "f"(b.x), "f"(b.y));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(ud) : "l"(ua), "l"(ub));
    f2 d;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(ud));
    return d;
}
__device__ inline uint32_t hmul2(uint32_t a, uint32_t b) {
    __half2 r = __hmul2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}

// ---------------------------------------------------------------------------
// Quantised K operand.  Thread t of a fragment reads its region of a token
// row and turns it into R = D/8 registers; register r = 2 ks + h holds the
// codes of channels 16 ks + 4 t + 2 h + {0, 1} in its two halves at bit
// position kpos(r), i.e. the f16 subnormals code * 2^(kpos - 24).
// ---------------------------------------------------------------------------
template <int BITS>
__host__ __device__ constexpr int kpos(int r) {
    return BITS == 2 ? ((r & 7) < 5 ? 2 * (r & 7) : 2 * ((r & 7) - 5))
         : BITS == 4 ? 4 * (r & 1)
                     : 2 * (r & 3);
}

template <int BITS, int D>
struct KRow {
    static constexpr int NLO = BITS == 4 ? D / 32 : D / 64;  // main-plane words of a thread region
    static constexpr int NHI = BITS == 3 ? (D >= 128 ? D / 128 : 1) : 0;
    uint32_t w[NLO];
    uint32_t hw[NHI > 0 ? NHI : 1];

    __device__ inline void load(const uint8_t *row, int t) {
        if constexpr (BITS == 2 || BITS == 3) {
            const uint8_t *p = row + t * (D / 16);
            if constexpr (NLO == 1) {
                w[0] = *reinterpret_cast<const uint32_t *>(p);
            } else if constexpr (NLO == 2) {
                const uint2 u = *reinterpret_cast<const uint2 *>(p);
                w[0] = u.x; w[1] = u.y;
            } else {
#pragma unroll
                for (int i = 0; i < NLO / 4; ++i) {
                    const uint4 u = reinterpret_cast<const uint4 *>(p)[i];
                    w[4 * i] = u.x; w[4 * i + 1] = u.y; w[4 * i + 2] = u.z; w[4 * i + 3] = u.w;
                }
            }
            if constexpr (BITS == 3) {
                const uint8_t *h = row + D / 4;  // high-bit plane after the four low regions
                if constexpr (D == 64) {
                    const uint32_t u = *reinterpret_cast<const uint16_t *>(h + 2 * t);
                    hw[0] = __byte_perm(u, 0u, 0x4140);  // half-0 byte -> bits 0-7, half-1 byte -> 16-23
                } else {
#pragma unroll
                    for (int i = 0; i < NHI; ++i) hw[i] = reinterpret_cast<const uint32_t *>(h + t * (D / 32))[i];
                }
            }
        } else {  // 4 bits
            const uint8_t *p = row + t * (D / 8);
            if constexpr (NLO == 2) {
                const uint2 u = *reinterpret_cast<const uint2 *>(p);
                w[0] = u.x; w[1] = u.y;
            } else {
#pragma unroll
                for (int i = 0; i < NLO / 4; ++i) {
                    const uint4 u = reinterpret_cast<const uint4 *>(p)[i];
                    w[4 * i] = u.x; w[4 * i + 1] = u.y; w[4 * i + 2] = u.z; w[4 * i + 3] = u.w;
                }
            }
        }
    }

    // operand register r (compile-time after unrolling)
    __device__ inline uint32_t reg(int r) const {
        if constexpr (BITS == 2) {
            const int u = r >> 3, j = r & 7;
            return j < 5 ? (w[u] & (0x00030003u << (2 * j))) : ((w[u] >> 10) & (0x00030003u << (2 * (j - 5))));
        } else if constexpr (BITS == 4) {
            const int u = r >> 2, j = r & 3;
            const uint32_t y = j < 2 ? w[u] : (w[u] >> 8);
            return y & (0x000F000Fu << (4 * (j & 1)));
        } else {
            const int u = r >> 3, j = r & 7, p = 2 * (j & 3);
            const uint32_t lo = j < 4 ? w[u] : (w[u] >> 8);
            const int set = 2 * (u & 1) + (j >> 2);
            const uint32_t h = hw[u >> 1];
            const uint32_t y = set == 0 ? (h << 2) : set == 1 ? (h << 1) : set == 2 ? (h >> 6) : (h >> 7);
            return (lo & (0x00030003u << p)) | (y & (0x00040004u << p));
        }
    }
};

// ---------------------------------------------------------------------------
// Quantised V operand.  Thread (g, t) reads its region (channels 16 mt + g
// and 16 mt + 8 + g, tokens 2t, 2t+1, 2t+8, 2t+9) and forms the four A
// registers of m-tile mt: a0 / a2 = channel 16 mt + g with tokens (2t, 2t+1)
// / (2t+8, 2t+9), a1 / a3 the same for channel 16 mt + 8 + g.  a2 and a3 sit
// VHI above a0 and a1 (the B operand of the second token pair carries
// 2^-VHI); a1 and a3 sit ROW8 above a0 and a2 (compensated on the output
// rows g+8).
// ---------------------------------------------------------------------------
template <int BITS, int D>
struct VReg {
    static constexpr int NW = BITS == 4 ? D / 16 : D / 32;  // main-plane words of the region
    static constexpr int NH = BITS == 3 ? D / 64 : 0;       // high-plane words (3 bits)
    static constexpr int VHI = BITS == 4 ? 4 : 2;
    static constexpr int ROW8 = BITS == 4 ? 0 : 4;
    uint32_t w[NW];
    uint32_t hw[NH > 0 ? NH : 1];

    template <int N>
    __device__ static inline void ld(uint32_t (&dst)[N], const uint8_t *p) {
        if constexpr (N == 1) {
            dst[0] = *reinterpret_cast<const uint32_t *>(p);
        } else if constexpr (N == 2) {
            const uint2 u = *reinterpret_cast<const uint2 *>(p);
            dst[0] = u.x; dst[1] = u.y;
        } else {
#pragma unroll
            for (int i = 0; i < N / 4; ++i) {
                const uint4 u = reinterpret_cast<const uint4 *>(p)[i];
                dst[4 * i] = u.x; dst[4 * i + 1] = u.y; dst[4 * i + 2] = u.z; dst[4 * i + 3] = u.w;
            }
        }
    }

    __device__ inline void load(const uint8_t *vb, int g, int t) {
        const int region = g * 4 + t;
        ld<NW>(w, vb + 4 * region * NW);
        if constexpr (BITS == 3) ld<NH>(hw, vb + 4 * D + 4 * region * NH);
    }

    __device__ inline void regs(int mt, uint32_t (&a)[4]) const {
        if constexpr (BITS == 4) {
            const uint32_t x = w[mt], y = x >> 8;
            a[0] = x & 0x000F000Fu; a[2] = x & 0x00F000F0u;
            a[1] = y & 0x000F000Fu; a[3] = y & 0x00F000F0u;
        } else {
            const int u = mt >> 1, m = mt & 1;
            const uint32_t y = m ? (w[u] >> 8) : w[u];
            if constexpr (BITS == 2) {
                a[0] = y & 0x00030003u; a[2] = y & 0x000C000Cu;
                a[1] = y & 0x00300030u; a[3] = y & 0x00C000C0u;
            } else {
                const int set = 2 * (u & 1) + m;
                const uint32_t h = hw[u >> 1];
                const uint32_t z = set == 0 ? (h << 2) : set == 1 ? (h << 1) : set == 2 ? (h >> 6) : (h >> 7);
                a[0] = (y & 0x00030003u) | (z & 0x00040004u);
                a[2] = (y & 0x000C000Cu) | (z & 0x00100010u);
                a[1] = (y & 0x00300030u) | (z & 0x00400040u);
                a[3] = (y & 0x00C000C0u) | (z & 0x01000100u);
            }
        }
    }
};

// NG fp16 values (one token's K scales) as floats.
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

// a ring stage given as a compile-time constant or at run time
template <int N>
__device__ constexpr int stage_value(std::integral_constant<int, N>) {
    return N;
}
__device__ inline int stage_value(int s) { return s; }

template <int BITS, int D, int NW>
__device__ __forceinline__ void draft_block(const DraftArgs &a, int split, int kvh, int b, int chunk,
                                            uint8_t *smem) {
    using C = Cfg<BITS, D, NW>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int p0 = split * chunk;
    const int32_t *trow = a.table + (int64_t)b * a.maxb;
    // The loads that depend on nothing else go out together: the group's
    // queries, the table entries of the warp's first 64 pages (read before
    // the length is known: every entry below maxb is in bounds) and the
    // length, so their latencies overlap at the start of the CTA.
    constexpr int QW = (8 * D / 2 + NW * 32 - 1) / (NW * 32);  // query words per thread
    uint32_t qreg[QW];
    {
        const uint32_t *src = reinterpret_cast<const uint32_t *>(a.q + ((int64_t)b * a.hq + kvh * a.grp) * D);
#pragma unroll
        for (int i = 0; i < QW; ++i) {
            const int e = threadIdx.x + i * NW * 32;
            qreg[i] = e < a.grp * D / 2 ? src[e] : 0u;
        }
    }
    auto raw_id = [&](int kk) -> int {
        const int pg = p0 + warp + NW * kk;
        return pg < a.maxb ? trow[pg] : -1;
    };
    const int raw0 = raw_id(lane), raw1 = raw_id(32 + lane);
    const int len = a.lens[b];
    const int npages = ceil_div(len, kPage);
    const int p1 = min(p0 + chunk, npages);
    uint8_t *ring = smem + warp * C::NSTAGE * C::STAGE;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (C::RING > C::COMBINE ? C::RING : C::COMBINE)) +
                     warp * C::NSTAGE;
    // pages of this warp: p0 + warp + NW k
    const int nw = p1 > p0 + warp ? ceil_div(p1 - (p0 + warp), NW) : 0;

    int *sflag = reinterpret_cast<int *>(reinterpret_cast<uint64_t *>(smem + (C::RING > C::COMBINE ? C::RING
                                                                                                : C::COMBINE)) +
                                         NW * C::NSTAGE) +
                 warp * C::NSTAGE;

    if (a.k_new != nullptr) {
        // vc_draft_step: the CTA whose pages hold slot[b] writes the step's
        // new entry there before any copy of that page is issued; the other
        // CTAs never read that page
        const int s = a.slot[b];
        if (split == 0 && kvh == 0 && (s < 0 || s >= len) && threadIdx.x == 0) report(a.status, VC_ERR_INVALID_ARG);
        const int pi = (s >= 0 && s < len) ? s / kPage : -1;
        if (pi >= p0 && pi < p1) {  // uniform over the CTA
            if (warp == 0) {
                __shared__ uint32_t krow[BITS == 16 ? 1 : D * BITS / 32];
                const int id = pi < a.maxb ? trow[pi] : -1;
                if (id >= 0 && id < a.n_pages) {
                    const int64_t off = ((int64_t)id * a.hkv + kvh) * C::HB;
                    const int64_t row = ((int64_t)b * a.hkv + kvh) * D;
                    qrow::append_entry<BITS, D>(reinterpret_cast<const uint8_t *>(a.k_new + row),
                                                reinterpret_cast<const uint8_t *>(a.v_new + row),
                                                const_cast<uint8_t *>(a.kp) + off, const_cast<uint8_t *>(a.vp) + off,
                                                s % kPage, lane, krow);
                    // the generic-proxy writes must be visible to the bulk
                    // copies (async proxy) issued after the barrier below
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                } else if (lane == 0) {
                    report(a.status, VC_ERR_BAD_INDEX);
                }
            }
            __syncthreads();
        }
    }

    // Head blocks (page id x hkv + kv head) of this warp's pages, 32 at a
    // time: lane i holds page 32 blk + i (-1: past the warp's pages or not a
    // valid page id).  Two blocks are kept so the table reads run a block
    // ahead of the copies.  The block is advanced once per four pages by the
    // loop driver, not per copy: this bookkeeping and the copy issue had cost
    // about a sixth of the kernel's instructions.
    auto head_row = [&](int kk, int id) -> int {
        return (kk < nw && id >= 0 && id < a.n_pages) ? id * a.hkv + kvh : -1;
    };
    auto load_rows = [&](int blk) -> int {
        const int kk = 32 * blk + lane;
        return kk < nw ? head_row(kk, raw_id(kk)) : -1;
    };
    int rows_cur = head_row(lane, raw0), rows_nxt = head_row(32 + lane, raw1), cur_blk = 0;
    auto advance_rows = [&](int k) {  // make page k's block current (k warp-uniform, non-decreasing)
        if ((k >> 5) != cur_blk) {
            rows_cur = rows_nxt;
            rows_nxt = load_rows((k >> 5) + 1);
            cur_blk = k >> 5;
        }
    };
    auto issue = [&](int k) {  // every lane (k warp-uniform, in the current block); lane 0 issues the copies
        const int row = __shfl_sync(0xffffffffu, rows_cur, k & 31);
        if (lane == 0 && !a.skip_copies) {
            // a bad page id is reported and page 0 copied in its place (the
            // stage then holds finite data; the request's result is void)
            const int st = k % C::NSTAGE;
            if constexpr (BITS == 16) sflag[st] = row >= 0;
            if (row < 0) report(a.status, VC_ERR_BAD_INDEX);
            const int64_t off = (int64_t)(row < 0 ? kvh : row) * C::HB;
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive_expect_tx(&bars[st], 2 * C::HB);
            bulk_g2s(ring + st * C::STAGE, a.kp + off, C::HB, &bars[st]);
            bulk_g2s(ring + st * C::STAGE + C::HB, a.vp + off, C::HB, &bars[st]);
        }
    };

    if (lane == 0) {
        for (int s = 0; s < C::NSTAGE; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    for (int k = 0; k < min(nw, C::NSTAGE); ++k) issue(k);

    // ---- the group's queries, staged once per CTA in shared memory ----
    uint16_t *qs = reinterpret_cast<uint16_t *>(smem + (C::RING > C::COMBINE ? C::RING : C::COMBINE) + C::BARS);
    float *qsum = reinterpret_cast<float *>(qs + 8 * D);  // [8 heads][NG] group sums, pre-scaled
    {
        uint32_t *dst = reinterpret_cast<uint32_t *>(qs);
#pragma unroll
        for (int i = 0; i < QW; ++i) {
            const int e = threadIdx.x + i * NW * 32;
            if (e < 8 * D / 2) dst[e] = qreg[i];
        }
        __syncthreads();
        if constexpr (BITS != 16) {
            for (int e = threadIdx.x; e < 8 * C::NG; e += NW * 32) {
                const int n = e / C::NG, gr = e % C::NG;
                float sum = 0.0f;
                for (int i = 0; i < kGroup; ++i) sum += bf16_bits_to_f32(qs[n * D + gr * kGroup + i]);
                qsum[e] = sum * a.scale_log2;
            }
            // Q fragments: B of S^T = K Q^T, column n = head g, k-slot pair of
            // register r pre-scaled by 2^-kpos(r) so every product is c q
            // 2^-24.  The same for every warp: packed once into shared memory
            // as [group][lane][k-step 2gr lo, hi, k-step 2gr+1 lo, hi], the
            // k-steps spread over the warps.
            uint32_t *qf = reinterpret_cast<uint32_t *>(qsum + 8 * C::NG);
#pragma unroll
            for (int ks = 0; ks < C::NT; ++ks) {
                if (ks % NW != warp) continue;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int c0 = 16 * ks + 4 * t + 2 * h;
                    const float f = __uint_as_float((uint32_t)(127 - kpos<BITS>(2 * ks + h)) << 23);
                    qf[((ks >> 1) * 32 + lane) * 4 + 2 * (ks & 1) + h] =
                        pack_f16(bf16_bits_to_f32(qs[g * D + c0]) * f, bf16_bits_to_f32(qs[g * D + c0 + 1]) * f);
                }
            }
            __syncthreads();
        }
    }

    float o[C::NT][4];
#pragma unroll
    for (int i = 0; i < C::NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.0f, 0.0f};
    static_assert(BITS == 16 || C::NG < 8, "the V zero-point MMA keeps one spare row for the P sums");
    const int src0 = t * 4 + (g >> 1), src1 = (t + 4) * 4 + (g >> 1);
    const bool odd_head = g & 1;

    if constexpr (BITS == 16) {
        // ---- bf16 token-drop cache: query fragments (B of S^T = K Q^T) ----
        uint32_t bq[C::NT][2];
#pragma unroll
        for (int ks = 0; ks < C::NT; ++ks) {
            // per pair of k-steps, thread t holds channels 8t..8t+7 of a 32-block
            const int kk = ks >> 1, second = ks & 1;
            const int c0 = 32 * kk + 8 * t + 4 * second;
            bq[ks][0] = pack_bf16(bf16_bits_to_f32(qs[g * D + c0]), bf16_bits_to_f32(qs[g * D + c0 + 1]));
            bq[ks][1] = pack_bf16(bf16_bits_to_f32(qs[g * D + c0 + 2]), bf16_bits_to_f32(qs[g * D + c0 + 3]));
        }
        for (int k = 0; k < nw; ++k) {
            const int st = k % C::NSTAGE;
            if (!mbar_wait(&bars[st], (k / C::NSTAGE) & 1, a.status, a.wait_ns)) break;
            const uint8_t *kb = ring + st * C::STAGE;
            uint8_t *vb = ring + st * C::STAGE + C::HB;
            const int pg = p0 + warp + NW * k;
            if (!sflag[st]) {  // reported at issue time; page 0's blocks landed here
                __syncwarp();
                if (k + C::NSTAGE < nw) {
                    advance_rows(k + C::NSTAGE);
                    issue(k + C::NSTAGE);
                }
                continue;
            }
            const int slot0 = 2 * g, slot1 = 2 * g + 1;
            const int pos0 = pg * kPage + slot0;
            // even and odd k-steps in two accumulators: two MMA chains of NT / 2
            float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < C::NT / 2; ++kk) {
                const uint4 u0 = *reinterpret_cast<const uint4 *>(kb + slot0 * D * 2 + (32 * kk + 8 * t) * 2);
                const uint4 u1 = *reinterpret_cast<const uint4 *>(kb + slot1 * D * 2 + (32 * kk + 8 * t) * 2);
                const uint32_t a0[4] = {u0.x, u1.x, u0.y, u1.y};
                const uint32_t a1[4] = {u0.z, u1.z, u0.w, u1.w};
                mma_bf16(acc, a0, bq[2 * kk][0], bq[2 * kk][1]);
                mma_bf16(acc2, a1, bq[2 * kk + 1][0], bq[2 * kk + 1][1]);
            }
            float s[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) s[j] = (acc[j] + acc2[j]) * a.scale_log2;
            if (pos0 >= len) s[0] = s[1] = -INFINITY;
            if (pos0 + 1 >= len) s[2] = s[3] = -INFINITY;

            float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            const float mn0 = mx0 > m[0] ? mx0 + kLazyRef : m[0];
            const float mn1 = mx1 > m[1] ? mx1 + kLazyRef : m[1];
            if (__any_sync(0xffffffffu, mn0 > m[0] || mn1 > m[1])) {
                const float al0 = mn0 == -INFINITY ? 1.0f : ex2(m[0] - mn0);
                const float al1 = mn1 == -INFINITY ? 1.0f : ex2(m[1] - mn1);
#pragma unroll
                for (int i = 0; i < C::NT; ++i) {
                    o[i][0] *= al0; o[i][2] *= al0;
                    o[i][1] *= al1; o[i][3] *= al1;
                }
                l[0] *= al0;
                l[1] *= al1;
                m[0] = mn0;
                m[1] = mn1;
            }
            const float ms0 = m[0] == -INFINITY ? 0.0f : m[0], ms1 = m[1] == -INFINITY ? 0.0f : m[1];
            const float p[4] = {ex2(s[0] - ms0), ex2(s[1] - ms1), ex2(s[2] - ms0), ex2(s[3] - ms1)};
            l[0] += p[0] + p[2];
            l[1] += p[1] + p[3];

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
            __syncwarp();
            if (k + C::NSTAGE < nw) {
                advance_rows(k + C::NSTAGE);
                issue(k + C::NSTAGE);
            }
        }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l[0] += __shfl_xor_sync(0xffffffffu, l[0], off);
            l[1] += __shfl_xor_sync(0xffffffffu, l[1], off);
        }
    } else {
        // ---- quantised cache ----
        // (query fragments packed in the prologue above)
        const uint32_t *qfrag = reinterpret_cast<const uint32_t *>(qsum + 8 * C::NG);
        // Zero-point term of the scores as one more MMA: k-slots (2t, 2t+1)
        // carry groups (2P, 2P+1), P = t & 1, as the hi (t < 2) or lo (t >= 2)
        // f16 part of the pre-scaled query group sums.
        const int zp = t & 1;
        const bool zuse = C::NG >= 4 || 2 * zp + 1 < C::NG;  // always with four or more groups
        uint32_t bz = 0u;
        if (zuse) {
            const float s0 = qsum[g * C::NG + 2 * zp], s1 = qsum[g * C::NG + 2 * zp + 1];
            const __half h0 = __float2half_rn(s0), h1 = __float2half_rn(s1);
            if (t < 2) {
                bz = pack_f16(__half2float(h0), __half2float(h1));
            } else {
                bz = pack_f16(s0 - __half2float(h0), s1 - __half2float(h1));
            }
        }
        float oz[4] = {0.f, 0.f, 0.f, 0.f};  // V zero-point term, rows = groups, columns = heads
        float ms0 = 0.0f, ms1 = 0.0f;         // running max as subtracted (0 while it is -inf)
        float nm[4] = {0.f, 0.f, 0.f, 0.f};   // minus the running max, per accumulator column
        bool fresh = true;                    // a head column has seen no score yet
        const float kscale = a.scale_log2 * 16777216.0f;  // products carry 2^-24
        constexpr float kVhi = VReg<BITS, D>::VHI == 4 ? 0.0625f : 0.25f;
        const uint32_t vhi_scale = pack_f16(kVhi, kVhi);

        // NPG (1 or 2) consecutive pages of the warp: k = the first page's
        // index, its ring stage S0 and S0 + 1 compile-time constants of the
        // unrolled driver below.  Two pages share the query-fragment loads,
        // the rescale check and the copy bookkeeping, and give the scheduler
        // two independent MMA chains.
        // MASK: the page may end inside (the request's ragged last page):
        // scores and V parameters of the slots past the end are masked.
        // Every other page is full.  S0 is a compile-time constant on the
        // unrolled path (an int for the masked last page).
        auto body = [&](int k, auto s0c, uint32_t parity, auto npc, auto maskc) -> bool {
            const int S0 = stage_value(s0c);
            constexpr int NPG = decltype(npc)::value;
            constexpr bool MASK = decltype(maskc)::value;
            int nvalid[NPG];
#pragma unroll
            for (int i = 0; i < NPG; ++i) {
                if (!mbar_wait(&bars[S0 + i], parity, a.status, a.wait_ns)) return false;
                // slots >= nvalid are past the end (used by the masked body only)
                const int pg = p0 + warp + NW * (k + i);
                nvalid[i] = len - pg * kPage;
            }

            // ---- shared-memory reads of the pages' K rows and parameters ----
            KRow<BITS, D> r0[NPG], r1[NPG];  // tokens g (rows g) and g+8 (rows g+8)
            float sc0[NPG][C::NG], sc1[NPG][C::NG];
            uint32_t kza0[NPG], kza1[NPG];
#pragma unroll
            for (int i = 0; i < NPG; ++i) {
                const uint8_t *kb = ring + (S0 + i) * C::STAGE;
                r0[i].load(kb + g * (D * BITS / 8), t);
                r1[i].load(kb + (g + 8) * (D * BITS / 8), t);
                const __half *ksc = reinterpret_cast<const __half *>(kb + C::CR);
                const __half *kzr = ksc + kPage * C::NG;
                load_halves<C::NG>(ksc + g * C::NG, sc0[i]);
                load_halves<C::NG>(ksc + (g + 8) * C::NG, sc1[i]);
                kza0[i] = kza1[i] = 0u;
                if (zuse) {
                    kza0[i] = *reinterpret_cast<const uint32_t *>(kzr + g * C::NG + 2 * zp);
                    kza1[i] = *reinterpret_cast<const uint32_t *>(kzr + (g + 8) * C::NG + 2 * zp);
                }
            }
            // ---- S^T = K Q^T per group, scaled and summed ----
            f2 s01[NPG], s23[NPG];
#pragma unroll
            for (int i = 0; i < NPG; ++i) s01[i] = s23[i] = f2{0.f, 0.f};
#pragma unroll
            for (int gr = 0; gr < C::NG; ++gr) {
                const uint4 qb = *reinterpret_cast<const uint4 *>(qfrag + (gr * 32 + lane) * 4);
#pragma unroll
                for (int i = 0; i < NPG; ++i) {
                    float acc[4];
                    {
                        const int ks = 2 * gr;
                        const uint32_t af[4] = {r0[i].reg(2 * ks), r1[i].reg(2 * ks), r0[i].reg(2 * ks + 1),
                                                r1[i].reg(2 * ks + 1)};
                        mma_f16_z(acc, af, qb.x, qb.y);
                    }
                    {
                        const int ks = 2 * gr + 1;
                        const uint32_t af[4] = {r0[i].reg(2 * ks), r1[i].reg(2 * ks), r0[i].reg(2 * ks + 1),
                                                r1[i].reg(2 * ks + 1)};
                        mma_f16(acc, af, qb.z, qb.w);
                    }
                    s01[i].x = fmaf(sc0[i][gr], acc[0], s01[i].x);
                    s01[i].y = fmaf(sc0[i][gr], acc[1], s01[i].y);
                    s23[i].x = fmaf(sc1[i][gr], acc[2], s23[i].x);
                    s23[i].y = fmaf(sc1[i][gr], acc[3], s23[i].y);
                }
            }
            // zero-point term, accumulated onto minus the running max
            float x[NPG][4];  // log2 score - running max
            float mx = -INFINITY;
#pragma unroll
            for (int i = 0; i < NPG; ++i) {
                float z[4];
                const uint32_t za[4] = {kza0[i], kza1[i], 0u, 0u};
                mma_f16_c(z, za, bz, 0u, nm);
                const f2 x01 = fma2(s01[i], f2{kscale, kscale}, f2{z[0], z[1]});
                const f2 x23 = fma2(s23[i], f2{kscale, kscale}, f2{z[2], z[3]});
                x[i][0] = x01.x; x[i][1] = x01.y; x[i][2] = x23.x; x[i][3] = x23.y;
                if (MASK && nvalid[i] < kPage) {  // ragged last page: mask the scores of empty slots
                    if (g >= nvalid[i]) x[i][0] = x[i][1] = -INFINITY;
                    if (g + 8 >= nvalid[i]) x[i][2] = x[i][3] = -INFINITY;
                }
                mx = fmaxf(mx, fmaxf(fmaxf(x[i][0], x[i][1]), fmaxf(x[i][2], x[i][3])));
            }

            // ---- online softmax: rescale only when a score beats the running reference ----
            if (__any_sync(0xffffffffu, mx > 0.0f || fresh)) {
                float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                for (int i = 0; i < NPG; ++i) {
                    x[i][0] += ms0; x[i][1] += ms1; x[i][2] += ms0; x[i][3] += ms1;
                    mx0 = fmaxf(mx0, fmaxf(x[i][0], x[i][2]));
                    mx1 = fmaxf(mx1, fmaxf(x[i][1], x[i][3]));
                }
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                }
                const float mn0 = mx0 > m[0] ? mx0 + kLazyRef : m[0];
                const float mn1 = mx1 > m[1] ? mx1 + kLazyRef : m[1];
                const float al0 = (mn0 == -INFINITY || m[0] == mn0) ? 1.0f : ex2(m[0] - mn0);
                const float al1 = (mn1 == -INFINITY || m[1] == mn1) ? 1.0f : ex2(m[1] - mn1);
#pragma unroll
                for (int i = 0; i < C::NT; ++i) {
                    o[i][0] *= al0; o[i][2] *= al0;
                    o[i][1] *= al1; o[i][3] *= al1;
                }
                oz[0] *= al0; oz[2] *= al0;
                oz[1] *= al1; oz[3] *= al1;
                m[0] = mn0;
                m[1] = mn1;
                fresh = mn0 == -INFINITY || mn1 == -INFINITY;
                ms0 = mn0 == -INFINITY ? 0.0f : mn0;
                ms1 = mn1 == -INFINITY ? 0.0f : mn1;
                nm[0] = nm[2] = -ms0;
                nm[1] = nm[3] = -ms1;
#pragma unroll
                for (int i = 0; i < NPG; ++i) {
                    x[i][0] -= ms0; x[i][1] -= ms1; x[i][2] -= ms0; x[i][3] -= ms1;
                }
            }
#pragma unroll
            for (int i = 0; i < NPG; ++i) {
                const uint8_t *vb = ring + (S0 + i) * C::STAGE + C::HB;
                const uint8_t *vpar = vb + C::CR;
                uint32_t vsc[2 * C::NG];  // per group: scales of tokens (2t, 2t+1), then (2t+8, 2t+9)
                {
                    const uint32_t *pp = reinterpret_cast<const uint32_t *>(vpar + t * 8 * C::NG);
#pragma unroll
                    for (int j = 0; j < 2 * C::NG; j += 4) {
                        const uint4 u = *reinterpret_cast<const uint4 *>(pp + j);
                        vsc[j] = u.x; vsc[j + 1] = u.y; vsc[j + 2] = u.z; vsc[j + 3] = u.w;
                    }
                }
                // A of the V zero-point MMA: rows 0..G-1 the group's zero
                // points of tokens (2t, 2t+1) / (2t+8, 2t+9); row G ones, so
                // the MMA also sums P over the page (the softmax denominator)
                // (every lane loads -- the rows past the groups read group 0's
                // words and drop them -- so the warp does not diverge)
                const int gz = g < C::NG ? g : 0;
                const uint2 u = *reinterpret_cast<const uint2 *>(vpar + kPage * C::NG * 2 + (t * C::NG + gz) * 8);
                const uint32_t vone = g == C::NG ? 0x3C003C00u : 0u;
                uint32_t vza0 = g < C::NG ? u.x : vone;
                uint32_t vza2 = g < C::NG ? u.y : vone;
                if (MASK && nvalid[i] < kPage) {  // empty slots' V parameters may hold anything (0 x NaN)
                    const int nv = nvalid[i];
                    const uint32_t mlo = (2 * t < nv ? 0x0000FFFFu : 0u) | (2 * t + 1 < nv ? 0xFFFF0000u : 0u);
                    const uint32_t mhi = (2 * t + 8 < nv ? 0x0000FFFFu : 0u) | (2 * t + 9 < nv ? 0xFFFF0000u : 0u);
#pragma unroll
                    for (int gr = 0; gr < C::NG; ++gr) {
                        vsc[2 * gr] &= mlo;
                        vsc[2 * gr + 1] &= mhi;
                    }
                    vza0 &= mlo;
                    vza2 &= mhi;
                }
                VReg<BITS, D> vs;
                vs.load(vb, g, t);
                const float p[4] = {ex2(x[i][0]), ex2(x[i][1]), ex2(x[i][2]), ex2(x[i][3])};

                // ---- P^T as the B operand (k-slot = token, column = head):
                // the score fragment rows 0-7 / 8-15 transposed ----
                const uint32_t blo = movmatrix_t(pack_f16(p[0], p[1]));
                const uint32_t bhi = movmatrix_t(pack_f16(p[2], p[3]));
                const uint32_t bhi_s = hmul2(bhi, vhi_scale);

                // ---- O^T += V^T (P s)^T, zero points as one more MMA ----
#pragma unroll
                for (int gr = 0; gr < C::NG; ++gr) {
                    const uint32_t b0 = hmul2(blo, vsc[2 * gr]), b1 = hmul2(bhi_s, vsc[2 * gr + 1]);
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int mt = 2 * gr + h2;
                        uint32_t af[4];
                        vs.regs(mt, af);
                        mma_f16(o[mt], af, b0, b1);
                    }
                }
                {
                    const uint32_t za[4] = {vza0, 0u, vza2, 0u};
                    mma_f16(oz, za, blo, bhi);
                }
            }
            __syncwarp();
#pragma unroll
            for (int i = 0; i < NPG; ++i)
                if (k + i + C::NSTAGE < nw) issue(k + i + C::NSTAGE);
            return true;
        };
        // driver: pairs of stages in order, the ring indices known at compile
        // time (NSTAGE = 4: pages k0, k0+1 in stages 0, 1; k0+2, k0+3 in 2, 3)
        static_assert(C::NSTAGE == 4, "the driver below unrolls a 4-stage ring");
        using I0 = std::integral_constant<int, 0>;
        using I1 = std::integral_constant<int, 1>;
        using I2 = std::integral_constant<int, 2>;
        // the warp's last page is masked on its own when the request ends
        // inside it; all other pages take the unmasked body (a bad page id is
        // reported, and its stage holds page 0's blocks: finite, the result
        // of that request void)
        using NoMask = std::false_type;
        const int last = nw - 1;
        const bool mask_last = nw > 0 && len - (p0 + warp + NW * last) * kPage < kPage;
        const int nfull = mask_last ? last : nw;
        bool ok = true;
        for (int k0 = 0; k0 < nfull && ok; k0 += C::NSTAGE) {
            const uint32_t parity = (uint32_t)(k0 / C::NSTAGE) & 1u;
            advance_rows(k0 + C::NSTAGE);  // the copies issued below: pages k0 + 4 .. k0 + 7, one block
            if (k0 + 1 < nfull)
                ok = body(k0, I0{}, parity, I2{}, NoMask{});
            else
                ok = body(k0, I0{}, parity, I1{}, NoMask{});
            if (!ok) break;
            if (k0 + 3 < nfull)
                ok = body(k0 + 2, I2{}, parity, I2{}, NoMask{});
            else if (k0 + 2 < nfull)
                ok = body(k0 + 2, I2{}, parity, I1{}, NoMask{});
        }
        if (ok && mask_last)
            body(last, last % C::NSTAGE, (uint32_t)(last / C::NSTAGE) & 1u, I1{}, std::true_type{});
        l[0] = __shfl_sync(0xffffffffu, oz[0], C::NG * 4 + t);
        l[1] = __shfl_sync(0xffffffffu, oz[1], C::NG * 4 + t);
        // ---- finish O^T: codes part (2^24, rows g+8 2^(24 - ROW8)) + zero-point part of the group ----
        constexpr float kRow8 = VReg<BITS, D>::ROW8 == 4 ? 1048576.0f : 16777216.0f;
#pragma unroll
        for (int gr = 0; gr < C::NG; ++gr) {
            const float z0 = __shfl_sync(0xffffffffu, oz[0], gr * 4 + t);
            const float z1 = __shfl_sync(0xffffffffu, oz[1], gr * 4 + t);
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int mt = 2 * gr + h2;
                o[mt][0] = fmaf(o[mt][0], 16777216.0f, z0);
                o[mt][1] = fmaf(o[mt][1], 16777216.0f, z1);
                o[mt][2] = fmaf(o[mt][2], kRow8, z0);
                o[mt][3] = fmaf(o[mt][3], kRow8, z1);
            }
        }
    }

    // ---- combine the warps of the CTA in shared memory ----
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

// Combine the first `count` chunk partials of one (request, head) row (of
// n_splits slots), in chunk order.
template <int D>
__device__ __forceinline__ void reduce_row(const float *ws_o, const float *ws_ml, int n_splits, int count,
                                           int64_t row, float *out, int tid, int nthreads) {
    combine_partials<D>(ws_o, ws_ml, n_splits, count, row, out, tid, nthreads);
}

}  // namespace draft
}  // namespace vc
