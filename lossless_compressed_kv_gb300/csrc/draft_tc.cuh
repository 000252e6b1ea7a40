// Draft attention over a quantised (2-, 3- or 4-bit) KV_comp on the
// 5th-generation tensor cores (tcgen05 + TMEM).  Device body shared by the
// draft launch and the mixed draft / verify launch.
//
// "VeriCache: Making Lossy KV Compression Exact", "The Core Idea" items 1-2
// (the drafter reads the compressed cache, one query per head and step) and
// "Verifying Without Giving Back the Speedup" (drafting is bound by the
// bytes of the compressed cache it streams).
//
// A CTA owns one (request, kv head, context chunk) and walks it in tiles of
// 8 pages = 128 tokens.  Roles (224 threads, two CTAs per SM):
//  - warp 4, producer: 16 lanes issue one bulk copy each per tile (the K and
//    the V head block of 8 pages) into a 3-stage ring.
//  - warps 0-3, 128 threads: thread i unpacks token i's K codes into TMEM
//    lane i (operand A1 of the score product) and channel i's V codes for the
//    tile's 128 tokens into TMEM lane i (operand A2 of the P V product); as
//    the owner of token i it turns its row of scores into probabilities and
//    writes token i's column of the P V product's B operand.  The loop is
//    software-pipelined: the next tile's K codes are unpacked and stored
//    while this tile's scores are read back, and the next tile's V codes
//    after this tile's probabilities.
//  - warp 5 issues the score products, warp 6 the P V products (one
//    tcgen05.mma costs its issuing thread about 100 cycles whatever its
//    size, so the two chains get a thread each).
// Products (f16 operands, fp32 accumulate; every code enters as an exact
// f16 subnormal code * 2^(P - 24), its partner operand pre-scaled by 2^-P):
//    S[t][g GP + h]  = sum_{c in group g} code_K[t][c] q_h[c]          (A1 x B1)
//    score_h[t]      = scale_log2 (2^24 sum_g scale_K[t][g] S[t][g GP + h]
//                                  + sum_g zero_K[t][g] q-sum_h[g])
//    O^T[c][g GP + h] += sum_t code_V[c][t] (p_h[t] scale_V[t][g] 2^-P)  (A2 x B2)
//    out_h[c]        = 2^24 O^T[c][g(c) GP + h] + sum_t zero_V[t][g(c)] p_h[t]
// so no dequantised value is ever rounded; the zero-point sums and the
// softmax denominators are fp32 per-thread partials, reduced at the end.
// Softmax: one reference maximum per head for the whole CTA, raised (with a
// rescale of O in TMEM and of the partials) only when a score passes it by
// more than 2^8, so P stays below 2^8; every tile the 128 threads vote on
// that with one named-barrier reduction.
#pragma once

#include "draft_impl.cuh"
#include "tmem_io.cuh"
#include "verify_tc.cuh"

namespace vc {
namespace dtc {

using draft::DraftArgs;

template <int BITS_, int D, int GP>
struct Cfg {
    static constexpr int BITS = BITS_;
    static constexpr int NG = D / 32;                  // quantisation groups
    static constexpr int HB = 2 * D * (BITS + 1);      // head block bytes
    static constexpr int CR = kPage * D * BITS / 8;    // code region bytes
    static constexpr int ROWB = D * BITS / 8;          // one token's K codes
    static constexpr int TP = 8;                       // pages per tile
    static constexpr int TOK = TP * kPage;             // tokens per tile (MMA M / K)
    static constexpr int STAGE = TP * 2 * HB;          // K blocks, then V blocks
    static constexpr int NST = 3;
    static constexpr int NC = NG * GP;                 // (group, head) columns of S and O
    static constexpr int N = NC < 16 ? 16 : NC;        // MMA N (multiple of 16)
    static constexpr int KAT1 = D / 64;                // 64-element swizzle atoms of B1 (K = D)
    static constexpr int KAT2 = TOK / 64;              // ... of B2 (K = 128 tokens)
    static constexpr int A1C = D / 2;                  // columns of A1
    // TMEM columns: O, two A2 buffers, A1, S
    static constexpr uint32_t O_COL = 0, A2_COL = 32, A1_COL = 160, D1_COL = 224;
    static constexpr int TMEM_COLS = 256;
    static_assert(N <= 32 && A1_COL + A1C <= D1_COL && D1_COL + N <= TMEM_COLS, "TMEM map");
    // shared memory, from a 1024-byte aligned base
    static constexpr int B1_BYTES = KAT1 * N * 128;              // [KAT1][N rows][128 B], K-major, 128B swizzle
    static constexpr int B2_BYTES = KAT2 * N * 128;              // per buffer, same layout, K = token
    static constexpr int OFF_B1 = 0;
    static constexpr int OFF_B2 = OFF_B1 + B1_BYTES;
    static constexpr int OFF_RING = OFF_B2 + 2 * B2_BYTES;
    static constexpr int OFF_MISC = OFF_RING + NST * STAGE;
    static constexpr int NRED = NC + GP;                         // reduced values per warp
    static constexpr int NBAR = 2 * NST + 8;
    static constexpr int OFF_QZ = NBAR * 8 + NST * 4 + 16;       // [NG][GP] scale_log2 x q group sums
    static constexpr int OFF_TMX = OFF_QZ + NG * GP * 4;         // [4][GP]
    static constexpr int OFF_RED = OFF_TMX + 4 * GP * 4;         // [4][NRED]
    static constexpr int MISC = OFF_RED + 4 * NRED * 4 + 16;
    static constexpr int SMEM = OFF_MISC + MISC + 1024;
    // staging area for the queries in the prologue (reuses the ring)
    static_assert(GP * D * 2 <= NST * STAGE, "query staging");
    // at most two CTAs per SM: each holds 256 TMEM columns
    static constexpr int SMEM_ALLOC = SMEM < 80 * 1024 ? 80 * 1024 : SMEM;
    static constexpr int THREADS = 224;
};

// Instruction descriptor, kind::f16: fp32 accumulate, f16 A and B, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16(int m, int n) {
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// Bit position of a 2-bit code's column register j (0..7) of a word after
// unpacking: j < 5 unshifted at 2 j, j >= 5 at 2 (j - 5) after a shift by 10.
__host__ __device__ constexpr int cpos(int j) { return j < 5 ? 2 * j : 2 * (j - 5); }

// Bit position (pre-scale exponent of the partner operand) of the V codes of
// token pair j = slot / 2 of a page in their A2 column register.
template <int BITS>
__host__ __device__ constexpr int vpos(int j) {
    return BITS == 2 ? cpos(j) : BITS == 3 ? 2 * (j & 3) : 4 * (j & 1);
}

// The 8 column registers of one word of 2-bit codes (code pairs at the same
// position of both halves, exact f16 subnormals code * 2^(cpos - 24)).
__device__ inline void unpack8(uint32_t w, uint32_t *r) {
    const uint32_t w10 = w >> 10;
    r[0] = w & 0x00030003u;
    r[1] = w & 0x000C000Cu;
    r[2] = w & 0x00300030u;
    r[3] = w & 0x00C000C0u;
    r[4] = w & 0x03000300u;
    r[5] = w10 & 0x00030003u;
    r[6] = w10 & 0x000C000Cu;
    r[7] = w10 & 0x00300030u;
}

// Channel c's V codes of one page (block code region vb) as its 8 A2
// column registers (token pairs (2j, 2j + 1)), exact f16 subnormals
// code * 2^(vpos(j) - 24).
template <int BITS, int D>
__device__ inline void unpack_v(const uint8_t *vb, int c, uint32_t *r) {
    if constexpr (BITS == 2) {
        unpack8(*reinterpret_cast<const uint32_t *>(vb + 4 * c), r);
    } else if constexpr (BITS == 3) {
        // low two bits as 2 bits at positions 2 (j & 3); the high bit from the
        // channel pair's word, moved to its code's bit 2
        const uint32_t lo = *reinterpret_cast<const uint32_t *>(vb + 4 * c);
        const uint32_t x = *reinterpret_cast<const uint32_t *>(vb + 4 * D + 4 * (c >> 1)) >> (c & 1);
        const uint32_t lo8 = lo >> 8, xl = x << 2, xr = x >> 6;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            r[j] = (lo & (0x00030003u << (2 * j))) | (xl & (0x00040004u << (2 * j)));
            r[4 + j] = (lo8 & (0x00030003u << (2 * j))) | (xr & (0x00040004u << (2 * j)));
        }
    } else {
        const uint2 u = *reinterpret_cast<const uint2 *>(vb + 8 * c);
        const uint32_t y0 = u.x >> 8, y1 = u.y >> 8;
        r[0] = u.x & 0x000F000Fu; r[1] = u.x & 0x00F000F0u; r[2] = y0 & 0x000F000Fu; r[3] = y0 & 0x00F000F0u;
        r[4] = u.y & 0x000F000Fu; r[5] = u.y & 0x00F000F0u; r[6] = y1 & 0x000F000Fu; r[7] = y1 & 0x00F000F0u;
    }
}

// A token's K codes (its row of a K head block) as its D/2 A1 column
// registers: column t (D/8) + r = register r of the row's thread region t,
// channels 16 (r >> 1) + 4 t + 2 (r & 1) + {0, 1}.
template <int BITS, int D>
__device__ inline void unpack_k(const uint8_t *row, uint32_t *r) {
    if constexpr (BITS == 2) {
        uint32_t wds[D / 16];
        const uint4 *rp = reinterpret_cast<const uint4 *>(row);
#pragma unroll
        for (int x = 0; x < D / 64; ++x) {
            const uint4 u = rp[x];
            wds[4 * x] = u.x; wds[4 * x + 1] = u.y; wds[4 * x + 2] = u.z; wds[4 * x + 3] = u.w;
        }
#pragma unroll
        for (int x = 0; x < D / 16; ++x) unpack8(wds[x], r + 8 * x);
    } else {
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            draft::KRow<BITS, D> kr;
            kr.load(row, t);
#pragma unroll
            for (int x = 0; x < D / 8; ++x) r[t * (D / 8) + x] = kr.reg(x);
        }
    }
}

// Named barrier 1 over the 128 threads of warps 0-3, OR of a predicate.
__device__ inline bool bar_or_128(bool v) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(out)
        : "r"((uint32_t)v)
        : "memory");
    return out != 0;
}
__device__ inline void bar_sync_128() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ inline float half_bits_to_f32(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// Byte offset of element (row n, K index k) of a K-major, 128-byte-swizzled
// operand tile of `rows` rows.
__device__ inline int kmaj(int n, int k, int rows) {
    return (k >> 6) * (rows * 128) + n * 128 + ((((k >> 3) & 7) ^ (n & 7)) << 4) + (k & 7) * 2;
}

template <int BITS, int D, int GP>
__device__ __forceinline__ void draft_tc_block(const DraftArgs &a, int split, int kvh, int b, int chunk,
                                               uint8_t *smem_raw) {
    using C = Cfg<BITS, D, GP>;
    using namespace tmemio;
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t *sB1 = smem + C::OFF_B1;
    uint8_t *sB2 = smem + C::OFF_B2;  // [2 buffers]
    uint8_t *ring = smem + C::OFF_RING;
    uint8_t *misc = smem + C::OFF_MISC;
    uint64_t *full = reinterpret_cast<uint64_t *>(misc);
    uint64_t *empty = full + C::NST;
    uint64_t *a1r = empty + C::NST;  // A1 written (one arrival per compute warp)
    uint64_t *sr = a1r + 1;          // scores ready (MMA commit)
    uint64_t *a2r = sr + 1;          // [2] A2 buffer written (4 arrivals)
    uint64_t *pr = a2r + 2;          // [2] B2 buffer written (4 arrivals)
    uint64_t *pvd = pr + 2;          // [2] P V of the buffer done (MMA commit)
    uint32_t *smask = reinterpret_cast<uint32_t *>(full + C::NBAR);  // [NST] valid pages of a stage
    uint32_t *tslot = smask + C::NST;
    int *dead_any = reinterpret_cast<int *>(tslot + 1);
    float *qz = reinterpret_cast<float *>(misc + C::OFF_QZ);
    float *tmx = reinterpret_cast<float *>(misc + C::OFF_TMX);
    float *red = reinterpret_cast<float *>(misc + C::OFF_RED);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int grp = a.grp;
    const int32_t *trow = a.table + (int64_t)b * a.maxb;
    const int len = a.lens[b];
    const int npages = ceil_div(len, kPage);
    const int p0 = split * chunk;
    const int p1 = min(p0 + chunk, npages);
    const int ntile = p1 > p0 ? ceil_div(p1 - p0, C::TP) : 0;

    // ---- set-up ----
    if (tid == 0) {
        for (int i = 0; i < C::NST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 4);
        }
        mbar_init(a1r, 4);
        mbar_init(sr, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&a2r[i], 4);
            mbar_init(&pr[i], 4);
            mbar_init(&pvd[i], 1);
        }
        *dead_any = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                     "r"(C::TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (a.k_new != nullptr && warp == 1) {
        // vc_draft_step: the CTA whose pages hold slot[b] writes the step's
        // new entry there before any copy is issued (no other CTA reads that
        // page)
        const int s = a.slot[b];
        if (split == 0 && kvh == 0 && (s < 0 || s >= len) && lane == 0) report(a.status, VC_ERR_INVALID_ARG);
        const int pi = (s >= 0 && s < len) ? s / kPage : -1;
        if (pi >= p0 && pi < p1) {
            __shared__ uint32_t krow[D * BITS / 32];
            const int id = pi < a.maxb ? trow[pi] : -1;
            if (id >= 0 && id < a.n_pages) {
                const int64_t off = ((int64_t)id * a.hkv + kvh) * C::HB;
                const int64_t row = ((int64_t)b * a.hkv + kvh) * D;
                qrow::append_entry<BITS, D>(reinterpret_cast<const uint8_t *>(a.k_new + row),
                                            reinterpret_cast<const uint8_t *>(a.v_new + row),
                                            const_cast<uint8_t *>(a.kp) + off, const_cast<uint8_t *>(a.vp) + off,
                                            s % kPage, lane, krow);
                // visible to the bulk copies (async proxy) issued after the barrier
                asm volatile("fence.proxy.async.global;" ::: "memory");
            } else if (lane == 0) {
                report(a.status, VC_ERR_BAD_INDEX);
            }
        }
    }
    // The group's queries, staged in the ring (refilled later): bf16 [GP][D]
    uint16_t *qs = reinterpret_cast<uint16_t *>(ring);
    {
        const uint32_t *src = reinterpret_cast<const uint32_t *>(a.q + ((int64_t)b * a.hq + kvh * grp) * D);
        uint32_t *dst = reinterpret_cast<uint32_t *>(qs);
        for (int e = tid; e < GP * D / 2; e += C::THREADS) dst[e] = e < grp * D / 2 ? src[e] : 0u;
    }
    __syncthreads();
    if (tid < C::NG * GP) {  // scale_log2 x the group sums of each head's query
        const int g = tid / GP, h = tid % GP;
        float sum = 0.0f;
        for (int i = 0; i < kGroup; ++i) sum += bf16_bits_to_f32(qs[h * D + g * kGroup + i]);
        qz[tid] = sum * a.scale_log2;
    }
    // B1 [N rows][D K elements]: row n < NC = (group g, head h) holds q_h
    // pre-scaled at the K elements of group g's channels; 0 elsewhere
    for (int e = tid; e < C::KAT1 * C::N * 8; e += C::THREADS) {
        const int at = e / (C::N * 8), n = (e / 8) % C::N, ch = e % 8;
        uint32_t w[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            float v2[2];
#pragma unroll
            for (int hl = 0; hl < 2; ++hl) {
                const int k = at * 64 + ch * 8 + 2 * x + hl;
                float v = 0.0f;
                const int g = n / GP, h = n % GP;
                if (n < C::NC && h < grp) {
                    const int col = k >> 1, t = col / (D / 8), r = col % (D / 8);
                    const int c = 16 * (r >> 1) + 4 * t + 2 * (r & 1) + hl;
                    if ((c >> 5) == g)
                        v = bf16_bits_to_f32(qs[h * D + c]) *
                            __uint_as_float((uint32_t)(127 - draft::kpos<BITS>(r)) << 23);
                }
                v2[hl] = v;
            }
            w[x] = pack_f16(v2[0], v2[1]);
        }
        *reinterpret_cast<uint4 *>(sB1 + at * (C::N * 128) + n * 128 + (((ch ^ (n & 7))) << 4)) =
            make_uint4(w[0], w[1], w[2], w[3]);
    }
    // B2 buffers: rows >= NC stay zero
    for (int e = tid; e < 2 * C::B2_BYTES / 16; e += C::THREADS)
        reinterpret_cast<uint4 *>(sB2)[e] = make_uint4(0u, 0u, 0u, 0u);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    vtc::tc_fence_before();
    __syncthreads();  // queries read: the ring is free for the copies
    vtc::tc_fence_after();
    const uint32_t tmem = *tslot;

    constexpr uint32_t IDESC = idesc_f16(128, C::N);
    const uint64_t kWait = a.wait_ns;

    if (warp == 4) {
        // ================= producer: bulk copies of 8 pages per tile =================
        bool alive = true;
        for (int j = 0; j < ntile && alive; ++j) {
            const int st = j % C::NST;
            if (j >= C::NST)
                alive = __all_sync(0xffffffffu, mbar_wait(&empty[st], ((j / C::NST) - 1) & 1, a.status, kWait));
            if (!alive) break;
            const int k = lane & 7, pg = p0 + j * C::TP + k;
            int id = -1;
            if (lane < 16 && pg < p1) {
                id = pg < a.maxb ? trow[pg] : -1;
                if (id < 0 || id >= a.n_pages) {
                    if (lane < 8) report(a.status, VC_ERR_BAD_INDEX);
                    id = -1;
                }
            }
            const uint32_t vm = __ballot_sync(0xffffffffu, lane < 8 && id >= 0);
            if (a.skip_copies) continue;  // fault injection: no copy and no arrival
            if (lane == 0) {
                smask[st] = vm;
                mbar_arrive_expect_tx(&full[st], (uint32_t)__popc(vm) * 2u * C::HB);
            }
            __syncwarp();
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            if (lane < 16 && id >= 0) {
                const int64_t off = ((int64_t)id * a.hkv + kvh) * C::HB;
                bulk_g2s(ring + st * C::STAGE + (lane < 8 ? 0 : C::TP * C::HB) + k * C::HB,
                         (lane < 8 ? a.kp : a.vp) + off, C::HB, &full[st]);
            }
        }
    } else if (warp == 5) {
        // ================= score products S = A1 B1 =================
        if (lane == 0) {
            for (int j = 0; j < ntile; ++j) {
                if (!mbar_wait(a1r, j & 1, a.status, kWait)) break;
                vtc::tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    vtc::umma_ta(tmem + C::D1_COL, tmem + C::A1_COL + ks * 8,
                                 vtc::sdesc(smem_u32(sB1) + (ks >> 2) * (C::N * 128) + (ks & 3) * 32, 16, 1024),
                                 IDESC, ks > 0);
                vtc::umma_commit(sr);
            }
        }
    } else if (warp == 6) {
        // ================= P V products O += A2 B2 =================
        if (lane == 0) {
            for (int j = 0; j < ntile; ++j) {
                const int bf = j & 1;
                if (!mbar_wait(&a2r[bf], (j >> 1) & 1, a.status, kWait)) break;
                if (!mbar_wait(&pr[bf], (j >> 1) & 1, a.status, kWait)) break;
                vtc::tc_fence_after();
                const uint32_t b2 = smem_u32(sB2 + bf * C::B2_BYTES);
#pragma unroll
                for (int kk = 0; kk < C::TOK / 16; ++kk)
                    vtc::umma_ta(tmem + C::O_COL, tmem + C::A2_COL + bf * 64 + kk * 8,
                                 vtc::sdesc(b2 + (kk >> 2) * (C::N * 128) + (kk & 3) * 32, 16, 1024), IDESC,
                                 (j > 0 || kk > 0));
                vtc::umma_commit(&pvd[bf]);
            }
        }
    } else {
        // ================= warps 0-3: unpack, softmax, partials =================
        const int i = tid;  // token of the tile (K side, softmax); channel (V side)
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const int pgk = i >> 4, slot = i & 15;
        const float pscale = __uint_as_float((uint32_t)(127 - vpos<BITS>(slot >> 1)) << 23);  // 2^-P of token i in A2
        const float kscale = a.scale_log2 * 16777216.0f;
        float mref[GP], lpart[GP], zpart[C::NG][GP];
#pragma unroll
        for (int h = 0; h < GP; ++h) {
            mref[h] = -INFINITY;
            lpart[h] = 0.0f;
#pragma unroll
            for (int g = 0; g < C::NG; ++g) zpart[g][h] = 0.0f;
        }
        bool dead = false;
        // every wait of these warps is warp-uniform; `dead` (a wait ran out)
        // skips all further tensor-memory work but keeps the loop and its
        // named barriers in step with the other compute warps
        auto wait_all = [&](uint64_t *bar, uint32_t parity) {
            if (!dead) dead = !__all_sync(0xffffffffu, mbar_wait(bar, parity, a.status, kWait));
        };
        auto stage_of = [&](int j) { return ring + (j % C::NST) * C::STAGE; };
        // A1 <- tile j's K codes of token i (a1_done signals the stored row)
        auto put_a1 = [&](int j) {
            wait_all(&full[j % C::NST], (j / C::NST) & 1);
            if (dead) return;
            uint32_t r[C::A1C];
            unpack_k<BITS, D>(stage_of(j) + pgk * C::HB + slot * C::ROWB, r);
            if constexpr (C::A1C == 64) tmem_st_x64(tmem + lane_base + C::A1_COL, r);
            else tmem_st_x32(tmem + lane_base + C::A1_COL, r);
        };
        auto a1_done = [&]() {
            if (dead) return;
            tmem_st_wait();
            vtc::tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(a1r);
        };
        // A2 buffer j & 1 <- tile j's V codes of channel i (after the P V of
        // tile j - 2, which read that buffer)
        auto put_a2 = [&](int j) {
            if (j >= 2) wait_all(&pvd[j & 1], ((j - 2) >> 1) & 1);
            if (dead) return;
            vtc::tc_fence_after();
            if (i < D) {
                uint32_t r[64];
                const uint8_t *vb = stage_of(j) + C::TP * C::HB;
#pragma unroll
                for (int p = 0; p < C::TP; ++p) unpack_v<BITS, D>(vb + p * C::HB, i, r + 8 * p);
                tmem_st_x64(tmem + lane_base + C::A2_COL + (j & 1) * 64, r);
                tmem_st_wait();
            }
            vtc::tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&a2r[j & 1]);
        };
        if (D < 128 && warp >= D / 32) {
            // channels past head_dim: their A2 lanes stay zero for the whole CTA
            uint32_t z[64];
#pragma unroll
            for (int x = 0; x < 64; ++x) z[x] = 0u;
            tmem_st_x64(tmem + lane_base + C::A2_COL, z);
            tmem_st_x64(tmem + lane_base + C::A2_COL + 64, z);
            tmem_st_wait();
        }
        if (ntile > 0) {
            put_a1(0);
            a1_done();
            put_a2(0);
        }
        for (int j = 0; j < ntile; ++j) {
            const uint8_t *stg = stage_of(j);
            const uint32_t vm = dead ? 0u : smask[j % C::NST];
            // ---- this tile's scores (the score product was issued on A1) ----
            wait_all(sr, j & 1);
            uint32_t d1r[C::N];
            if (!dead) {
                vtc::tc_fence_after();
                if constexpr (C::N == 16)
                    tmem_ld_x16(tmem + lane_base + C::D1_COL, *reinterpret_cast<uint32_t(*)[16]>(d1r));
                else
                    tmem_ld_x32(tmem + lane_base + C::D1_COL, *reinterpret_cast<uint32_t(*)[32]>(d1r));
            }
            // ---- meanwhile the next tile's K codes into A1 (its product is done) ----
            if (j + 1 < ntile) put_a1(j + 1);
            const int pos = (p0 + j * C::TP + pgk) * kPage + slot;
            const bool valid = !dead && ((vm >> pgk) & 1u) && pos < len;
            float s[GP];
            float sv[C::NG], zv[C::NG];
            if (!dead) {
                tmem_ld_wait();
                const uint16_t *kpar = reinterpret_cast<const uint16_t *>(stg + pgk * C::HB + C::CR) + slot * C::NG;
                const uint16_t *vpar =
                    reinterpret_cast<const uint16_t *>(stg + (C::TP + pgk) * C::HB + C::CR) + slot * C::NG;
                float sk[C::NG], zk[C::NG];
#pragma unroll
                for (int g = 0; g < C::NG; ++g) {
                    sk[g] = half_bits_to_f32(kpar[g]);
                    zk[g] = half_bits_to_f32(kpar[kPage * C::NG + g]);
                    sv[g] = half_bits_to_f32(vpar[g]);
                    zv[g] = half_bits_to_f32(vpar[kPage * C::NG + g]);
                }
#pragma unroll
                for (int h = 0; h < GP; ++h) {
                    float acc = 0.0f, zt = 0.0f;
#pragma unroll
                    for (int g = 0; g < C::NG; ++g) {
                        acc = fmaf(sk[g], __uint_as_float(d1r[g * GP + h]), acc);
                        zt = fmaf(zk[g], qz[g * GP + h], zt);
                    }
                    const float x = fmaf(acc, kscale, zt);
                    s[h] = (valid && h < grp) ? x : -INFINITY;
                }
            } else {
#pragma unroll
                for (int h = 0; h < GP; ++h) s[h] = -INFINITY;
#pragma unroll
                for (int g = 0; g < C::NG; ++g) sv[g] = zv[g] = 0.0f;
            }
            if (j + 1 < ntile) a1_done();  // the next score product may start
            // ---- reference maximum: raised only when a score passes it by 2^8 ----
            bool ex = false;
#pragma unroll
            for (int h = 0; h < GP; ++h) ex = ex || (s[h] > mref[h] + 8.0f);
            if (bar_or_128(ex)) {
                float wm[GP];
#pragma unroll
                for (int h = 0; h < GP; ++h) {
                    wm[h] = s[h];
#pragma unroll
                    for (int o = 16; o >= 1; o >>= 1) wm[h] = fmaxf(wm[h], __shfl_xor_sync(0xffffffffu, wm[h], o));
                }
                if (lane == 0)
#pragma unroll
                    for (int h = 0; h < GP; ++h) tmx[warp * GP + h] = wm[h];
                bar_sync_128();
                float alpha[GP];
                bool scale_o = false;
#pragma unroll
                for (int h = 0; h < GP; ++h) {
                    const float tm = fmaxf(fmaxf(tmx[h], tmx[GP + h]), fmaxf(tmx[2 * GP + h], tmx[3 * GP + h]));
                    const float mn = fmaxf(mref[h], tm);
                    alpha[h] = (mref[h] == -INFINITY || mn == mref[h]) ? 1.0f : ex2(mref[h] - mn);
                    scale_o = scale_o || alpha[h] != 1.0f;
                    mref[h] = mn;
                    lpart[h] *= alpha[h];
#pragma unroll
                    for (int g = 0; g < C::NG; ++g) zpart[g][h] *= alpha[h];
                }
                if (scale_o && j > 0) {
                    // O holds the P V of tiles < j: wait for the last of them
                    wait_all(&pvd[(j - 1) & 1], ((j - 1) >> 1) & 1);
                    if (!dead && warp < D / 32) {
                        vtc::tc_fence_after();
                        uint32_t ov[C::N];
                        if constexpr (C::N == 16)
                            tmem_ld_x16(tmem + lane_base + C::O_COL, *reinterpret_cast<uint32_t(*)[16]>(ov));
                        else
                            tmem_ld_x32(tmem + lane_base + C::O_COL, *reinterpret_cast<uint32_t(*)[32]>(ov));
                        tmem_ld_wait();
#pragma unroll
                        for (int n = 0; n < C::N; ++n)
                            ov[n] = __float_as_uint(__uint_as_float(ov[n]) * alpha[n % GP]);
                        if constexpr (C::N == 16)
                            tmem_st_x16(tmem + lane_base + C::O_COL, *reinterpret_cast<uint32_t(*)[16]>(ov));
                        else
                            tmem_st_x32(tmem + lane_base + C::O_COL, *reinterpret_cast<uint32_t(*)[32]>(ov));
                        tmem_st_wait();
                    }
                }
                bar_sync_128();  // tmx is read before anyone writes it again
            }
            // ---- probabilities, partial sums, token i's column of B2 ----
            float p[GP];
#pragma unroll
            for (int h = 0; h < GP; ++h) {
                p[h] = s[h] == -INFINITY ? 0.0f : ex2(s[h] - mref[h]);
                lpart[h] += p[h];
            }
            if (valid) {
#pragma unroll
                for (int g = 0; g < C::NG; ++g)
#pragma unroll
                    for (int h = 0; h < GP; ++h) zpart[g][h] = fmaf(zv[g], p[h], zpart[g][h]);
            }
            // B2 buffer j & 1 was read by the P V of tile j - 2
            if (j >= 2) wait_all(&pvd[j & 1], ((j - 2) >> 1) & 1);
            if (!dead) {
                uint8_t *b2 = sB2 + (j & 1) * C::B2_BYTES;
#pragma unroll
                for (int n = 0; n < C::NC; ++n) {
                    const float f = valid ? p[n % GP] * (sv[n / GP] * pscale) : 0.0f;
                    *reinterpret_cast<__half *>(b2 + kmaj(n, i, C::N)) = __float2half_rn(f);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                vtc::tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&pr[j & 1]);
            }
            // ---- the next tile's V codes (its stage has landed: put_a1 waited) ----
            if (j + 1 < ntile) put_a2(j + 1);
            if (!dead) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[j % C::NST]);  // every read of tile j's stage is done
            }
        }
        // ---- the chunk's partial result ----
        if (ntile > 0) wait_all(&pvd[(ntile - 1) & 1], ((ntile - 1) >> 1) & 1);
        float oc[GP];
#pragma unroll
        for (int h = 0; h < GP; ++h) oc[h] = 0.0f;
        if (!dead && ntile > 0 && warp < D / 32) {
            vtc::tc_fence_after();
            uint32_t ov[GP];
            // warp w holds channels 32 w .. 32 w + 31 = group w
            if constexpr (GP == 4) tmem_ld_x4(tmem + lane_base + C::O_COL + warp * GP, ov);
            else tmem_ld_x8(tmem + lane_base + C::O_COL + warp * GP, ov);
            tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < GP; ++h) oc[h] = __uint_as_float(ov[h]);
        }
        if (dead && lane == 0) *dead_any = 1;
        // fixed-order reduction of the zero-point and denominator partials
        float v[C::NRED];
#pragma unroll
        for (int g = 0; g < C::NG; ++g)
#pragma unroll
            for (int h = 0; h < GP; ++h) v[g * GP + h] = zpart[g][h];
#pragma unroll
        for (int h = 0; h < GP; ++h) v[C::NC + h] = lpart[h];
#pragma unroll
        for (int x = 0; x < C::NRED; ++x)
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) v[x] += __shfl_xor_sync(0xffffffffu, v[x], o);
        if (lane == 0)
#pragma unroll
            for (int x = 0; x < C::NRED; ++x) red[warp * C::NRED + x] = v[x];
        bar_sync_128();
        const bool bad = *dead_any != 0;
        if (i < D) {
            const int g = i >> 5;
#pragma unroll
            for (int h = 0; h < GP; ++h) {
                if (h >= grp) break;
                const int x = g * GP + h;
                const float z = ((red[x] + red[C::NRED + x]) + red[2 * C::NRED + x]) + red[3 * C::NRED + x];
                const int64_t row = ((int64_t)b * a.hq + kvh * grp + h) * a.n_splits + split;
                a.ws_o[row * D + i] = bad ? 0.0f : fmaf(oc[h], 16777216.0f, z);
            }
        }
        if (i < grp) {
            const int x = C::NC + i;
            const float l = ((red[x] + red[C::NRED + x]) + red[2 * C::NRED + x]) + red[3 * C::NRED + x];
            const int64_t row = ((int64_t)b * a.hq + kvh * grp + i) * a.n_splits + split;
            float m = -INFINITY;
#pragma unroll
            for (int h = 0; h < GP; ++h)
                if (h == i) m = mref[h];
            a.ws_ml[row * 2] = bad ? -INFINITY : m;
            a.ws_ml[row * 2 + 1] = bad ? 0.0f : l;
        }
    }
    vtc::tc_fence_before();
    __syncthreads();
    vtc::tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS));
}

}  // namespace dtc
}  // namespace vc
