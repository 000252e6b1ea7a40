// Verification attention on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// "VeriCache: Making Lossy KV Compression Exact", "The Core Idea" items 3-5:
// one pass over KV_full checks every drafted position; query i of the block
// attends causally to the prefix and the block up to itself.  The rows of a
// CTA are (query, head) pairs of one kv head's GQA group (one 128-row MMA
// tile, or two for more than 128 rows), so every K/V byte feeds n_q * G rows.
//
// Roles (one CTA = one (request, kv head, 3648-key split, row block)):
//  - producer warp: one thread streams 64-key blocks (4 pages) of K and V
//    into a shared-memory ring (3 stages for one tile, 4 for two) with TMA
//    tensor copies (one 16-row x 64-channel box per page and 128-byte column
//    chunk); the TMA unit writes the 128-byte-swizzled layout the tensor core
//    reads.  Full / empty mbarriers per stage (transaction bytes / MMA
//    completion).  The split's page ids are read into shared memory at
//    set-up, and the producer starts while the other warps stage Q.
//  - MMA warp: one thread issues every tcgen05.mma:  S = Q K^T (M 128, N 64,
//    K 16 steps) into TMEM, then O += P V (M 128, N = D) with P read from
//    TMEM as the A operand and V from shared memory (MN-major).  A one-tile
//    CTA keeps Q in TMEM too (its S MMAs read only the K block from shared
//    memory); a two-tile CTA keeps it in shared memory.
//  - 4 softmax warps per 128-row tile: each thread owns one row = one TMEM
//    lane; it loads the row's 64 scores from TMEM, masks (only blocks that
//    reach the query block), keeps a running max (rescaling O in TMEM only
//    when the max grows by more than 2^8), writes P (bf16 pairs) over the
//    first half of the S buffer it came from, and finally reads O.
//  A one-tile CTA uses 96 KB of shared memory and 256 TMEM columns with one
//  S buffer, so two CTAs share an SM and overlap each other's S / softmax /
//  P V chain; a two-tile CTA holds two S buffers per tile and runs alone.
// Every configuration uses the same 64-key blocks and each row's arithmetic
// depends on that row alone, with splits fixed by key position, so results
// do not depend on n_q, the row block or the batch.
// Every mbarrier wait is bounded; a timeout is reported and the CTA drains.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; maps are encoded by the host code)

#include "vc_internal.cuh"

namespace vc {
namespace vtc {

constexpr int kBlockKeys = 32;   // keys per MMA block (2 pages)
// Keys per split: fixed by position (a row's bits must not depend on n_q, the
// batch or the context), a multiple of the 64-key block.  3648 = 57 blocks
// rather than 4096: it cuts the usual contexts into pieces that fill whole
// waves of CTAs more evenly (measured: 32800 keys 213 -> 202 us, 41000 keys
// 407 -> 372 us, 131112 keys 999 -> 988 us on the bench shapes).
constexpr int kSplitPages = 228;
constexpr int kTileRows = 128;

struct Args {
    CUtensorMap kmap, vmap;  // K / V pools as [pages * hkv * 16 rows][D] bf16, box 16 x 64, 128B swizzle
    const uint16_t *q;  // [B][n_q][Hq][D]
    const uint8_t *kp, *vp;
    int64_t n_pages;
    const int32_t *table, *lens;
    int maxb;
    int n_q, hq, hkv, grp;
    float scale_log2;
    int n_splits;
    int rows_per_cta;   // QT * 128
    int rb0 = 0;        // row block of the first CTA row (a launch may cover the last row blocks only)
    float *ws_o;        // [B][n_q][Hq][n_splits][D]
    float *ws_ml;       // [..][2]
    int32_t *status;
    uint64_t wait_ns = kWaitNs;  // bounded-wait limit
    int skip_copies = 0;         // fault injection: the producer issues no copy
};

template <int D, int QT>
struct Cfg {
    static constexpr int NC = D / 64;                      // swizzle atoms along D
    static_assert(QT == 1 || QT == 2, "one or two 128-row tiles per CTA");
    // keys per block: the softmax round trip between the MMA warp and the
    // softmax warps (barrier wake-ups, TMEM load and store latencies) is paid
    // once per 64 keys
    static constexpr int BK = 64;
    // S buffers per tile in TMEM (P is written over its S buffer): two let a
    // tile's next S overlap its softmax; one-tile CTAs (two per SM, 256
    // columns each) take one so that Q fits in TMEM and the shared memory
    // holds three K/V stages -- the two CTAs of an SM overlap instead
    static constexpr int SB = QT == 2 ? 2 : 1;
    // Q as the TMEM A operand of S = Q K^T when it fits next to the S and O
    // columns (then the S MMAs read only the K block from shared memory);
    // otherwise Q stays in shared memory
    static constexpr int TMEM_LIMIT = QT == 1 ? 256 : 512;  // one-tile CTAs run two per SM
    static constexpr bool QTM = QT * SB * BK + QT * D + QT * D / 2 <= TMEM_LIMIT;
    static constexpr int QTILE = kTileRows * D * 2;        // one Q tile
    static constexpr int KTILE = BK * D * 2;               // one K (or V) block
    static constexpr int OFF_KV = QTM ? 0 : QT * QTILE;
    // K/V ring depth within the shared memory of the CTAs an SM holds
    static constexpr int STAGE_BYTES = 2 * KTILE;
    static constexpr int STAGES_FIT = ((QT == 1 ? 110 : 220) * 1024 - OFF_KV) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT < 8 ? STAGES_FIT : 8;
    static_assert(STAGES >= 2, "K/V ring needs two stages");
    static constexpr int OFF_BAR = OFF_KV + STAGES * 2 * KTILE;
    static constexpr int NBAR = QT * 6 + 2 * STAGES;  // s_ready, p_ready, pv_done ([QT][2] each), full, empty
    // page ids of the split (read once at set-up, so that the producer
    // issues a block's copies without waiting on table loads)
    static constexpr int OFF_PID = OFF_BAR + NBAR * 8 + 16;
    static constexpr int SMEM = OFF_PID + kSplitPages * 4 + 1024;
    static constexpr int TMEM_USED = QT * SB * BK + QT * D + (QTM ? QT * D / 2 : 0);
    static constexpr int TMEM_COLS = TMEM_USED <= 256 ? 256 : 512;
    static_assert(TMEM_USED <= TMEM_LIMIT, "S, O (and Q) columns exceed TMEM");
    // MMA-issuing warps: one per tile with two S buffers, so each tile's S /
    // P V chain is issued independently (one thread issuing both tiles'
    // MMAs in a fixed order stalls on the other tile's waits); one with a
    // single S buffer
    static constexpr int NMMA = SB == 2 ? QT : 1;
    static constexpr int THREADS = QT * 128 + 32 + 32 * NMMA;  // softmax warps + producer + MMA warps
    static constexpr int MIN_CTAS = QT == 1 ? 2 : 1;  // resident CTAs per SM (TMEM: 256 columns each)
    __host__ __device__ static constexpr uint32_t S_COL(int qt, int buf) { return (uint32_t)(qt * SB + buf) * BK; }
    __host__ __device__ static constexpr uint32_t O_COL(int qt) { return (uint32_t)(QT * SB * BK + qt * D); }
    // Q tile qt as bf16 pairs (D / 2 columns), when QTM
    __host__ __device__ static constexpr uint32_t Q_COL(int qt) {
        return (uint32_t)(QT * SB * BK + QT * D + qt * (D / 2));
    }
};

// --- tcgen05 / descriptor helpers ------------------------------------------
// Shared-memory matrix descriptor, 128-byte swizzle (layout type 2), version 1.
__device__ inline uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B, A K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}
__device__ inline void umma(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
// The same with the A operand (M lanes x 16 K elements, bf16 pairs per
// 32-bit column) read from TMEM.
__device__ inline void umma_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
        "r"(tmem_a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ inline void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
// One TMA tensor copy: box at (x = channel, y = row) of `map` -> dst.
__device__ inline void tma2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ inline void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ inline void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ inline void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ inline void tmem_st16(uint32_t taddr, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])));
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// N (32 or 64) consecutive columns of this thread's lane: one load, one wait
template <int N>
__device__ inline void tmem_ld_row(uint32_t taddr, float (&v)[N]) {
    static_assert(N == 32 || N == 64, "x32 or x64 loads");
    uint32_t r[N];
    if constexpr (N == 32) {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
            "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
            "tcgen05.wait::ld.sync.aligned;"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
              "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
              "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
            : "r"(taddr)
            : "memory");
    } else {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x64.b32 {"
            "%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
            "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
            "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
            "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63"
            "}, [%64];\n\t"
            "tcgen05.wait::ld.sync.aligned;"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
              "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
              "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
              "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
              "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
              "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
              "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
            : "r"(taddr)
            : "memory");
    }
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = __uint_as_float(r[i]);
}

// max of N values as a tree (log2 N dependent steps); exact, so the order
// does not change the result
template <int N>
__device__ inline float max_tree(const float (&v)[N]) {
    float m[N / 2];
#pragma unroll
    for (int i = 0; i < N / 2; ++i) m[i] = fmaxf(v[i], v[i + N / 2]);
#pragma unroll
    for (int w = N / 4; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) m[i] = fmaxf(m[i], m[i + w]);
    return m[0];
}

// 16 columns of this thread's lane, without waiting (tcgen05.wait::st follows)
__device__ inline void tmem_st16_nowait(uint32_t taddr, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}

// offset of (row, 16-byte chunk c) in a 128-byte-swizzled K-major tile whose
// rows are `rows` long per 64-element atom column
__device__ inline int sw128(int row, int c, int rows) {
    return (c >> 3) * rows * 128 + row * 128 + (((c & 7) ^ (row & 7)) << 4);
}

// --- the CTA body ------------------------------------------------------------
// FULL: every tile of this row block holds rows (the tile count is then a
// compile-time constant and the tile loops fold away); otherwise the last
// row block skips its empty tiles.
template <int D, int QT, bool FULL>
__device__ __forceinline__ void verify_tc_block(const Args &a, int split, int rb, int bk, uint8_t *smem_raw) {
    using C = Cfg<D, QT>;
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // 1024-byte aligned
    uint8_t *sq = smem;
    uint8_t *skv = smem + C::OFF_KV;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *s_ready = bars;             // [QT][2]
    uint64_t *p_ready = bars + QT * 2;    // [QT][2]
    uint64_t *pv_done = bars + QT * 4;    // [QT][2]
    uint64_t *full = bars + QT * 6;       // [STAGES]
    uint64_t *empty = full + C::STAGES;   // [STAGES]
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + C::NBAR);
    int32_t *spid = reinterpret_cast<int32_t *>(smem + C::OFF_PID);  // [nb * BK / 16] page ids

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool producer = warp == QT * 4;
    const bool mma_warp = warp > QT * 4 && warp <= QT * 4 + C::NMMA;
    const int mtile = warp - QT * 4 - 1;  // the tile an MMA warp issues for (two S buffers)
    const int b = bk / a.hkv, kvh = bk % a.hkv;
    const int len = a.lens[b];
    const bool len_ok = len >= a.n_q;
    if (!len_ok && tid == 0 && split == 0 && rb == 0 && kvh == 0) report(a.status, VC_ERR_BAD_INDEX);
    const int npages = len_ok ? ceil_div(len, kPage) : 0;
    const int p0 = split * kSplitPages;
    const int p1 = min(p0 + kSplitPages, npages);
    const int nkeys = max(0, min(p1 * kPage, len) - p0 * kPage);
    const int nb = ceil_div(nkeys, C::BK);
    const int nrows = a.n_q * a.grp;
    // tiles of this row block holding at least one row (the last row block
    // may fill fewer than QT): the others issue no MMA and run no softmax
    const int nt = FULL ? QT : min(QT, ceil_div(max(0, min(a.rows_per_cta, nrows - rb * a.rows_per_cta)), kTileRows));
    const int32_t *trow = a.table + (int64_t)b * a.maxb;

    // ---- set-up: barriers, TMEM, page ids, Q tiles ----
    // Page ids of the split's blocks, checked once (pages past the request's
    // end within its last block: any valid page, masked / zeroed later).
    // One dependent table load per page inside the producer loop would cap
    // the copy issue rate at a block per few table-load latencies.
    for (int i = tid; i < nb * (C::BK / kPage) && tid < C::THREADS; i += C::THREADS) {
        const int pidx = p0 + i;
        int id = 0;
        if (pidx < npages) {
            id = pidx < a.maxb ? trow[pidx] : -1;
            if (id < 0 || id >= a.n_pages) {
                report(a.status, VC_ERR_BAD_INDEX);
                id = 0;
            }
        }
        spid[i] = id;
    }
    if (tid == 0) {
        for (int i = 0; i < QT * 2; ++i) {
            mbar_init(&s_ready[i], 1);
            mbar_init(&p_ready[i], kTileRows);
        }
        for (int i = 0; i < QT * 2; ++i) mbar_init(&pv_done[i], 1);
        for (int i = 0; i < C::STAGES; ++i) {
            mbar_init(&full[i], 1);
            // a stage is free once every issuing thread's P V of it is done
            mbar_init(&empty[i], C::SB == 2 ? nt : 1);
        }
        fence_mbar_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                     "r"(C::TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    // The producer starts its copies now; the other warps stage the Q tiles
    // meanwhile (every load issued before any store) and meet at their own
    // barrier, so the first blocks' copy latency overlaps the Q loads.
    // (a launch with more threads than the roles need -- the mixed grid --
    // leaves the extra warps out of the staging and its barrier)
    if (!producer && warp < C::THREADS / 32) {
        if constexpr (!C::QTM) {
            constexpr int QE = QT * kTileRows * (D / 8);  // 16-byte chunks of the CTA's Q tiles
            constexpr int NQ = C::THREADS - 32;           // every thread but the producer warp's
            constexpr int QPT = (QE + NQ - 1) / NQ;
            const int qi = tid < QT * 128 ? tid : tid - 32;
            uint4 v[QPT];
#pragma unroll
            for (int u = 0; u < QPT; ++u) {
                const int e = qi + u * NQ;
                const int r = e / (D / 8), c = e % (D / 8);  // r: row within the CTA, c: 16-byte chunk
                const int rg = rb * a.rows_per_cta + r;
                v[u] = make_uint4(0, 0, 0, 0);
                if (e < QE && rg < nrows) {
                    const int i = rg / a.grp, n = rg % a.grp;
                    v[u] = *reinterpret_cast<const uint4 *>(
                        a.q + (((int64_t)b * a.n_q + i) * a.hq + kvh * a.grp + n) * D + c * 8);
                }
            }
#pragma unroll
            for (int u = 0; u < QPT; ++u) {
                const int e = qi + u * NQ;
                const int r = e / (D / 8), c = e % (D / 8);
                if (e < QE) *reinterpret_cast<uint4 *>(sq + (r >> 7) * C::QTILE + sw128(r & 127, c, kTileRows)) = v[u];
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        } else if (warp < QT * 4) {
            // each softmax thread writes its own row (= TMEM lane) of its
            // tile's Q as bf16 pairs (element 2c in the low half of column c)
            const int qt = warp >> 2;
            const int r = (warp & 3) * 32 + lane;
            const int rg = rb * a.rows_per_cta + qt * kTileRows + r;
            uint4 u[D / 8];
#pragma unroll
            for (int j = 0; j < D / 8; ++j) u[j] = make_uint4(0, 0, 0, 0);
            if (rg < nrows) {
                const int i = rg / a.grp, n = rg % a.grp;
                const uint4 *src =
                    reinterpret_cast<const uint4 *>(a.q + (((int64_t)b * a.n_q + i) * a.hq + kvh * a.grp + n) * D);
#pragma unroll
                for (int j = 0; j < D / 8; ++j) u[j] = src[j];
            }
            const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
#pragma unroll
            for (int c0 = 0; c0 < D / 2; c0 += 16) {
                float v[16];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    v[4 * j] = __uint_as_float(u[c0 / 4 + j].x);
                    v[4 * j + 1] = __uint_as_float(u[c0 / 4 + j].y);
                    v[4 * j + 2] = __uint_as_float(u[c0 / 4 + j].z);
                    v[4 * j + 3] = __uint_as_float(u[c0 / 4 + j].w);
                }
                tmem_st16(tmem + lane_base + C::Q_COL(qt) + c0, v);
            }
        }
        tc_fence_before();
        asm volatile("bar.sync 1, %0;" ::"r"(C::THREADS - 32) : "memory");
        tc_fence_after();
    }
    bool alive = true;

    constexpr uint32_t IQK = idesc_bf16(128, C::BK, false);
    constexpr uint32_t IPV = idesc_bf16(128, D, true);
    if (producer) {
        // ================= producer: TMA tensor copies into the stage ring =================
        if (lane == 0 && !a.skip_copies) {
            for (int j = 0; j < nb && alive; ++j) {
                const int st = j % C::STAGES;
                if (j >= C::STAGES) alive = mbar_wait(&empty[st], ((j / C::STAGES) - 1) & 1, a.status, a.wait_ns);
                if (!alive) break;
                uint8_t *kt = skv + st * 2 * C::KTILE;
                mbar_arrive_expect_tx(&full[st], 2 * C::KTILE);
#pragma unroll
                for (int pg = 0; pg < C::BK / kPage; ++pg) {
                    const int y = (spid[j * (C::BK / kPage) + pg] * a.hkv + kvh) * kPage;
#pragma unroll
                    for (int c = 0; c < C::NC; ++c) {
                        tma2d(kt + c * (C::BK * 128) + pg * (kPage * 128), &a.kmap, c * 64, y, &full[st]);
                        tma2d(kt + C::KTILE + c * (C::BK * 128) + pg * (kPage * 128), &a.vmap, c * 64, y,
                              &full[st]);
                    }
                }
            }
        }
    } else if (mma_warp) {
        // ================= MMA issue (one thread per MMA warp) =================
        if (lane == 0 && (C::SB != 2 || mtile < nt)) {
            auto issue_s = [&](int j, int qt, const uint8_t *kt) {
                if constexpr (C::QTM) {
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
                        umma_ta(tmem + C::S_COL(qt, j % C::SB), tmem + C::Q_COL(qt) + ks * 8,
                                sdesc(smem_u32(kt) + (ks >> 2) * (C::BK * 128) + (ks & 3) * 32, 16, 1024), IQK,
                                ks > 0);
                } else {
                    const uint8_t *qtile = sq + qt * C::QTILE;
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
                        umma(tmem + C::S_COL(qt, j % C::SB),
                             sdesc(smem_u32(qtile) + (ks >> 2) * (kTileRows * 128) + (ks & 3) * 32, 16, 1024),
                             sdesc(smem_u32(kt) + (ks >> 2) * (C::BK * 128) + (ks & 3) * 32, 16, 1024), IQK,
                             ks > 0);
                }
                umma_commit(&s_ready[qt * 2 + j % C::SB]);
            };
            auto issue_pv_tile = [&](int j, int qt) {
                const uint8_t *vt = skv + (j % C::STAGES) * 2 * C::KTILE + C::KTILE;
                // P of block j: bf16 pairs in the first half of its S buffer
#pragma unroll
                for (int kk = 0; kk < C::BK / 16; ++kk)
                    umma_ta(tmem + C::O_COL(qt), tmem + C::S_COL(qt, j % C::SB) + kk * 8,
                            sdesc(smem_u32(vt) + kk * 16 * 128, C::BK * 128, 1024), IPV, (j > 0 || kk > 0));
            };
            auto finish_pv = [&](int j, int qt) {  // the P V of tile qt (SB == 2) or of every tile
                if constexpr (C::SB == 2) {
                    umma_commit(&pv_done[qt * 2 + (j & 1)]);
                } else {
#pragma unroll
                    for (int t = 0; t < QT; ++t)
                        if (t < nt) umma_commit(&pv_done[t * 2 + (j & 1)]);
                }
                umma_commit(&empty[j % C::STAGES]);
            };
            auto wait_p = [&](int j, int qt) {
                alive = alive && mbar_wait(&p_ready[qt * 2 + j % C::SB], (j / C::SB) & 1, a.status, a.wait_ns);
                tc_fence_after();
            };
            for (int j = 0; j < nb && alive; ++j) {
                const int st = j % C::STAGES;
                alive = mbar_wait(&full[st], (j / C::STAGES) & 1, a.status, a.wait_ns);
                if (!alive) break;
                tc_fence_after();
                const uint8_t *kt = skv + st * 2 * C::KTILE;
                if constexpr (C::SB == 2) {
                    // this warp's tile: S of block j, then P V of block j - 1
                    issue_s(j, mtile, kt);
                    if (j >= 1) {
                        wait_p(j - 1, mtile);
                        if (!alive) break;
                        issue_pv_tile(j - 1, mtile);
                        finish_pv(j - 1, mtile);
                    }
                } else {
                    // one S buffer per tile: a tile's P V of block j - 1 reads
                    // the buffer its S of block j then overwrites (in order)
#pragma unroll
                    for (int qt = 0; qt < QT; ++qt) {
                        if (qt >= nt || !alive) continue;
                        if (j >= 1) {
                            wait_p(j - 1, qt);
                            if (!alive) break;
                            issue_pv_tile(j - 1, qt);
                        }
                        issue_s(j, qt, kt);
                    }
                    if (j >= 1 && alive) finish_pv(j - 1, 0);
                }
            }
            if (nb > 0 && alive) {
                if constexpr (C::SB == 2) {
                    wait_p(nb - 1, mtile);
                    if (alive) {
                        issue_pv_tile(nb - 1, mtile);
                        finish_pv(nb - 1, mtile);
                    }
                } else {
#pragma unroll
                    for (int qt = 0; qt < QT; ++qt)
                        if (qt < nt) wait_p(nb - 1, qt);
                    if (alive) {
#pragma unroll
                        for (int qt = 0; qt < QT; ++qt)
                            if (qt < nt) issue_pv_tile(nb - 1, qt);
                        finish_pv(nb - 1, 0);
                    }
                }
            }
        }
    } else if ((warp >> 2) >= nt) {
        // a tile without rows in this row block: nothing to do
    } else {
        // ================= softmax / epilogue: one thread per row =================
        const int qt = warp >> 2;
        const int r = (warp & 3) * 32 + lane;                 // row within the tile = TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const int rg = rb * a.rows_per_cta + qt * kTileRows + r;
        const bool rvalid = rg < nrows;
        const int qpos = len - a.n_q + (rvalid ? rg / a.grp : 0);
        float m_used = -INFINITY, l = 0.0f;
        bool o_touched = false;
        // tcgen05.ld / st are warp-collective: every lane of a softmax warp runs
        // them together (row validity and rescale decisions only pick values)
        for (int j = 0; j < nb && alive; ++j) {
            alive = __all_sync(0xffffffffu, mbar_wait(&s_ready[qt * 2 + j % C::SB], (j / C::SB) & 1, a.status, a.wait_ns));
            if (!alive) break;
            tc_fence_after();
            float s[C::BK];
            tmem_ld_row<C::BK>(tmem + lane_base + C::S_COL(qt, j % C::SB), s);
            const int key0 = p0 * kPage + j * C::BK;
            // raw-score max; masking only where the block reaches the query
            // block or the request's end (the same arithmetic either way, so a
            // row's bits do not depend on n_q)
            if (key0 + C::BK > len - a.n_q) {
#pragma unroll
                for (int c = 0; c < C::BK; ++c) {
                    const int key = key0 + c;
                    if (!(rvalid && key <= qpos && key < len)) s[c] = -INFINITY;
                }
            }
            const float mraw = max_tree<C::BK>(s);
            const float mb = mraw * a.scale_log2;
            // grow the reference max only when it rises by more than 2^8
            // (rare after the first block); O is rescaled in TMEM
            const bool grow = mb > m_used + 8.0f;
            const float f = grow ? (m_used == -INFINITY ? 0.0f : ex2(m_used - mb)) : 1.0f;
            if (__any_sync(0xffffffffu, grow) && o_touched) {
                // the previous block's P V must have landed before O is rescaled
                alive = __all_sync(0xffffffffu,
                                   mbar_wait(&pv_done[qt * 2 + ((j - 1) & 1)], ((j - 1) >> 1) & 1, a.status, a.wait_ns));
                if (!alive) break;
                tc_fence_after();
                for (int c0 = 0; c0 < D; c0 += 16) {
                    float v[16];
                    tmem_ld16(tmem + lane_base + C::O_COL(qt) + c0, v);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] *= f;
                    tmem_st16(tmem + lane_base + C::O_COL(qt) + c0, v);
                }
            }
            if (grow) {
                l *= f;
                m_used = mb;
            }
            const float nms = m_used == -INFINITY ? 0.0f : -m_used;
            // slots past the request's end (or of pages past it) may hold any
            // bytes: zero their V rows so that 0 * NaN never reaches P V.
            // Every tile does it before it signals its P: a tile's P V is
            // issued independently of the other tile's (zeros written twice
            // are still zeros)
            const int nvalid = len - key0;
            if (nvalid < C::BK) {
                uint8_t *vt = skv + (j % C::STAGES) * 2 * C::KTILE + C::KTILE;
                for (int e = r; e < (C::BK - nvalid) * (D / 8); e += kTileRows) {
                    const int kr = nvalid + e / (D / 8), c = e % (D / 8);
                    *reinterpret_cast<uint4 *>(vt + sw128(kr, c, C::BK)) = make_uint4(0, 0, 0, 0);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            // P (bf16 pairs) over the first half of this block's S buffer;
            // the buffer's previous P was read by block j - SB's P V, which the
            // MMA pipe finished before it wrote this block's S.  The block's P
            // sum in four interleaved partial sums (a fixed order, short
            // dependent chains).
            {
                float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int h = 0; h < C::BK / 32; ++h) {
                    float pk[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const float p0v = ex2(fmaf(s[h * 32 + 2 * c], a.scale_log2, nms));
                        const float p1v = ex2(fmaf(s[h * 32 + 2 * c + 1], a.scale_log2, nms));
                        ls[(2 * c) & 3] += p0v;
                        ls[(2 * c + 1) & 3] += p1v;
                        pk[c] = __uint_as_float(pack_bf16(p0v, p1v));
                    }
                    tmem_st16_nowait(tmem + lane_base + C::S_COL(qt, j % C::SB) + h * 16, pk);
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            }
            tc_fence_before();
            mbar_arrive(&p_ready[qt * 2 + j % C::SB]);
            o_touched = true;
        }
        pdl_trigger();  // the main loop is done: the next kernel may be scheduled
        // epilogue: the whole warp waits for the last P V and reads O
        float *dst = nullptr;
        int64_t row = 0;
        if (rvalid) {
            const int i = rg / a.grp, n = rg % a.grp;
            row = (((int64_t)b * a.n_q + i) * a.hq + kvh * a.grp + n) * a.n_splits + split;
            dst = a.ws_o + row * D;
        }
        bool have_o = nb > 0 && alive;
        if (have_o) {
            have_o = __all_sync(0xffffffffu,
                                mbar_wait(&pv_done[qt * 2 + ((nb - 1) & 1)], ((nb - 1) >> 1) & 1, a.status, a.wait_ns));
            alive = have_o;
        }
        if (have_o) {
            tc_fence_after();
            for (int c0 = 0; c0 < D; c0 += 16) {
                float v[16];
                tmem_ld16(tmem + lane_base + C::O_COL(qt) + c0, v);
                if (rvalid) {
#pragma unroll
                    for (int i2 = 0; i2 < 16; i2 += 4)
                        *reinterpret_cast<float4 *>(dst + c0 + i2) =
                            make_float4(v[i2], v[i2 + 1], v[i2 + 2], v[i2 + 3]);
                }
            }
        } else if (rvalid) {
            for (int c0 = 0; c0 < D; ++c0) dst[c0] = 0.0f;
            m_used = -INFINITY;
            l = 0.0f;
        }
        if (rvalid) {
            a.ws_ml[row * 2] = m_used;
            a.ws_ml[row * 2 + 1] = l;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS));
}

// The CTA body, with the tile count folded for full row blocks.
template <int D, int QT>
__device__ __forceinline__ void verify_tc_cta(const Args &a, int split, int rb, int bk, uint8_t *smem_raw) {
    const int rows_here = a.n_q * a.grp - rb * a.rows_per_cta;
    if (QT == 1 || rows_here > (QT - 1) * kTileRows)  // every tile holds rows
        verify_tc_block<D, QT, true>(a, split, rb, bk, smem_raw);
    else
        verify_tc_block<D, QT, false>(a, split, rb, bk, smem_raw);
}

// Combine the splits of one row in split order (fixed, so a row's result does
// not depend on how many empty splits follow it).
template <int D>
__device__ __forceinline__ void reduce_row(const float *ws_o, const float *ws_ml, int n_splits, int64_t row,
                                           float *out, int tid, int nthreads) {
    combine_partials<D>(ws_o, ws_ml, n_splits, n_splits, row, out, tid, nthreads);
}

}  // namespace vtc
}  // namespace vc
