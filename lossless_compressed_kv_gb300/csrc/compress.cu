// vc_compress: KV_full (bf16 pages) -> KV_comp entries.
//
// "VeriCache Guide", section "The Uniform Compressor Interface" (token
// eviction and low-bit quantisation behind one compress()) and the guide's
// compressor (K and V gathered with one sorted index list shared by all
// heads).  The bit format (asymmetric 32-channel groups, fp16 scale and
// zero, little-endian packing) is the library's reading; see vc.h.
//
// Quantised formats: one CTA per (KV_comp page, kv head) touched by a
// request's slot range.  It loads the page's K and V head blocks into shared
// memory, quantises the covered token slots (one warp per slot: 32 lanes own
// D/32 consecutive channels each, so a group's min/max is a shuffle over the
// lanes of that group), places the codes with comp_layout.cuh's map and
// writes both blocks back whole.  Slots outside the range keep their bytes.
// bf16 token drop: one warp per (kept entry, kv head) copies the row.
#include "comp_layout.cuh"
#include "quant_row.cuh"
#include "vc_internal.cuh"

namespace vc {
namespace {

constexpr int kWarps = 8;

struct CompressArgs {
    const uint8_t *fk, *fv;  // full pools
    int64_t f_pages;
    const int32_t *f_table, *f_lens;
    int f_maxb;
    uint8_t *ck, *cv;  // comp pools
    int64_t c_pages;
    const int32_t *c_table;
    int c_maxb;
    const int32_t *offs, *idx, *start;
    int hkv;
    int32_t *status;
};

// Replace the `width` bits at bit offset `off` of a shared-memory block.
__device__ inline void put_bits(uint32_t *blk, int off, int width, uint32_t v) {
    const uint32_t m = ((1u << width) - 1u) << (off & 31);
    atomicAnd(&blk[off >> 5], ~m);
    atomicOr(&blk[off >> 5], (v << (off & 31)) & m);
}

constexpr int kPageWarps = 8;
// Up to this many entries per request the token-parallel path is used.
constexpr int kTokenPathMax = 32;

template <int BITS, int D>
__global__ void __launch_bounds__(kPageWarps * 32) compress_page_kernel(CompressArgs a) {
    pdl_begin();
    constexpr int HB = 2 * D * (BITS + 1);    // head block bytes
    constexpr int CR = kPage * D * BITS / 8;  // code region bytes
    constexpr int G = D / kGroup, CPL = D / 32, LPG = kGroup / CPL;
    __shared__ __align__(16) uint32_t blk[2][HB / 4];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z, h = blockIdx.y;
    const int o0 = a.offs[b], n = a.offs[b + 1] - o0;
    if (n <= 0) return;
    const int start = a.start ? a.start[b] : 0;
    if (start < 0) {
        if (threadIdx.x == 0 && blockIdx.x == 0) report(a.status, VC_ERR_BAD_INDEX);
        return;
    }
    const int pg = start / kPage + blockIdx.x;
    const int s_lo = max(start, pg * kPage), s_hi = min(start + n, (pg + 1) * kPage);
    if (s_lo >= s_hi) return;
    const int cp = pg < a.c_maxb ? a.c_table[(int64_t)b * a.c_maxb + pg] : -1;
    if (cp < 0 || cp >= a.c_pages) {
        if (threadIdx.x == 0) report(a.status, VC_ERR_BAD_INDEX);
        return;
    }
    uint8_t *gk = a.ck + ((int64_t)cp * a.hkv + h) * HB;
    uint8_t *gv = a.cv + ((int64_t)cp * a.hkv + h) * HB;
    const int fhb = head_block_bytes(16, D);
    // Each warp's first slot: kept index -> page -> bf16 rows, started before
    // the old blocks are copied so the two chains of dependent loads overlap.
    int s = s_lo + warp;
    uint16_t xk[CPL], xv[CPL];
    int fp = -1;
    auto fetch = [&](int slot_pos) {
        const int t = a.idx[o0 + (slot_pos - start)];
        fp = (t >= 0 && t < a.f_lens[b] && t / kPage < a.f_maxb) ? a.f_table[(int64_t)b * a.f_maxb + t / kPage] : -1;
        if (fp >= 0 && fp < a.f_pages) {
            const int64_t fbase = ((int64_t)fp * a.hkv + h) * fhb + (int64_t)(t % kPage) * D * 2;
            qrow::load_lane_row<D>(a.fk + fbase, lane, xk);
            qrow::load_lane_row<D>(a.fv + fbase, lane, xv);
        } else {
            fp = -1;
        }
    };
    if (s < s_hi) fetch(s);
    for (int i = threadIdx.x; i < HB / 16; i += blockDim.x) {
        reinterpret_cast<uint4 *>(blk[0])[i] = reinterpret_cast<const uint4 *>(gk)[i];
        reinterpret_cast<uint4 *>(blk[1])[i] = reinterpret_cast<const uint4 *>(gv)[i];
    }
    __syncthreads();
    for (; s < s_hi; s += kPageWarps) {
        if (s != s_lo + warp) fetch(s);
        if (fp < 0) {  // bad kept index: the slot keeps its bytes
            if (lane == 0) report(a.status, VC_ERR_BAD_INDEX);
            continue;
        }
        const int slot = s % kPage;
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
            uint8_t code[CPL];
            uint16_t sh, zh;
            qrow::quantize_row<BITS, D>(kv ? xv : xk, code, sh, zh);
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                const int ch = lane * CPL + i;
                const int o = kv ? layout::v_bit(BITS, D, slot, ch, 0) : layout::k_bit(BITS, D, slot, ch, 0);
                if constexpr (BITS == 3) {
                    put_bits(blk[kv], o, 2, code[i] & 3u);
                    const int o1 = kv ? layout::v_bit(3, D, slot, ch, 1) : layout::k_bit(3, D, slot, ch, 1);
                    put_bits(blk[kv], o1, 1, code[i] >> 2);
                } else {
                    put_bits(blk[kv], o, BITS, code[i]);
                }
            }
            if (lane % LPG == 0) {
                const int gr = lane / LPG;
                const int e = kv ? layout::v_param(G, slot, gr) : slot * G + gr;
                uint16_t *par = reinterpret_cast<uint16_t *>(reinterpret_cast<uint8_t *>(blk[kv]) + CR);
                par[e] = sh;
                par[kPage * G + e] = zh;
            }
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < HB / 16; i += blockDim.x) {
        reinterpret_cast<uint4 *>(gk)[i] = reinterpret_cast<const uint4 *>(blk[0])[i];
        reinterpret_cast<uint4 *>(gv)[i] = reinterpret_cast<const uint4 *>(blk[1])[i];
    }
}

// Small appends (a few entries per request, e.g. one drafted token per draft
// step): one warp per (kept entry, kv head).  The token's K row and fp16
// parameters belong to it alone and are stored directly; its V codes share
// 32-bit words with the other tokens of the page and are merged with global
// AND / OR reductions (one thread per word, in program order).
template <int BITS, int D>
__global__ void __launch_bounds__(kWarps * 32) compress_token_kernel(CompressArgs a) {
    pdl_begin();
    constexpr int HB = 2 * D * (BITS + 1), RW = D * BITS / 32;  // K row words
    __shared__ uint32_t krow[kWarps][RW];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    const int item = blockIdx.x * kWarps + warp;  // (entry, head) pair
    const int j = item / a.hkv, h = item % a.hkv;
    const int o0 = a.offs[b], o1 = a.offs[b + 1];
    if (o0 + j >= o1) return;
    const int t = a.idx[o0 + j];
    const int slot_pos = (a.start ? a.start[b] : 0) + j;
    if (t < 0 || t >= a.f_lens[b] || t / kPage >= a.f_maxb || slot_pos < 0 || slot_pos / kPage >= a.c_maxb) {
        if (lane == 0) report(a.status, VC_ERR_BAD_INDEX);
        return;
    }
    const int fp = a.f_table[(int64_t)b * a.f_maxb + t / kPage];
    const int cp = a.c_table[(int64_t)b * a.c_maxb + slot_pos / kPage];
    if (fp < 0 || fp >= a.f_pages || cp < 0 || cp >= a.c_pages) {
        if (lane == 0) report(a.status, VC_ERR_BAD_INDEX);
        return;
    }
    const int fhb = head_block_bytes(16, D);
    const int64_t fbase = ((int64_t)fp * a.hkv + h) * fhb + (int64_t)(t % kPage) * D * 2;
    uint8_t *gk = a.ck + ((int64_t)cp * a.hkv + h) * HB;
    uint8_t *gv = a.cv + ((int64_t)cp * a.hkv + h) * HB;
    qrow::append_entry<BITS, D>(a.fk + fbase, a.fv + fbase, gk, gv, slot_pos % kPage, lane, krow[warp]);
}

// bf16 token drop: one warp per (kept entry, kv head) copies the row.
template <int D>
__global__ void __launch_bounds__(kWarps * 32) compress_bf16_kernel(CompressArgs a) {
    pdl_begin();
    constexpr int CPL = D / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    const int item = blockIdx.x * kWarps + warp;  // (entry, head) pair
    const int j = item / a.hkv, h = item % a.hkv;
    const int o0 = a.offs[b], o1 = a.offs[b + 1];
    if (o0 + j >= o1) return;
    const int t = a.idx[o0 + j];
    const int slot = (a.start ? a.start[b] : 0) + j;
    // bounds of every index read
    if (t < 0 || t >= a.f_lens[b] || t / kPage >= a.f_maxb || slot < 0 || slot / kPage >= a.c_maxb) {
        if (lane == 0) report(a.status, VC_ERR_BAD_INDEX);
        return;
    }
    const int fp = a.f_table[(int64_t)b * a.f_maxb + t / kPage];
    const int cp = a.c_table[(int64_t)b * a.c_maxb + slot / kPage];
    if (fp < 0 || fp >= a.f_pages || cp < 0 || cp >= a.c_pages) {
        if (lane == 0) report(a.status, VC_ERR_BAD_INDEX);
        return;
    }
    const int hb = head_block_bytes(16, D);
    const int64_t fbase = ((int64_t)fp * a.hkv + h) * hb + (int64_t)(t % kPage) * D * 2;
    const int64_t cbase = ((int64_t)cp * a.hkv + h) * hb + (int64_t)(slot % kPage) * D * 2;
#pragma unroll
    for (int kv = 0; kv < 2; ++kv) {
        uint16_t x[CPL];
        qrow::load_lane_row<D>((kv ? a.fv : a.fk) + fbase, lane, x);
        uint16_t *d16 = reinterpret_cast<uint16_t *>((kv ? a.cv : a.ck) + cbase);
#pragma unroll
        for (int i = 0; i < CPL; ++i) d16[lane * CPL + i] = x[i];
    }
}

template <int BITS, int D>
cudaError_t launch_bd(const CompressArgs &a, int batch, int max_kept, cudaStream_t st) {
    if constexpr (BITS == 16) {
        dim3 grid(ceil_div(max_kept * a.hkv, kWarps), batch);
        launch_pdl(compress_bf16_kernel<D>, grid, kWarps * 32, 0, st, a);
    } else if (max_kept <= kTokenPathMax) {
        dim3 grid(ceil_div(max_kept * a.hkv, kWarps), batch);
        launch_pdl(compress_token_kernel<BITS, D>, grid, kWarps * 32, 0, st, a);
    } else {
        // a range of max_kept slots starting anywhere touches at most this many pages
        dim3 grid(ceil_div(max_kept, kPage) + 1, a.hkv, batch);
        launch_pdl(compress_page_kernel<BITS, D>, grid, kPageWarps * 32, 0, st, a);
    }
    return cudaGetLastError();
}

template <int BITS>
cudaError_t launch_b(int d, const CompressArgs &a, int batch, int max_kept, cudaStream_t st) {
    switch (d) {
        case 32: if constexpr (BITS == 16) return launch_bd<BITS, 32>(a, batch, max_kept, st); break;
        case 64: return launch_bd<BITS, 64>(a, batch, max_kept, st);
        case 128: return launch_bd<BITS, 128>(a, batch, max_kept, st);
        case 256: return launch_bd<BITS, 256>(a, batch, max_kept, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

vc_status compress(const vc_paged_kv *full, const int32_t *kept_offsets, const int32_t *kept_idx,
                   const int32_t *comp_start, int32_t max_kept, const vc_paged_kv *comp,
                   int32_t *dev_status, cudaStream_t st) {
    if (!full || !comp || max_kept < 0 || full->batch < 0) return VC_ERR_INVALID_ARG;
    if (full->fmt.bits != 16) return VC_ERR_UNSUPPORTED;
    const int d = full->fmt.head_dim, hkv = full->fmt.num_kv_heads, bits = comp->fmt.bits;
    if (comp->fmt.head_dim != d || comp->fmt.num_kv_heads != hkv || full->batch != comp->batch)
        return VC_ERR_INVALID_ARG;
    if (!(d == 32 || d == 64 || d == 128 || d == 256) || hkv < 1) return VC_ERR_UNSUPPORTED;
    if (!(bits == 2 || bits == 3 || bits == 4 || bits == 16)) return VC_ERR_UNSUPPORTED;
    if (bits != 16 && d % 64) return VC_ERR_UNSUPPORTED;  // quantised formats: head_dim 64, 128, 256
    if (full->batch == 0 || max_kept == 0) return VC_OK;  // nothing is read or written
    if (!kept_offsets || !kept_idx || !full->k_pages || !full->v_pages || !full->block_table || !full->seq_lens ||
        !comp->k_pages || !comp->v_pages || !comp->block_table || full->max_blocks < 1 || comp->max_blocks < 1)
        return VC_ERR_INVALID_ARG;
    CompressArgs a;
    a.fk = (const uint8_t *)full->k_pages;
    a.fv = (const uint8_t *)full->v_pages;
    a.f_pages = full->num_pages;
    a.f_table = full->block_table;
    a.f_lens = full->seq_lens;
    a.f_maxb = full->max_blocks;
    a.ck = (uint8_t *)comp->k_pages;
    a.cv = (uint8_t *)comp->v_pages;
    a.c_pages = comp->num_pages;
    a.c_table = comp->block_table;
    a.c_maxb = comp->max_blocks;
    a.offs = kept_offsets;
    a.idx = kept_idx;
    a.start = comp_start;
    a.hkv = hkv;
    a.status = dev_status;
    cudaError_t e;
    switch (bits) {
        case 2: e = launch_b<2>(d, a, full->batch, max_kept, st); break;
        case 3: e = launch_b<3>(d, a, full->batch, max_kept, st); break;
        case 4: e = launch_b<4>(d, a, full->batch, max_kept, st); break;
        default: e = launch_b<16>(d, a, full->batch, max_kept, st); break;
    }
    return e == cudaSuccess ? VC_OK : VC_ERR_CUDA;
}

}  // namespace vc
