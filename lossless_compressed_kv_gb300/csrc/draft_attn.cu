// vc_draft_attn: single-query GQA decode attention over the compressed cache.
//
// "VeriCache: Making Lossy KV Compression Exact", section "The Core Idea"
// (the drafter runs the same model with the compressed KV cache, one token
// per step) and section "Verifying Without Giving Back the Speedup"
// (drafting from compressed KV is a memory-bandwidth problem: every step
// re-reads the whole compressed cache from HBM).
//
// Design (sm_103a):
//  - Work item = (request, kv head, context chunk); a CTA of 4 warps owns one
//    chunk, each warp a strided subset of its 16-token pages.  Pages are
//    staged in shared memory by bulk (TMA) copies, one per K and per V head
//    block, completion tracked by an mbarrier per stage (4-deep ring/warp).
//  - The G query heads of the kv head share every K/V byte.  Per page the
//    products S^T = K Q^T (16 tokens x 8 head columns) and O^T += V^T P^T
//    (16 channels x 8 heads) run on mma.sync m16n8k16 with fp32 accumulate:
//    with 2-bit codes a page-head costs 2*G*D FMAs for 96 bytes, more than
//    the CUDA cores can retire at HBM speed.
//  - Dequantisation is folded around the MMA: codes enter as exact small
//    integers (f16), a 32-channel group is reduced separately and scaled:
//      q . k_hat = sum_g s_g (sum_{i in g} q_i c_i) + z_g (sum_{i in g} q_i)
//      sum_t p_t v_hat_t = sum_t (p_t s_{t,g}) c_t + sum_t p_t z_{t,g}
//    so no dequantised value is ever rounded.  bf16 caches (token-drop
//    KV_comp) feed the bf16 MMA directly.
//  - Online softmax in fp32 (log2 domain) against a lazy reference (moved
//    3 above a new maximum, so slightly larger later scores do not rescale
//    again); partial (m, l, o) per chunk in the workspace, combined by
//    draft_reduce_kernel.  Only a warp's last page can end inside; it is
//    the one page drafted with the masking code.
#include "draft_impl.cuh"

namespace vc {
namespace {

using draft::Cfg;
using draft::DraftArgs;
constexpr int kWarps = 4;

// Resident CTAs per SM the register budget is cut for.  Four (128
// registers): a five-CTA cap (102 registers) fits the 2-bit body but the
// extra register pressure costs more instructions than the extra warps hide
// (measured: 73.4 vs 68.8 us on the 8B-shaped 32k 2-bit workload).
template <int BITS, int D>
constexpr int kMinCtas = 4;

// One CTA per (unit = request x kv head, context chunk): units 0 ..
// lo_units - 1 first, in n_lo chunks of chunk_pages each, then the others in
// n_hi (smaller) chunks of chunk_hi.
template <int BITS, int D>
__global__ void __launch_bounds__(kWarps * 32, kMinCtas<BITS, D>) draft_kernel(DraftArgs a) {
    pdl_begin();
    extern __shared__ __align__(128) uint8_t smem[];
    int c = blockIdx.x, unit, split, chunk;
    if (c < a.lo_units * a.n_lo) {
        unit = c / a.n_lo;
        split = c % a.n_lo;
        chunk = a.chunk_pages;
    } else {
        c -= a.lo_units * a.n_lo;
        unit = a.lo_units + c / a.n_hi;
        split = c % a.n_hi;
        chunk = a.chunk_hi;
    }
    draft::draft_block<BITS, D, kWarps>(a, split, unit % a.hkv, unit / a.hkv, chunk, smem);
}

template <int D>
__global__ void draft_reduce_kernel(const float *ws_o, const float *ws_ml, int n_splits, int grp, int hkv,
                                    int lo_units, int n_hi, int n_lo, float *out) {
    pdl_begin();
    const int64_t row = (int64_t)blockIdx.y * gridDim.x + blockIdx.x;  // b * Hq + h
    const int unit = blockIdx.y * hkv + blockIdx.x / grp;
    draft::reduce_row<D>(ws_o, ws_ml, n_splits, unit < lo_units ? n_lo : n_hi, row, out, threadIdx.x,
                         blockDim.x);
}

// lo_units units in n_lo chunks of chunk_pages, the others in n_hi chunks of
// chunk_hi pages (n_hi >= n_lo); n_splits = the workspace's chunk slots per row.
struct Plan {
    int chunk_pages, n_lo, lo_units, chunk_hi, n_hi, n_splits;
};

template <int BITS, int D>
int occupancy() {
    static int occ = -1;
    if (occ < 0) {
        using C = Cfg<BITS, D, kWarps>;
        set_smem_limit((const void *)draft_kernel<BITS, D>, C::SMEM);
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, draft_kernel<BITS, D>, kWarps * 32, C::SMEM) !=
                cudaSuccess ||
            n < 1)
            n = 1;
        occ = n;
    }
    return occ;
}

int num_sms() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n < 1) n = 1;
    }
    return n;
}

template <int BITS, int D>
Plan plan(int batch, int hkv, int max_seq_len) {
    // One full wave: as many CTAs as SMs x resident CTAs, every one inside
    // one unit.  When the slots are not a multiple of the units, (slots mod
    // units) units take one chunk more (smaller chunks), so that every slot
    // holds a CTA.  The block scheduler fills the SMs breadth first, so each
    // SM gets both sizes; the larger chunks are launched first, because the
    // warp schedulers favour a CTA's warps by age and the first CTAs on an
    // SM run faster: that way an SM's CTAs end closer together.
    const int max_pages = ceil_div(max_seq_len, kPage);
    const int64_t units = (int64_t)batch * hkv;
    const int64_t slots = (int64_t)num_sms() * occupancy<BITS, D>();
    const int cap = ceil_div(max_pages, kWarps);  // a warp needs a page
    const int64_t per_unit = slots / units;
    const int base = per_unit < 1 ? 1 : (per_unit > cap ? cap : (int)per_unit);
    auto chunk_for = [&](int splits) { return max(kWarps, ceil_div(ceil_div(max_pages, splits), kWarps) * kWarps); };
    Plan p;
    p.chunk_pages = chunk_for(base);
    p.n_lo = max(1, ceil_div(max_pages, p.chunk_pages));
    p.lo_units = (int)units;
    p.chunk_hi = p.chunk_pages;
    p.n_hi = p.n_lo;
    const int64_t extra = slots - (int64_t)base * units;
    if (base + 1 <= cap && extra > 0 && extra < units) {
        const int ch = chunk_for(base + 1);
        const int nh = max(1, ceil_div(max_pages, ch));
        if (nh > p.n_lo) {
            p.lo_units = (int)(units - extra);
            p.chunk_hi = ch;
            p.n_hi = nh;
        }
    }
    p.n_splits = max(p.n_hi, p.n_lo);
    return p;
}

template <int BITS>
Plan plan_b(int d, int batch, int hkv, int max_seq_len) {
    return d == 64 ? plan<BITS, 64>(batch, hkv, max_seq_len) : plan<BITS, 128>(batch, hkv, max_seq_len);
}

Plan plan_any(int bits, int d, int batch, int hkv, int max_seq_len) {
    switch (bits) {
        case 2: return plan_b<2>(d, batch, hkv, max_seq_len);
        case 3: return plan_b<3>(d, batch, hkv, max_seq_len);
        case 4: return plan_b<4>(d, batch, hkv, max_seq_len);
        default: return plan_b<16>(d, batch, hkv, max_seq_len);
    }
}

template <int BITS, int D>
cudaError_t launch(const DraftArgs &a, int batch, cudaStream_t st) {
    using C = Cfg<BITS, D, kWarps>;
    const cudaError_t e = set_smem_limit((const void *)draft_kernel<BITS, D>, C::SMEM);
    if (e != cudaSuccess) return e;
    const int64_t units = (int64_t)batch * a.hkv;
    const int64_t ctas = (int64_t)a.lo_units * a.n_lo + (units - a.lo_units) * a.n_hi;
    launch_pdl(draft_kernel<BITS, D>, dim3((unsigned)ctas), kWarps * 32, C::SMEM, st, a);
    return cudaGetLastError();
}

}  // namespace

bool draft_supported(const vc_kv_format &f, int hq) {
    const int d = f.head_dim, hkv = f.num_kv_heads, bits = f.bits;
    return (d == 64 || d == 128) && hkv >= 1 && hq >= hkv && hq % hkv == 0 && hq / hkv <= 8 &&
           (bits == 2 || bits == 3 || bits == 4 || bits == 16);
}

size_t draft_workspace(const vc_paged_kv &c, int hq, int max_seq_len) {
    if (max_seq_len <= 0) return 0;
    const Plan p = plan_any(c.fmt.bits, c.fmt.head_dim, c.batch, c.fmt.num_kv_heads, max_seq_len);
    return (size_t)c.batch * hq * p.n_splits * (c.fmt.head_dim + 2) * sizeof(float);
}

cudaError_t draft_launch(const void *q, int hq, const vc_paged_kv &c, float scale, float *out,
                         int max_seq_len, void *ws, int32_t *status, cudaStream_t st, const void *k_new,
                         const void *v_new, const int32_t *slot) {
    const int d = c.fmt.head_dim, bits = c.fmt.bits;
    DraftArgs a;
    const Plan p = plan_any(bits, d, c.batch, c.fmt.num_kv_heads, max(max_seq_len, 1));
    a.q = (const uint16_t *)q;
    a.kp = (const uint8_t *)c.k_pages;
    a.vp = (const uint8_t *)c.v_pages;
    a.n_pages = c.num_pages;
    a.table = c.block_table;
    a.lens = c.seq_lens;
    a.maxb = c.max_blocks;
    a.hq = hq;
    a.hkv = c.fmt.num_kv_heads;
    a.grp = hq / a.hkv;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.chunk_pages = p.chunk_pages;
    a.n_splits = p.n_splits;
    a.n_lo = p.n_lo;
    a.lo_units = p.lo_units;
    a.chunk_hi = p.chunk_hi;
    a.n_hi = p.n_hi;
    a.ws_o = (float *)ws;
    a.ws_ml = a.ws_o + (size_t)c.batch * hq * p.n_splits * d;
    a.status = status;
    a.wait_ns = wait_fault().wait_ns;
    a.skip_copies = wait_fault().skip_copies;
    a.k_new = (const uint16_t *)k_new;
    a.v_new = (const uint16_t *)v_new;
    a.slot = slot;
    cudaError_t e;
#define VC_L(B_, D_) launch<B_, D_>(a, c.batch, st)
    if (d == 64) {
        e = bits == 2 ? VC_L(2, 64) : bits == 3 ? VC_L(3, 64) : bits == 4 ? VC_L(4, 64) : VC_L(16, 64);
    } else {
        e = bits == 2 ? VC_L(2, 128) : bits == 3 ? VC_L(3, 128) : bits == 4 ? VC_L(4, 128) : VC_L(16, 128);
    }
#undef VC_L
    if (e != cudaSuccess) return e;
    dim3 rg(hq, c.batch);
    if (d == 64)
        launch_pdl(draft_reduce_kernel<64>, rg, 64, 0, st, a.ws_o, a.ws_ml, p.n_splits, a.grp, a.hkv, p.lo_units,
                   p.n_hi, p.n_lo, out);
    else
        launch_pdl(draft_reduce_kernel<128>, rg, 128, 0, st, a.ws_o, a.ws_ml, p.n_splits, a.grp, a.hkv,
                   p.lo_units, p.n_hi, p.n_lo, out);
    return cudaGetLastError();
}

}  // namespace vc
