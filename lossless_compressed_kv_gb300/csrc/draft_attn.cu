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
//  - Online softmax in fp32 (log2 domain), partial (m, l, o) per chunk in the
//    workspace, combined by draft_reduce_kernel.
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

template <int BITS, int D>
__global__ void __launch_bounds__(kWarps * 32, kMinCtas<BITS, D>) draft_kernel(DraftArgs a) {
    pdl_begin();
    extern __shared__ __align__(128) uint8_t smem[];
    draft::draft_block<BITS, D, kWarps>(a, blockIdx.x, blockIdx.y, blockIdx.z, smem);
}

template <int D>
__global__ void draft_reduce_kernel(const float *ws_o, const float *ws_ml, int n_splits, float *out) {
    pdl_begin();
    const int64_t row = (int64_t)blockIdx.y * gridDim.x + blockIdx.x;  // b * Hq + h
    draft::reduce_row<D>(ws_o, ws_ml, n_splits, row, out, threadIdx.x, blockDim.x);
}

struct Plan {
    int chunk_pages, n_splits;
};

template <int BITS, int D>
int occupancy() {
    static int occ = -1;
    if (occ < 0) {
        using C = Cfg<BITS, D, kWarps>;
        cudaFuncSetAttribute(draft_kernel<BITS, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
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
    // one full wave: at most SMs x resident CTAs work items, equal chunks
    const int max_pages = ceil_div(max_seq_len, kPage);
    const int64_t units = (int64_t)batch * hkv;
    const int64_t slots = (int64_t)num_sms() * occupancy<BITS, D>();
    int splits = (int)(slots / units);
    splits = max(1, min(splits, ceil_div(max_pages, kWarps)));
    int chunk = ceil_div(max_pages, splits);
    chunk = max(kWarps, ceil_div(chunk, kWarps) * kWarps);
    Plan p;
    p.chunk_pages = chunk;
    p.n_splits = max(1, ceil_div(max_pages, chunk));
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
    occupancy<BITS, D>();  // sets the shared-memory attribute once
    dim3 grid(a.n_splits, a.hkv, batch);
    launch_pdl(draft_kernel<BITS, D>, grid, kWarps * 32, C::SMEM, st, a);
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
    a.ws_o = (float *)ws;
    a.ws_ml = a.ws_o + (size_t)c.batch * hq * p.n_splits * d;
    a.status = status;
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
        launch_pdl(draft_reduce_kernel<64>, rg, 64, 0, st, a.ws_o, a.ws_ml, p.n_splits, out);
    else
        launch_pdl(draft_reduce_kernel<128>, rg, 128, 0, st, a.ws_o, a.ws_ml, p.n_splits, out);
    return cudaGetLastError();
}

}  // namespace vc
