// vc_mixed_attn: drafting and verifying requests in one launch.
//
// "VeriCache: Making Lossy KV Compression Exact", section "Verifying Without
// Giving Back the Speedup", Figure 2 (cross-resource staggering): instead of
// all requests drafting and then all verifying, some requests verify against
// their full cache while the others keep drafting from the compressed one.
// Drafting is HBM-bandwidth bound, verification brings dense tensor work, so
// one grid holding both keeps both busy.  The first blocks run the
// verification body for the items of the requests with role 1, the next
// ones the draft body (8 warps) for the items of the requests with role 0,
// both over each request's own length (the grid is sized for the longest
// request and the worst split of roles; blocks past the two lists exit).
// One combine launch finishes both.  Blocks have 8 warps: the draft body
// uses all of them (16 draft warps per SM at two blocks per SM, as many as
// the standalone draft kernel keeps), the verification body 6 (the other two
// only join its CTA barriers).  Measured on the 32-request 3-bit workload
// against 6-warp blocks: the launch 871 -> 768 us, its drafting half alone
// 428 -> 329 us.  Interleaving verification and draft blocks in the grid
// (so that an SM holds one of each) was tried and not kept (766 us).
#include "draft_impl.cuh"
#include "verify_tc.cuh"

namespace vc {
int verify_splits(int max_seq_len);
bool verify_args(vtc::Args &a, const void *q, int n_q, int hq, const vc_paged_kv &f, float scale,
                 int max_seq_len, void *ws, int32_t *status);

namespace {

// the verification body of one 128-row tile needs 4 softmax warps, a
// producer warp and an MMA warp; draft blocks use all 8
constexpr int kThreads = 256;
static_assert(kThreads >= vtc::Cfg<128, 1>::THREADS && kThreads >= vtc::Cfg<64, 1>::THREADS,
              "the verification body's roles fit in a block");
constexpr int kDraftWarps = kThreads / 32;

struct MixedArgs {
    draft::DraftArgs d;
    vtc::Args v;
    const int32_t *role;
    int n_verify_blocks, rb, batch;
};

template <int BITS, int D>
struct MCfg {
    static constexpr int DS = draft::Cfg<BITS, D, kDraftWarps>::SMEM;
    static constexpr int VS = vtc::Cfg<D, 1>::SMEM;
    static constexpr int SMEM = DS > VS ? DS : VS;
};

// Splits of request b's verification (fixed 3648-key pieces of its length;
// one for a request shorter than its block, whose single block reports the
// error and writes zeros) and chunks of its KV_comp (0 for an empty one).
__device__ inline int verify_splits_of(const MixedArgs &m, int b) {
    const int len = m.v.lens[b];
    return len >= m.v.n_q ? ceil_div(ceil_div(len, kPage), vtc::kSplitPages) : 1;
}
__device__ inline int draft_chunks_of(const MixedArgs &m, int b) {
    return ceil_div(ceil_div(max(m.d.lens[b], 0), kPage), m.d.chunk_pages);
}
__device__ inline int verify_items(const MixedArgs &m, int b) { return m.v.hkv * m.rb * verify_splits_of(m, b); }
__device__ inline int draft_items(const MixedArgs &m, int b) { return m.d.hkv * draft_chunks_of(m, b); }

template <int BITS, int D>
__global__ void __launch_bounds__(kThreads) mixed_kernel(const __grid_constant__ MixedArgs m) {
    pdl_begin();
    extern __shared__ __align__(1024) uint8_t smem[];
    // The grid's blocks cover, in this order, the verification items of the
    // requests with role 1 (kv head x row block x split over the request's
    // own length), then the draft items of the requests with role 0 (kv
    // head x chunk over its own KV_comp length); blocks past both lists
    // exit.  Each block finds its item from the roles and lengths, so no
    // block is spent on a request of the other role or past a request's end.
    __shared__ int item[4];  // kind (1 verify, 2 draft, 0 none), request, index within the request
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int k = blockIdx.x, kind = 0, req = 0, local = 0;
        for (int pass = 1; pass <= 2 && kind == 0; ++pass) {
            int base = 0;
            for (int b0 = 0; b0 < m.batch; b0 += 32) {
                const int b = b0 + lane;
                int cnt = 0;
                if (b < m.batch && m.role[b] == (pass == 1 ? 1 : 0))
                    cnt = pass == 1 ? verify_items(m, b) : draft_items(m, b);
                int incl = cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                const int excl = incl - cnt;
                const unsigned hit = __ballot_sync(0xffffffffu, cnt > 0 && k >= base + excl && k < base + incl);
                if (hit) {
                    const int src = __ffs(hit) - 1;
                    kind = pass;
                    req = b0 + src;
                    local = k - base - __shfl_sync(0xffffffffu, excl, src);
                    break;
                }
                base += __shfl_sync(0xffffffffu, incl, 31);
            }
            if (kind == 0) k -= base;  // the draft items follow the verification items
        }
        if (lane == 0) {
            item[0] = kind;
            item[1] = req;
            item[2] = local;
        }
    }
    __syncthreads();
    const int kind = item[0], b = item[1], local = item[2];
    if (kind == 1) {
        const int ns = verify_splits_of(m, b);
        const int split = local % ns, rest = local / ns;
        const int rb = rest % m.rb, kvh = rest / m.rb;
        vtc::verify_tc_cta<D, 1>(m.v, split, rb, b * m.v.hkv + kvh, smem);
    } else if (kind == 2) {
        const int nc = draft_chunks_of(m, b);
        draft::draft_block<BITS, D, kDraftWarps>(m.d, local % nc, local / nc, b, m.d.chunk_pages, smem);
    }
}

template <int D>
__global__ void mixed_reduce_kernel(MixedArgs m, float *out_draft, float *out_verify, int draft_rows) {
    pdl_begin();
    const int row = blockIdx.x;
    if (row < draft_rows) {  // row = b * Hq + h
        const int b = row / m.d.hq;
        if (m.role[b] != 0) return;
        combine_partials<D>(m.d.ws_o, m.d.ws_ml, m.d.n_splits, draft_chunks_of(m, b), row, out_draft, threadIdx.x,
                            blockDim.x);
    } else {  // ((b * n_q + i) * Hq + h)
        const int r = row - draft_rows;
        const int b = r / (m.v.n_q * m.v.hq);
        if (m.role[b] != 1) return;
        combine_partials<D>(m.v.ws_o, m.v.ws_ml, m.v.n_splits, verify_splits_of(m, b), r, out_verify, threadIdx.x,
                            blockDim.x);
    }
}

int sms() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n < 1) n = 1;
    }
    return n;
}

// Draft chunking of the mixed launch: at least two draft blocks per SM over
// the whole batch, and at most 64 pages per warp (512 per block), so that
// requests of very different lengths (blocks past a request's end exit at
// once, as do blocks of verifying requests) still spread evenly over the SMs.
// (Caps of 24 / 32 / 43 / 64 / 96 / 128 pages per warp measured 808 / 783 /
// 770 / 755 / 755 / 770 us on the 32-request 3-bit workload.)
void draft_plan(int batch, int hkv, int max_seq_len, int &chunk, int &splits) {
    const int max_pages = ceil_div(max_seq_len, kPage);
    const int64_t units = (int64_t)batch * hkv;
    int s = (int)((2LL * sms() + units - 1) / units);
    s = max(s, ceil_div(max_pages, 64 * kDraftWarps));
    s = max(1, min(s, ceil_div(max_pages, kDraftWarps)));
    chunk = ceil_div(max_pages, s);
    chunk = max(kDraftWarps, ceil_div(chunk, kDraftWarps) * kDraftWarps);
    splits = max(1, ceil_div(max_pages, chunk));
}

size_t draft_part(const vc_paged_kv &comp, int hq, int max_seq_len) {
    int chunk, splits;
    draft_plan(comp.batch, comp.fmt.num_kv_heads, max_seq_len, chunk, splits);
    return (size_t)comp.batch * hq * splits * (comp.fmt.head_dim + 2) * sizeof(float);
}

template <int BITS, int D>
cudaError_t launch(const MixedArgs &m, int batch, float *out_draft, float *out_verify, cudaStream_t st) {
    using C = MCfg<BITS, D>;
    cudaError_t e = set_smem_limit((const void *)mixed_kernel<BITS, D>, C::SMEM);
    if (e != cudaSuccess) return e;
    const int nd = m.d.n_splits * m.d.hkv * batch;
    launch_pdl(mixed_kernel<BITS, D>, m.n_verify_blocks + nd, kThreads, C::SMEM, st, m);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int draft_rows = batch * m.d.hq, verify_rows = batch * m.v.n_q * m.v.hq;
    launch_pdl(mixed_reduce_kernel<D>, draft_rows + verify_rows, D, 0, st, m, out_draft, out_verify, draft_rows);
    return cudaGetLastError();
}

}  // namespace

size_t mixed_workspace(const vc_paged_kv &comp, const vc_paged_kv &full, int n_q, int hq, int max_seq_len) {
    if (max_seq_len <= 0) return 0;
    const size_t v = (size_t)full.batch * n_q * hq * verify_splits(max_seq_len) * (full.fmt.head_dim + 2) *
                     sizeof(float);
    return draft_part(comp, hq, max_seq_len) + v;
}

cudaError_t mixed_launch(const int32_t *role, const void *q_draft, const vc_paged_kv &comp, float *out_draft,
                         const void *q_verify, int n_q, const vc_paged_kv &full, float *out_verify, int hq,
                         float scale, int max_seq_len, void *ws, int32_t *status, cudaStream_t st) {
    MixedArgs m;
    const int d = comp.fmt.head_dim, bits = comp.fmt.bits, batch = comp.batch;
    int chunk, splits;
    draft_plan(batch, comp.fmt.num_kv_heads, max_seq_len, chunk, splits);
    m.d.q = (const uint16_t *)q_draft;
    m.d.kp = (const uint8_t *)comp.k_pages;
    m.d.vp = (const uint8_t *)comp.v_pages;
    m.d.n_pages = comp.num_pages;
    m.d.table = comp.block_table;
    m.d.lens = comp.seq_lens;
    m.d.maxb = comp.max_blocks;
    m.d.hq = hq;
    m.d.hkv = comp.fmt.num_kv_heads;
    m.d.grp = hq / m.d.hkv;
    m.d.scale_log2 = scale * 1.4426950408889634f;
    m.d.chunk_pages = chunk;
    m.d.n_splits = splits;
    m.d.ws_o = (float *)ws;
    m.d.ws_ml = m.d.ws_o + (size_t)batch * hq * splits * d;
    m.d.status = status;
    m.d.wait_ns = wait_fault().wait_ns;
    m.d.skip_copies = wait_fault().skip_copies;
    void *vws = (uint8_t *)ws + draft_part(comp, hq, max_seq_len);
    if (!verify_args(m.v, q_verify, n_q, hq, full, scale, max_seq_len, vws, status)) return cudaErrorInvalidValue;
    m.role = role;
    m.batch = batch;
    m.rb = ceil_div(n_q * m.v.grp, vtc::kTileRows);
    m.n_verify_blocks = m.v.n_splits * m.rb * batch * m.v.hkv;
#define VC_L(B_, D_) launch<B_, D_>(m, batch, out_draft, out_verify, st)
    if (d == 64)
        return bits == 2 ? VC_L(2, 64) : bits == 3 ? VC_L(3, 64) : bits == 4 ? VC_L(4, 64) : VC_L(16, 64);
    return bits == 2 ? VC_L(2, 128) : bits == 3 ? VC_L(3, 128) : bits == 4 ? VC_L(4, 128) : VC_L(16, 128);
#undef VC_L
}

}  // namespace vc
