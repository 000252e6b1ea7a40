// vc_verify_attn: the verification pass over the full (bf16) cache.
//
// "VeriCache: Making Lossy KV Compression Exact", section "The Core Idea"
// items 3-5: one pass over KV_full checks all drafted positions in
// parallel; query i of the block attends causally to every earlier position
// and to itself ("KV Cache and Speculative Decoding": causal attention).
//
// Rows of the contraction are (query, head) pairs of one kv head's GQA
// group: n_q * G rows share every K/V byte, which makes QK^T / PV a dense
// contraction (128 rows for x = 32, G = 4).  Design:
//  - CTA = 8 warps x 16 rows (one m16 tile each) of one (request, kv head),
//    one split of 4096 keys (256 pages).  Splits are fixed by key position,
//    the pages of a split are visited in order and the split partials are
//    combined in split order, so a row's result never depends on n_q, on the
//    row's place in the block or on the batch.
//  - K/V pages staged in shared memory with cp.async (16-byte chunks, XOR
//    swizzle so ldmatrix is conflict-free), 4-stage ring, one barrier/page.
//  - S = Q K^T and O += P V on mma.sync m16n8k16 bf16, fp32 accumulate,
//    online softmax in fp32 (log2 domain).
#include "verify_impl.cuh"

namespace vc {
using verify::VerifyArgs;
using verify::VCfg;
using verify::kWarps;
using verify::kRows;
using verify::kSplitPages;
namespace {

template <int D>
__global__ void __launch_bounds__(verify::kMaxWarps * 32) verify_kernel(VerifyArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    verify::verify_block<D>(a, blockIdx.x, blockIdx.y, blockIdx.z, smem);
}

template <int D>
__global__ void verify_reduce_kernel(const float *ws_o, const float *ws_ml, int n_splits, float *out) {
    verify::reduce_row<D>(ws_o, ws_ml, n_splits, blockIdx.x, out, threadIdx.x, blockDim.x);
}

template <int D>
cudaError_t launch(const VerifyArgs &a, int batch, cudaStream_t st) {
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(verify_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, VCfg<D>::SMEM);
        attr = true;
    }
    // one warp per 16-row tile; as few CTAs per (request, kv head, split) as
    // the 16-warp limit allows, rows spread evenly over them
    const int tiles = ceil_div(a.n_q * a.grp, 16);
    const int rb = ceil_div(tiles, verify::kMaxWarps);
    const int warps = ceil_div(tiles, rb);
    dim3 grid(a.n_splits, rb, batch * a.hkv);
    verify_kernel<D><<<grid, warps * 32, VCfg<D>::SMEM, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return cudaSuccess;
}

}  // namespace

int verify_splits(int max_seq_len) { return max(1, ceil_div(ceil_div(max_seq_len, kPage), kSplitPages)); }

bool verify_supported(const vc_kv_format &f, int hq, int n_q) {
    const int d = f.head_dim, hkv = f.num_kv_heads;
    return f.bits == 16 && (d == 64 || d == 128) && hkv >= 1 && hq >= hkv && hq % hkv == 0 &&
           hq / hkv <= 8 && n_q >= 1 && n_q <= VC_MAX_VERIFY_QUERIES;
}

size_t verify_workspace(const vc_paged_kv &f, int n_q, int hq, int max_seq_len) {
    if (max_seq_len <= 0) return 0;
    return (size_t)f.batch * n_q * hq * verify_splits(max_seq_len) * (f.fmt.head_dim + 2) * sizeof(float);
}

// Fill the kernel arguments (shared with the mixed launch).
void verify_args(VerifyArgs &a, const void *q, int n_q, int hq, const vc_paged_kv &f, float scale,
                 int max_seq_len, void *ws, int32_t *status) {
    a.q = (const uint16_t *)q;
    a.kp = (const uint8_t *)f.k_pages;
    a.vp = (const uint8_t *)f.v_pages;
    a.n_pages = f.num_pages;
    a.table = f.block_table;
    a.lens = f.seq_lens;
    a.maxb = f.max_blocks;
    a.n_q = n_q;
    a.hq = hq;
    a.hkv = f.fmt.num_kv_heads;
    a.grp = hq / a.hkv;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.n_splits = verify_splits(max_seq_len);
    a.ws_o = (float *)ws;
    a.ws_ml = a.ws_o + (size_t)f.batch * n_q * hq * a.n_splits * f.fmt.head_dim;
    a.status = status;
}

cudaError_t verify_launch(const void *q, int n_q, int hq, const vc_paged_kv &f, float scale, float *out,
                          int max_seq_len, void *ws, int32_t *status, cudaStream_t st) {
    VerifyArgs a;
    verify_args(a, q, n_q, hq, f, scale, max(max_seq_len, 1), ws, status);
    const int d = f.fmt.head_dim;
    cudaError_t e = d == 64 ? launch<64>(a, f.batch, st) : launch<128>(a, f.batch, st);
    if (e != cudaSuccess) return e;
    const int rows = f.batch * n_q * hq;
    if (d == 64)
        verify_reduce_kernel<64><<<rows, 64, 0, st>>>(a.ws_o, a.ws_ml, a.n_splits, out);
    else
        verify_reduce_kernel<128><<<rows, 128, 0, st>>>(a.ws_o, a.ws_ml, a.n_splits, out);
    return cudaGetLastError();
}

}  // namespace vc
