// vc_verify_attn: the verification pass over the full (bf16) cache on
// tcgen05 / TMEM (see verify_tc.cuh for the design).
//
// "VeriCache: Making Lossy KV Compression Exact", section "The Core Idea"
// items 3-5: one pass over KV_full checks all drafted positions in
// parallel; query i of the block attends causally to every earlier position
// and to itself ("KV Cache and Speculative Decoding": causal attention).
// Launch: one CTA per (split of 3648 keys, row block, request x kv head);
// a row block holds one 128-row MMA tile of (query, head) rows when there
// are at most 128 rows, else two (more rows take further row blocks).  When
// the last row block would hold a single tile behind full two-tile blocks
// (e.g. 40 queries x 8 heads = 256 + 64 rows), it runs as a second launch of
// one-tile CTAs, which fit two to an SM instead of leaving half of a
// two-tile CTA idle.
#include <type_traits>

#include "verify_tc.cuh"

namespace vc {
using vtc::Args;
namespace {

template <int D, int QT>
__global__ void __launch_bounds__(vtc::Cfg<D, QT>::THREADS, vtc::Cfg<D, QT>::MIN_CTAS) verify_kernel(const __grid_constant__ Args a) {
    pdl_wait();
    extern __shared__ __align__(1024) uint8_t smem[];
    vtc::verify_tc_cta<D, QT>(a, blockIdx.x, blockIdx.y + a.rb0, blockIdx.z, smem);
}

template <int D>
__global__ void verify_reduce_kernel(const float *ws_o, const float *ws_ml, int n_splits, float *out) {
    pdl_begin();
    vtc::reduce_row<D>(ws_o, ws_ml, n_splits, blockIdx.x, out, threadIdx.x, blockDim.x);
}

// Row blocks rb0 .. rb0 + n_rb - 1 of QT tiles each.
template <int D, int QT>
cudaError_t launch(Args a, int batch, int rb0, int n_rb, cudaStream_t st) {
    using C = vtc::Cfg<D, QT>;
    const cudaError_t e = set_smem_limit((const void *)verify_kernel<D, QT>, C::SMEM);
    if (e != cudaSuccess) return e;
    a.rows_per_cta = QT * vtc::kTileRows;
    a.rb0 = rb0;
    dim3 grid(a.n_splits, n_rb, batch * a.hkv);
    launch_pdl(verify_kernel<D, QT>, grid, C::THREADS, C::SMEM, st, a);
    return cudaGetLastError();
}

typedef CUresult (*EncodeTiled)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
    static EncodeTiled fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    }
    return fn;
}

// A page pool seen by the TMA unit: rows = pages * kv heads * 16 tokens,
// D bf16 channels each; boxes of 16 rows x 64 channels, 128-byte swizzle.
bool encode_pool(CUtensorMap *m, const void *pool, int64_t n_pages, int hkv, int d) {
    EncodeTiled fn = encoder();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)n_pages * hkv * kPage};
    cuuint64_t strides[1] = {(cuuint64_t)d * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)kPage};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(pool), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int verify_splits(int max_seq_len) { return max(1, ceil_div(ceil_div(max_seq_len, kPage), vtc::kSplitPages)); }

bool verify_supported(const vc_kv_format &f, int hq, int n_q) {
    const int d = f.head_dim, hkv = f.num_kv_heads;
    return f.bits == 16 && (d == 64 || d == 128) && hkv >= 1 && hq >= hkv && hq % hkv == 0 &&
           hq / hkv <= 8 && n_q >= 1 && n_q <= VC_MAX_VERIFY_QUERIES;
}

size_t verify_workspace(const vc_paged_kv &f, int n_q, int hq, int max_seq_len) {
    if (max_seq_len <= 0) return 0;
    return (size_t)f.batch * n_q * hq * verify_splits(max_seq_len) * (f.fmt.head_dim + 2) * sizeof(float);
}

// Fill the kernel arguments (shared with the mixed launch); false when the
// tensor maps of the pools cannot be encoded.
bool verify_args(Args &a, const void *q, int n_q, int hq, const vc_paged_kv &f, float scale, int max_seq_len,
                 void *ws, int32_t *status) {
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
    a.rows_per_cta = vtc::kTileRows;
    a.ws_o = (float *)ws;
    a.ws_ml = a.ws_o + (size_t)f.batch * n_q * hq * a.n_splits * f.fmt.head_dim;
    a.status = status;
    a.wait_ns = wait_fault().wait_ns;
    a.skip_copies = wait_fault().skip_copies;
    return encode_pool(&a.kmap, f.k_pages, f.num_pages, a.hkv, f.fmt.head_dim) &&
           encode_pool(&a.vmap, f.v_pages, f.num_pages, a.hkv, f.fmt.head_dim);
}

cudaError_t verify_launch(const void *q, int n_q, int hq, const vc_paged_kv &f, float scale, float *out,
                          int max_seq_len, void *ws, int32_t *status, cudaStream_t st) {
    Args a;
    if (!verify_args(a, q, n_q, hq, f, scale, max(max_seq_len, 1), ws, status)) return cudaErrorInvalidValue;
    const int d = f.fmt.head_dim;
    // one tile for up to 128 rows, else row blocks of two tiles; a last row
    // block with one tile behind full two-tile blocks runs as one-tile CTAs.
    // Every configuration uses the same 64-key blocks and rows as its own
    // unit, so a row's bits do not depend on n_q or on the split
    const int rows = n_q * a.grp, pair = 2 * vtc::kTileRows;
    const int full2 = rows / pair, rem = rows % pair;
    auto go = [&](auto dc) -> cudaError_t {
        constexpr int D = decltype(dc)::value;
        if (rows <= vtc::kTileRows) return launch<D, 1>(a, f.batch, 0, 1, st);
        if (full2 >= 1 && rem > 0 && rem <= vtc::kTileRows) {
            const cudaError_t e2 = launch<D, 2>(a, f.batch, 0, full2, st);
            if (e2 != cudaSuccess) return e2;
            return launch<D, 1>(a, f.batch, 2 * full2, 1, st);
        }
        return launch<D, 2>(a, f.batch, 0, ceil_div(rows, pair), st);
    };
    const cudaError_t e =
        d == 64 ? go(std::integral_constant<int, 64>{}) : go(std::integral_constant<int, 128>{});
    if (e != cudaSuccess) return e;
    const int out_rows = f.batch * n_q * hq;
    if (d == 64)
        launch_pdl(verify_reduce_kernel<64>, out_rows, 64, 0, st, a.ws_o, a.ws_ml, a.n_splits, out);
    else
        launch_pdl(verify_reduce_kernel<128>, out_rows, 128, 0, st, a.ws_o, a.ws_ml, a.n_splits, out);
    return cudaGetLastError();
}

}  // namespace vc
