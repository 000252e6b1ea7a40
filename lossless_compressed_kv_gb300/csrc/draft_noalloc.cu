// vc_draft_attn_static: the draft attention with its split partials kept in
// a fixed array that lives in the library, so the caller passes no
// workspace and nothing is allocated at call time.
//
// For callers that cannot allocate device memory where they call the
// library: for instance a plugin run by a host engine that owns every device
// allocation and hands out no scratch buffers, or a latency-critical path
// that must not call cudaMalloc (which can synchronise the device).  The
// caller still provides q, the cache and `out`.
//
// The array is 8 MiB and is held on every GPU that loads the library until
// the process exits.  Host code cannot pass the array's name to a kernel (on
// the host it names a host-side stand-in, not device memory), so the device
// address is looked up with cudaGetSymbolAddress while that device is
// current, checked, cached, and passed to the kernels.  The first call on
// each device does this look-up.  The cache is keyed on the device's current
// context as well: after cudaDeviceReset (or any tear-down and re-creation
// of the primary context) the module is loaded again, the array may sit at
// another address, and the next call looks it up again.
#include <cuda.h>

#include <mutex>

#include "vc_internal.cuh"

namespace vc {
size_t draft_workspace(const vc_paged_kv &c, int hq, int max_seq_len);
bool draft_supported(const vc_kv_format &f, int hq);
cudaError_t draft_launch(const void *q, int hq, const vc_paged_kv &c, float scale, float *out,
                         int max_seq_len, void *ws, int32_t *status, cudaStream_t st,
                         const void *k_new = nullptr, const void *v_new = nullptr, const int32_t *slot = nullptr);

namespace {

constexpr size_t kScratchBytes = VC_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_draft_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices] = {};
CUcontext g_ctx[kMaxDevices] = {};

// The calling thread's current driver context (the runtime's primary
// context of the current device once the runtime has initialised it).
using CtxGetCurrent = CUresult (*)(CUcontext *);
cudaError_t current_context(CUcontext *ctx) {
    static CtxGetCurrent fn = nullptr;
    static bool looked = false;
    if (!looked) {  // under g_mu
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrent>(p);
        looked = true;
    }
    if (!fn) return cudaErrorNotSupported;
    return fn(ctx) == CUDA_SUCCESS ? cudaSuccess : cudaErrorContextIsDestroyed;
}

// Device address of g_draft_scratch on the current device, looked up again
// whenever the device's context is not the one the cached address came from.
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    // cudaGetSymbolAddress initialises the runtime (and loads the module)
    // first, so the context is read after it
    void *p = nullptr;
    CUcontext ctx = nullptr;
    if (g_addr[dev]) {
        e = current_context(&ctx);
        if (e != cudaSuccess) return e;
        if (ctx == g_ctx[dev]) {
            *out = g_addr[dev];
            return cudaSuccess;
        }
    }
    e = cudaGetSymbolAddress(&p, g_draft_scratch);
    if (e != cudaSuccess) return e;
    if (!p) return cudaErrorInvalidSymbol;
    e = current_context(&ctx);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
    g_ctx[dev] = ctx;
    *out = p;
    return cudaSuccess;
}

}  // namespace
}  // namespace vc

using namespace vc;

extern "C" {

size_t vc_static_scratch_bytes(void) { return kScratchBytes; }

vc_status vc_draft_attn_static(const void *q, int32_t num_q_heads, const vc_paged_kv *comp, float softmax_scale,
                               float *out, int32_t max_seq_len, int32_t *dev_status, vc_stream_t stream) {
    // the checks of vc_draft_attn, in its order: formats first, then a batch
    // of 0 returns VC_OK (its per-request pointers may be NULL), then the
    // pointers of a batch with requests
    if (!comp || comp->batch < 0 || comp->fmt.num_kv_heads < 1 || comp->fmt.head_dim < 32 ||
        comp->fmt.head_dim % 32 || comp->fmt.head_dim > VC_MAX_HEAD_DIM || max_seq_len < 0)
        return VC_ERR_INVALID_ARG;
    if (!draft_supported(comp->fmt, num_q_heads)) return VC_ERR_UNSUPPORTED;
    if (comp->batch == 0) return VC_OK;
    if (!q || !out || !comp->k_pages || !comp->v_pages || !comp->block_table || !comp->seq_lens ||
        comp->max_blocks < 1 || comp->num_pages < 1)
        return VC_ERR_INVALID_ARG;
    const int msl = max_seq_len > 0 ? max_seq_len : 1;
    // every partial the combine pass reads is written by the same call first,
    // so nothing in the array has to start at zero
    if (draft_workspace(*comp, num_q_heads, msl) > kScratchBytes) return VC_ERR_WORKSPACE;
    void *ws = nullptr;
    if (scratch_address(&ws) != cudaSuccess) {
        cudaGetLastError();
        return VC_ERR_CUDA;
    }
    return draft_launch(q, num_q_heads, *comp, softmax_scale, out, msl, ws, dev_status, (cudaStream_t)stream) ==
                   cudaSuccess
               ? VC_OK
               : VC_ERR_CUDA;
}

}  // extern "C"
