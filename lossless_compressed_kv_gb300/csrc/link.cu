// Paced host-to-device copies: a slower link emulated on one machine.
//
// "VeriCache: Making Lossy KV Compression Exact", the two serving settings:
// in remote prefix caching the compressed cache of a stored prefix is sent to
// the serving GPU, which can start decoding from it, while the full cache
// stays reachable for verification.  Study notes "VeriCache: Turning Lossy KV
// Cache into Lossless LLM Inference", case 3: the slow link carries KV_comp
// to the drafter, a fast link brings KV_full to the verifier.
//
// vc_link_clock stores the device's global timer (ns) as the link's time
// origin.  vc_stage_paced_async splits a copy into chunks; before chunk k a
// one-thread kernel on the copy stream waits until the timer reaches
// origin + (link_offset + end of chunk k) / rate, so each chunk lands no
// earlier than a link of that rate would deliver it.  The wait is bounded by
// its own deadline (the host rejects offsets beyond kMaxLinkNs) and by a
// second bound of kMaxLinkNs on the time spent waiting.
#include "vc_internal.cuh"

namespace vc {
namespace {

constexpr double kMaxLinkNs = 60e9;  // a paced copy may span at most 60 s of link time

__global__ void link_clock_kernel(int64_t *origin) {
    if (threadIdx.x == 0 && blockIdx.x == 0) *origin = (int64_t)global_ns();
}

__global__ void link_wait_kernel(const int64_t *origin, int64_t offset_ns) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    const uint64_t target = (uint64_t)(*origin + offset_ns);
    const uint64_t t0 = global_ns();
    for (;;) {
        const uint64_t now = global_ns();
        if (now >= target || now - t0 > (uint64_t)kMaxLinkNs) return;
        __nanosleep(1000);
    }
}

}  // namespace
}  // namespace vc

extern "C" {

vc_status vc_link_clock(int64_t *origin_ns, vc_stream_t stream) {
    if (!origin_ns) return VC_ERR_INVALID_ARG;
    vc::link_clock_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(origin_ns);
    return cudaGetLastError() == cudaSuccess ? VC_OK : VC_ERR_CUDA;
}

vc_status vc_stage_paced_async(void *dev_dst, const void *pinned_src, size_t bytes, size_t chunk_bytes,
                               double bytes_per_ns, const int64_t *origin_ns, size_t link_offset_bytes,
                               vc_stream_t side, vc_event_t done) {
    if (!dev_dst || !pinned_src || !origin_ns || chunk_bytes == 0 || !(bytes_per_ns > 0.0))
        return VC_ERR_INVALID_ARG;
    if ((double)(link_offset_bytes + bytes) / bytes_per_ns > vc::kMaxLinkNs) return VC_ERR_INVALID_ARG;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, pinned_src) != cudaSuccess) {
        cudaGetLastError();
        return VC_ERR_STAGING;
    }
    if (at.type != cudaMemoryTypeHost) return VC_ERR_STAGING;
    cudaStream_t s = (cudaStream_t)side;
    for (size_t off = 0; off < bytes; off += chunk_bytes) {
        const size_t n = bytes - off < chunk_bytes ? bytes - off : chunk_bytes;
        const int64_t release = (int64_t)((double)(link_offset_bytes + off + n) / bytes_per_ns);
        vc::link_wait_kernel<<<1, 32, 0, s>>>(origin_ns, release);
        if (cudaGetLastError() != cudaSuccess) return VC_ERR_CUDA;
        if (cudaMemcpyAsync((char *)dev_dst + off, (const char *)pinned_src + off, n, cudaMemcpyHostToDevice, s) !=
            cudaSuccess)
            return VC_ERR_CUDA;
    }
    if (done && cudaEventRecord((cudaEvent_t)done, s) != cudaSuccess) return VC_ERR_CUDA;
    return VC_OK;
}

}  // extern "C"
