// Internal helpers of libvc: device status reporting, bounded mbarrier waits,
// bulk (TMA) and cp.async copies, tensor-core fragments.  sm_103a only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <set>
#include <tuple>
#include <utility>

#include "vc.h"

namespace vc {

constexpr int kPage = VC_PAGE_TOKENS;  // tokens per page
constexpr int kGroup = VC_GROUP;       // channels per quantisation group

// Bytes of one kv head's block inside a page.
__host__ __device__ inline int head_block_bytes(int bits, int d) {
    return bits == 16 ? kPage * d * 2 : 2 * d * (bits + 1);
}
// Byte size of one token slot's packed codes.
__host__ __device__ inline int code_row_bytes(int bits, int d) { return d * bits / 8; }

// First error wins; the caller zeroes the word before the launch.
__device__ inline void report(int32_t *st, int code) {
    if (st) atomicCAS(st, 0, code);
}

// ---------------------------------------------------------------------------
// mbarrier + bulk copy (global -> shared, completion counted in bytes)
// ---------------------------------------------------------------------------
__device__ inline uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ inline void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ inline void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ inline void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ inline void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ inline bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    // no suspend-time hint: the poll returns after the hardware's own short
    // time limit even if the phase is still open (so the caller's wall-clock
    // bound holds), and a thread waiting on a phase that completes soon
    // resumes sooner than with a long hint (measured: verify 3 %, draft 2 %)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ inline uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait: gives up after limit_ns of wall-clock time (2 s unless a
// test lowered it with vc_debug_set_wait_fault), reports VC_ERR_TIMEOUT and
// returns false (the caller then drains and exits).
constexpr uint64_t kWaitNs = 2000000000ull;
__device__ inline bool mbar_wait(uint64_t *bar, uint32_t parity, int32_t *st, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) {
            report(st, VC_ERR_TIMEOUT);
            return false;
        }
    }
}

// Host-side fault injection for the tests of the bounded waits
// (vc_debug_set_wait_fault): the wait limit and whether the draft and
// verification kernels skip their KV copies, read by every launch.
struct WaitFault {
    uint64_t wait_ns = kWaitNs;
    int skip_copies = 0;
};
WaitFault wait_fault();

// One bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned).
__device__ inline void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ---------------------------------------------------------------------------
// cp.async (16 bytes, L2 only)
// ---------------------------------------------------------------------------
__device__ inline void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ inline void cp_async_zero16(void *dst, const void *src) {  // src-size 0: fills zeros
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, 0;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}
__device__ inline void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ inline void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------------------
// tensor-core fragments (mma.sync m16n8k16, fp32 accumulate)
// ---------------------------------------------------------------------------
__device__ inline void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// d = a b + c with separate accumulator input (c is left unchanged)
__device__ inline void mma_f16_c(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                 const float (&c)[4]) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
          "f"(c[3]));
}
// d = a b (zero accumulator input)
__device__ inline void mma_f16_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    const float z = 0.0f;
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
}
// Transpose an 8x8 matrix of 16-bit elements held in the mma fragment
// layout (thread (g, t) holds row g, columns 2t and 2t+1).
__device__ inline uint32_t movmatrix_t(uint32_t a) {
    uint32_t d;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

__device__ inline void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ inline void ldsm_x4_t(uint32_t (&r)[4], const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}

__device__ inline uint32_t pack_f16(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ inline uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ inline float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Combine the first `count` split partials (m, l, o) of one output row
// (`stride` slots per row; m in log2 units), in split order:
//   out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s,  M = max_s m_s
// (0 when no split saw a key).  The loads go out eight splits at a time --
// the partials come from L2, and one round trip per split would add up --
// while the arithmetic keeps split order.
template <int D>
__device__ __forceinline__ void combine_partials(const float *ws_o, const float *ws_ml, int stride, int count,
                                                 int64_t row, float *out, int tid, int nthreads) {
    constexpr int U = 8;
    const float *ml = ws_ml + row * stride * 2;
    float M = -INFINITY;
    for (int s0 = 0; s0 < count; s0 += U) {
        float m[U];
#pragma unroll
        for (int j = 0; j < U; ++j) m[j] = s0 + j < count ? ml[2 * (s0 + j)] : -INFINITY;
#pragma unroll
        for (int j = 0; j < U; ++j) M = fmaxf(M, m[j]);
    }
    for (int c = tid; c < D; c += nthreads) {
        float acc = 0.0f, L = 0.0f;
        if (M != -INFINITY) {
            for (int s0 = 0; s0 < count; s0 += U) {
                float mm[U], ll[U], oo[U];
#pragma unroll
                for (int j = 0; j < U; ++j) {
                    const bool in = s0 + j < count;
                    mm[j] = in ? ml[2 * (s0 + j)] : 0.0f;
                    ll[j] = in ? ml[2 * (s0 + j) + 1] : 0.0f;
                    oo[j] = in ? ws_o[(row * stride + s0 + j) * D + c] : 0.0f;
                }
#pragma unroll
                for (int j = 0; j < U; ++j) {
                    if (s0 + j < count) {
                        const float f = ex2(mm[j] - M);
                        acc += f * oo[j];
                        L += f * ll[j];
                    }
                }
            }
        }
        out[row * D + c] = L > 0.0f ? acc / L : 0.0f;
    }
}

__device__ inline float bf16_bits_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Kernels are launched with programmatic
// stream serialisation, so a kernel may be scheduled while the previous one
// on its stream is finishing (its launch and block set-up overlap that
// kernel's tail).  Every kernel starts with pdl_wait(): griddepcontrol.wait
// blocks until the previous kernel has completed and its memory is visible
// (so nothing it wrote or reads is touched before).  pdl_trigger()
// (griddepcontrol.launch_dependents) lets the next kernel be scheduled once
// every block of this one has called it or exited: short kernels call it at
// once (pdl_begin), long multi-wave kernels after their main loop, so that
// waiting blocks of the next kernel do not sit on SMs that still run this
// one's last wave.  Without the launch attribute both are no-ops.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_begin() {
    pdl_wait();
    pdl_trigger();
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// A kernel's dynamic shared-memory limit (needed above 48 KB), set once per
// (kernel, device, size): the attribute belongs to the device's context, so a
// process that drives several devices sets it on each of them.
inline cudaError_t set_smem_limit(const void *kernel, int bytes) {
    static std::mutex mu;
    static std::set<std::tuple<const void *, int, int>> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const auto key = std::make_tuple(kernel, dev, bytes);
    std::lock_guard<std::mutex> lock(mu);
    if (done.count(key)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.insert(key);
    return e;
}

}  // namespace vc
