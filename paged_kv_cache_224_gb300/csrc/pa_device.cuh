// Device-side building blocks shared by the paged-KV kernels (sm_103a):
// shared-memory addresses, mbarrier waits with an iteration limit, 1-D bulk
// (TMA) copies from global to shared memory, and 16-bit -> fp32 unpacking.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/pa.h"

namespace pa {

constexpr unsigned kFull = 0xffffffffu;

// Upper bound on mbarrier polls before a wait gives up and flags
// PA_DEVERR_TIMEOUT.  A poll that finds the phase incomplete suspends for a
// while (about 7800 SM cycles on a GB300, measured with the self-test), so
// 2^18 polls is about one second -- orders of magnitude above any legitimate
// copy or pipeline latency.
constexpr uint32_t kMaxPolls = 1u << 18;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void flag_error(int *d_err, int bits) {
    if (d_err) atomicOr(d_err, bits);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity.  Returns false (after
// kMaxPolls polls) if the phase never completed.  A phase that is already
// complete is seen by a plain test: a try_wait costs the thread about 200
// cycles even then (measured: 3-4% of the prefill kernel's time).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t max_polls = kMaxPolls) {
    if (mbar_test(bar, parity)) return true;
    for (uint32_t i = 0; i < max_polls; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// L2 policy for data read exactly once (KV tiles): evict first.
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// L2 policy for data that other CTAs read again soon (a prompt's prefix K/V,
// read by every row tile of its kv head): evict last.
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 1-D bulk copy global -> shared (TMA engine), completion signalled on `bar`
// as transaction bytes.  dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint4 lds128(const void *p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_addr(p)));
    return v;
}

// ---------------------------------------------------------------- 16-bit data

template <typename T> struct Elem;

template <> struct Elem<__nv_bfloat16> {
    // bf16 is the top half of an fp32: widening is a shift / mask.
    static __device__ __forceinline__ void unpack2(uint32_t w, float &lo, float &hi) {
        lo = __uint_as_float(w << 16);
        hi = __uint_as_float(w & 0xffff0000u);
    }
    static __device__ __forceinline__ uint32_t pack2(float lo, float hi) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&v);
    }
};

template <> struct Elem<__half> {
    static __device__ __forceinline__ void unpack2(uint32_t w, float &lo, float &hi) {
        __half2 h = *reinterpret_cast<__half2 *>(&w);
        float2 f = __half22float2(h);
        lo = f.x;
        hi = f.y;
    }
    static __device__ __forceinline__ uint32_t pack2(float lo, float hi) {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&v);
    }
};

template <typename T>
__device__ __forceinline__ void unpack8(const uint4 &u, float (&f)[8]) {
    Elem<T>::unpack2(u.x, f[0], f[1]);
    Elem<T>::unpack2(u.y, f[2], f[3]);
    Elem<T>::unpack2(u.z, f[4], f[5]);
    Elem<T>::unpack2(u.w, f[6], f[7]);
}

template <typename T>
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    uint4 u;
    u.x = Elem<T>::pack2(f[0], f[1]);
    u.y = Elem<T>::pack2(f[2], f[3]);
    u.z = Elem<T>::pack2(f[4], f[5]);
    u.w = Elem<T>::pack2(f[6], f[7]);
    return u;
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization (launch_pdl) may be scheduled before the kernel ahead of it
// on the stream has finished; pdl_wait() blocks until that kernel has
// completed and its writes are visible (a no-op for an ordinary launch), so
// it comes before a kernel's first global access.  pdl_trigger() lets the
// next such kernel be scheduled once every CTA of this one has called it.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// max(a, b, c) in one instruction (three-input max.f32, sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace pa
