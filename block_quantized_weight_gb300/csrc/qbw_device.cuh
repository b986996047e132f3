// qbw_device.cuh -- small device helpers shared by the qbw kernels: inline PTX
// for mbarriers, 1-D bulk asynchronous copies (TMA), packed fp32x2 arithmetic,
// bounded waits and the library's fault word.  sm_103a only.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace qbw {

// ------------------------------------------------------------------ fault word
// A kernel whose bounded wait expires sets a bit in the library's per-device
// fault word (passed to every kernel as a pointer) and returns; the host reads
// it with qbw_fault_read().
__device__ __forceinline__ void record_fault(unsigned int* fault, unsigned int code) {
    atomicOr(fault, 1u << code);
}

// ------------------------------------------------------------------ timers
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wall-clock bound of every spin-wait in the library.
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s

// ------------------------------------------------------------------ shared memory
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ float4 lds128f(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ float2 lds64f(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
    return v;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_inval(uint32_t bar) {
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Make mbarrier initialisation visible to the async proxy (bulk copies).
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) writes to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of the barrier to complete, giving up after
// limit_ns (kWaitLimitNs by default).  Returns false (and records `code`) on
// timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, unsigned int* fault,
                                                  unsigned int code, uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    uint32_t spins = 0;
    while (!mbar_try_wait(bar, parity)) {
        if ((++spins & 255u) == 0u && globaltimer_ns() - t0 > limit_ns) {
            record_fault(fault, code);
            return false;
        }
    }
    return true;
}

// Publish or clear a tagged 64-bit word (value in the lower half, tag in the
// upper): one store, so a reader sees the old word or the new one whole.
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// The launch's grid identifier (PTX %gridid): the same in every CTA of one
// grid, and different for grids launched at different times in this context.
__device__ __forceinline__ uint64_t grid_id() {
    uint64_t g;
    asm volatile("mov.u64 %0, %%gridid;" : "=l"(g));
    return g;
}

// Tag that marks a word published by this launch: 1 .. 2^32 - 1, different
// for any two grids fewer than 2^32 - 1 launches apart (0 means "no share").
__device__ __forceinline__ uint32_t launch_tag() { return (uint32_t)(grid_id() % 0xFFFFFFFFull) + 1u; }

// Wait until the 64-bit word at p carries `tag` in its upper half, reading it
// with relaxed gpu-scope loads, giving up after limit_ns.  A word with any
// other tag (consumed, stale, or another launch's) is not accepted.  Returns
// the last word read; on timeout records `code` (the word's tag is then not
// `tag`).
__device__ __forceinline__ unsigned long long wait_tag_u64(const unsigned long long* p, uint32_t tag,
                                                           unsigned int* fault, unsigned int code,
                                                           uint64_t limit_ns = kWaitLimitNs) {
    unsigned long long w;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
    if ((uint32_t)(w >> 32) == tag) return w;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
        if ((uint32_t)(w >> 32) == tag) return w;
        if (globaltimer_ns() - t0 > limit_ns) {
            record_fault(fault, code);
            return w;
        }
    }
}

// ------------------------------------------------------------------ bulk copy
// 1-D bulk copy global -> shared (TMA engine), completion counted in bytes on
// the given mbarrier.  src, dst 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// 2-D tensor copy global -> shared through a tensor map (TMA); the box lands
// row-major at dst (128-byte aligned); elements outside the tensor read as 0.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint32_t bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(tmap), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// Prefetch the box of a 2-D tensor map at (x, y) into L2 (no shared memory,
// no completion to wait for).
__device__ __forceinline__ void tma_prefetch_2d(const void* tmap, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(tmap), "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// Programmatic dependent launch: wait until the preceding grid on the stream
// has completed and its memory is visible (a no-op when the kernel was not
// launched as a programmatic dependent); allow the next grid to launch.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// L2 policy for data streamed exactly once (weights): evict first.
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ------------------------------------------------------------------ fp32x2
__device__ __forceinline__ uint64_t pack2(uint32_t lo, uint32_t hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1,%2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}

__device__ __forceinline__ uint64_t pack2f(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1,%2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ float2 unpack2f(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0,%1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}

// acc += a * b, element-wise on two fp32 lanes, round-to-nearest.
__device__ __forceinline__ void ffma2(uint64_t& acc, uint64_t a, uint64_t b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}

// a + b on two fp32 lanes.
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// ------------------------------------------------------------------ conversions
__device__ __forceinline__ float half_bits_to_float(uint32_t bits16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xFFFFu)));
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
    return __uint_as_float((bits16 & 0xFFFFu) << 16);
}

template <typename T>
__device__ __forceinline__ float load_act(const void* p, int64_t i);

template <>
__device__ __forceinline__ float load_act<float>(const void* p, int64_t i) {
    return __ldg(static_cast<const float*>(p) + i);
}

template <>
__device__ __forceinline__ float load_act<__nv_bfloat16>(const void* p, int64_t i) {
    return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
}

template <typename T>
__device__ __forceinline__ void store_out(void* p, int64_t i, float v);

template <>
__device__ __forceinline__ void store_out<float>(void* p, int64_t i, float v) {
    static_cast<float*>(p)[i] = v;
}

template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(void* p, int64_t i, float v) {
    static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
}

// gelu_tanh(v) = 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3))), fp32, with
// CUDA's tanhf (saturates to +-1 for large arguments, so no NaN for large |v|).
__device__ __forceinline__ float gelu_tanh(float v) {
    const float c = 0.7978845608028654f;   // sqrt(2/pi)
    const float inner = c * fmaf(0.044715f * v, v * v, v);
    return 0.5f * v * (1.0f + tanhf(inner));
}

}  // namespace qbw
