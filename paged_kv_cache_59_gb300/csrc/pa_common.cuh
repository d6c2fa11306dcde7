// Shared device helpers: status plumbing, bf16 packing, and thin inline-PTX
// wrappers for mbarrier waits and bulk asynchronous copies (sm_90+ ISA, used
// here on sm_103a). Every wait is bounded: it gives up after a wall-clock
// limit, sets PA_DEVERR_TIMEOUT in the device error word and reports failure
// so the caller can stop cleanly instead of hanging the GPU.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pagedkv.h"

#define PA_WAIT_LIMIT_NS 1000000000ull  // 1 s: far above any legitimate wait

// Address of the device error word for the current device (host side; the
// word lives in status.cu). Returns nullptr if the runtime call fails.
unsigned int* pa_device_error_ptr();

// Host: device address of a file-scope __device__ variable on the current
// device (host code cannot use the variable's name as a device address).
// The address is looked up with cudaGetSymbolAddress once per device and
// context and cached in *cache; a new context on the device (after a device
// reset) is looked up again. Thread-safe. nullptr if a runtime call fails.
struct PaSymbolCache;
PaSymbolCache* pa_symbol_cache_new();
void* pa_symbol_address(PaSymbolCache* cache, const void* symbol);

// Host-side helpers shared by the entry points.
static inline bool pa_aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Host: launches `kern` with programmatic stream serialization, so its launch
// and prologue overlap the tail of the previous kernel in the stream. The
// kernel must call pa::grid_dependency_wait() before it touches memory that
// earlier work in the stream reads or writes.
template <typename... KArgs, typename... Args>
static inline int pa_launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
               Args... args) {
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
    return cudaLaunchKernelEx(&cfg, kern, args...) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

namespace pa {

__device__ __forceinline__ void set_error(unsigned int* err, unsigned int bit) {
    if (err) atomicOr(err, bit);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Invalidates a barrier whose phases have all completed, before its memory
// is initialised again.
__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Makes barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Same test, but a thread whose phase is not complete may be suspended for up
// to `hint_ns` (or until the phase completes) instead of returning at once,
// so waiting warps take no issue slots from working ones.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity to complete. Returns false
// (and flags PA_DEVERR_TIMEOUT) if it did not complete within the limit.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned int* err,
                                          uint64_t limit_ns = PA_WAIT_LIMIT_NS) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0 && globaltimer_ns() - t0 > limit_ns) {
            set_error(err, PA_DEVERR_TIMEOUT);
            return false;
        }
    }
}

// ------------------------------------------------------- bulk async copies
// 1-D bulk copy global -> shared (this CTA), completion signalled on `bar`
// as transaction bytes. dst/src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// L2 policy for data read exactly once (the KV stream).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// ------------------------------------------------------------------ bf16
// bf16 -> fp32 is exact: the bf16 bits are the upper half of the fp32.
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
    float2 r;
    r.x = __uint_as_float(w << 16);
    r.y = __uint_as_float(w & 0xffff0000u);
    return r;
}

// fp32 -> bf16 round to nearest even (NaN kept quiet).
__device__ __forceinline__ uint32_t float2_to_bf16x2(float a, float b) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
}

// Four E4M3 codes (bytes 0..3 of w, byte 0 first) -> (v0, v1), (v2, v3).
// E4M3 values are a subset of fp16 values, so the hardware conversion to
// f16x2 and the widening to fp32 are both exact.
__device__ __forceinline__ void e4m3x4_to_float2x2(uint32_t w, float2& a, float2& b) {
    uint32_t h0, h1;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
        : "=r"(h0), "=r"(h1)
        : "r"(w));
    float f0, f1, f2, f3;
    asm("{\n\t.reg .f16 x, y;\n\t"
        "mov.b32 {x, y}, %2;\n\t"
        "cvt.f32.f16 %0, x;\n\t"
        "cvt.f32.f16 %1, y;\n\t}"
        : "=f"(f0), "=f"(f1)
        : "r"(h0));
    asm("{\n\t.reg .f16 x, y;\n\t"
        "mov.b32 {x, y}, %2;\n\t"
        "cvt.f32.f16 %0, x;\n\t"
        "cvt.f32.f16 %1, y;\n\t}"
        : "=f"(f2), "=f"(f3)
        : "r"(h1));
    a = make_float2(f0, f1);
    b = make_float2(f2, f3);
}

// Programmatic dependent launch: a kernel launched with the programmatic
// stream serialization attribute may start while the previous kernel in the
// stream is still running; grid_dependency_wait() blocks until that kernel
// has completed and its memory is visible (a no-op for ordinary launches).
// launch_dependents() lets the next such kernel be scheduled early.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace pa
