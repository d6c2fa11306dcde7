// Device error word and status strings.
//
// Kernels that find a fault they can only see on the device (a block id or
// slot outside the pool, a bulk-copy wait that timed out) set a bit in this
// word and skip the work instead of trapping, so the CUDA context stays
// usable. The host reads and clears it with pa_get_device_error().
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pa_common.cuh"

__device__ unsigned int g_pa_device_error = 0;

namespace {
constexpr int kMaxDevices = 64;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
std::once_flag g_ctx_fns_once;
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// Driver entry points resolved through the runtime (the library does not
// link libcuda directly).
void resolve_ctx_fns() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(fn);
}

// Unique id of the calling thread's current context; 0 if there is none yet
// (or the driver cannot tell).
unsigned long long current_context_id() {
    std::call_once(g_ctx_fns_once, resolve_ctx_fns);
    CUcontext c = nullptr;
    if (!g_ctx_get_current || g_ctx_get_current(&c) != CUDA_SUCCESS || !c) return 0;
    unsigned long long id = 0;
    if (!g_ctx_get_id || g_ctx_get_id(c, &id) != CUDA_SUCCESS) return 0;
    return id;
}
}  // namespace

struct PaSymbolCache {
    std::mutex mu;
    unsigned long long ctx_id[kMaxDevices] = {};
    void* addr[kMaxDevices] = {};
};

PaSymbolCache* pa_symbol_cache_new() { return new PaSymbolCache(); }  // lives until the process exits

void* pa_symbol_address(PaSymbolCache* cache, const void* symbol) {
    int dev = 0;
    if (!cache || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    const unsigned long long id = current_context_id();
    std::lock_guard<std::mutex> lock(cache->mu);
    if (id != 0 && cache->ctx_id[dev] == id && cache->addr[dev]) return cache->addr[dev];
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess || !p) return nullptr;
    // the lookup makes the device's primary context current if none was
    cache->ctx_id[dev] = id != 0 ? id : current_context_id();
    cache->addr[dev] = p;
    return p;
}

unsigned int* pa_device_error_ptr() {
    static PaSymbolCache* cache = pa_symbol_cache_new();
    return static_cast<unsigned int*>(pa_symbol_address(cache, &g_pa_device_error));
}

extern "C" int pa_get_device_error(int* flags_out) {
    if (!flags_out) return PA_ERR_INVALID_ARG;
    unsigned int v = 0, zero = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return PA_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&v, g_pa_device_error, sizeof(v)) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaMemcpyToSymbol(g_pa_device_error, &zero, sizeof(zero)) != cudaSuccess) return PA_ERR_CUDA;
    *flags_out = (int)v;
    return PA_OK;
}

extern "C" const char* pa_status_string(int status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported configuration";
        case PA_ERR_WORKSPACE: return "workspace missing or too small";
        case PA_ERR_CUDA: return "CUDA runtime error";
        case PA_ERR_DEVICE: return "device-side error flagged";
        case PA_ERR_OOM: return "out of KV blocks";
        case PA_ERR_REFCOUNT: return "unknown sequence or refcount misuse";
        case PA_ERR_CAPACITY: return "output buffer too small";
        default: return "unknown status";
    }
}

// Self-test of the bounded waits: one thread waits on an mbarrier that
// nothing arrives on, with a limit of `limit_us` microseconds. The wait must
// give up, set PA_DEVERR_TIMEOUT and return, leaving the context usable.
__global__ void pa_selftest_wait_kernel(unsigned long long limit_ns, unsigned int* err) {
    __shared__ __align__(8) uint64_t bar;
    pa::mbar_init(&bar, 1);
    pa::fence_mbar_init();
    pa::mbar_wait(&bar, 0, err, limit_ns);  // phase 0 never completes
}

extern "C" int pa_selftest_wait_timeout(int limit_us, pa_stream_t stream) {
    if (limit_us <= 0 || limit_us > 10000000) return PA_ERR_INVALID_ARG;
    unsigned int* err = pa_device_error_ptr();
    if (!err) return PA_ERR_CUDA;
    pa_selftest_wait_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        (unsigned long long)limit_us * 1000ull, err);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
