// Device error word and status strings.
//
// Kernels that find a fault they can only see on the device (a block id or
// slot outside the pool, a bulk-copy wait that timed out) set a bit in this
// word and skip the work instead of trapping, so the CUDA context stays
// usable. The host reads and clears it with pa_get_device_error().
#include <cuda_runtime.h>

#include "pa_common.cuh"

__device__ unsigned int g_pa_device_error = 0;

namespace {
constexpr int kMaxDevices = 64;
unsigned int* g_err_ptr[kMaxDevices] = {nullptr};
}

unsigned int* pa_device_error_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    if (!g_err_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pa_device_error) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<unsigned int*>(p);
    }
    return g_err_ptr[dev];
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
