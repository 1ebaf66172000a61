// api.cu -- status handling shared by every dsix entry point.
#include <mutex>
#include <vector>

#include "common.cuh"

namespace {
__device__ int g_status = 0;

template <typename T, typename F>
T per_device(std::vector<T>& cache, std::mutex& mu, F make) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return T{};
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= static_cast<int>(cache.size())) cache.resize(dev + 1, T{});
    if (cache[dev] == T{}) cache[dev] = make(dev);
    return cache[dev];
}
}  // namespace

namespace dsix {

int* status_ptr() {
    static std::mutex mu;
    static std::vector<int*> cache;
    return per_device(cache, mu, [](int) -> int* {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
        return static_cast<int*>(p);
    });
}

int launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? IX_OK : IX_ERR_CUDA;
}

// The calling thread's current CUDA context (the device's primary context once
// the runtime has used the device), through the driver entry point; NULL when
// there is none yet or on error.
void* current_context() {
    using Fn = CUresult (*)(CUcontext*);
    static std::once_flag once;
    static Fn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<Fn>(p);
    });
    if (!fn) return nullptr;
    CUcontext c = nullptr;
    if (fn(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}

int num_sms() {
    static std::mutex mu;
    static std::vector<int> cache;
    int n = per_device(cache, mu, [](int dev) -> int {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        return v;
    });
    return n > 0 ? n : -1;
}

}  // namespace dsix

extern "C" const char* ix_status_string(int status) {
    switch (status) {
        case IX_OK: return "IX_OK";
        case IX_ERR_NULL: return "IX_ERR_NULL: a required pointer is NULL";
        case IX_ERR_SHAPE: return "IX_ERR_SHAPE: a size or stride is negative or inconsistent";
        case IX_ERR_UNSUPPORTED: return "IX_ERR_UNSUPPORTED: shape or parameter not supported";
        case IX_ERR_ALIGN: return "IX_ERR_ALIGN: pointer or stride breaks the required alignment";
        case IX_ERR_WORKSPACE: return "IX_ERR_WORKSPACE: workspace missing or too small";
        case IX_ERR_CUDA: return "IX_ERR_CUDA: the CUDA runtime rejected a launch or query";
        case IX_ERR_DEVICE_CHECK: return "IX_ERR_DEVICE_CHECK: a device-side check fired";
        default: return "unknown dsix status";
    }
}

extern "C" int ix_device_status(int* status_out) {
    int v = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return IX_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return IX_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_status, &zero, sizeof(int)) != cudaSuccess) return IX_ERR_CUDA;
    if (status_out) *status_out = v;
    return v ? IX_ERR_DEVICE_CHECK : IX_OK;
}
