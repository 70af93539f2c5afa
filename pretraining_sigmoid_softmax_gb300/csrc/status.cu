// Library-wide entry points: status strings, sizes, the per-device status word and the
// device checks every other entry point relies on.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "sizes.h"

namespace {

constexpr int kMaxDevices = 64;

// {first error code, site that recorded it}; one copy per device that loads the library.
__device__ int g_status_word[2];

int* g_status_ptr[kMaxDevices] = {nullptr};
int g_sm_count[kMaxDevices] = {0};
int g_supported[kMaxDevices] = {0};  // 0 unknown, 1 yes, 2 no
std::mutex g_mu;
std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};

// Site recorded by the bounded-wait self-check.
constexpr int kSiteWaitCheck = 90;

// One mbarrier that nothing ever arrives on, waited on with the bounded wait every role of
// the grouped-GEMM kernels uses. Nothing is in flight: the wait runs out after `limit_ns`,
// records MOE_ERR_TIMEOUT and the kernel returns.
__global__ void bounded_wait_check_kernel(int* status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    moe::mbar_init(moe::smem_u32(&bar), 1);
    moe::fence_mbar_init();
    moe::mbar_wait_bounded(moe::smem_u32(&bar), 0u, &abort_flag, status, limit_ns,
                           kSiteWaitCheck);
}

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

}  // namespace

namespace moe {

int* device_status_word() {
    int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int*>(p);
    }
    return g_status_ptr[dev];
}

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(); }

int sm_count() {
    int dev = current_device();
    if (dev < 0) return 1;
    if (!g_sm_count[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        g_sm_count[dev] = n > 0 ? n : 1;
    }
    return g_sm_count[dev];
}

bool device_supported() {
    int dev = current_device();
    if (dev < 0) return false;
    if (!g_supported[dev]) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        g_supported[dev] = (major == 10 && minor == 3) ? 1 : 2;
    }
    return g_supported[dev] == 1;
}

}  // namespace moe

extern "C" {

const char* moe_status_string(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape or device";
        case MOE_ERR_WORKSPACE: return "workspace too small";
        case MOE_ERR_LAUNCH: return "CUDA launch or runtime error";
        case MOE_ERR_BAD_INDEX: return "expert index out of range or layout overflow";
        case MOE_ERR_TIMEOUT: return "bounded device wait ran out";
        case MOE_ERR_TOO_LARGE: return "sizes exceed the library's fixed scratch array";
        default: return "unknown status";
    }
}

int moe_version(void) { return 100; }

int64_t moe_padded_rows(int64_t T, int k, int E) {
    if (T <= 0 || k <= 0 || E <= 0) return 0;
    int64_t r = T * k + (int64_t)E * (MOE_ROW_ALIGN - 1);
    return (r + MOE_ROW_ALIGN - 1) / MOE_ROW_ALIGN * MOE_ROW_ALIGN;
}

size_t moe_workspace_bytes(int64_t T, int d, int E, int k) {
    if (T <= 0 || d <= 0 || E <= 0 || k <= 0) return 0;
    return moe::ws_total(T, d, E, k);
}

int moe_device_status(moe_stream_t stream, int* code, int* site) {
    if (!code) return MOE_ERR_INVALID_ARG;
    int* w = moe::device_status_word();
    if (!w) return MOE_ERR_LAUNCH;
    int host[2] = {0, 0};
    if (cudaMemcpyAsync(host, w, sizeof(host), cudaMemcpyDeviceToHost, (cudaStream_t)stream) !=
        cudaSuccess)
        return MOE_ERR_LAUNCH;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MOE_ERR_LAUNCH;
    *code = host[0];
    if (site) *site = host[1];
    return MOE_OK;
}

int moe_clear_device_status(moe_stream_t stream) {
    int* w = moe::device_status_word();
    if (!w) return MOE_ERR_LAUNCH;
    if (cudaMemsetAsync(w, 0, 2 * sizeof(int), (cudaStream_t)stream) != cudaSuccess)
        return MOE_ERR_LAUNCH;
    return MOE_OK;
}

void moe_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns); }

int moe_check_bounded_wait(uint64_t limit_ns, moe_stream_t stream) {
    if (limit_ns == 0 || limit_ns > 1000000000ull) return MOE_ERR_INVALID_ARG;
    if (!moe::device_supported()) return MOE_ERR_UNSUPPORTED;
    int* w = moe::device_status_word();
    if (!w) return MOE_ERR_LAUNCH;
    bounded_wait_check_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(w, limit_ns);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

}  // extern "C"
