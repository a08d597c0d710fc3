// Library-wide host state: error messages, device error word, SM count, wait limit, version.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>
#include <atomic>
#include <mutex>
#include <cuda.h>
#include <cudaTypedefs.h>
#include "common.cuh"

namespace moe {

// The device error word: [0] flags (kDevErrTimeout, kDevErrBadIndex), [1] site code of the last error.
// One copy per device that loads the library; kernels get its address from device_error_word().
static __device__ unsigned g_error_word[2];

static thread_local char t_msg[512] = "";

int set_error(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_msg, sizeof(t_msg), fmt, ap);
    va_end(ap);
    return code;
}

static std::atomic<unsigned long long> g_launches{0};

int check_launch(const char* what) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return MOE_OK;
}

int check_launch(cudaError_t launch_result, const char* what) {
    const int rc = check_launch(what);
    if (rc != MOE_OK) return rc;
    if (launch_result != cudaSuccess)
        return set_error(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(launch_result));
    return MOE_OK;
}

static constexpr int kMaxDevices = 64;
static std::mutex g_mu;
static int g_sms[kMaxDevices];
static unsigned* g_err_ptr[kMaxDevices];

int num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sms[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

unsigned long long context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    if (!get_current || !get_id) return 0;
    CUcontext c = nullptr;
    if (get_current(&c) != CUDA_SUCCESS || !c) return 0;
    unsigned long long id = 0;
    return get_id(c, &id) == CUDA_SUCCESS ? id : 0;
}

static unsigned long long g_err_ctx[kMaxDevices];

unsigned* device_error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    const unsigned long long ctx = context_id();
    if (!g_err_ptr[dev] || ctx == 0 || g_err_ctx[dev] != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<unsigned*>(p);
        g_err_ctx[dev] = context_id();       // the lookup above made the context current if there was none
    }
    return g_err_ptr[dev];
}

static long long g_wait_limit = 0;
static constexpr long long kDefaultWaitLimit = 1LL << 26;   // mbarrier polls (seconds of waiting)

long long wait_limit() { return g_wait_limit > 0 ? g_wait_limit : kDefaultWaitLimit; }

}  // namespace moe

using namespace moe;

extern "C" const char* moe_last_error_string(void) { return t_msg; }

extern "C" void moe_set_wait_limit(long long spins) { g_wait_limit = spins > 0 ? spins : 0; }

extern "C" unsigned long long moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" const char* moe_version(void) { return "moe-gb300 0.1 (sm_103a)"; }

extern "C" int moe_check_device_error(void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, "moe_check_device_error: %s", cudaGetErrorString(e));
    unsigned* p = device_error_word();
    if (!p) return set_error(MOE_ERR_CUDA, "moe_check_device_error: device error word unavailable");
    unsigned w[2] = {0, 0};
    e = cudaMemcpy(w, p, sizeof(w), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, "moe_check_device_error: %s", cudaGetErrorString(e));
    if (w[0] == 0) return MOE_OK;
    const unsigned zero[2] = {0, 0};
    e = cudaMemcpy(p, zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, "moe_check_device_error: %s", cudaGetErrorString(e));
    if (w[0] & kDevErrTimeout)
        return set_error(MOE_ERR_TIMEOUT, "device wait ran out (flags 0x%x, site 0x%x)", w[0], w[1]);
    return set_error(MOE_ERR_INVALID_ARG, "device input check failed: topk id out of range (flags 0x%x, site 0x%x)",
                     w[0], w[1]);
}
