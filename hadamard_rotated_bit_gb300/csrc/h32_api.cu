// Library-wide entry points: device checks, status reporting, wait bounds.
#include <atomic>
#include <mutex>

#include "h32_common.cuh"

namespace h32 {
// the status word of the router and combine kernels (h32_moe.cu)
h32_status moe_read_and_clear_status(cudaStream_t s);

namespace {

std::atomic<uint64_t> g_wait_polls{kDefaultWaitPolls};

struct DeviceInfo {
    int checked = 0;  // 0 = not yet, 1 = sm_103, -1 = not supported
    int sm_count = 0;
};

constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::mutex g_dev_mutex;

}  // namespace

uint64_t wait_limit() { return g_wait_polls.load(std::memory_order_relaxed); }

namespace {
thread_local const char *t_last_cuda_error = "no error";
}

h32_status launch_status(cudaError_t e) {
    if (e == cudaSuccess) return H32_OK;
    t_last_cuda_error = cudaGetErrorString(e);
    return H32_ERR_CUDA;
}

void note_error(const char *what) { t_last_cuda_error = what; }

h32_status check_device(int *sm_count) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        cudaGetLastError();
        return H32_ERR_UNSUPPORTED;
    }
    if (dev >= kMaxDevices) return H32_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo &info = g_devices[dev];
    if (info.checked == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return H32_ERR_UNSUPPORTED;
        }
        info.checked = (major == 10 && minor == 3) ? 1 : -1;
        info.sm_count = sms;
    }
    if (info.checked != 1) return H32_ERR_UNSUPPORTED;
    if (sm_count) *sm_count = info.sm_count;
    return H32_OK;
}

}  // namespace h32

extern "C" h32_status h32_device_status(void *stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    H32_TRY(h32::check_device(nullptr));
    const cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return h32::launch_status(e);
    // one caller at a time: each status word is taken through one device word
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    const h32_status st[4] = {h32::quant_read_and_clear_status(s),
                              h32::gemm_read_and_clear_status(s),
                              h32::tc_read_and_clear_status(s),
                              h32::moe_read_and_clear_status(s)};
    for (h32_status v : st)
        if (v == H32_ERR_CUDA) return H32_ERR_CUDA;
    for (h32_status v : st)
        if (v == H32_ERR_TIMEOUT) return H32_ERR_TIMEOUT;
    for (h32_status v : st)
        if (v != H32_OK) return v;
    return H32_OK;
}

extern "C" const char *h32_status_string(h32_status st) {
    switch (st) {
        case H32_OK: return "ok";
        case H32_ERR_INVALID_ARG: return "invalid argument";
        case H32_ERR_ALIGNMENT: return "pointer or row pitch not 16-byte aligned";
        case H32_ERR_UNSUPPORTED: return "no sm_103 CUDA device";
        case H32_ERR_CUDA: return "CUDA runtime error";
        case H32_ERR_TIMEOUT: return "a bounded device wait gave up";
        case H32_ERR_DEVICE_GUARD: return "device-side range check failed";
    }
    return "unknown status";
}

extern "C" void h32_set_wait_limit(uint64_t polls) {
    h32::g_wait_polls.store(polls == 0 ? h32::kDefaultWaitPolls : polls, std::memory_order_relaxed);
}

extern "C" int h32_version(void) { return 100; }

extern "C" const char *h32_last_cuda_error(void) { return h32::t_last_cuda_error; }
