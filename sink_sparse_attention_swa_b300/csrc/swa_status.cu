// swa_status.cu -- the per-device status word the kernels report into, and
// the SM count used to size persistent grids.
#include <mutex>

#include "swa_internal.h"

namespace swa {

// Bit 0: a bounded wait ran out (DEV_ERR_TIMEOUT); bit 1: a negative
// position was passed to decode or append (DEV_ERR_BAD_POS); bit 2: a debug
// build's bounds check failed (DEV_ERR_BOUNDS).
__device__ int g_swa_device_status;

namespace {
std::mutex g_mu;
int *g_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
// one-shot stall injection per device (swa_debug_inject_stall): the kind of
// launch it applies to (0 = none) and that launch's wait limit
int g_stall_kind[kMaxDevices] = {};
uint64_t g_stall_ns[kMaxDevices] = {};
}  // namespace

bool take_injected_stall(int kind, uint64_t *wait_ns)
{
    const int dev = current_device();
    if (dev < 0) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_stall_kind[dev] != kind) return false;
    g_stall_kind[dev] = 0;
    *wait_ns = g_stall_ns[dev];
    return true;
}

int set_injected_stall(int kind, int64_t wait_ns)
{
    if (kind != 0 && kind != SWA_STALL_PREFILL && kind != SWA_STALL_DECODE &&
        kind != INJECT_SHRINK_BOUNDS)
        return SWA_ERR_INVALID_ARG;
    if ((kind == SWA_STALL_PREFILL || kind == SWA_STALL_DECODE) &&
        (wait_ns < 100000 || wait_ns > 2000000000))
        return SWA_ERR_INVALID_ARG;
    const int dev = current_device();
    if (dev < 0) return SWA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    g_stall_kind[dev] = kind;
    g_stall_ns[dev] = kind != 0 ? static_cast<uint64_t>(wait_ns) : 0;
    return SWA_OK;
}

int current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

int *status_ptr()
{
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_swa_device_status) != cudaSuccess) return nullptr;
        g_ptr[dev] = static_cast<int *>(p);
    }
    return g_ptr[dev];
}

int num_sms()
{
    const int dev = current_device();
    if (dev < 0) return 1;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sms[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v < 1)
            v = 1;
        g_sms[dev] = v;
    }
    return g_sms[dev];
}

int read_and_clear_status(cudaStream_t stream)
{
    int *p = status_ptr();
    if (p == nullptr) return SWA_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return SWA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SWA_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return SWA_ERR_CUDA;
    if (v & DEV_ERR_TIMEOUT) return SWA_ERR_DEVICE_TIMEOUT;
    if (v & DEV_ERR_BOUNDS) return SWA_ERR_DEVICE_BOUNDS;
    if (v & DEV_ERR_BAD_POS) return SWA_ERR_INVALID_ARG;
    return SWA_OK;
}

}  // namespace swa
