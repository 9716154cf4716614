// swa_status.cu -- the per-device status word the kernels report into, and
// the SM count used to size persistent grids.
#include <mutex>

#include "swa_internal.h"

namespace swa {

// Bit 0: a bounded wait ran out (DEV_ERR_TIMEOUT); bit 1: a negative
// position was passed to decode or append (DEV_ERR_BAD_POS).
__device__ int g_swa_device_status;

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
int *g_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

int current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}
}  // namespace

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
    if (v & DEV_ERR_BAD_POS) return SWA_ERR_INVALID_ARG;
    return SWA_OK;
}

}  // namespace swa
