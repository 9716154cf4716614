// swa_decode_noalloc.cu -- swa_decode without any allocation, for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: plugins and embedded runtimes
// that are handed only their input and output buffers, processes whose device
// memory is owned entirely by another allocator (a framework's caching pool),
// and latency-critical loops where an allocation, and the device-wide
// synchronisation a cudaFree implies, is not allowed.  swa_decode
// grows a library workspace with cudaMalloc, and swa_decode_ex needs the caller
// to provide one; this entry point instead keeps the split-K partial results in
// a fixed array in the library's own device memory.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds it (SWA_NOALLOC_SCRATCH_BYTES) until the process exits.  In
// host code its name is only a host-side stand-in, never a device address: the
// device address is looked up with cudaGetSymbolAddress once per device, with
// that device current, on the first call made on that device.  Make that first
// call before any stream capture.
//
// Every call shares the one array and it keeps the last call's contents.
// Nothing in it needs to start at zero: each call's split pass writes every
// partial result that the same call's merge pass reads.  Calls whose kernels
// overlap on the GPU (concurrent streams, or concurrent host threads on one
// device) race on the array and must be serialised by the caller.
#include <mutex>

#include "swa_internal.h"

namespace {

constexpr size_t kScratchBytes = SWA_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up once
// per device); nullptr if the lookup fails.
void *scratch_address()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return nullptr;
        g_addr[dev] = p;
    }
    return g_addr[dev];
}

}  // namespace

extern "C" int swa_decode_noalloc(const void *q, const void *Kcache, const void *Vcache,
                                  const int32_t *pos, int B, int H, int Hkv, int d, int w, int g,
                                  float scale, void *O, swa_stream_t stream)
{
    // Workspace the automatic split count needs (0 for invalid sizes, which
    // swa_decode_ex then rejects); larger than the built-in array -> refuse.
    const size_t need = swa_decode_workspace_bytes(B, H, Hkv, d, w, g, 0);
    if (need > kScratchBytes) return SWA_ERR_WORKSPACE;
    void *ws = scratch_address();
    if (ws == nullptr) return SWA_ERR_CUDA;
    return swa_decode_ex(q, Kcache, Vcache, pos, B, H, Hkv, d, w, g, scale, O, nullptr, SWA_BF16, 0,
                         ws, kScratchBytes, stream);
}
