// swa_chunk.cu -- the key lists of a chunked prefill.
//
// ("Sliding Window and Sparse Attention, from Longformer to CSA2", section 1:
// prefill processes many query positions at once, decode one; section 2: the
// rolling buffer keeps position i in slot i mod w and the first g positions
// permanently.)  A chunk of T new tokens at positions pos0 .. pos0+T-1 reads
// keys from the rolling cache (positions before pos0) and from itself.  This
// kernel lays them out, per (sequence, kv head), in the order the prefill
// kernels expect (swa_internal.h, chunk_*):
//   rows 0 .. S-1        sink slots w .. w+S-1 (positions 0 .. S-1)
//   rows S .. S+p-1      zero (the alignment padding, p = chunk_pad)
//   rows S+p .. S+p+A-1  ring slots of positions W0 .. pos0-1 (A = pos0 - W0)
//   then T rows          the chunk's own keys (positions pos0 .. pos0+T-1)
//   the remaining rows   zero (never read by a valid query; zero so that the
//                        unused rows of a partial key tile hold finite values)
// so the prefill kernels read each key with a 2-D tiled copy of contiguous
// rows, whatever the ring's wrap-around.
#include <cuda_bf16.h>

#include "swa_internal.h"

namespace swa {
namespace {

template <typename T, int HD>
__global__ void swa_chunk_gather_k(T *__restrict__ Kx, T *__restrict__ Vx, const T *__restrict__ Kc,
                                   const T *__restrict__ Vc, const T *__restrict__ kn,
                                   const T *__restrict__ vn, const int32_t *__restrict__ pos0,
                                   int B, int Hkv, int Tn, int w, int g, int rows, int *status)
{
    constexpr int C = HD * static_cast<int>(sizeof(T)) / 16;  // 16-byte pieces per row
    const size_t total = static_cast<size_t>(B) * Hkv * rows * C;
    const size_t slots = static_cast<size_t>(w) + g;
    for (size_t x = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; x < total;
         x += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int c = static_cast<int>(x % C);
        const int r = static_cast<int>((x / C) % rows);
        const size_t bk = x / C / rows;  // b * Hkv + kv head
        const int b = static_cast<int>(bk / Hkv);
        int ps = pos0[b];
        if (ps < 0 || ps > INT32_MAX - Tn) {  // invalid: report it, read the cache as if empty
            if (r == 0 && c == 0 && bk % Hkv == 0) atomicOr(status, DEV_ERR_BAD_POS);
            ps = 0;
        }
        const int S = chunk_sinks(ps, g), W0 = chunk_w0(ps, w, g), pad = chunk_pad(ps, w, g);
        const int L = S + pad + (ps - W0) + Tn;
        uint4 kv = make_uint4(0u, 0u, 0u, 0u), vv = kv;
        if (r < L && (r < S || r >= S + pad)) {
            const T *ks, *vs;
            if (r < S) {  // a sink slot
                const size_t off = (bk * slots + w + r) * HD;
                ks = Kc + off;
                vs = Vc + off;
            } else {
                const int pos = W0 + (r - S - pad);
                if (pos < ps) {  // still in the ring
                    const size_t off = (bk * slots + pos % w) * HD;
                    ks = Kc + off;
                    vs = Vc + off;
                } else {  // the chunk itself
                    const size_t off = (bk * Tn + (pos - ps)) * HD;
                    ks = kn + off;
                    vs = vn + off;
                }
            }
            // debug builds: the row read lies in the cache or the chunk
            [[maybe_unused]] const int pr = W0 + (r - S - pad);
            if (SWA_BOUNDS(r < S ? r < g : (pr >= 0 && (pr < ps || pr - ps < Tn)), status)) {
                kv = reinterpret_cast<const uint4 *>(ks)[c];
                vv = reinterpret_cast<const uint4 *>(vs)[c];
            }
        }
        reinterpret_cast<uint4 *>(Kx + (bk * rows + r) * HD)[c] = kv;
        reinterpret_cast<uint4 *>(Vx + (bk * rows + r) * HD)[c] = vv;
    }
}

template <typename T, int HD>
int launch_gather_t(void *Kx, void *Vx, const void *Kc, const void *Vc, const void *kn,
                    const void *vn, const int32_t *pos0, int B, int Hkv, int Tn, int w, int g,
                    cudaStream_t stream)
{
    const long long rows = chunk_rows_max(w, g, Tn);
    constexpr int C = HD * static_cast<int>(sizeof(T)) / 16;
    const size_t total = static_cast<size_t>(B) * Hkv * rows * C;
    const int threads = 256;
    size_t blocks = (total + threads - 1) / threads;
    const size_t cap = static_cast<size_t>(num_sms()) * 16;
    if (blocks > cap) blocks = cap;
    int *st = status_ptr();
    if (st == nullptr) return SWA_ERR_CUDA;
    swa_chunk_gather_k<T, HD><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
        static_cast<T *>(Kx), static_cast<T *>(Vx), static_cast<const T *>(Kc),
        static_cast<const T *>(Vc), static_cast<const T *>(kn), static_cast<const T *>(vn), pos0, B,
        Hkv, Tn, w, g, static_cast<int>(rows), st);
    return cudaGetLastError() == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
}

}  // namespace

int launch_chunk_gather(void *Kx, void *Vx, const void *Kc, const void *Vc, const void *k_new,
                        const void *v_new, const int32_t *pos0, int B, int Hkv, int T, int d,
                        int w, int g, swa_dtype dt, cudaStream_t stream)
{
    if (dt == SWA_BF16) {
        if (d == 128)
            return launch_gather_t<__nv_bfloat16, 128>(Kx, Vx, Kc, Vc, k_new, v_new, pos0, B, Hkv,
                                                       T, w, g, stream);
        if (d == 64)
            return launch_gather_t<__nv_bfloat16, 64>(Kx, Vx, Kc, Vc, k_new, v_new, pos0, B, Hkv,
                                                      T, w, g, stream);
    } else {
        if (d == 128)
            return launch_gather_t<float, 128>(Kx, Vx, Kc, Vc, k_new, v_new, pos0, B, Hkv, T, w,
                                               g, stream);
        if (d == 64)
            return launch_gather_t<float, 64>(Kx, Vx, Kc, Vc, k_new, v_new, pos0, B, Hkv, T, w, g,
                                              stream);
    }
    return SWA_ERR_UNSUPPORTED;
}

}  // namespace swa
