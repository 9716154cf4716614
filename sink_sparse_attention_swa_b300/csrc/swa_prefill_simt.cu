// swa_prefill_simt.cu -- fp32 sliding-window (+ sinks) prefill on the CUDA
// cores.  Same semantics and the same block-sparse tile walk as the bf16
// tensor-core kernel, fp32 end to end, for inputs that must keep fp32
// precision (tensor-core TF32/BF16 cannot meet a 1e-5 error bound).
//
// ("Sliding Window and Sparse Attention, from Longformer to CSA2", sections
// 1-2; "Local and Sparse Attention: Reading Fewer Token Positions", Figures
// 1-2.)  One CTA per (q tile of 64 rows, residue class, head, batch); one
// query row per thread; key/value tiles of 32 rows staged in shared memory;
// online softmax in base 2 with the scale folded in.  The fixed patterns run
// as in the tensor-core kernel: residue classes (R > 1) address rows c + R t
// of class c; landmark tiles (rl > 0) read the rows 0, rl, 2 rl, ... .
#include <cmath>

#include "swa_internal.h"

namespace swa {
namespace {

constexpr int TM = 64;
constexpr int TN = 32;

template <int HD>
__global__ void __launch_bounds__(TM)
    swa_prefill_f32_simt(const float *__restrict__ Q, const float *__restrict__ K,
                         const float *__restrict__ V, float *__restrict__ O,
                         float *__restrict__ lse, const float *__restrict__ sink, int H,
                         int Hkv, int n, int n_k, int w, int g, float sl2,
                         const int32_t *__restrict__ pos0, int R, int rl, int *status)
{
    __shared__ __align__(16) float sK[TN][HD];
    __shared__ __align__(16) float sV[TN][HD];
    const int cls = blockIdx.x % R, qt = blockIdx.x / R, h = blockIdx.y, b = blockIdx.z;
    const int kvh = h / (H / Hkv);
    const int r = threadIdx.x;
    // rows (and keys) of this class: indices into its subsequence c, c+R, ...
    const int nq = (n - cls + R - 1) / R;
    const int nk = R == 1 ? n_k : nq;
    if (qt * TM >= nq) return;  // a class one row short may have one tile less
    // query row t of this thread; its index in the key list is i = t + off
    // (a chunked prefill lists its keys from chunk_offset(pos0[b]) on)
    int off = 0;
    if (pos0 != nullptr) {
        const int ps = pos0[b];
        off = chunk_offset(ps < 0 ? 0 : ps, w, g);
    }
    const int t = qt * TM + r;
    const int i = t + off;
    const size_t qrow = (static_cast<size_t>(b) * H + h) * n + cls + static_cast<size_t>(R) * t;
    const float *Kb = K + (static_cast<size_t>(b) * Hkv + kvh) * n_k * HD;
    const float *Vb = V + (static_cast<size_t>(b) * Hkv + kvh) * n_k * HD;

    float q[HD], acc[HD];
#pragma unroll
    for (int e = 0; e < HD; ++e) {
        q[e] = (t < nq) ? Q[qrow * HD + e] : 0.f;
        acc[e] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    const int q0 = qt * TM;
    TileRange tr = tile_range_at(q0 + off, (q0 + TM < nq ? q0 + TM : nq) - 1 + off, w, g, TN);
    add_landmarks(tr, w, g, rl, TN);
    const int lo = i - w + 1;
    const int lhi = land_hi(i, w, rl > 0 ? rl : 1), llo = rl > 0 ? land_lo(g, rl) : 0;
    for (int j = 0; j < tr.count; ++j) {
        // landmark tiles first (k a landmark index, key row rl k), then the
        // sink and band tiles (k an index into the class, key row c + R k)
        const bool land = j < tr.nl;
        const int k0 = (land ? tr.lt0 + j : tile_kt(tr, j - tr.nl)) * TN;
        const int khi = land ? lhi : i, klo = land ? llo : lo, kgs = land ? 0 : g;
        __syncthreads();
        for (int x = r; x < TN * HD / 4; x += TM) {
            const int row = x / (HD / 4), c4 = x % (HD / 4);
            const int kk = k0 + row;
            const long long krow = land ? static_cast<long long>(rl) * kk
                                        : cls + static_cast<long long>(R) * kk;
            float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
            if (land ? krow < n_k : kk < nk) {
                kv = reinterpret_cast<const float4 *>(Kb + static_cast<size_t>(krow) * HD)[c4];
                vv = reinterpret_cast<const float4 *>(Vb + static_cast<size_t>(krow) * HD)[c4];
            }
            reinterpret_cast<float4 *>(&sK[row][0])[c4] = kv;
            reinterpret_cast<float4 *>(&sV[row][0])[c4] = vv;
        }
        __syncthreads();
        float s[TN];
        float mt = -INFINITY;
#pragma unroll
        for (int c = 0; c < TN; ++c) {
            const int jj = k0 + c;
            const bool allowed = (t < nq) && (jj <= khi) && (jj >= klo || jj < kgs);
            float dot = 0.f;
#pragma unroll
            for (int e = 0; e < HD; ++e) dot = fmaf(q[e], sK[c][e], dot);
            s[c] = allowed ? dot * sl2 : -INFINITY;
            mt = fmaxf(mt, s[c]);
        }
        if (mt == -INFINITY) continue;  // no allowed key for this row in the tile
        const float m_new = fmaxf(m, mt);
        const float alpha = (m == -INFINITY) ? 0.f : exp2f(m - m_new);
        l *= alpha;
#pragma unroll
        for (int e = 0; e < HD; ++e) acc[e] *= alpha;
#pragma unroll
        for (int c = 0; c < TN; ++c) {
            const float pc = exp2f(s[c] - m_new);
            l += pc;
#pragma unroll
            for (int e = 0; e < HD; ++e) acc[e] = fmaf(pc, sV[c][e], acc[e]);
        }
        m = m_new;
    }
    if (t < nq && SWA_BOUNDS(qrow < static_cast<size_t>(gridDim.z) * H * n, status)) {
        float row_lse;
        const float inv = finish_row(m, l, sink, h, &row_lse);
#pragma unroll
        for (int e = 0; e < HD; ++e) O[qrow * HD + e] = acc[e] * inv;
        if (lse != nullptr) lse[qrow] = row_lse;
    }
}

template <int HD>
int launch_hd(const void *Q, const void *K, const void *V, void *O, float *lse, const float *sink,
              int B, int H, int Hkv, int n, int n_k, int w, int g, float scale,
              const int32_t *pos0, int R, int rl, cudaStream_t stream)
{
    if (rl > 0) R = 1;
    const int n_hi = (n + R - 1) / R;
    dim3 grid(((n_hi + TM - 1) / TM) * R, H, B);
    swa_prefill_f32_simt<HD><<<grid, TM, 0, stream>>>(
        static_cast<const float *>(Q), static_cast<const float *>(K),
        static_cast<const float *>(V), static_cast<float *>(O), lse, sink, H, Hkv, n, n_k, w, g,
        scale * 1.4426950408889634f, pos0, R, rl, status_ptr());
    return cudaGetLastError() == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
}

}  // namespace

int launch_prefill_f32(const void *Q, const void *K, const void *V, void *O, float *lse,
                       const float *sink, int B, int H, int Hkv, int n, int n_k, int d, int w,
                       int g, float scale, const int32_t *pos0, int R, int rl,
                       cudaStream_t stream)
{
    if (d == 64)
        return launch_hd<64>(Q, K, V, O, lse, sink, B, H, Hkv, n, n_k, w, g, scale, pos0, R, rl,
                             stream);
    if (d == 128)
        return launch_hd<128>(Q, K, V, O, lse, sink, B, H, Hkv, n, n_k, w, g, scale, pos0, R, rl,
                              stream);
    return SWA_ERR_UNSUPPORTED;
}

}  // namespace swa
