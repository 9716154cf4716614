// swa_decode.cu -- single-token decode over the rolling-buffer KV cache, and
// the cache append that fills it.
//
// ("Sliding Window and Sparse Attention, from Longformer to CSA2", section 1:
// decode reads the whole cache from HBM for every generated token, so memory
// bandwidth sets the speed; section 2: the rolling buffer, position i in slot
// i mod w, and attention sinks kept permanently; section 6: the log-sum-exp
// merges partial results over disjoint key sets exactly.  "Local and Sparse
// Attention: Reading Fewer Token Positions", Figure 4: the rolling cache.)
//
// Cache layout [B][Hkv][w+g][d]: ring slots 0..w-1, then sink slots w..w+g-1.
// For a query at position pos the keys it reads are stored in
//   ring slots 0 .. nring-1,  nring = min(w, pos+1)   (a ring slot t < nring
//                             holds a position in pos-w+1 .. pos)
//   sink slots w .. w+nsink-1, nsink = clamp(pos-w+1, 0, g)  (sinks that have
//                             left the window; the others are read from the
//                             ring, so no key is read twice)
// so the valid slots form two contiguous runs, enumerated as a virtual index
// v in [0, nring+nsink).
//
// Pass 1 (split kernel): CTA (split s, kv head, batch) streams its share of
// the valid slots once with 16-byte coalesced loads, keeps the G query heads
// of the group together so each key/value row is read once for all of them,
// and runs a per-warp online softmax (base 2, scale folded into q).  The CTA's
// warps merge in shared memory and write (m, l, unnormalised o) per head.
// Pass 2 (merge kernel): per (batch, head), the log-sum-exp merge of the
// splits.  With a single split pass 1 writes the final output itself.
#include <cmath>
#include <cstdlib>

#include "swa_internal.h"
#include "swa_ptx.cuh"

namespace swa {
namespace {

constexpr int DEC_WARPS = 4;
constexpr int KEYS_PER_GROUP = 8;
constexpr float LN2 = 0.69314718055994530942f;

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <typename T>
struct Elem;
template <>
struct Elem<__nv_bfloat16> {
    static constexpr int PER16 = 8;  // elements per 16 bytes
    __device__ static void unpack(const uint4 &u, float (&f)[8])
    {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            f[2 * k] = __uint_as_float(w[k] << 16);
            f[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
        }
    }
    __device__ static float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
    __device__ static __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};
template <>
struct Elem<float> {
    static constexpr int PER16 = 4;
    __device__ static void unpack(const uint4 &u, float (&f)[4])
    {
        f[0] = __uint_as_float(u.x);
        f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z);
        f[3] = __uint_as_float(u.w);
    }
    __device__ static float to_f(float x) { return x; }
    __device__ static float from_f(float x) { return x; }
};

struct DecodeParams {
    int B, H, Hkv, w, g, S;  // S = number of splits
    float sl2;
    const int32_t *pos;
    int *status; // device status word (a negative position is reported there)
    float *ws;   // [B][H][S][d+2] when S > 1
    void *O;     // [B][H][d]
    float *lse;  // [B][H] or null
};

// slot of the v-th valid key
__device__ __forceinline__ int valid_slot(int v, int nring, int w) { return v < nring ? v : w + (v - nring); }

template <typename T, int HD, int G>
__global__ void __launch_bounds__(DEC_WARPS * 32)
    swa_decode_split(const T *__restrict__ q, const T *__restrict__ Kc, const T *__restrict__ Vc,
                     const DecodeParams p)
{
    using E = Elem<T>;
    constexpr int EPL = E::PER16;            // elements per lane per row chunk
    constexpr int LPR = HD / EPL;            // lanes per key row
    constexpr int RPI = 32 / LPR;            // key rows per warp load
    constexpr int NI = KEYS_PER_GROUP / RPI; // loads per lane per group
    static_assert(LPR <= 32 && 32 % LPR == 0 && KEYS_PER_GROUP % RPI == 0, "lane mapping");

    __shared__ float sm_m[DEC_WARPS][G], sm_l[DEC_WARPS][G];
    __shared__ float sm_o[DEC_WARPS][G][HD];

    const int s = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cidx = lane % LPR, rr = lane / LPR;
    int pos = p.pos[b];
    if (pos < 0) {  // invalid: read nothing, report it, output zeros
        if (threadIdx.x == 0 && s == 0 && kvh == 0) atomicOr(p.status, DEV_ERR_BAD_POS);
        pos = -1;
    }
    const int nring = pos + 1 < p.w ? pos + 1 : p.w;
    int nsink = pos - p.w + 1;
    nsink = nsink < 0 ? 0 : (nsink > p.g ? p.g : nsink);
    const int nvalid = nring + nsink;
    const int chunk = (nvalid + p.S - 1) / p.S;
    const int v_begin = s * chunk;
    const int v_end = min(v_begin + chunk, nvalid);
    const size_t slots = static_cast<size_t>(p.w) + p.g;
    const T *Kb = Kc + (static_cast<size_t>(b) * p.Hkv + kvh) * slots * HD + cidx * EPL;
    const T *Vb = Vc + (static_cast<size_t>(b) * p.Hkv + kvh) * slots * HD + cidx * EPL;

    // this lane's slice of the G query rows, pre-multiplied by scale*log2(e)
    float qf[G][EPL];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        const T *qr = q + (static_cast<size_t>(b) * p.H + kvh * G + hh) * HD + cidx * EPL;
#pragma unroll
        for (int e = 0; e < EPL; ++e) qf[hh][e] = E::to_f(qr[e]) * p.sl2;
    }
    float m[G], l[G], acc[G][EPL];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        m[hh] = -INFINITY;
        l[hh] = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[hh][e] = 0.f;
    }

    constexpr int STRIDE = DEC_WARPS * KEYS_PER_GROUP;
    uint4 kc[NI], vc[NI], kn[NI], vn[NI];
    auto load = [&](int g0, uint4 (&kr)[NI], uint4 (&vr)[NI]) {
#pragma unroll
        for (int k = 0; k < NI; ++k) {
            const int v = g0 + k * RPI + rr;
            if (v < v_end) {
                const size_t off = static_cast<size_t>(valid_slot(v, nring, p.w)) * HD;
                kr[k] = __ldcs(reinterpret_cast<const uint4 *>(Kb + off));
                vr[k] = __ldcs(reinterpret_cast<const uint4 *>(Vb + off));
            } else {
                kr[k] = make_uint4(0, 0, 0, 0);
                vr[k] = make_uint4(0, 0, 0, 0);
            }
        }
    };
    int g0 = v_begin + warp * KEYS_PER_GROUP;
    if (g0 < v_end) load(g0, kc, vc);
    for (; g0 < v_end; g0 += STRIDE) {
        const int gn = g0 + STRIDE;
        if (gn < v_end) load(gn, kn, vn);
        // scores: partial dot products, then a butterfly over the LPR lanes of a row
        float sc[NI][G];
#pragma unroll
        for (int k = 0; k < NI; ++k) {
            float kf[EPL];
            E::unpack(kc[k], kf);
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                float d0 = 0.f;
#pragma unroll
                for (int e = 0; e < EPL; ++e) d0 = fmaf(qf[hh][e], kf[e], d0);
                sc[k][hh] = d0;
            }
        }
#pragma unroll
        for (int off = 1; off < LPR; off <<= 1)
#pragma unroll
            for (int k = 0; k < NI; ++k)
#pragma unroll
                for (int hh = 0; hh < G; ++hh)
                    sc[k][hh] += __shfl_xor_sync(0xffffffffu, sc[k][hh], off);
#pragma unroll
        for (int k = 0; k < NI; ++k)
            if (g0 + k * RPI + rr >= v_end)
#pragma unroll
                for (int hh = 0; hh < G; ++hh) sc[k][hh] = -INFINITY;
        // online softmax per head over the group's keys (all lanes agree)
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            float mt = sc[0][hh];
#pragma unroll
            for (int k = 1; k < NI; ++k) mt = fmaxf(mt, sc[k][hh]);
#pragma unroll
            for (int off = LPR; off < 32; off <<= 1)
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
            const float m_new = fmaxf(m[hh], mt);
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = ex2(m[hh] - m_use);
            float ls = 0.f;
            float pk[NI];
#pragma unroll
            for (int k = 0; k < NI; ++k) {
                pk[k] = ex2(sc[k][hh] - m_use);
                ls += pk[k];
            }
#pragma unroll
            for (int off = LPR; off < 32; off <<= 1) ls += __shfl_xor_sync(0xffffffffu, ls, off);
            l[hh] = l[hh] * alpha + ls;
            m[hh] = m_new;
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[hh][e] *= alpha;
#pragma unroll
            for (int k = 0; k < NI; ++k) {
                float vf[EPL];
                E::unpack(vc[k], vf);
#pragma unroll
                for (int e = 0; e < EPL; ++e) acc[hh][e] = fmaf(pk[k], vf[e], acc[hh][e]);
            }
        }
#pragma unroll
        for (int k = 0; k < NI; ++k) {
            kc[k] = kn[k];
            vc[k] = vn[k];
        }
    }
    // combine the RPI row groups of the warp, then the warps of the CTA
#pragma unroll
    for (int hh = 0; hh < G; ++hh)
#pragma unroll
        for (int e = 0; e < EPL; ++e)
#pragma unroll
            for (int off = LPR; off < 32; off <<= 1)
                acc[hh][e] += __shfl_xor_sync(0xffffffffu, acc[hh][e], off);
    if (lane < LPR) {
#pragma unroll
        for (int hh = 0; hh < G; ++hh)
#pragma unroll
            for (int e = 0; e < EPL; ++e) sm_o[warp][hh][cidx * EPL + e] = acc[hh][e];
    }
    if (lane == 0) {
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            sm_m[warp][hh] = m[hh];
            sm_l[warp][hh] = l[hh];
        }
    }
    __syncthreads();
    for (int x = threadIdx.x; x < G * HD; x += DEC_WARPS * 32) {
        const int hh = x / HD, col = x % HD;
        float M = -INFINITY;
#pragma unroll
        for (int wv = 0; wv < DEC_WARPS; ++wv) M = fmaxf(M, sm_m[wv][hh]);
        const float Mu = (M == -INFINITY) ? 0.f : M;
        float Lsum = 0.f, o = 0.f;
#pragma unroll
        for (int wv = 0; wv < DEC_WARPS; ++wv) {
            const float sc = ex2(sm_m[wv][hh] - Mu);
            Lsum += sc * sm_l[wv][hh];
            o += sc * sm_o[wv][hh][col];
        }
        const int h = kvh * G + hh;
        if (p.S == 1) {
            T *Or = static_cast<T *>(p.O) + (static_cast<size_t>(b) * p.H + h) * HD;
            Or[col] = E::from_f(Lsum > 0.f ? o / Lsum : 0.f);
            if (col == 0 && p.lse != nullptr)
                p.lse[static_cast<size_t>(b) * p.H + h] = (M + log2f(Lsum)) * LN2;
        } else {
            float *wr = p.ws + ((static_cast<size_t>(b) * p.H + h) * p.S + s) * (HD + 2);
            if (col == 0) {
                wr[0] = M;
                wr[1] = Lsum;
            }
            wr[2 + col] = o;
        }
    }
}

template <typename T, int HD>
__global__ void __launch_bounds__(HD) swa_decode_merge(const DecodeParams p)
{
    using E = Elem<T>;
    const int bh = blockIdx.x;  // b * H + h
    const int col = threadIdx.x;
    const float *wr = p.ws + static_cast<size_t>(bh) * p.S * (HD + 2);
    float M = -INFINITY;
    for (int s = 0; s < p.S; ++s) M = fmaxf(M, wr[s * (HD + 2)]);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float L = 0.f, o = 0.f;
    for (int s = 0; s < p.S; ++s) {
        const float *x = wr + s * (HD + 2);
        const float sc = ex2(x[0] - Mu);
        L += sc * x[1];
        o += sc * x[2 + col];
    }
    static_cast<T *>(p.O)[static_cast<size_t>(bh) * HD + col] = E::from_f(L > 0.f ? o / L : 0.f);
    if (col == 0 && p.lse != nullptr) p.lse[bh] = (M + log2f(L)) * LN2;
}

template <typename T, int HD, int G>
int launch_decode_t(const void *q, const void *Kc, const void *Vc, const DecodeParams &p,
                    cudaStream_t stream)
{
    dim3 grid(p.S, p.Hkv, p.B);
    swa_decode_split<T, HD, G><<<grid, DEC_WARPS * 32, 0, stream>>>(
        static_cast<const T *>(q), static_cast<const T *>(Kc), static_cast<const T *>(Vc), p);
    if (cudaGetLastError() != cudaSuccess) return SWA_ERR_CUDA;
    if (p.S > 1) {
        swa_decode_merge<T, HD><<<p.B * p.H, HD, 0, stream>>>(p);
        if (cudaGetLastError() != cudaSuccess) return SWA_ERR_CUDA;
    }
    return SWA_OK;
}

template <typename T, int HD>
int dispatch_g(const void *q, const void *Kc, const void *Vc, const DecodeParams &p, int G,
               cudaStream_t stream)
{
    switch (G) {
    case 1: return launch_decode_t<T, HD, 1>(q, Kc, Vc, p, stream);
    case 2: return launch_decode_t<T, HD, 2>(q, Kc, Vc, p, stream);
    case 4: return launch_decode_t<T, HD, 4>(q, Kc, Vc, p, stream);
    case 8: return launch_decode_t<T, HD, 8>(q, Kc, Vc, p, stream);
    default: return SWA_ERR_UNSUPPORTED;
    }
}

// -------------------------------------------------------------- append
template <typename T, int HD>
__global__ void swa_cache_append_k(T *__restrict__ Kc, T *__restrict__ Vc,
                                   const T *__restrict__ kn, const T *__restrict__ vn,
                                   const int32_t *__restrict__ pos0, int T_new, int B, int Hkv,
                                   int w, int g, int *status)
{
    constexpr int C = HD * static_cast<int>(sizeof(T)) / 16;  // 16-byte chunks per row
    const size_t total = static_cast<size_t>(B) * Hkv * T_new * C;
    const size_t slots = static_cast<size_t>(w) + g;
    for (size_t x = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; x < total;
         x += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int c = static_cast<int>(x % C);
        const size_t row = x / C;  // (b * Hkv + kvh) * T_new + t
        const int t = static_cast<int>(row % T_new);
        const size_t bk = row / T_new;
        const int b = static_cast<int>(bk / Hkv);
        const int p0 = pos0[b];
        if (p0 < 0) {  // invalid: write nothing, report it
            if (c == 0 && t == 0) atomicOr(status, DEV_ERR_BAD_POS);
            continue;
        }
        const int p = p0 + t;
        const uint4 kv = reinterpret_cast<const uint4 *>(kn + row * HD)[c];
        const uint4 vv = reinterpret_cast<const uint4 *>(vn + row * HD)[c];
        T *kbase = Kc + bk * slots * HD;
        T *vbase = Vc + bk * slots * HD;
        if (t >= T_new - w) {  // only the last w new positions survive in the ring
            const size_t slot = static_cast<size_t>(p % w);
            reinterpret_cast<uint4 *>(kbase + slot * HD)[c] = kv;
            reinterpret_cast<uint4 *>(vbase + slot * HD)[c] = vv;
        }
        if (p < g) {
            const size_t slot = static_cast<size_t>(w) + p;
            reinterpret_cast<uint4 *>(kbase + slot * HD)[c] = kv;
            reinterpret_cast<uint4 *>(vbase + slot * HD)[c] = vv;
        }
    }
}

template <typename T, int HD>
int launch_append_t(void *Kc, void *Vc, const void *kn, const void *vn, const int32_t *pos0,
                    int T_new, int B, int Hkv, int w, int g, cudaStream_t stream)
{
    constexpr int C = HD * static_cast<int>(sizeof(T)) / 16;
    const size_t total = static_cast<size_t>(B) * Hkv * T_new * C;
    const int threads = 256;
    size_t blocks = (total + threads - 1) / threads;
    const size_t cap = static_cast<size_t>(num_sms()) * 16;
    if (blocks > cap) blocks = cap;
    if (blocks == 0) return SWA_OK;
    swa_cache_append_k<T, HD><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
        static_cast<T *>(Kc), static_cast<T *>(Vc), static_cast<const T *>(kn),
        static_cast<const T *>(vn), pos0, T_new, B, Hkv, w, g, status_ptr());
    return cudaGetLastError() == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
}

}  // namespace

int choose_decode_splits(int B, int Hkv, int w, int g)
{
    if (const char *e = std::getenv("SWA_FORCE_SPLITS")) {
        const int s = std::atoi(e);
        if (s >= 1 && s <= 1024) return s;
    }
    // enough CTAs for several waves of resident CTAs, but chunks of at least
    // 256 keys so the split bookkeeping stays small next to the key stream
    const long long slots = static_cast<long long>(w) + g;
    const long long ctas_wanted = 8LL * num_sms();
    long long s = (ctas_wanted + static_cast<long long>(B) * Hkv - 1) / (static_cast<long long>(B) * Hkv);
    const long long max_s = (slots + 255) / 256;
    if (s > max_s) s = max_s;
    if (s < 1) s = 1;
    if (s > 1024) s = 1024;
    return static_cast<int>(s);
}

size_t decode_workspace_bytes(int B, int H, int d, int splits)
{
    if (splits <= 1) return 0;
    return static_cast<size_t>(B) * H * splits * (d + 2) * sizeof(float);
}

int launch_decode(const void *q, const void *Kc, const void *Vc, const int32_t *pos, int B, int H,
                  int Hkv, int d, int w, int g, float scale, void *O, float *lse, swa_dtype dt,
                  int splits, void *ws, cudaStream_t stream)
{
    DecodeParams p;
    p.B = B;
    p.H = H;
    p.Hkv = Hkv;
    p.w = w;
    p.g = g;
    p.S = splits;
    p.sl2 = scale * 1.4426950408889634f;
    p.pos = pos;
    p.status = status_ptr();
    if (p.status == nullptr) return SWA_ERR_CUDA;
    p.ws = static_cast<float *>(ws);
    p.O = O;
    p.lse = lse;
    const int G = H / Hkv;
    if (dt == SWA_BF16) {
        if (d == 128) return dispatch_g<__nv_bfloat16, 128>(q, Kc, Vc, p, G, stream);
        if (d == 64) return dispatch_g<__nv_bfloat16, 64>(q, Kc, Vc, p, G, stream);
    } else {
        if (d == 128) return dispatch_g<float, 128>(q, Kc, Vc, p, G, stream);
        if (d == 64) return dispatch_g<float, 64>(q, Kc, Vc, p, G, stream);
    }
    return SWA_ERR_UNSUPPORTED;
}

int launch_cache_append(void *Kc, void *Vc, const void *kn, const void *vn, const int32_t *pos0,
                        int T, int B, int Hkv, int d, int w, int g, swa_dtype dt,
                        cudaStream_t stream)
{
    if (dt == SWA_BF16) {
        if (d == 128) return launch_append_t<__nv_bfloat16, 128>(Kc, Vc, kn, vn, pos0, T, B, Hkv, w, g, stream);
        if (d == 64) return launch_append_t<__nv_bfloat16, 64>(Kc, Vc, kn, vn, pos0, T, B, Hkv, w, g, stream);
    } else {
        if (d == 128) return launch_append_t<float, 128>(Kc, Vc, kn, vn, pos0, T, B, Hkv, w, g, stream);
        if (d == 64) return launch_append_t<float, 64>(Kc, Vc, kn, vn, pos0, T, B, Hkv, w, g, stream);
    }
    return SWA_ERR_UNSUPPORTED;
}

}  // namespace swa
