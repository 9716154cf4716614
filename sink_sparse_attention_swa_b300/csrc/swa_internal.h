// swa_internal.h -- declarations shared by the translation units of libswa.
// Not part of the public ABI (that is include/swa.h).
#pragma once

#include <atomic>
#include <cmath>
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "swa.h"

namespace swa {

// ---------------------------------------------------------------------------
// Block-sparse tile enumeration for prefill ("Sliding Window and Sparse
// Attention, from Longformer to CSA2", section 1 last paragraph and section 4
// "Block-sparse attention": skip whole key tiles that miss the band).
//
// For query tile qt (rows q0 .. q1, q1 the last row that exists) the key
// tiles with at least one allowed pair are
//   band tiles  kt_lo .. kt_hi, kt_lo = max(0, q0-w+1)/BN, kt_hi = q1/BN
//   sink tiles  0 .. (min(g, q1+1)-1)/BN   (when g > 0)
// visited as: the sink tiles below kt_lo first, then the band tiles, so a
// tile in both sets is visited once.  A tile is full (no element mask) when
// every key is causal for every row (k1 <= q0) and every key not below g is
// inside every row's window (max(k0, g) > k1 or max(k0, g) >= q1-w+1).
// Used by the kernels and by the host helper swa_enumerate_tiles; the tests
// compare the latter with the oracle's brute force.
// ---------------------------------------------------------------------------
struct TileRange {
    int q0, q1;   // first and last existing query row of the tile
    int nl;       // landmark key tiles (visited first: lt0 .. lt0+nl-1), see add_landmarks
    int lt0;
    int ns;       // number of sink-only key tiles (visited next: 0 .. ns-1)
    int kt_lo;    // first band key tile
    int count;    // total key tiles visited (nl + ns + band tiles)
};

// The key tiles for query rows q0 .. q1 (indices into the key list; any
// alignment).
__host__ __device__ inline TileRange tile_range_at(int q0, int q1, int w, int g, int BN)
{
    TileRange r;
    r.q0 = q0;
    r.q1 = q1;
    r.nl = 0;
    r.lt0 = 0;
    int lo = r.q0 - w + 1;
    if (lo < 0) lo = 0;
    r.kt_lo = lo / BN;
    const int kt_hi = r.q1 / BN;
    int ns = 0;
    if (g > 0) {
        const int last_sink = (g < r.q1 + 1 ? g : r.q1 + 1) - 1;
        const int s_hi = last_sink / BN;
        ns = (s_hi + 1 < r.kt_lo) ? s_hi + 1 : r.kt_lo;
    }
    r.ns = ns;
    r.count = ns + (kt_hi - r.kt_lo + 1);
    return r;
}

__host__ __device__ inline TileRange tile_range(int qt, int n, int w, int g, int BM, int BN)
{
    const int q0 = qt * BM;
    return tile_range_at(q0, (q0 + BM < n ? q0 + BM : n) - 1, w, g, BN);
}

// ---------------------------------------------------------------------------
// Chunked prefill ("Sliding Window and Sparse Attention, from Longformer to
// CSA2", section 2: the rolling buffer; section 1: prefill vs decode).  A
// chunk of T new tokens at positions pos0 .. pos0+T-1 attends to the rolling
// cache and to itself.  Its keys are laid out as one list:
//   indices 0 .. S-1        positions 0 .. S-1 (the sinks, S = min(g, pos0)),
//   indices S .. S+pad-1    padding (zero rows no query reads),
//   indices S+pad ..        positions W0 .. pos0+T-1 (window part of the
//                           cache, then the chunk), W0 = max(S, pos0-w+1).
// Positions S .. W0-1 are left out: no query of the chunk reads them.  Index
// differences equal position differences after the sinks, and the sinks are
// the first g indices (or all positions, when pos0 < g), so the prefill mask
// (j <= i, j >= i-w+1 or j < g) holds on list indices with query t at index
// t + chunk_offset.  The padding only exists once the window has moved past
// the sinks (S = g and W0 = pos0-w+1 > g-1): then every padding index is
// >= g and below the band of the chunk's first query, and pad makes
// chunk_offset a multiple of the 128-row query tile, so the chunk's query
// tiles meet the key tiles as aligned as in a plain prefill.
// ---------------------------------------------------------------------------
constexpr int CHUNK_ALIGN = 128;
__host__ __device__ inline int chunk_sinks(int pos0, int g) { return pos0 < g ? pos0 : g; }
__host__ __device__ inline int chunk_w0(int pos0, int w, int g)
{
    const int s = chunk_sinks(pos0, g), a = pos0 - w + 1;
    return s > a ? s : a;
}
__host__ __device__ inline int chunk_pad(int pos0, int w, int g)
{
    if (pos0 < g || pos0 - w + 1 < g) return 0;
    const int r = (g + w - 1) % CHUNK_ALIGN;
    return r == 0 ? 0 : CHUNK_ALIGN - r;
}
__host__ __device__ inline int chunk_offset(int pos0, int w, int g)
{
    return pos0 + chunk_sinks(pos0, g) + chunk_pad(pos0, w, g) - chunk_w0(pos0, w, g);
}
// rows of the key list for a chunk of T tokens at pos0
__host__ __device__ inline int chunk_keys(int pos0, int w, int g, int T)
{
    return chunk_offset(pos0, w, g) + T;
}
// the largest key list over all pos0, rounded up to whole 128-row tiles
// (chunk_offset <= roundup(g + w - 1, 128))
__host__ __device__ inline long long chunk_rows_max(int w, int g, int T)
{
    const long long a = CHUNK_ALIGN;
    return (static_cast<long long>(g) + w - 1 + a - 1) / a * a + (static_cast<long long>(T) + a - 1) / a * a;
}

// ---------------------------------------------------------------------------
// Landmarks ("Local and Sparse Attention: Reading Fewer Token Positions",
// Figure 2, right): besides the band and the sinks, a query i reads every
// position j = rl * m <= i.  A landmark inside the band is read there, one
// below g as a sink, so the landmark tiles carry only the rest:
//     g <= rl * m <= i - w,  i.e.  land_lo <= m <= land_hi(i),
// with m the index into the landmark list (positions 0, rl, 2 rl, ...), which
// the kernels load as dense 128-row tiles through a view of K and V whose row
// stride is rl rows.  Landmark tiles are visited before the sink and band
// tiles.
// ---------------------------------------------------------------------------
__host__ __device__ inline int land_lo(int g, int rl) { return (g + rl - 1) / rl; }
__host__ __device__ inline int land_hi(int i, int w, int rl) { return i >= w ? (i - w) / rl : -1; }
__host__ __device__ inline void add_landmarks(TileRange &r, int w, int g, int rl, int BN)
{
    if (rl <= 0) return;
    const int a = land_lo(g, rl), z = land_hi(r.q1, w, rl);
    if (z < a) return;
    r.lt0 = a / BN;
    r.nl = z / BN - r.lt0 + 1;
    r.count += r.nl;
}
// every landmark of tile lt is read by every row of the tile
__host__ __device__ inline bool land_full(const TileRange &r, int lt, int w, int g, int rl, int BN)
{
    return lt * BN >= land_lo(g, rl) && lt * BN + BN - 1 <= land_hi(r.q0, w, rl);
}

__host__ __device__ inline int tile_kt(const TileRange &r, int j)
{
    return j < r.ns ? j : r.kt_lo + (j - r.ns);
}

__host__ __device__ inline bool tile_full(const TileRange &r, int kt, int w, int g, int BN)
{
    const int k0 = kt * BN, k1 = k0 + BN - 1;
    if (k1 > r.q0) return false;
    const int a = k0 > g ? k0 : g;
    return a > k1 || a >= r.q1 - w + 1;
}

// ---------------------------------------------------------------------------
// Final normalisation of a row's online softmax kept in base 2: m is the
// reference maximum (scores times scale*log2(e)) and l the sum of
// exp2(score - m).  An optional learned sink logit of the row's head
// ("Sliding Window and Sparse Attention, from Longformer to CSA2", section 6,
// stage 3: a per-head logit that absorbs mass, i.e. one more softmax entry
// with a zero value) joins the normalising sum: sink [H] in natural-log
// units, or null.  Returns the factor the unnormalised output is multiplied
// by and sets *lse (natural log).  Without a sink this is 1/l and m + log2 l.
// ---------------------------------------------------------------------------
#ifdef __CUDACC__
__device__ __forceinline__ float finish_row(float m, float l, const float *sink, int h, float *lse)
{
    const float sig = (sink != nullptr) ? sink[h] * 1.4426950408889634f : -INFINITY;
    const float M = fmaxf(m, sig);
    if (M == -INFINITY) {
        *lse = -INFINITY;
        return 0.f;
    }
    const float a = exp2f(m - M);
    const float L = l * a + exp2f(sig - M);
    *lse = (M + log2f(L)) * 0.69314718055994530942f;
    return L > 0.f ? a / L : 0.f;
}
#endif

// ---------------------------------------------------------------------------
// Device status word (one per device, in swa_status.cu).  Kernels OR an error
// code into it when a bounded wait runs out.
// ---------------------------------------------------------------------------
enum : int { DEV_ERR_TIMEOUT = 1, DEV_ERR_BAD_POS = 2, DEV_ERR_BOUNDS = 4 };

// Bounds checks of the debug build (compiled with SWA_DEBUG): SWA_BOUNDS(cond,
// status) is cond, and when cond is false it also records DEV_ERR_BOUNDS in
// the device status word; the caller skips the access it guards.  In the
// product build it is the constant true and its arguments are not compiled.
#ifdef SWA_DEBUG
#define SWA_BOUNDS(cond, status) ((cond) || (atomicOr((status), DEV_ERR_BOUNDS), false))
#else
#define SWA_BOUNDS(cond, status) true
#endif
// the injection of swa_debug_shrink_bounds (an internal kind of the one-shot
// launch settings below)
constexpr int INJECT_SHRINK_BOUNDS = 3;

int *status_ptr();          // device address of the current device's status word
int read_and_clear_status(cudaStream_t stream);

// A stall injected by swa_debug_inject_stall for the next launch of one kind
// on the current device: returns true (once) and sets *wait_ns to the wait
// limit that launch must use; false (and *wait_ns untouched) otherwise.
bool take_injected_stall(int kind, uint64_t *wait_ns);
int set_injected_stall(int kind, int64_t wait_ns);

// ---------------------------------------------------------------------------
// Opt-in to more than 48 KB of dynamic shared memory for one kernel.  The
// attribute belongs to the current device, so it is set once per (kernel,
// device): a process that calls the library on several GPUs sets it on each.
// ---------------------------------------------------------------------------
constexpr int kMaxDevices = 64;
int current_device();  // the current device, or -1 if none (or beyond kMaxDevices)
#ifdef __CUDACC__
template <auto Kernel>
cudaError_t smem_opt_in(int bytes)
{
    static std::atomic<int> done[kMaxDevices];  // static storage: starts at zero
    const int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    if (done[dev].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
    const cudaError_t e =
        cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done[dev].store(bytes, std::memory_order_release);
    return e;
}
#endif

// ---------------------------------------------------------------------------
// Launchers (each validates nothing: the public entry points do that).
// ---------------------------------------------------------------------------
// sink: per-head sink logits [H] (device, fp32) or null, for every launcher.
// n: query rows (Q, O); n_k: key rows (K, V); pos0: device int32 [B] for a
// chunked prefill over key lists (query t at index t + chunk_offset(pos0[b])),
// or null for a plain prefill (n_k == n, query i at index i).
// R, rl: the fixed pattern (R = 1, rl = 0 for the window and sinks).
//   R > 1   residue classes: query i and key j meet only when i = j (mod R),
//           and each class c (positions c, c+R, c+2R, ...) is a window
//           prefill of its own over that subsequence (the dilated pattern;
//           the strided one is the same with w >= ceil(n/R)); needs n_k == n,
//           pos0 == null, g == 0.
//   rl > 0  landmarks every rl positions (add_landmarks); needs R == 1 and
//           pos0 == null.
// walk: a diagnostic log of the key tiles the kernels load (the layout of
// swa_debug_prefill_walk, its capacity in its header), or null for a plain
// launch.  cta_pairs: run the window path on the CTA-pair kernel
// (swa_debug_prefill_cta_pairs; SWA_ERR_UNSUPPORTED where it does not apply).
int launch_prefill_bf16(const void *Q, const void *K, const void *V, void *O, float *lse,
                        const float *sink, int B, int H, int Hkv, int n, int n_k, int d, int w,
                        int g, float scale, const int32_t *pos0, int R, int rl,
                        cudaStream_t stream, int32_t *walk = nullptr, bool cta_pairs = false);
int launch_prefill_f32(const void *Q, const void *K, const void *V, void *O, float *lse,
                       const float *sink, int B, int H, int Hkv, int n, int n_k, int d, int w,
                       int g, float scale, const int32_t *pos0, int R, int rl,
                       cudaStream_t stream);
// Builds the key lists of a chunked prefill: Kx, Vx [B][Hkv][rows][d] from
// the rolling cache and the chunk; rows = chunk_rows_max(w, g, T).
int launch_chunk_gather(void *Kx, void *Vx, const void *Kc, const void *Vc, const void *k_new,
                        const void *v_new, const int32_t *pos0, int B, int Hkv, int T, int d,
                        int w, int g, swa_dtype dt, cudaStream_t stream);
// Decode of any GQA group size G: the G query heads of a kv head are split
// into nsub = ceil(G / 8) sub-groups of Gs = ceil(G / nsub) heads, each padded
// to Gp (the next of 1, 2, 4, 8, the group widths the decode kernels are built
// for) with dummy heads whose results are never written.  A sub-group is a
// "virtual kv head": Hv = Hkv * nsub of them, sub-group u of kv head k being
// virtual head k * nsub + u, which reads kv head k's cache and query heads
// k * G + u * Gs + (0 .. Gs-1).
struct DecodeGroups {
    int nsub, Gs, Gp;
};
__host__ __device__ inline DecodeGroups decode_groups(int G)
{
    DecodeGroups r;
    r.nsub = (G + 7) / 8;
    r.Gs = (G + r.nsub - 1) / r.nsub;
    r.Gp = 1;
    while (r.Gp < r.Gs) r.Gp <<= 1;
    return r;
}
// CTAs of the decode split pass: num_splits > 0 asks for about that many per
// (sequence, virtual kv head); 0 picks one resident wave on the current device.
int decode_ctas(int B, int H, int Hkv, int w, int g, int num_splits);
size_t decode_workspace_bytes(int B, int H, int Hkv, int d, int ctas);
int launch_decode(const void *q, const void *Kc, const void *Vc, const int32_t *pos,
                  const float *sink, int B,
                  int H, int Hkv, int d, int w, int g, float scale, void *O, float *lse,
                  swa_dtype dt, int ctas, void *ws, cudaStream_t stream);
int launch_cache_append(void *Kc, void *Vc, const void *kn, const void *vn, const int32_t *pos0,
                        int T, int B, int Hkv, int d, int w, int g, swa_dtype dt,
                        cudaStream_t stream);
int launch_selftest_umma(const void *A, const void *Bk, const void *Bn, float *D1, float *D2,
                         cudaStream_t stream);

int num_sms();

}  // namespace swa
