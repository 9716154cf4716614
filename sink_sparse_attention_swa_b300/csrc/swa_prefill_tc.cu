// swa_prefill_tc.cu -- bf16 block-sparse sliding-window (+ sinks) prefill on
// the sm_103a tensor cores.
//
// What it computes ("Sliding Window and Sparse Attention, from Longformer to
// CSA2", sections 1-2; "Local and Sparse Attention: Reading Fewer Token
// Positions", Figures 1-2): O = softmax(scale * Q K^T + mask) V per head, the
// mask -inf outside {i-w+1 .. i} u {0 .. g-1} n {j <= i}.  Exact: the
// FlashAttention-style tiling and online softmax change the order of the
// arithmetic, not the result ("Sparse Attention ..." social post, section 2;
// the walkthrough's section 1 last paragraph).
//
// Design (B300-native; the pages give no kernel):
//  * Two kernels: the pair kernel (below; two query heads of a GQA group per
//    work item for even groups, two adjacent q tiles of one head for odd
//    groups) and the single-head kernel described here (odd groups under the
//    fixed patterns).
//  * Persistent CTAs, one per SM.  A work item is (b, kv head, q tile of 128
//    rows, query head or head pair, residue class for the fixed patterns);
//    items are ranked q tile first (decode_level_item), so the CTAs running at
//    the same time share one band position of every kv head in L2.
//  * Only key tiles (128 keys) that meet the band or the sink columns are
//    visited (tile_range); the element mask is applied only on partial tiles.
//  * Warp roles of the single-head kernel (192 threads):
//      warp 0  TMA producer: Q tile (double-buffered), K and V tiles into a
//              2-stage ring, 128-byte swizzled boxes of 64 columns.
//      warp 1  MMA issuer: S = Q K^T (both operands from shared memory) into
//              one of two TMEM S buffers; O += P V with P read from TMEM and V
//              N-major from shared memory.  tcgen05.commit signals mbarriers.
//      warps 2-5  softmax: one query row per thread (its TMEM lane), fp32
//              online softmax in base 2 with the scale folded in, lazy O
//              rescaling (only when a row max grows by more than 2^8), P to
//              TMEM as bf16, then the epilogue O / l -> bf16 and the LSE.
//  * TMEM (512 columns): O [0, d), S0 [128, 256), S1 [256, 384),
//    P0 [384, 448), P1 [448, 512).
//  * Every mbarrier wait is bounded (mbar_wait): on a timeout the CTA marks
//    the device status word, all roles stop, in-flight TMA loads and MMAs are
//    drained with bounded waits, and TMEM is freed before exit.
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <type_traits>

#include "swa_internal.h"
#include "swa_ptx.cuh"

namespace swa {
namespace {

using namespace ptx;

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int STAGES = 2;
constexpr int NTHREADS = 192;
constexpr uint64_t TIMEOUT_NS = 2000000000ull;  // 2 s: far beyond any legitimate wait
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t S_COL0 = 128;
constexpr uint32_t P_COL0 = 384;
constexpr float RESCALE_LOG2 = 8.0f;

// Compile-time loop: f(integral_constant<int, I>) for I = B .. E-1.
template <int B, int E, class F>
__device__ __forceinline__ void static_for(F &&f)
{
    if constexpr (B < E) {
        f(std::integral_constant<int, B>{});
        static_for<B + 1, E>(f);
    }
}

// One S column (index C, an immediate) set to -inf as a predicated select:
// past cb; before ca; or outside "C <= cb and (C >= ca or C < cg)".
template <int C>
__device__ __forceinline__ void mask_after(uint32_t &v, int cb)
{
    asm("{\n\t.reg .pred p;\n\tsetp.lt.s32 p, %1, %2;\n\tselp.b32 %0, 0xFF800000, %0, p;\n\t}"
        : "+r"(v)
        : "r"(cb), "n"(C));
}
template <int C>
__device__ __forceinline__ void mask_before(uint32_t &v, int ca)
{
    asm("{\n\t.reg .pred p;\n\tsetp.gt.s32 p, %1, %2;\n\tselp.b32 %0, 0xFF800000, %0, p;\n\t}"
        : "+r"(v)
        : "r"(ca), "n"(C));
}
template <int C>
__device__ __forceinline__ void mask_general(uint32_t &v, int ca, int cb, int cg)
{
    asm("{\n\t.reg .pred a, b;\n\t"
        "setp.le.s32 b, %3, %4;\n\t"        // C >= cg: not a sink column
        "setp.gt.and.s32 b, %1, %4, b;\n\t"  // and C < ca: before the band
        "setp.lt.or.s32 a, %2, %4, b;\n\t"   // or C > cb: past the diagonal
        "selp.b32 %0, 0xFF800000, %0, a;\n\t}"
        : "+r"(v)
        : "r"(ca), "r"(cb), "r"(cg), "n"(C));
}

// The mask of a partial tile on one row of S (s[4][32], column c = 32 q + e):
// a key is allowed iff c <= cb and (c >= ca or c < cg).  Nearly always one
// bound alone decides (the diagonal tile: c <= cb; the tile where the band
// starts: c >= ca), and those rows test one bound per column.  Every column is
// a predicated select, never a branch: written as a per-column `if`, tiles
// where both rules apply measured up to seven times a full tile's softmax.
__device__ __forceinline__ void mask_cols(uint32_t (&s)[4][32], int ca, int cb, int cg)
{
    if (cg >= ca || ca <= 0) {
        // the sinks (if any) reach the band, or the band covers c >= 0
        static_for<0, BN>([&](auto ic) {
            constexpr int c = decltype(ic)::value;
            mask_after<c>(s[c / 32][c % 32], cb);
        });
    } else if (cb >= BN - 1 && cg <= 0) {
        static_for<0, BN>([&](auto ic) {
            constexpr int c = decltype(ic)::value;
            mask_before<c>(s[c / 32][c % 32], ca);
        });
    } else {
        static_for<0, BN>([&](auto ic) {
            constexpr int c = decltype(ic)::value;
            mask_general<c>(s[c / 32][c % 32], ca, cb, cg);
        });
    }
}

// Tensor-memory columns are compile-time offsets from the allocated base.
// One-head kernel: O in [0, HD), two S buffers from S_COL0, two P halves from
// P_COL0.  Head-pair kernels: O_X at 256x, S_X / P_X at 256x + 128.
static_assert(S_COL0 >= 128 && P_COL0 >= S_COL0 + 2 * BN && P_COL0 + 2 * (BN / 2) <= TMEM_COLS,
              "one-head kernel's tensor-memory columns");
static_assert(256 + 128 + BN <= TMEM_COLS, "head-pair kernels' tensor-memory columns");

#ifdef SWA_DEBUG
// Debug builds: the base the allocator returned is lane 0, with every
// allocated column after it inside the SM's 512.  A kernel whose base fails
// skips its work and goes straight to its teardown.
__device__ __forceinline__ bool tmem_base_ok(uint32_t tmem, int *status)
{
    return SWA_BOUNDS((tmem >> 16) == 0u && (tmem & 0xFFFFu) + TMEM_COLS <= 512u, status);
}
#endif

// Epilogue staging: each softmax warp turns its 32 rows x 32 columns of the
// output (64 bytes of bf16 per row) around in shared memory so that its global
// stores cover whole 64-byte row segments, 8 rows per instruction, instead of
// 16 bytes of 32 different rows.  Rows are padded to 80 bytes, so the 16-byte
// accesses of 8 lanes in a row fall in distinct banks.
constexpr uint32_t STAGE_ROW = 80;
constexpr uint32_t STAGE_WARP = 32 * STAGE_ROW;

template <int HD>
struct Layout {
    static constexpr uint32_t QB = BM * HD * 2;    // one Q tile
    static constexpr uint32_t KB = BN * HD * 2;    // one K (or V) tile
    static constexpr uint32_t Q_OFF = 0;           // 2 Q buffers
    static constexpr uint32_t K_OFF = Q_OFF + 2 * QB;
    static constexpr uint32_t V_OFF = K_OFF + STAGES * KB;
    static constexpr uint32_t BAR_OFF = V_OFF + STAGES * KB;
    enum {
        Q_FULL = 0,
        Q_EMPTY = 2,
        K_FULL = 4,
        V_FULL = K_FULL + STAGES,
        KV_EMPTY = V_FULL + STAGES,
        S_FULL = KV_EMPTY + STAGES,
        S_EMPTY = S_FULL + 2,
        P_FULL = S_EMPTY + 2,
        PV_DONE = P_FULL + 2,
        O_EMPTY = PV_DONE + 2,
        DRAIN = O_EMPTY + 1,
        NBAR = DRAIN + 1
    };
    static constexpr uint32_t MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr uint32_t STAGE_OFF = (MISC_OFF + 16 + 15) & ~15u;  // 4 softmax warps
    static constexpr uint32_t BYTES = STAGE_OFF + 4 * STAGE_WARP;
    // > half of the SM's shared memory, so that exactly one CTA (and one
    // 512-column TMEM allocation) lives on an SM.
    static constexpr uint32_t DYN_SMEM = (BYTES + 1024 > 120 * 1024) ? BYTES + 1024 : 120 * 1024;
};

struct PrefillParams {
    int B, H, Hkv, n, w, g, G, n_qt, num_items;
    int n_k;                 // key rows (K, V); n is the query rows (Q, O)
    const int32_t *pos0;     // chunked prefill: chunk start per sequence, or null
    // residue classes (dilated and strided patterns; R = 1 otherwise): class c
    // holds n_hi rows if c < rem, else n_lo; the last q-tile level holds
    // R_top classes (those with a row in it)
    int R, rem, n_hi, n_lo, R_top;
    int rl;                  // landmark stride, 0 for none
    float sl2;  // scale * log2(e)
    __nv_bfloat16 *O;
    float *lse;
    const float *sink;  // per-head sink logits [H] or null
    int *status;
    uint64_t wait_ns;   // limit of every bounded wait of the roles (2 s unless a test sets it)
    int skip_first_kv;  // test injection: the first key/value copy is left out (see swa.h)
#ifdef SWA_DEBUG
    long long dbg_orows;  // output rows the bounds checks allow (B*H*n; one fewer when shrunk)
#endif
};

// One entry of the tile-walk log per key tile a producer issues: the item's
// rank, sequence, kv head, unit (head pair, head, or q-tile pair), q tile,
// residue class, the tile's first key index, and flags (1 full, 2 landmark
// tile).  log[0] counts the entries, log[2..3] holds the
// capacity (a 64-bit count of entries); entry e is at log[WALK_HDR +
// WALK_ENTRY * e].  The log is a kernel argument of its own, kept out of
// PrefillParams (a larger parameter block made the control warpgroup spill),
// and the producers write it only in the WALK instantiations that
// swa_debug_prefill_walk launches: a per-tile check for a null log cost the
// product kernels up to 2% on short items.
constexpr int WALK_HDR = 8, WALK_ENTRY = 8;
__device__ __forceinline__ void log_walk(int32_t *log, int t, int b, int kvh, int u, int qt, int cls,
                                         int k0, int flags)
{
    const long long e = atomicAdd(log, 1);
    if (e >= *reinterpret_cast<const long long *>(log + 2)) return;
    int32_t *w = log + WALK_HDR + WALK_ENTRY * e;
    w[0] = t;
    w[1] = b;
    w[2] = kvh;
    w[3] = u;
    w[4] = qt;
    w[5] = cls;
    w[6] = k0;
    w[7] = flags;
}

// Work order of both kernels.  Items are ranked by q tile, the last q tile
// (the most key tiles) first; within a q tile by unit (query head, or head
// pair), residue class, kv head and sequence, the unit fastest, so the CTAs
// working at the same time share one band position of every kv head (a few
// MB of K/V in L2) and, with residue classes, neighbouring rows of it.  Only
// the last level can hold fewer classes (R_top): a class whose subsequence is
// one row shorter may end a tile earlier.  No item is empty.
template <bool PAT>
__device__ __forceinline__ void decode_level_item(int r, const PrefillParams &p, int U, int &b,
                                                  int &u, int &kvh, int &qt, int &cls)
{
    const int per_c = p.B * p.Hkv * U;
    if constexpr (!PAT) {  // one class: levels of per_c items
        qt = p.n_qt - 1 - r / per_c;
        r %= per_c;
        u = r % U;
        r /= U;
        cls = 0;
        kvh = r % p.Hkv;
        b = r / p.Hkv;
        return;
    }
    const int top = p.R_top * per_c;
    int Rl = p.R_top;
    if (r < top) {
        qt = p.n_qt - 1;
    } else {
        r -= top;
        const int per_qt = p.R * per_c;
        qt = p.n_qt - 2 - r / per_qt;
        r %= per_qt;
        Rl = p.R;
    }
    u = r % U;
    r /= U;
    cls = r % Rl;
    r /= Rl;
    kvh = r % p.Hkv;
    b = r / p.Hkv;
}

// Key tiles of query tile qt of sequence b (residue class cls), in key-list
// indices; *off is the list index of query row 0 (0 for a plain prefill,
// chunk_offset(pos0[b]) for a chunked one).  With residue classes, rows and
// keys are indices into the class's subsequence.
// QP: the item is a pair of q tiles of one head (the pair kernel on an odd
// group; n_qt then counts pairs of q tiles)
template <bool PAT, bool QP = false>
__device__ __forceinline__ TileRange item_tiles(const PrefillParams &p, int b, int qt, int cls,
                                                int &off)
{
    off = 0;
    if (p.pos0 != nullptr) {
        const int ps = __ldg(p.pos0 + b);
        off = chunk_offset(ps < 0 ? 0 : ps, p.w, p.g);
    }
    const int nq = !PAT ? p.n : cls < p.rem ? p.n_hi : p.n_lo;
    // with q-tile pairs the walk covers the key tiles of both q tiles
    const int rows = QP ? 2 * BM : BM;
    const int q0 = qt * rows, q1 = (q0 + rows < nq ? q0 + rows : nq) - 1;
    TileRange tr = tile_range_at(q0 + off, q1 + off, p.w, p.g, BN);
    if constexpr (PAT) add_landmarks(tr, p.w, p.g, p.rl, BN);
    return tr;
}

// Key-tile j of an item: its first row in the key source, which view to load
// it from (landmark tiles: the stride-rl view at class 0), and the element
// mask a row i applies to it: key index k allowed iff k <= hi and (k >= lo or
// k < gs), hi/lo/gs per tile kind.
struct KeyTile {
    int k0;
    bool land;
    bool full;
};
template <bool PAT>
__device__ __forceinline__ KeyTile key_tile(const TileRange &tr, int j, const PrefillParams &p)
{
    KeyTile kt;
    kt.land = PAT && j < tr.nl;
    if (kt.land) {
        const int lt = tr.lt0 + j;
        kt.k0 = lt * BN;
        kt.full = land_full(tr, lt, p.w, p.g, p.rl, BN);
    } else {
        const int t = tile_kt(tr, PAT ? j - tr.nl : j);
        kt.k0 = t * BN;
        kt.full = tile_full(tr, t, p.w, p.g, BN);
    }
    return kt;
}

// Debug builds: the key tile's first key lies in the key list it is read
// from (the keys, the landmark list, or the residue class's subsequence).
template <bool PAT>
__device__ __forceinline__ bool key_tile_in_range(const KeyTile &kt, int cls, const PrefillParams &p)
{
    if constexpr (!PAT) return kt.k0 >= 0 && kt.k0 < p.n_k;
    const int lim = kt.land ? (p.n_k + p.rl - 1) / p.rl : (cls < p.rem ? p.n_hi : p.n_lo);
    return kt.k0 >= 0 && kt.k0 < lim;
}
#define SWA_ITEM_IN_RANGE(p, b, kvh, qt, cls) \
    ((b) >= 0 && (b) < (p).B && (kvh) >= 0 && (kvh) < (p).Hkv && (qt) >= 0 && (qt) < (p).n_qt && \
     (cls) >= 0 && (cls) < (p).R)

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// All 32 lanes wait; the outcome is made warp-uniform.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          int *status, uint64_t limit_ns)
{
    const bool ok = mbar_wait(bar, parity, abort, status, limit_ns);
    return __all_sync(0xffffffffu, ok);
}

// Epilogue of one warp: the 32 query rows of its TMEM lane quarter (one per
// lane), O[:, 0:HD) at o_addr, times inv_l, rounded to bf16 and stored to
// orow (this lane's output row; row_ok false for rows past the end) through
// the warp's staging area `stage` (STAGE_WARP bytes of shared memory).
template <int HD>
__device__ __forceinline__ void store_o_rows(uint32_t o_addr, float inv_l,
                                             __nv_bfloat16 *orow, bool row_ok, uint8_t *stage,
                                             int lane)
{
    // the row each lane writes back in step s: 8 rows per step, 4 lanes a row
    const int sub = lane & 3;
    uint64_t dst[4];
    bool dok[4];
#pragma unroll
    for (int st = 0; st < 4; ++st) {
        const int src = st * 8 + (lane >> 2);
        dst[st] = __shfl_sync(0xffffffffu, reinterpret_cast<uint64_t>(orow), src);
        dok[st] = __shfl_sync(0xffffffffu, row_ok ? 1 : 0, src) != 0;
    }
    uint4 *mine = reinterpret_cast<uint4 *>(stage + lane * STAGE_ROW);
    // all of the row's O columns in one round of tensor-memory loads
    uint32_t o[HD / 32][32];
#pragma unroll
    for (int q = 0; q < HD / 32; ++q) tmem_ld32(o_addr + q * 32, o[q]);
    tmem_ld_wait();
#pragma unroll
    for (int q = 0; q < HD / 32; ++q) reg_fence32(o[q]);
#pragma unroll
    for (int q = 0; q < HD / 32; ++q) {
#pragma unroll
        for (int v = 0; v < 4; ++v)
            mine[v] = make_uint4(pack_bf16x2(__uint_as_float(o[q][8 * v]) * inv_l,
                                             __uint_as_float(o[q][8 * v + 1]) * inv_l),
                                 pack_bf16x2(__uint_as_float(o[q][8 * v + 2]) * inv_l,
                                             __uint_as_float(o[q][8 * v + 3]) * inv_l),
                                 pack_bf16x2(__uint_as_float(o[q][8 * v + 4]) * inv_l,
                                             __uint_as_float(o[q][8 * v + 5]) * inv_l),
                                 pack_bf16x2(__uint_as_float(o[q][8 * v + 6]) * inv_l,
                                             __uint_as_float(o[q][8 * v + 7]) * inv_l));
        __syncwarp();
#pragma unroll
        for (int st = 0; st < 4; ++st) {
            const uint4 val =
                *reinterpret_cast<const uint4 *>(stage + (st * 8 + (lane >> 2)) * STAGE_ROW + sub * 16);
            if (dok[st])
                reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(dst[st]) + q * 32)[sub] =
                    val;
        }
        __syncwarp();
    }
}

// The same epilogue in rounds of 32 columns, for a warp with few registers:
// each round loads 32 columns of O from tensor memory, scales and rounds them,
// turns them around in `stage` and stores them.  Once the last round's load
// has completed the warp arrives on `empty_bar` (the O columns may be
// overwritten), before that round's stores; with CLUSTER, `empty_bar` is a
// shared::cluster address (a barrier of either CTA of a pair).
template <int HD, bool CLUSTER = false>
__device__ __forceinline__ void store_o_rows_chunked(uint32_t o_addr, float inv_l,
                                                     __nv_bfloat16 *orow, bool row_ok,
                                                     uint8_t *stage, int lane, uint32_t empty_bar)
{
    const int sub = lane & 3;
    uint64_t dst[4];
    bool dok[4];
#pragma unroll
    for (int st = 0; st < 4; ++st) {
        const int src = st * 8 + (lane >> 2);
        dst[st] = __shfl_sync(0xffffffffu, reinterpret_cast<uint64_t>(orow), src);
        dok[st] = __shfl_sync(0xffffffffu, row_ok ? 1 : 0, src) != 0;
    }
    uint4 *mine = reinterpret_cast<uint4 *>(stage + lane * STAGE_ROW);
#pragma unroll 1
    for (int q = 0; q < HD / 32; ++q) {
        uint32_t o[32];
        tmem_ld32(o_addr + q * 32, o);
        tmem_ld_wait();
        reg_fence32(o);
        if (q == HD / 32 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (CLUSTER)
                    mbar_arrive_cluster(empty_bar);  // a shared::cluster address
                else
                    mbar_arrive(empty_bar);
            }
        }
#pragma unroll
        for (int v = 0; v < 4; ++v)
            mine[v] = make_uint4(pack_bf16x2(__uint_as_float(o[8 * v]) * inv_l,
                                             __uint_as_float(o[8 * v + 1]) * inv_l),
                                 pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv_l,
                                             __uint_as_float(o[8 * v + 3]) * inv_l),
                                 pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv_l,
                                             __uint_as_float(o[8 * v + 5]) * inv_l),
                                 pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv_l,
                                             __uint_as_float(o[8 * v + 7]) * inv_l));
        __syncwarp();
#pragma unroll
        for (int st = 0; st < 4; ++st) {
            const uint4 val =
                *reinterpret_cast<const uint4 *>(stage + (st * 8 + (lane >> 2)) * STAGE_ROW + sub * 16);
            if (dok[st])
                reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(dst[st]) + q * 32)[sub] =
                    val;
        }
        __syncwarp();
    }
}

// Units of the pair kernel per kv head: head pairs of an even group, or single
// heads whose two halves are two q tiles (odd groups); and the head of half x.
template <bool QP>
__device__ __forceinline__ int pair_units(const PrefillParams &p)
{
    return QP ? p.G : (p.G >> 1);
}
template <bool QP>
__device__ __forceinline__ int pair_head(const PrefillParams &p, int kvh, int u, int x)
{
    return QP ? kvh * p.G + u : kvh * p.G + 2 * u + x;
}

// One box of rows: with the fixed patterns through the 4-D views (class
// coordinate cls), otherwise through the plain 3-D maps.
template <bool PAT>
__device__ __forceinline__ void load_rows(uint32_t dst, const CUtensorMap *map, uint32_t bar, int x,
                                          int cls, int row, int z)
{
    if constexpr (PAT)
        tma_load_4d(dst, map, bar, x, cls, row, z);
    else
        tma_load_3d(dst, map, bar, x, row, z);
}

template <int HD, bool PAT, bool WALK>
__global__ void __launch_bounds__(NTHREADS, 1)
    swa_prefill_bf16_sm103(const __grid_constant__ CUtensorMap tmQ,
                           const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV,
                           const __grid_constant__ CUtensorMap tmQ2,
                           const __grid_constant__ CUtensorMap tmK2,
                           const __grid_constant__ CUtensorMap tmV2, const PrefillParams p,
                           int32_t *walk)
{
    using L = Layout<HD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(smem);
    const uint32_t sQ = sb + L::Q_OFF, sK = sb + L::K_OFF, sV = sb + L::V_OFF;
    const uint32_t bars = sb + L::BAR_OFF;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::MISC_OFF + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#define BAR(i) (bars + 8u * static_cast<uint32_t>(i))

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(BAR(L::Q_FULL + i), 1);
            mbar_init(BAR(L::Q_EMPTY + i), 1);
            mbar_init(BAR(L::S_FULL + i), 1);
            mbar_init(BAR(L::S_EMPTY + i), 4);
            mbar_init(BAR(L::P_FULL + i), 4);
            mbar_init(BAR(L::PV_DONE + i), 1);
        }
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(BAR(L::K_FULL + i), 1);
            mbar_init(BAR(L::V_FULL + i), 1);
            mbar_init(BAR(L::KV_EMPTY + i), 1);
        }
        mbar_init(BAR(L::O_EMPTY), 4);
        mbar_init(BAR(L::DRAIN), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch(&tmQ);
        tma_prefetch(&tmK);
        tma_prefetch(&tmV);
        tma_prefetch(&tmQ2);
        tma_prefetch(&tmK2);
        tma_prefetch(&tmV2);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
#ifdef SWA_DEBUG
    if (!tmem_base_ok(tmem, p.status)) goto teardown;
#endif

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int kv_iter = 0, it = 0;
            int last_k_par[STAGES], last_q_par[2];
            for (int s = 0; s < STAGES; ++s) last_k_par[s] = -1;
            last_q_par[0] = last_q_par[1] = -1;
            bool ok = true;
            auto load_q = [&](int item, int idx) -> bool {
                int b, hg, kvh, qt, cls;
                decode_level_item<PAT>(item, p, p.G, b, hg, kvh, qt, cls);
                const int h = kvh * p.G + hg;
                const int qb = idx & 1;
                if (!mbar_wait(BAR(L::Q_EMPTY + qb), ((idx >> 1) & 1) ^ 1, abort_flag, p.status,
                               p.wait_ns))
                    return false;
                mbar_expect_tx(BAR(L::Q_FULL + qb), L::QB);
                const CUtensorMap *mq = (!PAT || cls < p.rem) ? &tmQ : &tmQ2;
                for (int c = 0; c < HD / 64; ++c)
                    load_rows<PAT>(sQ + qb * L::QB + c * (BM * 128), mq, BAR(L::Q_FULL + qb),
                                   c * 64, cls, qt * BM, b * p.H + h);
                last_q_par[qb] = (idx >> 1) & 1;
                return true;
            };
            if (static_cast<int>(blockIdx.x) < p.num_items) ok = load_q(blockIdx.x, 0);
            for (int t = blockIdx.x; ok && t < p.num_items; t += gridDim.x, ++it) {
                int b, hg, kvh, qt, cls;
                decode_level_item<PAT>(t, p, p.G, b, hg, kvh, qt, cls);
                (void)SWA_BOUNDS(SWA_ITEM_IN_RANGE(p, b, kvh, qt, cls), p.status);
                int off;
                const TileRange tr = item_tiles<PAT>(p, b, qt, cls, off);
                for (int j = 0; j < tr.count; ++j, ++kv_iter) {
                    const int st = kv_iter % STAGES;
                    const uint32_t ph = (kv_iter / STAGES) & 1;
                    if (!mbar_wait(BAR(L::KV_EMPTY + st), ph ^ 1, abort_flag, p.status,
                                   p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    const KeyTile kt = key_tile<PAT>(tr, j, p);
                    (void)SWA_BOUNDS(key_tile_in_range<PAT>(kt, cls, p), p.status);
                    const int zkv = b * p.Hkv + kvh;
                    // landmark tiles: class 0 of the stride-rl view; others: this class
                    const int kc = kt.land ? 0 : cls;
                    const bool hi = !PAT || kt.land || cls < p.rem;
                    if constexpr (WALK)
                        log_walk(walk, t, b, kvh, hg, qt, cls, kt.k0,
                                 (kt.full ? 1 : 0) | (kt.land ? 2 : 0));
                    // test injection: this stage's copies never start, so the MMA
                    // warp's wait for them runs out (nothing is in flight to drain)
                    if (p.skip_first_kv && kv_iter == 0) continue;
                    mbar_expect_tx(BAR(L::K_FULL + st), L::KB);
                    for (int c = 0; c < HD / 64; ++c)
                        load_rows<PAT>(sK + st * L::KB + c * (BN * 128), hi ? &tmK : &tmK2,
                                    BAR(L::K_FULL + st), c * 64, kc, kt.k0, zkv);
                    mbar_expect_tx(BAR(L::V_FULL + st), L::KB);
                    for (int c = 0; c < HD / 64; ++c)
                        load_rows<PAT>(sV + st * L::KB + c * (BN * 128), hi ? &tmV : &tmV2,
                                    BAR(L::V_FULL + st), c * 64, kc, kt.k0, zkv);
                    last_k_par[st] = static_cast<int>(ph);
                    if (j == 0 && t + static_cast<int>(gridDim.x) < p.num_items) {
                        // prefetch the next item's Q one item ahead
                        if (!load_q(t + gridDim.x, it + 1)) {
                            ok = false;
                            break;
                        }
                    }
                }
            }
            if (!ok) {
                // drain: wait (bounded, ignoring the abort flag) for every load
                // still in flight to land before the CTA may exit
                for (int s = 0; s < STAGES; ++s)
                    if (last_k_par[s] >= 0) {
                        mbar_wait(BAR(L::K_FULL + s), last_k_par[s], nullptr, nullptr, TIMEOUT_NS);
                        mbar_wait(BAR(L::V_FULL + s), last_k_par[s], nullptr, nullptr, TIMEOUT_NS);
                    }
                for (int q = 0; q < 2; ++q)
                    if (last_q_par[q] >= 0)
                        mbar_wait(BAR(L::Q_FULL + q), last_q_par[q], nullptr, nullptr, TIMEOUT_NS);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop; each MMA and commit is issued by one
        // elected lane, with descriptor bases computed once per group.
        {
            const uint32_t idesc_s = idesc_bf16_f32(128, BN, 0);
            const uint32_t idesc_o = idesc_bf16_f32(128, HD, 1);
            int kv_iter = 0, it = 0, c = 0;
            bool ok = true;
            // the PV product of the previous tile, issued after the next S
            bool have_prev = false;
            int prev_st = 0, prev_c = 0, prev_it = 0;
            uint32_t prev_ph = 0;
            bool prev_first = false;
            auto issue_pv = [&]() -> bool {
                const int pb = prev_c & 1;
                if (!warp_wait(BAR(L::P_FULL + pb), (prev_c >> 1) & 1, abort_flag, p.status, p.wait_ns))
                    return false;
                if (!warp_wait(BAR(L::V_FULL + prev_st), prev_ph, abort_flag, p.status, p.wait_ns))
                    return false;
                if (prev_first &&
                    !warp_wait(BAR(L::O_EMPTY), (prev_it & 1) ^ 1, abort_flag, p.status, p.wait_ns))
                    return false;
                tc_fence_after();
                const uint64_t vb = smem_desc_sw128(sV + prev_st * L::KB, BN * 128, 1024);
                const uint32_t p_t = tmem + P_COL0 + pb * (BN / 2);
                mma_ts_e(tmem, p_t, vb, idesc_o, prev_first ? 0u : 1u);
#pragma unroll
                for (int ks = 1; ks < BN / 16; ++ks)
                    mma_ts_e(tmem, p_t + ks * 8, vb + static_cast<uint64_t>((ks * 16 * 128) >> 4),
                             idesc_o, 1u);
                tc_commit_e(BAR(L::KV_EMPTY + prev_st));
                tc_commit_e(BAR(L::PV_DONE + pb));
                return true;
            };
            for (int t = blockIdx.x; ok && t < p.num_items; t += gridDim.x, ++it) {
                int b, hg, kvh, qt, cls;
                decode_level_item<PAT>(t, p, p.G, b, hg, kvh, qt, cls);
                int off;
                const TileRange tr = item_tiles<PAT>(p, b, qt, cls, off);
                const int qb = it & 1;
                if (!warp_wait(BAR(L::Q_FULL + qb), (it >> 1) & 1, abort_flag, p.status, p.wait_ns)) {
                    ok = false;
                    break;
                }
                for (int j = 0; j < tr.count; ++j, ++kv_iter, ++c) {
                    const int st = kv_iter % STAGES;
                    const uint32_t ph = (kv_iter / STAGES) & 1;
                    const int sbuf = c & 1;
                    if (!warp_wait(BAR(L::K_FULL + st), ph, abort_flag, p.status, p.wait_ns) ||
                        !warp_wait(BAR(L::S_EMPTY + sbuf), ((c >> 1) & 1) ^ 1, abort_flag,
                                   p.status, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t qd = smem_desc_sw128(sQ + qb * L::QB, 16, 1024);
                    const uint64_t kd = smem_desc_sw128(sK + st * L::KB, 16, 1024);
#pragma unroll
                    for (int ks = 0; ks < HD / 16; ++ks) {
                        const uint32_t qo = ((ks >> 2) * (BM * 128) + (ks & 3) * 32) >> 4;
                        const uint32_t ko = ((ks >> 2) * (BN * 128) + (ks & 3) * 32) >> 4;
                        mma_ss_e(tmem + S_COL0 + sbuf * BN, qd + qo, kd + ko, idesc_s,
                                 ks > 0 ? 1u : 0u);
                    }
                    tc_commit_e(BAR(L::S_FULL + sbuf));
                    if (j == tr.count - 1) tc_commit_e(BAR(L::Q_EMPTY + qb));
                    if (have_prev && !issue_pv()) {
                        ok = false;
                        break;
                    }
                    have_prev = true;
                    prev_st = st;
                    prev_ph = ph;
                    prev_c = c;
                    prev_it = it;
                    prev_first = (j == 0);
                }
            }
            if (ok && have_prev) issue_pv();
            // drain: every MMA this warp issued has completed before exit
            tc_commit_e(BAR(L::DRAIN));
            warp_wait(BAR(L::DRAIN), 0, nullptr, nullptr, TIMEOUT_NS);
        }
    } else {
        // ------------------------------------------------------------ softmax
        const int sub = warp & 3;                 // TMEM lane quarter this warp may access
        const int r = sub * 32 + lane;            // query row within the tile
        const uint32_t lane_off = static_cast<uint32_t>(sub * 32) << 16;
        const float sl2 = p.sl2;
        int c = 0, it = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < p.num_items; t += gridDim.x, ++it) {
            int b, hg, kvh, qt, cls;
            decode_level_item<PAT>(t, p, p.G, b, hg, kvh, qt, cls);
            const int h = kvh * p.G + hg;
            int off;
            const TileRange tr = item_tiles<PAT>(p, b, qt, cls, off);
            const int i = tr.q0 + r;
            const int lo = i - p.w + 1;
            const int lhi = PAT ? land_hi(i, p.w, p.rl > 0 ? p.rl : 1) : 0;
            const int llo = PAT && p.rl > 0 ? land_lo(p.g, p.rl) : 0;
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < tr.count; ++j, ++c) {
                const int sbuf = c & 1;
                if (!warp_wait(BAR(L::S_FULL + sbuf), (c >> 1) & 1, abort_flag, p.status, p.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t s[4][32];
                const uint32_t sa = tmem + lane_off + S_COL0 + sbuf * BN;
#pragma unroll
                for (int q = 0; q < 4; ++q) tmem_ld32(sa + q * 32, s[q]);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 4; ++q) reg_fence32(s[q]);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(L::S_EMPTY + sbuf));

                const KeyTile kt = key_tile<PAT>(tr, j, p);
                if (!kt.full) {
                    // band and sink tiles: k <= i and (k >= i-w+1 or k < g); landmark
                    // tiles (k a landmark index): land_lo <= k <= land_hi(i)
                    const int khi = kt.land ? lhi : i, klo = kt.land ? llo : lo;
                    const int kgs = kt.land ? 0 : p.g;
                    // allowed: k <= khi and (k >= klo or k < kgs), in tile columns k - k0
                    mask_cols(s, klo - kt.k0, khi - kt.k0, kgs - kt.k0);
                }
                float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    mx0 = fmaxf(mx0, __uint_as_float(s[0][e]));
                    mx1 = fmaxf(mx1, __uint_as_float(s[1][e]));
                    mx2 = fmaxf(mx2, __uint_as_float(s[2][e]));
                    mx3 = fmaxf(mx3, __uint_as_float(s[3][e]));
                }
                const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
                const float m_new = fmaxf(m, m_tile);
                if (j == 0) {
                    m = m_new;  // O is overwritten by this item's first P V product
                } else {
                    const bool need = m_new > m + RESCALE_LOG2;
                    if (__any_sync(0xffffffffu, need)) {
                        const float alpha = need ? ex2(m - m_new) : 1.f;
                        if (need) m = m_new;
                        l *= alpha;
                        // O must be complete: wait for the previous tile's P V
                        const int pc = c - 1;
                        if (!warp_wait(BAR(L::PV_DONE + (pc & 1)), (pc >> 1) & 1, abort_flag,
                                       p.status, p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll 1
                        for (int q = 0; q < HD / 32; ++q) {
                            uint32_t o[32];
                            tmem_ld32(tmem + lane_off + q * 32, o);
                            tmem_ld_wait();
                            reg_fence32(o);
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st32(tmem + lane_off + q * 32, o);
                        }
                        tmem_st_wait();
                    }
                }
                const float m_use = (m == -INFINITY) ? 0.f : m;
                uint32_t pk[2][32];
                float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float p0 = ex2(fmaf(__uint_as_float(s[q][e]), sl2, -m_use));
                        const float p1 = ex2(fmaf(__uint_as_float(s[q][e + 1]), sl2, -m_use));
                        if (e & 2) {
                            l2 += p0;
                            l3 += p1;
                        } else {
                            l0 += p0;
                            l1 += p1;
                        }
                        pk[q >> 1][(q & 1) * 16 + (e >> 1)] = pack_bf16x2(p0, p1);
                    }
                l += (l0 + l1) + (l2 + l3);
                // P buffer (c & 1) is free once the P V of tile c-2 has completed
                if (c >= 2 && !warp_wait(BAR(L::PV_DONE + (c & 1)), ((c >> 1) & 1) ^ 1, abort_flag,
                                         p.status, p.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t pa = tmem + lane_off + P_COL0 + (c & 1) * (BN / 2);
                tmem_st32(pa, pk[0]);
                tmem_st32(pa + 32, pk[1]);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(L::P_FULL + (c & 1)));
            }
            if (!ok) break;
            // ---------------------------------------------------------- epilogue
            const int pc = c - 1;
            if (!warp_wait(BAR(L::PV_DONE + (pc & 1)), (pc >> 1) & 1, abort_flag, p.status, p.wait_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float row_lse;
            const float inv_l = finish_row(m, l, p.sink, h, &row_lse);
            // the query row of this thread: its index in the class subsequence,
            // and its position c + R t
            const int t_row = i - off;
            const size_t orow_i = static_cast<size_t>(b * p.H + h) * p.n +
                                  (PAT ? cls + static_cast<size_t>(p.R) * t_row : t_row);
            const bool row_ok = t_row < (!PAT ? p.n : cls < p.rem ? p.n_hi : p.n_lo) &&
                                SWA_BOUNDS(static_cast<long long>(orow_i) < p.dbg_orows, p.status);
            __nv_bfloat16 *orow = p.O + orow_i * HD;
            store_o_rows<HD>(tmem + lane_off, inv_l, orow, row_ok,
                             smem + L::STAGE_OFF + (warp - 2) * STAGE_WARP, lane);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(L::O_EMPTY));
            if (p.lse != nullptr && row_ok) p.lse[orow_i] = row_lse;
        }
    }
#undef BAR
#ifdef SWA_DEBUG
teardown:
#endif
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

// ------------------------------------------------------------------------
// Pair kernel: two query heads of one GQA group per work item.
//
// The two heads read the same key/value tiles, so each K/V tile staged in
// shared memory feeds four MMAs (S_A, S_B, P_A V, P_B V) instead of two.  Two
// softmax warpgroups (A: warps 4-7, B: warps 8-11) work on the two heads and
// take turns with the tensor core; the MMA warp issues, per key tile c,
//     P_A(c-1) V, S_A(c) = Q_A K^T, P_B(c-1) V, S_B(c) = Q_B K^T
// so softmax A(c) runs while the tensor core computes P_B(c-1) V and S_B(c),
// and the other way round.  512 threads in four warpgroups: warpgroup 0 holds
// the TMA warp (0) and the MMA warp (1), warpgroups 1 and 2 run the softmax of
// the two heads, and warpgroup 3 writes the output.  setmaxnreg moves
// registers from warpgroups 0 and 3 to the softmax warpgroups (REGS_SOFTMAX),
// so a full 128-column S row stays in registers.  TMEM (512 columns): O_A
// [0,128), S_A [128,256), O_B [256,384), S_B [384,512); P (bf16) is written
// back over the first half of its S buffer.  A tcgen05.commit tracks every MMA
// issued before it, so the S_X(c) barrier also tells softmax X that P_X(c-1) V
// has landed in O_X and that O_X may be rescaled.
// The epilogue warpgroup takes each item's output off the softmax warps'
// path: after its last tile a softmax warp only leaves the row's normaliser
// and LSE in shared memory and goes on with the next item; the epilogue warps
// wait for the item's last P V (O_FULL), read O_X out of tensor memory (each
// warp its TMEM lane quarter), free it for the next item (O_EMPTY), and store
// it through STAGE_WARP bytes of shared memory per warp (store_o_rows_chunked).
// ------------------------------------------------------------------------
constexpr int NTHREADS2 = 512;
// named barriers 1 (head A) and 2 (head B): a softmax warpgroup's 128 threads
// arrive when all of P is in tensor memory, the 32 threads of the MMA warp
// wait; 3 (A) and 4 (B) likewise when P's first 64 keys are (the pair kernel
// hands P over in two halves, so that the first half's P V runs while the
// second half is exponentiated)
constexpr int P_BAR_THREADS = 128 + 32;
// registers per thread after the hand-over: 128 * (80 + 176 + 176 + 80)
// equals the 512 * 128 registers the kernel is launched with
constexpr int REGS_CTRL = 80;
constexpr int REGS_SOFTMAX = 176;
constexpr int REGS_EPI = 80;

template <int HD>
struct Layout2 {
    static constexpr uint32_t QB = BM * HD * 2;
    static constexpr uint32_t KB = BN * HD * 2;
    static constexpr uint32_t Q_OFF = 0;  // Q_A, Q_B
    static constexpr uint32_t K_OFF = Q_OFF + 2 * QB;
    static constexpr uint32_t V_OFF = K_OFF + STAGES * KB;
    static constexpr uint32_t BAR_OFF = V_OFF + STAGES * KB;
    enum {
        Q_FULL = 0,
        Q_EMPTY = 2,
        K_FULL = 4,                  // K(c) and V(c-1) have landed (tile c's barrier)
        V_EMPTY = K_FULL + STAGES,   // a V slot is free (after the second head's P V)
        KV_EMPTY = V_EMPTY + STAGES, // a K slot is free (after the second head's S)
        S_FULL = KV_EMPTY + STAGES,
        P_FULL = S_FULL + 2,
        O_FULL = P_FULL + 2,
        O_EMPTY = O_FULL + 2,
        ROW_STATS = O_EMPTY + 2,  // [head x][item parity]: a row's normaliser and LSE are posted
        DRAIN = ROW_STATS + 4,
        NBAR = DRAIN + 1
    };
    static constexpr uint32_t MISC_OFF = BAR_OFF + NBAR * 8;
    // the producer's item-info ring (4 ints): the MMA warp's tile count per
    // item under the combined-stage protocol, so that it decodes no items
    static constexpr uint32_t INFO_OFF = MISC_OFF + 16;
    // (1/l, lse) per row: [item parity][head x][BM rows] float2
    static constexpr uint32_t STATS_OFF = (INFO_OFF + 16 + 15) & ~15u;
    static constexpr uint32_t STAGE_OFF = STATS_OFF + 2 * 2 * BM * 8;  // 4 epilogue warps
    static constexpr uint32_t BYTES = STAGE_OFF + 4 * STAGE_WARP;
    static constexpr uint32_t DYN_SMEM = (BYTES + 1024 > 120 * 1024) ? BYTES + 1024 : 120 * 1024;
};

// Work order of the pair kernel.  Items are ranked q tile first, the last q
// tile (the most key tiles) first; within a q tile by sequence, kv head and
// head pair, so the CTAs working at the same time share one band position of
// every kv head (a few MB of K/V in L2).  Rank r goes to CTA r % P in even
// rounds and P-1 - r % P in odd rounds (a snake), which evens out the cheaper
// q tiles at the start of the sequence across the CTAs.  CTA c's k-th item has
// rank pair_item_rank(c, k); ranks >= num_items end its loop.
__device__ __forceinline__ int pair_item_rank(int c, int k)
{
    const int P = static_cast<int>(gridDim.x);
    return k * P + ((k & 1) ? P - 1 - c : c);
}


// Softmax warpgroup x: P_x of the current key tile is in tensor memory.
__device__ __forceinline__ void p_arrive(int x)
{
    if (x == 0)
        asm volatile("bar.arrive 1, %0;" ::"n"(128 + 32) : "memory");
    else
        asm volatile("bar.arrive 2, %0;" ::"n"(128 + 32) : "memory");
}
// ... and its first 64 keys (pair kernel)
__device__ __forceinline__ void p_arrive_half(int x)
{
    if (x == 0)
        asm volatile("bar.arrive 3, %0;" ::"n"(128 + 32) : "memory");
    else
        asm volatile("bar.arrive 4, %0;" ::"n"(128 + 32) : "memory");
}

__device__ __forceinline__ uint64_t pack2(uint32_t lo, uint32_t hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.ftz.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.ftz.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float max3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Softmax over 64 columns (two 32-column halves of s) of one row: p =
// exp2(s * sl2 - m), accumulated into the pair-sum `acc2`, packed to bf16 pairs.
__device__ __forceinline__ void softmax_half(const uint32_t (&sa)[32], const uint32_t (&sb)[32],
                                             uint64_t sl2x2, uint64_t negm2, uint64_t &acc2,
                                             uint32_t (&pk)[32])
{
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
        float x0, x1, y0, y1;
        unpack2(fma2(pack2(sa[e], sa[e + 1]), sl2x2, negm2), x0, x1);
        unpack2(fma2(pack2(sb[e], sb[e + 1]), sl2x2, negm2), y0, y1);
        const float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(y0), p3 = ex2(y1);
        acc2 = add2(acc2, add2(pack2(__float_as_uint(p0), __float_as_uint(p1)),
                               pack2(__float_as_uint(p2), __float_as_uint(p3))));
        pk[e >> 1] = pack_bf16x2(p0, p1);
        pk[16 + (e >> 1)] = pack_bf16x2(p2, p3);
    }
}

template <int HD, bool PAT, bool QP, bool SKEW, bool WALK>
__global__ void __launch_bounds__(NTHREADS2, 1)
    swa_prefill_bf16_pair_sm103(const __grid_constant__ CUtensorMap tmQ,
                                const __grid_constant__ CUtensorMap tmK,
                                const __grid_constant__ CUtensorMap tmV,
                                const __grid_constant__ CUtensorMap tmQ2,
                                const __grid_constant__ CUtensorMap tmK2,
                                const __grid_constant__ CUtensorMap tmV2, const PrefillParams p,
                           int32_t *walk)
{
    using L = Layout2<HD>;
    // SKEW, the K/V protocol: tile c's barrier carries K(c) and V(c-1), with the
    // K and V slots freed separately, so K(c) is requested a tile period early
    // (items of many key tiles: the window path, landmark and dilated
    // patterns); otherwise one K/V stage per tile, freed after the second
    // head's P V (items of one or two tiles, where a P V product should not
    // wait for the next tile's K).  See the producer.
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(smem);
    const uint32_t sQ = sb + L::Q_OFF, sK = sb + L::K_OFF, sV = sb + L::V_OFF;
    const uint32_t bars = sb + L::BAR_OFF;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::MISC_OFF + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pairs_per_item_count = p.num_items;
    // item it's key-tile count at [it & 3] (the combined-stage protocol):
    // written by the producer before any copy of the item completes a barrier,
    // read by the MMA warp after the item's first Q barrier
    volatile int *item_info = reinterpret_cast<volatile int *>(smem + L::INFO_OFF);
#define BAR(i) (bars + 8u * static_cast<uint32_t>(i))

    if (threadIdx.x == 0) {
        for (int x = 0; x < 2; ++x) {
            mbar_init(BAR(L::Q_FULL + x), 1);
            mbar_init(BAR(L::Q_EMPTY + x), 1);
            mbar_init(BAR(L::S_FULL + x), 1);
            mbar_init(BAR(L::P_FULL + x), 4);
            mbar_init(BAR(L::O_FULL + x), 1);
            mbar_init(BAR(L::O_EMPTY + x), 4);
            mbar_init(BAR(L::ROW_STATS + 2 * x), 4);
            mbar_init(BAR(L::ROW_STATS + 2 * x + 1), 4);
        }
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(BAR(L::K_FULL + i), 1);
            mbar_init(BAR(L::V_EMPTY + i), 1);
            mbar_init(BAR(L::KV_EMPTY + i), 1);
        }
        mbar_init(BAR(L::DRAIN), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch(&tmQ);
        tma_prefetch(&tmK);
        tma_prefetch(&tmV);
        tma_prefetch(&tmQ2);
        tma_prefetch(&tmK2);
        tma_prefetch(&tmV2);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
#ifdef SWA_DEBUG
    if (!tmem_base_ok(tmem, p.status)) goto teardown;
#endif

    if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_CTRL));
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            if constexpr (!SKEW) {
                // one stage and one barrier per tile for K and V, freed after the
                // second head's P V; the Q tiles go first (fixed patterns with
                // items of one or two key tiles)
                int kv_iter = 0, it = 0;
                int last_k_par[STAGES], last_q_par[2] = {-1, -1};
                for (int s = 0; s < STAGES; ++s) last_k_par[s] = -1;
                bool ok = true;
                for (int t = pair_item_rank(blockIdx.x, 0); ok && t < pairs_per_item_count;
                     t = pair_item_rank(blockIdx.x, ++it)) {
                    int b, hp, kvh, qt, cls;
                    decode_level_item<PAT>(t, p, pair_units<QP>(p), b, hp, kvh, qt, cls);
                    (void)SWA_BOUNDS(SWA_ITEM_IN_RANGE(p, b, kvh, qt, cls), p.status);
                    int off;
                    const TileRange tr = item_tiles<PAT, QP>(p, b, qt, cls, off);
                    item_info[it & 3] = tr.count;
                    const CUtensorMap *mq = (!PAT || cls < p.rem) ? &tmQ : &tmQ2;
                    for (int x = 0; x < 2 && ok; ++x) {
                        if (!mbar_wait(BAR(L::Q_EMPTY + x), (it & 1) ^ 1, abort_flag, p.status,
                                       p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        mbar_expect_tx(BAR(L::Q_FULL + x), L::QB);
                        const int hx = pair_head<QP>(p, kvh, hp, x);
                        const int qrow = QP ? (2 * qt + x) * BM : qt * BM;
                        for (int c = 0; c < HD / 64; ++c)
                            load_rows<PAT>(sQ + x * L::QB + c * (BM * 128), mq, BAR(L::Q_FULL + x),
                                           c * 64, cls, qrow, b * p.H + hx);
                        last_q_par[x] = it & 1;
                    }
                    for (int j = 0; ok && j < tr.count; ++j, ++kv_iter) {
                        const int st = kv_iter % STAGES;
                        const uint32_t ph = (kv_iter / STAGES) & 1;
                        if (!mbar_wait(BAR(L::KV_EMPTY + st), ph ^ 1, abort_flag, p.status,
                                       p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        const KeyTile kt = key_tile<PAT>(tr, j, p);
                        (void)SWA_BOUNDS(key_tile_in_range<PAT>(kt, cls, p), p.status);
                        const int zkv = b * p.Hkv + kvh;
                        // landmark tiles: class 0 of the stride-rl view; others: this class
                        const int kc = kt.land ? 0 : cls;
                        const bool hi = !PAT || kt.land || cls < p.rem;
                        if constexpr (WALK)
                            log_walk(walk, t, b, kvh, hp, qt, cls, kt.k0,
                                     (kt.full ? 1 : 0) | (kt.land ? 2 : 0));
                        // test injection: this stage's copies never start, so the MMA
                        // warp's wait for them runs out (nothing is in flight to drain)
                        if (p.skip_first_kv && kv_iter == 0) continue;
                        mbar_expect_tx(BAR(L::K_FULL + st), 2 * L::KB);
                        for (int c = 0; c < HD / 64; ++c)
                            load_rows<PAT>(sK + st * L::KB + c * (BN * 128), hi ? &tmK : &tmK2,
                                           BAR(L::K_FULL + st), c * 64, kc, kt.k0, zkv);
                        for (int c = 0; c < HD / 64; ++c)
                            load_rows<PAT>(sV + st * L::KB + c * (BN * 128), hi ? &tmV : &tmV2,
                                           BAR(L::K_FULL + st), c * 64, kc, kt.k0, zkv);
                        last_k_par[st] = static_cast<int>(ph);
                    }
                }
                if (!ok) {
                    for (int s = 0; s < STAGES; ++s)
                        if (last_k_par[s] >= 0)
                            mbar_wait(BAR(L::K_FULL + s), last_k_par[s], nullptr, nullptr, TIMEOUT_NS);
                    for (int x = 0; x < 2; ++x)
                        if (last_q_par[x] >= 0)
                            mbar_wait(BAR(L::Q_FULL + x), last_q_par[x], nullptr, nullptr, TIMEOUT_NS);
                }
            } else {
                int kv_iter = 0, it = 0;
                int last_k_par[STAGES], last_q_par[2] = {-1, -1};
                for (int s = 0; s < STAGES; ++s) last_k_par[s] = -1;
                bool ok = true;
                // Tile c's barrier (K_FULL slot c % STAGES) carries K(c) and V(c-1): the
                // K slot is freed after the second head's S (a tile earlier than a
                // combined K/V stage would be), so K(c) is requested a whole tile
                // period before S_A(c) needs it, and the MMA warp still waits once per
                // tile.  The last tile's V rides on the barrier of the tile after it.
                // pv_*: the previous tile's V, still to be loaded.
                bool pv_have = false;
                int pv_k0 = 0, pv_kc = 0, pv_z = 0;
                const CUtensorMap *pv_map = &tmV;
                // waits until V slot (c_next - 1) % STAGES is free for V(c_next - 1)
                auto load_prev_v = [&](int c_next) -> bool {
                    const int vc = c_next - 1, vs = vc % STAGES;
                    if (!mbar_wait(BAR(L::V_EMPTY + vs), ((vc / STAGES) & 1) ^ 1, abort_flag, p.status,
                                   p.wait_ns))
                        return false;
                    return true;
                };
                auto issue_prev_v = [&](int c_next, uint32_t bar) {
                    const int vs = (c_next - 1) % STAGES;
                    for (int c = 0; c < HD / 64; ++c)
                        load_rows<PAT>(sV + vs * L::KB + c * (BN * 128), pv_map, bar, c * 64, pv_kc,
                                       pv_k0, pv_z);
                };
                for (int t = pair_item_rank(blockIdx.x, 0); ok && t < pairs_per_item_count;
                     t = pair_item_rank(blockIdx.x, ++it)) {
                    int b, hp, kvh, qt, cls;
                    decode_level_item<PAT>(t, p, pair_units<QP>(p), b, hp, kvh, qt, cls);
                    (void)SWA_BOUNDS(SWA_ITEM_IN_RANGE(p, b, kvh, qt, cls), p.status);
                    int off;
                    const TileRange tr = item_tiles<PAT, QP>(p, b, qt, cls, off);
                    const CUtensorMap *mq = (!PAT || cls < p.rem) ? &tmQ : &tmQ2;
                    // the item's Q tiles.  Their buffers free up only at the
                    // previous item's last S, and the MMA warp first needs the
                    // previous item's last value tile, so on the window path they
                    // go after the item's first key tile (which carries that V):
                    // 1-4% faster than the other order.  For the fixed patterns
                    // they go first: 2-4% faster there.
                    auto load_q_tiles = [&]() -> bool {
                        for (int x = 0; x < 2; ++x) {
                            if (!mbar_wait(BAR(L::Q_EMPTY + x), (it & 1) ^ 1, abort_flag, p.status,
                                           p.wait_ns))
                                return false;
                            mbar_expect_tx(BAR(L::Q_FULL + x), L::QB);
                            const int hx = pair_head<QP>(p, kvh, hp, x);
                            const int qrow = QP ? (2 * qt + x) * BM : qt * BM;
                            for (int c = 0; c < HD / 64; ++c)
                                load_rows<PAT>(sQ + x * L::QB + c * (BM * 128), mq,
                                               BAR(L::Q_FULL + x), c * 64, cls, qrow, b * p.H + hx);
                            last_q_par[x] = it & 1;
                        }
                        return true;
                    };
                    if (PAT && !load_q_tiles()) ok = false;
                    for (int j = 0; ok && j < tr.count; ++j, ++kv_iter) {
                        const int st = kv_iter % STAGES;
                        const uint32_t ph = (kv_iter / STAGES) & 1;
                        if ((pv_have && !load_prev_v(kv_iter)) ||
                            !mbar_wait(BAR(L::KV_EMPTY + st), ph ^ 1, abort_flag, p.status,
                                       p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        const KeyTile kt = key_tile<PAT>(tr, j, p);
                        (void)SWA_BOUNDS(key_tile_in_range<PAT>(kt, cls, p), p.status);
                        const int zkv = b * p.Hkv + kvh;
                        // landmark tiles: class 0 of the stride-rl view; others: this class
                        const int kc = kt.land ? 0 : cls;
                        const bool hi = !PAT || kt.land || cls < p.rem;
                        // test injection: this stage's copies never start, so the MMA
                        // warp's wait for them runs out (nothing is in flight to drain)
                        if (p.skip_first_kv && kv_iter == 0) {
                            pv_have = false;
                            continue;
                        }
                        // this tile's K and the previous tile's V complete this tile's
                        // barrier
                        if constexpr (WALK)
                            log_walk(walk, t, b, kvh, hp, qt, cls, kt.k0,
                                     (kt.full ? 1 : 0) | (kt.land ? 2 : 0));
                        const CUtensorMap *mk = hi ? &tmK : &tmK2;
                        const CUtensorMap *mv = hi ? &tmV : &tmV2;
                        mbar_expect_tx(BAR(L::K_FULL + st), pv_have ? 2 * L::KB : L::KB);
                        if (pv_have) issue_prev_v(kv_iter, BAR(L::K_FULL + st));
                        for (int c = 0; c < HD / 64; ++c)
                            load_rows<PAT>(sK + st * L::KB + c * (BN * 128), mk, BAR(L::K_FULL + st),
                                           c * 64, kc, kt.k0, zkv);
                        last_k_par[st] = static_cast<int>(ph);
                        pv_have = true;
                        pv_k0 = kt.k0;
                        pv_kc = kc;
                        pv_z = zkv;
                        pv_map = mv;
                        if (!PAT && j == 0 && !load_q_tiles()) {
                            ok = false;
                            break;
                        }
                    }
                }
                // the last tile's V, on the barrier of the tile after it
                if (ok && pv_have) {
                    const int st = kv_iter % STAGES;
                    const uint32_t ph = (kv_iter / STAGES) & 1;
                    // the barrier's previous phase (tile kv_iter - 2) must be complete
                    // before it is armed again: its K slot release says so
                    if (!load_prev_v(kv_iter) ||
                        !mbar_wait(BAR(L::KV_EMPTY + st), ph ^ 1, abort_flag, p.status, p.wait_ns)) {
                        ok = false;
                    } else {
                        mbar_expect_tx(BAR(L::K_FULL + st), L::KB);
                        issue_prev_v(kv_iter, BAR(L::K_FULL + st));
                        last_k_par[st] = static_cast<int>(ph);
                    }
                }
                if (!ok) {
                    for (int s = 0; s < STAGES; ++s)
                        if (last_k_par[s] >= 0)
                            mbar_wait(BAR(L::K_FULL + s), last_k_par[s], nullptr, nullptr, TIMEOUT_NS);
                    for (int x = 0; x < 2; ++x)
                        if (last_q_par[x] >= 0)
                            mbar_wait(BAR(L::Q_FULL + x), last_q_par[x], nullptr, nullptr, TIMEOUT_NS);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The issuing warp shares its SM sub-partition with two softmax warps,
        // and a single thread issues a 128x128x16 MMA only a little faster than
        // the tensor core executes it, so the issue path is kept short: the
        // whole warp runs the loop (waits, bookkeeping) and each MMA and commit
        // is issued by one elected lane; descriptor bases are computed once per
        // group and the K-steps are unrolled with compile-time offsets.
        {
            const uint32_t idesc_s = idesc_bf16_f32(128, BN, 0);
            const uint32_t idesc_o = idesc_bf16_f32(128, HD, 1);
            int kv_iter = 0, it = 0, c = 0;
            bool ok = true;
            bool have_prev = false, prev_first = false, prev_last = false;
            int prev_st = 0, prev_c = 0, prev_it = 0;
            // P_X(prev) V into O_X
            auto issue_pv = [&](auto xc) -> bool {
                constexpr int x = decltype(xc)::value;
                // P_X(prev) stored: softmax warpgroup X arrives on named barrier
                // 1 + x (a hardware barrier wakes the issuer sooner than an
                // mbarrier).  A warpgroup that gives up arrives once more and sets
                // the abort flag, which is checked after every meeting, so this
                // never waits for an arrival that will not come.
                // P_X's first 64 keys: their half of P V goes to the tensor core
                // while the softmax warpgroup exponentiates the other half
                asm volatile("bar.sync %0, %1;" ::"n"(3 + x), "n"(P_BAR_THREADS) : "memory");
                if (prev_first && !warp_wait(BAR(L::O_EMPTY + x), (prev_it & 1) ^ 1, abort_flag,
                                             p.status, p.wait_ns))
                    return false;
                tc_fence_after();
                const uint64_t vb = smem_desc_sw128(sV + prev_st * L::KB, BN * 128, 1024);
                const uint32_t o_t = tmem + x * 256, p_t = tmem + x * 256 + 128;
                mma_ts_group4(o_t, p_t, vb, idesc_o, prev_first ? 0u : 1u);
                asm volatile("bar.sync %0, %1;" ::"n"(1 + x), "n"(P_BAR_THREADS) : "memory");
                tc_fence_after();
                // keys 64..127: P columns 32.., V rows 64.. (64 * 128 B >> 4)
                mma_ts_group4(o_t, p_t + 32, vb + 512, idesc_o, 1u);
                // the V slot (window path) or the whole K/V stage (fixed patterns)
                if (x == 1) tc_commit_e(BAR((SKEW ? L::V_EMPTY : L::KV_EMPTY) + prev_st));
                if (prev_last) tc_commit_e(BAR(L::O_FULL + x));
                // a softmax warpgroup that gave up arrived once more on the barrier
                // above; the product just issued read a garbage P, which is harmless
                return !*abort_flag;
            };
            // S_X = Q_X K^T
            auto issue_s = [&](auto xc, int st, bool last) {
                constexpr int x = decltype(xc)::value;
                const uint64_t qb = smem_desc_sw128(sQ + x * L::QB, 16, 1024);
                const uint64_t kb = smem_desc_sw128(sK + st * L::KB, 16, 1024);
                const uint32_t s_t = tmem + x * 256 + 128;
                mma_ss_group<HD / 16>(s_t, qb, kb, idesc_s);
                tc_commit_e(BAR(L::S_FULL + x));
                if (last) tc_commit_e(BAR(L::Q_EMPTY + x));
                if (SKEW && x == 1) tc_commit_e(BAR(L::KV_EMPTY + st));  // the K slot
            };
            using X0 = std::integral_constant<int, 0>;
            using X1 = std::integral_constant<int, 1>;
            for (int t = pair_item_rank(blockIdx.x, 0); ok && t < pairs_per_item_count;
                 t = pair_item_rank(blockIdx.x, ++it)) {
                // the item's tile count: worked out here on the skewed path
                // (items of many tiles); for items of one or two
                // tiles, where the issuer's own index arithmetic showed, taken
                // from the producer (item_info) once the item's first Q barrier
                // has passed (measured 4% faster on the strided pattern, no
                // gain or 1% slower on long items)
                int count = 1;
                if constexpr (SKEW) {
                    int b, hp, kvh, qt, cls, off;
                    decode_level_item<PAT>(t, p, pair_units<QP>(p), b, hp, kvh, qt, cls);
                    count = item_tiles<PAT, QP>(p, b, qt, cls, off).count;
                }
                for (int j = 0; j < count; ++j, ++kv_iter, ++c) {
                    const int st = kv_iter % STAGES;
                    const uint32_t ph = (kv_iter / STAGES) & 1;
                    // window path: K(c) and V(c-1) have landed (one wait per tile,
                    // before P_A(c-1) V); fixed patterns: K(c) and V(c), after it
                    if (SKEW &&
                        !warp_wait(BAR(L::K_FULL + st), ph, abort_flag, p.status, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    // head A: P_A(c-1) V, then S_A(c)
                    if (have_prev && !issue_pv(X0{})) {
                        ok = false;
                        break;
                    }
                    if ((j == 0 &&
                         !warp_wait(BAR(L::Q_FULL + 0), it & 1, abort_flag, p.status, p.wait_ns)) ||
                        (!SKEW &&
                         !warp_wait(BAR(L::K_FULL + st), ph, abort_flag, p.status, p.wait_ns))) {
                        ok = false;
                        break;
                    }
                    if (!SKEW && j == 0) count = item_info[it & 3];
                    const bool last = (j == count - 1);
                    tc_fence_after();
                    issue_s(X0{}, st, last);
                    // head B: P_B(c-1) V, then S_B(c)
                    if (have_prev && !issue_pv(X1{})) {
                        ok = false;
                        break;
                    }
                    if (j == 0 && !warp_wait(BAR(L::Q_FULL + 1), it & 1, abort_flag, p.status, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_s(X1{}, st, last);
                    have_prev = true;
                    prev_st = st;
                    prev_c = c;
                    prev_it = it;
                    prev_first = (j == 0);
                    prev_last = last;
                }
            }
            // the last tile's V (window path: on the barrier of the tile after it)
            if (ok && have_prev &&
                (!SKEW || warp_wait(BAR(L::K_FULL + kv_iter % STAGES), (kv_iter / STAGES) & 1,
                                    abort_flag, p.status, p.wait_ns))) {
                if (issue_pv(X0{})) issue_pv(X1{});
            }
            // drain: every MMA this warp issued has completed before exit
            tc_commit_e(BAR(L::DRAIN));
            warp_wait(BAR(L::DRAIN), 0, nullptr, nullptr, TIMEOUT_NS);
        }
    }
    } else if (warp < 12) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REGS_SOFTMAX));
        // ------------------------------------------------------------ softmax A / B
        const int x = (warp >> 2) - 1;           // 0: head h0 (warps 4-7), 1: h0+1 (warps 8-11)
        const int sub = warp & 3;                // TMEM lane quarter this warp may access
        const int r = sub * 32 + lane;           // query row within the tile
        const uint32_t lane_off = static_cast<uint32_t>(sub * 32) << 16;
        const uint32_t o_addr = tmem + lane_off + x * 256;
        const uint32_t s_addr = o_addr + 128;
        const float sl2 = p.sl2;
        const uint64_t sl2x2 = pack2(__float_as_uint(sl2), __float_as_uint(sl2));
        float2 *stats = reinterpret_cast<float2 *>(smem + L::STATS_OFF);
        int c = 0, it = 0;
        bool ok = true;
        // the item's sequence, head, class, query offset and key tiles; the next
        // item's are worked out while this one's last P V runs
        struct Item {
            int b, h, cls, off;
            TileRange tr;
        };
        auto load_item = [&](int t, Item &e) {
            int hp, kvh, qt;
            decode_level_item<PAT>(t, p, pair_units<QP>(p), e.b, hp, kvh, qt, e.cls);
            e.h = pair_head<QP>(p, kvh, hp, x);
            e.tr = item_tiles<PAT, QP>(p, e.b, qt, e.cls, e.off);
        };
        Item nxt;
        int t = pair_item_rank(blockIdx.x, 0);
        if (t < pairs_per_item_count) load_item(t, nxt);
        while (ok && t < pairs_per_item_count) {
            const int h = nxt.h;
            const TileRange tr = nxt.tr;
            // this half's own rows: with q-tile pairs, half x is q tile 2k + x,
            // and tiles of the walk are classed (full or not) against its rows
            constexpr bool qp = QP;
            TileRange trx = tr;
            if constexpr (qp) {
                trx.q0 = tr.q0 + x * BM;
                const int e1 = trx.q0 + BM - 1;
                trx.q1 = e1 < tr.q1 ? e1 : tr.q1;
            }
            const int i = trx.q0 + r;
            const int lo = i - p.w + 1;
            const int lhi = PAT ? land_hi(i, p.w, p.rl > 0 ? p.rl : 1) : 0;
            const int llo = PAT && p.rl > 0 ? land_lo(p.g, p.rl) : 0;
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < tr.count; ++j, ++c) {
                if (!warp_wait(BAR(L::S_FULL + x), c & 1, abort_flag, p.status, p.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t s[4][32];
#pragma unroll
                for (int q = 0; q < 4; ++q) tmem_ld32(s_addr + q * 32, s[q]);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 4; ++q) reg_fence32(s[q]);
                const KeyTile kt = key_tile<PAT>(tr, j, p);
                const bool full = qp ? tile_full(trx, kt.k0 / BN, p.w, p.g, BN) : kt.full;
                if (!full) {
                    // band and sink tiles: k <= i and (k >= i-w+1 or k < g); landmark
                    // tiles (k a landmark index): land_lo <= k <= land_hi(i)
                    const int khi = kt.land ? lhi : i, klo = kt.land ? llo : lo;
                    const int kgs = kt.land ? 0 : p.g;
                    // allowed: k <= khi and (k >= klo or k < kgs), in tile columns k - k0
                    mask_cols(s, klo - kt.k0, khi - kt.k0, kgs - kt.k0);
                }
                float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    mx0 = max3(mx0, __uint_as_float(s[0][e]), __uint_as_float(s[0][e + 1]));
                    mx1 = max3(mx1, __uint_as_float(s[1][e]), __uint_as_float(s[1][e + 1]));
                    mx2 = max3(mx2, __uint_as_float(s[2][e]), __uint_as_float(s[2][e + 1]));
                    mx3 = max3(mx3, __uint_as_float(s[3][e]), __uint_as_float(s[3][e + 1]));
                }
                const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
                const float m_new = fmaxf(m, m_tile);
                if (j == 0) {
                    m = m_new;
                } else {
                    const bool need = m_new > m + RESCALE_LOG2;
                    if (__any_sync(0xffffffffu, need)) {
                        // O_X is complete: the S_X(c) commit covered P_X(c-1) V
                        const float alpha = need ? ex2(m - m_new) : 1.f;
                        if (need) m = m_new;
                        l *= alpha;
#pragma unroll 1
                        for (int q = 0; q < HD / 32; ++q) {
                            uint32_t o[32];
                            tmem_ld32(o_addr + q * 32, o);
                            tmem_ld_wait();
                            reg_fence32(o);
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st32(o_addr + q * 32, o);
                        }
                    }
                }
                const float m_use = (m == -INFINITY) ? 0.f : m;
                const uint64_t negm2 = pack2(__float_as_uint(-m_use), __float_as_uint(-m_use));
                uint64_t acc2 = 0;  // two fp32 zeros
                uint32_t pk[32];
                // keys 0..63, handed over first, then keys 64..127
                softmax_half(s[0], s[1], sl2x2, negm2, acc2, pk);
                tmem_st32(s_addr, pk);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                p_arrive_half(x);
                softmax_half(s[2], s[3], sl2x2, negm2, acc2, pk);
                tmem_st32(s_addr + 32, pk);
                float a0, a1;
                unpack2(acc2, a0, a1);
                l += a0 + a1;
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                p_arrive(x);
            }
            if (!ok) break;
            // the row's normaliser and LSE to the epilogue warpgroup, which
            // writes this item's output while this warp goes on with the next
            float row_lse;
            const float inv_l = finish_row(m, l, p.sink, h, &row_lse);
            stats[((it & 1) * 2 + x) * BM + r] = make_float2(inv_l, row_lse);
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(L::ROW_STATS + 2 * x + (it & 1)));
            const int t_next = pair_item_rank(blockIdx.x, it + 1);
            if (t_next < pairs_per_item_count) load_item(t_next, nxt);
            ++it;
            t = t_next;
        }
        // gave up (a wait ran out): one more arrival on each of this head's
        // two P barriers lets an issuer that is already waiting on either meet,
        // see the abort flag and stop
        if (!ok) {
            *abort_flag = 1;
            __syncwarp();
            p_arrive_half(x);
            p_arrive(x);
        }
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_EPI));
        // ------------------------------------------------------------ epilogue
        // Per item and head: wait for the softmax's row statistics and for the
        // item's last P V, then write O / l as bf16 (and the LSE).
        const int sub = warp & 3;                // TMEM lane quarter this warp may access
        const int r = sub * 32 + lane;           // query row within the tile
        const uint32_t lane_off = static_cast<uint32_t>(sub * 32) << 16;
        const float2 *stats = reinterpret_cast<const float2 *>(smem + L::STATS_OFF);
        uint8_t *stage = smem + L::STAGE_OFF + sub * STAGE_WARP;
        int it = 0;
        bool ok = true;
        for (int t = pair_item_rank(blockIdx.x, 0); ok && t < pairs_per_item_count;
             t = pair_item_rank(blockIdx.x, ++it)) {
            int b, hp, kvh, qt, cls, off;
            decode_level_item<PAT>(t, p, pair_units<QP>(p), b, hp, kvh, qt, cls);
            const TileRange tr = item_tiles<PAT, QP>(p, b, qt, cls, off);
            const int nq = !PAT ? p.n : cls < p.rem ? p.n_hi : p.n_lo;
#pragma unroll 1
            for (int x = 0; x < 2; ++x) {
                if (!warp_wait(BAR(L::ROW_STATS + 2 * x + (it & 1)), (it >> 1) & 1, abort_flag,
                               p.status, p.wait_ns) ||
                    !warp_wait(BAR(L::O_FULL + x), it & 1, abort_flag, p.status, p.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float2 sv = stats[((it & 1) * 2 + x) * BM + r];
                const int h = pair_head<QP>(p, kvh, hp, x);
                // this thread's query row: half x of a q-tile pair is q tile 2k + x
                const int i = tr.q0 + (QP ? x * BM : 0) + r;
                const int t_row = i - off;
                const size_t orow_i = static_cast<size_t>(b * p.H + h) * p.n +
                                      (PAT ? cls + static_cast<size_t>(p.R) * t_row : t_row);
                const bool row_ok =
                    t_row < nq && SWA_BOUNDS(static_cast<long long>(orow_i) < p.dbg_orows, p.status);
                store_o_rows_chunked<HD>(tmem + lane_off + x * 256, sv.x, p.O + orow_i * HD,
                                         row_ok, stage, lane, BAR(L::O_EMPTY + x));
                if (p.lse != nullptr && row_ok) p.lse[orow_i] = sv.y;
            }
        }
    }
#undef BAR
#ifdef SWA_DEBUG
teardown:
#endif
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

// ------------------------------------------------------------------------
// One-tile self-test of the operand encodings (no counterpart on the pages).
// ------------------------------------------------------------------------
__global__ void __launch_bounds__(128, 1)
    swa_selftest_umma_sm103(const __grid_constant__ CUtensorMap tmA,
                            const __grid_constant__ CUtensorMap tmBk,
                            const __grid_constant__ CUtensorMap tmBn, const __nv_bfloat16 *A,
                            float *D1, float *D2, int *status)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(smem);
    const uint32_t sA = sb, sBk = sb + 32768, sBn = sb + 65536;
    const uint32_t bar_ld = sb + 98304, bar_mma = bar_ld + 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + 98304 + 16);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(bar_ld, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;
    if (threadIdx.x == 0) {
        mbar_expect_tx(bar_ld, 3 * 32768);
        for (int c = 0; c < 2; ++c) {
            tma_load_3d(sA + c * 16384, &tmA, bar_ld, c * 64, 0, 0);
            tma_load_3d(sBk + c * 16384, &tmBk, bar_ld, c * 64, 0, 0);
            tma_load_3d(sBn + c * 16384, &tmBn, bar_ld, c * 64, 0, 0);
        }
        ok = mbar_wait(bar_ld, 0, nullptr, status, TIMEOUT_NS);
    }
    // A into TMEM columns 256..319 as bf16 pairs, one row per thread
    {
        const int r = threadIdx.x;
        const uint32_t *arow = reinterpret_cast<const uint32_t *>(A + r * 128);
        uint32_t v[2][32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            v[0][e] = arow[e];
            v[1][e] = arow[32 + e];
        }
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        tmem_st32(tmem + lane_off + 256, v[0]);
        tmem_st32(tmem + lane_off + 288, v[1]);
        tmem_st_wait();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0 && ok) {
        const uint32_t id1 = idesc_bf16_f32(128, 128, 0);
        const uint32_t id2 = idesc_bf16_f32(128, 128, 1);
        for (int ks = 0; ks < 8; ++ks) {
            const uint32_t blk = ks >> 2, sub = ks & 3;
            mma_ss(tmem + 0, smem_desc_sw128(sA + blk * 16384 + sub * 32, 16, 1024),
                   smem_desc_sw128(sBk + blk * 16384 + sub * 32, 16, 1024), id1, ks > 0);
        }
        for (int ks = 0; ks < 8; ++ks)
            mma_ts(tmem + 128, tmem + 256 + ks * 8, smem_desc_sw128(sBn + ks * 2048, 16384, 1024),
                   id2, ks > 0);
        tc_commit(bar_mma);
        mbar_wait(bar_mma, 0, nullptr, status, TIMEOUT_NS);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    {
        const int r = threadIdx.x;
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        for (int q = 0; q < 4; ++q) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_off + q * 32, o);
            tmem_ld_wait();
            reg_fence32(o);
            for (int e = 0; e < 32; ++e) D1[r * 128 + q * 32 + e] = __uint_as_float(o[e]);
            tmem_ld32(tmem + lane_off + 128 + q * 32, o);
            tmem_ld_wait();
            reg_fence32(o);
            for (int e = 0; e < 32; ++e) D2[r * 128 + q * 32 + e] = __uint_as_float(o[e]);
        }
    }
    (void)lane;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------------
// Host side: tensor maps and launches.
// ------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// bf16 tensor [d2][d1][d0] (d0 contiguous) tiled in boxes of {64, rows, 1},
// 128-byte swizzle, zero fill outside the tensor.
bool make_map_3d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
                 uint32_t rows)
{
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
    cuuint32_t box[3] = {64, rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A 4-D view of a bf16 tensor [Z][rows_total][d]: dims (d, R, rows, Z), byte
// strides (d*2, R*d*2, rows_total*d*2), so element (x, c, k, z) is column x of
// row c + R*k of slice z, and a box (64, 1, box_rows, 1) taken at class c is
// box_rows rows R apart.  R = 1 is the plain row-major tensor.  The caller
// keeps c + R*(rows-1) < rows_total for every class a box is taken at, so no
// box reaches past its slice.
bool make_view(CUtensorMap *m, const void *base, uint64_t d, uint64_t R, uint64_t rows,
               uint64_t Z, uint64_t rows_total, uint32_t box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[4] = {d, R, rows, Z};
    cuuint64_t strides[3] = {d * 2, R * d * 2, rows_total * d * 2};
    cuuint32_t box[4] = {64, 1, box_rows, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The window path on CTA pairs (cta_group::2): see swa_prefill_duo.cuh.
#include "swa_prefill_duo.cuh"

// Clusters of two CTAs of the CTA-pair kernel that fit on the device at once
// (0 if it cannot run), worked out once per device.
template <int HD, bool SHARED>
int duo_clusters()
{
    static std::atomic<int> known[kMaxDevices];  // 0: not yet known; else clusters + 1
    const int dev = current_device();
    if (dev < 0) return 0;
    const int k = known[dev].load(std::memory_order_acquire);
    if (k > 0) return k - 1;
    using L = LayoutD<HD, SHARED>;
    int n = 0;
    if (smem_opt_in<swa_prefill_bf16_duo_sm103<HD, SHARED>>(L::DYN_SMEM) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (num_sms() / 2));
        cfg.blockDim = dim3(NTHREADS2);
        cfg.dynamicSmemBytes = L::DYN_SMEM;
        if (cudaOccupancyMaxActiveClusters(&n, swa_prefill_bf16_duo_sm103<HD, SHARED>, &cfg) !=
            cudaSuccess)
            n = 0;
    }
    (void)cudaGetLastError();  // a refusal above is an answer, not an error to keep
    known[dev].store(n + 1, std::memory_order_release);
    return n;
}

// One launch of the CTA-pair kernel (window path, even group, H % 4 == 0);
// SWA_ERR_UNSUPPORTED if no cluster of two fits.
template <int HD, bool SHARED>
int launch_duo(const CUtensorMap &mq, const CUtensorMap &mkh, const CUtensorMap &mv,
               PrefillParams p, cudaStream_t stream)
{
    using L = LayoutD<HD, SHARED>;
    const int fit = duo_clusters<HD, SHARED>();
    if (fit <= 0) return SWA_ERR_UNSUPPORTED;
    p.num_items = p.B * (p.H / 4) * p.n_qt;
    const int clusters = p.num_items < fit ? p.num_items : fit;
    swa_prefill_bf16_duo_sm103<HD, SHARED>
        <<<2 * clusters, NTHREADS2, L::DYN_SMEM, stream>>>(mq, mkh, mv, p);
    return cudaGetLastError() == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
}

// One launch of the pair kernel: head pairs of an even group, or (QP) pairs of
// adjacent q tiles of one head for an odd group.
template <int HD, bool WALK, bool PAT, bool QP, bool SKEW = true>
int launch_pair(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                const CUtensorMap &mq2, const CUtensorMap &mk2, const CUtensorMap &mv2,
                PrefillParams p, int per_unit, cudaStream_t stream, int32_t *walk)
{
    using L2 = Layout2<HD>;
    if (smem_opt_in<swa_prefill_bf16_pair_sm103<HD, PAT, QP, SKEW, WALK>>(L2::DYN_SMEM) !=
        cudaSuccess)
        return SWA_ERR_CUDA;
    if constexpr (QP) {
        p.n_qt = (p.n + 2 * BM - 1) / (2 * BM);  // levels of q-tile pairs
        p.num_items = p.B * p.H * p.n_qt;
    } else {
        p.num_items = p.B * p.Hkv * (p.G / 2) * per_unit;
    }
    const int grid = p.num_items < num_sms() ? p.num_items : num_sms();
    swa_prefill_bf16_pair_sm103<HD, PAT, QP, SKEW, WALK>
        <<<grid, NTHREADS2, L2::DYN_SMEM, stream>>>(mq, mk, mv, mq2, mk2, mv2, p, walk);
    return cudaGetLastError() == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
}

template <int HD, bool WALK, bool PAT>
int launch_kernels(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                   const CUtensorMap &mq2, const CUtensorMap &mk2, const CUtensorMap &mv2,
                   PrefillParams p, int per_unit, cudaStream_t stream, int32_t *walk)
{
    // pair<QP, SKEW>(): one launch of that pair-kernel instantiation
    auto pair = [&](auto qp, auto skew) {
        return launch_pair<HD, WALK, PAT, decltype(qp)::value, decltype(skew)::value>(
            mq, mk, mv, mq2, mk2, mv2, p, per_unit, stream, walk);
    };
    using T = std::true_type;
    using F = std::false_type;
    if constexpr (!PAT) {
        // the window path: head pairs; an odd group pairs adjacent q tiles of one head
        return p.G % 2 == 0 ? pair(F{}, T{}) : pair(T{}, T{});
    } else {
        // the fixed patterns: head pairs for even groups, the single-head kernel
        // for odd ones.  An item's key tiles number about min(window, class
        // rows) / BN + 1: the skewed K/V protocol for four tiles' worth and more
        // (landmarks, dilated windows), one stage per tile below that (the
        // strided head's short classes).
        if (p.G % 2 == 0) {
            const int span = p.w < p.n_hi ? p.w : p.n_hi;
            return span >= 4 * BN ? pair(F{}, T{}) : pair(F{}, F{});
        }
        using L = Layout<HD>;
        if (smem_opt_in<swa_prefill_bf16_sm103<HD, PAT, WALK>>(L::DYN_SMEM) != cudaSuccess)
            return SWA_ERR_CUDA;
        p.num_items = p.B * p.H * per_unit;
        const int grid = p.num_items < num_sms() ? p.num_items : num_sms();
        swa_prefill_bf16_sm103<HD, PAT, WALK>
            <<<grid, NTHREADS, L::DYN_SMEM, stream>>>(mq, mk, mv, mq2, mk2, mv2, p, walk);
        return cudaGetLastError() == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
    }
}

template <int HD>
int launch_hd(const void *Q, const void *K, const void *V, void *O, float *lse, const float *sink,
              int B, int H, int Hkv, int n, int n_k, int w, int g, float scale,
              const int32_t *pos0, int R, int rl, cudaStream_t stream, int32_t *walk,
              bool cta_pairs)
{
    if (rl > 0) R = 1;
    const bool pat = R > 1 || rl > 0;
    // residue classes: class c has n_hi rows if c < rem, else n_lo
    const int n_hi = (n + R - 1) / R, n_lo = n / R, rem = n % R;
    const uint64_t ZQ = static_cast<uint64_t>(B) * H, ZK = static_cast<uint64_t>(B) * Hkv;
    // maps: tmX for classes below rem (and the landmark view), tmX2 for the rest
    CUtensorMap mq, mk, mv, mq2, mk2, mv2;
    bool ok;
    if (!pat) {
        ok = make_map_3d(&mq, Q, HD, n, ZQ, BM) && make_map_3d(&mk, K, HD, n_k, ZK, BN) &&
             make_map_3d(&mv, V, HD, n_k, ZK, BN);
        mq2 = mq;
        mk2 = mk;
        mv2 = mv;
    } else if (rl > 0) {
        // landmarks: Q, K, V as they are, and K, V as the stride-rl view whose
        // class 0 lists positions 0, rl, 2 rl, ... (ceil(n/rl) of them)
        const uint64_t nlm = (static_cast<uint64_t>(n_k) + rl - 1) / rl;
        ok = make_view(&mq2, Q, HD, 1, n, ZQ, n, BM) && make_view(&mk2, K, HD, 1, n_k, ZK, n_k, BN) &&
             make_view(&mv2, V, HD, 1, n_k, ZK, n_k, BN) &&
             make_view(&mk, K, HD, rl, nlm, ZK, n_k, BN) && make_view(&mv, V, HD, rl, nlm, ZK, n_k, BN);
        mq = mq2;
    } else {
        ok = make_view(&mq, Q, HD, R, n_hi, ZQ, n, BM) &&
             make_view(&mk, K, HD, R, n_hi, ZK, n_k, BN) &&
             make_view(&mv, V, HD, R, n_hi, ZK, n_k, BN);
        if (ok && n_lo > 0 && n_lo != n_hi) {
            ok = make_view(&mq2, Q, HD, R, n_lo, ZQ, n, BM) &&
                 make_view(&mk2, K, HD, R, n_lo, ZK, n_k, BN) &&
                 make_view(&mv2, V, HD, R, n_lo, ZK, n_k, BN);
        } else {
            mq2 = mq;
            mk2 = mk;
            mv2 = mv;
        }
    }
    if (!ok) return SWA_ERR_CUDA;
    PrefillParams p;
    p.B = B;
    p.H = H;
    p.Hkv = Hkv;
    p.n = n;
    p.n_k = n_k;
    p.pos0 = pos0;
    p.w = w;
    p.g = g;
    p.G = H / Hkv;
    p.R = R;
    p.rem = rem;
    p.n_hi = n_hi;
    p.n_lo = n_lo;
    p.rl = rl;
    p.n_qt = (n_hi + BM - 1) / BM;
    p.R_top = n_lo > (p.n_qt - 1) * BM ? R : rem;
    p.num_items = 0;
    // items per unit (query head or head pair) of one kv head of one sequence
    const int per_unit = p.R_top + (p.n_qt - 1) * R;
    p.sl2 = scale * 1.4426950408889634f;
    p.O = static_cast<__nv_bfloat16 *>(O);
    p.lse = lse;
    p.sink = sink;
    p.status = status_ptr();
    if (p.status == nullptr) return SWA_ERR_CUDA;
    p.wait_ns = TIMEOUT_NS;
    p.skip_first_kv = take_injected_stall(SWA_STALL_PREFILL, &p.wait_ns) ? 1 : 0;
#ifdef SWA_DEBUG
    {
        uint64_t unused = 0;
        p.dbg_orows = static_cast<long long>(B) * H * n -
                      (take_injected_stall(INJECT_SHRINK_BOUNDS, &unused) ? 1 : 0);
    }
#endif
    // the logged walk is a kernel of its own, so the product kernels carry no
    // per-tile check for it
    // the window path on CTA pairs, on request only (it measured 4-9% slower
    // than the pair kernel on the Mistral-like, Gemma-3-like and long layers):
    // d = 128, an even group, heads in quads
    if (cta_pairs) {
        if constexpr (HD == 128) {
            if (!pat && walk == nullptr && p.G % 2 == 0 && H % 4 == 0) {
                CUtensorMap mkh;
                if (!make_map_3d(&mkh, K, HD, n_k, ZK, BN / 2)) return SWA_ERR_CUDA;
                return p.G % 4 == 0 ? launch_duo<HD, true>(mq, mkh, mv, p, stream)
                                    : launch_duo<HD, false>(mq, mkh, mv, p, stream);
            }
        }
        return SWA_ERR_UNSUPPORTED;
    }
    auto launch = [&](auto walk_on, auto pat_on) {
        return launch_kernels<HD, decltype(walk_on)::value, decltype(pat_on)::value>(
            mq, mk, mv, mq2, mk2, mv2, p, per_unit, stream, walk);
    };
    using T = std::true_type;
    using F = std::false_type;
    if (walk != nullptr) return pat ? launch(T{}, T{}) : launch(T{}, F{});
    return pat ? launch(F{}, T{}) : launch(F{}, F{});
}

}  // namespace

int launch_prefill_bf16(const void *Q, const void *K, const void *V, void *O, float *lse,
                        const float *sink, int B, int H, int Hkv, int n, int n_k, int d, int w,
                        int g, float scale, const int32_t *pos0, int R, int rl,
                        cudaStream_t stream, int32_t *walk, bool cta_pairs)
{
    if (d == 128)
        return launch_hd<128>(Q, K, V, O, lse, sink, B, H, Hkv, n, n_k, w, g, scale, pos0, R, rl,
                              stream, walk, cta_pairs);
    if (d == 64)
        return launch_hd<64>(Q, K, V, O, lse, sink, B, H, Hkv, n, n_k, w, g, scale, pos0, R, rl,
                             stream, walk, cta_pairs);
    return SWA_ERR_UNSUPPORTED;
}

int launch_selftest_umma(const void *A, const void *Bk, const void *Bn, float *D1, float *D2,
                         cudaStream_t stream)
{
    CUtensorMap ma, mbk, mbn;
    if (!make_map_3d(&ma, A, 128, 128, 1, 128) || !make_map_3d(&mbk, Bk, 128, 128, 1, 128) ||
        !make_map_3d(&mbn, Bn, 128, 128, 1, 128))
        return SWA_ERR_CUDA;
    const int smem = 98304 + 64 + 1024;
    if (cudaFuncSetAttribute(swa_selftest_umma_sm103, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
        return SWA_ERR_CUDA;
    int *st = status_ptr();
    if (st == nullptr) return SWA_ERR_CUDA;
    swa_selftest_umma_sm103<<<1, 128, smem, stream>>>(
        ma, mbk, mbn, static_cast<const __nv_bfloat16 *>(A), D1, D2, st);
    return cudaGetLastError() == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
}

}  // namespace swa
