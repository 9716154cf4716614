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
// so the keys of one (sequence, kv head) are two contiguous runs of rows.
//
// Split pass (swa_decode_split): a persistent grid of P CTAs.  The slots of
// all (sequence, kv head) segments, laid end to end (B*Hkv*(w+g) rows), are
// cut into P equal contiguous ranges, one per CTA, so every CTA streams the
// same number of bytes whatever B, Hkv and w are.  In each CTA one producer
// thread copies the valid rows of its range, 64 at a time, into a ring of
// shared-memory stages with bulk asynchronous copies (cp.async.bulk, one per
// contiguous run of rows, completion on an mbarrier); four consumer warps take
// two groups of 8 rows of each stage each.  A consumer warp
//   * scores its 8 keys against the G query heads of the group with packed
//     fp32x2 FMAs (8 lanes per key row, q pre-scaled by scale*log2(e)),
//   * finishes the dot products with a reduce-scatter butterfly over the 8
//     lanes, so each lane ends with whole scores and every exp2 is computed
//     once,
//   * keeps an online softmax per head in base 2 whose reference maximum is
//     only raised when a score exceeds it by more than 2^8 (exact: the same
//     reference divides out at the end),
//   * and accumulates P.V with 16 lanes per value row.
// When its range leaves a segment, the CTA merges its warps and writes one
// partial (m, l, o) per head for that segment.
// Merge pass (swa_decode_merge): per (sequence, kv head) and head of the
// group, the log-sum-exp merge of the partials of the CTAs whose ranges met
// the segment.  It is launched as a programmatic dependent launch, so its
// launch overlaps the split pass; it waits for the split pass to complete
// before reading.  Its blocks are small (one head, HD threads, at most 64
// registers each), so one fits on each SM beside the two split CTAs and is
// already resident when the split pass ends.
#include <cmath>
#include <cstdlib>

#include "swa_internal.h"
#include "swa_ptx.cuh"

namespace swa {
namespace {

using namespace ptx;

constexpr int DEC_CWARPS = 4;                       // consumer warps per CTA
constexpr int DEC_THREADS = (DEC_CWARPS + 1) * 32;  // + one producer warp
constexpr int GROUP_ROWS = 8;                       // rows of one consumer-warp group
constexpr int DEC_GPW = 2;                          // groups per consumer warp per stage
constexpr int STAGE_ROWS = DEC_CWARPS * GROUP_ROWS * DEC_GPW;
constexpr int DEC_CTAS_PER_SM = 2;
constexpr int DEC_STAGE_BUDGET = 96 * 1024;         // shared memory for the stage ring
constexpr int MIN_SLOTS_PER_CTA = 64;
constexpr float RESCALE_LOG2 = 8.0f;
constexpr float M_EMPTY = -1.0e30f;  // running max before any key (finite: no inf-inf)
constexpr uint64_t DEC_TIMEOUT_NS = 2000000000ull;

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint64_t pk2(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void upk2(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// 16 bytes of T as fp32 pairs (element 2i in the low half of pair i).
template <typename T>
struct Unpack;
template <>
struct Unpack<__nv_bfloat16> {
    static constexpr int PAIRS = 4;
    __device__ static void run(const uint4 &u, uint64_t (&o)[4])
    {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
            o[k] = pk2(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xFFFF0000u));
    }
    __device__ static float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
    __device__ static __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};
template <>
struct Unpack<float> {
    static constexpr int PAIRS = 2;
    __device__ static void run(const uint4 &u, uint64_t (&o)[2])
    {
        o[0] = pk2(__uint_as_float(u.x), __uint_as_float(u.y));
        o[1] = pk2(__uint_as_float(u.z), __uint_as_float(u.w));
    }
    __device__ static float to_f(float x) { return x; }
    __device__ static float from_f(float x) { return x; }
};

template <typename T, int HD, int G>
struct DecCfg {
    static constexpr int RB = HD * static_cast<int>(sizeof(T));  // bytes per cache row
    static constexpr int EPC = 16 / static_cast<int>(sizeof(T));  // elements per 16 bytes
    // key rows: 8 lanes per row, 4 rows per pass, 2 passes per 8-row group
    static constexpr int EK = HD / 8;     // elements of a key row per lane
    static constexpr int CPL = EK / EPC;  // 16-byte chunks of a key row per lane
    static constexpr int KPL = GROUP_ROWS / 4;  // key rows per lane per group
    static constexpr int NV = KPL * G;    // partial dot products per lane
    static constexpr int NR = NV >= 8 ? NV / 8 : 1;  // whole scores per lane after the butterfly
    // value rows: 16 lanes per row, 2 rows per pass, 4 passes per group
    static constexpr int EV = HD / 16;    // columns per lane
    static constexpr int VB = EV * static_cast<int>(sizeof(T));  // bytes per lane per value row
    static constexpr int STAGE_BYTES = 2 * STAGE_ROWS * RB;
    static constexpr int NS_RAW = (DEC_STAGE_BUDGET) / STAGE_BYTES;
    static constexpr int NS = NS_RAW < 2 ? 2 : (NS_RAW > 8 ? 8 : NS_RAW);  // stages
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = NS * STAGE_ROWS * RB;
    static constexpr int BAR_OFF = 2 * NS * STAGE_ROWS * RB;  // full[NS], empty[NS], sync[2]
    static constexpr int FLAG_OFF = BAR_OFF + (2 * NS + 2) * 8;
    static constexpr int P_OFF = FLAG_OFF + 16;                  // [warp][8 rows][G] fp32 pairs
    static constexpr int P_BYTES = GROUP_ROWS * G * 8;
    static constexpr int F_OFF = P_OFF + DEC_CWARPS * P_BYTES;   // [warp][G][HD + 2] fp32
    static constexpr int BYTES = F_OFF + DEC_CWARPS * G * (HD + 2) * 4;
    static constexpr int MIN_BLOCKS = G >= 8 ? 1 : DEC_CTAS_PER_SM;
    static_assert(CPL >= 1 && EK % EPC == 0, "key lane mapping");
    static_assert(VB == 8 || VB == 16 || VB == 32, "value lane mapping");
};

struct DecodeParams {
    int B, H, Hkv, w, g;
    int G;          // query heads per kv head
    int nsub, Gs;   // sub-groups per kv head and real heads per sub-group (decode_groups)
    int Hv;         // virtual kv heads, Hkv * nsub: one segment per (sequence, virtual head)
    int P;          // CTAs of the split pass
    long long T;    // B * Hv * (w + g) slots, laid end to end
    float sl2;      // scale * log2(e)
    const int32_t *pos;
    int *status;    // device status word (a negative position is reported there)
    float *ws;      // partials [P + B*Hv][Gp][HD + 2]: m, l, o
    void *O;        // [B][H][d]
    float *lse;     // [B][H] or null
    const float *sink;  // per-head sink logits [H] or null
    uint64_t wait_ns;   // limit of every bounded wait of the roles (2 s unless a test sets it)
    int skip_first_stage;  // test injection: the first stage's copies are left out (see swa.h)
};

__host__ __device__ __forceinline__ long long cta_begin(long long T, int P, int c)
{
    const long long base = T / P, rem = T % P;
    return c * base + (c < rem ? c : rem);
}
// The CTA whose range holds slot x.
__device__ __forceinline__ int cta_of(long long T, int P, long long x)
{
    const long long base = T / P, rem = T % P;
    const long long big = rem * (base + 1);
    return static_cast<int>(x < big ? x / (base + 1) : rem + (x - big) / base);
}

struct Seg {
    int b, kvh, bk;
    int h0;      // the first query head of the segment's sub-group
    int nh;      // its real heads (the rest, up to the group width, are padding)
    int ring_lo, ring_hi;  // valid ring rows of this CTA's share of the segment
    int sink_lo, sink_hi;  // valid sink rows (slot numbers w..)
    bool bad_pos;
};

__device__ __forceinline__ Seg make_seg(const DecodeParams &p, long long bk, int t0, int t1)
{
    Seg s;
    s.bk = static_cast<int>(bk);
    s.b = static_cast<int>(bk / p.Hv);
    const int v = static_cast<int>(bk % p.Hv);
    s.kvh = v / p.nsub;
    const int u = v % p.nsub;
    s.h0 = s.kvh * p.G + u * p.Gs;
    s.nh = min(p.Gs, p.G - u * p.Gs);
    // 64-bit: pos may be as large as INT32_MAX
    long long pos = __ldg(p.pos + s.b);
    s.bad_pos = pos < 0;
    if (pos < 0) pos = -1;
    const int nring = static_cast<int>(pos + 1 < p.w ? pos + 1 : p.w);
    long long ns = pos - p.w + 1;
    const int nsink = static_cast<int>(ns < 0 ? 0 : (ns > p.g ? p.g : ns));
    s.ring_lo = t0;
    s.ring_hi = t1 < nring ? t1 : nring;
    s.sink_lo = t0 > p.w ? t0 : p.w;
    s.sink_hi = t1 < p.w + nsink ? t1 : p.w + nsink;
    return s;
}

// Walks this CTA's range segment by segment and stage by stage (at most
// STAGE_ROWS contiguous valid rows of one segment per stage).  The producer
// and the consumers run the same walk, so they agree on every stage.
// on_stage returns false to stop (a bounded wait ran out).
template <class Begin, class Stage, class End>
__device__ __forceinline__ bool walk(const DecodeParams &p, Begin on_begin, Stage on_stage,
                                     End on_end)
{
    const long long S = static_cast<long long>(p.w) + p.g;
    const long long lo = cta_begin(p.T, p.P, blockIdx.x), hi = cta_begin(p.T, p.P, blockIdx.x + 1);
    int it = 0;
    for (long long x = lo; x < hi;) {
        const long long bk = x / S, base = bk * S;
        const int t0 = static_cast<int>(x - base);
        const int t1 = static_cast<int>(hi - base < S ? hi - base : S);
        const Seg s = make_seg(p, bk, t0, t1);
        on_begin(s);
        for (int r = s.ring_lo; r < s.ring_hi; r += STAGE_ROWS, ++it)
            if (!on_stage(it, s, r, min(STAGE_ROWS, s.ring_hi - r))) return false;
        for (int r = s.sink_lo; r < s.sink_hi; r += STAGE_ROWS, ++it)
            if (!on_stage(it, s, r, min(STAGE_ROWS, s.sink_hi - r))) return false;
        on_end(s);
        x = base + t1;
    }
    return true;
}

// One level of the reduce-scatter butterfly over the lanes that differ in
// `mask`: with N >= 2 values the lane keeps half of them (the upper half if
// its mask bit is set) and adds the partner's copy of that half; with one
// value left it adds the partner's value (all-reduce).
template <int N, int MASK>
__device__ __forceinline__ void rs_level(float *v, int lane)
{
    if constexpr (N >= 2) {
        const bool up = (lane & MASK) != 0;
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            const float send = up ? v[i] : v[i + N / 2];
            const float keep = up ? v[i + N / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, MASK);
        }
    } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], MASK);
    }
}

template <typename T, int HD, int G>
__global__ void __launch_bounds__(DEC_THREADS, DecCfg<T, HD, G>::MIN_BLOCKS)
    swa_decode_split(const T *__restrict__ q, const T *__restrict__ Kc, const T *__restrict__ Vc,
                     const DecodeParams p)
{
    using C = DecCfg<T, HD, G>;
    using U = Unpack<T>;
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t sb = smem_u32(smem);
    const uint32_t bars = sb + C::BAR_OFF;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::FLAG_OFF);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#define FULL(s) (bars + 8u * static_cast<uint32_t>(s))
#define EMPTY(s) (bars + 8u * static_cast<uint32_t>(C::NS + (s)))
#define SYNC(i) (bars + 8u * static_cast<uint32_t>(2 * C::NS + (i)))

    // let the merge pass be scheduled as soon as every CTA of this grid runs
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(FULL(s), 1);
            mbar_init(EMPTY(s), DEC_CWARPS);
        }
        mbar_init(SYNC(0), DEC_CWARPS);
        mbar_init(SYNC(1), DEC_CWARPS);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const size_t S = static_cast<size_t>(p.w) + p.g;

    if (warp == DEC_CWARPS) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        int last_par[C::NS];
#pragma unroll
        for (int s = 0; s < C::NS; ++s) last_par[s] = -1;
        const bool ok = walk(
            p, [](const Seg &) {},
            [&](int it, const Seg &s, int row, int count) -> bool {
                const int slot = it % C::NS;
                const uint32_t ph = (it / C::NS) & 1;
                if (!mbar_wait(EMPTY(slot), ph ^ 1, abort_flag, p.status, p.wait_ns))
                    return false;
                // test injection: this stage's copies never start, so the
                // consumers' wait for it runs out (nothing is in flight to drain)
                if (p.skip_first_stage && it == 0) return true;
                // debug builds: the rows lie in the segment's cache (a copy that
                // fails the check is not made, and the consumers' wait runs out)
                if (!SWA_BOUNDS(s.b < p.B && s.kvh < p.Hkv && row >= 0 &&
                                    static_cast<size_t>(row) + count <= S,
                                p.status))
                    return true;
                const uint32_t bytes = static_cast<uint32_t>(count * C::RB);
                mbar_expect_tx(FULL(slot), 2 * bytes);
                const size_t off = ((static_cast<size_t>(s.b) * p.Hkv + s.kvh) * S + row) * HD;
                const uint32_t dk = sb + C::K_OFF + slot * STAGE_ROWS * C::RB;
                const uint32_t dv = sb + C::V_OFF + slot * STAGE_ROWS * C::RB;
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
                    " [%0], [%1], %2, [%3];" ::"r"(dk),
                    "l"(Kc + off), "r"(bytes), "r"(FULL(slot))
                    : "memory");
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
                    " [%0], [%1], %2, [%3];" ::"r"(dv),
                    "l"(Vc + off), "r"(bytes), "r"(FULL(slot))
                    : "memory");
                last_par[slot] = static_cast<int>(ph);
                return true;
            },
            [](const Seg &) {});
        if (!ok) {
            // stopped early: wait (bounded, ignoring the abort flag) for every
            // copy still in flight before the CTA may exit
            for (int s = 0; s < C::NS; ++s)
                if (last_par[s] >= 0)
                    mbar_wait(FULL(s), last_par[s], nullptr, nullptr, DEC_TIMEOUT_NS);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int rg = lane >> 3, cidx = lane & 7;   // key layout: row group, lane in row
    const int vr = lane >> 4, vc = lane & 15;    // value layout
    const int rot = (cidx * C::CPL) >> 3;        // chunk rotation: conflict-free smem reads
    const int j0 = (cidx * C::NV) >> 3;          // first whole score this lane holds
    const bool owner = C::NV >= 8 || (cidx & ((8 / C::NV) - 1)) == 0;
    uint64_t *Pw = reinterpret_cast<uint64_t *>(smem + C::P_OFF + warp * C::P_BYTES);
    float *Fl = reinterpret_cast<float *>(smem + C::F_OFF);

    uint64_t q2[G][C::EK / 2];       // this lane's key-layout slice of q, times scale*log2(e)
    uint64_t acc[G][C::EV / 2];      // unnormalised output columns vc*EV .. (value layout)
    float m[G];                      // reference maximum per head (warp-uniform)
    float mv[C::NR], lv[C::NR];      // per held score: its head's reference, its sum of p

    auto on_begin = [&](const Seg &s) {
        if (s.bad_pos && threadIdx.x == 0) atomicOr(p.status, DEV_ERR_BAD_POS);
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            // a padding head of the sub-group scores with q = 0 (never written out)
            const bool real = hh < s.nh &&
                              SWA_BOUNDS(s.b < p.B && s.h0 + hh < p.H, p.status);
            const T *qr = q + (static_cast<size_t>(s.b) * p.H + s.h0 + (real ? hh : 0)) * HD;
#pragma unroll
            for (int c = 0; c < C::CPL; ++c) {
                const int chunk = cidx * C::CPL + ((c + rot) % C::CPL);
#pragma unroll
                for (int e = 0; e < C::EPC; e += 2)
                    q2[hh][(c * C::EPC + e) / 2] =
                        real ? pk2(U::to_f(qr[chunk * C::EPC + e]) * p.sl2,
                                   U::to_f(qr[chunk * C::EPC + e + 1]) * p.sl2)
                             : pk2(0.f, 0.f);
            }
            m[hh] = M_EMPTY;
#pragma unroll
            for (int e = 0; e < C::EV / 2; ++e) acc[hh][e] = 0;
        }
#pragma unroll
        for (int t = 0; t < C::NR; ++t) {
            mv[t] = M_EMPTY;
            lv[t] = 0.f;
        }
    };

    auto on_stage = [&](int it, const Seg &, int, int count) -> bool {
        const int slot = it % C::NS;
        const uint32_t ph = (it / C::NS) & 1;
        if (!__all_sync(0xffffffffu,
                        mbar_wait(FULL(slot), ph, abort_flag, p.status, p.wait_ns)))
            return false;
#pragma unroll 1
        for (int gi = 0; gi < DEC_GPW; ++gi) {
        const int row0 = (gi * DEC_CWARPS + warp) * GROUP_ROWS;
        const int nrows = count - row0;  // rows of this warp's group that exist (may be <= 0)
        if (nrows > 0) {
            const uint8_t *kst = smem + C::K_OFF + (slot * STAGE_ROWS + row0) * C::RB;
            const uint8_t *vst = smem + C::V_OFF + (slot * STAGE_ROWS + row0) * C::RB;
            // ---- scores: 8 lanes per key row
            float sv[C::NV];
#pragma unroll
            for (int k = 0; k < C::KPL; ++k) {
                const int row = 4 * k + rg;
                uint64_t kp[C::EK / 2];
#pragma unroll
                for (int c = 0; c < C::CPL; ++c) {
                    const int chunk = cidx * C::CPL + ((c + rot) % C::CPL);
                    const uint4 u = *reinterpret_cast<const uint4 *>(kst + row * C::RB + chunk * 16);
                    uint64_t pr[U::PAIRS];
                    U::run(u, pr);
#pragma unroll
                    for (int e = 0; e < U::PAIRS; ++e) kp[c * U::PAIRS + e] = pr[e];
                }
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    uint64_t a = 0;
#pragma unroll
                    for (int i = 0; i < C::EK / 2; ++i) a = ffma2(q2[hh][i], kp[i], a);
                    float lo, hi;
                    upk2(a, lo, hi);
                    sv[k * G + hh] = lo + hi;
                }
            }
            rs_level<C::NV, 4>(sv, lane);
            rs_level<(C::NV >= 2 ? C::NV / 2 : 1), 2>(sv, lane);
            rs_level<(C::NV >= 4 ? C::NV / 4 : 1), 1>(sv, lane);
            // sv[0 .. NR-1]: whole scores j0 .. j0+NR-1, score j = (key k = j / G, head j % G)
#pragma unroll
            for (int t = 0; t < C::NR; ++t) {
                const int row = 4 * ((j0 + t) / G) + rg;
                if (row >= nrows) sv[t] = -INFINITY;
            }
            bool need = false;
#pragma unroll
            for (int t = 0; t < C::NR; ++t) need |= sv[t] > mv[t] + RESCALE_LOG2;
            if (__any_sync(0xffffffffu, need)) {
                // raise the reference maximum of every head to the running maximum
                float gm[G];
#pragma unroll
                for (int hh = 0; hh < G; ++hh) gm[hh] = -INFINITY;
#pragma unroll
                for (int t = 0; t < C::NR; ++t)
#pragma unroll
                    for (int hh = 0; hh < G; ++hh)
                        if ((j0 + t) % G == hh) gm[hh] = fmaxf(gm[hh], sv[t]);
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1)
                        gm[hh] = fmaxf(gm[hh], __shfl_xor_sync(0xffffffffu, gm[hh], off));
                    const float mn = fmaxf(m[hh], gm[hh]);
                    const float alpha = ex2(m[hh] - mn);
                    m[hh] = mn;
                    const uint64_t a2 = pk2(alpha, alpha);
#pragma unroll
                    for (int e = 0; e < C::EV / 2; ++e) acc[hh][e] = fmul2(acc[hh][e], a2);
#pragma unroll
                    for (int t = 0; t < C::NR; ++t)
                        if ((j0 + t) % G == hh) {
                            lv[t] *= alpha;
                            mv[t] = mn;
                        }
                }
            }
            // ---- probabilities to shared memory (fp32 pairs p, p), one writer per score
#pragma unroll
            for (int t = 0; t < C::NR; ++t) {
                const float pr = ex2(sv[t] - mv[t]);
                if (owner) {
                    lv[t] += pr;
                    const int j = j0 + t;
                    Pw[(4 * (j / G) + rg) * G + (j % G)] = pk2(pr, pr);
                }
            }
            __syncwarp();
            // ---- P.V: 16 lanes per value row
#pragma unroll
            for (int k = 0; k < GROUP_ROWS / 2; ++k) {
                const int row = 2 * k + vr;
                uint64_t v2[C::EV / 2];
                const uint8_t *src = vst + row * C::RB + vc * C::VB;
                if constexpr (C::VB == 8) {
                    const uint2 u = *reinterpret_cast<const uint2 *>(src);
                    uint64_t pr[U::PAIRS];
                    U::run(make_uint4(u.x, u.y, 0u, 0u), pr);
#pragma unroll
                    for (int e = 0; e < C::EV / 2; ++e) v2[e] = pr[e];
                } else {
#pragma unroll
                    for (int c = 0; c < C::VB / 16; ++c) {
                        const uint4 u = *reinterpret_cast<const uint4 *>(src + c * 16);
                        uint64_t pr[U::PAIRS];
                        U::run(u, pr);
#pragma unroll
                        for (int e = 0; e < U::PAIRS; ++e) v2[c * U::PAIRS + e] = pr[e];
                    }
                }
                if (row >= nrows) {
                    // a row past the stage's end: stale shared memory, and p = 0
#pragma unroll
                    for (int e = 0; e < C::EV / 2; ++e) v2[e] = 0;
                }
                const uint64_t *prow = Pw + row * G;
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    const uint64_t pp = prow[hh];
#pragma unroll
                    for (int e = 0; e < C::EV / 2; ++e) acc[hh][e] = ffma2(pp, v2[e], acc[hh][e]);
                }
            }
        }
        __syncwarp();  // the warp's P rows are reused by its next group
        }
        if (lane == 0) mbar_arrive(EMPTY(slot));
        return true;
    };

    // the consumer warps meet at a segment's end through two mbarriers (bounded
    // waits, so a warp that stopped early cannot leave the others hanging)
    int nflush = 0;
    auto cta_sync = [&](int which) -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(SYNC(which));
        return __all_sync(0xffffffffu, mbar_wait(SYNC(which), nflush & 1, abort_flag, p.status,
                                                 p.wait_ns));
    };

    auto on_end = [&](const Seg &s) {
        // this warp's (m, l, o) per head into shared memory
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            float lh = 0.f;
#pragma unroll
            for (int t = 0; t < C::NR; ++t)
                if ((j0 + t) % G == hh && owner) lh += lv[t];
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) lh += __shfl_xor_sync(0xffffffffu, lh, off);
            float *f = Fl + (warp * G + hh) * (HD + 2);
#pragma unroll
            for (int e = 0; e < C::EV / 2; ++e) {
                float lo, hi;
                upk2(acc[hh][e], lo, hi);
                lo += __shfl_xor_sync(0xffffffffu, lo, 16);
                hi += __shfl_xor_sync(0xffffffffu, hi, 16);
                if (vr == 0) {
                    f[2 + vc * C::EV + 2 * e] = lo;
                    f[2 + vc * C::EV + 2 * e + 1] = hi;
                }
            }
            if (lane == 0) {
                f[0] = m[hh];
                f[1] = lh;
            }
        }
        if (!cta_sync(0)) return;
        // the CTA's partial for this segment
        float *wsp = p.ws + (static_cast<size_t>(blockIdx.x) + s.bk) * G * (HD + 2);
        // debug builds: the partial's index lies in the workspace (ctas + B*Hv partials)
        const bool w_ok = SWA_BOUNDS(static_cast<long long>(blockIdx.x) + s.bk <
                                         static_cast<long long>(p.P) + static_cast<long long>(p.B) * p.Hv,
                                     p.status);
        for (int x = threadIdx.x; w_ok && x < G * (HD + 2); x += DEC_CWARPS * 32) {
            const int hh = x / (HD + 2), col = x % (HD + 2);
            float M = M_EMPTY;
#pragma unroll
            for (int wv = 0; wv < DEC_CWARPS; ++wv) M = fmaxf(M, Fl[(wv * G + hh) * (HD + 2)]);
            float r = M;
            if (col > 0) {
                r = 0.f;
#pragma unroll
                for (int wv = 0; wv < DEC_CWARPS; ++wv) {
                    const float *f = Fl + (wv * G + hh) * (HD + 2);
                    r += ex2(f[0] - M) * f[col];
                }
            }
            wsp[x] = r;
        }
        cta_sync(1);
        ++nflush;
    };

    walk(p, on_begin, on_stage, on_end);
#undef FULL
#undef EMPTY
#undef SYNC
}

// Block (segment bk, head hh of the sub-group); thread col is one output column.
template <typename T, int HD, int G>
__global__ void __launch_bounds__(HD, 8) swa_decode_merge(const DecodeParams p)
{
    using U = Unpack<T>;
    // wait until the split pass has completed and its writes are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int bk = blockIdx.x;
    const int hh = blockIdx.y, col = threadIdx.x;
    const long long S = static_cast<long long>(p.w) + p.g;
    int c_lo = cta_of(p.T, p.P, bk * S), c_hi = cta_of(p.T, p.P, bk * S + S - 1);
    // debug builds: the partials lie in the workspace (else none is read)
    if (!SWA_BOUNDS(c_lo >= 0 && c_hi < p.P, p.status)) c_hi = c_lo - 1;
    // the first NU partials (usually all of them) are loaded in one round
    constexpr int NU = 4;
    float mv[NU], lv[NU], ov[NU];
#pragma unroll
    for (int k = 0; k < NU; ++k) {
        mv[k] = M_EMPTY;
        lv[k] = 0.f;
        ov[k] = 0.f;
        if (c_lo + k <= c_hi) {
            const float *x = p.ws + ((static_cast<size_t>(c_lo + k) + bk) * G + hh) * (HD + 2);
            mv[k] = x[0];
            lv[k] = x[1];
            ov[k] = x[2 + col];
        }
    }
    float M = fmaxf(fmaxf(mv[0], mv[1]), fmaxf(mv[2], mv[3]));
    for (int c = c_lo + NU; c <= c_hi; ++c)
        M = fmaxf(M, p.ws[((static_cast<size_t>(c) + bk) * G + hh) * (HD + 2)]);
    float L = 0.f, o = 0.f;
#pragma unroll
    for (int k = 0; k < NU; ++k) {
        const float sc = ex2(mv[k] - M);
        L += sc * lv[k];
        o += sc * ov[k];
    }
    for (int c = c_lo + NU; c <= c_hi; ++c) {
        const float *x = p.ws + ((static_cast<size_t>(c) + bk) * G + hh) * (HD + 2);
        const float sc = ex2(x[0] - M);
        L += sc * x[1];
        o += sc * x[2 + col];
    }
    const int b = bk / p.Hv, v = bk % p.Hv, u = v % p.nsub;
    if (hh >= min(p.Gs, p.G - u * p.Gs)) return;  // a padding head of the sub-group
    const int h = (v / p.nsub) * p.G + u * p.Gs + hh;
    const size_t bh = static_cast<size_t>(b) * p.H + h;
    float row_lse;
    const float f = L > 0.f ? finish_row(M, L, p.sink, h, &row_lse) : 0.f;
    if (!(L > 0.f)) row_lse = -INFINITY;
    if (!SWA_BOUNDS(bh < static_cast<size_t>(p.B) * p.H, p.status)) return;
    static_cast<T *>(p.O)[bh * HD + col] = U::from_f(o * f);
    if (col == 0 && p.lse != nullptr) p.lse[bh] = row_lse;
}

template <typename T, int HD, int G>
int launch_decode_t(const void *q, const void *Kc, const void *Vc, const DecodeParams &p,
                    cudaStream_t stream)
{
    using C = DecCfg<T, HD, G>;
    if (smem_opt_in<swa_decode_split<T, HD, G>>(C::BYTES) != cudaSuccess) return SWA_ERR_CUDA;
    swa_decode_split<T, HD, G><<<p.P, DEC_THREADS, C::BYTES, stream>>>(
        static_cast<const T *>(q), static_cast<const T *>(Kc), static_cast<const T *>(Vc), p);
    if (cudaGetLastError() != cudaSuccess) return SWA_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.B * p.Hv), static_cast<unsigned>(G));
    cfg.blockDim = dim3(HD);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, swa_decode_merge<T, HD, G>, p) != cudaSuccess) return SWA_ERR_CUDA;
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
        // invalid: a negative start, or one whose last position p0+T_new-1
        // passes INT32_MAX; write nothing and report it
        if (p0 < 0 || p0 > INT32_MAX - T_new) {
            if (c == 0 && t == 0) atomicOr(status, DEV_ERR_BAD_POS);
            continue;
        }
        const int p = p0 + t;
        const uint4 kv = reinterpret_cast<const uint4 *>(kn + row * HD)[c];
        const uint4 vv = reinterpret_cast<const uint4 *>(vn + row * HD)[c];
        T *kbase = Kc + bk * slots * HD;
        T *vbase = Vc + bk * slots * HD;
        if (t >= T_new - w && SWA_BOUNDS(p % w < w, status)) {  // the last w survive in the ring
            const size_t slot = static_cast<size_t>(p % w);
            reinterpret_cast<uint4 *>(kbase + slot * HD)[c] = kv;
            reinterpret_cast<uint4 *>(vbase + slot * HD)[c] = vv;
        }
        if (p < g && SWA_BOUNDS(static_cast<size_t>(w) + p < slots, status)) {
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

int decode_ctas(int B, int H, int Hkv, int w, int g, int num_splits)
{
    const long long Hv = static_cast<long long>(Hkv) * decode_groups(H / Hkv).nsub;
    const long long T = static_cast<long long>(B) * Hv * (static_cast<long long>(w) + g);
    long long P;
    if (num_splits > 0) {
        // about num_splits CTAs per (sequence, virtual kv head) segment
        P = static_cast<long long>(num_splits) * B * Hv;
    } else {
        // one resident wave, each CTA streaming at least MIN_SLOTS_PER_CTA rows
        P = static_cast<long long>(DEC_CTAS_PER_SM) * num_sms();
        const long long cap = T / MIN_SLOTS_PER_CTA;
        if (P > cap) P = cap;
    }
    if (P > T) P = T;
    if (P > (1LL << 30)) P = 1LL << 30;
    if (P < 1) P = 1;
    return static_cast<int>(P);
}

size_t decode_workspace_bytes(int B, int H, int Hkv, int d, int ctas)
{
    // one partial (m, l, o[d]) per head of the padded sub-group for every
    // (CTA, segment) pair that meets: at most ctas + B*Hv - 1 of them, indexed
    // cta + segment
    const DecodeGroups dg = decode_groups(H / Hkv);
    return (static_cast<size_t>(ctas) + static_cast<size_t>(B) * Hkv * dg.nsub) * dg.Gp *
           (static_cast<size_t>(d) + 2) * sizeof(float);
}

int launch_decode(const void *q, const void *Kc, const void *Vc, const int32_t *pos,
                  const float *sink, int B, int H,
                  int Hkv, int d, int w, int g, float scale, void *O, float *lse, swa_dtype dt,
                  int ctas, void *ws, cudaStream_t stream)
{
    DecodeParams p;
    p.B = B;
    p.H = H;
    p.Hkv = Hkv;
    p.w = w;
    p.g = g;
    const DecodeGroups dg = decode_groups(H / Hkv);
    p.G = H / Hkv;
    p.nsub = dg.nsub;
    p.Gs = dg.Gs;
    p.Hv = Hkv * dg.nsub;
    p.P = ctas;
    p.T = static_cast<long long>(B) * p.Hv * (static_cast<long long>(w) + g);
    p.sl2 = scale * 1.4426950408889634f;
    p.pos = pos;
    p.status = status_ptr();
    if (p.status == nullptr) return SWA_ERR_CUDA;
    p.ws = static_cast<float *>(ws);
    p.O = O;
    p.lse = lse;
    p.sink = sink;
    p.wait_ns = DEC_TIMEOUT_NS;
    p.skip_first_stage = take_injected_stall(SWA_STALL_DECODE, &p.wait_ns) ? 1 : 0;
    const int G = dg.Gp;  // the kernels' group width
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
