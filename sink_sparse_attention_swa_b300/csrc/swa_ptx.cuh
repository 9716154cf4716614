// swa_ptx.cuh -- thin inline-PTX wrappers for the sm_103a features the
// kernels use: mbarriers with bounded waits, TMA (cp.async.bulk.tensor),
// tensor memory (tcgen05.alloc/ld/st) and the 5th-generation tensor-core MMA
// (tcgen05.mma, kind::f16).  Encodings follow the public PTX ISA.
#pragma once

#include <cstdint>

#include <cuda.h>  // CUtensorMap (type only; the driver is reached at run time)
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace swa {
namespace ptx {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase of parity `parity` to complete.  Gives up after
// `timeout_ns` (or as soon as *abort is set), records DEV_ERR_TIMEOUT in the
// device status word on a timeout, sets *abort so that the CTA's other roles
// stop too, and returns false.  No trap, no endless spin.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          int *status, uint64_t timeout_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31u) == 0) {
            if (abort != nullptr && *abort) return false;
            if (globaltimer_ns() - t0 > timeout_ns) {
                if (abort != nullptr) *abort = 1;
                if (status != nullptr) atomicOr(status, 1);
                return false;
            }
        }
    }
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_prefetch(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load of one box into shared memory, completing `bytes` on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1, int c2)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// 4-D tiled load of one box into shared memory, completing on an mbarrier.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1, int c2, int c3)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// 3-D tiled store of one box from shared memory (bulk-group completion).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int c0, int c1,
                                             int c2)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::
            "l"(reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0()
{
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Make generic-proxy writes to shared memory visible to the async proxy
// (tensor core / TMA reads of data written by ordinary stores).
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ tensor memory
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive once on `bar` when every tcgen05 async operation this thread issued
// so far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The same two MMAs and the commit, issued by one lane elected from the
// calling warp (elect.sync); the whole warp executes the call.  Issuing from a
// converged warp this way takes the MMA issue path about a quarter fewer
// cycles per instruction than a loop that only lane 0 runs.
__device__ __forceinline__ void mma_ss_e(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_ts_e(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tc_commit_e(uint32_t bar)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}

// Grouped issue: one asm block elects a lane once and issues a whole K-loop
// of MMAs, with the k-step offsets added to the low word of each shared-memory
// descriptor (the start-address field; these offsets never carry out of it).
// One instruction stream with independent adds keeps the issuing warp short.
// S = A * B^T over K = 16*NK with both operands K-major in 128-byte swizzled
// 64-column chunks of 128 rows (16 KB apart): k-step ks adds
// ((ks>>2)*16384 + (ks&3)*32) >> 4 to both descriptors' start address.
template <int NK>
__device__ __forceinline__ void mma_ss_group(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc)
{
    const uint32_t al = static_cast<uint32_t>(a), ah = static_cast<uint32_t>(a >> 32);
    const uint32_t bl = static_cast<uint32_t>(b), bh = static_cast<uint32_t>(b >> 32);
#define SWA_MMA_SS(OFF) \
    "add.u32 xl, %1, " #OFF ";\n\tadd.u32 yl, %3, " #OFF ";\n\t" \
    "mov.b64 xd, {xl, %2};\n\tmov.b64 yd, {yl, %4};\n\t" \
    "@e tcgen05.mma.cta_group::1.kind::f16 [%0], xd, yd, %5, t;\n\t"
    if constexpr (NK == 8) {
        asm volatile("{\n\t.reg .pred e, f, t;\n\t.reg .b32 xl, yl;\n\t.reg .b64 xd, yd;\n\t"
                     "elect.sync _|e, 0xffffffff;\n\t"
                     "setp.ne.b32 f, %5, %5;\n\tsetp.eq.b32 t, %5, %5;\n\t"
                     "mov.b64 xd, {%1, %2};\n\tmov.b64 yd, {%3, %4};\n\t"
                     "@e tcgen05.mma.cta_group::1.kind::f16 [%0], xd, yd, %5, f;\n\t"
                     SWA_MMA_SS(2) SWA_MMA_SS(4) SWA_MMA_SS(6) SWA_MMA_SS(1024) SWA_MMA_SS(1026)
                     SWA_MMA_SS(1028) SWA_MMA_SS(1030) "}\n" ::"r"(d),
                     "r"(al), "r"(ah), "r"(bl), "r"(bh), "r"(idesc)
                     : "memory");
    } else {
        asm volatile("{\n\t.reg .pred e, f, t;\n\t.reg .b32 xl, yl;\n\t.reg .b64 xd, yd;\n\t"
                     "elect.sync _|e, 0xffffffff;\n\t"
                     "setp.ne.b32 f, %5, %5;\n\tsetp.eq.b32 t, %5, %5;\n\t"
                     "mov.b64 xd, {%1, %2};\n\tmov.b64 yd, {%3, %4};\n\t"
                     "@e tcgen05.mma.cta_group::1.kind::f16 [%0], xd, yd, %5, f;\n\t"
                     SWA_MMA_SS(2) SWA_MMA_SS(4) SWA_MMA_SS(6) "}\n" ::"r"(d),
                     "r"(al), "r"(ah), "r"(bl), "r"(bh), "r"(idesc)
                     : "memory");
    }
#undef SWA_MMA_SS
}
// O (+)= P * V over K = 128 keys: P in tensor memory (8 columns per k-step),
// V N-major in shared memory (k-step ks adds ks*16 rows * 128 B >> 4 = 128).
__device__ __forceinline__ void mma_ts_group8(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                              uint32_t acc0)
{
    const uint32_t bl = static_cast<uint32_t>(b), bh = static_cast<uint32_t>(b >> 32);
#define SWA_MMA_TS(AO, BO) \
    "add.u32 ta, %1, " #AO ";\n\tadd.u32 yl, %2, " #BO ";\n\tmov.b64 yd, {yl, %3};\n\t" \
    "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], yd, %4, t;\n\t"
    asm volatile("{\n\t.reg .pred e, f, t;\n\t.reg .b32 ta, yl;\n\t.reg .b64 yd;\n\t"
                 "elect.sync _|e, 0xffffffff;\n\t"
                 "setp.ne.b32 f, %5, 0;\n\tsetp.eq.b32 t, %4, %4;\n\t"
                 "mov.b64 yd, {%2, %3};\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], yd, %4, f;\n\t"
                 SWA_MMA_TS(8, 128) SWA_MMA_TS(16, 256) SWA_MMA_TS(24, 384) SWA_MMA_TS(32, 512)
                 SWA_MMA_TS(40, 640) SWA_MMA_TS(48, 768) SWA_MMA_TS(56, 896) "}\n" ::"r"(d),
                 "r"(a_tmem), "r"(bl), "r"(bh), "r"(idesc), "r"(acc0)
                 : "memory");
#undef SWA_MMA_TS
}

// Half of mma_ts_group8: O (+)= P * V over 64 keys, four k-steps from the
// given P columns and V rows (the first four of a 128-key tile, or with
// a_tmem + 32 and the V descriptor advanced 64 rows, the last four).
__device__ __forceinline__ void mma_ts_group4(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                              uint32_t acc0)
{
    const uint32_t bl = static_cast<uint32_t>(b), bh = static_cast<uint32_t>(b >> 32);
#define SWA_MMA_TS(AO, BO) \
    "add.u32 ta, %1, " #AO ";\n\tadd.u32 yl, %2, " #BO ";\n\tmov.b64 yd, {yl, %3};\n\t" \
    "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], yd, %4, t;\n\t"
    asm volatile("{\n\t.reg .pred e, f, t;\n\t.reg .b32 ta, yl;\n\t.reg .b64 yd;\n\t"
                 "elect.sync _|e, 0xffffffff;\n\t"
                 "setp.ne.b32 f, %5, 0;\n\tsetp.eq.b32 t, %4, %4;\n\t"
                 "mov.b64 yd, {%2, %3};\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], yd, %4, f;\n\t"
                 SWA_MMA_TS(8, 128) SWA_MMA_TS(16, 256) SWA_MMA_TS(24, 384) "}\n" ::"r"(d),
                 "r"(a_tmem), "r"(bl), "r"(bh), "r"(idesc), "r"(acc0)
                 : "memory");
#undef SWA_MMA_TS
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, A K-major,
// B K-major (b_mn_major = 0) or N-major (1), shape M x N.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format,
//   15 A major, 16 B major, 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int b_mn_major)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(b_mn_major) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Shared-memory matrix descriptor with the 128-byte swizzle: start address,
// leading- and stride-dimension byte offsets (all >> 4), the fixed version
// field (bit 46) and the layout type 2 (SWIZZLE_128B) in bits 61-63.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                    uint32_t sbo_bytes)
{
    uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// 32 lanes x 32 columns of 32-bit words: thread t of the warp receives lane
// (base lane + t), columns col .. col+31 in r[0..31].
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Orders later uses of r[] after a preceding tcgen05.wait::ld (an empty
// volatile asm that "rewrites" the registers; volatile asm keeps its order).
__device__ __forceinline__ void reg_fence32(uint32_t (&r)[32])
{
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]),
                   "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]),
                   "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (low 16 bits), .y = hi
    return *reinterpret_cast<uint32_t *>(&v);
}


// ------------------------------------------------------------------ CTA pairs
// Two CTAs of a cluster of two sharing one tcgen05 MMA (cta_group::2): the
// MMA of M = 256 rows takes rows 0-127 of A from the even CTA's shared (or
// tensor) memory and rows 128-255 from the odd CTA's, splits B along N between
// the two (each CTA holds N/2 of its rows, at the same shared-memory offset)
// and writes each CTA's 128 rows of D into that CTA's tensor memory.  Every
// tcgen05 instruction of such a kernel names cta_group::2.

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The shared::cluster address of shared-memory address `addr` in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// One arrival on an mbarrier given by its shared::cluster address (this CTA's
// or the peer's).  The arrivals that cross the pair follow a completed
// tensor-memory store (tcgen05.wait::st, then tcgen05.fence::before_thread_sync)
// or a completed tensor-memory load, so they need no cluster-scope release;
// with .release.cluster (and .acquire.cluster on the waiting side) the
// pair kernel's hand-offs took 1.3x as long.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cl_bar)
{
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cl_bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// mbar_wait for a barrier that the peer CTA's threads or copies also complete;
// the same bound and error reporting.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, volatile int *abort,
                                                  int *status, uint64_t timeout_ns)
{
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((it & 31u) == 0) {
            if (abort != nullptr && *abort) return false;
            if (globaltimer_ns() - t0 > timeout_ns) {
                if (abort != nullptr) *abort = 1;
                if (status != nullptr) atomicOr(status, 1);
                return false;
            }
        }
    }
}

// Every thread of both CTAs: arrive, then wait for all the others (the
// per-thread form: a warp need not be converged).
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release;\n\t"
                 "barrier.cluster.wait.acquire;" ::: "memory");
}

// 3-D tiled load into this CTA's shared memory whose completion is counted on
// an mbarrier of either CTA of the pair (its shared::cluster address).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap *map,
                                                 uint32_t cl_bar, int c0, int c1, int c2)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".cta_group::2 [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(cl_bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// Tensor memory of a CTA pair: one warp of each CTA allocates (the same
// columns in both) and frees.
__device__ __forceinline__ void tmem_alloc2(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish2()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// One arrival on the mbarrier at shared-memory offset `bar` of each CTA in
// `mask` (bit r: cluster rank r) once every MMA issued before has completed;
// issued by one elected lane of the calling warp.
__device__ __forceinline__ void tc_commit2_mc(uint32_t bar, uint16_t mask)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;\n\t}" ::"r"(bar),
        "h"(mask)
        : "memory");
}

// S = A * B^T over K = 128 for a CTA pair (M = 256): A K-major in 64-column
// chunks of 128 rows (16 KB apart), B K-major in 64-column chunks of the
// CTA's N/2 = 64 rows (8 KB apart); k-step ks adds (ks & 3) * 32 bytes within
// a chunk.  Descriptor start addresses are in 16-byte units.
__device__ __forceinline__ void mma2_ss_group8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc)
{
    const uint32_t al = static_cast<uint32_t>(a), ah = static_cast<uint32_t>(a >> 32);
    const uint32_t bl = static_cast<uint32_t>(b), bh = static_cast<uint32_t>(b >> 32);
#define SWA_MMA2_SS(AO, BO) \
    "add.u32 xl, %1, " #AO ";\n\tadd.u32 yl, %3, " #BO ";\n\t" \
    "mov.b64 xd, {xl, %2};\n\tmov.b64 yd, {yl, %4};\n\t" \
    "@e tcgen05.mma.cta_group::2.kind::f16 [%0], xd, yd, %5, t;\n\t"
    asm volatile("{\n\t.reg .pred e, f, t;\n\t.reg .b32 xl, yl;\n\t.reg .b64 xd, yd;\n\t"
                 "elect.sync _|e, 0xffffffff;\n\t"
                 "setp.ne.b32 f, %5, %5;\n\tsetp.eq.b32 t, %5, %5;\n\t"
                 "mov.b64 xd, {%1, %2};\n\tmov.b64 yd, {%3, %4};\n\t"
                 "@e tcgen05.mma.cta_group::2.kind::f16 [%0], xd, yd, %5, f;\n\t"
                 SWA_MMA2_SS(2, 2) SWA_MMA2_SS(4, 4) SWA_MMA2_SS(6, 6) SWA_MMA2_SS(1024, 512)
                 SWA_MMA2_SS(1026, 514) SWA_MMA2_SS(1028, 516) SWA_MMA2_SS(1030, 518) "}\n" ::"r"(d),
                 "r"(al), "r"(ah), "r"(bl), "r"(bh), "r"(idesc)
                 : "memory");
#undef SWA_MMA2_SS
}

// O (+)= P * V over K = 128 keys for a CTA pair: P in each CTA's tensor memory
// (8 columns per k-step), V N-major in shared memory, the CTA's N/2 = 64
// columns (k-step ks adds ks * 16 rows * 128 B).
__device__ __forceinline__ void mma2_ts_group8(uint32_t d, uint32_t a_tmem, uint64_t b,
                                               uint32_t idesc, uint32_t acc0)
{
    const uint32_t bl = static_cast<uint32_t>(b), bh = static_cast<uint32_t>(b >> 32);
#define SWA_MMA2_TS(AO, BO) \
    "add.u32 ta, %1, " #AO ";\n\tadd.u32 yl, %2, " #BO ";\n\tmov.b64 yd, {yl, %3};\n\t" \
    "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [ta], yd, %4, t;\n\t"
    asm volatile("{\n\t.reg .pred e, f, t;\n\t.reg .b32 ta, yl;\n\t.reg .b64 yd;\n\t"
                 "elect.sync _|e, 0xffffffff;\n\t"
                 "setp.ne.b32 f, %5, 0;\n\tsetp.eq.b32 t, %4, %4;\n\t"
                 "mov.b64 yd, {%2, %3};\n\t"
                 "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], yd, %4, f;\n\t"
                 SWA_MMA2_TS(8, 128) SWA_MMA2_TS(16, 256) SWA_MMA2_TS(24, 384) SWA_MMA2_TS(32, 512)
                 SWA_MMA2_TS(40, 640) SWA_MMA2_TS(48, 768) SWA_MMA2_TS(56, 896) "}\n" ::"r"(d),
                 "r"(a_tmem), "r"(bl), "r"(bh), "r"(idesc), "r"(acc0)
                 : "memory");
#undef SWA_MMA2_TS
}

}  // namespace ptx
}  // namespace swa
