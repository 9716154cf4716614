// swa_prefill_duo.cuh -- the window-path prefill on CTA pairs (cta_group::2).
//
// Included by swa_prefill_tc.cu inside its namespace: it uses that file's
// tile walk (item_tiles, key_tile), softmax pieces (softmax_half, finish_row),
// epilogue (store_o_rows_chunked) and parameter block.
//
// What it computes is the pair kernel's: causal sliding-window attention with
// sinks ("Sliding Window and Sparse Attention, from Longformer to CSA2",
// sections 2 and 4; "Local and Sparse Attention: Reading Fewer Token
// Positions", Figures 1-2), exact softmax by the online (flash) recurrence,
// only the key tiles that meet the band or the sinks.
//
// Why pairs.  With one CTA per work item, each 128x128x16 MMA of S = Q K^T
// reads 8 KB of operands from shared memory for 64 cycles of math, which is
// the shared-memory port's whole rate; with the P V operands and the TMA
// writes of K and V, the port is busier than the tensor core and sets the
// tile period.  A cluster of two CTAs sharing one MMA of M = 256 rows halves
// what each SM reads of B (K for S, V for P V) and what each loads of K and V:
// CTA r holds keys 64r .. 64r+63 of every K tile and value columns
// 64r .. 64r+63 of every V tile.
//
// Work item: four query heads h = 4q + 2x + r (q a quad of heads, x the half,
// r the CTA's rank in the cluster) over one 128-row q tile.  Half x is one
// MMA of 256 rows: head 4q + 2x in CTA 0 and head 4q + 2x + 1 in CTA 1, which
// read the same kv head (the group size G is even).  When G % 4 == 0 the two
// halves read the same kv head too and share one K/V stream (SHARED);
// otherwise each half has its own.
//
// Roles (512 threads per CTA, as the pair kernel): warp 0 loads (each CTA its
// own rows and halves, completing on barriers of CTA 0), warp 1 of CTA 0
// issues every MMA, warpgroups 1 and 2 run the softmax of halves 0 and 1 on
// the CTA's own rows, warpgroup 3 writes the output.  Tensor memory as the
// pair kernel: O_0 [0,128), S_0 [128,256), O_1 [256,384), S_1 [384,512).
// K/V protocol: the pair kernel's skewed one (tile c's barrier carries K(c)
// and V(c-1), K and V slots freed separately).
//
// Synchronisation across the pair: the MMA warp's commits arrive on the
// barriers of both CTAs (multicast); the loads of both CTAs complete on CTA
// 0's full barriers, which CTA 0's producer arms with both CTAs' bytes; the
// softmax and epilogue warps of both CTAs arrive on CTA 0's P_FULL and
// O_EMPTY barriers.  Every wait is bounded (a timeout sets the device status
// word and ends the CTA's roles).

template <int HD, bool SHARED>
struct LayoutD {
    static constexpr int NSTR = SHARED ? 1 : 2;        // K/V streams
    // K/V ring depth: one shared stream fits four stages in the shared memory
    // that two streams fill with two
    static constexpr int DUO_STAGES = SHARED ? 4 : 2;
    static constexpr uint32_t QB = BM * HD * 2;        // one half's 128 query rows
    static constexpr uint32_t KH = (BN / 2) * HD * 2;  // this CTA's 64 keys of a K tile
    static constexpr uint32_t VH = BN * (HD / 2) * 2;  // this CTA's HD/2 columns of a V tile
    static constexpr uint32_t Q_OFF = 0;
    static constexpr uint32_t K_OFF = Q_OFF + 2 * QB;
    static constexpr uint32_t V_OFF = K_OFF + DUO_STAGES * NSTR * KH;
    static constexpr uint32_t BAR_OFF = V_OFF + DUO_STAGES * NSTR * VH;
    enum {
        Q_FULL = 0,                       // CTA 0: both CTAs' Q rows of half x landed
        Q_EMPTY = 2,                      // both: half x's Q buffer is free
        K_FULL = 4,                       // CTA 0: K(c) and V(c-1) landed in both CTAs
        V_EMPTY = K_FULL + DUO_STAGES,    // both: a V slot is free
        KV_EMPTY = V_EMPTY + DUO_STAGES,  // both: a K slot is free
        S_FULL = KV_EMPTY + DUO_STAGES,   // both: S_x is in tensor memory
        P_FULL = S_FULL + 2,              // CTA 0: P_x written by all 8 softmax warps
        O_FULL = P_FULL + 2,              // both: the item's last P_x V has landed
        O_EMPTY = O_FULL + 2,             // CTA 0: O_x read out by all 8 epilogue warps
        ROW_STATS = O_EMPTY + 2,          // both, local: [half x][item parity]
        DRAIN = ROW_STATS + 4,
        NBAR = DRAIN + 1
    };
    static constexpr uint32_t MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr uint32_t STATS_OFF = (MISC_OFF + 16 + 15) & ~15u;
    static constexpr uint32_t STAGE_OFF = STATS_OFF + 2 * 2 * BM * 8;
    static constexpr uint32_t BYTES = STAGE_OFF + 4 * STAGE_WARP;
    static constexpr uint32_t DYN_SMEM = BYTES + 1024;
};

// Work order: q tiles from the last (the most key tiles) down; within a q
// tile the quad of heads fastest, then the sequence.  Cluster c's k-th item
// has rank duo_item_rank(c, k) (the pair kernel's snake over clusters).
__device__ __forceinline__ void duo_item(int r, const PrefillParams &p, int &b, int &q, int &qt)
{
    const int quads = p.H >> 2, per = p.B * quads;
    qt = p.n_qt - 1 - r / per;
    r %= per;
    q = r % quads;
    b = r / quads;
}
__device__ __forceinline__ int duo_item_rank(int c, int k)
{
    const int P = static_cast<int>(gridDim.x) >> 1;
    return k * P + ((k & 1) ? P - 1 - c : c);
}

template <int HD, bool SHARED>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS2, 1)
    swa_prefill_bf16_duo_sm103(const __grid_constant__ CUtensorMap tmQ,
                               const __grid_constant__ CUtensorMap tmKh,
                               const __grid_constant__ CUtensorMap tmV, const PrefillParams p)
{
    static_assert(HD == 128, "the CTA-pair kernel splits 128 value columns into two 64-column halves");
    using L = LayoutD<HD, SHARED>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(smem);
    const uint32_t sQ = sb + L::Q_OFF, sK = sb + L::K_OFF, sV = sb + L::V_OFF;
    const uint32_t bars = sb + L::BAR_OFF;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::MISC_OFF + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = static_cast<int>(cluster_ctarank());
    const int cl = static_cast<int>(blockIdx.x) >> 1;
    const int num_items = p.num_items;
    // this CTA's barriers, and CTA 0's (the one the MMA warp waits on) in the
    // cluster's shared window
    const uint32_t lead = mapa_shared(bars, 0);
#define BAR(i) (bars + 8u * static_cast<uint32_t>(i))
#define LBAR(i) (lead + 8u * static_cast<uint32_t>(i))

    if (threadIdx.x == 0) {
        for (int x = 0; x < 2; ++x) {
            mbar_init(BAR(L::Q_FULL + x), 1);
            mbar_init(BAR(L::Q_EMPTY + x), 1);
            mbar_init(BAR(L::S_FULL + x), 1);
            mbar_init(BAR(L::P_FULL + x), 8);
            mbar_init(BAR(L::O_FULL + x), 1);
            mbar_init(BAR(L::O_EMPTY + x), 8);
            mbar_init(BAR(L::ROW_STATS + 2 * x), 4);
            mbar_init(BAR(L::ROW_STATS + 2 * x + 1), 4);
        }
        for (int i = 0; i < L::DUO_STAGES; ++i) {
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
        tma_prefetch(&tmKh);
        tma_prefetch(&tmV);
    }
    if (warp == 1) {
        tmem_alloc2(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish2();
    }
    // both CTAs' barriers are initialised and their tensor memory allocated
    // before either CTA's copies, commits or arrivals can reach the other
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
#ifdef SWA_DEBUG
    if (!tmem_base_ok(tmem, p.status)) goto teardown;
#endif

    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_CTRL));
        if (warp == 0) {
            // -------------------------------------------------------- producer
            // Both CTAs walk the same items and tiles.  CTA r loads its own Q
            // rows (head 4q + 2x + r), keys 64r .. 64r+63 of each K tile and
            // value columns 64r .. 64r+63 of each V tile; every copy completes
            // on CTA 0's barrier, which CTA 0 arms with both CTAs' bytes (a
            // copy of CTA 1 may land before the arming: the phase still needs
            // CTA 0's arrival).  The empty barriers are this CTA's own (the
            // MMA warp's commits reach both).
            if (lane == 0) {
                int kv_iter = 0, it = 0;
                bool ok = true;
                bool pv_have = false;
                int pv_k0 = 0, pv_z[2] = {0, 0};
                auto issue_prev_v = [&](int c_next, uint32_t cl_bar) {
                    const int vs = (c_next - 1) % L::DUO_STAGES;
                    for (int s = 0; s < L::NSTR; ++s)
                        tma_load_3d_pair(sV + (vs * L::NSTR + s) * L::VH, &tmV, cl_bar,
                                         rank * (HD / 2), pv_k0, pv_z[s]);
                };
                // V slot (c_next - 1) % stages free for V(c_next - 1)
                auto wait_prev_v = [&](int c_next) -> bool {
                    const int vc = c_next - 1;
                    return mbar_wait(BAR(L::V_EMPTY + vc % L::DUO_STAGES), ((vc / L::DUO_STAGES) & 1) ^ 1,
                                     abort_flag, p.status, p.wait_ns);
                };
                for (int t = duo_item_rank(cl, 0); ok && t < num_items;
                     t = duo_item_rank(cl, ++it)) {
                    int b, q, qt, off;
                    duo_item(t, p, b, q, qt);
                    const TileRange tr = item_tiles<false>(p, b, qt, 0, off);
                    const int z0 = b * p.Hkv + (4 * q) / p.G;
                    const int z1 = SHARED ? z0 : b * p.Hkv + (4 * q + 2) / p.G;
                    // the item's Q rows, after its first key tile (which carries
                    // the previous item's last V, needed first)
                    auto load_q = [&]() -> bool {
                        for (int x = 0; x < 2; ++x) {
                            if (!mbar_wait(BAR(L::Q_EMPTY + x), (it & 1) ^ 1, abort_flag, p.status,
                                           p.wait_ns))
                                return false;
                            if (rank == 0) mbar_expect_tx(BAR(L::Q_FULL + x), 2 * L::QB);
                            const int h = 4 * q + 2 * x + rank;
                            for (int c = 0; c < HD / 64; ++c)
                                tma_load_3d_pair(sQ + x * L::QB + c * (BM * 128), &tmQ,
                                                 LBAR(L::Q_FULL + x), c * 64, qt * BM, b * p.H + h);
                        }
                        return true;
                    };
                    for (int j = 0; ok && j < tr.count; ++j, ++kv_iter) {
                        const int st = kv_iter % L::DUO_STAGES;
                        const uint32_t ph = (kv_iter / L::DUO_STAGES) & 1;
                        if ((pv_have && !wait_prev_v(kv_iter)) ||
                            !mbar_wait(BAR(L::KV_EMPTY + st), ph ^ 1, abort_flag, p.status,
                                       p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        const KeyTile kt = key_tile<false>(tr, j, p);
                        // test injection: this tile's copies never start, so the
                        // MMA warp's wait for them runs out
                        if (p.skip_first_kv && kv_iter == 0) {
                            pv_have = false;
                            continue;
                        }
                        if (rank == 0)
                            mbar_expect_tx(BAR(L::K_FULL + st),
                                           2u * L::NSTR * (L::KH + (pv_have ? L::VH : 0u)));
                        if (pv_have) issue_prev_v(kv_iter, LBAR(L::K_FULL + st));
                        const int zs[2] = {z0, z1};
                        for (int s = 0; s < L::NSTR; ++s)
                            for (int c = 0; c < HD / 64; ++c)
                                tma_load_3d_pair(sK + (st * L::NSTR + s) * L::KH + c * (BN / 2 * 128),
                                                 &tmKh, LBAR(L::K_FULL + st), c * 64,
                                                 kt.k0 + rank * (BN / 2), zs[s]);
                        pv_have = true;
                        pv_k0 = kt.k0;
                        pv_z[0] = z0;
                        pv_z[1] = z1;
                        if (j == 0 && !load_q()) {
                            ok = false;
                            break;
                        }
                    }
                }
                // the last tile's V, on the barrier of the tile after it (whose
                // previous phase must be complete before it is armed again)
                if (ok && pv_have) {
                    const int st = kv_iter % L::DUO_STAGES;
                    const uint32_t ph = (kv_iter / L::DUO_STAGES) & 1;
                    if (wait_prev_v(kv_iter) &&
                        mbar_wait(BAR(L::KV_EMPTY + st), ph ^ 1, abort_flag, p.status, p.wait_ns)) {
                        if (rank == 0) mbar_expect_tx(BAR(L::K_FULL + st), 2u * L::NSTR * L::VH);
                        issue_prev_v(kv_iter, LBAR(L::K_FULL + st));
                    }
                }
            }
        } else if (warp == 1 && rank == 0) {
            // ------------------------------------------------------ MMA issuer
            // One MMA of 256 rows per k-step serves both CTAs.  Order per key
            // tile c, as the pair kernel: [K(c), V(c-1) landed] P_0(c-1) V,
            // S_0(c), P_1(c-1) V, S_1(c).
            const uint32_t idesc_s = idesc_bf16_f32(256, BN, 0);
            const uint32_t idesc_o = idesc_bf16_f32(256, HD, 1);
            constexpr uint16_t BOTH = 3;
            int kv_iter = 0, it = 0, c = 0;
            bool ok = true;
            bool have_prev = false, prev_first = false, prev_last = false;
            int prev_st = 0, prev_c = 0, prev_it = 0;
            auto wait_cl = [&](uint32_t bar, uint32_t parity) -> bool {
                const bool r_ok = mbar_wait_cluster(bar, parity, abort_flag, p.status, p.wait_ns);
                return __all_sync(0xffffffffu, r_ok);
            };
            auto issue_pv = [&](auto xc) -> bool {
                constexpr int x = decltype(xc)::value;
                constexpr int sx = SHARED ? 0 : x;
                if (!wait_cl(BAR(L::P_FULL + x), prev_c & 1)) return false;
                if (prev_first && !wait_cl(BAR(L::O_EMPTY + x), (prev_it & 1) ^ 1)) return false;
                tc_fence_after();
                const uint64_t vb =
                    smem_desc_sw128(sV + (prev_st * L::NSTR + sx) * L::VH, BN * 128, 1024);
                mma2_ts_group8(tmem + x * 256, tmem + x * 256 + 128, vb, idesc_o,
                               prev_first ? 0u : 1u);
                if (x == 1) tc_commit2_mc(BAR(L::V_EMPTY + prev_st), BOTH);
                if (prev_last) tc_commit2_mc(BAR(L::O_FULL + x), BOTH);
                return true;
            };
            auto issue_s = [&](auto xc, int st, bool last) {
                constexpr int x = decltype(xc)::value;
                constexpr int sx = SHARED ? 0 : x;
                const uint64_t qb = smem_desc_sw128(sQ + x * L::QB, 16, 1024);
                const uint64_t kb = smem_desc_sw128(sK + (st * L::NSTR + sx) * L::KH, 16, 1024);
                mma2_ss_group8(tmem + x * 256 + 128, qb, kb, idesc_s);
                tc_commit2_mc(BAR(L::S_FULL + x), BOTH);
                if (last) tc_commit2_mc(BAR(L::Q_EMPTY + x), BOTH);
                if (x == 1) tc_commit2_mc(BAR(L::KV_EMPTY + st), BOTH);
            };
            using X0 = std::integral_constant<int, 0>;
            using X1 = std::integral_constant<int, 1>;
            for (int t = duo_item_rank(cl, 0); ok && t < num_items; t = duo_item_rank(cl, ++it)) {
                int b, q, qt, off;
                duo_item(t, p, b, q, qt);
                const TileRange tr = item_tiles<false>(p, b, qt, 0, off);
                for (int j = 0; j < tr.count; ++j, ++kv_iter, ++c) {
                    const int st = kv_iter % L::DUO_STAGES;
                    const uint32_t ph = (kv_iter / L::DUO_STAGES) & 1;
                    const bool last = (j == tr.count - 1);
                    if (!wait_cl(BAR(L::K_FULL + st), ph)) {
                        ok = false;
                        break;
                    }
                    if (have_prev && !issue_pv(X0{})) {
                        ok = false;
                        break;
                    }
                    if (j == 0 && !wait_cl(BAR(L::Q_FULL + 0), it & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_s(X0{}, st, last);
                    if (have_prev && !issue_pv(X1{})) {
                        ok = false;
                        break;
                    }
                    if (j == 0 && !wait_cl(BAR(L::Q_FULL + 1), it & 1)) {
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
            // the last tile's V rides on the barrier of the tile after it
            if (ok && have_prev &&
                wait_cl(BAR(L::K_FULL + kv_iter % L::DUO_STAGES), (kv_iter / L::DUO_STAGES) & 1)) {
                if (issue_pv(X0{})) issue_pv(X1{});
            }
            // every MMA issued has completed before the CTAs leave
            tc_commit2_mc(BAR(L::DRAIN), 1);
            warp_wait(BAR(L::DRAIN), 0, nullptr, nullptr, TIMEOUT_NS);
        }
    } else if (warp < 12) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REGS_SOFTMAX));
        // ------------------------------------------------------------ softmax
        // Half x on this CTA's 128 rows of head 4q + 2x + rank: the pair
        // kernel's online softmax (window path), P handed to CTA 0's MMA warp
        // through its P_FULL barrier.
        const int x = (warp >> 2) - 1;
        const int sub = warp & 3;
        const int r = sub * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(sub * 32) << 16;
        const uint32_t o_addr = tmem + lane_off + x * 256;
        const uint32_t s_addr = o_addr + 128;
        const float sl2 = p.sl2;
        const uint64_t sl2x2 = pack2(__float_as_uint(sl2), __float_as_uint(sl2));
        float2 *stats = reinterpret_cast<float2 *>(smem + L::STATS_OFF);
        const uint32_t p_full = LBAR(L::P_FULL + x);
        int c = 0, it = 0;
        bool ok = true;
        for (int t = duo_item_rank(cl, 0); ok && t < num_items; t = duo_item_rank(cl, ++it)) {
            int b, q, qt, off;
            duo_item(t, p, b, q, qt);
            const TileRange tr = item_tiles<false>(p, b, qt, 0, off);
            const int h = 4 * q + 2 * x + rank;
            const int i = tr.q0 + r;
            const int lo = i - p.w + 1;
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < tr.count; ++j, ++c) {
                if (!warp_wait(BAR(L::S_FULL + x), c & 1, abort_flag, p.status, p.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t s[4][32];
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) tmem_ld32(s_addr + qq * 32, s[qq]);
                tmem_ld_wait();
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) reg_fence32(s[qq]);
                const KeyTile kt = key_tile<false>(tr, j, p);
                if (!kt.full) {
                    // k <= i and (k >= i-w+1 or k < g), in tile columns
                    mask_cols(s, lo - kt.k0, i - kt.k0, p.g - kt.k0);
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
                        // O_x is complete: the S_x(c) commit covered P_x(c-1) V
                        const float alpha = need ? ex2(m - m_new) : 1.f;
                        if (need) m = m_new;
                        l *= alpha;
#pragma unroll 1
                        for (int qq = 0; qq < HD / 32; ++qq) {
                            uint32_t o[32];
                            tmem_ld32(o_addr + qq * 32, o);
                            tmem_ld_wait();
                            reg_fence32(o);
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st32(o_addr + qq * 32, o);
                        }
                    }
                }
                const float m_use = (m == -INFINITY) ? 0.f : m;
                const uint64_t negm2 = pack2(__float_as_uint(-m_use), __float_as_uint(-m_use));
                uint64_t acc2 = 0;
                uint32_t pk[32];
                softmax_half(s[0], s[1], sl2x2, negm2, acc2, pk);
                tmem_st32(s_addr, pk);
                softmax_half(s[2], s[3], sl2x2, negm2, acc2, pk);
                tmem_st32(s_addr + 32, pk);
                float a0, a1;
                unpack2(acc2, a0, a1);
                l += a0 + a1;
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(p_full);
            }
            if (!ok) break;
            float row_lse;
            const float inv_l = finish_row(m, l, p.sink, h, &row_lse);
            stats[((it & 1) * 2 + x) * BM + r] = make_float2(inv_l, row_lse);
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(L::ROW_STATS + 2 * x + (it & 1)));
        }
        if (!ok) *abort_flag = 1;
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_EPI));
        // ------------------------------------------------------------ epilogue
        // Per item and half: the softmax's row statistics and the item's last
        // P V, then O / l as bf16 (and the LSE) for this CTA's head; O_x is
        // released on CTA 0's O_EMPTY barrier.
        const int sub = warp & 3;
        const int r = sub * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(sub * 32) << 16;
        const float2 *stats = reinterpret_cast<const float2 *>(smem + L::STATS_OFF);
        uint8_t *stage = smem + L::STAGE_OFF + sub * STAGE_WARP;
        int it = 0;
        bool ok = true;
        for (int t = duo_item_rank(cl, 0); ok && t < num_items; t = duo_item_rank(cl, ++it)) {
            int b, q, qt, off;
            duo_item(t, p, b, q, qt);
            const TileRange tr = item_tiles<false>(p, b, qt, 0, off);
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
                const int h = 4 * q + 2 * x + rank;
                const int t_row = tr.q0 + r - off;
                const size_t orow_i = static_cast<size_t>(b * p.H + h) * p.n + t_row;
                const bool row_ok =
                    t_row < p.n && SWA_BOUNDS(static_cast<long long>(orow_i) < p.dbg_orows, p.status);
                store_o_rows_chunked<HD, true>(tmem + lane_off + x * 256, sv.x, p.O + orow_i * HD,
                                               row_ok, stage, lane, LBAR(L::O_EMPTY + x));
                if (p.lse != nullptr && row_ok) p.lse[orow_i] = sv.y;
            }
        }
    }
#undef LBAR
#undef BAR
    // neither CTA leaves (nor frees its tensor memory) while the other may
    // still reach its barriers or tensor memory
#ifdef SWA_DEBUG
teardown:
#endif
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc2(tmem, TMEM_COLS);
    }
}
