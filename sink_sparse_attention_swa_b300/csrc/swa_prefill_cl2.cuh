// swa_prefill_cl2.cuh -- the window-path prefill on CTA pairs with one query
// head per CTA and the score tile double-buffered.
//
// Included by swa_prefill_tc.cu inside its namespace (it uses that file's tile
// walk, softmax pieces, epilogue and parameter block, and the CTA-pair PTX
// wrappers).  It computes what the pair kernel computes: causal sliding-window
// attention with sinks ("Sliding Window and Sparse Attention, from Longformer
// to CSA2", sections 2 and 4), exact softmax by the online recurrence, only
// the key tiles that meet the band or the sinks.
//
// Why this shape.  In the pair kernel each head's P overwrites its S in tensor
// memory, so S(c+1) cannot start before P(c) V has been issued: per key tile,
// each head waits for its own S -> softmax -> P -> P V chain, and the other
// head covers that only in part.  Here the two CTAs of a cluster take the two
// heads of one pair (head 2u + r in CTA r, both reading kv head 2u / G), and
// one MMA of 256 rows serves both (tcgen05 cta_group::2; CTA r holds keys
// 64r..64r+63 of every K tile and value columns 64r..64r+63 of every V tile).
// One head per CTA leaves room in tensor memory for two S buffers and two O
// buffers: S(c+1) is computed while the softmax works on S(c), and the next
// item's first products need not wait for this item's output to be read out.
// Q is double-buffered in shared memory for the same reason.
//
// Roles (512 threads per CTA): warp 0 loads; warp 1 of CTA 0 issues every MMA;
// warpgroups 1 and 2 run the softmax of the CTA's 128 rows, warpgroup 1 on
// key columns 0..63 of each tile and warpgroup 2 on 64..127 (they share each
// row's maximum through shared memory and a two-warp mbarrier);
// warpgroup 3 writes the output.
//
// Tensor memory (512 columns): O buffers [0,128) and [128,256) by item
// parity, S buffers [256,384) and [384,512) by tile parity.  P (bf16) of keys
// 0..63 is written over the S buffer's columns 0..31, of keys 64..127 over its
// columns 64..95: each softmax warpgroup writes only columns it has read.
//
// MMA order per key tile c: [K(c), V(c-1) landed] S(c) into buffer c % 2, then
// P(c-1) V in two halves (keys 0..63 as soon as warpgroup 1's P is in, keys
// 64..127 after warpgroup 2's).  An O rescale (rare: the running maximum rose
// by more than 2^8) waits for the previous P V to complete (PV_DONE).
//
// Every wait is bounded; a timeout sets the device status word and ends the
// CTA's roles, which meet at a cluster barrier before either CTA exits.

template <int HD>
struct LayoutC {
    static constexpr int NST = 4;                      // K/V ring depth
    static constexpr uint32_t QB = BM * HD * 2;        // one head's 128 query rows
    static constexpr uint32_t KH = (BN / 2) * HD * 2;  // this CTA's 64 keys of a K tile
    static constexpr uint32_t VH = BN * (HD / 2) * 2;  // this CTA's HD/2 columns of a V tile
    static constexpr uint32_t Q_OFF = 0;               // two Q buffers (item parity)
    static constexpr uint32_t K_OFF = Q_OFF + 2 * QB;
    static constexpr uint32_t V_OFF = K_OFF + NST * KH;
    static constexpr uint32_t BAR_OFF = V_OFF + NST * VH;
    enum {
        Q_FULL = 0,                  // CTA 0 [item parity]: both CTAs' Q rows landed
        Q_EMPTY = 2,                 // both [item parity]: the Q buffer is free
        K_FULL = 4,                  // CTA 0 [slot]: K(c) and V(c-1) landed in both CTAs
        V_EMPTY = K_FULL + NST,      // both [slot]: a V slot is free
        KV_EMPTY = V_EMPTY + NST,    // both [slot]: a K slot is free
        S_FULL = KV_EMPTY + NST,     // both [tile parity]: S is in tensor memory
        P_LEFT = S_FULL + 2,         // CTA 0 [tile parity]: P of keys 0..63 (8 warps)
        P_RIGHT = P_LEFT + 2,        // CTA 0 [tile parity]: P of keys 64..127 (8 warps)
        PV_DONE = P_RIGHT + 2,       // both [tile parity]: that tile's P V has completed
        O_FULL = PV_DONE + 2,        // both [item parity]: the item's last P V landed
        O_EMPTY = O_FULL + 2,        // CTA 0 [item parity]: O read out (8 epilogue warps)
        ROW_STATS = O_EMPTY + 2,     // local [item parity]: (m, l) of both sides posted
        STATS_EMPTY = ROW_STATS + 2, // local [item parity]: the epilogue has read them
        DRAIN = STATS_EMPTY + 2,
        MAXX = DRAIN + 1,            // local [lane quarter][tile parity]: both sides' maxima posted
        NBAR = MAXX + 8
    };
    static constexpr uint32_t MISC_OFF = BAR_OFF + NBAR * 8;
    // row-maximum exchange: float [tile parity][side][128 rows]
    static constexpr uint32_t MAX_OFF = (MISC_OFF + 16 + 15) & ~15u;
    // (m, l) per row: float2 [item parity][side][128 rows]
    static constexpr uint32_t STATS_OFF = MAX_OFF + 2 * 2 * BM * 4;
    static constexpr uint32_t STAGE_OFF = STATS_OFF + 2 * 2 * BM * 8;
    static constexpr uint32_t BYTES = STAGE_OFF + 4 * STAGE_WARP;
    static constexpr uint32_t DYN_SMEM = BYTES + 1024;
};
static_assert(LayoutC<128>::DYN_SMEM <= 227 * 1024, "shared memory of the CTA-pair kernel");

// Work order: q tiles from the last (the most key tiles) down; within a q
// tile the head pair fastest, then the sequence.  Cluster c's k-th item has
// rank duo_item_rank(c, k).
__device__ __forceinline__ void cl2_item(int r, const PrefillParams &p, int &b, int &u, int &qt)
{
    const int pairs = p.H >> 1, per = p.B * pairs;
    qt = p.n_qt - 1 - r / per;
    r %= per;
    u = r % pairs;
    b = r / pairs;
}

template <int HD>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS2, 1)
    swa_prefill_bf16_cl2_sm103(const __grid_constant__ CUtensorMap tmQ,
                               const __grid_constant__ CUtensorMap tmKh,
                               const __grid_constant__ CUtensorMap tmV, const PrefillParams p)
{
    static_assert(HD == 128, "the CTA-pair kernel splits 128 value columns into two 64-column halves");
    using L = LayoutC<HD>;
    constexpr int NST = L::NST;
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
    const uint32_t lead = mapa_shared(bars, 0);  // CTA 0's barriers, cluster window
#define BAR(i) (bars + 8u * static_cast<uint32_t>(i))
#define LBAR(i) (lead + 8u * static_cast<uint32_t>(i))

    if (threadIdx.x == 0) {
        for (int x = 0; x < 2; ++x) {
            mbar_init(BAR(L::Q_FULL + x), 1);
            mbar_init(BAR(L::Q_EMPTY + x), 1);
            mbar_init(BAR(L::S_FULL + x), 1);
            mbar_init(BAR(L::P_LEFT + x), 8);
            mbar_init(BAR(L::P_RIGHT + x), 8);
            mbar_init(BAR(L::PV_DONE + x), 1);
            mbar_init(BAR(L::O_FULL + x), 1);
            mbar_init(BAR(L::O_EMPTY + x), 8);
            mbar_init(BAR(L::ROW_STATS + x), 8);
            mbar_init(BAR(L::STATS_EMPTY + x), 4);
        }
        for (int i = 0; i < NST; ++i) {
            mbar_init(BAR(L::K_FULL + i), 1);
            mbar_init(BAR(L::V_EMPTY + i), 1);
            mbar_init(BAR(L::KV_EMPTY + i), 1);
        }
        mbar_init(BAR(L::DRAIN), 1);
        for (int i = 0; i < 8; ++i) mbar_init(BAR(L::MAXX + i), 2);
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
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_CTRL));
        if (warp == 0) {
            // -------------------------------------------------------- producer
            // Both CTAs walk the same items and tiles.  Per item: its Q rows
            // into Q buffer (item parity) as soon as that buffer is free (item
            // it-2's last S), then per tile c the skewed K/V copies: K(c) and
            // V(c-1) complete tile c's barrier, in CTA 0, which CTA 0 arms
            // with both CTAs' bytes.
            if (lane == 0) {
                int kv_iter = 0, it = 0;
                bool ok = true;
                bool pv_have = false;
                int pv_k0 = 0, pv_z = 0;
                auto wait_prev_v = [&](int c_next) -> bool {
                    const int vc = c_next - 1;
                    return mbar_wait(BAR(L::V_EMPTY + vc % NST), ((vc / NST) & 1) ^ 1, abort_flag,
                                     p.status, p.wait_ns);
                };
                auto issue_prev_v = [&](int c_next, uint32_t cl_bar) {
                    tma_load_3d_pair(sV + ((c_next - 1) % NST) * L::VH, &tmV, cl_bar,
                                     rank * (HD / 2), pv_k0, pv_z);
                };
                for (int t = duo_item_rank(cl, 0); ok && t < num_items;
                     t = duo_item_rank(cl, ++it)) {
                    int b, u, qt, off;
                    cl2_item(t, p, b, u, qt);
                    const TileRange tr = item_tiles<false>(p, b, qt, 0, off);
                    const int h = 2 * u + rank;
                    const int z = b * p.Hkv + (2 * u) / p.G;
                    const int qb = it & 1;
                    if (!mbar_wait(BAR(L::Q_EMPTY + qb), ((it >> 1) & 1) ^ 1, abort_flag, p.status,
                                   p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    if (rank == 0) mbar_expect_tx(BAR(L::Q_FULL + qb), 2 * L::QB);
                    for (int c = 0; c < HD / 64; ++c)
                        tma_load_3d_pair(sQ + qb * L::QB + c * (BM * 128), &tmQ, LBAR(L::Q_FULL + qb),
                                         c * 64, qt * BM, b * p.H + h);
                    for (int j = 0; ok && j < tr.count; ++j, ++kv_iter) {
                        const int st = kv_iter % NST;
                        const uint32_t ph = (kv_iter / NST) & 1;
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
                                           2u * (L::KH + (pv_have ? L::VH : 0u)));
                        if (pv_have) issue_prev_v(kv_iter, LBAR(L::K_FULL + st));
                        for (int c = 0; c < HD / 64; ++c)
                            tma_load_3d_pair(sK + st * L::KH + c * (BN / 2 * 128), &tmKh,
                                             LBAR(L::K_FULL + st), c * 64, kt.k0 + rank * (BN / 2), z);
                        pv_have = true;
                        pv_k0 = kt.k0;
                        pv_z = z;
                    }
                }
                // the last tile's V, on the barrier of the tile after it (whose
                // previous phase must be complete before it is armed again)
                if (ok && pv_have) {
                    const int st = kv_iter % NST;
                    const uint32_t ph = (kv_iter / NST) & 1;
                    if (wait_prev_v(kv_iter) &&
                        mbar_wait(BAR(L::KV_EMPTY + st), ph ^ 1, abort_flag, p.status, p.wait_ns)) {
                        if (rank == 0) mbar_expect_tx(BAR(L::K_FULL + st), 2u * L::VH);
                        issue_prev_v(kv_iter, LBAR(L::K_FULL + st));
                    }
                }
            }
        } else if (warp == 1 && rank == 0) {
            // ------------------------------------------------------ MMA issuer
            const uint32_t idesc_s = idesc_bf16_f32(256, BN, 0);
            const uint32_t idesc_o = idesc_bf16_f32(256, HD, 1);
            constexpr uint16_t BOTH = 3;
            int c = 0, it = 0;
            bool ok = true;
            bool have_prev = false, prev_first = false, prev_last = false;
            int prev_c = 0, prev_it = 0;
            auto wait_cl = [&](uint32_t bar, uint32_t parity) -> bool {
                const bool r_ok = mbar_wait_cluster(bar, parity, abort_flag, p.status, p.wait_ns);
                return __all_sync(0xffffffffu, r_ok);
            };
            // P(prev) V into the O buffer of the item it belongs to, keys 0..63
            // on the left softmax's P, keys 64..127 on the right's
            auto issue_pv = [&]() -> bool {
                const int pb = prev_c & 1, pst = prev_c % NST;
                const uint32_t par = (prev_c >> 1) & 1;
                const uint32_t o_t = tmem + (prev_it & 1) * 128;
                const uint32_t p_t = tmem + 256 + pb * 128;
                if (!wait_cl(BAR(L::P_LEFT + pb), par)) return false;
                if (prev_first &&
                    !wait_cl(BAR(L::O_EMPTY + (prev_it & 1)), ((prev_it >> 1) & 1) ^ 1))
                    return false;
                tc_fence_after();
                const uint64_t vb = smem_desc_sw128(sV + pst * L::VH, BN * 128, 1024);
                mma2_ts_group4(o_t, p_t, vb, idesc_o, prev_first ? 0u : 1u);
                if (!wait_cl(BAR(L::P_RIGHT + pb), par)) return false;
                tc_fence_after();
                // keys 64..127: P columns 64.., V rows 64.. (64 * 128 B >> 4)
                mma2_ts_group4(o_t, p_t + 64, vb + 512, idesc_o, 1u);
                tc_commit2_mc(BAR(L::V_EMPTY + pst), BOTH);
                tc_commit2_mc(BAR(L::PV_DONE + pb), BOTH);
                if (prev_last) tc_commit2_mc(BAR(L::O_FULL + (prev_it & 1)), BOTH);
                return true;
            };
            for (int t = duo_item_rank(cl, 0); ok && t < num_items; t = duo_item_rank(cl, ++it)) {
                int b, u, qt, off;
                cl2_item(t, p, b, u, qt);
                const TileRange tr = item_tiles<false>(p, b, qt, 0, off);
                const int qb = it & 1;
                for (int j = 0; j < tr.count; ++j, ++c) {
                    const int st = c % NST;
                    const uint32_t ph = (c / NST) & 1;
                    const bool last = (j == tr.count - 1);
                    if (!wait_cl(BAR(L::K_FULL + st), ph) ||
                        (j == 0 && !wait_cl(BAR(L::Q_FULL + qb), (it >> 1) & 1))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // S(c) = Q K(c)^T into S buffer c % 2
                    {
                        const uint64_t qd = smem_desc_sw128(sQ + qb * L::QB, 16, 1024);
                        const uint64_t kd = smem_desc_sw128(sK + st * L::KH, 16, 1024);
                        mma2_ss_group8(tmem + 256 + (c & 1) * 128, qd, kd, idesc_s);
                        tc_commit2_mc(BAR(L::S_FULL + (c & 1)), BOTH);
                        if (last) tc_commit2_mc(BAR(L::Q_EMPTY + qb), BOTH);
                        tc_commit2_mc(BAR(L::KV_EMPTY + st), BOTH);  // the K slot
                    }
                    // then P(c-1) V (the previous tile, possibly the previous item's)
                    if (have_prev && !issue_pv()) {
                        ok = false;
                        break;
                    }
                    have_prev = true;
                    prev_c = c;
                    prev_it = it;
                    prev_first = (j == 0);
                    prev_last = last;
                }
            }
            // the last tile's V rides on the barrier of the tile after it
            if (ok && have_prev && wait_cl(BAR(L::K_FULL + c % NST), (c / NST) & 1)) issue_pv();
            tc_commit2_mc(BAR(L::DRAIN), 1);
            warp_wait(BAR(L::DRAIN), 0, nullptr, nullptr, TIMEOUT_NS);
        }
    } else if (warp < 12) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REGS_SOFTMAX));
        // ------------------------------------------------------------ softmax
        // Side s of the CTA's rows: key columns 64s .. 64s+63 of every tile.
        // The warps of the two sides that hold the same 32 rows (TMEM lane
        // quarter q) post their partial row maxima in shared memory and meet
        // on mbarrier MAXX[q][tile parity] (a bounded wait: a named barrier
        // could wait forever for a side that gave up), so both use the same
        // running maximum m; each keeps its own part of the row sum l and
        // rescales its own half of O.
        const int s = (warp >> 2) - 1;
        const int q = warp & 3;
        const int r = q * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        const float sl2 = p.sl2;
        const uint64_t sl2x2 = pack2(__float_as_uint(sl2), __float_as_uint(sl2));
        float *maxbuf = reinterpret_cast<float *>(smem + L::MAX_OFF);
        float2 *stats = reinterpret_cast<float2 *>(smem + L::STATS_OFF);
        const uint32_t p_bar = s == 0 ? LBAR(L::P_LEFT) : LBAR(L::P_RIGHT);
        int c = 0, it = 0;
        bool ok = true;
        for (int t = duo_item_rank(cl, 0); ok && t < num_items; t = duo_item_rank(cl, ++it)) {
            int b, u, qt, off;
            cl2_item(t, p, b, u, qt);
            const TileRange tr = item_tiles<false>(p, b, qt, 0, off);
            const int i = tr.q0 + r;
            const int lo = i - p.w + 1;
            const uint32_t o_addr = tmem + lane_off + (it & 1) * 128 + s * 64;
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < tr.count; ++j, ++c) {
                const int sbuf = c & 1;
                if (!warp_wait(BAR(L::S_FULL + sbuf), (c >> 1) & 1, abort_flag, p.status,
                               p.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t s_addr = tmem + lane_off + 256 + sbuf * 128;
                uint32_t sv[2][32];
                tmem_ld32(s_addr + s * 64, sv[0]);
                tmem_ld32(s_addr + s * 64 + 32, sv[1]);
                tmem_ld_wait();
                reg_fence32(sv[0]);
                reg_fence32(sv[1]);
                const KeyTile kt = key_tile<false>(tr, j, p);
                if (!kt.full) {
                    // k <= i and (k >= i-w+1 or k < g), in this side's tile columns
                    const int k0 = kt.k0 + s * 64;
                    const int ca = lo - k0, cb = i - k0, cg = p.g - k0;
#pragma unroll
                    for (int qq = 0; qq < 2; ++qq)
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const int cc = qq * 32 + e;
                            if (!(cc <= cb && (cc >= ca || cc < cg)))
                                sv[qq][e] = __float_as_uint(-INFINITY);
                        }
                }
                float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    mx0 = max3(mx0, __uint_as_float(sv[0][e]), __uint_as_float(sv[0][e + 1]));
                    mx1 = max3(mx1, __uint_as_float(sv[1][e]), __uint_as_float(sv[1][e + 1]));
                }
                // the row maximum over both sides
                float *mb = maxbuf + sbuf * 2 * BM;
                mb[s * BM + r] = fmaxf(mx0, mx1);
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(L::MAXX + 2 * q + sbuf));
                if (!warp_wait(BAR(L::MAXX + 2 * q + sbuf), (c >> 1) & 1, abort_flag, p.status,
                               p.wait_ns)) {
                    ok = false;
                    break;
                }
                const float m_tile = fmaxf(mb[r], mb[BM + r]) * sl2;
                const float m_new = fmaxf(m, m_tile);
                if (j == 0) {
                    m = m_new;
                } else {
                    const bool need = m_new > m + RESCALE_LOG2;
                    if (__any_sync(0xffffffffu, need)) {
                        // this side's half of O, once the previous tile's P V is in
                        if (!warp_wait(BAR(L::PV_DONE + ((c - 1) & 1)), ((c - 1) >> 1) & 1,
                                       abort_flag, p.status, p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const float alpha = need ? ex2(m - m_new) : 1.f;
                        if (need) m = m_new;
                        l *= alpha;
#pragma unroll 1
                        for (int qq = 0; qq < 2; ++qq) {
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
                softmax_half(sv[0], sv[1], sl2x2, negm2, acc2, pk);
                // P of this side's 64 keys over its own first 32 S columns
                tmem_st32(s_addr + s * 64, pk);
                float a0, a1;
                unpack2(acc2, a0, a1);
                l += a0 + a1;
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(p_bar + 8u * static_cast<uint32_t>(sbuf));
            }
            if (!ok) break;
            // this side's (m, l) for the epilogue, once it has read item it-2's
            if (!warp_wait(BAR(L::STATS_EMPTY + (it & 1)), ((it >> 1) & 1) ^ 1, abort_flag,
                           p.status, p.wait_ns)) {
                ok = false;
                break;
            }
            stats[((it & 1) * 2 + s) * BM + r] = make_float2(m, l);
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(L::ROW_STATS + (it & 1)));
        }
        if (!ok) *abort_flag = 1;
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_EPI));
        // ------------------------------------------------------------ epilogue
        // Per item: both sides' (m, l) and the item's last P V, then O / l as
        // bf16 (and the LSE) for this CTA's head; the O buffer is released on
        // CTA 0's O_EMPTY barrier.
        const int sub = warp & 3;
        const int r = sub * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(sub * 32) << 16;
        const float2 *stats = reinterpret_cast<const float2 *>(smem + L::STATS_OFF);
        uint8_t *stage = smem + L::STAGE_OFF + sub * STAGE_WARP;
        int it = 0;
        for (int t = duo_item_rank(cl, 0); t < num_items; t = duo_item_rank(cl, ++it)) {
            int b, u, qt, off;
            cl2_item(t, p, b, u, qt);
            const TileRange tr = item_tiles<false>(p, b, qt, 0, off);
            const int ib = it & 1;
            if (!warp_wait(BAR(L::ROW_STATS + ib), (it >> 1) & 1, abort_flag, p.status, p.wait_ns) ||
                !warp_wait(BAR(L::O_FULL + ib), (it >> 1) & 1, abort_flag, p.status, p.wait_ns))
                break;
            tc_fence_after();
            const float2 s0 = stats[(ib * 2 + 0) * BM + r], s1 = stats[(ib * 2 + 1) * BM + r];
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(L::STATS_EMPTY + ib));
            const int h = 2 * u + rank;
            float row_lse;
            const float inv_l = finish_row(s0.x, s0.y + s1.y, p.sink, h, &row_lse);
            const int t_row = tr.q0 + r - off;
            const bool row_ok = t_row < p.n;
            const size_t orow_i = static_cast<size_t>(b * p.H + h) * p.n + t_row;
            store_o_rows_chunked<HD, true>(tmem + lane_off + ib * 128, inv_l, p.O + orow_i * HD,
                                           row_ok, stage, lane, LBAR(L::O_EMPTY + ib));
            if (p.lse != nullptr && row_ok) p.lse[orow_i] = row_lse;
        }
    }
#undef LBAR
#undef BAR
    // neither CTA leaves (nor frees its tensor memory) while the other may
    // still reach its barriers or tensor memory
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc2(tmem, TMEM_COLS);
    }
}
