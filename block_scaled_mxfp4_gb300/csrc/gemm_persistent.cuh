// Persistent stream-K form of the block-scaled MXFP4 GEMM (included by
// gemm_sm103.cu, which provides Cfg, the scale-atom helpers, the epilogue
// stores and the device status word).
//
// Grid = G CTAs, all resident.  CTA c walks a list of work items
// (tile, K-stage range): first whole tiles c, c+G, ... for the full waves,
// then its share [c*S/G, (c+1)*S/G) of the remaining tiles' K stages, so every
// CTA gets the same number of stages.  A stream-K tile is split into
// consecutive K segments owned by consecutive CTAs; the owner of segment 0
// (which reaches it last, at the end of its own list) completes the tile:
// it waits for the per-CTA ready flags of the other owners, adds their fp32
// partials to its own accumulator in segment order (deterministic), and
// writes D.  Every other segment owner writes its partial and sets its flag
// to this call's epoch (a per-call number that is never 0, so flags left by
// earlier calls never look ready).  A CTA writes at most one partial (its
// first item) and completes at most one tile this way (its last item).  The
// completing CTA brings the partials in with bulk copies into its (by then
// idle) operand ring, two 32-column chunks in flight at a time.
//
// Roles as in the one-tile kernel (warps 0-3 epilogue, 4 TMA producer, 5 MMA);
// the accumulator has NACC TMEM buffers, and the epilogue hands a buffer back
// to the MMA warp as soon as it has read it, so the next item's MMAs overlap
// the previous item's stores.
//
// Scales, in the order the producer prefers them:
//   relaid atoms (prepacked)  one bulk copy per 128-row block per stage;
//   row-major, TMA-able       one 2-D TMA per operand per PAIR of stages
//                             (a 16-byte x rows box = 16 scale blocks per row)
//                             into an NSLOT-deep staging ring requested up to
//                             NSLOT-1 pairs ahead; the warp then rebuilds the
//                             stage's atoms from shared memory (8-byte reads,
//                             16-byte writes per lane);
//   row-major, 4-byte aligned 4-byte cp.async per scale word;
//   otherwise                 plain loads by the warp.
#pragma once

namespace mxfp4 {

enum ItemKind : int { kItemFull = 0, kItemPartial = 1, kItemFinal = 2 };

struct Item {
    int tile, k0, k1, kind;
    int wait_lo, wait_hi;   // kItemFinal: the CTAs whose partials complete the tile
};

__device__ __forceinline__ long long sk_bound(const Sched &s, int c)
{
    return static_cast<long long>(c) * s.sk_units / s.ctas;
}

// Whether CTA c has any stream-K units (with fewer units than CTAs some ranges
// are empty; such CTAs write no partial and must not be waited for).
__device__ __forceinline__ bool sk_has_units(const Sched &s, int c)
{
    return sk_bound(s, c) < sk_bound(s, c + 1);
}

// CTA whose stream-K range holds unit u.
__device__ __forceinline__ int sk_owner(const Sched &s, long long u)
{
    int c = static_cast<int>(u * s.ctas / s.sk_units);
    if (c > s.ctas - 1)
        c = s.ctas - 1;
    while (c < s.ctas - 1 && sk_bound(s, c + 1) <= u)
        ++c;
    while (c > 0 && sk_bound(s, c) > u)
        --c;
    return c;
}

struct ItemIter {
    int cta, j;
    long long u, uend;
    __device__ ItemIter(const Sched &s, int c)
        : cta(c), j(0), u(sk_bound(s, c)), uend(sk_bound(s, c + 1)) {}

    __device__ bool next(const Sched &s, Item &it)
    {
        it.wait_lo = it.wait_hi = 0;
        if (j < s.dp_waves) {
            it.tile = cta + j * s.ctas;
            it.k0 = 0;
            it.k1 = s.kt;
            it.kind = kItemFull;
            ++j;
            return true;
        }
        if (u >= uend)
            return false;
        const long long tl = u / s.kt;
        const int k0 = static_cast<int>(u - tl * s.kt);
        const long long rem = uend - u;
        const int k1 = static_cast<int>(min(static_cast<long long>(s.kt), k0 + rem));
        it.tile = s.sk_tile0 + static_cast<int>(tl);
        it.k0 = k0;
        it.k1 = k1;
        if (k0 == 0 && k1 == s.kt) {
            it.kind = kItemFull;
        } else if (k0 == 0) {
            it.kind = kItemFinal;
            it.wait_lo = cta + 1;
            it.wait_hi = sk_owner(s, (tl + 1) * s.kt - 1);
        } else {
            it.kind = kItemPartial;
        }
        u += k1 - k0;
        return true;
    }
};

// The (tile, stage pair) sequence a CTA consumes, for scale requests ahead
// of the stages that use them.  Pair p covers stages 2p and 2p+1.
struct PairCursor {
    ItemIter it;
    Item cur;
    bool valid;
    int pair, pair_end;
    __device__ PairCursor(const Sched &s, int c) : it(s, c)
    {
        valid = it.next(s, cur);
        if (valid) {
            pair = cur.k0 / 2;
            pair_end = (cur.k1 - 1) / 2;
        }
    }
    __device__ bool next(const Sched &s, int &tile, int &pr)
    {
        if (!valid)
            return false;
        tile = cur.tile;
        pr = pair;
        if (++pair > pair_end) {
            valid = it.next(s, cur);
            if (valid) {
                pair = cur.k0 / 2;
                pair_end = (cur.k1 - 1) / 2;
            }
        }
        return true;
    }
};

// Tile t -> (tile row along P, tile column along Q), rows grouped by s.group
// so that the tiles in flight at once share a few P panels.
__device__ __forceinline__ void tile_coords(const Sched &s, int t, int &pt, int &qt)
{
    const int per_group = s.group * s.tiles_q;
    const int g = t / per_group;
    const int within = t - g * per_group;
    const int gh = min(s.group, s.tiles_p - g * s.group);
    pt = g * s.group + within % gh;
    qt = within / gh;
}

__device__ __forceinline__ int ld_acquire(const int *p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(int *p, int v)
{
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

template <int BN, int STAGES, int NACC, int NSLOT>
struct PCfg {
    using Base = Cfg<BN, STAGES>;
    static constexpr int TMEM_USED = NACC * BN + STAGES * Base::SF_COLS;
    static constexpr int TMEM_COLS = TMEM_USED <= 32    ? 32
                                     : TMEM_USED <= 64  ? 64
                                     : TMEM_USED <= 128 ? 128
                                     : TMEM_USED <= 256 ? 256
                                                        : 512;
    static constexpr int RING_BYTES = STAGES * Base::STAGE_BYTES;
    static constexpr int STG_P = kTileM * 16;               // 128 rows x 16 scale bytes
    static constexpr int STG_Q = BN * 16;                   // BN rows x 16 scale bytes
    static constexpr int SLOT_BYTES = STG_P + STG_Q;
    static constexpr int BAR_BYTES = 512;
    static constexpr int SMEM_BYTES = RING_BYTES + NSLOT * SLOT_BYTES + BAR_BYTES + 1024;
    static constexpr int FIX_CHUNK = 32 * kTileM * 4;       // one 32-column partial chunk
    static constexpr int FIX_CAP = RING_BYTES / 2 / FIX_CHUNK;  // chunks per fix-up buffer
    static_assert(TMEM_USED <= 512, "tensor memory budget");
    static_assert(NACC == 1 || NACC == 2, "accumulator buffers");
    static_assert(NSLOT >= 2, "scale staging ring");
    static_assert(SLOT_BYTES % 1024 == 0, "staging alignment");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static_assert(FIX_CAP >= 2, "fix-up buffers");
};

template <int BN, int STAGES, bool SWAP, int NACC, int NSLOT>
__global__ void __launch_bounds__(192, 1)
    gemm_mxf4_persistent(const __grid_constant__ GemmArgs a, const __grid_constant__ Sched sch,
                         const __grid_constant__ CUtensorMap tmP,
                         const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmSP,
                         const __grid_constant__ CUtensorMap tmSQ)
{
    using Cf = Cfg<BN, STAGES>;
    using PC = PCfg<BN, STAGES, NACC, NSLOT>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t *stg = smem + PC::RING_BYTES;                    // scale staging ring
    uint64_t *full = reinterpret_cast<uint64_t *>(stg + NSLOT * PC::SLOT_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *acc_full = empty + STAGES;
    uint64_t *acc_empty = acc_full + NACC;
    uint64_t *epi_go = acc_empty + NACC;   // flags of a final item have all been seen
    uint64_t *epi_done = epi_go + 1;       // all epilogue warps finished an item's stores
    uint64_t *drain = epi_done + 1;        // MMA drain on abort
    uint64_t *sf_full = drain + 1;         // [NSLOT] scale staging slots landed
    uint64_t *sf_empty = sf_full + NSLOT;  // [NSLOT] scale staging slots consumed
    uint64_t *fix_full = sf_empty + NSLOT; // [2] fix-up chunk buffers landed
    uint64_t *fix_free = fix_full + 2;     // [2] fix-up chunk buffers read by all warps
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fix_free + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cta = blockIdx.x;

    if (threadIdx.x == 0) {
        const uint32_t full_count = (a.sf_tma || !a.sf_rowmajor) ? 1 : a.sf_async ? 33 : 2;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], full_count);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < NACC; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], 4);
        }
        mbar_init(epi_go, 1);
        mbar_init(epi_done, 4);
        mbar_init(drain, 1);
        for (int i = 0; i < NSLOT; ++i) {
            mbar_init(&sf_full[i], 1);
            mbar_init(&sf_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&fix_full[i], 1);
            mbar_init(&fix_free[i], 4);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(tmem_slot, PC::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
        prefetch_tensormap(&tmP);
        prefetch_tensormap(&tmQ);
        if (a.sf_tma) {
            prefetch_tensormap(&tmSP);
            prefetch_tensormap(&tmSQ);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int kblocks = a.K / 32;

    if (warp == 4) {
        // ------------------------------------------------------ producer --
        const uint64_t pol_p = a.stream_p ? l2_policy_evict_first() : l2_policy_evict_last();
        const uint64_t pol_q = l2_policy_evict_last();
        // Row-major scales without TMA: the whole warp builds the atoms.
        const bool warp_sf = a.sf_rowmajor != 0 && !a.sf_tma;
        ItemIter it(sch, cta);
        PairCursor pc(sch, cta);
        Item item;
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;
        int n_req = 0, n_pass = 0;                     // scale pairs requested / reached
        bool stop = false;
        while (!stop && it.next(sch, item)) {
            int pt, qt;
            tile_coords(sch, item.tile, pt, qt);
            const int p0 = pt * kTileM, q0 = qt * BN;
            for (int kt = item.k0; kt < item.k1; ++kt) {
                bool ok = true;
                if (warp_sf || lane == 0)
                    ok = mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.wait_limit,
                                   &g_device_status);
                if (warp_sf)
                    ok = __all_sync(0xffffffffu, ok);
                if (!ok) {
                    stop = true;
                    break;
                }
                uint8_t *st = smem + stage * Cf::STAGE_BYTES;
                uint8_t *sf_s = st + Cf::P_BYTES + Cf::Q_BYTES;
                if (a.sf_tma) {
                    // One thread: operand tiles, and the scale pairs up to
                    // NSLOT-1 pairs ahead (a slot is reused once the MMA warp
                    // has rebuilt the atoms of the pair it held).
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&full[stage], Cf::P_BYTES + Cf::Q_BYTES);
                        tma_load_2d(st, &tmP, &full[stage], kt * 128, p0, pol_p);
                        tma_load_2d(st + Cf::P_BYTES, &tmQ, &full[stage], kt * 128, q0, pol_q);
                        if (kt == item.k0 || (kt & 1) == 0) {
                            ++n_pass;
                            int rt, rp;
                            while (!stop && n_req < n_pass - 1 + NSLOT && pc.next(sch, rt, rp)) {
                                const int slot = n_req % NSLOT;
                                if (n_req >= NSLOT &&
                                    !mbar_wait(&sf_empty[slot], ((n_req / NSLOT) - 1) & 1u,
                                               abort_flag, a.wait_limit, &g_device_status)) {
                                    stop = true;
                                    break;
                                }
                                int rpt, rqt;
                                tile_coords(sch, rt, rpt, rqt);
                                uint8_t *dst = stg + slot * PC::SLOT_BYTES;
                                mbar_arrive_expect_tx(&sf_full[slot], PC::SLOT_BYTES);
                                tma_load_2d(dst, &tmSP, &sf_full[slot], rp * 16, rpt * kTileM,
                                            pol_p);
                                tma_load_2d(dst + PC::STG_P, &tmSQ, &sf_full[slot], rp * 16,
                                            rqt * BN, pol_q);
                                ++n_req;
                            }
                        }
                    }
                } else if (!warp_sf) {
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&full[stage], Cf::STAGE_BYTES);
                        tma_load_2d(st, &tmP, &full[stage], kt * 128, p0, pol_p);
                        tma_load_2d(st + Cf::P_BYTES, &tmQ, &full[stage], kt * 128, q0, pol_q);
                        const int64_t sf_off = static_cast<int64_t>(kt) * 2 * kSfAtomBytes;
                        bulk_load(sf_s,
                                  a.sfP + static_cast<int64_t>(p0 / kSfRowBlock) * a.sf_rb_stride +
                                      sf_off,
                                  Cf::SFP_BYTES, &full[stage], pol_p);
#pragma unroll
                        for (int r = 0; r < Cf::NQ; ++r)
                            bulk_load(sf_s + Cf::SFP_BYTES + r * 2 * kSfAtomBytes,
                                      a.sfQ +
                                          static_cast<int64_t>(q0 / kSfRowBlock + r) *
                                              a.sf_rb_stride +
                                          sf_off,
                                      2 * kSfAtomBytes, &full[stage], pol_q);
                    }
                } else {
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&full[stage], Cf::P_BYTES + Cf::Q_BYTES);
                        tma_load_2d(st, &tmP, &full[stage], kt * 128, p0, pol_p);
                        tma_load_2d(st + Cf::P_BYTES, &tmQ, &full[stage], kt * 128, q0, pol_q);
                    }
                    if (a.sf_async) {
                        copy_sf_rows_async(sf_s, a.sfP, a.ldsP, a.rowsP, kblocks, p0, kt, lane);
#pragma unroll
                        for (int r = 0; r < Cf::NQ; ++r)
                            copy_sf_rows_async(sf_s + Cf::SFP_BYTES + r * 2 * kSfAtomBytes, a.sfQ,
                                               a.ldsQ, a.rowsQ, kblocks, q0 + r * kSfRowBlock, kt,
                                               lane);
                        cp_async_mbar_arrive(&full[stage]);
                    } else {
                        uint32_t w[4][2];
                        load_sf_rows(a.sfP, a.ldsP, a.rowsP, kblocks, p0, kt, a.sf_vec8, lane, w);
                        store_sf_lines(sf_s, w, lane);
#pragma unroll
                        for (int r = 0; r < Cf::NQ; ++r) {
                            load_sf_rows(a.sfQ, a.ldsQ, a.rowsQ, kblocks, q0 + r * kSfRowBlock, kt,
                                         a.sf_vec8, lane, w);
                            store_sf_lines(sf_s + Cf::SFP_BYTES + r * 2 * kSfAtomBytes, w, lane);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0)
                            mbar_arrive(&full[stage]);
                    }
                }
                ++issued;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (lane == 0 && *abort_flag) {
            for (int i = max(0, issued - STAGES); i < issued; ++i)
                mbar_wait_drain(&full[i % STAGES], (i / STAGES) & 1u, a.wait_limit);
            for (int n = max(0, n_req - NSLOT); n < n_req; ++n)
                mbar_wait_drain(&sf_full[n % NSLOT], (n / NSLOT) & 1u, a.wait_limit);
        }
    } else if (warp == 5) {
        // ---------------------------------------------------- MMA issuer --
        // One thread issues the tensor-core work.  With TMA-staged scales the
        // whole warp first rebuilds each stage's atoms from the staging ring
        // (and fences its own writes for the async proxy).
        const bool warp_mma = a.sf_tma != 0;
        if (warp_mma || lane == 0) {
            const uint32_t idesc = idesc_mxf4(kTileM, BN);
            const uint32_t t_sf = tmem + NACC * BN;
            ItemIter it(sch, cta);
            Item item;
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            int n_con = 0, cslot = 0;
            bool stop = false;
            while (!stop && it.next(sch, item)) {
                bool ok = mbar_wait(&acc_empty[acc], acc_phase ^ 1u, abort_flag, a.wait_limit,
                                    &g_device_status);
                if (warp_mma)
                    ok = __all_sync(0xffffffffu, ok);
                if (!ok)
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + acc * BN;
                int pt, qt;
                tile_coords(sch, item.tile, pt, qt);
                const uint32_t q_off =
                    (BN < 128 && !a.sf_rowmajor)
                        ? static_cast<uint32_t>(((qt * BN) % kSfRowBlock) / 32)
                        : 0u;
                for (int kt = item.k0; kt < item.k1; ++kt) {
                    ok = mbar_wait(&full[stage], phase, abort_flag, a.wait_limit, &g_device_status);
                    if (warp_mma)
                        ok = __all_sync(0xffffffffu, ok);
                    if (!ok) {
                        stop = true;
                        break;
                    }
                    uint8_t *st = smem + stage * Cf::STAGE_BYTES;
                    uint8_t *sf_s = st + Cf::P_BYTES + Cf::Q_BYTES;
                    if (warp_mma) {
                        if (kt == item.k0 || (kt & 1) == 0) {
                            cslot = n_con % NSLOT;
                            const uint32_t cph = static_cast<uint32_t>(n_con / NSLOT) & 1u;
                            ++n_con;
                            ok = mbar_wait(&sf_full[cslot], cph, abort_flag, a.wait_limit,
                                           &g_device_status);
                            if (!__all_sync(0xffffffffu, ok)) {
                                stop = true;
                                break;
                            }
                        }
                        // Atoms of this stage from half (kt & 1) of each staged row.
                        const uint8_t *sp = stg + cslot * PC::SLOT_BYTES + 8 * (kt & 1);
                        uint32_t w[4][2];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint2 v =
                                *reinterpret_cast<const uint2 *>(sp + (lane + 32 * j) * 16);
                            w[j][0] = v.x;
                            w[j][1] = v.y;
                        }
                        store_sf_lines(sf_s, w, lane);
#pragma unroll
                        for (int r = 0; r < Cf::NQ; ++r) {
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const int qr = r * kSfRowBlock + lane + 32 * j;
                                if (qr < BN) {
                                    const uint2 v = *reinterpret_cast<const uint2 *>(
                                        sp + PC::STG_P + qr * 16);
                                    w[j][0] = v.x;
                                    w[j][1] = v.y;
                                } else {
                                    w[j][0] = w[j][1] = 0u;
                                }
                            }
                            store_sf_lines(sf_s + Cf::SFP_BYTES + r * 2 * kSfAtomBytes, w, lane);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0 && ((kt & 1) == 1 || kt + 1 == item.k1))
                            mbar_arrive(&sf_empty[cslot]);   // last stage of the pair: slot free
                    } else if (a.sf_rowmajor) {
                        fence_proxy_async_smem();
                    }
                    if (lane == 0) {
                        tc_fence_after();
                        const uint32_t sfp_t = t_sf + stage * Cf::SF_COLS;
                        const uint32_t sfq_t = sfp_t + Cf::SF_COLS_P;
                        const uint32_t sfp_s = smem_addr(sf_s);
                        const uint32_t sfq_s = sfp_s + Cf::SFP_BYTES;
#pragma unroll
                        for (int g = 0; g < 2; ++g) {
                            tmem_cp_32x128b_x4(sfp_t + g * 4,
                                               sdesc_sf_block(sfp_s + g * kSfAtomBytes));
#pragma unroll
                            for (int r = 0; r < Cf::NQ; ++r)
                                tmem_cp_32x128b_x4(sfq_t + g * 4 * Cf::NQ + r * 4,
                                                   sdesc_sf_block(sfq_s + r * 2 * kSfAtomBytes +
                                                                  g * kSfAtomBytes));
                        }
                        const uint64_t adesc = sdesc_kmajor_sw128(smem_addr(st));
                        const uint64_t bdesc = sdesc_kmajor_sw128(smem_addr(st + Cf::P_BYTES));
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint32_t sf_id = (j & 1) * 2;
                            mma_mxf4(d_tmem, adesc + 2 * j, bdesc + 2 * j,
                                     idesc_sf_ids(idesc, sf_id, sf_id), sfp_t + (j >> 1) * 4,
                                     sfq_t + (j >> 1) * 4 * Cf::NQ + q_off,
                                     (kt > item.k0 || j > 0) ? 1u : 0u);
                        }
                        mma_commit(&empty[stage]);
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (lane == 0)
                    mma_commit(&acc_full[acc]);
                if (++acc == NACC) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (lane == 0 && *abort_flag) {
                mma_commit(drain);
                mbar_wait_drain(drain, 0, a.wait_limit);   // MMAs in flight land first
            }
        }
    } else {
        // ------------------------------------------------------ epilogue --
        const int row = warp * 32 + lane;
        ItemIter it(sch, cta);
        Item item;
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t done_phase = 0;
        while (it.next(sch, item)) {
            bool ok = mbar_wait(&acc_full[acc], acc_phase, abort_flag, a.wait_limit,
                                &g_device_status);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok)
                break;
            tc_fence_after();
            int pt, qt;
            tile_coords(sch, item.tile, pt, qt);
            const int p0 = pt * kTileM, q0 = qt * BN;
            const int qrows = SWAP ? a.M : a.N;
            const bool final_item = item.kind == kItemFinal;
            // Completing CTA: the contributing CTAs (non-empty ranges, in
            // segment order), of which the first FIX_CAP come in by bulk copy.
            int contrib[PC::FIX_CAP];
            int ncontrib = 0;
            int chunks = 0;                            // 32-column chunks of the tile to write
            if (final_item) {
                if (threadIdx.x == 0) {
                    for (int c = item.wait_lo; c <= item.wait_hi; ++c) {
                        if (!sk_has_units(sch, c))
                            continue;
                        const long long t0 = clock64();
                        while (ld_acquire(sch.flags + c) != sch.epoch) {
                            if (*abort_flag)
                                break;
                            if (clock64() - t0 > a.wait_limit) {
                                atomicExch(&g_device_status, -6);
                                *abort_flag = 1;
                                break;
                            }
                        }
                    }
                    mbar_arrive(epi_go);
                }
                ok = mbar_wait(epi_go, 0, abort_flag, a.wait_limit, &g_device_status);
                ok = __all_sync(0xffffffffu, ok && !*abort_flag);
                for (int c = item.wait_lo; c <= item.wait_hi && ncontrib < PC::FIX_CAP; ++c)
                    if (sk_has_units(sch, c))
                        contrib[ncontrib++] = c;
                for (int c0 = 0; c0 < BN && c0 < sch.pcols; c0 += 32)
                    ++chunks;
                if (SWAP)
                    chunks = min(chunks, (a.M - q0 + 31) / 32);
            }
            // Bulk copies of chunk ci of every bulk contributor into buffer ci & 1.
            const uint64_t pol_fix = l2_policy_evict_first();
            auto fix_issue = [&](int ci) {
                const int c0 = ci * 32;
                const int ncols = min(32, sch.pcols - c0);
                uint8_t *buf = smem + (ci & 1) * (PC::RING_BYTES / 2);
                mbar_arrive_expect_tx(&fix_full[ci & 1], ncontrib * ncols * kTileM * 4);
                for (int k = 0; k < ncontrib; ++k)
                    bulk_load(buf + k * PC::FIX_CHUNK,
                              sch.partials + (static_cast<int64_t>(contrib[k]) * sch.pcols + c0) *
                                                 kTileM,
                              ncols * kTileM * 4, &fix_full[ci & 1], pol_fix);
            };
            if (final_item && ok && threadIdx.x == 0 && chunks > 0)
                fix_issue(0);
            const uint32_t t_row = tmem + acc * BN + (static_cast<uint32_t>(warp * 32) << 16);
            bool released = false;
#pragma unroll 1
            for (int ci = 0, c0 = 0; c0 < BN; ++ci, c0 += 32) {
                if (SWAP && q0 + c0 >= a.M)
                    break;                                   // padding columns of D^T
                if (final_item && ok && threadIdx.x == 0 && ci + 1 < chunks) {
                    // Prefetch the next chunk once its buffer has been read.
                    if (ci >= 1)
                        mbar_wait(&fix_free[(ci + 1) & 1], ((ci - 1) >> 1) & 1u, abort_flag,
                                  a.wait_limit, &g_device_status);
                    fix_issue(ci + 1);
                }
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_row + c0, r);
                tmem_ld_wait();
                if (c0 + 32 >= BN || (SWAP && q0 + c0 + 32 >= a.M)) {
                    // Accumulator fully read: hand it back to the MMA warp.
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&acc_empty[acc]);
                    released = true;
                }
                if (!ok)
                    continue;
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    v[i] = __uint_as_float(r[i]);
                if (item.kind == kItemPartial) {
                    float *dst =
                        sch.partials + (static_cast<int64_t>(cta) * sch.pcols + c0) * kTileM + row;
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (q0 + c0 + i < qrows && c0 + i < sch.pcols)
                            __stcg(dst + i * kTileM, v[i]);
                    continue;
                }
                if (final_item && ci < chunks) {
                    const bool got = mbar_wait(&fix_full[ci & 1], (ci >> 1) & 1u, abort_flag,
                                               a.wait_limit, &g_device_status);
                    const float *buf =
                        reinterpret_cast<const float *>(smem + (ci & 1) * (PC::RING_BYTES / 2));
                    if (got) {
                        // Segment order: own accumulator, then the contributors in order.
                        for (int k = 0; k < ncontrib; ++k) {
                            const float *src = buf + k * (PC::FIX_CHUNK / 4) + row;
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                if (q0 + c0 + i < qrows && c0 + i < sch.pcols)
                                    v[i] += src[i * kTileM];
                        }
                    }
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&fix_free[ci & 1]);
                    // Contributors beyond the bulk buffers (rare): read directly.
                    int seen = 0;
                    for (int c = item.wait_lo; c <= item.wait_hi; ++c) {
                        if (!sk_has_units(sch, c) || seen++ < ncontrib)
                            continue;
                        const float *src =
                            sch.partials + (static_cast<int64_t>(c) * sch.pcols + c0) * kTileM + row;
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (q0 + c0 + i < qrows && c0 + i < sch.pcols)
                                v[i] += __ldcg(src + i * kTileM);
                    }
                }
                if (!SWAP) {
                    const int m = p0 + row;
                    if (m < a.M && q0 + c0 < a.N)
                        store_d_row(a, m, q0 + c0, v);
                } else {
                    store_d_col(a, q0 + c0, p0 + row, v);
                }
            }
            if (!released) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&acc_empty[acc]);
            }
            if (item.kind == kItemPartial && ok) {
                // All four warps done with this item's partial stores: publish.
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(epi_done);
                if (threadIdx.x == 0 &&
                    mbar_wait(epi_done, done_phase, abort_flag, a.wait_limit, &g_device_status)) {
                    __threadfence();
                    st_release(sch.flags + cta, sch.epoch);   // this call's partial is ready
                }
                done_phase ^= 1u;
            }
            if (++acc == NACC) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, PC::TMEM_COLS);
    }
}

}  // namespace mxfp4
