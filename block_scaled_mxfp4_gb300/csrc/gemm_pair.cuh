// CTA-pair (2-SM) form of the block-scaled MXFP4 GEMM for large shapes
// (included by gemm_sm103.cu).
//
// A cluster of two CTAs computes one 256 x 256 output tile with
// tcgen05.mma.cta_group::2 (M = 256): CTA r of the pair holds rows
// [128r, 128r+128) of the tile's A panel and rows [128r, 128r+128) of its B
// panel (half of N) in its own shared memory, and its own 128 rows x 256
// columns of the fp32 accumulator in its own tensor memory.  Per 256-K stage
// each CTA therefore stages 16 KB of A and 16 KB of B for 128 x 256 x 256
// multiply-adds -- two thirds of the one-CTA 128 x 256 tile's 48 KB -- which
// is what lets the ring keep the tensor pipe fed from L2.
//
//   warp 4 (each CTA)  TMA producer: its A half, its B half, its 128 rows of
//                      scale-A atoms and all 256 rows of scale-B atoms; every
//                      copy is counted on the LEADER's full barrier (the
//                      cta_group::2 form of the TMA signals the pair), which
//                      only the leader arrives on, expecting both CTAs' bytes.
//   warp 5 (leader)    waits on its full barrier, copies both CTAs' scale atoms
//                      into their own tensor memory (tcgen05.cp.cta_group::2),
//                      issues four K=64 M=256 MMAs, commits the stage to BOTH
//                      CTAs' empty barriers, and each tile to both CTAs'
//                      accumulator-full barriers.
//   warps 0-3 (each)   drain their CTA's accumulator rows, release the
//                      leader's accumulator (4 warps x 2 CTAs), store D.
// Persistent over tiles: pair i takes tiles i, i + pairs, ...  Scales are
// relaid atoms (read through a 2-D uint32 view: 128 words = one atom).
#pragma once

namespace mxfp4 {

template <int STAGES>
struct PairCfg {
    static constexpr int A_BYTES = kTileM * 128;          // 128 rows x 128 bytes
    static constexpr int B_BYTES = kTileM * 128;          // this CTA's half of N
    static constexpr int SFA_BYTES = 2 * kSfAtomBytes;    // 128 rows, 2 k-groups
    static constexpr int SFB_BYTES = 4 * kSfAtomBytes;    // 256 rows, 2 k-groups
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM_BYTES = RING_BYTES + BAR_BYTES + 1024;
    static constexpr int SF_COLS_A = 8;                   // 2 groups x 4 columns
    static constexpr int SF_COLS_B = 16;                  // 2 groups x 2 blocks x 4 columns
    static constexpr int SF_COLS = SF_COLS_A + SF_COLS_B;
    static constexpr int TMEM_USED = 256 + STAGES * SF_COLS;
    static constexpr int TMEM_COLS = TMEM_USED <= 256 ? 256 : 512;
    static_assert(TMEM_USED <= 512, "tensor memory budget");
    static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

struct PairSched {
    int tiles_p, tiles_q;   // 256 x 256 output tiles
    int kt;                 // K stages per tile
    int group;              // raster: groups of `group` tile rows
};

__device__ __forceinline__ void pair_tile_coords(const PairSched &s, int t, int &pt, int &qt)
{
    const int per_group = s.group * s.tiles_q;
    const int g = t / per_group;
    const int within = t - g * per_group;
    const int gh = min(s.group, s.tiles_p - g * s.group);
    pt = g * s.group + within % gh;
    qt = within / gh;
}

template <int STAGES>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(192, 1)
    gemm_mxf4_pair(const __grid_constant__ GemmArgs a, const __grid_constant__ PairSched ps,
                   const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB)
{
    using PC = PairCfg<STAGES>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + PC::RING_BYTES);   // leader's are used
    uint64_t *empty = full + STAGES;
    uint64_t *acc_full = empty + STAGES;
    uint64_t *acc_empty = acc_full + 1;                                      // leader's is used
    uint64_t *drain = acc_empty + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;
    const int tiles = ps.tiles_p * ps.tiles_q;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);          // the leader's expect-tx arrival (both CTAs' bytes)
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 8);             // four epilogue warps in each CTA
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc_pair(tmem_slot, PC::TMEM_COLS);
        tmem_relinquish_pair();
    }
    if (warp == 4 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        prefetch_tensormap(&tmSA);
        prefetch_tensormap(&tmSB);
    }
    tc_fence_before();
    cluster_sync();                          // barriers of both CTAs initialised
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int64_t groups = sf_groups(a.K);

    if (warp == 4) {
        // ------------------------------------------------------ producer --
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            bool stop = false;
            for (int t = pair; t < tiles && !stop; t += npairs) {
                int pt, qt;
                pair_tile_coords(ps, t, pt, qt);
                const int arow = pt * 256 + static_cast<int>(rank) * kTileM;
                const int brow = qt * 256 + static_cast<int>(rank) * kTileM;
                const int64_t sfa_atom = static_cast<int64_t>(pt * 2 + rank) * groups;
                const int64_t sfb_atom0 = static_cast<int64_t>(qt * 2) * groups;
                for (int kt = 0; kt < ps.kt; ++kt) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.wait_limit,
                                   &g_device_status)) {
                        stop = true;
                        break;
                    }
                    uint8_t *st = smem + stage * PC::STAGE_BYTES;
                    const uint32_t lbar = map_to_rank(smem_addr(&full[stage]), 0);
                    // Only the leader arrives, expecting both CTAs' bytes: a
                    // cluster-scope arrive from the peer costs ~0.5 us a stage.
                    // The peer's copies just complete their bytes on the
                    // leader's barrier (it cannot start the next phase of this
                    // stage before the leader's MMAs have freed it).
                    if (leader)
                        mbar_arrive_expect_tx(&full[stage], 2 * PC::STAGE_BYTES);
                    tma_load_2d_pair(st, &tmA, lbar, kt * 128, arow, pol);
                    tma_load_2d_pair(st + PC::A_BYTES, &tmB, lbar, kt * 128, brow, pol);
                    uint8_t *sf = st + PC::A_BYTES + PC::B_BYTES;
                    tma_load_2d_pair(sf, &tmSA, lbar, 0, static_cast<int>(sfa_atom + 2 * kt), pol);
                    tma_load_2d_pair(sf + PC::SFA_BYTES, &tmSB, lbar, 0,
                                     static_cast<int>(sfb_atom0 + 2 * kt), pol);
                    tma_load_2d_pair(sf + PC::SFA_BYTES + 2 * kSfAtomBytes, &tmSB, lbar, 0,
                                     static_cast<int>(sfb_atom0 + groups + 2 * kt), pol);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------ MMA (leader) --
        if (leader && lane == 0) {
            const uint32_t idesc = idesc_mxf4(256, 256);
            const uint32_t t_sf = tmem + 256;
            int stage = 0;
            uint32_t phase = 0;
            uint32_t acc_phase = 0;
            bool stop = false;
            // Scale atoms of stage s into that stage's tensor-memory slot.
            auto sf_copy = [&](int s) {
                uint8_t *st = smem + s * PC::STAGE_BYTES;
                const uint32_t sfa_t = t_sf + s * PC::SF_COLS;
                const uint32_t sfb_t = sfa_t + PC::SF_COLS_A;
                const uint32_t sfa_s = smem_addr(st + PC::A_BYTES + PC::B_BYTES);
                const uint32_t sfb_s = sfa_s + PC::SFA_BYTES;
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    tmem_cp_32x128b_x4_pair(sfa_t + g * 4, sdesc_sf_block(sfa_s + g * kSfAtomBytes));
#pragma unroll
                    for (int r = 0; r < 2; ++r)
                        tmem_cp_32x128b_x4_pair(
                            sfb_t + g * 8 + r * 4,
                            sdesc_sf_block(sfb_s + r * 2 * kSfAtomBytes + g * kSfAtomBytes));
                }
            };
            for (int t = pair; t < tiles && !stop; t += npairs) {
                if (!mbar_wait(acc_empty, acc_phase ^ 1u, abort_flag, a.wait_limit,
                               &g_device_status))
                    break;
                tc_fence_after();
                // tcgen05.cp and tcgen05.mma execute in issue order on the
                // tensor pipe, so issuing the next stage's scale copies ahead
                // of this stage's MMAs gains nothing (measured slower); the
                // plain order keeps one full-barrier wait per stage.
                for (int kt = 0; kt < ps.kt; ++kt) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, a.wait_limit,
                                   &g_device_status)) {
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    sf_copy(stage);
                    uint8_t *st = smem + stage * PC::STAGE_BYTES;
                    const uint32_t sfa_t = t_sf + stage * PC::SF_COLS;
                    const uint32_t sfb_t = sfa_t + PC::SF_COLS_A;
                    const uint64_t adesc = sdesc_kmajor_sw128(smem_addr(st));
                    const uint64_t bdesc = sdesc_kmajor_sw128(smem_addr(st + PC::A_BYTES));
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t sf_id = (j & 1) * 2;
                        mma_mxf4_pair(tmem, adesc + 2 * j, bdesc + 2 * j,
                                      idesc_sf_ids(idesc, sf_id, sf_id), sfa_t + (j >> 1) * 4,
                                      sfb_t + (j >> 1) * 8, (kt > 0 || j > 0) ? 1u : 0u);
                    }
                    mma_commit_pair(&empty[stage], 0x3);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                mma_commit_pair(acc_full, 0x3);
                acc_phase ^= 1u;
            }
            if (*abort_flag) {
                mma_commit_pair(drain, 0x1);
                mbar_wait_drain(drain, 0, a.wait_limit);
            }
        }
    } else {
        // ------------------------------------------------------ epilogue --
        const int row = warp * 32 + lane;
        const uint32_t lead_acc_empty = map_to_rank(smem_addr(acc_empty), 0);
        uint32_t acc_phase = 0;
        for (int t = pair; t < tiles; t += npairs) {
            bool ok = mbar_wait(acc_full, acc_phase, abort_flag, a.wait_limit, &g_device_status);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok)
                break;
            acc_phase ^= 1u;
            tc_fence_after();
            int pt, qt;
            pair_tile_coords(ps, t, pt, qt);
            const int m = pt * 256 + static_cast<int>(rank) * kTileM + row;
            const int n0 = qt * 256;
            const uint32_t t_row = tmem + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll 1
            for (int c0 = 0; c0 < 256; c0 += 32) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_row + c0, r);
                tmem_ld_wait();
                if (c0 == 256 - 32) {
                    // Accumulator rows of this warp read: release them to the leader.
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive_cluster(lead_acc_empty);
                }
                if (m < a.M && n0 + c0 < a.N) {
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        v[i] = __uint_as_float(r[i]);
                    store_d_row(a, m, n0 + c0, v);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();            // no CTA leaves while its peer may still signal it
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, PC::TMEM_COLS);
    }
}

}  // namespace mxfp4
