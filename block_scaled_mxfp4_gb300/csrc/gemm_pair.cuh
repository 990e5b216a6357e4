// CTA-pair (2-SM) form of the block-scaled MXFP4 GEMM for large shapes
// (included by gemm_sm103.cu).
//
// A cluster of two CTAs computes one 256 x 256 output tile with
// tcgen05.mma.cta_group::2 (M = 256): CTA r of the pair holds rows
// [128r, 128r+128) of the tile's A panel and rows [128r, 128r+128) of its B
// panel (half of N) in its own shared memory, and its own 128 rows x 256
// columns of the fp32 accumulator in its own tensor memory.  Per 256-K stage
// each CTA therefore stages 16 KB of A and 16 KB of B (plus the stage's scale
// atoms) for 128 x 256 x 256 multiply-adds -- against 48 KB for a one-CTA
// 128 x 256 tile -- so that six stages fit, enough to keep the tensor pipe
// fed across the TMA round trip.  One accumulator (256 of the 512 tensor-
// memory columns) and one scale slot per stage (6 x 24 columns).
//
// NV = true is the NVFP4 form: kind::mxf4nvf4 with one UE4M3 scale per 16 K
// (scale_vec::4X).  A stage then carries four scale atoms per 128-row block
// instead of two (each atom spans 64 K), a scale slot takes 48 columns, and
// five stages fit the tensor memory (256 + 5 x 48 = 496 columns).
//
// Roles (512 threads = 16 warps per CTA):
//   warps 4, 6, 7 (each CTA)  TMA producers: A half, B half, and the scale
//                      atoms (this CTA's 128 rows of scale-A; all BN rows of
//                      scale-B in one 3-D box of 2 K-groups x 2 row blocks),
//                      each completing its bytes on this CTA's full barrier.
//                      A thread waits out each copy instruction it issues
//                      (hundreds of cycles), hence three issuing warps.
//   warps 12-15 (each CTA)  scale writers, warp w for TMEM lanes 32(w%4)..+31:
//                      once a stage has landed in this CTA, each lane reads
//                      its 16-byte lines of the stage's atoms from shared
//                      memory and writes them with tcgen05.st into its TMEM
//                      lane of the stage's scale slot (the four warps lay
//                      down the four replicas), waits for the stores, and
//                      arrives on the LEADER's sf_ready barrier (the peer's
//                      warps with a relaxed remote arrive).  tcgen05.st does
//                      not queue behind the MMAs already issued (a
//                      shared-to-tensor-memory copy would), so the scales of
//                      later stages are ready well ahead.
//   warp 5 (leader)    waits for the accumulator to be free, then per stage
//                      for sf_ready (8 arrivals: both CTAs' data landed and
//                      both CTAs' scales written); issues four K=64 M=256
//                      N=256 MMAs and commits the stage to BOTH CTAs' empty
//                      barriers, and each tile to both CTAs' accumulator-full
//                      barriers.
//   warps 0-3 / 8-11 (each CTA)  epilogue, columns [0, 128) / [128, 256):
//                      read the accumulator (warp w owns TMEM lanes
//                      32(w%4)..+31 = tile rows), release the buffer to the
//                      leader as soon as the reads are done (8 warps x 2
//                      CTAs), form alpha*acc + beta*C and round once to bf16
//                      in registers, then store D -- so the next tile's MMAs
//                      wait for neither the arithmetic nor the stores.
// Persistent over tiles: pair i takes tiles i, i + pairs, ...  Scales are
// relaid atoms (a 2-D uint32 view for scale-A, 3-D for scale-B: 128 words =
// one atom).  A stage's scale slot in tensor memory is rewritten only after
// the MMAs that read it completed: that is implied by the stage's full
// barrier (the producers waited for the stage's previous MMAs).
// Launched as a programmatic dependent: right after this library's scale
// relayout (whose grid waits for the work before it), only the scale loads
// wait for the preceding grid; otherwise every load, and the epilogue, waits.
#pragma once

namespace mxfp4 {

template <int STAGES, bool NV>
struct PairCfg {
    static constexpr int BN = 256;                        // tile N
    static constexpr int B_ROWS = BN / 2;                 // this CTA's rows of the B tile
    static constexpr int GROUPS = NV ? 4 : 2;             // scale atoms per stage and row block
    static constexpr int A_BYTES = kTileM * 128;          // 128 rows x 128 bytes (256 K)
    static constexpr int B_BYTES = B_ROWS * 128;
    static constexpr int SFB_RB = 2;                      // 128-row scale blocks a tile can touch
    static constexpr int SFA_BYTES = GROUPS * kSfAtomBytes;           // 128 rows
    static constexpr int SFB_BYTES = SFB_RB * GROUPS * kSfAtomBytes;
    static constexpr int SF_BYTES = SFA_BYTES + SFB_BYTES;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SF_BYTES;
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    static constexpr int BAR_BYTES = 512;
    static constexpr int SMEM_BYTES = RING_BYTES + BAR_BYTES + 1024;
    static constexpr int SF_COLS_A = 4 * GROUPS;          // 4 columns per k-group
    static constexpr int SF_COLS_B = 4 * GROUPS * SFB_RB; // and per 128-row block
    static constexpr int SF_COLS = SF_COLS_A + SF_COLS_B; // one scale slot per stage
    static constexpr int HALF = BN / 2;                   // columns per epilogue warp
    static constexpr int TMEM_USED = BN + STAGES * SF_COLS;
    static constexpr int TMEM_COLS = TMEM_USED <= 256 ? 256 : 512;
    static constexpr int THREADS = 512;
    static constexpr int EPI_WARPS = 8;                   // per CTA
    static_assert(TMEM_USED <= 512, "tensor memory budget");
    static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static_assert(HALF == 128, "epilogue columns");
};

struct PairSched {
    int tiles_p, tiles_q;   // 256 x 256 output tiles
    int kt;                 // K stages (256 K each) per tile
    int group;              // raster: groups of `group` tile rows
};

// Tile t -> its row of tiles pt and column qt, over tiles_p x tiles_q tiles
// rastered in bands of `group` tile rows.
__device__ __forceinline__ void pair_tile_coords(const PairSched &s, int t, int &pt, int &qt)
{
    const int per_group = s.group * s.tiles_q;
    const int g = t / per_group;
    const int within = t - g * per_group;
    const int gh = min(s.group, s.tiles_p - g * s.group);
    pt = g * s.group + within % gh;
    qt = within / gh;
}

// One epilogue thread's HALF columns of one accumulator row, rounded: out[j]
// holds columns n0 + 2j and n0 + 2j + 1 as packed bf16.  Stores them to D
// row m: 32-byte stores when the row segment is whole and aligned, with a
// short pause after every 64 bytes.  The stores overlap the next tile's main
// loop, and global stores share the memory-instruction queue with the
// mbarrier polls of the producer, scale-writer and MMA warps: a burst of 64 KB of
// stores per CTA delays those polls by thousands of cycles, so the epilogue
// uses the widest stores and spreads them out.  D goes to L2 as evict-first:
// written once and not read back, it should not push out the A and B panels
// that later tiles load again (the operands are loaded as evict-last).
template <int HALF>
__device__ __forceinline__ void pair_store_row(const GemmArgs &a, int m, int n0,
                                               const uint32_t (&out)[HALF / 2])
{
    if (m >= a.M || n0 >= a.N)
        return;
    uint16_t *d = a.D + static_cast<int64_t>(m) * a.ldd + n0;
    if (a.vec32_ok && n0 + HALF <= a.N) {
        const uint64_t pol = l2_policy_evict_first();
#pragma unroll
        for (int j = 0; j < HALF / 2; j += 8) {
            st_global_v8_hint(d + 2 * j, out[j], out[j + 1], out[j + 2], out[j + 3], out[j + 4],
                              out[j + 5], out[j + 6], out[j + 7], pol);
            if ((j & 15) == 8)
                __nanosleep(400);
        }
    } else if (a.vec_ok && n0 + HALF <= a.N) {
#pragma unroll
        for (int j = 0; j < HALF / 2; j += 4)
            *reinterpret_cast<uint4 *>(d + 2 * j) = make_uint4(out[j], out[j + 1], out[j + 2], out[j + 3]);
    } else {
#pragma unroll
        for (int j = 0; j < HALF / 2; ++j) {
            if (n0 + 2 * j < a.N)
                d[2 * j] = static_cast<uint16_t>(out[j] & 0xFFFFu);
            if (n0 + 2 * j + 1 < a.N)
                d[2 * j + 1] = static_cast<uint16_t>(out[j] >> 16);
        }
    }
}

// alpha * acc (+ beta * C) for W (16 or 32) columns of row m starting at n,
// rounded once; out receives W / 2 packed bf16 pairs.
template <int W>
__device__ __forceinline__ void pair_round_chunk(const GemmArgs &a, int m, int n, const uint32_t (&r)[W],
                                                 uint32_t *out)
{
    float v[W];
#pragma unroll
    for (int i = 0; i < W; ++i)
        v[i] = a.alpha * __uint_as_float(r[i]);
    if (a.beta != 0.0f && m < a.M) {
        const uint16_t *c = a.C + static_cast<int64_t>(m) * a.ldc + n;
        if (a.vec_ok && n + W <= a.N) {
#pragma unroll
            for (int i = 0; i < W; i += 8) {
                const uint4 w = *reinterpret_cast<const uint4 *>(c + i);
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    v[i + 2 * j] = fmaf(a.beta, bf16_bits_to_float(ww[j] & 0xFFFF), v[i + 2 * j]);
                    v[i + 2 * j + 1] = fmaf(a.beta, bf16_bits_to_float(ww[j] >> 16), v[i + 2 * j + 1]);
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < W; ++i)
                if (n + i < a.N)
                    v[i] = fmaf(a.beta, bf16_bits_to_float(c[i]), v[i]);
        }
    }
#pragma unroll
    for (int j = 0; j < W / 2; ++j)
        out[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
}

template <int STAGES, bool NV>
__global__ void __launch_bounds__(PairCfg<STAGES, NV>::THREADS, 1)
    gemm_mxf4_pair(const __grid_constant__ GemmArgs a, const __grid_constant__ PairSched ps,
                   const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB)
{
    using PC = PairCfg<STAGES, NV>;
    constexpr int BN = PC::BN;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + PC::RING_BYTES);   // leader's are used
    uint64_t *empty = full + STAGES;
    uint64_t *sf_ready = empty + STAGES;                                    // leader's are used
    uint64_t *acc_full = sf_ready + STAGES;
    uint64_t *acc_empty = acc_full + 1;                                     // leader's used
    uint64_t *drain = acc_empty + 1;                                        // [3]: MMA
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 3);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank() & 1u;   // rank within the pair
    const uint32_t lead = 0;                        // cluster rank of the leader
    const bool leader = rank == 0;
    const int cl = blockIdx.x / 2;
    const int ncl = gridDim.x / 2;
    const int tiles = ps.tiles_p * ps.tiles_q;
    const int my_tiles = cl < tiles ? (tiles - 1 - cl) / ncl + 1 : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 3);          // this CTA's three producers
            mbar_init(&empty[s], 1);         // the pair's MMA commit
            mbar_init(&sf_ready[s], 8);      // the scale writers of both CTAs (leader's used)
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 2 * PC::EPI_WARPS);
        for (int i = 0; i < 3; ++i)
            mbar_init(&drain[i], 1);
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
    const int64_t groups = NV ? sf_groups_nv(a.K) : sf_groups(a.K);
    const int total_stages = my_tiles * ps.kt;
    // The next kernel on the stream may launch; it waits in-kernel for this
    // grid before touching anything this grid writes.
    if (threadIdx.x == 0)
        pdl_launch_dependents();

    if (warp == 4 || warp == 6 || warp == 7) {
        // ------------------------------------------------------ producers --
        if (lane == 0) {
            const int role = warp == 4 ? 0 : warp - 5;   // 0: A, 1: B, 2: scales
            const uint64_t pol = l2_policy_evict_last();
            // After this library's relayout (whose grid waited for the work
            // before it) only the relaid scales depend on the preceding grid.
            if (role == 2 || !a.ab_early)
                pdl_wait_prerequisites();
            const uint32_t unit = role == 0 ? PC::A_BYTES : role == 1 ? PC::B_BYTES : PC::SF_BYTES;
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool stop = false;
            for (int t = cl; t < tiles && !stop; t += ncl) {
                int pt, qt;
                pair_tile_coords(ps, t, pt, qt);
                const int arow = pt * 256 + static_cast<int>(rank) * kTileM;
                const int brow = qt * BN + static_cast<int>(rank) * PC::B_ROWS;
                const int sfa_atom = static_cast<int>(static_cast<int64_t>(pt * 2 + rank) * groups);
                const int sfb_rb = (qt * BN) / kSfRowBlock;
                for (int kt = 0; kt < ps.kt; ++kt) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.wait_limit,
                                   &g_device_status)) {
                        stop = true;
                        break;
                    }
                    uint8_t *st = smem + stage * PC::STAGE_BYTES;
                    mbar_arrive_expect_tx(&full[stage], unit);
                    if (role == 0) {
                        tma_load_2d(st, &tmA, &full[stage], kt * 128, arow, pol);
                    } else if (role == 1) {
                        tma_load_2d(st + PC::A_BYTES, &tmB, &full[stage], kt * 128, brow, pol);
                    } else {
                        uint8_t *sf = st + PC::A_BYTES + PC::B_BYTES;
                        tma_load_2d(sf, &tmSA, &full[stage], 0, sfa_atom + PC::GROUPS * kt, pol);
                        tma_load_3d(sf + PC::SFA_BYTES, &tmSB, &full[stage], 0, PC::GROUPS * kt,
                                    sfb_rb, pol);
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (*abort_flag) {
                // Let the copies already issued land before the CTA exits.
                for (int i = max(0, issued - STAGES); i < issued; ++i)
                    mbar_wait_drain(&full[i % STAGES], (i / STAGES) & 1u, a.wait_limit);
            }
        }
    } else if (warp >= 12) {
        // ------------------------------------------- scale writers (each CTA) --
        const int quarter = warp & 3;
        const uint32_t t_q = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + BN;
        const uint32_t lead_ready = map_to_rank(smem_addr(&sf_ready[0]), lead);
        int stage = 0;
        uint32_t phase = 0;
        for (int i = 0; i < total_stages; ++i) {
            bool ok = mbar_wait(&full[stage], phase, abort_flag, a.wait_limit, &g_device_status);
            if (!__all_sync(0xffffffffu, ok))
                break;
            // Line `lane` of every atom of the stage: scale-A atoms g (columns
            // 4g .. 4g+3); scale-B (atom g, row block rb; in shared memory at
            // rb*GROUPS + g) -> columns SF_COLS_A + g*4*SFB_RB + rb*4.
            const uint8_t *sf_s = smem + stage * PC::STAGE_BYTES + PC::A_BYTES + PC::B_BYTES;
            uint32_t wa[4 * PC::GROUPS];
            uint32_t wb[4 * PC::GROUPS * PC::SFB_RB];
#pragma unroll
            for (int g = 0; g < PC::GROUPS; ++g) {
                const uint4 v = *reinterpret_cast<const uint4 *>(sf_s + g * kSfAtomBytes + 16 * lane);
                wa[4 * g] = v.x;
                wa[4 * g + 1] = v.y;
                wa[4 * g + 2] = v.z;
                wa[4 * g + 3] = v.w;
#pragma unroll
                for (int rb = 0; rb < PC::SFB_RB; ++rb) {
                    const uint4 u = *reinterpret_cast<const uint4 *>(
                        sf_s + PC::SFA_BYTES + (rb * PC::GROUPS + g) * kSfAtomBytes + 16 * lane);
                    const int o = (g * PC::SFB_RB + rb) * 4;
                    wb[o] = u.x;
                    wb[o + 1] = u.y;
                    wb[o + 2] = u.z;
                    wb[o + 3] = u.w;
                }
            }
            const uint32_t slot = t_q + stage * PC::SF_COLS;
            if constexpr (NV) {
                tmem_st_32x32b_x16(slot, wa);
                tmem_st_32x32b_x32(slot + PC::SF_COLS_A, wb);
            } else {
                tmem_st_32x32b_x8(slot, wa);
                tmem_st_32x32b_x16(slot + PC::SF_COLS_A, wb);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader)
                    mbar_arrive(&sf_ready[stage]);
                else
                    mbar_arrive_cluster_relaxed(lead_ready + static_cast<uint32_t>(stage * sizeof(uint64_t)));
            }
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------ MMA (leader) --
        // The whole warp runs the loop (warp-uniform descriptors and
        // barrier polls); one elected lane issues each MMA and commit.
        if (leader) {
            const uint32_t idesc = NV ? idesc_nvf4(256, BN) : idesc_mxf4(256, BN);
            const uint32_t t_sf = tmem + BN;
            int stage = 0;
            uint32_t phase = 0;
            uint32_t acc_phase = 0;         // parity of the accumulator's next use
            bool stop = false;
            for (int t = cl; t < tiles && !stop; t += ncl) {
                if (!mbar_wait(acc_empty, acc_phase ^ 1u, abort_flag, a.wait_limit,
                               &g_device_status))
                    break;
                tc_fence_after();
                int pt, qt;
                pair_tile_coords(ps, t, pt, qt);
                const uint32_t q_off = static_cast<uint32_t>(((qt * BN) % kSfRowBlock) / 32);
                const uint32_t d_tmem = tmem;
                for (int kt = 0; kt < ps.kt; ++kt) {
                    // sf_ready completes after the scale writers observed the
                    // stage's full barrier (all of its bytes landed), so it
                    // stands for both: one poll per stage.
                    if (!mbar_wait(&sf_ready[stage], phase, abort_flag, a.wait_limit,
                                   &g_device_status)) {
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sfa_t = t_sf + stage * PC::SF_COLS;
                    const uint32_t sfb_t = sfa_t + PC::SF_COLS_A + q_off;
                    const uint32_t st = smem_addr(smem + stage * PC::STAGE_BYTES);
                    const uint64_t adesc = sdesc_kmajor_sw128(st);
                    const uint64_t bdesc = sdesc_kmajor_sw128(st + PC::A_BYTES);
                    // Four K=64 MMAs per 256-K stage.
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if constexpr (NV) {
                            // Atom j holds the MMA's four blocks of 16.
                            mma_nvf4_pair_elect(d_tmem, adesc + 2 * j, bdesc + 2 * j, idesc,
                                                sfa_t + j * 4, sfb_t + j * 4 * PC::SFB_RB,
                                                (kt > 0 || j > 0) ? 1u : 0u);
                        } else {
                            const uint32_t sf_id = (j & 1) * 2;
                            const int g = j >> 1;                    // scale k-group
                            mma_mxf4_pair_elect(d_tmem, adesc + 2 * j, bdesc + 2 * j,
                                                idesc_sf_ids(idesc, sf_id, sf_id), sfa_t + g * 4,
                                                sfb_t + g * 4 * PC::SFB_RB,
                                                (kt > 0 || j > 0) ? 1u : 0u);
                        }
                    }
                    // Frees the stage in both CTAs of the pair.
                    mma_commit_pair_elect(&empty[stage], static_cast<uint16_t>(3u));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                mma_commit_pair_elect(acc_full, static_cast<uint16_t>(3u));
                acc_phase ^= 1u;
            }
            if (*abort_flag) {
                mma_commit_pair_elect(&drain[0], static_cast<uint16_t>(1u << lead));
                mbar_wait_drain(&drain[0], 0, a.wait_limit);
            }
        }
    } else {
        // ------------------------------------------------------ epilogue --
        // warps 0-3: columns [0, HALF), warps 8-11: columns [HALF, BN).
        // C and D may belong to the work before this grid.
        pdl_wait_prerequisites();
        const int quarter = warp & 3;
        const int half = warp >> 3;
        const int row = quarter * 32 + lane;
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + half * PC::HALF;
        uint32_t acc_phase = 0;
        for (int t = cl; t < tiles; t += ncl) {
            bool ok = mbar_wait(acc_full, acc_phase, abort_flag, a.wait_limit, &g_device_status);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok)
                break;
            acc_phase ^= 1u;
            tc_fence_after();
            int pt, qt;
            pair_tile_coords(ps, t, pt, qt);
            const int m = pt * 256 + static_cast<int>(rank) * kTileM + row;
            const int n0 = qt * BN + half * PC::HALF;
            const uint32_t t_row = t_lane;
            uint32_t out[PC::HALF / 2];
            // Columns 0-63 are read and rounded; 64-127 are read, the
            // accumulator released, and only then rounded: the next tile's
            // MMAs wait for the reads alone, not the arithmetic.  Once this
            // warp's accumulator cells are read (tcgen05.wait::ld has
            // returned, so no TMEM read is outstanding) they are released to
            // the leader.  No memory fence is needed for that, and a
            // cluster-scope release arrive costs ~1000 cycles, so the leader's
            // warps arrive locally and the peer's with a relaxed remote arrive.
            uint32_t r0[32], r1[32];
            tmem_ld_32x32b_x32(t_row, r0);
            tmem_ld_32x32b_x32(t_row + 32, r1);
            tmem_ld_wait(r0, r1);
            pair_round_chunk<32>(a, m, n0, r0, out);
            pair_round_chunk<32>(a, m, n0 + 32, r1, out + 16);
            tmem_ld_32x32b_x32(t_row + 64, r0);
            tmem_ld_32x32b_x32(t_row + 96, r1);
            tmem_ld_wait(r0, r1);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader)
                    mbar_arrive(acc_empty);
                else
                    mbar_arrive_cluster_relaxed(map_to_rank(smem_addr(acc_empty), lead));
            }
            pair_round_chunk<32>(a, m, n0 + 64, r0, out + 32);
            pair_round_chunk<32>(a, m, n0 + 96, r1, out + 48);
            pair_store_row<PC::HALF>(a, m, n0, out);
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
