// C ABI of the block-scaled MXFP4 GEMM: argument checks, the tile / split-K
// plan, TMA tensor maps and the launch sequence (optional scale relayout ->
// GEMM, whose split-K partials are summed inside the GEMM; prepacked scales
// come from mxfp4_scale_relayout).  Declared in include/mxfp4_gemm.h.
#include <atomic>
#include <chrono>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "../../include/mxfp4_gemm.h"
#include "internal.h"

using namespace mxfp4;

namespace {

constexpr int kMaxSplit = 16;
constexpr int kMaxClusterSplit = 8;   // splits a (portable) cluster holds
constexpr int kDefaultSms = 152;
constexpr size_t kAlign = 256;

std::atomic<long long> g_wait_limit{1LL << 32};

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct DeviceInfo {
    bool valid = false;
    bool sm103 = false;
    int sms = 0;
};

std::mutex g_dev_mutex;
DeviceInfo g_dev[64];

// Current device's properties, cached; nullptr if no device is usable.
const DeviceInfo *current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo &d = g_dev[dev];
    if (!d.valid) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        d.sm103 = (major == 10 && minor == 3);
        d.sms = sms;
        d.valid = true;
    }
    return &d;
}

int device_sms_or_default()
{
    const DeviceInfo *d = current_device();
    return (d && d->sms > 0) ? d->sms : kDefaultSms;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// 2-D uint8 view [rows, K/2] of a packed operand with row stride ld/2 bytes;
// box 128 bytes x box_rows, 128-byte swizzle, zero fill out of bounds.
bool encode_operand(CUtensorMap *map, const void *base, int rows, int K, int64_t ld, int box_rows)
{
    auto enc = tensor_map_encoder();
    if (!enc)
        return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld / 2)};
    cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D uint8 view [rows, K/32] of row-major E8M0 scales (row stride ld bytes,
// a multiple of 16); box 16 bytes x box_rows, no swizzle, zero fill.
// kbytes: scale bytes per row (K / 32, or K / 16 for NVFP4).
bool encode_scales(CUtensorMap *map, const void *base, int rows, int kbytes, int64_t ld, int box_rows)
{
    auto enc = tensor_map_encoder();
    if (!enc)
        return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kbytes), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld)};
    cuuint32_t box[2] = {16u, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Relaid scale atoms viewed as 2-D uint32 [atoms, 128] (one 512-byte atom per
// row); a box of 2 rows = the two atoms of one 256-K stage of a 128-row block.
// groups: atoms per 128-row block (sf_groups(K), or sf_groups_nv(K) for NVFP4).
bool encode_atoms(CUtensorMap *map, const void *base, int rows, int64_t groups, int box_atoms)
{
    auto enc = tensor_map_encoder();
    if (!enc)
        return false;
    const int64_t atoms = sf_row_blocks(rows) * groups;
    cuuint64_t dims[2] = {128u, static_cast<cuuint64_t>(atoms)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(kSfAtomBytes)};
    cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_atoms)};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Relaid scale atoms viewed as 3-D uint32 [row blocks][k-groups][128]; a box
// of box_groups k-groups (2 per 256 K of a stage) x box_rb row blocks = the
// 128-row blocks a pair tile's B rows touch for one stage, in smem order (row
// block, k-group); a tile that starts inside a block reads past its last rows
// (zero fill beyond the end).
bool encode_atoms_3d(CUtensorMap *map, const void *base, int rows, int64_t groups, int box_rb,
                     int box_groups)
{
    auto enc = tensor_map_encoder();
    if (!enc)
        return false;
    cuuint64_t dims[3] = {128u, static_cast<cuuint64_t>(groups),
                          static_cast<cuuint64_t>(sf_row_blocks(rows))};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(kSfAtomBytes),
                             static_cast<cuuint64_t>(groups * kSfAtomBytes)};
    cuuint32_t box[3] = {128u, static_cast<cuuint32_t>(box_groups), static_cast<cuuint32_t>(box_rb)};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

struct Candidate {
    int tile_n;
    int stages;
    int ctas_per_sm;
};

// Tile / swap / split-K choice.  Candidates are scored as the page's section
// "Tile selection heuristic" scores its tiles: fewest waves (ceil(tiles /
// resident CTA slots)), then the fullest last wave, then the larger
// tile_m*tile_n/(tile_m+tile_n); the fixed candidate order breaks ties.
// split_k >= 1 runs one CTA per (tile, K split); for split_k > 1 the CTA that
// completes a tile sums the fp32 partials in split order.  split_k == 0 picks
// the split itself: 1 when the tiles fill at least half a wave, else enough
// splits to fill the resident CTA slots, each split keeping at least
// kMinSplitStages K stages.  Shapes whose 256 x 256 tiles fill every SM pair
// at least once run the CTA-pair kernel instead (split_k == 0 only).
constexpr int kMinSplitStages = 8;

// Bytes of the split-K area of a workspace: one 8-byte counter per tile, then
// one partial slot (128 rows x part_cols fp32, columns rounded up to 4) per
// tile and split, each part 256-byte aligned.
size_t splitk_bytes(int64_t tiles, int split, int part_cols)
{
    const size_t cols4 = static_cast<size_t>((part_cols + 3) / 4 * 4);
    return align_up(static_cast<size_t>(tiles) * 8) +
           align_up(static_cast<size_t>(tiles) * split * kTileM * cols4 * sizeof(float));
}

int make_plan(int M, int N, int K, int split_req, int sms, mxfp4_plan *out, GemmShape *shape,
              bool fp8 = false)
{
    if (M < 1 || N < 1 || K < 32 || (K % 32) != 0 || split_req < 0 || split_req > kMaxSplit)
        return MXFP4_ERR_INVALID_ARG;
    if (sms <= 0)
        sms = kDefaultSms;
    const int swap = (M <= 64 && N > M) ? 1 : 0;
    const int64_t P = swap ? N : M;
    const int64_t Q = swap ? M : N;
    const int kt = (K + kTileK - 1) / kTileK;
    const int64_t tiles256 = ((static_cast<int64_t>(M) + 255) / 256) * ((static_cast<int64_t>(N) + 255) / 256);
    // The CTA-pair kernel takes shapes whose 256 x 256 tiles fill at least one
    // wave of SM pairs.
    const bool use_pair = !fp8 && !swap && split_req == 0 && M >= 256 && N >= 256 &&
                          tiles256 >= sms / 2;

    Candidate cands[3];
    int nc = 0;
    if (swap) {
        cands[nc++] = {64, 4, 2};             // two 4-stage CTAs per SM
    } else {
        cands[nc++] = {256, 4, 1};
        cands[nc++] = {128, 6, 1};
        if (Q <= 64)
            cands[nc++] = {64, 8, 1};
    }
    int best = -1;
    int64_t best_waves = 0;
    double best_occ = 0, best_ratio = 0;
    for (int i = 0; i < nc; ++i) {
        // The one-tile launch puts the tile columns on grid.y (at most 65535):
        // a tile that needs more columns than that is not a candidate.
        if ((Q + cands[i].tile_n - 1) / cands[i].tile_n > 65535)
            continue;
        const int64_t tiles = ((P + kTileM - 1) / kTileM) * ((Q + cands[i].tile_n - 1) / cands[i].tile_n);
        const int64_t slots = static_cast<int64_t>(sms) * cands[i].ctas_per_sm;
        const int64_t waves = (tiles + slots - 1) / slots;
        const double occ = static_cast<double>(tiles) / static_cast<double>(waves * slots);
        const double ratio = static_cast<double>(kTileM * cands[i].tile_n) / (kTileM + cands[i].tile_n);
        bool better = best < 0 || waves < best_waves ||
                      (waves == best_waves && (occ > best_occ + 1e-12 ||
                                               (occ > best_occ - 1e-12 && ratio > best_ratio)));
        if (better) {
            best = i;
            best_waves = waves;
            best_occ = occ;
            best_ratio = ratio;
        }
    }
    if (best < 0 && !use_pair)
        return MXFP4_ERR_UNSUPPORTED_SHAPE;
    const Candidate c = best >= 0 ? cands[best] : Candidate{256, 4, 1};
    const int64_t gx = (P + kTileM - 1) / kTileM;
    const int64_t gy = (Q + c.tile_n - 1) / c.tile_n;
    if (!use_pair && (gy > 65535 || gx > 0x7FFFFFFF || gx * gy > 0x7FFFFFFF))
        return MXFP4_ERR_UNSUPPORTED_SHAPE;
    const int64_t tiles = gx * gy;
    const int64_t slots = static_cast<int64_t>(sms) * c.ctas_per_sm;

    int split = 1;
    if (split_req > 0) {
        split = split_req;
    } else if (!use_pair && 2 * tiles < slots) {
        const int64_t by_slots = slots / tiles;
        const int64_t by_k = kt / kMinSplitStages;
        int64_t s = by_slots < by_k ? by_slots : by_k;
        if (s > kMaxSplit)
            s = kMaxSplit;
        split = s > 1 ? static_cast<int>(s) : 1;
    }
    if (split > kt)
        split = kt;
    const int per = (kt + split - 1) / split;
    split = (kt + per - 1) / per;   // every split gets >= 1 stage

    std::memset(out, 0, sizeof(*out));
    out->swap_ab = swap;
    out->tile_m = kTileM;
    out->tile_n = c.tile_n;
    out->tile_k = kTileK;
    out->stages = c.stages;
    out->split_k = split;
    out->k_tiles_per_split = per;
    out->grid_x = static_cast<int>(gx);
    out->grid_y = static_cast<int>(gy);
    out->grid_z = split;
    const int part_cols = static_cast<int>(Q < c.tile_n ? Q : c.tile_n);
    // Up to kMaxClusterSplit splits reduce inside each tile's cluster and need
    // no workspace; more keep fp32 partials and tile counters in it.
    out->workspace_bytes = split > kMaxClusterSplit ? splitk_bytes(tiles, split, part_cols) : 0;
    out->pair = use_pair ? 1 : 0;
    if (use_pair) {
        // Persistent: one CTA pair per two SMs, each taking every pairs-th
        // 256 x 256 tile.
        const int64_t tiles_q = (static_cast<int64_t>(N) + 255) / 256;
        const int64_t ptiles = ((static_cast<int64_t>(M) + 255) / 256) * tiles_q;
        const int64_t pairs = sms / 2;
        out->tile_m = 256;
        out->tile_n = 256;
        out->tile_k = 256;
        out->stages = 6;
        out->split_k = 1;
        out->k_tiles_per_split = kt;
        out->waves = static_cast<int>((ptiles + pairs - 1) / pairs);
        out->ctas = 2 * static_cast<int>(ptiles < pairs ? ptiles : pairs);
        out->grid_x = out->ctas;
        out->grid_y = 1;
        out->grid_z = 1;
        out->workspace_bytes = 0;
    }
    // With enough tiles to fill the GPU the GEMM is compute-bound: mxfp4_gemm
    // then relays the row-major scales out in a separate pass (a few us) so
    // the mainloop can move whole scale atoms with bulk copies.  Skinny and
    // small shapes build the atoms inside the GEMM instead (no extra launches).
    // (The CTA-pair kernel always reads relaid atoms.)
    out->relayout_pass = (use_pair || (!swap && tiles >= sms)) ? 1 : 0;
    if (shape) {
        shape->tile_n = use_pair ? 256 : c.tile_n;
        shape->stages = out->stages;
        shape->swap = swap;
        shape->ctas_per_sm = c.ctas_per_sm;
        shape->pair = use_pair;
        shape->pair_ctas = out->ctas;
        shape->fp8 = fp8 ? 1 : 0;
        shape->nv = 0;
    }
    return MXFP4_OK;
}

int check_device()
{
    const DeviceInfo *d = current_device();
    if (!d)
        return MXFP4_ERR_CUDA;
    return d->sm103 ? MXFP4_OK : MXFP4_ERR_ARCH;
}

int check_common(const void *D, int64_t ldd, const void *C, int64_t ldc, const void *A, int64_t lda,
                 const void *B, int64_t ldb, float beta, int M, int N, int K, int split_k)
{
    if (!D || !A || !B)
        return MXFP4_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 32 || (K % 32) != 0 || split_k < 0 || split_k > kMaxSplit)
        return MXFP4_ERR_INVALID_ARG;
    if (lda < K || ldb < K || ldd < N)
        return MXFP4_ERR_INVALID_ARG;
    if (beta != 0.0f && (!C || ldc < N))
        return MXFP4_ERR_INVALID_ARG;
    if ((lda % 32) != 0 || (ldb % 32) != 0 || !aligned(A, 16) || !aligned(B, 16))
        return MXFP4_ERR_MISALIGNED;
    return MXFP4_OK;
}

// Scale relayout (if needed) has been done; run the GEMM.
// Scales as the kernel will read them: row-major [rows, ld] (atoms built in
// the kernel) or already relaid into atoms.
struct Scales {
    const uint8_t *a, *b;
    int64_t ld_a, ld_b;
    bool rowmajor;
};

std::atomic<unsigned> g_epoch{0};
std::once_flag g_epoch_once;

// Next per-call tag of the split-K tile counters (never 0).  The count starts
// from a clock-derived value so that a fresh workspace holding small integers
// does not look tagged by chance; counters of earlier calls hold earlier
// tags and never match.
uint32_t next_epoch()
{
    std::call_once(g_epoch_once, [] {
        const auto t = std::chrono::steady_clock::now().time_since_epoch().count();
        g_epoch.store(static_cast<unsigned>((t ^ (t >> 29)) * 2654435761u) | 0x40000000u);
    });
    unsigned e = ++g_epoch;
    while (e == 0)
        e = ++g_epoch;
    return e;
}

// ws: workspace base (split-K counters and partials), or nullptr when the
// plan needs none.  flags: MXFP4_FLAG_* of the call.
int run_gemm(void *D, int64_t ldd, const void *C, int64_t ldc, const void *A, int64_t lda,
             const void *B, int64_t ldb, const Scales &sc, float alpha, float beta, int M, int N,
             int K, const mxfp4_plan &plan, const GemmShape &shape, uint8_t *ws,
             cudaStream_t stream, bool after_relayout = false, int fmt_a = 0, int fmt_b = 0,
             unsigned flags = 0, bool nv = false)
{
    if (shape.pair) {
        if (sc.rowmajor)
            return MXFP4_ERR_INVALID_ARG;            // the pair kernel reads relaid atoms
        // Atoms per stage and 128-row block: 2 (128 K each), or 4 for NVFP4.
        const int per_stage = nv ? 4 : 2;
        const int64_t groups = nv ? sf_groups_nv(K) : sf_groups(K);
        CUtensorMap tmA, tmB, tmSA, tmSB;
        if (!encode_operand(&tmA, A, M, K, lda, kTileM) ||
            !encode_operand(&tmB, B, N, K, ldb, 128) ||
            !encode_atoms(&tmSA, sc.a, M, groups, per_stage) ||
            !encode_atoms_3d(&tmSB, sc.b, N, groups, 2, per_stage))
            return MXFP4_ERR_CUDA;
        GemmArgs a;
        std::memset(&a, 0, sizeof(a));
        a.M = M;
        a.N = N;
        a.K = K;
        a.kt_total = (K + kTileK - 1) / kTileK;
        a.alpha = alpha;
        a.beta = beta;
        a.C = static_cast<const uint16_t *>(beta != 0.0f ? C : nullptr);
        a.ldc = ldc;
        a.D = static_cast<uint16_t *>(D);
        a.ldd = ldd;
        a.vec_ok = aligned(D, 16) && (ldd % 8) == 0 &&
                   (beta == 0.0f || (aligned(C, 16) && (ldc % 8) == 0));
        a.vec32_ok = a.vec_ok && aligned(D, 32) && (ldd % 16) == 0;
        a.ab_early = after_relayout ? 1 : 0;
        a.wait_limit = g_wait_limit.load();
        const int tiles_p = (M + 255) / 256, tiles_q = (N + 255) / 256;
        if (launch_gemm_pair(a, tiles_p, tiles_q, shape.pair_ctas, tmA, tmB, tmSA, tmSB, nv,
                             stream) != cudaSuccess)
            return MXFP4_ERR_CUDA;
        return MXFP4_OK;
    }
    const bool swap = shape.swap != 0;
    CUtensorMap tmP, tmQ;
    const void *Pp = swap ? B : A;
    const void *Qp = swap ? A : B;
    const int Prows = swap ? N : M, Qrows = swap ? M : N;
    const int64_t ldP = swap ? ldb : lda, ldQ = swap ? lda : ldb;
    // An 8-bit row of K elements holds the bytes of an fp4 row of 2K.
    const int kx = shape.fp8 ? 2 : 1;
    // Q tiles copy only the rows Q has (rounded up to 8, the swizzle atom):
    // a skinny M then moves M rows per stage, not tile_n.
    const int q_box = Qrows < shape.tile_n ? (Qrows + 7) / 8 * 8 : shape.tile_n;
    if (!encode_operand(&tmP, Pp, Prows, K * kx, ldP * kx, kTileM) ||
        !encode_operand(&tmQ, Qp, Qrows, K * kx, ldQ * kx, q_box))
        return MXFP4_ERR_CUDA;

    GemmArgs a;
    std::memset(&a, 0, sizeof(a));
    a.sfP = swap ? sc.b : sc.a;
    a.sfQ = swap ? sc.a : sc.b;
    a.sf_rb_stride = sf_groups(K) * kSfAtomBytes;
    a.sf_rowmajor = sc.rowmajor ? 1 : 0;
    a.ldsP = swap ? sc.ld_b : sc.ld_a;
    a.ldsQ = swap ? sc.ld_a : sc.ld_b;
    a.sf_vec8 = sc.rowmajor && aligned(sc.a, 8) && aligned(sc.b, 8) && (sc.ld_a % 8) == 0 &&
                (sc.ld_b % 8) == 0;
    a.sf_async = sc.rowmajor && aligned(sc.a, 4) && aligned(sc.b, 4) && (sc.ld_a % 4) == 0 &&
                 (sc.ld_b % 4) == 0;
    // Row-major scales whose rows are 16-byte aligned come by TMA (one copy
    // per operand and stage); others are gathered with 4-byte copies.
    a.sf_tma = sc.rowmajor && aligned(sc.a, 16) && aligned(sc.b, 16) && (sc.ld_a % 16) == 0 &&
               (sc.ld_b % 16) == 0;
    a.q_box_rows = q_box;
    CUtensorMap tmSP = tmP, tmSQ = tmQ;   // unused unless a.sf_tma
    const int kbytes = nv ? K / 16 : K / 32;
    if (a.sf_tma && (!encode_scales(&tmSP, a.sfP, Prows, kbytes, a.ldsP, kTileM) ||
                     !encode_scales(&tmSQ, a.sfQ, Qrows, kbytes, a.ldsQ, q_box)))
        return MXFP4_ERR_CUDA;
    a.rowsP = Prows;
    a.rowsQ = Qrows;
    a.M = M;
    a.N = N;
    a.K = K;
    a.kt_total = (K * kx + kTileK - 1) / kTileK;
    a.kt_per_split = plan.k_tiles_per_split;
    a.fmt_p = swap ? fmt_b : fmt_a;
    a.fmt_q = swap ? fmt_a : fmt_b;
    a.split_k = plan.split_k;
    a.alpha = alpha;
    a.beta = beta;
    a.C = static_cast<const uint16_t *>(beta != 0.0f ? C : nullptr);
    a.ldc = ldc;
    a.D = static_cast<uint16_t *>(D);
    a.ldd = ldd;
    if (plan.split_k > 1 && plan.split_k <= kMaxClusterSplit) {
        a.part_cols = Qrows < shape.tile_n ? Qrows : shape.tile_n;
        a.cluster_reduce = 1;
    } else if (plan.split_k > 1) {
        if (!ws)
            return MXFP4_ERR_WORKSPACE;
        const int64_t tiles = static_cast<int64_t>(plan.grid_x) * plan.grid_y;
        a.part_cols = Qrows < shape.tile_n ? Qrows : shape.tile_n;
        a.tile_count = reinterpret_cast<unsigned long long *>(ws);
        a.partials = reinterpret_cast<float *>(ws + align_up(static_cast<size_t>(tiles) * 8));
        a.epoch = next_epoch();
    }
    a.vec_ok = aligned(D, 16) && (ldd % 8) == 0 &&
               (beta == 0.0f || (aligned(C, 16) && (ldc % 8) == 0));
    a.vec32_ok = a.vec_ok && aligned(D, 32) && (ldd % 16) == 0;
    a.stream_p = swap ? 1 : 0;
    a.p_is_b = swap ? 1 : 0;
    // B (and its scales) may be read before the preceding work ends only
    // when the caller says that work does not write them, and when no
    // relayout pass of this call is that work.
    a.b_early = ((flags & MXFP4_FLAG_B_STATIC) && !after_relayout) ? 1 : 0;
    a.wait_limit = g_wait_limit.load();

    dim3 grid(plan.grid_x, plan.grid_y, plan.grid_z);
    if (launch_gemm(a, tmP, tmQ, tmSP, tmSQ, shape, grid, stream) != cudaSuccess)
        return MXFP4_ERR_CUDA;
    return MXFP4_OK;
}

}  // namespace

extern "C" {

int mxfp4_version(void) { return 1 * 10000 + 0 * 100 + 0; }

const char *mxfp4_strerror(int status)
{
    switch (status) {
    case MXFP4_OK: return "ok";
    case MXFP4_ERR_INVALID_ARG: return "invalid argument";
    case MXFP4_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MXFP4_ERR_MISALIGNED: return "misaligned pointer or stride";
    case MXFP4_ERR_WORKSPACE: return "workspace missing or too small";
    case MXFP4_ERR_CUDA: return "CUDA runtime error";
    case MXFP4_ERR_TIMEOUT: return "in-kernel wait timed out";
    case MXFP4_ERR_ARCH: return "device is not sm_103";
    default: return "unknown status";
    }
}

void mxfp4_set_wait_limit(long long cycles) { g_wait_limit.store(cycles > 0 ? cycles : 1); }

int mxfp4_plan_gemm(int M, int N, int K, int split_k, int num_sms, mxfp4_plan *out)
{
    if (!out)
        return MXFP4_ERR_INVALID_ARG;
    if (num_sms <= 0)
        num_sms = device_sms_or_default();
    return make_plan(M, N, K, split_k, num_sms, out, nullptr);
}

size_t mxfp4_scale_relayout_size(int rows, int K)
{
    if (rows < 1 || K < 32 || (K % 32) != 0)
        return 0;
    return sf_relaid_bytes(rows, K);
}

size_t mxfp4_gemm_prepacked_workspace_size(int M, int N, int K, int split_k)
{
    mxfp4_plan plan;
    if (make_plan(M, N, K, split_k, device_sms_or_default(), &plan, nullptr) != MXFP4_OK)
        return 0;
    return plan.workspace_bytes;
}

size_t mxfp4_gemm_workspace_size(int M, int N, int K, int split_k)
{
    mxfp4_plan plan;
    if (make_plan(M, N, K, split_k, device_sms_or_default(), &plan, nullptr) != MXFP4_OK)
        return 0;
    size_t ws = plan.workspace_bytes;
    if (plan.relayout_pass)
        ws += align_up(sf_relaid_bytes(M, K)) + align_up(sf_relaid_bytes(N, K));
    return ws;
}

int mxfp4_scale_relayout(void *dst, const void *src, int rows, int K, int64_t ld_src, void *stream)
{
    if (!dst || !src || rows < 1 || K < 32 || (K % 32) != 0 || ld_src < K / 32)
        return MXFP4_ERR_INVALID_ARG;
    if (!aligned(dst, 16))
        return MXFP4_ERR_MISALIGNED;
    if (sf_row_blocks(rows) > 0x7FFFFFFF)
        return MXFP4_ERR_UNSUPPORTED_SHAPE;
    int st = check_device();
    if (st != MXFP4_OK)
        return st;
    if (launch_scale_relayout(static_cast<uint8_t *>(dst), static_cast<const uint8_t *>(src), rows, K,
                              ld_src, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MXFP4_ERR_CUDA;
    return MXFP4_OK;
}

int mxfp4_scale_relayout2(void *dst_a, const void *src_a, int rows_a, int64_t ld_a, void *dst_b,
                          const void *src_b, int rows_b, int64_t ld_b, int K, void *stream)
{
    if (!dst_a || !src_a || !dst_b || !src_b || rows_a < 1 || rows_b < 1 || K < 32 ||
        (K % 32) != 0 || ld_a < K / 32 || ld_b < K / 32)
        return MXFP4_ERR_INVALID_ARG;
    if (!aligned(dst_a, 16) || !aligned(dst_b, 16))
        return MXFP4_ERR_MISALIGNED;
    if (sf_row_blocks(rows_a) + sf_row_blocks(rows_b) > 0x7FFFFFFF)
        return MXFP4_ERR_UNSUPPORTED_SHAPE;
    int st = check_device();
    if (st != MXFP4_OK)
        return st;
    if (launch_scale_relayout2(static_cast<uint8_t *>(dst_a), static_cast<const uint8_t *>(src_a),
                               rows_a, ld_a, static_cast<uint8_t *>(dst_b),
                               static_cast<const uint8_t *>(src_b), rows_b, ld_b, K,
                               static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MXFP4_ERR_CUDA;
    return MXFP4_OK;
}

// Shared body of mxfp4_gemm and mxfp4_gemm_prepacked after their own checks.
// fp8: K counts 8-bit elements (the plan is that of an fp4 GEMM of 2K).
static int gemm_entry(void *D, int64_t ldd, const void *C, int64_t ldc, const void *A, int64_t lda,
                      const void *B, int64_t ldb, const Scales &sc, float alpha, float beta, int M,
                      int N, int K, int split_k, void *workspace, size_t workspace_bytes,
                      void *stream, bool fp8 = false, int fmt_a = 0, int fmt_b = 0)
{
    const int sms = device_sms_or_default();
    mxfp4_plan plan;
    GemmShape shape;
    int st = make_plan(M, N, fp8 ? 2 * K : K, split_k, sms, &plan, &shape, fp8);
    if (st != MXFP4_OK)
        return st;
    if (plan.workspace_bytes > 0) {
        if (!workspace || workspace_bytes < plan.workspace_bytes)
            return MXFP4_ERR_WORKSPACE;
        if (!aligned(workspace, kAlign))
            return MXFP4_ERR_MISALIGNED;
    }
    st = check_device();
    if (st != MXFP4_OK)
        return st;
    return run_gemm(D, ldd, C, ldc, A, lda, B, ldb, sc, alpha, beta, M, N, K, plan, shape,
                    plan.workspace_bytes ? static_cast<uint8_t *>(workspace) : nullptr,
                    static_cast<cudaStream_t>(stream), false, fmt_a, fmt_b);
}

int mxfp4_gemm_prepacked(void *D, int64_t ldd, const void *C, int64_t ldc, const void *A,
                         int64_t lda, const void *B, int64_t ldb, const void *scaleA_relaid,
                         const void *scaleB_relaid, float alpha, float beta, int M, int N, int K,
                         int split_k, void *workspace, size_t workspace_bytes, void *stream)
{
    int st = check_common(D, ldd, C, ldc, A, lda, B, ldb, beta, M, N, K, split_k);
    if (st != MXFP4_OK)
        return st;
    if (!scaleA_relaid || !scaleB_relaid)
        return MXFP4_ERR_INVALID_ARG;
    if (!aligned(scaleA_relaid, 16) || !aligned(scaleB_relaid, 16))
        return MXFP4_ERR_MISALIGNED;
    const Scales sc{static_cast<const uint8_t *>(scaleA_relaid),
                    static_cast<const uint8_t *>(scaleB_relaid), 0, 0, false};
    return gemm_entry(D, ldd, C, ldc, A, lda, B, ldb, sc, alpha, beta, M, N, K, split_k, workspace,
                      workspace_bytes, stream);
}

// mxfp4_gemm and mxfp8_gemm: row-major scales, relaid into the workspace
// first when the plan asks for it.  fp8: K counts 8-bit elements (the plan
// is that of an fp4 GEMM of 2K, which has the same bytes per row).
// Element formats of the one-byte-per-element GEMM; each enum value is the
// format's code in the kind::mxf8f6f4 instruction descriptor.
static bool byte_format_ok(int fmt)
{
    return fmt == MXFP8_E4M3 || fmt == MXFP8_E5M2 || fmt == MXFP6_E2M3 || fmt == MXFP6_E3M2 ||
           fmt == MXFP4_E2M1_PADDED;
}

static int gemm_rowmajor(void *D, int64_t ldd, const void *C, int64_t ldc, const void *A,
                         int64_t lda, const void *B, int64_t ldb, const void *scaleA,
                         int64_t ld_sa, const void *scaleB, int64_t ld_sb, float alpha, float beta,
                         int M, int N, int K, int split_k, void *workspace, size_t workspace_bytes,
                         void *stream, bool fp8, int fmt_a, int fmt_b, unsigned flags = 0)
{
    const int kx = fp8 ? 2 : 1;
    if (fp8 && (K > (1 << 29) || lda > (INT64_MAX / 4) || ldb > (INT64_MAX / 4)))
        return MXFP4_ERR_INVALID_ARG;
    int st = check_common(D, ldd, C, ldc, A, lda * kx, B, ldb * kx, beta, M, N, K * kx, split_k);
    if (st != MXFP4_OK)
        return st;
    if (K < 32 || (K % 32) != 0)
        return MXFP4_ERR_INVALID_ARG;
    if (!scaleA || !scaleB || ld_sa < K / 32 || ld_sb < K / 32)
        return MXFP4_ERR_INVALID_ARG;
    if (fp8 && (!byte_format_ok(fmt_a) || !byte_format_ok(fmt_b)))
        return MXFP4_ERR_INVALID_ARG;
    if (workspace && !aligned(workspace, kAlign))
        return MXFP4_ERR_MISALIGNED;
    const int sms = device_sms_or_default();
    mxfp4_plan plan;
    GemmShape shape;
    st = make_plan(M, N, K * kx, split_k, sms, &plan, &shape, fp8);
    if (st != MXFP4_OK)
        return st;
    const size_t sfa_bytes = plan.relayout_pass ? align_up(sf_relaid_bytes(M, K)) : 0;
    const size_t sfb_bytes = plan.relayout_pass ? align_up(sf_relaid_bytes(N, K)) : 0;
    // Layout: [split-K counters + partials (plan.workspace_bytes)][relaid A][relaid B].
    const size_t head = plan.workspace_bytes;
    const size_t need = head + sfa_bytes + sfb_bytes;
    if (need > 0 && (!workspace || workspace_bytes < need))
        return MXFP4_ERR_WORKSPACE;
    st = check_device();
    if (st != MXFP4_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    Scales sc{static_cast<const uint8_t *>(scaleA), static_cast<const uint8_t *>(scaleB), ld_sa,
              ld_sb, true};
    if (plan.relayout_pass) {
        uint8_t *sfa = ws + head;
        uint8_t *sfb = sfa + sfa_bytes;
        if (launch_scale_relayout2(sfa, sc.a, M, ld_sa, sfb, sc.b, N, ld_sb, K, s) != cudaSuccess)
            return MXFP4_ERR_CUDA;
        sc = Scales{sfa, sfb, 0, 0, false};
    }
    return run_gemm(D, ldd, C, ldc, A, lda, B, ldb, sc, alpha, beta, M, N, K, plan, shape,
                    plan.workspace_bytes ? ws : nullptr, s, plan.relayout_pass != 0, fmt_a,
                    fmt_b, flags);
}

int mxfp4_gemm(void *D, int64_t ldd, const void *C, int64_t ldc, const void *A, int64_t lda,
               const void *B, int64_t ldb, const void *scaleA, int64_t ld_sa, const void *scaleB,
               int64_t ld_sb, float alpha, float beta, int M, int N, int K, int split_k,
               void *workspace, size_t workspace_bytes, void *stream)
{
    return gemm_rowmajor(D, ldd, C, ldc, A, lda, B, ldb, scaleA, ld_sa, scaleB, ld_sb, alpha, beta,
                         M, N, K, split_k, workspace, workspace_bytes, stream, false, 0, 0);
}

int mxfp4_gemm_ex(void *D, int64_t ldd, const void *C, int64_t ldc, const void *A, int64_t lda,
                  const void *B, int64_t ldb, const void *scaleA, int64_t ld_sa, const void *scaleB,
                  int64_t ld_sb, float alpha, float beta, int M, int N, int K, int split_k,
                  unsigned flags, void *workspace, size_t workspace_bytes, void *stream)
{
    if ((flags & ~static_cast<unsigned>(MXFP4_FLAG_B_STATIC)) != 0)
        return MXFP4_ERR_INVALID_ARG;
    return gemm_rowmajor(D, ldd, C, ldc, A, lda, B, ldb, scaleA, ld_sa, scaleB, ld_sb, alpha, beta,
                         M, N, K, split_k, workspace, workspace_bytes, stream, false, 0, 0, flags);
}

int mxfp8_gemm(void *D, int64_t ldd, const void *C, int64_t ldc, const void *A, int64_t lda,
               const void *B, int64_t ldb, const void *scaleA, int64_t ld_sa, const void *scaleB,
               int64_t ld_sb, int fmt_a, int fmt_b, float alpha, float beta, int M, int N, int K,
               int split_k, void *workspace, size_t workspace_bytes, void *stream)
{
    return gemm_rowmajor(D, ldd, C, ldc, A, lda, B, ldb, scaleA, ld_sa, scaleB, ld_sb, alpha, beta,
                         M, N, K, split_k, workspace, workspace_bytes, stream, true, fmt_a, fmt_b);
}

// NVFP4 plan: skinny shapes (M <= 64, swap-AB) run the one-tile kernel with
// the MXFP4 plan's tile and split and the row-major scales read by TMA (no
// workspace up to 8 splits); every other shape runs the CTA-pair kernel on
// relaid scales.
static bool nv_one_tile(int M, int N, int K, mxfp4_plan *plan, GemmShape *shape)
{
    if (!(M <= 64 && N > M))
        return false;
    return make_plan(M, N, K, 0, device_sms_or_default(), plan, shape, false) == MXFP4_OK &&
           plan->swap_ab == 1 && plan->pair == 0 && plan->split_k <= kMaxClusterSplit;
}

size_t nvfp4_gemm_workspace_size(int M, int N, int K)
{
    if (M < 1 || N < 1 || K < 32 || (K % 32) != 0)
        return 0;
    // The relaid scales of the pair kernel.  (The skinny path needs none when
    // the caller's scale rows are 16-byte aligned; with other scale rows it
    // falls back to the pair kernel, so the size covers that case too.)
    return align_up(sf_relaid_bytes_nv(M, K)) + align_up(sf_relaid_bytes_nv(N, K));
}

// NVFP4: the scales are relaid into the workspace (one launch for both
// operands), then the CTA-pair kernel runs as its programmatic dependent, for
// every shape.
int nvfp4_gemm(void *D, int64_t ldd, const void *C, int64_t ldc, const void *A, int64_t lda,
               const void *B, int64_t ldb, const void *scaleA, int64_t ld_sa, const void *scaleB,
               int64_t ld_sb, float alpha, float beta, int M, int N, int K, void *workspace,
               size_t workspace_bytes, void *stream)
{
    int st = check_common(D, ldd, C, ldc, A, lda, B, ldb, beta, M, N, K, 0);
    if (st != MXFP4_OK)
        return st;
    if (!scaleA || !scaleB || ld_sa < K / 16 || ld_sb < K / 16)
        return MXFP4_ERR_INVALID_ARG;
    const int64_t tiles = ((static_cast<int64_t>(M) + 255) / 256) * ((static_cast<int64_t>(N) + 255) / 256);
    if (tiles > 0x7FFFFFFF)
        return MXFP4_ERR_UNSUPPORTED_SHAPE;
    {
        mxfp4_plan plan;
        GemmShape shape;
        if (nv_one_tile(M, N, K, &plan, &shape) && aligned(scaleA, 16) && aligned(scaleB, 16) &&
            (ld_sa % 16) == 0 && (ld_sb % 16) == 0) {
            if (workspace && !aligned(workspace, kAlign))
                return MXFP4_ERR_MISALIGNED;
            st = check_device();
            if (st != MXFP4_OK)
                return st;
            shape.nv = 1;
            const Scales sc{static_cast<const uint8_t *>(scaleA), static_cast<const uint8_t *>(scaleB),
                            ld_sa, ld_sb, true};
            return run_gemm(D, ldd, C, ldc, A, lda, B, ldb, sc, alpha, beta, M, N, K, plan, shape,
                            nullptr, static_cast<cudaStream_t>(stream), false, 0, 0, 0, true);
        }
    }
    const size_t sfa_bytes = align_up(sf_relaid_bytes_nv(M, K));
    const size_t sfb_bytes = align_up(sf_relaid_bytes_nv(N, K));
    if (!workspace || workspace_bytes < sfa_bytes + sfb_bytes)
        return MXFP4_ERR_WORKSPACE;
    if (!aligned(workspace, kAlign))
        return MXFP4_ERR_MISALIGNED;
    st = check_device();
    if (st != MXFP4_OK)
        return st;
    const int64_t pairs = device_sms_or_default() / 2;
    mxfp4_plan plan;
    std::memset(&plan, 0, sizeof(plan));
    GemmShape shape;
    std::memset(&shape, 0, sizeof(shape));
    shape.tile_n = 256;
    shape.stages = 5;
    shape.ctas_per_sm = 1;
    shape.pair = 1;
    shape.pair_ctas = 2 * static_cast<int>(tiles < pairs ? tiles : pairs);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *sfa = static_cast<uint8_t *>(workspace);
    uint8_t *sfb = sfa + sfa_bytes;
    if (launch_scale_relayout2_nv(sfa, static_cast<const uint8_t *>(scaleA), M, ld_sa, sfb,
                                  static_cast<const uint8_t *>(scaleB), N, ld_sb, K, s) != cudaSuccess)
        return MXFP4_ERR_CUDA;
    const Scales sc{sfa, sfb, 0, 0, false};
    return run_gemm(D, ldd, C, ldc, A, lda, B, ldb, sc, alpha, beta, M, N, K, plan, shape, nullptr,
                    s, true, 0, 0, 0, true);
}

int mxfp8_gemm_prepacked(void *D, int64_t ldd, const void *C, int64_t ldc, const void *A,
                         int64_t lda, const void *B, int64_t ldb, const void *scaleA_relaid,
                         const void *scaleB_relaid, int fmt_a, int fmt_b, float alpha, float beta,
                         int M, int N, int K, int split_k, void *workspace, size_t workspace_bytes,
                         void *stream)
{
    if (K > (1 << 29) || lda > (INT64_MAX / 4) || ldb > (INT64_MAX / 4))
        return MXFP4_ERR_INVALID_ARG;
    int st = check_common(D, ldd, C, ldc, A, lda * 2, B, ldb * 2, beta, M, N, K * 2, split_k);
    if (st != MXFP4_OK)
        return st;
    if (K < 32 || (K % 32) != 0 || !scaleA_relaid || !scaleB_relaid)
        return MXFP4_ERR_INVALID_ARG;
    if (!byte_format_ok(fmt_a) || !byte_format_ok(fmt_b))
        return MXFP4_ERR_INVALID_ARG;
    if (!aligned(scaleA_relaid, 16) || !aligned(scaleB_relaid, 16))
        return MXFP4_ERR_MISALIGNED;
    const Scales sc{static_cast<const uint8_t *>(scaleA_relaid),
                    static_cast<const uint8_t *>(scaleB_relaid), 0, 0, false};
    return gemm_entry(D, ldd, C, ldc, A, lda, B, ldb, sc, alpha, beta, M, N, K, split_k, workspace,
                      workspace_bytes, stream, true, fmt_a, fmt_b);
}

size_t mxfp8_gemm_prepacked_workspace_size(int M, int N, int K, int split_k)
{
    mxfp4_plan plan;
    if (K < 32 || (K % 32) != 0 || K > (1 << 29) ||
        make_plan(M, N, 2 * K, split_k, device_sms_or_default(), &plan, nullptr, true) != MXFP4_OK)
        return 0;
    return plan.workspace_bytes;
}

int mxfp8_plan_gemm(int M, int N, int K, int split_k, int num_sms, mxfp4_plan *out)
{
    if (!out || K < 32 || (K % 32) != 0 || K > (1 << 29))
        return MXFP4_ERR_INVALID_ARG;
    if (num_sms <= 0)
        num_sms = device_sms_or_default();
    const int st = make_plan(M, N, 2 * K, split_k, num_sms, out, nullptr, true);
    if (st == MXFP4_OK)
        out->tile_k = kTileK / 2;           // 8-bit elements per stage
    return st;
}

size_t mxfp8_gemm_workspace_size(int M, int N, int K, int split_k)
{
    mxfp4_plan plan;
    if (K < 32 || (K % 32) != 0 || K > (1 << 29) ||
        make_plan(M, N, 2 * K, split_k, device_sms_or_default(), &plan, nullptr, true) != MXFP4_OK)
        return 0;
    size_t ws = plan.workspace_bytes;
    if (plan.relayout_pass)
        ws += align_up(sf_relaid_bytes(M, K)) + align_up(sf_relaid_bytes(N, K));
    return ws;
}

// Rows per panel of the pipelined host call: eight panels of a multiple of
// 256 rows once M reaches 2048 (each panel still fills the GPU with 256-row
// pair tiles); one panel below that.
static int host_panel_rows(int M)
{
    if (M < 2048)
        return M;
    const int rows = (M + 7) / 8;
    return (rows + 255) / 256 * 256;
}

// Columns per block of the pipelined host call: with row panels and N >= 2048
// two halves (a multiple of 256 columns each), so that the first GEMM waits
// for half of B rather than all of it; otherwise all N columns.
static int host_block_cols(int M, int N)
{
    if (M < 2048 || N < 2048)
        return N;
    return ((N + 1) / 2 + 255) / 256 * 256;
}

// Element form of a host-buffer call: packed E2M1 (two per byte) or one of
// the byte forms of mxfp8_gemm (fmt_a / fmt_b are then its format codes).
struct HostForm {
    bool bytes;
    int fmt_a, fmt_b;
};

static size_t host_arena_size(int M, int N, int K, int split_k, int with_c, HostForm f)
{
    if (M < 1 || N < 1 || K < 32 || (K % 32) != 0 || split_k < 0 || split_k > kMaxSplit)
        return 0;
    // Workspace of the block GEMMs: the largest over the block shapes (full
    // and last row panel x full and last column block).
    const int mp = host_panel_rows(M), nc = host_block_cols(M, N);
    const int rows[2] = {mp, M - (M - 1) / mp * mp};
    const int cols[2] = {nc, N - (N - 1) / nc * nc};
    size_t ws = 0;
    for (int r : rows)
        for (int c : cols) {
            const size_t w = f.bytes ? mxfp8_gemm_workspace_size(r, c, K, split_k)
                                     : mxfp4_gemm_workspace_size(r, c, K, split_k);
            ws = w > ws ? w : ws;
        }
    const size_t row = f.bytes ? static_cast<size_t>(K) : static_cast<size_t>(K) / 2;
    const size_t mn2 = align_up(static_cast<size_t>(M) * N * 2);
    return align_up(static_cast<size_t>(M) * row) + align_up(static_cast<size_t>(N) * row) +
           align_up(static_cast<size_t>(M) * K / 32) + align_up(static_cast<size_t>(N) * K / 32) +
           (with_c ? mn2 : 0) + mn2 + ws;
}

size_t mxfp4_gemm_host_arena_size(int M, int N, int K, int split_k, int with_c)
{
    return host_arena_size(M, N, K, split_k, with_c, HostForm{false, 0, 0});
}

size_t mxfp8_gemm_host_arena_size(int M, int N, int K, int split_k, int with_c)
{
    return host_arena_size(M, N, K, split_k, with_c, HostForm{true, 0, 0});
}

namespace {

// Per-device copy streams and events of the pipelined host call, created on
// first use and reused under a lock (a later record of an event does not
// affect waits enqueued before it).
constexpr int kHostMaxPanels = 8;
constexpr int kHostMaxColBlocks = 2;
struct HostPipe {
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t b_in[kHostMaxColBlocks] = {}, in[kHostMaxPanels] = {};
    cudaEvent_t out[kHostMaxPanels * kHostMaxColBlocks] = {};
    std::mutex lock;
};

HostPipe *host_pipe(int dev)
{
    static HostPipe pipes[64];
    static std::mutex init_lock;
    if (dev < 0 || dev >= 64)
        return nullptr;
    HostPipe *p = &pipes[dev];
    std::lock_guard<std::mutex> g(init_lock);
    if (!p->h2d) {
        auto ev = [](cudaEvent_t *e) { return cudaEventCreateWithFlags(e, cudaEventDisableTiming); };
        if (cudaStreamCreateWithFlags(&p->h2d, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&p->d2h, cudaStreamNonBlocking) != cudaSuccess ||
            ev(&p->start) != cudaSuccess || ev(&p->done) != cudaSuccess) {
            p->h2d = nullptr;
            return nullptr;
        }
        bool made = true;
        for (cudaEvent_t &e : p->b_in)
            made = made && ev(&e) == cudaSuccess;
        for (cudaEvent_t &e : p->in)
            made = made && ev(&e) == cudaSuccess;
        for (cudaEvent_t &e : p->out)
            made = made && ev(&e) == cudaSuccess;
        if (!made) {
            p->h2d = nullptr;
            return nullptr;
        }
    }
    return p;
}

}  // namespace

static int gemm_host(void *D_host, const void *C_host, const void *A_host, const void *B_host,
                     const void *scaleA_host, const void *scaleB_host, float alpha, float beta,
                     int M, int N, int K, int split_k, void *device_arena, size_t arena_bytes,
                     void *stream, HostForm form)
{
    if (!D_host || !A_host || !B_host || !scaleA_host || !scaleB_host || !device_arena)
        return MXFP4_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 32 || (K % 32) != 0 || split_k < 0 || split_k > kMaxSplit)
        return MXFP4_ERR_INVALID_ARG;
    if (beta != 0.0f && !C_host)
        return MXFP4_ERR_INVALID_ARG;
    if (form.bytes && (!byte_format_ok(form.fmt_a) || !byte_format_ok(form.fmt_b)))
        return MXFP4_ERR_INVALID_ARG;
    if (!aligned(device_arena, kAlign))
        return MXFP4_ERR_MISALIGNED;
    const int with_c = beta != 0.0f;
    const size_t need = host_arena_size(M, N, K, split_k, with_c, form);
    if (need == 0 || arena_bytes < need)
        return MXFP4_ERR_WORKSPACE;
    int st = check_device();
    if (st != MXFP4_OK)
        return st;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return MXFP4_ERR_CUDA;
    HostPipe *pipe = host_pipe(dev);
    if (!pipe)
        return MXFP4_ERR_CUDA;
    uint8_t *p = static_cast<uint8_t *>(device_arena);
    const size_t arow = form.bytes ? static_cast<size_t>(K) : static_cast<size_t>(K) / 2;
    const size_t srow = static_cast<size_t>(K) / 32;
    const size_t drow = static_cast<size_t>(N) * 2;
    const size_t a_b = static_cast<size_t>(M) * arow, b_b = static_cast<size_t>(N) * arow;
    const size_t sa_b = static_cast<size_t>(M) * srow, sb_b = static_cast<size_t>(N) * srow;
    const size_t mn2 = static_cast<size_t>(M) * drow;
    uint8_t *dA = p;
    p += align_up(a_b);
    uint8_t *dB = p;
    p += align_up(b_b);
    uint8_t *dSA = p;
    p += align_up(sa_b);
    uint8_t *dSB = p;
    p += align_up(sb_b);
    uint8_t *dC = nullptr;
    if (with_c) {
        dC = p;
        p += align_up(mn2);
    }
    uint8_t *dD = p;
    p += align_up(mn2);
    uint8_t *ws = p;
    const size_t ws_bytes = arena_bytes - static_cast<size_t>(p - static_cast<uint8_t *>(device_arena));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const auto *hA = static_cast<const uint8_t *>(A_host);
    const auto *hSA = static_cast<const uint8_t *>(scaleA_host);
    const auto *hC = static_cast<const uint8_t *>(C_host);
    auto *hD = static_cast<uint8_t *>(D_host);

    // Blocks of row panels x column blocks.  On the copy-in stream: column
    // block 0 of B and its scales, then each row panel of A with its scales
    // and C, then the other column blocks of B.  The GEMMs run on `stream`,
    // column block by column block, each row panel once its rows (and the
    // block's B) landed; each block of D goes back on the copy-out stream
    // while the next computes.  The copy streams start after the work
    // already on `stream`, and `stream` ends after the last copy of D.
    const int mp = host_panel_rows(M), nc = host_block_cols(M, N);
    const int panels = (M + mp - 1) / mp, blocks = (N + nc - 1) / nc;
    std::lock_guard<std::mutex> g(pipe->lock);
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    auto copy_b = [&](int j) {
        const size_t n0 = static_cast<size_t>(j) * nc;
        const size_t cols = N - n0 < static_cast<size_t>(nc) ? N - n0 : nc;
        return ok(cudaMemcpyAsync(dB + n0 * arow, static_cast<const uint8_t *>(B_host) + n0 * arow,
                                  cols * arow, cudaMemcpyHostToDevice, pipe->h2d)) &&
               ok(cudaMemcpyAsync(dSB + n0 * srow,
                                  static_cast<const uint8_t *>(scaleB_host) + n0 * srow,
                                  cols * srow, cudaMemcpyHostToDevice, pipe->h2d)) &&
               ok(cudaEventRecord(pipe->b_in[j], pipe->h2d));
    };
    if (!ok(cudaEventRecord(pipe->start, s)) || !ok(cudaStreamWaitEvent(pipe->h2d, pipe->start, 0)) ||
        !ok(cudaStreamWaitEvent(pipe->d2h, pipe->start, 0)) || !copy_b(0))
        return MXFP4_ERR_CUDA;
    for (int i = 0; i < panels; ++i) {
        const size_t m0 = static_cast<size_t>(i) * mp;
        const size_t rows = M - m0 < static_cast<size_t>(mp) ? M - m0 : mp;
        if (!ok(cudaMemcpyAsync(dA + m0 * arow, hA + m0 * arow, rows * arow, cudaMemcpyHostToDevice,
                                pipe->h2d)) ||
            !ok(cudaMemcpyAsync(dSA + m0 * srow, hSA + m0 * srow, rows * srow,
                                cudaMemcpyHostToDevice, pipe->h2d)) ||
            (with_c && !ok(cudaMemcpyAsync(dC + m0 * drow, hC + m0 * drow, rows * drow,
                                           cudaMemcpyHostToDevice, pipe->h2d))) ||
            !ok(cudaEventRecord(pipe->in[i], pipe->h2d)))
            return MXFP4_ERR_CUDA;
    }
    for (int j = 1; j < blocks; ++j)
        if (!copy_b(j))
            return MXFP4_ERR_CUDA;
    for (int j = 0; j < blocks; ++j) {
        const size_t n0 = static_cast<size_t>(j) * nc;
        const int cols = static_cast<int>(N - n0 < static_cast<size_t>(nc) ? N - n0 : nc);
        if (!ok(cudaStreamWaitEvent(s, pipe->b_in[j], 0)))
            return MXFP4_ERR_CUDA;
        for (int i = 0; i < panels; ++i) {
            const size_t m0 = static_cast<size_t>(i) * mp;
            const int rows = static_cast<int>(M - m0 < static_cast<size_t>(mp) ? M - m0 : mp);
            const size_t d_off = m0 * drow + n0 * 2;
            if (j == 0 && !ok(cudaStreamWaitEvent(s, pipe->in[i], 0)))
                return MXFP4_ERR_CUDA;
            if (form.bytes)
                st = mxfp8_gemm(dD + d_off, N, with_c ? dC + d_off : nullptr, N, dA + m0 * arow,
                                K, dB + n0 * arow, K, dSA + m0 * srow, K / 32, dSB + n0 * srow,
                                K / 32, form.fmt_a, form.fmt_b, alpha, beta, rows, cols, K,
                                split_k, ws, ws_bytes, stream);
            else
                st = mxfp4_gemm(dD + d_off, N, with_c ? dC + d_off : nullptr, N, dA + m0 * arow,
                                K, dB + n0 * arow, K, dSA + m0 * srow, K / 32, dSB + n0 * srow,
                                K / 32, alpha, beta, rows, cols, K, split_k, ws, ws_bytes, stream);
            if (st != MXFP4_OK)
                return st;
            cudaEvent_t out = pipe->out[j * kHostMaxPanels + i];
            if (!ok(cudaEventRecord(out, s)) || !ok(cudaStreamWaitEvent(pipe->d2h, out, 0)) ||
                !ok(cudaMemcpy2DAsync(hD + d_off, drow, dD + d_off, drow, static_cast<size_t>(cols) * 2,
                                      rows, cudaMemcpyDeviceToHost, pipe->d2h)))
                return MXFP4_ERR_CUDA;
        }
    }
    if (!ok(cudaEventRecord(pipe->done, pipe->d2h)) || !ok(cudaStreamWaitEvent(s, pipe->done, 0)))
        return MXFP4_ERR_CUDA;
    return MXFP4_OK;
}

int mxfp4_gemm_host(void *D_host, const void *C_host, const void *A_host, const void *B_host,
                    const void *scaleA_host, const void *scaleB_host, float alpha, float beta,
                    int M, int N, int K, int split_k, void *device_arena, size_t arena_bytes,
                    void *stream)
{
    return gemm_host(D_host, C_host, A_host, B_host, scaleA_host, scaleB_host, alpha, beta, M, N,
                     K, split_k, device_arena, arena_bytes, stream, HostForm{false, 0, 0});
}

int mxfp8_gemm_host(void *D_host, const void *C_host, const void *A_host, const void *B_host,
                    const void *scaleA_host, const void *scaleB_host, int fmt_a, int fmt_b,
                    float alpha, float beta, int M, int N, int K, int split_k,
                    void *device_arena, size_t arena_bytes, void *stream)
{
    return gemm_host(D_host, C_host, A_host, B_host, scaleA_host, scaleB_host, alpha, beta, M, N,
                     K, split_k, device_arena, arena_bytes, stream, HostForm{true, fmt_a, fmt_b});
}

int mxfp4_device_status(int *status, int reset)
{
    if (!status)
        return MXFP4_ERR_INVALID_ARG;
    int st = check_device();
    if (st != MXFP4_OK)
        return st;
    return read_device_status(status, reset) == cudaSuccess ? MXFP4_OK : MXFP4_ERR_CUDA;
}

int mxfp4_wait_timeout_probe(long long limit_cycles, void *stream)
{
    if (limit_cycles <= 0)
        return MXFP4_ERR_INVALID_ARG;
    int st = check_device();
    if (st != MXFP4_OK)
        return st;
    return launch_wait_probe(limit_cycles, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? MXFP4_OK
               : MXFP4_ERR_CUDA;
}

int mxfp8_quantize(void *Q, int64_t ldq, void *S, int64_t lds, const void *X, int64_t ldx,
                   int rows, int K, int fmt, void *stream)
{
    if (!Q || !S || !X || rows < 1 || K < 32 || (K % 32) != 0 || ldx < K || ldq < K ||
        lds < K / 32 || !byte_format_ok(fmt))
        return MXFP4_ERR_INVALID_ARG;
    if (!aligned(X, 16) || (ldx % 8) != 0 || !aligned(Q, 16) || (ldq % 16) != 0)
        return MXFP4_ERR_MISALIGNED;
    int st = check_device();
    if (st != MXFP4_OK)
        return st;
    return launch_quantize8(static_cast<uint8_t *>(Q), ldq, static_cast<uint8_t *>(S), lds,
                            static_cast<const uint16_t *>(X), ldx, rows, K, fmt,
                            device_sms_or_default(), static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? MXFP4_OK
               : MXFP4_ERR_CUDA;
}

int mxfp4_quantize(void *Q, int64_t ldq, void *S, int64_t lds, const void *X, int64_t ldx,
                   int rows, int K, void *stream)
{
    if (!Q || !S || !X || rows < 1 || K < 32 || (K % 32) != 0 || ldx < K || ldq < K ||
        lds < K / 32)
        return MXFP4_ERR_INVALID_ARG;
    if (!aligned(X, 16) || (ldx % 8) != 0 || !aligned(Q, 16) || (ldq % 32) != 0)
        return MXFP4_ERR_MISALIGNED;
    int st = check_device();
    if (st != MXFP4_OK)
        return st;
    return launch_quantize(static_cast<uint8_t *>(Q), ldq / 2, static_cast<uint8_t *>(S), lds,
                           static_cast<const uint16_t *>(X), ldx, rows, K, device_sms_or_default(),
                           static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? MXFP4_OK
               : MXFP4_ERR_CUDA;
}

}  // extern "C"
