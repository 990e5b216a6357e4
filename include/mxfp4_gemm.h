/*
 * mxfp4_gemm.h -- C ABI of the GB300 (sm_103a) block-scaled MXFP4 GEMM.
 *
 *     D[M,N] (bf16) = alpha * A[M,K] (mxfp4) * B[N,K]^T (mxfp4) + beta * C[M,N] (bf16)
 *
 * The operation and its operand formats are those of the page "asm_f4gemm --
 * driving aiter's gfx950 MXFP4 GEMM code objects" (the formula at the top,
 * section "Data layouts", section "Kernel ABI"):
 *   - A [M, K/2] and B [N, K/2]: packed fp4x2 E2M1 bytes, row-major; byte i
 *     of a row holds element 2i in its low nibble and 2i+1 in its high nibble;
 *     magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}, sign in bit 3.
 *   - scaleA [M, K/32] and scaleB [N, K/32]: one E8M0 byte (value 2^(e-127))
 *     per 32 consecutive K elements of a row, row-major.
 *   - C, D: bf16 [M, N] row-major.
 * Each scale multiplies its 32 inputs before they are accumulated (page
 * "CDNA4 dense MFMA builtins", section "Mixed-precision with scaling").
 * Products accumulate in fp32; D is rounded once to bf16 (nearest even).
 *
 * Conventions shared by every entry point:
 *   - All data pointers are DEVICE pointers owned by the caller unless an
 *     entry point says otherwise.  The library never allocates, frees or
 *     retains them, never synchronises the device, and enqueues work on
 *     `stream` only (a cudaStream_t; NULL is the legacy default stream).
 *   - A/B row strides (lda, ldb) are counted in fp4 ELEMENTS, as the page's
 *     kernarg block counts them (stride in bytes = ld / 2).  Scale row strides
 *     (ld_sa, ld_sb) are in bytes.  C/D strides (ldc, ldd) are in elements.
 *   - Every argument is validated before anything is enqueued; on an error
 *     the call returns a negative mxfp4_status and enqueues nothing.  Errors
 *     raised by the CUDA runtime at launch return MXFP4_ERR_CUDA.  Waits
 *     inside the kernels are bounded: one that runs out records
 *     MXFP4_ERR_TIMEOUT in a device status word (mxfp4_device_status) and
 *     the kernel returns instead of hanging.
 *   - Only sm_103 devices are accepted (MXFP4_ERR_ARCH otherwise).
 *   - Functions are safe to call from several host threads.
 *   - mxfp4_gemm, mxfp4_gemm_ex, mxfp4_gemm_prepacked, mxfp4_gemm_host,
 *     the mxfp8_gemm family, the quantisers and the scale relayout can be
 *     captured into a CUDA graph (stream capture), including their
 *     dependent, cluster and split-K launches and the host-buffer entries'
 *     internal copy streams, which fork from and join back to `stream`.  The
 *     first call on a device sets kernel attributes and creates those
 *     streams: make it before capturing.  A replay reads the buffers'
 *     contents at replay time.
 */
#ifndef MXFP4_GEMM_H
#define MXFP4_GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mxfp4_status {
    MXFP4_OK = 0,
    MXFP4_ERR_INVALID_ARG = -1,       /* null pointer, bad size or stride */
    MXFP4_ERR_UNSUPPORTED_SHAPE = -2, /* shape outside what the kernels take */
    MXFP4_ERR_MISALIGNED = -3,        /* pointer or stride breaks a 16-byte rule */
    MXFP4_ERR_WORKSPACE = -4,         /* workspace missing or too small */
    MXFP4_ERR_CUDA = -5,              /* the CUDA runtime reported an error */
    MXFP4_ERR_TIMEOUT = -6,           /* a bounded in-kernel wait ran out */
    MXFP4_ERR_ARCH = -7               /* current device is not sm_103 */
} mxfp4_status;

/* The launch configuration mxfp4_gemm would use for a shape (host only). */
typedef struct mxfp4_plan {
    int swap_ab;            /* 1: computes D^T = B . A^T (skinny M) */
    int tile_m;             /* MMA M rows per tile (rows of A, or of B if swapped) */
    int tile_n;             /* MMA N columns per tile */
    int tile_k;             /* K elements per pipeline stage */
    int stages;             /* shared-memory ring depth */
    int split_k;            /* K splits; > 1: fp32 partials summed in the GEMM */
    int k_tiles_per_split;  /* tile_k blocks handled by one split */
    int grid_x, grid_y, grid_z;
    size_t workspace_bytes; /* split-K tile counters and partials (what
                               mxfp4_gemm_prepacked needs) */
    int relayout_pass;      /* 1: mxfp4_gemm relays the scales out in a separate
                               pass into its workspace (compute-bound shapes);
                               0: the GEMM builds the scale layout itself */
    int pair;               /* 1: CTA-pair kernel (256 x 256 tiles over two SMs) */
    int ctas;               /* pair kernel: CTAs launched (persistent) */
    int waves;              /* pair kernel: most tiles one CTA pair computes */
} mxfp4_plan;

/*
 * Choose tile, swap and split-K for a shape (the tile heuristic of the page's
 * section "Tile selection heuristic": fewest waves over the SMs, then SM
 * occupancy of the last wave, then tile area over perimeter; ties resolved by
 * a fixed candidate order).  split_k = 0 lets the heuristic choose: the
 * CTA-pair kernel (256 x 256 tiles over two SMs) when those tiles fill every
 * SM pair at least once; else no split when the tiles fill at least half a
 * wave, or enough splits to fill the SMs with at least 8 K stages each.
 * 1..16 forces that many splits (clamped to the number of K blocks) on the
 * one-tile kernel.  num_sms = 0 uses the current device's SM count (or 152
 * when no device is visible).  Pure host logic: no GPU work.  Returns
 * MXFP4_OK or MXFP4_ERR_INVALID_ARG.
 */
int mxfp4_plan_gemm(int M, int N, int K, int split_k, int num_sms, mxfp4_plan *out);

/*
 * Bytes of device workspace mxfp4_gemm needs: when the plan splits K, one
 * 8-byte counter per output tile and one fp32 partial tile per (tile, split)
 * (its columns rounded up to a multiple of 4);
 * plus both relaid scale buffers when the plan has a relayout pass; 0 when
 * neither applies (then the workspace may be NULL).  Returns 0 for invalid
 * sizes too (mxfp4_plan_gemm tells them apart).
 */
size_t mxfp4_gemm_workspace_size(int M, int N, int K, int split_k);

/*
 * Bytes of a relaid scale buffer for `rows` rows of K elements:
 * 2*ceil(rows/256) * 2*ceil(K/256) * 512 (row blocks of 128, their count
 * rounded up to even so a 256-row tile never reads past the end).
 */
size_t mxfp4_scale_relayout_size(int rows, int K);

/*
 * Relayout of E8M0 scales (page section "Data layouts", subsection
 * "A_scale / B_scale": one scale per 32 K, padded with 0x7F = 1.0) from
 * row-major [rows, K/32] (row stride ld_src bytes) into the tcgen05
 * block-scale layout the GEMM stages into tensor memory: 512-byte atoms of
 * 128 rows x 4 scale blocks, atom (rb, g) at byte (rb * 2*ceil(K/256) + g)*512,
 * and inside an atom row r = 32*j + i, block b at byte 16*i + 4*j + b.
 * Rows >= rows and blocks >= K/32 are filled with 0x7F.
 * dst: device, mxfp4_scale_relayout_size(rows, K) bytes, 16-byte aligned.
 * Use it to prepack weight scales once for mxfp4_gemm_prepacked.
 */
int mxfp4_scale_relayout(void *dst, const void *src, int rows, int K, int64_t ld_src,
                         void *stream);

/*
 * mxfp4_scale_relayout of both operands' scales (the same K) in one launch:
 * src_a [rows_a, ld_a] -> dst_a and src_b [rows_b, ld_b] -> dst_b, each dst
 * mxfp4_scale_relayout_size(rows, K) bytes, 16-byte aligned, not overlapping.
 * Same layout, fill and errors as mxfp4_scale_relayout; mxfp4_gemm uses it
 * for its relayout pass.
 */
int mxfp4_scale_relayout2(void *dst_a, const void *src_a, int rows_a, int64_t ld_a, void *dst_b,
                          const void *src_b, int rows_b, int64_t ld_b, int K, void *stream);

/*
 * The GEMM (page formula; section "Kernel ABI" for the argument set).
 *   D       bf16 [M, ldd]           output; ldd >= N
 *   C       bf16 [M, ldc] or NULL   read only when beta != 0; may alias D
 *                                   only with ldc == ldd
 *   A       uint8 [M, lda/2]        lda >= K, lda % 32 == 0 (16-byte rows)
 *   B       uint8 [N, ldb/2]        ldb >= K, ldb % 32 == 0
 *   scaleA  uint8 [M, ld_sa]        ld_sa >= K/32
 *   scaleB  uint8 [N, ld_sb]        ld_sb >= K/32
 *   M, N >= 1; K >= 32, K % 32 == 0 (the scale block).  A, B 16-byte aligned.
 *   split_k  0 = heuristic, else 1..16.  Each split parks an fp32 partial
 *            tile in the workspace; the CTA that finishes a tile last sums
 *            its partials in split order 0, 1, ... (whichever split finished
 *            last), so results are bitwise reproducible run to run.
 *   workspace  device, >= mxfp4_gemm_workspace_size(M, N, K, split_k) bytes,
 *              256-byte aligned, contents need not be initialised (counters
 *              carry a per-call tag and are reset by the call that completes
 *              them); NULL when that size is 0.  Calls that may run at the
 *              same time need workspaces of their own.  After a call stopped
 *              on MXFP4_ERR_TIMEOUT, re-capture graphs that hold split-K
 *              calls on the same workspace (a replay repeats the tag).
 * The scales are read row-major.  Compute-bound shapes (plan.relayout_pass)
 * first relay them out into the workspace with the relayout kernel; the
 * others build the tcgen05 scale layout inside the GEMM itself.
 * Every kernel of the call is launched as a programmatic dependent of the work on
 * `stream`: it may start while that work drains (its set-up overlaps the
 * other kernel's tail) and waits for it in-kernel before reading any input or
 * writing any output, so ordering on the stream is as for plain launches.
 */
int mxfp4_gemm(void *D, int64_t ldd, const void *C, int64_t ldc,
               const void *A, int64_t lda, const void *B, int64_t ldb,
               const void *scaleA, int64_t ld_sa, const void *scaleB, int64_t ld_sb,
               float alpha, float beta, int M, int N, int K, int split_k,
               void *workspace, size_t workspace_bytes, void *stream);

/*
 * mxfp4_gemm with flags.  MXFP4_FLAG_B_STATIC: the caller guarantees that the
 * work enqueued on `stream` before this call does not write B or scaleB (for
 * example weights that stay fixed across a decode loop).  The GEMM then
 * starts copying B and scaleB into its pipeline before waiting for that
 * work, so the weight stream of one call can start before the kernel ahead
 * of it has finished; A, C and D are still touched only after that work has
 * finished.
 * The flag has no effect on plans with a relayout pass (their B scales come
 * from this call's own relayout).  Other arguments and results as for
 * mxfp4_gemm (bit-identical output); unknown flag bits: MXFP4_ERR_INVALID_ARG.
 */
#define MXFP4_FLAG_B_STATIC 1u

int mxfp4_gemm_ex(void *D, int64_t ldd, const void *C, int64_t ldc,
                  const void *A, int64_t lda, const void *B, int64_t ldb,
                  const void *scaleA, int64_t ld_sa, const void *scaleB, int64_t ld_sb,
                  float alpha, float beta, int M, int N, int K, int split_k, unsigned flags,
                  void *workspace, size_t workspace_bytes, void *stream);

/*
 * MXFP8 / MXFP6 form of mxfp4_gemm: D[M,N] = alpha * A[M,K] . B[N,K]^T +
 * beta * C[M,N] with 8-bit, 6-bit or padded 4-bit elements (one byte of
 * footprint each), one E8M0 scale per 32 K as for
 * MXFP4 (page "CDNA4 dense MFMA builtins", section "FP8 and BF8 matrix
 * inputs": FP8 = E4M3, BF8 = E5M2; section "Mixed-precision with scaling":
 * also FP6 = E2M3 or E3M2, scaled per block, A and B formats chosen
 * independently).  Encodings: the OCP formats (E4M3: bias 7, no infinity,
 * NaN = S.1111.111, largest 448; E5M2: bias 15, IEEE-style infinities and
 * NaNs, largest 57344; E2M3: bias 1, largest 7.5; E3M2: bias 3, largest 28;
 * the 6-bit formats have no infinity or NaN).
 *   A: uint8 [M, lda] device, lda >= K elements (= bytes), lda % 16 == 0,
 *      16-byte aligned; B likewise [N, ldb].  8-bit formats: one code per
 *      byte.  6-bit formats: the layout the tensor cores read -- every 16
 *      consecutive elements of a row take 16 bytes, their codes packed
 *      little-endian into the first 12 (element i of the group in bits
 *      6i .. 6i+5, sign in the top bit of each code) and 4 padding bytes
 *      that are not read.  MXFP4_E2M1_PADDED: E2M1 (the MXFP4 element) in
 *      the same kind of layout, so that it mixes with the formats above --
 *      every 16 elements take 16 bytes, the first 8 holding two codes each
 *      (element 2i of the group in the low nibble of byte i, as in packed
 *      MXFP4 rows) and 8 padding bytes that are not read.  Either way one
 *      byte per element of footprint.
 *   fmt_a, fmt_b: MXFP8_E4M3, MXFP8_E5M2, MXFP6_E2M3, MXFP6_E3M2 or
 *      MXFP4_E2M1_PADDED (each value is the format's code in the
 *      kind::mxf8f6f4 instruction).  For E2M1 x E2M1 with packed rows,
 *      mxfp4_gemm is the faster path (kind::mxf4, twice the rate).
 *   Scales, C, D, alpha, beta, split_k, workspace, stream: as for
 *   mxfp4_gemm (mxfp8_gemm_workspace_size gives the workspace).
 * Runs the one-tile tcgen05 kernel (kind::mxf8f6f4, K = 32 per MMA; FP6 at
 * the FP8 rate) with the same tile / split-K / swap-AB plan as an MXFP4 GEMM
 * whose rows hold as many bytes (mxfp8_plan_gemm reports it; tile_k there
 * counts elements).
 * Errors: as for mxfp4_gemm, plus MXFP4_ERR_INVALID_ARG for a bad format.
 */
enum { MXFP8_E4M3 = 0, MXFP8_E5M2 = 1, MXFP6_E2M3 = 3, MXFP6_E3M2 = 4, MXFP4_E2M1_PADDED = 5 };
int mxfp8_gemm(void *D, int64_t ldd, const void *C, int64_t ldc,
               const void *A, int64_t lda, const void *B, int64_t ldb,
               const void *scaleA, int64_t ld_sa, const void *scaleB, int64_t ld_sb,
               int fmt_a, int fmt_b, float alpha, float beta, int M, int N, int K, int split_k,
               void *workspace, size_t workspace_bytes, void *stream);
int mxfp8_plan_gemm(int M, int N, int K, int split_k, int num_sms, mxfp4_plan *out);
size_t mxfp8_gemm_workspace_size(int M, int N, int K, int split_k);

/*
 * mxfp8_gemm on scales already relaid by mxfp4_scale_relayout(dst, src, rows,
 * K, ...) with this call's K (the relaid layout depends only on rows and the
 * number of 32-K blocks, not on the element format), e.g. weights prepared
 * once.  Arguments as mxfp8_gemm without the scale strides; workspace:
 * mxfp8_gemm_prepacked_workspace_size.
 */
int mxfp8_gemm_prepacked(void *D, int64_t ldd, const void *C, int64_t ldc,
                         const void *A, int64_t lda, const void *B, int64_t ldb,
                         const void *scaleA_relaid, const void *scaleB_relaid,
                         int fmt_a, int fmt_b, float alpha, float beta, int M, int N, int K,
                         int split_k, void *workspace, size_t workspace_bytes, void *stream);
size_t mxfp8_gemm_prepacked_workspace_size(int M, int N, int K, int split_k);

/*
 * NVFP4 form of the GEMM: the pages describe no such format (they cover
 * E8M0 block scales only); it is the other block-scaled FP4 variant of the
 * same tensor-core instruction family.  A and B are packed E2M1 exactly as
 * for mxfp4_gemm; each row of A and B carries one scale per 16 consecutive K
 * elements instead of 32, stored as an unsigned E4M3 byte (UE4M3:
 * (1 + m/8) * 2^(e-7), exponent field 0 subnormal (m/8) * 2^-6, 0x7F NaN;
 * bit 7 must be 0 -- such bytes are not checked and give undefined
 * results).  scaleA: [M, ld_sa] bytes, ld_sa >= K / 16; scaleB likewise.
 * A per-tensor scale, where the caller has one, folds into alpha.
 *
 *   D = alpha * (A . B^T) + beta * C, one bf16 rounding, as mxfp4_gemm.
 *
 * Skinny shapes (M <= 64 and N > M) whose scale rows are 16-byte aligned
 * (scaleA, scaleB, ld_sa, ld_sb) run the one-tile kernel with mxfp4_gemm's
 * plan (swap-AB, split-K inside the launch) and leave the workspace
 * untouched (it may be NULL).  Every other call relays the scales into
 * `workspace` (>= nvfp4_gemm_workspace_size(M, N, K) bytes, 256-byte
 * aligned, owned by the caller, free again once the call's work on `stream`
 * has finished) and runs the CTA-pair kernel (256 x 256 tiles).  K % 32 == 0
 * and the 16-byte rules of mxfp4_gemm apply.  Errors as mxfp4_gemm.
 */
int nvfp4_gemm(void *D, int64_t ldd, const void *C, int64_t ldc,
               const void *A, int64_t lda, const void *B, int64_t ldb,
               const void *scaleA, int64_t ld_sa, const void *scaleB, int64_t ld_sb,
               float alpha, float beta, int M, int N, int K,
               void *workspace, size_t workspace_bytes, void *stream);
size_t nvfp4_gemm_workspace_size(int M, int N, int K);

/*
 * As mxfp4_gemm, with both scale buffers already in the relaid layout
 * produced by mxfp4_scale_relayout (scaleA for M rows, scaleB for N rows, at
 * the same K); the GEMM then copies whole scale atoms with bulk copies.  The
 * workspace holds the split-K partials: mxfp4_gemm_prepacked_workspace_size
 * bytes (plan.workspace_bytes).
 */
int mxfp4_gemm_prepacked(void *D, int64_t ldd, const void *C, int64_t ldc,
                         const void *A, int64_t lda, const void *B, int64_t ldb,
                         const void *scaleA_relaid, const void *scaleB_relaid,
                         float alpha, float beta, int M, int N, int K, int split_k,
                         void *workspace, size_t workspace_bytes, void *stream);

size_t mxfp4_gemm_prepacked_workspace_size(int M, int N, int K, int split_k);

/*
 * End-to-end call on HOST buffers: copies A, B, scaleA, scaleB (and C when
 * beta != 0) from host memory into `device_arena`, runs mxfp4_gemm there and
 * copies D back to host memory.  For M >= 2048 the work goes in blocks so
 * the copies overlap the compute: the rows in eight panels (multiples of 256
 * rows) and, when N >= 2048 too, the columns in two halves (a multiple of 256
 * columns each).  On an internal copy stream: the first column block of B
 * and its scales, then each panel's A, scales and C rows, then the rest of
 * B.  The block GEMMs run on `stream`, first column block first; each block
 * of D returns on a second internal copy stream while the next computes.  The
 * internal streams start after the work already enqueued on `stream`, and
 * `stream` waits for the last copy of D, so the call is ordered on `stream`
 * as a whole (pinned host memory makes the copies asynchronous).  Host
 * arrays are dense (ld = K for A/B, K/32 for scales, N for C/D).  The call
 * returns after enqueueing; synchronise `stream` before reading D_host.
 * device_arena: >= mxfp4_gemm_host_arena_size(M, N, K, split_k, beta != 0)
 * bytes of device memory, 256-byte aligned, owned by the caller.
 */
int mxfp4_gemm_host(void *D_host, const void *C_host, const void *A_host, const void *B_host,
                    const void *scaleA_host, const void *scaleB_host,
                    float alpha, float beta, int M, int N, int K, int split_k,
                    void *device_arena, size_t arena_bytes, void *stream);

size_t mxfp4_gemm_host_arena_size(int M, int N, int K, int split_k, int with_c);

/*
 * mxfp4_gemm_host for the operand forms of mxfp8_gemm: the same pipelined
 * copies and blocks, with A [M, K] and B [N, K] host arrays of one byte per
 * element (fmt_a / fmt_b as for mxfp8_gemm: MXFP8_E4M3, MXFP8_E5M2,
 * MXFP6_E2M3, MXFP6_E3M2, MXFP4_E2M1_PADDED) and each block computed by
 * mxfp8_gemm.  device_arena: >= mxfp8_gemm_host_arena_size(M, N, K, split_k,
 * beta != 0) bytes, 256-byte aligned.  Errors: as mxfp4_gemm_host, plus
 * MXFP4_ERR_INVALID_ARG for a bad format.
 */
int mxfp8_gemm_host(void *D_host, const void *C_host, const void *A_host, const void *B_host,
                    const void *scaleA_host, const void *scaleB_host, int fmt_a, int fmt_b,
                    float alpha, float beta, int M, int N, int K, int split_k,
                    void *device_arena, size_t arena_bytes, void *stream);

size_t mxfp8_gemm_host_arena_size(int M, int N, int K, int split_k, int with_c);

/*
 * mxfp4_gemm for callers that cannot allocate device memory (the page has no
 * counterpart: it exists for users whose allocator is owned by someone else
 * or who may not synchronise the device through a cudaMalloc mid-run).  Same
 * arguments and results as mxfp4_gemm minus the workspace: the scratch (relaid
 * scales, split-K tile counters and partials) lives in one array of
 * MXFP4_NOALLOC_SCRATCH_BYTES inside the library's device image, held by
 * every GPU that loads the library until exit.  Shapes whose
 * mxfp4_gemm_workspace_size exceeds it are rejected with MXFP4_ERR_WORKSPACE
 * before anything is enqueued.  `stream` must belong to the current device
 * (MXFP4_ERR_INVALID_ARG otherwise), whose copy of the array is used.  The
 * first call on a device looks up the array's device address (a runtime
 * query); make that first call before capturing the stream into a graph.  All
 * calls share the array: calls that overlap on the GPU race on it and must be
 * serialised by the caller.  Nothing needs clearing between calls: each call
 * rewrites the relaid scales and partials before it reads them, and the tile
 * counters carry a per-call tag, so a counter left by an earlier call reads as
 * zero.
 */
#define MXFP4_NOALLOC_SCRATCH_BYTES (32u << 20)

int mxfp4_gemm_noalloc(void *D, int64_t ldd, const void *C, int64_t ldc,
                       const void *A, int64_t lda, const void *B, int64_t ldb,
                       const void *scaleA, int64_t ld_sa, const void *scaleB, int64_t ld_sb,
                       float alpha, float beta, int M, int N, int K, int split_k, void *stream);

/*
 * Read the device status word that bounded waits write on timeout into
 * *status (MXFP4_OK or MXFP4_ERR_TIMEOUT); if reset != 0 clear it.
 * Synchronous (it copies one int from the device).
 */
int mxfp4_device_status(int *status, int reset);

/*
 * Test hook for the bounded waits: launches one CTA that waits on an
 * mbarrier nothing ever arrives at, with a limit of `limit_cycles` SM clock
 * cycles, through the same wait routine the GEMM uses.  The wait runs out,
 * records MXFP4_ERR_TIMEOUT in the device status word and the kernel
 * returns.  The page has no counterpart: this exists so tests can show a
 * stuck wait ends cleanly without faulting the GPU.
 */
int mxfp4_wait_timeout_probe(long long limit_cycles, void *stream);

/*
 * MXFP4 quantiser: bf16 rows -> the operand format mxfp4_gemm takes.
 *   X  bf16 [rows, ldx]     input, ldx >= K elements, ldx % 8 == 0, 16-byte aligned
 *   Q  uint8 [rows, ldq/2]  output codes, packed two per byte (element 2i in the
 *                           low nibble); ldq >= K counted in fp4 elements like
 *                           lda, ldq % 32 == 0, 16-byte aligned
 *   S  uint8 [rows, lds]    output E8M0 scale codes, one per 1x32 block, lds >= K/32
 * Per block: s = floor(log2(amax / 6)) (the largest integer with
 * 6 * 2^s <= amax; 0 for an all-zero block), clamped to [-127, 127], scale code
 * s + 127; each element is x / 2^s rounded to the nearest E2M1 value (ties to
 * even, saturating at +-6) with the sign of x (so small negatives give -0).
 * This is the quantisation rule the benchmark workloads' operands follow; the
 * asm_f4gemm page lists operand generation among its reference helpers
 * (section "Files") without stating it.  Inputs must be finite.  rows >= 1,
 * K >= 32, K % 32 == 0.  Errors: MXFP4_ERR_INVALID_ARG (null pointer, sizes,
 * strides), MXFP4_ERR_MISALIGNED, device errors.  Enqueued on `stream`.
 */
int mxfp4_quantize(void *Q, int64_t ldq, void *S, int64_t lds, const void *X, int64_t ldx,
                   int rows, int K, void *stream);

/*
 * MXFP8 quantiser: bf16 rows -> the operand format mxfp8_gemm takes.
 *   X  bf16 [rows, ldx]   input, ldx >= K, ldx % 8 == 0, 16-byte aligned
 *   Q  uint8 [rows, ldq]  output codes in mxfp8_gemm's operand form for
 *                         fmt: one per byte (MXFP8_E4M3 / MXFP8_E5M2), or
 *                         the padded 16-per-16-bytes forms (MXFP6_E2M3 /
 *                         MXFP6_E3M2 / MXFP4_E2M1_PADDED, padding written as
 *                         zeros), ldq >= K, ldq % 16 == 0, 16-byte aligned
 *   S  uint8 [rows, lds]  output E8M0 scale codes, one per 1x32 block
 * Per block: s = floor(log2 amax) - emax, with emax the exponent of the
 * format's largest binade (8 for E4M3, 15 for E5M2, 2 for E2M3 and E2M1, 4
 * for E3M2: the OCP MX scale rule); 0 for an all-zero block; clamped to
 * [-127, 127]; scale code s + 127.  Each element is x / 2^s rounded to the
 * nearest finite value of the format (ties to even, saturating at 448 /
 * 57344 / 7.5 / 28 / 6) with the sign of x.  Inputs must
 * be finite.  rows >= 1, K >= 32, K % 32 == 0.  Errors: MXFP4_ERR_INVALID_ARG
 * (null pointer, sizes, strides, format), MXFP4_ERR_MISALIGNED, device
 * errors.  Enqueued on `stream`.
 */
int mxfp8_quantize(void *Q, int64_t ldq, void *S, int64_t lds, const void *X, int64_t ldx,
                   int rows, int K, int fmt, void *stream);

/* Set the in-kernel wait limit in SM clock cycles (default 2^32, ~2 s). */
void mxfp4_set_wait_limit(long long cycles);

/* Human-readable name of a status code (never NULL). */
const char *mxfp4_strerror(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
int mxfp4_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MXFP4_GEMM_H */
