/*
 * tg.h -- C ABI of the GB300 (sm_103a) TMA-fed bf16 GEMM and TMA tile-copy library.
 *
 * Sources for the operations (page title, section):
 *  [GEMM]  "GEMM: la moltiplicazione di matrici sull'hardware": section "Il conto, e il
 *          problema della versione ingenua" (C_ij = sum_k A_ik B_kj, 2MNK flops) and
 *          section "I tensor core" (C <- alpha*A*B + beta*C, 16-bit inputs with a 32-bit
 *          accumulator); section "In pratica" (16-byte alignment of the leading
 *          dimension, wave quantisation).
 *  [TMA]   "2 . Le Tensor Memory Accelerator": 2.2 (the 128-byte CUtensorMap descriptor,
 *          up to 5 dimensions, one thread issues a copy by coordinates), 2.3 (descriptor
 *          rules: 16-byte base, 16-byte-multiple strides, 128-byte shared destination,
 *          swizzle limits the box width; a violation yields silent wrong data), 2.5
 *          (out-of-bounds fill, TMA store for the epilogue, cluster multicast).
 *  [MAP]   "H100 . cuTensorMap (TMA descriptor)": 8 (rank, 16-byte global address,
 *          dims up to 2^32, strides in bytes, innermost stride implicit), 9 (boxDim,
 *          elementStrides non-zero and <= 8; innermost box extent <= swizzle size),
 *          11 (swizzle), 14 (OOB fill in shared memory: zero or NaN).
 *  [PIPE]  "1 . Asynchronisme et mbarrier": 1.4-1.5 (mbarrier with transaction bytes
 *          and a phase bit; the full/empty stage ring).
 *
 * Conventions shared by every entry point
 *  - Ownership: the caller owns every buffer.  Device pointers come from any CUDA
 *    allocator (a Python caller gets them from torch).  The library allocates nothing
 *    per call; on first use of a device it allocates one 16-byte device status word for
 *    that device, and on the first stream-K GEMM issued on a stream it allocates that
 *    stream's workspace (128 KiB per SM of fp32 partials plus one flag per SM; up to 16
 *    streams per device, beyond which GEMMs on further streams run data-parallel).  All
 *    are kept until process exit.  GEMMs on one stream are ordered, so they never share
 *    partials in flight.
 *  - Asynchrony: GPU work is enqueued on `stream` (0 = legacy default stream) and the
 *    call returns at once.  GEMM and tile-copy kernels are launched with programmatic
 *    stream serialisation: their start-up may overlap the end of the kernel before them
 *    on the stream, but they touch no global memory before that kernel has completed, so
 *    stream order holds as for any launch.  Every error the host can detect is returned
 *    synchronously, before anything is launched.  Errors found on the device (a pipeline wait that
 *    exceeded its time limit) are latched in the device status word and reported by
 *    tg_status_sync().
 *  - Errors: no entry point falls back to another implementation; each rule of the
 *    pages that the hardware would otherwise violate silently has its own status code.
 *  - Thread safety: calls may be made from several host threads; calls that share a
 *    device share its status word.
 *  - Memory: every buffer a kernel reads or writes (GEMM operands and C, copy tensors and
 *    images, the probe's timing words) must be device memory of the device that is
 *    current when the call is made.  Host memory (pinned or not), managed memory and
 *    another GPU's memory are refused with TG_ERR_INVALID_VALUE before anything is
 *    encoded or launched (checked with cudaPointerGetAttributes after the rules below),
 *    so no tensor map ever covers memory other than this GPU's own.
 */
#ifndef TG_H_
#define TG_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h> /* cudaStream_t */

#ifdef __cplusplus
extern "C" {
#endif

typedef enum tg_status {
    TG_OK = 0,
    TG_ERR_INVALID_VALUE = 1,    /* a size, enum or pointer argument is out of range      */
    TG_ERR_MISALIGNED = 2,       /* a base address, stride or box width breaks the 16-byte
                                    rules of [TMA] 2.3 / [MAP] 8                          */
    TG_ERR_UNSUPPORTED = 3,      /* valid per the pages but not provided by this library   */
    TG_ERR_BUFFER_TOO_SMALL = 4, /* the output buffer cannot hold the result               */
    TG_ERR_CUDA = 5,             /* a CUDA runtime/driver call failed                      */
    TG_ERR_NO_DRIVER_SYMBOL = 6, /* the driver does not export cuTensorMapEncodeTiled      */
    TG_ERR_DEVICE_TIMEOUT = 7    /* a device-side pipeline wait exceeded its time limit    */
} tg_status;

/* Human-readable name of a status code (static storage; never NULL). */
const char *tg_status_string(tg_status status);

/* Synchronises `stream`, then returns and clears the status latched on the current
 * device by kernels of this library (TG_OK if none).  A CUDA error raised while
 * synchronising is returned as TG_ERR_CUDA. */
tg_status tg_status_sync(cudaStream_t stream);

/* Diagnostic: looks a CUDA driver entry point up by name exactly as the library looks up
 * cuTensorMapEncodeTiled before its first tensor map (cudaGetDriverEntryPointByVersion,
 * CUDA 12.0 ABI).  TG_OK when the installed driver exports it, TG_ERR_NO_DRIVER_SYMBOL when
 * it does not (the status every encoding call returns on such a driver), TG_ERR_CUDA when
 * no usable driver can be asked, TG_ERR_INVALID_VALUE for NULL.  Host-only. */
tg_status tg_driver_symbol_status(const char *symbol);

/* Raw 32-bit status word last returned by tg_status_sync on this thread: the low byte
 * is the tg_status code; for TG_ERR_DEVICE_TIMEOUT, bits 8-11 name the role that gave
 * up (1 producer, 2 MMA issuer, 3 epilogue, 4 copy engine) and bits 16-31 the block. */
uint32_t tg_status_detail(void);

/* ------------------------------------------------------------------------------------
 * GEMM:  C <- alpha * A * B + beta * C    [GEMM] "I tensor core"
 *
 *  A: M x K bf16.  K-major (default): element (i,k) at A[i*lda + k], lda >= K;
 *     M-major (layout bit 0): element (i,k) at A[k*lda + i], lda >= M.
 *  B: the K x N operand.  K-major (default): stored as an N x K row-major array,
 *     element (k,j) at B[j*ldb + k], ldb >= K; N-major (layout bit 1): stored as a K x N
 *     row-major array, element (k,j) at B[k*ldb + j], ldb >= N.
 *  C: M x N row-major, element (i,j) at C[i*ldc + j], fp32, bf16 or fp16 (layout bits
 *     2-3), ldc >= N; read only when beta != 0 (so NaNs in C do not propagate when
 *     beta == 0).
 *  A and B hold bf16 (default), fp16, E4M3, E5M2 or tf32 values (layout bits 4-6).  The
 *  pages name 16-bit inputs and shorter ones such as FP8 as the tensor cores' formats
 *  ([GEMM] "In pratica: forme tonde e mezza precisione"), and tf32 as a third path:
 *  float32 inputs truncated to 10 mantissa bits ([GEMM] "I tensor core").  E4M3 is the
 *  variant without infinities (S.1111.111 is NaN); E5M2 has IEEE-style infinities and
 *  NaNs; both are passed as bytes, one element per byte.  tf32 operands are passed as
 *  ordinary binary32 arrays; only their top 19 bits take part.  8-bit and tf32 operands
 *  are K-major only.  Products are formed from the inputs and accumulated in fp32;
 *  alpha*acc + beta*C is computed in fp32 and rounded to nearest-even for a bf16 or
 *  fp16 C.
 *
 *  layout: bit 0 = A is M-major, bit 1 = B is N-major (each operand is staged by TMA in
 *          its own storage order and read by the tensor core through the matching
 *          shared-memory descriptor; no transposed copy is made),
 *          bits 2-3 = C element type (TG_C_F32, TG_C_BF16 or TG_C_F16),
 *          bits 4-6 = A and B element type (TG_IN_BF16, TG_IN_F16, TG_IN_E4M3,
 *          TG_IN_E5M2 or TG_IN_TF32; the MX types belong to gemm_mx); other bits 0.
 *  Rules (each returns before launch):
 *   M, N, K in [0, 2^31-1]                                   else TG_ERR_INVALID_VALUE
 *   M == 0 or N == 0: nothing to do, TG_OK (pointers are not inspected)
 *   K == 0: C <- beta*C (A and B are not read and may be NULL)
 *   lda, ldb >= their row length (above), ldc >= N; A, B, C non-NULL when read
 *                                                             else TG_ERR_INVALID_VALUE
 *   8-bit or tf32 A and B with bit 0 or bit 1 set            else TG_ERR_UNSUPPORTED
 *   (gemm_bf16_ex) an N-major B with tile_n 224               else TG_ERR_UNSUPPORTED
 *   A, B, C 16-byte aligned; lda, ldb, ldc times their element sizes multiples of 16
 *   (lda, ldb multiples of 8 elements for 16-bit, 16 for 8-bit, 4 for tf32 operands)
 *                                                             else TG_ERR_MISALIGNED
 *   row strides in bytes < 2^40                               else TG_ERR_INVALID_VALUE
 * ---------------------------------------------------------------------------------- */
#define TG_LAYOUT_A_MN_MAJOR 0x1u
#define TG_LAYOUT_B_MN_MAJOR 0x2u
#define TG_C_F32 (0u << 2)
#define TG_C_BF16 (1u << 2)
#define TG_C_F16 (2u << 2)
#define TG_IN_BF16 (0u << 4)
#define TG_IN_F16 (1u << 4)
#define TG_IN_E4M3 (2u << 4)
#define TG_IN_E5M2 (3u << 4)
#define TG_IN_TF32 (4u << 4)
#define TG_IN_MXE4M3 (5u << 4) /* gemm_mx only: E4M3 elements with E8M0 block scales */
#define TG_IN_MXE5M2 (6u << 4) /* gemm_mx only: E5M2 elements with E8M0 block scales */

tg_status gemm_bf16(int64_t M, int64_t N, int64_t K,
                    const void *A, int64_t lda,
                    const void *B, int64_t ldb,
                    void *C, int64_t ldc,
                    float alpha, float beta,
                    uint32_t layout, cudaStream_t stream);

/* Tuning knobs of the GEMM kernel ([PIPE] 1.3 "Combien d'étages ?": sweep the stage
 * count; [TMA] 2.5 multicast).  Zero in any field selects the default; for stages,
 * cluster, tile_n and mma the default is chosen per problem (the launch is reported by
 * tg_gemm_last_plan). */
typedef struct tg_gemm_config {
    uint32_t stages;     /* smem ring depth, 2..6 (limited by shared memory per tile);
                            0 = 6 for CTA pairs whose k-loop has at least 32 k-blocks
                            (the epilogue then keeps 2 staging buffers per warp), else 5;
                            4 or 6 for the per-CTA kernel (tile width 256 / 128)        */
    uint32_t cluster;    /* 1 = one CTA per tile; 2 = CTA pairs along M that load half
                            of the shared B tile each and multicast it to both (with mma
                            1: a single-GPU option, refused with TG_ERR_UNSUPPORTED when
                            the process can see more than one device); 4 = two CTA pairs
                            (mma 3, same single-GPU rule)                                 */
    uint32_t tile_n;     /* output tile width per CTA: 128 or 256 (tile height is 128);
                            224 with mma 2: a 256 x 224 pair tile, which divides widths of
                            a multiple of 4096 into a number of tiles that fills the SMs
                            more evenly (4096 / 224 -> 19 columns, x 4 rows = 76 pairs)    */
    uint32_t group_m;    /* rasterisation: tiles walk down groups of this many M tiles  */
    uint32_t max_ctas;   /* cap on persistent CTAs (0 = as many as fit, one per SM)     */
    uint32_t flags;      /* TG_GEMM_FLAG_* */
    uint64_t timeout_ns; /* device-side limit of every pipeline wait (default 1 s)      */
    uint32_t mma;        /* 1 = each CTA issues its own 128 x tile_n MMAs; 2 = a cluster of
                            two CTAs issues 256 x tile_n pair MMAs (tcgen05 cta_group::2),
                            each CTA staging half of the B tile (needs cluster 2); 3 = a
                            cluster of four CTAs holding two such pairs stacked along M,
                            each CTA loading a quarter of the shared B tile and multicasting
                            it to the same-parity CTA of the other pair (cluster 4; 16-bit
                            K-major operands, whole tiles, no dynamic schedule; a single-GPU
                            option like the B multicast of mma 1).  0 with cluster 0 = auto:
                            the pair, or mma 3 when A's or B's rows are not 128-byte
                            multiples (their TMA rows then straddle two L2 lines and the
                            shared B cuts the L2 requests per k-block by 23 %), M >= 512,
                            16-bit K-major operands and one visible device.  The automatic
                            choice depends on the strides, which tg_gemm_plan_for takes as
                            tightly packed: tg_gemm_plan_ld takes them, and tg_gemm_last_plan
                            reports the launch made.                                      */
    uint32_t schedule;   /* 0 = auto; 1 = data-parallel (whole tiles strided over the
                            persistent clusters; a last wave at most half full runs as
                            half-width tiles, TG_GEMM_FLAG_NO_SPLIT_TAIL); 2 = stream-K hybrid where the problem
                            allows it: whole tiles for all but the last full wave, then
                            the k-blocks of the remaining tiles split evenly over all
                            clusters, partial sums combined in fp32 ("GEMM: la
                            moltiplicazione ..." "In pratica": wave quantisation).  Auto
                            picks stream-K when there is at least one full wave and whole
                            tiles would leave more than 5 % of the cluster-waves idle;
                            3 = dynamic: one cluster per tile is launched, and a running
                            cluster takes over the tiles of clusters it cancels before
                            they start (cluster launch control), so clusters that finish
                            early, or start late because other kernels hold SMs, balance
                            out; needs max_ctas 0.  Never chosen by auto.                */
    uint32_t epi_bufs;   /* staging buffers per epilogue warp: 0 = 4 when they fit next
                            to the ring, else 2; or exactly 2 or 4                        */
    uint32_t reserved;   /* must be 0 */
    void *workspace;     /* NULL, or caller-owned device memory (16-byte aligned) that a
                            stream-K launch uses for its fp32 partials instead of the
                            library's per-stream workspace: tg_gemm_plan.workspace_bytes
                            bytes, zero-filled by the caller once before its first use and
                            never touched by the caller afterwards (the library keeps it
                            valid for the next launch).  GEMMs that may run at the same
                            time must not share one.                                      */
    uint64_t workspace_bytes; /* its size; 0 with a NULL workspace                        */
} tg_gemm_config;

/* Test hook: the producers of the first cluster (its one or two CTAs) issue no copies at
 * all, so the MMA issuer's first wait must run out and report TG_ERR_DEVICE_TIMEOUT while
 * no copy is in flight in that cluster.  Honoured by every kernel; other clusters of the
 * launch stop at their next wait and drain the copies they have in flight. */
#define TG_GEMM_FLAG_TEST_SKIP_FIRST_LOAD 0x1u

/* Split tail (data-parallel schedule, on by default): when the tiles left for a last wave
 * would occupy at most half of the persistent CTA pairs, each of them is computed as two
 * half-width tiles (256 x 128 pair MMAs), so that the last wave takes about half as long
 * ("GEMM: la moltiplicazione ...", "In pratica": wave quantisation; here the tile size
 * is chosen per tile rather than per launch).  Applies to CTA-pair launches with 256-wide
 * tiles and B read K-major; this flag turns it off. */
#define TG_GEMM_FLAG_NO_SPLIT_TAIL 0x2u

/* Fills *cfg with the defaults used by gemm_bf16: 0 (chosen per problem) in stages,
 * cluster, tile_n and mma; group_m 16; a 1 s wait limit; everything else 0. */
void tg_gemm_config_default(tg_gemm_config *cfg);

/* gemm_bf16 with explicit tuning knobs (cfg may be NULL = defaults).  Additional
 * rules: stages in {0, 2..6}, cluster in {0, 1, 2}, tile_n in {0, 128, 224, 256} (224 only
 * with mma 2), mma in
 * {0, 1, 2}, mma 2 with cluster 1, schedule > 3, schedule 3 with max_ctas != 0, epi_bufs
 * not in {0, 2, 4}, reserved != 0, a workspace without a size or a size without a
 * workspace, else TG_ERR_INVALID_VALUE; a workspace not 16-byte aligned ->
 * TG_ERR_MISALIGNED; a stream-K launch whose workspace is smaller than the plan's
 * workspace_bytes -> TG_ERR_BUFFER_TOO_SMALL; a
 * combination whose ring does not fit in shared memory returns TG_ERR_UNSUPPORTED, and so
 * does the B multicast (cluster 2 with mma 1, or mma 3) when more than one device is
 * visible; mma 3 with 8-bit or tf32 operands or an N-major B -> TG_ERR_UNSUPPORTED.
 *
 * Stream-K workspace without a caller-owned one: the library allocates one per (device,
 * stream) on the first stream-K launch on that stream (streams are told apart by
 * cudaStreamGetId, so every host thread's per-thread default stream has its own), clears
 * its flags with a memset enqueued on that stream, and keeps it until exit.  It never
 * synchronises the device.  A launch that cannot have one -- the stream is being
 * captured (pass a caller-owned workspace to capture stream-K launches), 16 streams of
 * this device already hold one, or the allocation failed -- runs with whole tiles
 * instead; tg_gemm_last_plan reports which.  The first call on a device allocates the
 * 16-byte status word: make it before any stream capture begins. */
tg_status gemm_bf16_ex(int64_t M, int64_t N, int64_t K,
                       const void *A, int64_t lda,
                       const void *B, int64_t ldb,
                       void *C, int64_t ldc,
                       float alpha, float beta,
                       uint32_t layout, const tg_gemm_config *cfg,
                       cudaStream_t stream);

/* gemm_bf16 for callers that cannot allocate device memory.  The paper has no
 * counterpart to this entry point; it exists for callers such as code running while a
 * CUDA stream is being captured (where cudaMalloc is not permitted), code whose device
 * memory is owned entirely by another allocator or a fixed budget, and code that must
 * not make the implicitly synchronising allocation calls.  gemm_bf16 allocates its
 * 16-byte status word with cudaMalloc on the first call on a device; this variant calls
 * no cudaMalloc, cudaFree or allocating library routine at any time.
 *
 * Same arguments, rules and result as gemm_bf16 (default tuning), plus:
 *  status_out  NULL, or device memory / page-locked host memory that receives,
 *              asynchronously on `stream` after the kernel, the kernel's 32-bit status
 *              word (0 = OK; otherwise the layout described at tg_status_detail).  It is
 *              written only when a kernel is launched (not for M == 0 or N == 0 or when
 *              an error is returned).  tg_status_sync does not see this variant's errors.
 *  Scratch     the kernel's status words live in a 256-byte file-scope array inside the
 *              library's device image (every GPU that loads the library holds it until
 *              the process exits).  A call needs 8 bytes of it whatever M, N and K are;
 *              a call needing more than the 256 bytes would return TG_ERR_UNSUPPORTED.
 *              Each call clears the words it uses (cudaMemsetAsync on `stream`) before
 *              its kernel.  Every call shares the array: calls whose work overlaps on the
 *              GPU (different streams, or different host threads, on one device) race
 *              on it and may report each other's status; serialise them on one stream.
 *  Set-up      the first call on a device looks up that device's address of the array
 *              (cudaGetSymbolAddress, with the device current); make that first call
 *              before any stream capture begins.
 */
tg_status gemm_bf16_noalloc(int64_t M, int64_t N, int64_t K,
                            const void *A, int64_t lda,
                            const void *B, int64_t ldb,
                            void *C, int64_t ldc,
                            float alpha, float beta,
                            uint32_t layout, uint32_t *status_out,
                            cudaStream_t stream);

/* ------------------------------------------------------------------------------------
 * MX (microscaling) GEMM:  C <- alpha * (A . Sa) * (B . Sb) + beta * C
 *
 * The TMA page (2.8, Blackwell) names block-scaled formats among what Blackwell adds; the
 * definition followed is the OCP Microscaling Formats (MX) specification v1.0: blocks of
 * 32 consecutive elements along K share one E8M0 scale X, an unsigned biased exponent
 * worth 2^(X - 127) (X = 255 is NaN), and an element's value is its own value times its
 * block's scale.  The tensor core multiplies such operands directly (tcgen05.mma
 * kind::mxf8f6f4 with block scales), accumulating in fp32.
 *
 *  A, B    as for gemm_bf16 with layout bits 4-6 = TG_IN_MXE4M3 or TG_IN_MXE5M2 (both
 *          operands one type), K-major only (bits 0-1 zero); one byte per element; lda,
 *          ldb multiples of 16.
 *  sfa,sfb E8M0 scale bytes of A (M rows) and of B (N rows), gemm_mx_scale_bytes(M, K)
 *          and gemm_mx_scale_bytes(N, K) bytes, device memory, 16-byte aligned, in 512-byte
 *          atoms: the scale of row r, 32-element block j (j = k / 32) is the byte at
 *            ((j / 4) * RB + r / 128) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + j % 4,
 *          RB = ceil(rows / 128).  (One atom is what the tensor core's scale copy takes in
 *          one instruction.)  Bytes no scale occupies must not be 255: a NaN scale times
 *          an out-of-range element, which reads as zero, is NaN.
 *  C       fp32, bf16 or fp16 (bits 2-3), as for gemm_bf16.
 *  cfg     NULL or: max_ctas, timeout_ns, flags, group_m, schedule 0/1 and no workspace;
 *          the kernel by mma:
 *            0 or 2  CTA pairs with 256 x 256 tiles (the default; cluster 0/2, tile_n
 *                    0/256, stages 0 (= 4) or 2..5), a single 256-column accumulator
 *                    beside the per-stage scale columns in TMEM;
 *            1       one CTA per 128 x 128 tile (cluster 0/1, tile_n 0/128, stages 0
 *                    (= 5) or 2..5), two accumulators;
 *          anything else TG_ERR_INVALID_VALUE.  A ring too deep for shared memory (6
 *          stages) returns TG_ERR_UNSUPPORTED.
 *  Rules: those of gemm_bf16_ex, plus sfa / sfb NULL with K > 0 -> TG_ERR_INVALID_VALUE,
 *  not 16-byte aligned -> TG_ERR_MISALIGNED, not device memory of the current device ->
 *  TG_ERR_INVALID_VALUE; a layout without an MX operand type -> TG_ERR_INVALID_VALUE.
 *  gemm_bf16, gemm_bf16_ex and gemm_bf16_noalloc refuse the MX types (TG_ERR_UNSUPPORTED).
 * ---------------------------------------------------------------------------------- */
tg_status gemm_mx(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *sfa,
                  const void *B, int64_t ldb, const void *sfb, void *C, int64_t ldc, float alpha,
                  float beta, uint32_t layout, const tg_gemm_config *cfg, cudaStream_t stream);

/* Bytes of the scales of an MX operand with `rows` rows and K columns: 512 times the
 * number of (128-row, 128-element) atoms, both counts rounded up (0 if rows or K <= 0). */
size_t gemm_mx_scale_bytes(int64_t rows, int64_t K);

/* Host-only: the launch that gemm_bf16_ex would make for these sizes on `sm_count`
 * SMs (0 = query the current device), for tightly packed operand rows (see
 * tg_gemm_plan_ld for other strides), without validating pointers or launching. */
typedef struct tg_gemm_plan {
    uint32_t tile_m, tile_n, tile_k; /* CTA tile and k-block (elements: 128 bytes deep,
                                        64 16-bit, 128 8-bit or 32 tf32 elements)       */
    uint32_t stages, cluster;
    uint64_t tiles_m, tiles_n;       /* output tiles along M and N                      */
    uint64_t k_blocks;               /* k-blocks per tile                               */
    uint32_t grid;                   /* persistent CTAs launched                        */
    uint32_t smem_bytes;             /* dynamic shared memory per CTA                   */
    uint32_t stage_bytes;            /* bytes one ring stage of one CTA receives by TMA */
    uint32_t mma;                    /* 1 = per-CTA MMA, 2 = CTA-pair MMA               */
    uint32_t dp_units;               /* scheduling units computed whole                 */
    uint64_t sk_iters;               /* stream-K (unit, k-block) iterations; 0 = none   */
    uint32_t split_units;            /* units of the last wave computed as two half-width
                                        tiles each (TG_GEMM_FLAG_NO_SPLIT_TAIL); 0 = none */
    uint64_t workspace_bytes;        /* bytes of a caller-owned workspace this launch needs
                                        (0 when it splits no tile)                        */
    uint32_t workspace;              /* tg_gemm_last_plan: 0 none, 1 the library's
                                        per-stream workspace, 2 the caller's              */
    uint32_t sk_fallback;            /* tg_gemm_last_plan: stream-K was planned but the
                                        launch ran whole tiles because 1 = 16 streams
                                        already hold a workspace, 2 = the stream was being
                                        captured and no caller-owned workspace was given,
                                        3 = allocation failed; 0 = no fallback            */
} tg_gemm_plan;

tg_status tg_gemm_plan_for(int64_t M, int64_t N, int64_t K, uint32_t layout,
                           const tg_gemm_config *cfg, uint32_t sm_count,
                           tg_gemm_plan *plan);

/* tg_gemm_plan_for for given row strides of A and B (in elements, as passed to
 * gemm_bf16_ex): the automatic kernel choice depends on them (cfg.mma); tg_gemm_plan_for
 * is this call with tightly packed rows (lda = K or M, ldb = K or N).  With sm_count 0 the
 * grid is the one the launch uses on the current device (its occupancy query for the
 * chosen cluster size); with sm_count > 0 it assumes every cluster fits and one visible
 * device.  The strides are not otherwise validated here. */
tg_status tg_gemm_plan_ld(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                          uint32_t layout, const tg_gemm_config *cfg, uint32_t sm_count,
                          tg_gemm_plan *plan);

/* The launch that the calling host thread's last successful gemm_bf16 / gemm_bf16_ex
 * call made (zeros before the first): its tiles, grid and schedule as launched, which
 * workspace its stream-K part used and, if stream-K was planned but could not run, why
 * (sk_fallback).  Host-only; plan NULL -> TG_ERR_INVALID_VALUE. */
tg_status tg_gemm_last_plan(tg_gemm_plan *plan);

/* ------------------------------------------------------------------------------------
 * TMA tile copy: the descriptor path on its own   [TMA] 2.2-2.5, [MAP] 8-11, 14
 *
 * For every box (bi, bj) of a 2-D tensor (row-major over the box grid, outer index
 * slowest) one thread issues a TMA load of the box into a 1024-byte-aligned shared
 * memory stage -- with the requested swizzle and out-of-bounds fill -- and the raw
 * stage bytes are then written to out + (bi*nbj + bj) * box_bytes, where
 * box_bytes = box.inner * box.outer * element size.  The output is therefore the exact
 * shared-memory image of every box.
 * ---------------------------------------------------------------------------------- */
typedef enum tg_dtype {
    TG_DTYPE_U8 = 0,   /* 1 byte  */
    TG_DTYPE_BF16 = 1, /* 2 bytes */
    TG_DTYPE_F16 = 2,  /* 2 bytes */
    TG_DTYPE_F32 = 3   /* 4 bytes */
} tg_dtype;

typedef struct tg_tensor2d {
    const void *base;      /* device address of element (0,0); 16-byte aligned          */
    uint32_t dtype;        /* tg_dtype                                                  */
    uint32_t rank;         /* must be 2 (1..5 are valid descriptors; only 2 is provided)*/
    uint64_t dims[2];      /* dims[0] = inner (contiguous) extent, dims[1] = outer      */
    uint64_t stride_bytes; /* bytes between consecutive outer indices; multiple of 16   */
} tg_tensor2d;

typedef struct tg_box {
    uint32_t inner; /* elements along dims[0], 1..256; inner*elem size multiple of 16    */
    uint32_t outer; /* elements along dims[1], 1..256                                    */
} tg_box;

typedef enum tg_swizzle {
    TG_SWZ_NONE = 0,
    TG_SWZ_32B = 1,  /* 16-byte units permuted within 32-byte spans   (a[4]   ^= a[7])   */
    TG_SWZ_64B = 2,  /* ... within 64-byte spans                      (a[5:4] ^= a[8:7]) */
    TG_SWZ_128B = 3  /* ... within 128-byte spans                     (a[6:4] ^= a[9:7]) */
} tg_swizzle;

typedef enum tg_oob {
    TG_OOB_ZERO = 0, /* out-of-bounds elements read as zero                              */
    TG_OOB_NAN = 1   /* out-of-bounds elements read as NaN (floating-point dtypes only)  */
} tg_oob;

/* Host-only checks of the descriptor rules ([TMA] 2.3, [MAP] 8-9), in this order:
 *   tensor/box NULL, rank 0 or > 5, unknown dtype, a dim of 0 or > 2^32, base NULL,
 *   stride < dims[0]*elem or >= 2^40, box extents 0 or > 256, unknown swizzle,
 *   swizzled box inner bytes > swizzle span          -> TG_ERR_INVALID_VALUE
 *   base not 16-byte aligned, stride not a multiple of 16,
 *   box inner bytes not a multiple of 16             -> TG_ERR_MISALIGNED
 *   rank != 2                                        -> TG_ERR_UNSUPPORTED
 * No GPU is touched. */
tg_status tma_validate(const tg_tensor2d *tensor, const tg_box *box, tg_swizzle swizzle);

/* Bytes of the image tma_tile_copy writes (0 if tensor/box are NULL or degenerate). */
size_t tma_tile_copy_image_bytes(const tg_tensor2d *tensor, const tg_box *box);

/* Enqueues the copy on `stream`.  In addition to tma_validate's rules:
 *   out NULL, unknown oob, NaN fill with an integer dtype -> TG_ERR_INVALID_VALUE
 *   out not 16-byte aligned                             -> TG_ERR_MISALIGNED
 *   out_bytes < tma_tile_copy_image_bytes()             -> TG_ERR_BUFFER_TOO_SMALL
 *   box bytes > 65536; a swizzled box whose inner bytes differ from the swizzle span
 *   (the hardware places narrower rows at the span's pitch, so the image would not be
 *   the dense box); a swizzled box whose bytes are not a multiple of 128
 *                                                       -> TG_ERR_UNSUPPORTED
 * The source tensor is never written ([MAP] 14). */
tg_status tma_tile_copy(const tg_tensor2d *tensor, const tg_box *box, tg_swizzle swizzle,
                        tg_oob oob, void *out, size_t out_bytes, cudaStream_t stream);

/* Tuning knobs of the tile copy ("1 . Asynchronisme et mbarrier" 1.3: stage count vs
 * shared memory).  Zero selects the default. */
typedef struct tg_copy_config {
    uint32_t stages;        /* boxes in flight per CTA, 2..16 (default 4)                  */
    uint32_t blocks_per_sm; /* resident CTAs per SM, 1..32 (default: as many as fit)       */
    uint32_t order;         /* order in which boxes are processed (the image layout does
                               not change): 0/1 = row-major over the box grid, 2 = column-
                               major                                                      */
    uint32_t l2_promotion;  /* descriptor L2 promotion ("H100 . cuTensorMap" 13): 0 =
                               default (256 B), 1 = none, 2 = 64 B, 3 = 128 B, 4 = 256 B  */
} tg_copy_config;

/* tma_tile_copy with explicit knobs (cfg may be NULL).  stages outside 2..16 or
 * blocks_per_sm above 32 -> TG_ERR_INVALID_VALUE; a ring that does not fit in shared
 * memory -> TG_ERR_UNSUPPORTED; order > 2 or l2_promotion > 4 -> TG_ERR_INVALID_VALUE. */
tg_status tma_tile_copy_ex(const tg_tensor2d *tensor, const tg_box *box, tg_swizzle swizzle,
                           tg_oob oob, void *out, size_t out_bytes, const tg_copy_config *cfg,
                           cudaStream_t stream);

/* ------------------------------------------------------------------------------------
 * Rank 1..5 tile copy with element strides   [MAP] 8-9, [TMA] 2.2 (up to 5 dimensions)
 *
 * Dimension i has dims[i] elements (dims[0] innermost and contiguous); consecutive
 * indices of dimension i >= 1 are strides[i-1] bytes apart.  A box has traversal extent
 * extent[i] and element stride element_strides[i]: it holds L_i = ceil(extent[i] /
 * element_strides[i]) elements along dimension i, element j taken from index
 * b_i*extent[i] + j*element_strides[i] of box b_i (nb_i = ceil(dims[i]/extent[i]) boxes;
 * indices beyond dims[i] read the fill value).  The image of a box is the dense
 * L_{rank-1} x ... x L_0 array (dimension 0 fastest) with the swizzle applied to its byte
 * offsets; boxes follow each other row-major over the box grid (dimension 0 fastest),
 * Π L_i * elem bytes apart.  With rank 2 and unit strides this is tma_tile_copy's image.
 * ---------------------------------------------------------------------------------- */
typedef struct tg_tensor_nd {
    const void *base;     /* device address of element 0; 16-byte aligned                */
    uint32_t dtype;       /* tg_dtype                                                     */
    uint32_t rank;        /* 1..5                                                         */
    uint64_t dims[5];     /* extents, dims[0] innermost; entries >= rank ignored           */
    uint64_t strides[4];  /* strides[i-1]: bytes between indices of dimension i >= 1     */
} tg_tensor_nd;

typedef struct tg_box_nd {
    uint32_t extent[5];          /* traversal box per dimension, 1..256                     */
    uint32_t element_strides[5]; /* 1..8; element_strides[0] must be 1 (the hardware does
                                    not stride the innermost dimension)                   */
} tg_box_nd;

/* Host-only rules: tensor/box NULL, rank 0 or > 5, unknown dtype, a dim of 0 or > 2^32,
 * base NULL, a stride >= 2^40 or smaller than the packed extent below it (strides[0] <
 * dims[0]*elem, strides[i] < dims[i]*strides[i-1]), an extent of 0 or > 256, an element
 * stride of 0 or > 8 or element_strides[0] != 1, unknown swizzle, swizzled inner bytes >
 * span -> TG_ERR_INVALID_VALUE; base not 16-byte aligned, a stride not a multiple of 16,
 * inner box bytes not a multiple of 16 -> TG_ERR_MISALIGNED. */
tg_status tma_validate_nd(const tg_tensor_nd *tensor, const tg_box_nd *box, tg_swizzle swizzle);

/* Bytes of the image tma_tile_copy_nd writes (0 for NULL or degenerate arguments). */
size_t tma_tile_copy_nd_image_bytes(const tg_tensor_nd *tensor, const tg_box_nd *box);

/* Enqueues the copy (cfg may be NULL).  Same additional rules as tma_tile_copy_ex, with
 * the box bytes being Π L_i * elem. */
tg_status tma_tile_copy_nd(const tg_tensor_nd *tensor, const tg_box_nd *box, tg_swizzle swizzle,
                           tg_oob oob, void *out, size_t out_bytes, const tg_copy_config *cfg,
                           cudaStream_t stream);

/* ------------------------------------------------------------------------------------
 * Tensor-core rate probe (measurement only; the pages state no tensor rate for this part).
 *
 *  Launches one CTA pair per two SMs; each pair issues `iters` x 4 back-to-back pair MMAs
 *  of 256 x 256 x (128 bytes of K) on zeroed operands already in shared memory, with no
 *  loads and no epilogue.  FLOPs = pairs * iters * 4 * 2 * 256 * 256 * K_mma, with K_mma =
 *  16 (bf16, fp16), 32 (E4M3, E5M2) or 8 (tf32); time it with events on `stream`.  The
 *  rate divided by the SM count and the clock is the per-SM dense FLOP per clock of the
 *  nameplate peak.  layout: only bits 4-6 (the operand type) may be set; iters in
 *  [1, 2^24]; else TG_ERR_INVALID_VALUE.  *pairs (may be NULL) receives the pairs
 *  launched.  Allocates nothing beyond the device status word.
 * ---------------------------------------------------------------------------------- */
tg_status tg_tensor_rate_probe(uint32_t layout, uint64_t iters, uint32_t *pairs,
                               cudaStream_t stream);

/* The same probe, timed by the GPU itself: `timing` is a device pointer to two uint64
 * (8-byte aligned; NULL -> TG_ERR_INVALID_VALUE, misaligned -> TG_ERR_MISALIGNED) that
 * receive, once the launch completes, the SM cycles (clock64) and the nanoseconds
 * (globaltimer) that the first pair's leader CTA spent from just before its first MMA to
 * the completion of its last.  FLOPs of one pair / cycles / 2 is then the per-SM dense
 * FLOP per clock at the clock the SMs actually ran, and cycles / ns that clock.  The
 * caller owns the buffer and synchronises `stream` before reading it. */
tg_status tg_tensor_rate_probe_timed(uint32_t layout, uint64_t iters, uint32_t *pairs,
                                     uint64_t *timing, cudaStream_t stream);

/* ------------------------------------------------------------------------------------
 * Copy back: the inverse of tma_tile_copy_nd.  [TMA] 2.5 "Copies dans les deux sens"
 * (shared -> global copies with the same descriptors) and [MAP] 11 (the swizzle is the
 * copy engine's, in both directions).
 *
 *  Reads an image laid out as tma_tile_copy_nd writes it (same tensor, box and swizzle)
 *  and writes every box back into the tensor through a tensor store with the same
 *  descriptor, which undoes the swizzle and writes only the elements inside the tensor.
 *  A round trip therefore restores the tensor; the library's test suite uses it to check
 *  its model of the swizzled image against the hardware.  Rules: those of
 *  tma_tile_copy_nd (with `image` / `image_bytes` in place of out / out_bytes, NULL image
 *  -> TG_ERR_INVALID_VALUE); element strides other than 1, or a row of dims[0] elements
 *  whose byte length is not a multiple of 16 -> TG_ERR_UNSUPPORTED (a tensor store writes
 *  whole 16-byte units at the right edge).  The tensor's storage is written; overlapping
 *  boxes cannot occur.
 * ---------------------------------------------------------------------------------- */
tg_status tma_tile_copy_back_nd(const tg_tensor_nd *tensor, const tg_box_nd *box,
                                tg_swizzle swizzle, const void *image, size_t image_bytes,
                                const tg_copy_config *cfg, cudaStream_t stream);

/* ------------------------------------------------------------------------------------
 * Region copy: the box grid starts anywhere.  [TMA] "Remplissage des bords" and [MAP]
 * section 14 (out-of-bounds fill: the parts of a box outside the tensor are filled in
 * shared memory, the tensor in global memory is never touched).
 *
 *  Along dimension i (i < rank) the grid holds nboxes[i] boxes; box b covers indices
 *  origin[i] + b * extent[i] ... + extent[i] - 1 (stepping by element_strides[i]).
 *  origin[i] may be negative and boxes may run past dims[i]: every index outside
 *  [0, dims[i]) reads the fill value (zero, or NaN with TG_OOB_NAN) -- the pages only
 *  describe a box running past the tensor's end; an index below 0 is taken to be out of
 *  bounds the same way.  tma_tile_copy_nd is the case origin 0, nboxes[i] =
 *  ceil(dims[i] / extent[i]).  The image layout is the same: boxes row-major over the
 *  grid, dimension 0 fastest.  Entries at or beyond `rank` are ignored.
 *
 *  Rules on top of tma_validate_nd: origin or nboxes NULL, a box count of 0 or above
 *  2^32-1, or a box coordinate outside the int32 range -> TG_ERR_INVALID_VALUE;
 *  origin[0] * element size not a multiple of 16 -> TG_ERR_MISALIGNED (a copy starts on
 *  a 16-byte boundary).
 * ---------------------------------------------------------------------------------- */
tg_status tma_validate_region_nd(const tg_tensor_nd *tensor, const tg_box_nd *box,
                                 const int32_t origin[5], const uint32_t nboxes[5],
                                 tg_swizzle swizzle);

/* Bytes of the image tma_tile_copy_region_nd writes (0 for NULL or degenerate arguments). */
size_t tma_tile_copy_region_nd_image_bytes(const tg_tensor_nd *tensor, const tg_box_nd *box,
                                           const uint32_t nboxes[5]);

/* Enqueues the region copy (cfg may be NULL); the other rules are tma_tile_copy_nd's. */
tg_status tma_tile_copy_region_nd(const tg_tensor_nd *tensor, const tg_box_nd *box,
                                  const int32_t origin[5], const uint32_t nboxes[5],
                                  tg_swizzle swizzle, tg_oob oob, void *out, size_t out_bytes,
                                  const tg_copy_config *cfg, cudaStream_t stream);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* TG_H_ */
