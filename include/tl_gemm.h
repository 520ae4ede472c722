/*
 * tl_gemm.h -- C ABI of the GB300 (sm_103a) tiled GEMM with a fused epilogue.
 *
 *   C = epi(op(A) . op(B)),  epi in {identity, ReLU},  fp16/bf16 in and out,
 *   fp32 accumulation in Tensor Memory, round-to-nearest-even on the output.
 *
 * The same pipeline also serves 8-bit operands (tl_gemm_fp8: one product scale;
 * tl_gemm_mx: one E8M0 scale per 32 K elements) and the attention forward pass
 * (tl_attention_fwd); each declaration below states its own semantics and sources.
 *
 * Sources of the semantics (the pages the operation is described on):
 *   - The tiled GEMM itself: the quickstart kernel copies A and B tiles global ->
 *     shared, multiplies them into an fp32 accumulator under a multi-stage
 *     software pipeline, and copies the accumulator back to global ("TileLang: a
 *     tile language one level below Triton", section "first kernel: GEMM";
 *     "TileLang: from tile dataflow to controllable AI kernels", section "minimal
 *     but complete GEMM skeleton": fp16 inputs, fp32 accumulation, cast to the
 *     output dtype at the end).
 *   - transpose_A / transpose_B: A is [M,K] or, transposed, [K,M]; B is [K,N] or,
 *     transposed, [N,K] ("TileLang core primitives" page, section 3.3 "T.gemm").
 *   - The ReLU epilogue max(x, 0) on the fp32 accumulator before the cast ("NVIDIA
 *     backend codegen" page, section 1, the GEMM+ReLU quickstart; "TileLang core
 *     primitives" page, section 3.8).
 *   - Partial tiles: out-of-range source elements read as 0 and out-of-range
 *     destination elements are never written ("TileLang core primitives" page,
 *     section 4.2 "out of bounds and padding"; TMA zero fill, "NVIDIA backend
 *     codegen" page, section 4.4.3).
 *   - Argument checks at the ABI boundary, before any launch ("TileLang: from tile
 *     dataflow to controllable AI kernels", section "automatically generated host
 *     checks"), and explicit failure instead of a silent fallback ("NVIDIA backend
 *     codegen" page, section 4.3.2).
 *
 * All pointers to matrices are DEVICE pointers of the current CUDA device.  The
 * library never frees or retains caller memory.  Every call is asynchronous on
 * `stream` (NULL = the legacy default stream) and returns once the work is
 * enqueued.  The library holds only per-device caches of kernel attributes and a
 * bounded host-side cache of encoded tensor-map descriptors (each a pure function of
 * a buffer's address, extents and pitch, so a stale entry is never wrong); it is
 * safe to call from several host threads.  The GEMM kernel is launched with
 * programmatic stream serialization and signals at its start that dependents may
 * launch: it does its own set-up while the previous kernel of the stream finishes,
 * and waits for that kernel before touching memory.  A kernel of the caller that is
 * itself launched with programmatic serialization after a GEMM may therefore start
 * before the GEMM ends, and must wait for it (cudaGridDependencySynchronize) before
 * using C, as CUDA requires of such kernels; ordinary launches are unaffected.
 */
#ifndef TL_GEMM_H
#define TL_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream, without requiring the CUDA headers. */
struct CUstream_st;
typedef struct CUstream_st* tl_stream_t;

/* Element types.  fp16 and bf16 are operand and output types of tl_gemm(); the
 * 8-bit E4M3 ("fn": finite only, bias 7, largest 448) and E5M2 (bias 15, with
 * infinities) are operand types of tl_gemm_fp8() only, whose output is fp16 or bf16.
 * The planning functions accept all four (8-bit: plans for tl_gemm_fp8). */
typedef enum { TL_F16 = 0, TL_BF16 = 1, TL_E4M3 = 2, TL_E5M2 = 3 } tl_dtype;

typedef enum { TL_EPI_NONE = 0, TL_EPI_RELU = 1 } tl_epilogue;

typedef enum {
  TL_OK = 0,
  TL_ERR_INVALID_ARG = 1,  /* negative size, ld too small, bad enum, bad plan      */
  TL_ERR_NULL_PTR = 2,     /* NULL matrix pointer with a non-empty extent          */
  TL_ERR_ALIGNMENT = 3,    /* a matrix pointer not aligned to its 2-byte element   */
  TL_ERR_UNSUPPORTED = 4,  /* valid request the library cannot run (no sm_103 GPU,*/
                           /* size beyond the library's limits)                    */
  TL_ERR_ALIAS = 5,        /* C overlaps A or B                                    */
  TL_ERR_DEVICE = 6,       /* pointer not on the current device, CUDA query failed */
  TL_ERR_LAUNCH = 7,       /* a kernel or an allocation failed to enqueue          */
  TL_ERR_TIMEOUT = 8       /* a device-side wait ran out (read by tl_device_status)*/
} tl_status;

/*
 * One execution plan: the tiling and scheduling the kernel runs with.
 * tl_gemm_plan() fills it from (M, N, K, dtype, transposes) without touching a
 * GPU; tl_gemm_with_plan() runs a given plan.
 */
typedef struct {
  int32_t bm;            /* output rows per tile: 128 (one CTA) or 256 (a CTA pair   */
                         /* in a 2-CTA cluster sharing each MMA, 128 rows each)     */
  int32_t bn;            /* output columns per tile (64, 128, 256; pairs 128, 256;  */
                         /* 16 or 32 with bk 128 when the kernel's B is K-major)    */
  int32_t bk;            /* K elements per pipeline stage: 64 or 128 (one or two    */
                         /* 128-byte swizzle rows per matrix row)                   */
  int32_t stages;        /* depth of the shared-memory ring                         */
  int32_t raster_group;  /* tile rows per L2 rasterisation group                    */
  int32_t grid;          /* persistent CTAs launched (0 = one per SM or SM pair,    */
                         /* capped by the tiles and by the resident clusters)       */
  int64_t tiles_m, tiles_n, tiles, k_blocks;
  int64_t ring_bytes;    /* per CTA: stages * (128*bk + (bn/cg)*bk) * 2, cg = bm/128 */
  int64_t smem_bytes;    /* dynamic shared memory per CTA (ring + staging + bars)   */
  int32_t tmem_cols;     /* Tensor Memory columns allocated per CTA (2 accumulators,*/
                         /* at least 32)                                            */
  int32_t tx_bytes;      /* bytes one stage's TMA loads deliver to one CTA          */
  int32_t repack_a;      /* A is staged through a pitch-padded workspace (plans     */
  int32_t repack_b;      /* from tl_gemm_plan assume aligned operands: 0)           */
  int32_t tma_store;     /* C written by TMA bulk stores when C is 16-byte aligned  */
                         /* (else predicated stores)                                */
  int32_t l2_prefetch;   /* k-blocks prefetched into L2 ahead of the ring (0 = off) */
  int32_t producers;     /* TMA producer threads taking turns by stage (1..3, at    */
                         /* most `stages`; 0 = default)                             */
  int32_t stream_k;      /* -1 off, 0 automatic, 1 on: the k-blocks of the last     */
                         /* waves' tiles are split evenly over all CTAs (pairs)     */
  int32_t dp_tiles;      /* tiles run whole before the split region                 */
  int32_t swap_ab;       /* 1: the kernel computes C^T = op(B)^T . op(A)^T (the     */
                         /* skinny-M plan: N on the MMA's 128 rows, M <= bn on its  */
                         /* narrow side) and writes it transposed into C; tiles_m,  */
                         /* tiles_n then count tiles of C^T.  0: C directly.        */
  int64_t sk_iters;      /* k-block iterations split evenly (0: no split)           */
  int64_t workspace_bytes; /* bytes of the stream-ordered workspace (repacked       */
                         /* operands, stream-K partial sums and flags)              */
  int32_t ksplit;        /* cluster split-K, bm = 128 and bn a power of two only:   */
                         /* 2 = two CTAs of a cluster share each tile's k-blocks,   */
                         /* each handing the fp32 partial sums of half the tile's   */
                         /* columns to the other through distributed shared memory; */
                         /* 1 = off; 0 (input) = automatic (when the tiles fill at  */
                         /* most half the SMs and k_blocks >= 4)                    */
} tl_plan;

/*
 * C = epi(op(A) . op(B)).
 *
 *   A  device pointer; op(A)[i,k] = A[i*lda + k], or A[k*lda + i] if trans_a.
 *   B  device pointer; op(B)[k,j] = B[k*ldb + j], or B[j*ldb + k] if trans_b.
 *   C  device pointer; C[i*ldc + j] for 0 <= i < M, 0 <= j < N.  Nothing outside
 *      that region is written.  C must not overlap A or B.
 *   M, N, K >= 0.  M == 0 or N == 0: returns TL_OK, launches nothing.  K == 0:
 *      C is filled with epi(0) = +0.
 *   lda >= (trans_a ? M : K), ldb >= (trans_b ? K : N), ldc >= N (elements).
 *   dtype: element type of A, B and C.  Accumulation is fp32; the output rounds
 *      to nearest even.  epilogue: TL_EPI_NONE or TL_EPI_RELU (applied to the fp32
 *      accumulator; negative values give +0).
 *   stream: CUDA stream to enqueue on.
 *
 * Operands whose base or pitch is not 16-byte aligned (tensor-memory-access rule:
 * the leading pitch in bytes must be a multiple of 16) are first copied on
 * `stream` into a workspace with the pitch rounded up, allocated and freed with
 * the stream-ordered allocator; an unaligned C is written by predicated stores.
 * When the tiles do not fill whole waves of the GPU, the k-blocks of the last
 * waves are split evenly over all CTAs (stream-K); the fp32 partial sums of split
 * tiles pass through the same kind of workspace and are added in a fixed order, so
 * results are deterministic for a given plan and GPU.
 *
 * Errors are returned before anything is enqueued: TL_ERR_INVALID_ARG,
 * TL_ERR_NULL_PTR, TL_ERR_ALIGNMENT, TL_ERR_ALIAS, TL_ERR_DEVICE,
 * TL_ERR_UNSUPPORTED.  TL_ERR_LAUNCH means an enqueue failed.
 */
tl_status tl_gemm(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                  int64_t lda, int64_t ldb, int64_t ldc, tl_dtype dtype, int trans_a,
                  int trans_b, tl_epilogue epilogue, tl_stream_t stream);

/*
 * The plan tl_gemm() would run for this problem.  Host only: touches no GPU (the
 * SM count is taken as `num_sms`, or 152 (GB300) when num_sms <= 0).  Returns
 * TL_ERR_INVALID_ARG for negative sizes or bad enums.  The resource figures follow
 * the pages' shared-memory model S = stages * (BM*BK*s_A + BK*BN*s_B) + S_other
 * ("TileLang: from tile dataflow to controllable AI kernels", section "more
 * stages is not always better").
 */
tl_status tl_gemm_plan(int64_t M, int64_t N, int64_t K, tl_dtype dtype, int trans_a,
                       int trans_b, int num_sms, tl_plan* plan);

/*
 * Fill the derived fields of `plan` (tiles, k-blocks, ring/smem bytes, TMEM
 * columns, tx bytes) from its bm/bn/bk/stages and the problem size.  Host only.
 * Returns TL_ERR_INVALID_ARG when the tiling is not one the kernel supports:
 *   16-bit operands: bm = 128 with bn in {64,128,256}, or bm = 256 with bn in
 *     {128,256}, bk = 64 or 128; bm = 128 with bn in {16,32} (skinny plans) or
 *     bm in {128,256} with bn in {192,224}, bk = 128 only, and for those a
 *     K-major B (trans_b = 1; with swap_ab, an A that is not transposed);
 *   8-bit operands (tl_gemm_fp8): bm = 128 with bn in {64,128,256}, or bm = 256
 *     with bn in {128,256}, bk = 128 or 256, no swap_ab;
 *   stages 2..8 and shared memory within the per-CTA limit;
 *   ksplit = 2 only with bm = 128 and a power-of-two bn.
 */
tl_status tl_plan_complete(int64_t M, int64_t N, int64_t K, tl_dtype dtype, int trans_a,
                           int trans_b, int num_sms, tl_plan* plan);

/*
 * tl_gemm() with an explicit plan (bm, bn, bk, stages, raster_group, grid,
 * l2_prefetch, producers, stream_k and swap_ab are read, and tma_store = -1 asks
 * for plain stores of C; the rest is recomputed; l2_prefetch < 0, producers <= 0
 * and stream_k = 0 select the defaults).  Used
 * to run a workload at a fixed tiling, e.g. the
 * pages' quickstart 128x128x64 with 3 stages.  Same arguments and errors as
 * tl_gemm(), plus TL_ERR_INVALID_ARG for an unsupported plan.
 */
tl_status tl_gemm_with_plan(const void* A, const void* B, void* C, int64_t M, int64_t N,
                            int64_t K, int64_t lda, int64_t ldb, int64_t ldc, tl_dtype dtype,
                            int trans_a, int trans_b, tl_epilogue epilogue,
                            const tl_plan* plan, tl_stream_t stream);

/*
 * C = epi(alpha * op(A) . op(B)) with 8-bit floating-point operands.  (The pages'
 * Blackwell GEMM also runs on low-precision operands: "NVIDIA backend codegen"
 * page, section 4.6.3, and the block-scaled MMA of "TileLang: a tile language one
 * level below Triton", where 32 consecutive K elements share one exponent; this
 * entry point takes one scale for the whole product, which is that form with every
 * block scale equal.)
 *
 *   A, B     device pointers to 8-bit codes: A of format a_type, B of b_type (each
 *            TL_E4M3 or TL_E5M2; the two may differ).  op(A) and op(B) as in
 *            tl_gemm(); lda, ldb, ldc in elements (bytes for A and B).
 *   C        device pointer to c_type elements (TL_F16 or TL_BF16), written as in
 *            tl_gemm(); C must not overlap A or B.
 *   alpha    finite fp32 scale applied to the fp32 accumulator before the epilogue
 *            (ReLU on alpha * sum) and the round-to-nearest-even cast.
 *   plan     NULL for the planner's choice (tl_gemm_plan with dtype = a_type gives
 *            it), or a plan whose bk is 128 or 256 (K elements per stage: one or two
 *            128-byte chunks) and bn >= 64; with B N-major (trans_b = 0) each CTA's
 *            share of the tile's columns (bn, or bn/2 for pairs) must be a multiple
 *            of 128.  No operand swap.
 * Operands whose base or pitch is not 16-byte aligned are copied to a padded pitch
 * as in tl_gemm() (stream-ordered workspace).  Accumulation is fp32 in Tensor
 * Memory; each product of two 8-bit values is exact in it.  Errors as tl_gemm(),
 * plus TL_ERR_INVALID_ARG for a non-8-bit operand type, a non-16-bit c_type, a
 * non-finite alpha or an unsupported plan.
 */
tl_status tl_gemm_fp8(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                      int64_t lda, int64_t ldb, int64_t ldc, tl_dtype a_type, tl_dtype b_type,
                      tl_dtype c_type, int trans_a, int trans_b, float alpha,
                      tl_epilogue epilogue, const tl_plan* plan, tl_stream_t stream);

/*
 * tl_gemm() for callers that cannot allocate device memory.  (This entry point has
 * no counterpart on the pages the GEMM is described on; it is a property of this
 * library's C ABI.)
 *
 * Who needs it: tl_gemm() takes a temporary buffer from the stream-ordered
 * allocator when A or B has a base or leading dimension the tensor-memory-access
 * unit cannot address (not 16-byte aligned) and must first be copied with a padded
 * pitch.  Some callers cannot allow that: a framework that owns all device memory
 * through its own pool and must not see a second allocator fragment or exceed its
 * budget; a serving process that has reserved nearly all HBM for its caches, where
 * any extra allocation fails; a real-time loop that must not allocate after start-up.
 * tl_gemm_noalloc() calls no cudaMalloc, cudaFree or allocating library routine.
 *
 * Instead it copies such operands into one fixed scratch array of
 * tl_gemm_noalloc_scratch_bytes() bytes (32 MiB) that the library defines as device
 * global memory: every GPU that loads the library holds it until the process exits.
 *   - Same arguments, semantics and errors as tl_gemm(), plus TL_ERR_UNSUPPORTED
 *     (returned before anything is enqueued) when the operands that need a copy do
 *     not fit the array: rows * (pitch rounded up to 8 elements) * 2 bytes for A,
 *     rounded up to 256 bytes, plus the same for B, must not exceed 32 MiB.
 *     Operands that need no copy use no scratch and have no size limit.
 *   - The first call on each device (that passes the argument checks) performs a
 *     one-time set-up: it looks up the array's device address with that device
 *     current.  Make that first call before any stream capture.  If that lookup
 *     failed, later calls on the device that need a copy return TL_ERR_DEVICE; calls
 *     that need none still run.
 *   - Every call shares the one array, and it keeps whatever the last call left in
 *     it (nothing read from it depends on that).  Calls whose work overlaps on the
 *     GPU (different streams, or host threads enqueueing concurrently) race on the
 *     array: serialise them, e.g. keep them on one stream.
 */
tl_status tl_gemm_noalloc(const void* A, const void* B, void* C, int64_t M, int64_t N,
                          int64_t K, int64_t lda, int64_t ldb, int64_t ldc, tl_dtype dtype,
                          int trans_a, int trans_b, tl_epilogue epilogue, tl_stream_t stream);

/* Size in bytes of the scratch array tl_gemm_noalloc() uses (33554432). */
int64_t tl_gemm_noalloc_scratch_bytes(void);

/* Static, NUL-terminated name of a status code ("TL_OK", ...). */
const char* tl_status_string(tl_status status);

/*
 * Outcome of the device-side bounded waits since the last reset, for the current
 * device: TL_OK, or TL_ERR_TIMEOUT if some wait of some kernel gave up (the
 * kernel then set this flag, drained its own copies, freed its Tensor Memory and
 * returned; its output is undefined).  Synchronises the device.  If `reset` is
 * non-zero the flag is cleared afterwards.  `detail`, if not NULL, receives the
 * raw status word (role and wait site of the first timeout).
 */
tl_status tl_device_status(int reset, uint32_t* detail);

/*
 * The same outcome without reset or detail: synchronises the current device and
 * returns TL_OK, or the status of the first device-side wait that gave up since the
 * flag was last cleared (tl_device_status with reset = 1 clears it).  A debugging
 * aid for use after a sync point; TL_ERR_DEVICE if the device cannot be queried.
 */
tl_status tl_last_device_status(void);

/*
 * Limit of every device-side wait for kernels enqueued after this call, in
 * nanoseconds at an SM clock of 4 GHz (default 1e9): the kernels count 4 SM cycles
 * per nanosecond, so at the GPU's real clock (about 2 GHz) a wait gives up after
 * two to four times this value.  Clamped to [1e5, 6e10].  Host only.
 */
void tl_set_wait_timeout_ns(uint64_t ns);

/*
 * Block-scaled 8-bit GEMM (the MX formats): 8-bit operands in which every 32
 * consecutive K elements of a row share one power-of-two scale ("NVIDIA backend
 * codegen" page, section 4.6.3: the block-scaled MMA, tcgen05 kind::mxf8f6f4 with
 * the scale factors in Tensor Memory):
 *
 *   C[i*ldc+j] = epi( sum_k x(A[i*lda+k]) 2^(SFA[i*sfa_ld+k/32] - 127)
 *                           * x(B[j*ldb+k]) 2^(SFB[j*sfb_ld+k/32] - 127) )
 *
 *   A        device pointer, M x K codes of a_type (TL_E4M3 or TL_E5M2), K-major.
 *   B        device pointer, N x K codes of b_type, K-major (the MX layout: C = A B^T).
 *   SFA/SFB  device pointers to E8M0 scale codes (the value 2^(e-127); 255 is NaN),
 *            one byte per 32-element block of each row of A / B.  Their row pitches
 *            sfa_ld / sfb_ld are in bytes, at least 4*ceil(K/128) (whole groups of four
 *            blocks); codes of blocks past K/32 and of the padding are ignored.
 *   C        device pointer, M x N of c_type (TL_F16 or TL_BF16), rounded once from
 *            the fp32 accumulator; epilogue TL_EPI_NONE or TL_EPI_RELU.
 * K must be a multiple of 32 (TL_ERR_INVALID_ARG).  A, B, SFA and SFB must be 16-byte
 * aligned with lda, ldb, sfa_ld and sfb_ld multiples of 16 (all four are read by the
 * TMA unit); C 2-byte aligned (TL_ERR_ALIGNMENT otherwise).  C must not overlap an input (TL_ERR_ALIAS).
 * M or N == 0: TL_OK, nothing launched; K == 0: C = 0.  Asynchronous on `stream`;
 * the caller owns every buffer; errors are returned before anything is enqueued, a
 * device-side timeout is read with tl_device_status().
 */
tl_status tl_gemm_mx(const void* A, const void* B, const void* SFA, const void* SFB, void* C,
                     int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                     int64_t sfa_ld, int64_t sfb_ld, tl_dtype a_type, tl_dtype b_type,
                     tl_dtype c_type, tl_epilogue epilogue, tl_stream_t stream);

/*
 * Attention forward pass: O = softmax(Q K^T / sqrt(D)) V for every batch and head,
 * optionally causal (query i attends to keys j <= i).  This is the pages' second
 * workload on the same tile primitives ("TileLang: a tile language one level below
 * Triton", section "FlashAttention: online softmax as tile code"), with their layout
 * and scale: Q, K, V and O are [B, S, H, D] row-major (batch, sequence, heads, head
 * dim), scores scaled by 1/sqrt(D).
 *
 *   Q, K, V, O  device pointers to dtype elements (TL_F16 or TL_BF16), 16-byte
 *               aligned (TL_ERR_ALIGNMENT otherwise); O must not overlap Q, K or V.
 *   D           64 or 128 (TL_ERR_UNSUPPORTED otherwise).
 *   causal      0 or 1.
 * B, S or H == 0: returns TL_OK, launches nothing.  Scores and the softmax statistics
 * are fp32; the probabilities enter the PV product rounded to dtype (as in the
 * pages' kernel, which casts them to fp16); O accumulates in fp32 and is rounded once.
 * Asynchronous on `stream`; errors are returned before anything is enqueued, a
 * device-side timeout is read with tl_device_status().
 */
tl_status tl_attention_fwd(const void* Q, const void* K, const void* V, void* O, int64_t B,
                           int64_t S, int64_t H, int64_t D, tl_dtype dtype, int causal,
                           tl_stream_t stream);

/*
 * Test hook for the failure-detection path; not for production use.  mode 1: every
 * GEMM kernel launched afterwards has its MMA thread wait first on a barrier that
 * nothing arrives on, as if its operands never came.  The wait runs out after the
 * limit set by tl_set_wait_timeout_ns(); the kernel then records TL_ERR_TIMEOUT with
 * wait site 7 in the device status word, every role unwinds (issued loads land,
 * Tensor Memory is freed) and the kernel returns with C unwritten.  mode 0 (the
 * default) turns it off.  No compute fault, trap or unbounded wait is involved.
 */
void tl_debug_set_stall(int mode);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int tl_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TL_GEMM_H */
