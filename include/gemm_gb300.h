/*
 * gemm_gb300.h -- C ABI of the GB300 (sm_103a) tcgen05 dense GEMM library.
 *
 *     D[M,N] = A[M,K] * B[N,K]^T      fp32 accumulation, bf16 output
 *
 * The operation is the dense GEMM of b200-gemm-optimization-ladder ("E --
 * Executable steps", step 1: fix the math definition, layout and dtype; "A1 --
 * The nine-level route": data path GMEM -> SMEM -> tcgen05 -> TMEM ->
 * registers/SMEM -> GMEM), with the block-scaled variant whose scale factors
 * are staged SMEM -> TMEM by tcgen05.cp (b200-tmem-lifecycle-planner, "A1 --
 * Case 2: block-scaled MMA").
 *
 * Layout (all matrices row-major, leading dimensions in ELEMENTS):
 *   A  [M, K] with row pitch lda >= K          (K contiguous)
 *   B  [N, K] with row pitch ldb >= K          (K contiguous, "K-major")
 *   D  [M, N] with row pitch ldd >= N          (bf16, round-to-nearest-even)
 *
 * Ownership: every pointer is a caller-owned DEVICE pointer (e.g. a torch CUDA
 * tensor).  The library never allocates or frees device memory; its only
 * device state is one status word per device, read by gemm_last_status().
 * A, B, SFA, SFB must not overlap D.
 *
 * Ordering: calls are asynchronous on `stream` (0 = the legacy default
 * stream), like cuBLAS.  Argument errors are returned synchronously; a
 * device-side watchdog timeout is reported by gemm_last_status().
 *
 * Errors: every entry point returns a gemm_status_t:
 *   GEMM_ERR_INVALID_ARG  M, N or K negative or >= 2^31, a NULL pointer,
 *                         lda < K, ldb < K, ldd < N, a pointer that is not
 *                         device memory, an unknown variant
 *   GEMM_ERR_ALIGNMENT    A or B not 16-byte aligned, or an A/B row pitch
 *                         whose byte size is not a multiple of 16 (the TMA
 *                         engine's rule): bf16 needs lda, ldb multiples of
 *                         8, E4M3 multiples of 16 (MXFP8 scale matrices
 *                         take any pitch and alignment); or D (C, bias of a
 *                         fused epilogue) not aligned to its element size
 *   GEMM_ERR_UNSUPPORTED_DEVICE  the current device is not compute
 *                         capability 10.3 (sm_103); there is no fallback
 *   GEMM_ERR_LAUNCH       the CUDA launch (or tensor-map encoding) failed
 * M == 0 or N == 0 is a no-op that returns GEMM_OK.  K == 0 writes D = 0
 * (the empty sum).  D may have any pitch (ldd >= N) and any element-aligned
 * base: when its rows are not 16-byte aligned the epilogue uses masked stores
 * instead of TMA stores.
 */
#ifndef GEMM_GB300_H
#define GEMM_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#ifndef __DRIVER_TYPES_H__
typedef struct CUstream_st* cudaStream_t;
#endif

typedef enum {
  GEMM_OK = 0,
  GEMM_ERR_INVALID_ARG = -1,
  GEMM_ERR_ALIGNMENT = -2,
  GEMM_ERR_UNSUPPORTED_DEVICE = -3,
  GEMM_ERR_LAUNCH = -4,
  GEMM_ERR_TIMEOUT = -5,
  GEMM_ERR_DEVICE_FAULT = -6
} gemm_status_t;

/* Kernel choice for gemm_bf16_variant / gemm_mxfp8_variant. */
typedef enum {
  GEMM_VARIANT_AUTO = 0,        /* the fastest path for the arguments              */
  GEMM_VARIANT_1CTA = 1,        /* persistent warp-specialised, cta_group::1,
                                   128x256 tiles (bf16) or 128x224 tiles (MXFP8)
                                   (ladder levels 4-7)                             */
  GEMM_VARIANT_2CTA = 2,        /* persistent warp-specialised CTA pair,
                                   cta_group::2, 256x256 tiles (bf16) or 256x224
                                   tiles (MXFP8) (ladder level 8)                  */
  GEMM_VARIANT_SYNC = 3,        /* one 128x128 tile per CTA, synchronous copies
                                   (ladder levels 1-3; bf16 only, reference rung)  */
  GEMM_VARIANT_SMALLK = 4,      /* bf16 only, 1 <= K <= 16: CUDA-core kernel for
                                   the HBM-bound case (a write of D at about 8
                                   flops per byte), aligned 16-byte row stores     */
  GEMM_VARIANT_SMALLK_TC = 5,   /* bf16 only, 1 <= K <= 16: one tcgen05.mma per
                                   128x256 tile (operands loaded at their real K,
                                   rows grouped by residue mod 8 so that every
                                   store is an aligned 16-byte one); AUTO picks
                                   for plain calls with K <= 16 the CUDA-core
                                   kernel below 48 MB of output, this one above  */
  GEMM_VARIANT_DIRECT_STORE = 0x100  /* flag: masked st.global epilogue instead of
                                        TMA stores, even when D is aligned.  Without
                                        it the library picks: TMA stores where D is
                                        16-byte aligned with ldd and N multiples of
                                        8 (64-column boxes for bf16, 32-column for
                                        MXFP8), except that a stream-K launch that
                                        splits tiles (bf16, or MXFP8 on one CTA)
                                        takes the masked kernel, whose two epilogue
                                        warpgroups share the partial sums, and so
                                        does a bf16 fused epilogue on one CTA      */
} gemm_variant_t;

/*
 * bf16 GEMM: D = A * B^T with A, B, D bf16 (IEEE bfloat16 bit patterns).
 * Runs the persistent tcgen05 kernel chosen for the shape (GEMM_VARIANT_AUTO:
 * the CTA pair, or one CTA when M <= 128), or, for K <= 16, the small-K
 * CUDA-core kernel (GEMM_VARIANT_SMALLK).
 */
int gemm_bf16(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
              int64_t lda, int64_t ldb, int64_t ldd, cudaStream_t stream);

/* bf16 GEMM on an explicitly chosen kernel (a gemm_variant_t value, optionally
 * OR-ed with GEMM_VARIANT_DIRECT_STORE).  Same arguments and errors. */
int gemm_bf16_variant(int variant, const void* A, const void* B, void* D, int64_t M, int64_t N,
                      int64_t K, int64_t lda, int64_t ldb, int64_t ldd, cudaStream_t stream);

/*
 * Block-scaled MXFP8 GEMM:  D[i,j] = sum_k a(i,k) * b(j,k),
 *   a(i,k) = 2^(SFA[i*ldsfa + k/32] - 127) * e4m3(A[i*lda + k])
 *   b(j,k) = 2^(SFB[j*ldsfb + k/32] - 127) * e4m3(B[j*ldb + k])
 * A [M, K], B [N, K]: E4M3 ("e4m3fn") bytes, lda/ldb multiples of 16.
 * SFA [M, ldsfa], SFB [N, ldsfb]: UE8M0 scale bytes (2^(e-127), 255 = NaN), one
 * per 32 consecutive k (the last block may be partial), row-major; ldsfa,
 * ldsfb are row pitches in bytes, any value >= ceil(K/32) (the dense layout
 * ld = ceil(K/32) included), with any alignment of SFA/SFB.  When both are
 * 16-byte aligned with pitches that are multiples of 16, the scale bytes
 * travel by TMA; otherwise the kernel's scale-factor warp gathers them with
 * plain loads (same results; slower for large K).  Bytes at k-blocks
 * >= ceil(K/32) are never read.  D bf16 as above.
 */
int gemm_mxfp8(const void* A, const void* B, const void* SFA, const void* SFB, void* D,
               int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldsfa,
               int64_t ldsfb, int64_t ldd, cudaStream_t stream);

int gemm_mxfp8_variant(int variant, const void* A, const void* B, const void* SFA,
                       const void* SFB, void* D, int64_t M, int64_t N, int64_t K, int64_t lda,
                       int64_t ldb, int64_t ldsfa, int64_t ldsfb, int64_t ldd,
                       cudaStream_t stream);

/*
 * Block-scaled MXFP8 GEMM with the scale matrices already in the tensor
 * core's chunk layout (b200-tmem-lifecycle-planner, "A1 -- Case 2": scale
 * factors are staged SMEM -> TMEM by tcgen05.cp in their own layout; here
 * they arrive in that layout, so TMA moves them into each pipeline stage
 * with the operands and no thread touches them).  Same D and A/B operands,
 * values and errors as gemm_mxfp8; the scales of an R-row operand
 * (R = M for SFA, N for SFB) with nblk = ceil(K/32) blocks per row are
 *     ceil(R/128) x ceil(nblk/4) chunks of 512 bytes, chunk (rb, g) at byte
 *     512 * (rb * ceil(nblk/4) + g); inside it the scale byte of row
 *     r = 128 rb + 32 c + l and block b = 4 g + j (0 <= l < 32, c, j < 4)
 *     sits at byte 16 l + 4 c + j
 * (the layout cuBLASLt's block-scaled GEMMs take).  SFA, SFB: 16-byte
 * aligned device buffers of that size.  Bytes of rows >= R are never
 * applied to D; bytes of blocks >= nblk multiply zero-filled operands and
 * must not hold 255 (NaN): zero them.  Kernel: the CTA pair on 256x256 tiles
 * (GEMM_VARIANT_AUTO / _2CTA) or one CTA on 128x256 tiles (_1CTA), one
 * 256-column accumulator; optionally | GEMM_VARIANT_DIRECT_STORE.  Errors as
 * gemm_mxfp8, plus GEMM_ERR_ALIGNMENT for SFA/SFB not 16-byte aligned and
 * GEMM_ERR_INVALID_ARG when ceil(R/128) * ceil(K/128) * 32 exceeds 2^31 - 1.
 */
int gemm_mxfp8_tiled(int variant, const void* A, const void* B, const void* SFA, const void* SFB,
                     void* D, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                     int64_t ldd, cudaStream_t stream);

/*
 * Fused epilogue, applied to the fp32 accumulator on its way from TMEM to
 * memory (the readback step where "cast/epilogue/store" happen:
 * b200-tmem-lifecycle-planner, "A1 -- Case 1: dense MMA accumulator";
 * custom fusion is the reason to own the kernel: b200-gemm-optimization-
 * ladder, "B -- Boundaries", "Do not use when").  The pages name no
 * particular epilogue; this is the plain linear-layer one, in fp32:
 *
 *     v = alpha * acc + beta * C[i,j] + bias[j]          (terms absent when NULL)
 *     D[i,j] = act(v), rounded once to the output type (RNE)
 *
 * act: GEMM_ACT_NONE; GEMM_ACT_RELU (0 where v < 0, NaN kept); GEMM_ACT_GELU
 * v * Phi(v) = v (1 + erf(v / sqrt 2)) / 2.
 * out_dtype: GEMM_DTYPE_BF16 or GEMM_DTYPE_F32; it is also C's type.  C is
 * [M, N] with pitch ldc >= N elements, any alignment; C may be D itself
 * (in-place update) only with ldc == ldd, and must not overlap D otherwise.
 * bias: N values of bias_dtype (GEMM_DTYPE_BF16 or GEMM_DTYPE_F32), any
 * alignment.  All pointers are device pointers.
 */
enum { GEMM_DTYPE_BF16 = 0, GEMM_DTYPE_F32 = 1 };
enum { GEMM_ACT_NONE = 0, GEMM_ACT_RELU = 1, GEMM_ACT_GELU = 2 };
typedef struct gemm_epilogue {
  float alpha;
  float beta;
  const void* C;
  int64_t ldc;
  const void* bias;
  int32_t bias_dtype;
  int32_t activation;
  int32_t out_dtype;
  int32_t reserved;  /* must be 0 */
} gemm_epilogue_t;

/* gemm_bf16_variant / gemm_mxfp8_variant with a fused epilogue (variants 0,
 * 1, 2, optionally | GEMM_VARIANT_DIRECT_STORE; an fp32 output, and a bf16
 * call that runs on one CTA, always use the masked-store epilogue).  `epi` NULL means alpha = 1 and nothing else
 * (the plain entry points).  D holds elements of epi->out_dtype with pitch
 * ldd.  K == 0 gives D = act(alpha * 0 + beta * C + bias).  Errors as the
 * plain entry points, plus GEMM_ERR_INVALID_ARG for an unknown dtype or
 * activation, reserved != 0, ldc < N, a host C or bias, or C == D with
 * ldc != ldd; GEMM_VARIANT_SYNC is not offered. */
int gemm_bf16_fused(int variant, const void* A, const void* B, void* D, int64_t M, int64_t N,
                    int64_t K, int64_t lda, int64_t ldb, int64_t ldd, const gemm_epilogue_t* epi,
                    cudaStream_t stream);
int gemm_mxfp8_fused(int variant, const void* A, const void* B, const void* SFA, const void* SFB,
                     void* D, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                     int64_t ldsfa, int64_t ldsfb, int64_t ldd, const gemm_epilogue_t* epi,
                     cudaStream_t stream);

/*
 * Stream-K schedule (the scheduler row "dynamic / stream-K scheduling" of the
 * optimisation ladder's persistent level: "check the tail and tile order",
 * b200-gemm-optimization-ladder, "E -- Executable steps", level 6).  Same
 * arguments and results as gemm_bf16_variant / gemm_mxfp8_variant (variants
 * 0, 1, 2, optionally with GEMM_VARIANT_DIRECT_STORE), plus a caller-owned
 * device workspace.  When the tiles do not fill the last wave of resident
 * CTAs and the mode set by gemm_set_streamk_mode allows it (by default: where
 * a cost model predicts a gain), the tiles of that partial wave and of one
 * full wave before it -- or all tiles, when there are fewer tiles than
 * resident CTAs -- are cut along K and spread evenly over the CTAs; a tile's
 * first K-range owner adds the later ranges' fp32 partials (parked in the
 * workspace) in K order before storing D, so results are deterministic.
 * Otherwise the call behaves like the data-parallel entry point.
 * workspace: 16-byte aligned device memory of at least
 * gemm_streamk_workspace_bytes() bytes: 32 bytes of flags per CTA, then the
 * partial slots.  ZERO IT ONCE before its first use.  Later calls need no
 * clearing: a completed call leaves its flag words zero again, and a call
 * that ended in GEMM_ERR_TIMEOUT leaves flag values that identify its own
 * launch (a process-wide launch sequence number), which no later launch
 * waits for.  Calls that share a workspace must not overlap on the GPU.  Errors as the data-parallel entry points,
 * plus GEMM_ERR_INVALID_ARG for a NULL, short or misaligned workspace.
 */
int gemm_bf16_streamk(int variant, const void* A, const void* B, void* D, int64_t M, int64_t N,
                      int64_t K, int64_t lda, int64_t ldb, int64_t ldd, void* workspace,
                      int64_t workspace_bytes, cudaStream_t stream);
int gemm_mxfp8_streamk(int variant, const void* A, const void* B, const void* SFA,
                       const void* SFB, void* D, int64_t M, int64_t N, int64_t K, int64_t lda,
                       int64_t ldb, int64_t ldsfa, int64_t ldsfb, int64_t ldd, void* workspace,
                       int64_t workspace_bytes, cudaStream_t stream);

/*
 * gemm_bf16_streamk without a caller workspace; it allocates nothing.  The
 * pages have no counterpart: this entry point exists for callers that must
 * not allocate device memory where they multiply -- code inside a memory
 * allocator's own out-of-memory or defragmentation path, where an allocation
 * would re-enter the allocator, or a serving loop that reserves its device
 * memory at start-up and may not grow it later.  The scratch is a library-owned
 * static device buffer of 24 MiB per device (enough for 191 resident CTAs;
 * a GB300 runs 152).  Same arguments, results and errors as
 * gemm_bf16_streamk (variants 0, 1, 2, optionally | GEMM_VARIANT_DIRECT_STORE)
 * minus the workspace, plus GEMM_ERR_INVALID_ARG when the device would need
 * more scratch than the buffer holds.
 * First call per device: with that device current, it looks up the buffer's
 * address (cudaGetSymbolAddress) and clears the buffer with a
 * cudaMemsetAsync queued on `stream` ahead of its own kernel, so make the
 * first call for each device before any stream capture begins.  Later calls
 * do not clear it (nothing needs clearing, also after a GEMM_ERR_TIMEOUT).
 * Every call on a device shares the one buffer: calls that overlap on the GPU
 * (other streams, other host threads) race and give wrong results; order
 * them on one stream or synchronise between them.  The buffer's address is
 * kept for the life of the process: calling cudaDeviceReset() and then this
 * entry point is not supported (nor, for the same reason, any other entry
 * point of the library, which keeps its status word's address the same way).
 */
int gemm_bf16_streamk_noalloc(int variant, const void* A, const void* B, void* D, int64_t M,
                              int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldd,
                              cudaStream_t stream);

/* When the stream-K entry points split tiles, for later calls in this
 * process: GEMM_STREAMK_AUTO (default) splits only where a cost model of the
 * kernel (whole-tile waves against split ranges plus the fix-up of each
 * split tile) predicts a gain of 5% or more; GEMM_STREAMK_ALWAYS splits
 * whenever the tiles leave a partial wave and K has two units or more;
 * GEMM_STREAMK_NEVER always runs the data-parallel schedule.  Returns the
 * previous mode, or GEMM_ERR_INVALID_ARG for another value. */
enum { GEMM_STREAMK_AUTO = 0, GEMM_STREAMK_ALWAYS = 1, GEMM_STREAMK_NEVER = 2 };
int gemm_set_streamk_mode(int mode);

/* The schedule the stream-K entry points would use (host only, no device
 * needed): for `tiles` output tiles, `resident` co-resident clusters, K-tiles
 * per tile and K-tiles per stream-K unit (1 for bf16, 4 for MXFP8) under
 * `mode`, out[0] = tiles computed whole, out[1] = tiles split along K,
 * out[2] = clusters launched (0 when there is nothing to compute).  `out`
 * holds 3 values.  GEMM_ERR_INVALID_ARG for out-of-range arguments. */
int gemm_streamk_plan(int64_t tiles, int64_t resident, int64_t k_tiles, int64_t unit, int mode,
                      int64_t* out);

/* Workspace bytes the stream-K entry points need on the current device for a
 * kernel variant (mxfp8: 0 = bf16, 1 = MXFP8); negative gemm_status_t on error. */
int64_t gemm_streamk_workspace_bytes(int mxfp8, int variant);

/*
 * MXFP8 quantisation on the GPU: the encoding the block-scaled GEMM consumes
 * (b200-tmem-lifecycle-planner, "A1 -- Case 2: block-scaled MMA").
 * X [rows, K]: float32, row pitch ldx >= K elements (any alignment).
 * For every row and every block of 32 consecutive k (the last may be partial):
 *   amax = largest |x| over the block's finite values;
 *   e    = smallest integer with amax <= 448 * 2^e, clamped to [-127, 127]
 *          (amax = 0 gives e = -127);
 *   SF[r * ldsf + b] = e + 127 (UE8M0);
 *   Q[r * ldq + k]   = x * 2^-e rounded to E4M3 ("e4m3fn"), nearest even;
 *                      NaN and +-Inf encode as E4M3 NaN with their sign.
 * Q [rows, ldq >= K] and SF [rows, ldsf >= ceil(K/32)] are caller-owned device
 * buffers; a gemm_mxfp8 call may consume them directly (its own rules on lda
 * and ldsf apply there).  Asynchronous on `stream`.  Errors: INVALID_ARG for
 * negative or too-large sizes, short pitches, NULL or non-device pointers;
 * rows == 0 or K == 0 is a no-op.
 */
int gemm_mxfp8_quantize(const float* X, int64_t rows, int64_t K, int64_t ldx, void* Q,
                        int64_t ldq, void* SF, int64_t ldsf, cudaStream_t stream);

/* gemm_mxfp8_quantize writing the scale bytes in the tiled layout that
 * gemm_mxfp8_tiled takes (no counterpart on the pages beyond the scale
 * layout itself): SF receives ceil(rows/128) * ceil(ceil(K/32)/4) * 512
 * bytes, every one written -- the scales, and zero in the padding (rows past
 * `rows` in the last row block, blocks past ceil(K/32) in the last group).
 * Q as for gemm_mxfp8_quantize.  Same errors, minus the scale pitch. */
int gemm_mxfp8_quantize_tiled(const float* X, int64_t rows, int64_t K, int64_t ldx, void* Q,
                              int64_t ldq, void* SF, cudaStream_t stream);

/*
 * Synchronises `stream`, then returns and clears the current device's status
 * word: GEMM_OK, GEMM_ERR_TIMEOUT when a kernel's bounded barrier wait gave up
 * (the kernel released its TMEM and returned; D is undefined), or
 * GEMM_ERR_DEVICE_FAULT when the stream reports a CUDA error.
 */
int gemm_last_status(cudaStream_t stream);

/* Raw status word of the last watchdog event (0 if none) without clearing it:
 * bits 56-63 code, 48-55 wait site, 0-31 CTA index.  Synchronises `stream`. */
uint64_t gemm_last_status_word(cudaStream_t stream);

/* The CUDA runtime error (cudaError_t value) behind the calling thread's most
 * recent GEMM_ERR_LAUNCH, or 100000 + CUresult when the driver rejected a
 * tensor map; 0 if none.  Diagnostic only. */
int gemm_last_cuda_error(void);

/* Schedule of the calling thread's most recent persistent-kernel launch
 * (diagnostic, no counterpart on the pages): out[0] clusters launched,
 * out[1] CTAs per cluster, out[2] tiles computed whole (column halves
 * included), out[3] tiles split along K by the stream-K schedule, out[4]
 * K-tiles per stream-K unit, out[5] tiles of the last round cut into two
 * column halves (the tail split below), out[6] 1 when right-edge tiles were
 * dealt last (gemm_set_edge_last below).  `out` holds 7 values.  Returns
 * GEMM_OK, or GEMM_ERR_INVALID_ARG for NULL. */
int gemm_last_schedule(int64_t* out);

/* Tail split of the data-parallel schedule (b200-gemm-optimization-ladder,
 * level 6, "check the tail and tile order").  With T output tiles over G
 * co-resident clusters, the last round holds r = T mod G tiles (all T when
 * T < G) and would leave G - r clusters idle for a whole tile's time.  When
 * 2r <= G, the persistent kernels (bf16, and MXFP8 with tiled scales) cut
 * those r tiles into two halves of UMMA_N / 2 columns each, which run as
 * separate work items with N = UMMA_N / 2 MMAs: the round then takes about
 * half a tile's time.  The halves cover disjoint columns of D, so nothing is
 * summed across them and each element is computed exactly as in the whole
 * tile.  Not applied to stream-K launches that split tiles along K, nor to
 * the MXFP8 kernels with row-major scales.
 * gemm_set_tail_split(1) (the default) enables it process-wide, 0 disables
 * it; returns the previous setting, or GEMM_ERR_INVALID_ARG for another
 * value.  gemm_tail_split_plan returns the number of tiles the launchers cut
 * for `tiles` tiles over `resident` clusters under the current setting
 * (host only), or GEMM_ERR_INVALID_ARG for negative or > 2^32 - 1 inputs. */
int gemm_set_tail_split(int enable);
int64_t gemm_tail_split_plan(int64_t tiles, int64_t resident);

/* Right-edge tiles last (the same ladder level: tile order and tail).  When N
 * is not a multiple of the tile width and the last column block holds at most
 * half of it (1 <= N mod 256 <= 128), a plain bf16 launch (gemm_bf16 with no
 * epilogue, no stream-K split) orders the tiles of that block after all
 * others, runs each of them as a first column half (MMAs with N = 128), and
 * deals rounds to clusters in alternating directions: the cheap edge tiles
 * then fill the last round and land on the clusters that took full tiles
 * last, where a tail split would have cut full tiles.  No tail split is made
 * for such a launch.  Each element of D is computed as in a whole tile.
 * gemm_set_edge_last(1) (the default) enables it process-wide, 0 disables
 * it; returns the previous setting, or GEMM_ERR_INVALID_ARG for another
 * value. */
int gemm_set_edge_last(int enable);

/* Test hook for the device watchdog (no counterpart on the pages: it exists to
 * exercise the failure path without faulting a GPU).  The calling thread's NEXT
 * persistent-kernel launch (gemm_bf16/gemm_mxfp8 variants 0-2) withholds the
 * operand loads of the given K-tile iteration in every CTA, so the consumers'
 * bounded waits run out: that launch then releases its TMEM, returns, leaves D
 * undefined, and gemm_last_status() reports GEMM_ERR_TIMEOUT.  Pair it with a
 * short gemm_set_watchdog_ms().  Returns GEMM_ERR_INVALID_ARG for a negative
 * iteration. */
int gemm_debug_stall_next_launch(int64_t k_iteration);

/* Static text for a gemm_status_t value. */
const char* gemm_status_string(int status);

/* Per-wait watchdog limit in milliseconds for later launches on this process
 * (default 2000, also read once from GEMM_WATCHDOG_MS); returns the old one. */
int64_t gemm_set_watchdog_ms(int64_t ms);

/* Compile-time plan of a kernel variant, for reports: pipeline stages,
 * dynamic shared memory bytes, TMEM columns, threads per CTA, CTAs per
 * cluster, tile M and N.  mxfp8: 0 = bf16, 1 = MXFP8 (row-major scales),
 * 2 = MXFP8 with tiled scales (gemm_mxfp8_tiled).  Returns GEMM_OK or
 * GEMM_ERR_INVALID_ARG. */
int gemm_kernel_plan(int mxfp8, int variant, int32_t* stages, int32_t* smem_bytes,
                     int32_t* tmem_cols, int32_t* threads, int32_t* cluster, int32_t* tile_m,
                     int32_t* tile_n);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_GB300_H */
