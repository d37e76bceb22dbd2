/*
 * gptq_q4.h -- C ABI of the GB300 (sm_103a) fused GPTQ W4A16 linear layer.
 *
 *     y[M][N] = x[M][K] . W[K][N] + bias[N]
 *
 * W is a GPTQ (v1) 4-bit weight matrix:
 *   qweight  int32 [K/8][N]   eight 4-bit codes per word along K, code k%8 in
 *                             bits 4(k%8) .. 4(k%8)+3 (lowest nibble first)
 *   qzeros   int32 [G][N/8]   eight 4-bit zero points per word along N, same
 *                             nibble order
 *   scales   fp16  [G][N]     one scale per (group, column)
 *   g_idx    int32 [K]        group of each row (act-order), or NULL
 *   w[k][n] = scales[g][n] * (q[k][n] - (z[g][n] + 1)),  g = g_idx[k]
 *             (g = k / groupsize when g_idx is NULL; G = K / groupsize, or
 *              G = 1 and one group over all of K when groupsize == -1)
 *
 * Sources (web pages; sections named):
 *   "GPTQ's 'Exllama Kernel Not Installed' Warning" -- "Why the kernel is
 *     missing" (4-bit integers packed in 32-bit words, a scale and a zero per
 *     group) and "What the fallback actually does" (the fused kernel reads
 *     packed weights, dequantizes in registers and never writes a dequantized
 *     matrix; the fallback rebuilds W and runs an ordinary matmul, reaching the
 *     same answer with several times the memory traffic).
 *   "Implementation: Predibase Lorax GPTQ Exllama V1" -- "Description" (a
 *     Q4Matrix handle built from qweight, qzeros, scales and optional g_idx;
 *     q4_matmul computes x @ q4 into a (batch, width) fp16 output; temp_state
 *     reorders activations for act-order; temp_dq holds dequantized weights
 *     for the prefill matmul; create_exllama_buffers sizes both) and "I/O
 *     Contract" (dtypes; bits must be 4; None or trivial g_idx = no act-order).
 *   "Inference Backends" -- "Packing, conversion, and runtime initialization"
 *     (runtime init repacks into a private execution layout and builds native
 *     handles), "Numeric epilogues and input gradients" (bias joins the fp32
 *     accumulator before the one final cast; split reductions stay fp32;
 *     no atomic partial-output reduction), "Strided tensor operands" (one
 *     stable argsort gives the reorder; an identity permutation skips the
 *     gather), "Runtime cache lifetime" (no dense weight cache is kept
 *     between operations).
 *
 * Conventions for every entry point:
 *   - Pointers marked "device" must be CUDA device (or managed) memory of the
 *     device that is current when the call is made; "host" means host memory.
 *     Arrays are dense and row-major; fp16 values are passed as their 16-bit
 *     patterns (uint16_t).
 *   - Every call except gptq_q4_make returns GPTQ_Q4_OK (0) or a negative
 *     status.  gptq_q4_make returns NULL on failure.  The status and a message
 *     with the specific reason are kept per host thread and read back with
 *     gptq_q4_last_status() / gptq_q4_last_error().  Nothing is ever printed,
 *     and no call silently falls back to another route: there is no CPU path.
 *   - Work is enqueued on the caller's stream and the calls return without
 *     waiting, except gptq_q4_make, gptq_q4_reserve, gptq_q4_free and
 *     gptq_q4_device_error, which synchronize as stated.
 *   - A handle may be used from one stream at a time (its workspaces are
 *     reused by every call).  Distinct handles are independent.
 */
#ifndef GPTQ_Q4_H
#define GPTQ_Q4_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ status codes */
#define GPTQ_Q4_OK                 0
#define GPTQ_Q4_INVALID_ARGUMENT (-1) /* NULL, bad sizes, g_idx out of range, misalignment */
#define GPTQ_Q4_UNSUPPORTED      (-2) /* valid GPTQ data outside what the GPU kernels take,
                                         or a device that is not sm_103 */
#define GPTQ_Q4_CUDA_ERROR       (-3) /* a CUDA runtime call failed; message holds its text */
#define GPTQ_Q4_OUT_OF_MEMORY    (-4) /* a device allocation failed */
#define GPTQ_Q4_DEVICE_FAULT     (-5) /* a kernel reported an error through its status word */

/* Paths gptq_q4_matmul can take (see gptq_q4_set_path). */
#define GPTQ_Q4_PATH_AUTO      0  /* decode below the prefill threshold, fused prefill above */
#define GPTQ_Q4_PATH_DECODE    1  /* always decode: the stream-K kernel on tall layers of 100 Mi
                                     weights or more that the column tiles cannot fill (K >= 2 N,
                                     fewer than two 32-column tiles per SM) at M = 1 with groups of
                                     at most 128 rows, at M = 2 with 32-row groups and at M = 3..8
                                     with groups of 128 rows or more; otherwise the
                                     register-streaming kernel at M <= 4, at M <= 8 on layers below
                                     64 Mi weights or with groups of at most 64 rows, and on any
                                     layer below 24 Mi weights; the TMA-ring kernel (M <= 16)
                                     elsewhere, where the shape allows it */
#define GPTQ_Q4_PATH_PREFILL   2  /* always the fused shared-memory-dequant tensor-core kernel */
#define GPTQ_Q4_PATH_DECODE_MMA 3 /* always the register-streaming decode kernel */
#define GPTQ_Q4_PATH_DECODE_TC 4  /* decode on tcgen05 with one tensor-memory accumulator per
                                     quantization group (M <= 16 on 4-bit handles with fp16
                                     activations; otherwise as GPTQ_Q4_PATH_DECODE) */
#define GPTQ_Q4_PATH_DECODE_RING 5 /* the TMA-ring decode kernel whenever the shape allows it
                                      (M <= 16, a K slice within 48 groups), else
                                      register-streaming */
#define GPTQ_Q4_PATH_DECODE_STREAM 6 /* the stream-K decode kernel (M <= 8): every warp of the
                                        grid streams an equal run of 32-column x 64-row units,
                                        quantization groups ride in the MMAs' spare columns;
                                        larger M as GPTQ_Q4_PATH_DECODE */

typedef struct gptq_q4_s *gptq_q4_handle;   /* opaque; owns device memory */

/* Build a handle (the Q4Matrix of the Lorax page's "Description": make_q4).
 *
 *   qweight  device int32 [K/8][N]
 *   qzeros   device int32 [G][N/8]
 *   scales   device fp16  [G][N]
 *   g_idx    device int32 [K], or NULL for the trivial map k / groupsize
 *   groupsize  > 0 dividing K, or -1 for one group over all of K
 *
 * Validates the arguments; copies g_idx to the host, checks every entry is in
 * [0, G), and derives the act-order row permutation P with one stable argsort
 * (rows sorted by group, original order kept within a group).  An identity P
 * means no act-order.  When the groups do not all hold the same whole number
 * of 32-row blocks (g_idx with groups of unequal size, or a groupsize that is
 * not a multiple of 32), every group is padded to the largest one rounded up
 * to 32 rows: the padding rows hold code 0 and P = -1, and the activation
 * gather writes 0 for them, so they add nothing to y.  Then repacks the codes,
 * in P order, into a private tile-ordered layout (same byte count as qweight
 * without padding), and the scales into a private pairing; zero points keep
 * the checkpoint layout.  All of it is
 * copied into handle-owned device memory, so the caller may free or change its
 * tensors afterwards.  Also sizes the split-K workspace for M <= 16.
 * Synchronizes the device before returning.  The caller must have finished
 * writing the input tensors (e.g. synchronized its stream) before the call.
 *
 * Errors (NULL return; reason in gptq_q4_last_error):
 *   INVALID_ARGUMENT  NULL qweight/qzeros/scales, K or N <= 0, K % 8 or N % 8
 *                     != 0, groupsize not -1 and not a positive divisor of K,
 *                     a g_idx entry outside [0, G), a pointer that is not
 *                     device memory of the current device
 *   UNSUPPORTED       K % 64 or N % 64 != 0; groups whose padding to the
 *                     largest one would make the layout more than 4 x K
 *                     rows; current device is not compute 10.3
 *   OUT_OF_MEMORY, CUDA_ERROR */
gptq_q4_handle gptq_q4_make(const int32_t *qweight, const int32_t *qzeros,
                            const uint16_t *scales, const int32_t *g_idx,
                            int K, int N, int groupsize);

/* Attach (or with NULL, detach) a bias: device fp16 [N], copied into the
 * handle.  Bias is added to the fp32 accumulator before the single rounding
 * to fp16 ("Inference Backends", "Numeric epilogues and input gradients").
 * Enqueued on the legacy default stream and synchronized before returning.
 * Errors: INVALID_ARGUMENT (NULL handle), OUT_OF_MEMORY, CUDA_ERROR. */
int gptq_q4_set_bias(gptq_q4_handle h, const uint16_t *bias);

/* Size the handle's work buffers for calls with up to max_m rows: the
 * act-order activation buffer temp_state [max_m][K] fp16 and the split-K
 * partial sums.  The counterpart of the Lorax page's create_exllama_buffers
 * (max_total_tokens).  A later gptq_q4_matmul with more rows grows the buffers
 * itself (stream-ordered allocation on the caller's stream); calling this
 * first keeps allocation out of gptq_q4_matmul.  Synchronizes the device.
 * Errors: INVALID_ARGUMENT (NULL handle, max_m < 0), OUT_OF_MEMORY. */
int gptq_q4_reserve(gptq_q4_handle h, int max_m);

/* out = x . W + bias  (q4_matmul; the Lorax page's "Description").
 *
 *   x    device [M][K] of the handle's activation type (fp16 by default;
 *        bf16 or fp32 after gptq_q4_set_act_dtype), 16-byte aligned
 *   out  device [M][N] of the same type, 16-byte aligned; written entirely,
 *        never read
 *   M    rows; 0 is a valid no-op
 *
 * With act-order, x is first gathered into temp_state (temp_state[m][j] =
 * x[m][P[j]]).  Rows below the prefill threshold run one of two decode
 * kernels (GPTQ_Q4_PATH_DECODE says which).  The TMA-ring kernel (M <= 16):
 * packed-word tiles and x tiles stream through a ring of shared-memory
 * stages by TMA; each warp owns 32 columns for a whole K slice, turns code
 * pairs into fp16 with one LOP3 each and accumulates on mma.sync in fp32,
 * the zero point removed per group from MMA-accumulated sums of x; the K
 * slices of a 128-column tile (at most 8) are summed in slice order inside a
 * thread-block cluster.  The register-streaming kernel: packed weights
 * streamed with 128-bit loads, through a per-warp ring of asynchronous
 * copies in shared memory at M <= 8 (x staged once per CTA, or carried with
 * each chunk when the x slice is long) and straight into registers above,
 * exact (q - z - 1) in fp16 (or raw code pairs with per-group sums of x),
 * fp32 accumulation on mma.sync, split-K summed in a fixed order inside a
 * cluster or, past eight slices, by the last CTA to finish.
 * GPTQ_Q4_PATH_DECODE_TC selects the
 * tcgen05 decode instead (M <= 16): packed weights streamed by TMA,
 * dequantized in shared memory to the exact integers (q - z - 1), one
 * tensor-memory accumulator per quantization group, scales applied once per
 * group in an fp32 epilogue.
 * Larger M runs the fused prefill (tcgen05/TMEM with shared-memory
 * dequantization).  Results do not depend on the path beyond fp32 rounding.
 * Errors: INVALID_ARGUMENT (NULL handle/pointers with M > 0, M < 0,
 * misaligned x or out, handle made on another device), OUT_OF_MEMORY (growing
 * a work buffer), CUDA_ERROR (launch failure). */
int gptq_q4_matmul(gptq_q4_handle h, const void *x, int M, void *out,
                   cudaStream_t stream);

/* temp_dq[k][n] = fp16(scales[g][n] * (q[k][n] - (z[g][n] + 1))), rounded
 * once to nearest-even, in the ORIGINAL row order (the permutation is undone
 * on write).  The dequantized matrix of the Lorax page's "Description"
 * (temp_dq), used for debugging and by the unfused prefill comparison.
 *   temp_dq  device fp16 [K][N], 16-byte aligned, caller-owned: the handle
 *            keeps no dense copy ("Runtime cache lifetime").
 * Errors: INVALID_ARGUMENT, CUDA_ERROR. */
int gptq_q4_dequant(gptq_q4_handle h, uint16_t *temp_dq, cudaStream_t stream);

/* The unpacked codes, read back from the handle's private layout (a debug
 * read-back; no passage of the pages defines it: "Inference Backends",
 * "Packing, conversion, and runtime initialization" only says runtime
 * initialization may repack into a private layout, and this call shows that
 * the repack kept every code):
 *   q  device uint8 [K][N], q[k][n] in 0..15, ORIGINAL row order
 *   z  device uint8 [G][N], stored zero points (without the +1)
 * Either pointer may be NULL to skip it.  For checking the repack bit-exactly.
 * Errors: INVALID_ARGUMENT, CUDA_ERROR. */
int gptq_q4_debug_unpack(gptq_q4_handle h, uint8_t *q, uint8_t *z, cudaStream_t stream);

/* The unfused comparison route ("What the fallback actually does", with the
 * matmul on the tensor cores): gptq_q4_dequant into the caller's temp_dq, then
 * out = x . temp_dq + bias by the tcgen05 GEMM below.  Same arguments as
 * gptq_q4_matmul plus temp_dq (device fp16 [K][N], caller-owned scratch).
 * Errors: as gptq_q4_matmul and gptq_q4_dequant. */
int gptq_q4_matmul_unfused(gptq_q4_handle h, const void *x, int M,
                           uint16_t *temp_dq, void *out, cudaStream_t stream);

/* Dense fp16 GEMM on the 5th-generation tensor cores (tcgen05, accumulators
 * in tensor memory, operands staged by TMA): out = a . b + bias with fp32
 * accumulation and one rounding to fp16.  The matmul the Lorax page runs on
 * temp_dq "during prefill".
 *   a     device fp16 [M][K] row-major, b device fp16 [K][N] row-major,
 *   bias  device fp16 [N] or NULL, out device fp16 [M][N];
 *   all 16-byte aligned; K % 64 == 0, N % 64 == 0, M >= 0.
 * Errors: INVALID_ARGUMENT, UNSUPPORTED (sizes), CUDA_ERROR. */
int gptq_q4_gemm_f16(const uint16_t *a, const uint16_t *b, const uint16_t *bias,
                     int M, int K, int N, uint16_t *out, cudaStream_t stream);

/* Bytes of the fixed device scratch used by gptq_q4_matmul_noalloc (16 MiB). */
#define GPTQ_Q4_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/* out = x . W + bias through the decode kernel, allocating nothing.
 *
 * The web pages this library follows have no counterpart for this call.  It
 * is for callers that cannot allocate device memory while they run a layer:
 * a plugin inside a framework that owns all device memory, a service whose
 * device memory is budgeted in full up front, a loop that must never hit
 * cudaMalloc/cudaFree (which can synchronize the device).  gptq_q4_matmul may
 * grow the handle's work buffers; this call never allocates or frees.
 *
 * It runs the decode kernel (any M) with its scratch -- split-K partial sums,
 * per-tile tickets and, for act-order, temp_state -- taken from one static
 * device array of GPTQ_Q4_NOALLOC_SCRATCH_BYTES bytes that every GPU loading
 * the library holds until the process exits.  Arguments, layouts and results
 * are those of gptq_q4_matmul (x, out: device fp16, 16-byte aligned).
 *
 *   - The first call in each CUDA context does a one-time set-up: it looks
 *     up the array's device address with cudaGetSymbolAddress, with the
 *     handle's device current, and keeps it keyed by the context's unique ID
 *     (the primary context, or one the caller made current).  A context made
 *     after cudaDeviceReset is a new context and gets its own set-up.  Make
 *     the first call in a context before any stream capture.
 *   - All calls share the one array, which keeps the last call's contents;
 *     the call clears what must start at zero (the tickets) on its stream.
 *     Calls that overlap on the GPU (other streams, other handles, other
 *     threads) race on the array: order them, e.g. use one stream.
 *   - Errors: as gptq_q4_matmul, plus INVALID_ARGUMENT when M (with this
 *     layer's K and N) would need more scratch than the array holds; the
 *     message gives both sizes. */
int gptq_q4_matmul_noalloc(gptq_q4_handle h, const uint16_t *x, int M, uint16_t *out,
                           cudaStream_t stream);

/* Force a path for gptq_q4_matmul (tests, benchmarks): GPTQ_Q4_PATH_*. */
int gptq_q4_set_path(gptq_q4_handle h, int path);

/* GPU packer ("Inference Backends", "Packing, conversion, and runtime
 * initialization": packing takes the original layer's weights with the
 * quantizer's scales, zeros and optional act-order index; a GPU path does the
 * packing math; symmetric modules without zeros use 2^(bits-1)).
 *   w       dev [K][N] fp16, the float weights (row k = input feature k)
 *   scales  dev [G][N] fp16
 *   zeros   dev [G][N] int32 effective zero points (0..15), or NULL: all 8
 *   g_idx   dev [K] int32 group of each row, or NULL: k / groupsize
 *   format  GPTQ_Q4_FORMAT_GPTQ (stores z - 1) or GPTQ_Q4_FORMAT_GPTQ_V2 (z)
 *   qweight dev [K/8][N] int32 out, qzeros dev [G][N/8] int32 out
 * Code q = clamp(rint(w / s) + z, 0, 15) with w / s the IEEE binary32
 * quotient, ties to even (0/0 gives z); qweight and qzeros in the
 * checkpoint layout gptq_q4_make reads; stored zeros are taken mod 16.
 * Asynchronous on `stream` once its arguments are checked (g_idx is copied to
 * the host for the range check).  Errors: INVALID_ARGUMENT (NULL, sizes,
 * groupsize, format, g_idx out of [0, G), non-device pointers), CUDA_ERROR. */
int gptq_q4_pack(const uint16_t *w, const uint16_t *scales, const int32_t *zeros, const int32_t *g_idx, int K,
                 int N, int groupsize, int format, int32_t *qweight, int32_t *qzeros, cudaStream_t stream);

/* Test hook for failure detection (the pages have no counterpart).  The TMA
 * and tcgen05 kernels bound every mbarrier wait: a wait that runs out sets
 * a bit in the handle's status word (reported by gptq_q4_device_error) and
 * the kernel returns instead of hanging.  This launches one CTA whose thread
 * runs that same wait, limited to limit_us microseconds (1 .. 2,000,000), on
 * an mbarrier that nothing arrives at; when the limit runs out it ORs 1 into
 * *status (a device int the caller owns and zeroes).  Asynchronous on
 * `stream`.  Errors: INVALID_ARGUMENT (NULL status, limit out of range),
 * CUDA_ERROR (launch). */
int gptq_q4_debug_wait_probe(int *status, unsigned limit_us, cudaStream_t stream);

/* Test hook, host only (no device call): the work split that the fused
 * prefill ("Inference Backends", "How AUTO selection works": the prefill
 * path for larger M) plans for an M x K x N call on a GPU with `sms` SMs.
 * out[0..6] (caller-owned host ints) = tile rows BM, tile columns BN,
 * stream-K (1) or whole tiles round robin (0), CTAs of the stream-K launch
 * (0 for round robin), the most pieces any tile is cut into, whether each
 * cut tile is finished by the CTA holding its first k blocks (1) or by every
 * piece's CTA, a share of the rows each (0), and the rows of K per pipeline
 * stage (64, or 128).  Errors: INVALID_ARGUMENT
 * (NULL out, M < 1, K or N not a positive multiple of 64, sms < 1). */
int gptq_q4_debug_prefill_plan(int M, int K, int N, int sms, int *out);

/* Test hook, host only (no device call): the kernel that gptq_q4_matmul runs
 * for M fp16 rows on a K x N layer with this group size (-1: one group; no
 * padding, GPTQ zero points), with `path` as the handle's
 * GPTQ_Q4_PATH_* setting (AUTO resolved by the default prefill threshold)
 * on a GPU with `sms` SMs.  *kernel (caller-owned host int) = 0 the fused
 * prefill, 1 the register-streaming decode, 2 the stream-K decode, 3 the
 * TMA-ring decode, 4 the tcgen05 decode.  Errors: INVALID_ARGUMENT (NULL
 * kernel, M < 1, K or N not a positive multiple of 64, a group size that is
 * not -1 or a multiple of 32 dividing K, sms < 1, an unknown path). */
int gptq_q4_debug_dispatch(int M, int K, int N, int groupsize, int path, int sms, int *kernel);

/* Projection fusion ("Inference Backends", "How AUTO selection works":
 * post-quantization QKV or gate/up projections that read the same input are
 * combined into one call).  One handle over `parts` GPTQ layers that share
 * K, groupsize and g_idx, concatenated along N in the given order:
 *   qweight[i] dev [K/8][N[i]], qzeros[i] dev [G][N[i]/8], scales[i] dev
 *   [G][N[i]] fp16, N[i] a positive multiple of 8, sum of N[i] a multiple of
 *   64 (the handle's N); g_idx as for gptq_q4_make, shared by all parts.
 * gptq_q4_matmul on the handle writes out [M][sum N[i]]: part i occupies
 * columns [sum_{j<i} N[j], + N[i]) of each row (views of one buffer, no copy);
 * a bias set with gptq_q4_set_bias is the parts' biases concatenated the same
 * way.  The parts' tensors are copied; the caller may free them on return.
 * Returns NULL on error (status and message as for gptq_q4_make). */
#define GPTQ_Q4_MAX_FUSED_PARTS 16
gptq_q4_handle gptq_q4_make_fused(int parts, const int32_t *const *qweight, const int32_t *const *qzeros,
                                  const uint16_t *const *scales, const int32_t *g_idx, int K, const int *N,
                                  int groupsize);

/* Checkpoint zero-point convention of a handle ("Inference Backends",
 * "Concepts": GPTQ and GPTQ_V2 are distinct checkpoint formats).  The two
 * store qweight, qzeros and scales in the same layout and differ in the
 * zero point: GPTQ keeps z_eff - 1 in qzeros, so w = s * (q - (z + 1));
 * GPTQ_V2 keeps z_eff itself, so w = s * (q - z).  Default GPTQ.  Changes
 * what later matmul/dequant calls compute; the handle's other state is
 * untouched.  Errors: INVALID_ARGUMENT (NULL handle, unknown format). */
#define GPTQ_Q4_FORMAT_GPTQ    0
#define GPTQ_Q4_FORMAT_GPTQ_V2 1
int gptq_q4_set_format(gptq_q4_handle h, int format);

/* Type of x and out for later matmul calls on this handle ("Inference
 * Backends", "Hardware, dependency, and format requirements": the ExLlama v2
 * row declares FP16/BF16/FP32 activation dtypes, keeps the activation/output
 * dtype, fp16 scales and fp32 accumulation).  Default FP16.  bias stays the
 * handle's fp16.
 *   BF16: x and out are bf16 [M][K] / [M][N]; every row of x is first scaled
 *     by a power of two 2^-e (its largest magnitude times 2^-e in [2^14,
 *     2^15)) and rounded once to fp16 (exact for values within ~2^28 of the
 *     row's largest: bf16 has an 8-bit significand), the fp16 kernels run
 *     unchanged, and each output is acc * 2^e + bias rounded once to bf16.
 *     Covers gptq_q4_matmul, gptq_q4_matmul_unfused and
 *     gptq_q4_matmul_noalloc; one extra launch per call prepares x (fused
 *     with the act-order gather).
 *   FP32: x and out are fp32 [M][K] / [M][N]; every row is scaled by 2^-e
 *     as above and split into two fp16 rows, hi = fp16(v) and lo = fp16(v -
 *     hi) (v - hi is exact, so hi + lo carries v to about 2^-22 of itself);
 *     the fp16 kernels run on the 2M rows and write their raw fp32 sums, and
 *     a last launch forms out = (sum_hi + sum_lo) * 2^e + bias in fp32 (no
 *     rounding to a narrower type).  Covers gptq_q4_matmul and
 *     gptq_q4_matmul_unfused (two extra launches per call);
 *     gptq_q4_matmul_noalloc returns UNSUPPORTED for an FP32 handle.
 * Errors: INVALID_ARGUMENT (NULL handle, unknown dtype). */
#define GPTQ_Q4_DTYPE_FP16 0
#define GPTQ_Q4_DTYPE_BF16 1
#define GPTQ_Q4_DTYPE_FP32 2
int gptq_q4_set_act_dtype(gptq_q4_handle h, int dtype);

/* Rows at and above which GPTQ_Q4_PATH_AUTO takes the prefill kernel (the
 * decode/prefill switch of the Lorax page's set_tuning_params).  Default 17,
 * or 9 for groups of at most 32 rows and for groups of at most 64 rows on
 * layers of 100 Mi weights or more: measured on GB300, the fused prefill is
 * faster than the decode kernels from there.  Results never depend on it. */
int gptq_q4_set_prefill_min_m(gptq_q4_handle h, int min_m);

/* Facts about a handle (host outputs; any pointer may be NULL). */
int gptq_q4_info(gptq_q4_handle h, int *K, int *N, int *groupsize, int *G,
                 int *act_order, size_t *device_bytes);

/* Synchronize the handle's device and return GPTQ_Q4_DEVICE_FAULT if any
 * kernel of this handle has set its status word (a bounded wait that ran out,
 * a failed internal check), else GPTQ_Q4_OK.  Clears the word. */
int gptq_q4_device_error(gptq_q4_handle h);

/* Release everything the handle owns (synchronizes its device).  NULL is a
 * no-op.  Lifecycle only; the pages' nearest passage is "Inference
 * Backends", "Runtime cache lifetime" (native runtime storage belongs to the
 * handle, and nothing outlives it). */
void gptq_q4_free(gptq_q4_handle h);

/* Q4Matrix handle for an 8-bit GPTQ layer.  "Inference Backends",
 * "Hardware, dependency, and format requirements": the GPTQ Marlin row
 * declares bits 4 and 8, and the Swordfish row says GPTQ supports 4/8-bit.
 * The pages print no 8-bit layout; this library reads it as the 4-bit
 * GPTQ packing with 32 / 8 = 4 codes per int32:
 *   qweight  device int32 [K/4][N]   four 8-bit codes per word along K,
 *                                   lowest byte = lowest row
 *   qzeros   device int32 [G][N/4]   four 8-bit zero points per word along N
 *   scales   device fp16  [G][N], |scale| < 4094
 *   g_idx, groupsize as for gptq_q4_make
 * w[k][n] = scales[g][n] * (q[k][n] - (z[g][n] + 1)) (GPTQ; GPTQ_V2 after
 * gptq_q4_set_format: q - z).  With q = 16 qh + ql and z = 16 zh + zl,
 * s (q - z - 1) = 16 s (qh - zh) + s (ql - zl - 1) exactly, so the handle
 * holds a 4-bit layer over 2K rows (the high nibbles with scale 16 s and zero
 * offset 0, then the low nibbles with scale s) whose two halves read the same
 * column of x; every matmul path, gptq_q4_dequant and gptq_q4_debug_unpack
 * (8-bit codes and zero points, one byte each) work as for 4-bit handles,
 * with twice the packed bytes.  gptq_q4_info reports the caller's K and G.
 * Errors as for gptq_q4_make. */
gptq_q4_handle gptq_q4_make8(const int32_t *qweight, const int32_t *qzeros,
                             const uint16_t *scales, const int32_t *g_idx,
                             int K, int N, int groupsize);

/* Status and message of the last call made on this host thread.
 * "Inference Backends", "Hardware, dependency, and format requirements":
 * device-validation errors keep the kernel's specific reason (an unsupported
 * compute capability, a missing kernel image) instead of a generic one; the
 * message names the argument or limit that failed. */
int gptq_q4_last_status(void);
const char *gptq_q4_last_error(void);

/* Number of kernels this library has launched in this process. */
uint64_t gptq_q4_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* GPTQ_Q4_H */
