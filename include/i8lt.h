/*
 * i8lt.h -- C ABI of the GB300 (sm_103a) int8 quantized linear layer.
 *
 * The layer is the memory-efficient Linear8bitLt of bitsandbytes PR #33
 * "Memory efficient backward":
 *   - weights live as row-major int8 codes CB [N, K] with one fp32 absmax per
 *     output row SCB [N] (PR description, "Stores int8 weights in row-major
 *     format");
 *   - the forward casts A to fp16, quantizes it row-wise (vector-wise absmax),
 *     takes columns with an element above the outlier threshold out as subA and
 *     multiplies them in fp16 against the matching weight columns subB
 *     (review thread, "4. Mixed-precision decomposition matmul"), dequantizes,
 *     adds the bias and casts back to A's dtype (PR description, "Cast inputs
 *     and outputs of the 8bit layer to fp16 and back");
 *   - the backward rebuilds fp16 weights CB * (SCB * (1/127)) inside the GEMM
 *     and never stores them (PR description, backward bullet; review thread on
 *     ".mul(1/127.0)"), and sums grad_bias from the uncast grad_output (PR
 *     conversation, "grad_bias is now computed on natural grad_output").
 * Beside it: the MLP's SiLU (with an optional fusion into the forward
 * epilogue), a token-sharded forward, the weight gradient of the
 * trainable-weight mode, the 4-bit (NF4 and FP4) weight-only layers of QLoRA
 * fine-tuning, an entry point that allocates nothing, per-launch timing and
 * a diagnostic of the bounded waits (each documented below).
 *
 * Conventions for every entry point:
 *   - Matrices are row-major and contiguous.  Device pointers unless stated.
 *     Base pointers of matrices must be 16-byte aligned.
 *   - The caller owns every buffer, including the workspace.  The library
 *     allocates no device memory.
 *   - `stream` is a cudaStream_t passed as void*.  Work is asynchronous on it;
 *     nothing synchronizes except i8lt_read_device_status and
 *     i8lt_noalloc_read_device_status.
 *   - Errors found on the host are returned before anything is launched.
 *     Errors found on the device (outlier capacity exceeded, a pipeline wait
 *     that timed out) are written to the status word at the start of the
 *     workspace, which every forward / backward call clears when it starts;
 *     the outputs of that call are then unspecified.
 *   - No C++ exception crosses this boundary.
 */
#ifndef I8LT_H_
#define I8LT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  I8LT_OK = 0,
  I8LT_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad shape */
  I8LT_ERR_UNSUPPORTED_DTYPE = 2, /* dtype not in i8lt_dtype */
  I8LT_ERR_MISALIGNED = 3,        /* a matrix base pointer is not 16-byte aligned */
  I8LT_ERR_WORKSPACE = 4,         /* workspace null or smaller than required */
  I8LT_ERR_K_TOO_LARGE = 5,       /* int32 accumulator could overflow */
  I8LT_ERR_OUTLIER_CAPACITY = 6,  /* device: more outlier columns than max_outliers */
  I8LT_ERR_TIMEOUT = 7,           /* device: a pipeline wait ran out of time */
  I8LT_ERR_CUDA = 8,              /* a CUDA runtime / driver call failed */
  I8LT_ERR_DEVICE = 9,            /* the current device is not sm_103 */
  I8LT_ERR_SCRATCH_LIMIT = 10     /* the problem needs more scratch than the
                                     static buffer of the no-alloc entry point */
} i8lt_status;

typedef enum { I8LT_F16 = 0, I8LT_BF16 = 1, I8LT_F32 = 2 } i8lt_dtype;

/* Largest in_features for which K * 127 * 127 < 2^31 (exact int32 sums). */
#define I8LT_MAX_K 133144

/* Version of this ABI; bumped on any incompatible change (3: the 4-bit
 * input gradients take grad_bias; 4: the double-quantized absmax entry
 * points and their kernel id, I8LT_K_COUNT = 21). */
int i8lt_abi_version(void);

/* Human-readable name of a status code (static storage). */
const char* i8lt_status_string(int status);

/* Leading dimension (elements) of the int8 weight CB for in_features K:
 * K rounded up to a multiple of 16, so that every row starts on 16 bytes. */
int64_t i8lt_weight_ld(int64_t K);

/*
 * Weight quantization (once per weight; "memory_efficient_backward" keeps
 * only CB and SCB, the fp16 weight is not kept).
 *   W    [N, K] in dtype `wt` (read only)
 *   CB   [N, i8lt_weight_ld(K)] int8 (written; columns >= K are set to 0)
 *   SCB  [N] fp32 (written)
 * W16 = fp16_rn(W); SCB[n] = max_k |W16[n,k]|;
 * CB[n,k] = round_half_even(fp32(W16[n,k]) * (127 / SCB[n])) in IEEE fp32,
 * 0 for a row whose absmax is 0.
 */
int i8lt_quantize_weight(const void* W, int wt, int64_t N, int64_t K,
                         int8_t* CB, float* SCB, void* stream);

/* Workspace of i8lt_forward, in bytes.  max_outliers is the capacity for
 * outlier columns (0 when the threshold disables the decomposition). */
size_t i8lt_forward_workspace_size(int64_t M, int64_t K, int64_t N,
                                   int64_t max_outliers);

/* Byte offsets of the regions of the forward workspace (for tests and
 * debugging; every region is 256-byte aligned):
 *   status  int32[4]: {status, outlier count found, count used, spare}
 *   colmax  uint32[K]: per column, fp16 bits of max_m |A16[m,k]|
 *   mask    uint32[ceil(K/32)]: bit k set when column k is an outlier
 *   idx     int32[cap_pad]: ascending outlier column indices
 *   SCA     fp32[M]: row absmax of A16 outside the outlier columns
 *   asq     uint32[ceil(M/256), nch]: per 256-row tile and 1024-column chunk
 *                      (nch = ceil(K_pad/1024)), the largest sum of squared
 *                      codes of a row of the tile in that chunk
 *   bsq     uint32[ceil(N/256), nch]: the same for the weight's code rows
 *   plan    uint32[ceil(M/256) * ceil(N/256)]: per tile pair, the chunks per
 *                      exact fp32 accumulation unit (bits 0-15; a group of
 *                      chunks G qualifies when sum_G asq * sum_G bsq < 2^48,
 *                      which bounds every partial sum below 2^24 by
 *                      Cauchy-Schwarz) and bit 16 set when every unit stays
 *                      below 2^22
 *   Aq      fp16[M, K_pad]: the int8 codes of A, stored as exact fp16 integers
 *                           (the form the fp16 tensor cores read)
 *   subA    fp16[M, cap_pad]: A16[:, idx], zero past the count
 *   subB    fp16[N, cap_pad]: dequantized weight columns W_dq[:, idx]
 *   CBh     fp16[N, K_pad]: the weight's int8 codes as exact fp16 values,
 *                           rebuilt on every call (the operand form the
 *                           tensor-core pipeline loads)
 * cap = min(max_outliers, K); cap_pad = cap rounded up to a multiple of 64. */
typedef struct {
  size_t status, asq, bsq, colmax, mask, idx, sca, plan, aq, suba, subb, cbh, total;
  int64_t k_pad, cap_pad;
} i8lt_fwd_layout;
int i8lt_forward_workspace_layout(int64_t M, int64_t K, int64_t N,
                                  int64_t max_outliers, i8lt_fwd_layout* out);

/* Optional extra outputs of the forward for parity checks.  Any field may be
 * NULL.  acc_i32 [M, N] receives the exact int32 accumulator
 * sum_k Aq[m,k] * CB[n,k] of the int8 part. */
typedef struct {
  int32_t* acc_i32;
} i8lt_fwd_debug;

/*
 * Forward: out = to_dtype(at)( Cacc[m,n] * SCA[m] * SCB[n] / 127^2
 *                             + sum_j subA[m,j] * subB[n,j]
 *                             + bias[n] + residual[m,n] )
 *   A        [M, K] dtype `at` in {f16, bf16, f32}; cast to fp16 first
 *   CB, SCB  from i8lt_quantize_weight (CB leading dimension i8lt_weight_ld(K))
 *   bias     [N] dtype `bt`, or NULL
 *   residual [M, N] dtype `at`, or NULL (added before the single rounding)
 *   threshold outlier threshold: column k is an outlier when some row has
 *            |A16[m,k]| > threshold; a value that is not a positive finite
 *            number disables the decomposition
 *   out      [M, N] dtype `at`
 *   ws       workspace of at least i8lt_forward_workspace_size bytes,
 *            256-byte aligned
 *   max_outliers capacity for outlier columns; more columns than this sets
 *            I8LT_ERR_OUTLIER_CAPACITY in the device status word
 *   dbg      optional debug outputs, or NULL
 * Returns I8LT_ERR_K_TOO_LARGE for K > I8LT_MAX_K.
 */
int i8lt_forward(const void* A, int at, int64_t M, int64_t K,
                 const int8_t* CB, const float* SCB, int64_t N,
                 const void* bias, int bt, float threshold,
                 const void* residual, void* out,
                 void* ws, size_t ws_bytes, int64_t max_outliers,
                 const i8lt_fwd_debug* dbg, void* stream);

/*
 * i8lt_forward_silu -- i8lt_forward for the hidden layer of an MLP (Dense ->
 * SiLU -> Dense), with the SiLU and the next layer's outlier detection fused
 * into the GEMM epilogue:
 *   out        [M, N] dtype `at`: the layer's output h, as i8lt_forward
 *   act        [M, N] dtype `at`: silu(h) computed from the stored h with
 *              the same arithmetic as i8lt_silu_forward (bit-identical)
 *   act_colmax [N] uint32, device: cleared by the call, then set to the
 *              per-column maxima of |fp16(act)| as fp16 bit patterns -- the
 *              column maxima step of the next layer's forward.  Pass the
 *              colmax region of the next layer's workspace
 *              (i8lt_fwd_layout.colmax) and run that layer with
 *              i8lt_forward_from_colmax: the pass of the standalone SiLU
 *              kernel and the next layer's column-maxima pass are saved.
 * Other arguments and errors as i8lt_forward; act 16-byte aligned,
 * act_colmax 4-byte aligned, neither may be NULL.
 */
int i8lt_forward_silu(const void* A, int at, int64_t M, int64_t K,
                      const int8_t* CB, const float* SCB, int64_t N,
                      const void* bias, int bt, float threshold,
                      const void* residual, void* out, void* act, uint32_t* act_colmax,
                      void* ws, size_t ws_bytes, int64_t max_outliers,
                      const i8lt_fwd_debug* dbg, void* stream);

/*
 * Token-sharded forward (one batch whose rows are split over several ranks,
 * each with its own workspace).  The outlier columns are a property of the
 * whole batch (a column is an outlier when some row of the batch exceeds the
 * threshold), so the ranks exchange one K-sized vector before quantizing:
 *   1. i8lt_forward_colmax: clears the workspace's status word and column
 *      maxima, then writes the column maxima of |fp16(A)| over this rank's M
 *      rows (M may be 0) into the colmax region of `ws`
 *      (i8lt_fwd_layout.colmax: K uint32 values, the fp16 bit pattern of
 *      each magnitude; integer order = magnitude order).  Arguments as in
 *      i8lt_forward (N and max_outliers size the workspace).
 *   2. the caller combines the K values of all ranks with an element-wise
 *      maximum (e.g. an all-reduce MAX over the region viewed as int32) and
 *      writes the result back into every rank's region;
 *   3. i8lt_forward_from_colmax: i8lt_forward on this rank's rows, taking the
 *      colmax region as given instead of computing it.
 * The rows of all ranks together then equal i8lt_forward on the whole batch,
 * bit for bit.  With a disabled threshold the exchange changes nothing.
 * No counterpart on the pages (their layer runs on one device); it is the
 * exchange step a token-sharded version of the method needs.
 */
int i8lt_forward_colmax(const void* A, int at, int64_t M, int64_t K, int64_t N,
                        void* ws, size_t ws_bytes, int64_t max_outliers, void* stream);
int i8lt_forward_from_colmax(const void* A, int at, int64_t M, int64_t K,
                             const int8_t* CB, const float* SCB, int64_t N,
                             const void* bias, int bt, float threshold,
                             const void* residual, void* out,
                             void* ws, size_t ws_bytes, int64_t max_outliers,
                             const i8lt_fwd_debug* dbg, void* stream);

/* Workspace of i8lt_backward_input, in bytes.
 * i8lt_backward_workspace_size: the minimum, for the fused schedule (status
 * word, grad_bias partial sums, and the fp16 copy of grad_output when it is
 * not already fp16 with N a multiple of 8).
 * i8lt_backward_workspace_size_dq: the minimum plus the transient
 * dequantized weight of the materialized schedule, K_pad x N_pad fp16
 * (K_pad = i8lt_weight_ld(K), N_pad = N rounded up to 8). */
size_t i8lt_backward_workspace_size(int64_t M, int64_t N, int gt);
size_t i8lt_backward_workspace_size_dq(int64_t M, int64_t N, int64_t K, int gt);

/*
 * Memory-efficient backward to the input (no weight gradient: the weight is
 * frozen in this mode).
 *   G         [M, N] grad_output, dtype `gt` (the layer's output dtype)
 *   CB, SCB   the quantized weight, CB leading dimension i8lt_weight_ld(K)
 *   addend    [M, K] dtype `gt`, or NULL: added to grad_A before rounding
 *   grad_A    [M, K] dtype `gt`, or NULL to skip:
 *             grad_A = to_dtype( fp16(G) @ W_dq ),
 *             W_dq[n,k] = fp16_rn(fp32(CB[n,k]) * (SCB[n] * fp32(1/127)))
 *             (bitsandbytes PR #33, "Memory efficient backward": the int8
 *             weight is dequantized to fp16 for the backward matmul on every
 *             call and the fp16 weight is not kept between calls)
 *   grad_bias [N] dtype `bt`, or NULL to skip: sum over rows of the uncast G
 *   ws        workspace of at least i8lt_backward_workspace_size bytes.  The
 *             size picks the schedule (same results either way):
 *             ws_bytes >= i8lt_backward_workspace_size_dq: materialized --
 *               a memory-bound prepass writes W_dq transposed into the
 *               workspace, then a plain fp16 GEMM reads it (the faster one);
 *             otherwise fused -- W_dq is rebuilt tile by tile in shared
 *               memory inside the GEMM and never stored (no N x K buffer).
 */
int i8lt_backward_input(const void* G, int gt, int64_t M, int64_t N,
                        const int8_t* CB, const float* SCB, int64_t K,
                        const void* addend, void* grad_A,
                        void* grad_bias, int bt,
                        void* ws, size_t ws_bytes, void* stream);

/*
 * i8lt_backward_input_noalloc -- the same computation as i8lt_backward_input,
 * for callers that cannot allocate device memory: a host framework that has
 * reserved the GPU's memory for its own pool at start-up (so a cudaMalloc
 * would fail or fragment it), code that runs inside another library's
 * allocator or memory-pressure callback, or a latency-critical loop that must
 * not enter the driver's allocator.  No counterpart on the pages: it is an
 * interface addition, not part of the method.
 *
 * The scratch (status word, grad_bias partial sums, fp16 copy of G) lives in
 * one static device array of I8LT_NOALLOC_SCRATCH_BYTES that every GPU which
 * loads this library holds until the process exits.  The caller still passes
 * every input and output.  A problem whose scratch
 * (i8lt_backward_workspace_size(M, N, gt)) exceeds that size is rejected with
 * I8LT_ERR_SCRATCH_LIMIT before anything is launched.  The call allocates no
 * device memory (no cudaMalloc / cudaFree, no allocating library routine);
 * with kernel timing switched on (i8lt_profile_start) the library creates
 * CUDA events, so such callers should leave timing off.
 *
 * The first call on each device looks up the device address of the array
 * (once per device, with that device current) and keeps it for the life of
 * the process; make that first call before any stream capture.  A
 * cudaDeviceReset of a device that has used this entry point leaves that
 * address stale: do not reset such a device while the library is loaded.
 * Every call shares the one array, which keeps the last call's contents
 * (each call clears the status word it needs): calls whose work overlaps on
 * the GPU (other streams, other threads) race on it and must be serialised
 * by the caller.  Device-side errors (a pipeline wait that timed out) are
 * recorded in the array's status word; read them with
 * i8lt_noalloc_read_device_status.
 */
#define I8LT_NOALLOC_SCRATCH_BYTES (32u << 20)
int i8lt_backward_input_noalloc(const void* G, int gt, int64_t M, int64_t N,
                                const int8_t* CB, const float* SCB, int64_t K,
                                const void* addend, void* grad_A,
                                void* grad_bias, int bt, void* stream);
/* Synchronizes `stream`, then reads the status word of the no-alloc scratch
 * on the current device (the result of the last i8lt_backward_input_noalloc
 * call there) into *status (may be NULL) and clears a recorded error, like
 * i8lt_read_device_status does for a workspace.  Allocates nothing (one
 * small device-to-host copy into this function's own stack).  Returns
 * I8LT_OK or the status the device recorded. */
int i8lt_noalloc_read_device_status(int32_t* status, void* stream);

/*
 * Weight gradient of the trainable-weight mode (bitsandbytes'
 * has_fp16_weights=True: the float weight is the parameter and is quantized
 * afresh on every forward with i8lt_quantize_weight):
 *   grad_W [N, K] dtype `wt` = sum over the M tokens of G[m, n] A[m, k],
 * computed in int8: G [M, N] (dtype gt) and A [M, K] (dtype at), both cast to
 * fp16, are quantized column by column -- one absmax scale per output
 * feature n and per input feature k, taken over the tokens -- the codes are
 * multiplied exactly (int32, so M <= I8LT_MAX_K, else I8LT_ERR_K_TOO_LARGE)
 * and grad_W = Cacc * scale_G[n] * scale_A[k] / 127^2, rounded once.  The
 * per-column scales keep an outlier feature from spoiling the others, so no
 * separate outlier product is taken.  Interface addition: the pages' layer
 * runs in the memory-efficient mode, where the weight is frozen.
 *   ws  at least i8lt_grad_weight_workspace_size(M, N, K) bytes
 */
size_t i8lt_grad_weight_workspace_size(int64_t M, int64_t N, int64_t K);
int i8lt_grad_weight(const void* G, int gt, const void* A, int at,
                     int64_t M, int64_t N, int64_t K,
                     void* grad_W, int wt, void* ws, size_t ws_bytes, void* stream);

/*
 * 4-bit weight-only layers: QLoRA fine-tuning keeps the frozen base weights
 * in 4 bits and runs every matmul in the 16-bit compute dtype ("Support
 * QLoRA 4-bit finetuning with bitsandbytes", lit-gpt PR #275: the bnb.nf4
 * and bnb.fp4 quantize options, Llama-2-7B runs with --precision
 * bf16-true).  The page names both formats without defining them.  Both
 * share one storage:
 *   blocks   64 consecutive elements of a weight row share one fp32 absmax;
 *   packing  row n of `packed` holds i8lt_nf4_row_bytes(K) bytes, two codes
 *            per byte, element 2j in the high nibble of byte j; padding and
 *            all-zero blocks hold the zero code;
 *   dequantization  Wdq[n, k] = rn(levels[code] * absmax[n, k / 64]), one
 *            fp32 multiply rounded once to the compute dtype.
 * NF4 follows QLoRA's published 4-bit NormalFloat construction:
 *   levels   16 fp32 values from -1 to 1 with an exact 0 (code 7): 7 negated
 *            and 8 positive standard-normal quantiles of evenly spaced
 *            probabilities between 1/2 and ((1 - 1/30) + (1 - 1/32)) / 2,
 *            divided by the largest (i8lt_nf4_levels returns them);
 *   codes    the nearest level to x / absmax (one fp32 division), decided
 *            against the fp32 midpoints of adjacent levels (a value equal to
 *            a midpoint takes the lower level).
 * FP4 is the 4-bit floating-point format E2M1 (1 sign, 2 exponent, 1
 * mantissa bits; exponent 0 subnormal), scaled so that the block's absmax
 * is its largest magnitude 6:
 *   levels   code = 8 s + c, c = the 3 exponent-mantissa bits with the
 *            magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; levels[code] =
 *            (-1)^s * E2M1(c) / 6 in fp32 (i8lt_fp4_levels; code 8 is -0);
 *   codes    c is the magnitude nearest to |x / absmax| (one fp32
 *            division), decided against the fp32 midpoints of adjacent
 *            magnitude levels, a tie taking the c whose mantissa bit is 0
 *            (round half to even); s = 1 for x < 0 unless c = 0 (zero is
 *            always code 0).
 * The nf4-dq / fp4-dq variants (absmax stored in 8 bits) are not provided.
 * The entry points of the two formats take the same arguments.
 */
#define I8LT_NF4_BLOCK 64
/* out[16]: the levels, by code (ascending for NF4). */
int i8lt_nf4_levels(float* out);
int i8lt_fp4_levels(float* out);
/* Bytes per packed row: round_up(K, 64) / 2 (a multiple of 32); -1 for K < 0. */
int64_t i8lt_nf4_row_bytes(int64_t K);
/* absmax values per row: ceil(K / 64); -1 for K < 0. */
int64_t i8lt_nf4_blocks(int64_t K);
/* W [N, K] row-major (dtype wt, device) -> packed [N, row_bytes] uint8 and
 * absmax [N, blocks] fp32, both device, caller-owned.  packed 16-byte
 * aligned. */
int i8lt_nf4_quantize(const void* W, int wt, int64_t N, int64_t K,
                      uint8_t* packed, float* absmax, void* stream);
int i8lt_fp4_quantize(const void* W, int wt, int64_t N, int64_t K,
                      uint8_t* packed, float* absmax, void* stream);
/* The dequantized weight Wdq [N, K] row-major in dtype dt (device). */
int i8lt_nf4_dequantize(const uint8_t* packed, const float* absmax, int64_t N,
                        int64_t K, void* out, int dt, void* stream);
int i8lt_fp4_dequantize(const uint8_t* packed, const float* absmax, int64_t N,
                        int64_t K, void* out, int dt, void* stream);
/* Workspace of the two matmuls: the device status word (256 bytes).  The
 * weight is then decoded stage by stage inside the GEMM and never stored. */
size_t i8lt_nf4_workspace_size(void);
/* A workspace of at least this many bytes (256 + N * K * 2; 0 for invalid
 * sizes) selects the materialized schedule instead: a prepass writes the
 * dequantized weight into the workspace (Wdq [N, K] for the forward, Wdq^T
 * [K, N] for the input gradient) and a TMA-fed GEMM reads it.  Same results
 * bit for bit, more memory, faster. */
size_t i8lt_nf4_workspace_size_dq(int64_t K, int64_t N);
/* Extra workspace bytes of an input gradient that also returns grad_bias
 * (the fp32 partial sums of 128-token chunks, ceil(M / 128) x N): they
 * follow the status word, and the dequantized weight of the materialized
 * schedule, if it fits, follows them. */
size_t i8lt_nf4_grad_bias_bytes(int64_t M, int64_t N);
/*
 * out [M, N] = rn(A [M, K] @ Wdq^T + bias), A and out in the compute dtype
 * at (I8LT_F16 or I8LT_BF16), fp32 accumulation on the tensor
 * cores; the weight is decoded stage by stage in shared memory and never
 * stored.  bias [N] of dtype bt or NULL.  K a multiple of 8 (16-byte rows
 * for the tensor-memory copies), else I8LT_ERR_INVALID_ARG; A, packed, out
 * 16-byte aligned; ws of i8lt_nf4_workspace_size bytes (or
 * i8lt_nf4_workspace_size_dq, see there), 256-byte aligned.
 */
int i8lt_nf4_forward(const void* A, int at, int64_t M, int64_t K,
                     const uint8_t* packed, const float* absmax, int64_t N,
                     const void* bias, int bt, void* out,
                     void* ws, size_t ws_bytes, void* stream);
int i8lt_fp4_forward(const void* A, int at, int64_t M, int64_t K,
                     const uint8_t* packed, const float* absmax, int64_t N,
                     const void* bias, int bt, void* out,
                     void* ws, size_t ws_bytes, void* stream);
/*
 * The gradients of the frozen 4-bit layer (the weight has none):
 *   grad_A [M, K] = rn(G [M, N] @ Wdq) in the compute dtype gt, or NULL to
 *            skip, with the weight decoded the same way;
 *   grad_bias [N] = the sum over the tokens of G, dtype bt, or NULL: fp32
 *            partial sums of 128-token chunks (each in a fixed order), then
 *            summed over the chunks in order; reduced inside the GEMM by its
 *            epilogue warps while the tensor cores run, or by a pass of its
 *            own when grad_A is NULL -- the same bits either way.
 * N a multiple of 8; ws at least i8lt_nf4_workspace_size() +
 * (grad_bias ? i8lt_nf4_grad_bias_bytes(M, N) : 0) bytes, and that plus
 * N * K * 2 (rounded up to 256) selects the materialized schedule; other
 * rules as i8lt_nf4_forward.
 */
int i8lt_nf4_backward_input(const void* G, int gt, int64_t M, int64_t N,
                            const uint8_t* packed, const float* absmax,
                            int64_t K, void* grad_A, void* grad_bias, int bt,
                            void* ws, size_t ws_bytes, void* stream);
int i8lt_fp4_backward_input(const void* G, int gt, int64_t M, int64_t N,
                            const uint8_t* packed, const float* absmax,
                            int64_t K, void* grad_A, void* grad_bias, int bt,
                            void* ws, size_t ws_bytes, void* stream);

/*
 * Double-quantized absmax: the `bnb.nf4-dq` and `bnb.fp4-dq` options of
 * "Support QLoRA 4-bit finetuning with bitsandbytes" (lit-gpt PR #275), which
 * store the fp32 absmax values of the 64-element blocks in 8 bits (QLoRA's
 * double quantization).  The page names the options without a definition;
 * the reading:
 *   offset   = fp32(S / count), S the sum of all `count` absmax values exactly
 *              rounded to float64, an IEEE float64 division;
 *   d        = fp32(c - offset) for every value c (row-major order);
 *   absmax2  = max |d| over each block of 256 consecutive values (fp32);
 *   q        = the FP8 E4M3 code (1 sign, 4 exponent bits with bias 7, 3
 *              mantissa bits, subnormals, largest finite 448) nearest to
 *              fp32(d * fp32(448 / absmax2)) (0 for a block of zeros), ties
 *              to the even code, saturating at +-448, the sign kept;
 *   decoded  = fp32(fp32(E4M3(q) * fp32(absmax2 * fp32(1 / 448))) + offset).
 * The 4-bit codes are those of the plain format; the matmuls take the
 * decoded absmax (i8lt_absmax8_dequantize writes it, fp32 [N, blocks per
 * row], e.g. into a buffer reused across layers).  Storage: 1 byte per
 * 64-element block plus 4 bytes per 256 blocks and 4 bytes, instead of 4
 * bytes per block.
 *
 * i8lt_absmax8_blocks(count): ceil(count / 256), the length of absmax2.
 * i8lt_absmax8_quantize: absmax [count] fp32 (finite, >= 0, as
 *   i8lt_nf4_quantize / i8lt_fp4_quantize write them) -> q [count] u8,
 *   absmax2 [i8lt_absmax8_blocks(count)] fp32, *offset (one fp32, device
 *   memory); ws of i8lt_absmax8_workspace_size() bytes, 256-byte aligned
 *   (scratch for the exact sum).  count == 0 writes offset = 0.
 * i8lt_absmax8_dequantize: q, absmax2, offset (device) -> out [count] fp32.
 * All pointers are device pointers owned by the caller; asynchronous on
 * `stream`.  Errors: I8LT_ERR_INVALID_ARG (count < 0 or > 2^40, a NULL
 * pointer), I8LT_ERR_WORKSPACE, I8LT_ERR_MISALIGNED.
 */
int64_t i8lt_absmax8_blocks(int64_t count);
size_t i8lt_absmax8_workspace_size(void);
int i8lt_absmax8_quantize(const float* absmax, int64_t count, uint8_t* q,
                          float* absmax2, float* offset, void* ws,
                          size_t ws_bytes, void* stream);
int i8lt_absmax8_dequantize(const uint8_t* q, const float* absmax2,
                            const float* offset, int64_t count, float* out,
                            void* stream);

/* SiLU between the two layers of an MLP: out = h * sigmoid(h), and its
 * backward out = g * silu'(h).  n elements of dtype dt. */
int i8lt_silu_forward(const void* h, int dt, int64_t n, void* out, void* stream);
int i8lt_silu_backward(const void* g, const void* h, int dt, int64_t n,
                       void* out, void* stream);

/* Kernel-level timing.  Between i8lt_profile_start and i8lt_profile_stop
 * the library records a CUDA event before and after every kernel it
 * launches, on the launch stream (no synchronization while recording).
 * i8lt_profile_stop waits for the recorded events, writes up to `cap`
 * {kernel id, milliseconds} records in launch order, sets *n_records to the
 * number written and *n_launches to the number of kernel launches made while
 * recording, and stops recording.  Host-side state only; at most
 * `max_launches` launches are timed (later ones are counted, not timed). */
typedef enum {
  I8LT_K_QUANTIZE_WEIGHT = 0, I8LT_K_COLMAX = 1, I8LT_K_OUTLIER_INDEX = 2, I8LT_K_ROW_QUANTIZE = 3,
  I8LT_K_SUBB = 4, I8LT_K_FWD_GEMM = 5, I8LT_K_GRADOUT_PREPASS = 6, I8LT_K_GRAD_BIAS_FINALIZE = 7,
  I8LT_K_BWD_GEMM = 8, I8LT_K_SILU = 9, I8LT_K_SILU_BACKWARD = 10, I8LT_K_WIDEN_CODES = 11,
  I8LT_K_DEQUANT_WEIGHT = 12, I8LT_K_COL_QUANTIZE = 13, I8LT_K_WGRAD_GEMM = 14, I8LT_K_UNIT_PLAN = 15,
  I8LT_K_NF4_QUANTIZE = 16, I8LT_K_NF4_DEQUANTIZE = 17, I8LT_K_NF4_GEMM_FWD = 18, I8LT_K_NF4_GEMM_BWD = 19,
  I8LT_K_ABSMAX8 = 20, I8LT_K_COUNT = 21
} i8lt_kernel_id;
typedef struct {
  int kernel;
  float ms;
} i8lt_kernel_time;
int i8lt_profile_start(int max_launches);
/* Diagnostic of the failure path.  Every pipeline wait of the library is
 * bounded: a wait that has not completed after its limit (4 s in the
 * kernels) records I8LT_ERR_TIMEOUT in the workspace status word, the kernel
 * winds down and the CUDA context stays usable.  This entry point runs that
 * same wait, limit_ns long (0 < limit_ns <= 2e9), on a barrier that nothing
 * completes, so that a caller or a test can see the error come back through
 * i8lt_read_device_status.  ws: at least 256 bytes, 256-byte aligned (its
 * status word is cleared first).  No counterpart on the pages. */
int i8lt_debug_wait_timeout(int64_t limit_ns, void* ws, size_t ws_bytes, void* stream);
/* The same for the grid-wide wait of the fused activation quantization: two
 * blocks of a cooperative launch wait, limit_ns long, at a barrier that is
 * one arrival short of complete (the arrival counter at byte 64 of ws, as in
 * the forward workspace); each records I8LT_ERR_TIMEOUT (role 7) and
 * returns.  ws: at least 256 bytes, 256-byte aligned, cleared first. */
int i8lt_debug_grid_wait_timeout(int64_t limit_ns, void* ws, size_t ws_bytes, void* stream);

/* Launch shape the library uses for the persistent GEMM kernels
 * (kernel = I8LT_K_FWD_GEMM or I8LT_K_BWD_GEMM): CTAs (pairs x 2), threads
 * per CTA and dynamic shared memory per CTA on the current device.  Any
 * output pointer may be NULL. */
int i8lt_gemm_launch_info(int kernel, int* ctas, int* threads, int* smem_bytes);
int i8lt_profile_stop(i8lt_kernel_time* out, int cap, int* n_records, int* n_launches);
const char* i8lt_kernel_name(int kernel);

/* Synchronizes `stream`, then reads the status word of a forward or backward
 * workspace, i.e. of the last call that used it (status and the number of
 * outlier columns found; either output pointer may be NULL), and clears the
 * status.  Returns I8LT_OK or the status the device recorded. */
int i8lt_read_device_status(void* ws, int32_t* status, int32_t* outliers,
                            void* stream);

#ifdef __cplusplus
}
#endif
#endif /* I8LT_H_ */
