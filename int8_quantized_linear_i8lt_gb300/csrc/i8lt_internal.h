// Host-side launchers shared between the translation units of libi8lt.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "i8lt_common.cuh"

namespace i8lt {

inline int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }
inline int64_t ceil_div(int64_t x, int64_t m) { return (x + m - 1) / m; }

// ---- kernel timing (i8lt_api.cu): no-ops unless i8lt_profile_start ran ----
void prof_begin(int kernel_id, cudaStream_t s);
void prof_end(cudaStream_t s);

struct ProfScope {
  cudaStream_t s;
  ProfScope(int id, cudaStream_t st) : s(st) { prof_begin(id, st); }
  ~ProfScope() { prof_end(s); }
};

// ---- memory-bound kernels (i8lt_quant.cu) --------------------------------

// K1: W [N,K] (dtype wt) -> CB int8 [N, ld] (zero pad), SCB fp32 [N].
cudaError_t launch_quantize_weight(const void* W, int wt, int64_t N, int64_t K, int64_t ld, bool vec,
                                   int8_t* CB, float* SCB, cudaStream_t s);

// K2: colmax[k] = fp16 bits of max_m |fp16(A[m,k])| (atomic max; colmax must
// be zeroed first).
cudaError_t launch_colmax(const void* A, int at, int64_t M, int64_t K, bool vec, uint32_t* colmax,
                          cudaStream_t s);

// Outlier set from colmax: mask bits, ascending idx[], found/used counts.
cudaError_t launch_outlier_index(const uint32_t* colmax, int64_t K, float thr, int64_t cap, int* idx,
                                 uint32_t* mask, DevStatus* st, cudaStream_t s);

// K3: SCA[m], Aq [M, K_pad] (codes as exact fp16), subA [M, cap_pad], and
// the activation side of the accumulation plan: asq[(m / 256) * nchunks + c]
// raised to the sum of squared codes of row m in the 1024-column chunk c
// (asq zeroed, [ceil(M / 256), ceil(K_pad / 1024)]).
cudaError_t launch_row_quantize(const void* A, int at, int64_t M, int64_t K, int64_t K_pad, bool vec,
                                const uint32_t* mask, const int* idx, DevStatus* st, int64_t cap_pad,
                                float* SCA, __half* Aq, __half* subA, uint32_t* asq, cudaStream_t s);

// K2 + K3 in one launch (i8lt_actquant.cu), for 16-bit A with K a multiple
// of 8 up to 32768 (act_quant_fused_supported): with do_colmax, the column
// maxima of A's rows into colmax (zeroed), by a cooperative launch with
// bounded grid-wide waits (arrive: a zeroed counter); then (or from the given
// colmax) the outlier set -- block 0 writes mask, idx and the counts in st --
// and SCA, Aq, subA and asq as launch_row_quantize.
// W [N, K] 16-bit -> CB int8 [N, k_pad], SCB [N] by the fused kernel's row
// pass (K % 8 == 0, k_pad <= 32768; act_quant_fused_supported).
cudaError_t launch_quantize_weight_fused(const void* W, int wt, int64_t N, int64_t K, int64_t k_pad, int8_t* CB,
                                         float* SCB, cudaStream_t s);
// Two blocks of a cooperative launch wait at a grid-wide barrier that one
// arrival short of complete, with the given limit (a test of the timeout path).
cudaError_t launch_grid_wait_probe(DevStatus* st, unsigned* arrive, unsigned long long limit_ns, cudaStream_t s);
bool act_quant_fused_supported(int at, int64_t K);
cudaError_t launch_act_quant_fused(const void* A, int at, int64_t M, int64_t K, int64_t k_pad, bool enabled,
                                   float thr, bool do_colmax, int64_t cap, int64_t cap_pad, uint32_t* colmax,
                                   uint32_t* mask, int* idx, DevStatus* st, unsigned* arrive, float* SCA,
                                   __half* Aq, __half* subA, uint32_t* asq, cudaStream_t s);

// Blocks of a kernel resident per SM at a given block size and dynamic shared
// memory, cached per (kernel, device, size): no query while a stream is
// being captured.
int cached_blocks_per_sm(const void* fn, int threads, int smem);

// K4: subB[n, j] = fp16(fp32(CB[n, idx[j]]) * SCB[n] * fp32(1/127)).
cudaError_t launch_build_subB(const int8_t* CB, int64_t ld, const float* SCB, int64_t N, const int* idx,
                              const DevStatus* st, int64_t cap_pad, __half* subB, cudaStream_t s);

// grad_bias is reduced in chunks of this many rows of G: partial[c, n] = the
// sum of G[m, n] over the rows m of chunk c (128 c <= m < 128 c + 128), in a
// fixed order that every kernel producing partial sums follows; then
// grad_bias[n] = sum over c, in order.
constexpr int kBiasChunkRows = 128;

// K7: grad_bias partial sums of the uncast G and (optionally) G16 = fp16(G)
// with N padded to N_pad; then the finalize (when grad_bias is given).
cudaError_t launch_gradout_prepass(const void* G, int gt, int64_t M, int64_t N, bool vec, __half* G16,
                                   int64_t N_pad, void* grad_bias, int bt, float* partial,
                                   int64_t max_chunks, cudaStream_t s);
// grad_bias[n] = sum over the chunks c (in order) of partial[c, n].
cudaError_t launch_grad_bias_finalize(const float* partial, int64_t M, int64_t N, void* grad_bias, int bt,
                                      cudaStream_t s);
int64_t gradout_partial_chunks(int64_t M);

cudaError_t launch_silu(const void* h, int dt, int64_t n, bool vec, void* out, cudaStream_t s);

// Diagnostic of the bounded waits: a wait that nothing completes, limit_ns long.
cudaError_t launch_wait_limit(DevStatus* st, unsigned long long limit_ns, cudaStream_t s);

// Trainable-weight mode: column-wise quantization of X [R, C] (dtype xt) into
// Xt [C, R_pad] fp16 codes and scale [C], from the column maxima colmax [C]
// (launch_colmax).  With sq ([C, ceil(R_pad / 1024)] int32, zeroed) and tsq
// ([ceil(C / 256), ceil(R_pad / 1024)] uint32, zeroed): the per-tile chunk
// maxima of the squared codes, for the GEMM's accumulation plan.
cudaError_t launch_col_quantize(const void* X, int xt, int64_t R, int64_t C, bool vec, const uint32_t* colmax,
                                int64_t R_pad, float* scale, __half* Xt, int* sq, uint32_t* tsq, cudaStream_t s);
cudaError_t launch_silu_backward(const void* g, const void* h, int dt, int64_t n, bool vec, void* out,
                                 cudaStream_t s);

// ---- tensor-core GEMMs (i8lt_gemm.cu) -------------------------------------

struct FwdGemmArgs {
  CUtensorMap tmA;    // Aq fp16 [M, K_pad], box 64 x 128, 128B swizzle
  CUtensorMap tmB;    // CBh fp16 [N, K_pad] (widened codes), box 64 x 128, 128B swizzle
  CUtensorMap tmSA;   // subA fp16 [M, cap_pad], box 64 x 128, 128B swizzle
  CUtensorMap tmSB;   // subB fp16 [N, cap_pad], box 64 x 128, 128B swizzle
};

struct FwdEpiArgs {
  int M, N, K_pad;
  int use_outliers;       // 0: decomposition disabled
  const float* SCA;
  const uint32_t* plan;   // per pair tile [num_m x num_n] (launch_unit_plan): bits 0-15 chunks of
                          // 1024 products per accumulation unit, bit 16 fast exact conversion
  const float* SCB;
  const void* bias;
  int bias_dt;
  const void* residual;
  void* out;
  int out_dt;
  int32_t* acc_i32;       // optional raw accumulator
  void* act;              // optional: silu(out) [M, N] in out_dt (MLP hidden layer)
  uint32_t* act_colmax;   // with act: per column max of |fp16(act)| bits, atomically raised
  DevStatus* st;
};

cudaError_t launch_fwd_gemm(const FwdGemmArgs& g, const FwdEpiArgs& e, cudaStream_t s, int prof_id = 5 /*K_FWD_GEMM*/);

// Forward prepass: CBh = fp16(CB) (exact), CB [N, k_pad]; and, for the
// accumulation plan, bsq[n / 256, c] raised to the sum of squares of the codes
// of row n in the 1024-column chunk c (bsq zeroed, [ceil(N / 256), nchunks]).
cudaError_t launch_widen_codes(const int8_t* CB, __half* CBh, int64_t N, int64_t k_pad, uint32_t* bsq,
                               cudaStream_t s);

// Exact-accumulation plan of the int8 GEMM.  asq [num_m, nchunks] and bsq
// [num_n, nchunks] hold, per 256-row tile of each operand and per 1024-deep
// chunk of the reduction, the largest sum of squares of a row's codes in that
// chunk.  By Cauchy-Schwarz every partial sum of a group of chunks G is at
// most sqrt(sum_G asq * sum_G bsq), so a group with sum_G asq * sum_G bsq <
// 2^48 accumulates exactly in fp32 (|partial| < 2^24), and one below 2^44
// (|partial| < 2^22) drains with the fast conversion.  plan[tm * num_n + tn] =
// L | fast << 16 with L the largest number of chunks per group such that every
// aligned group of L chunks of that tile pair is below 2^48 (a single chunk
// always is: (1024 * 127^2)^2 < 2^48).
cudaError_t launch_unit_plan(const uint32_t* asq, const uint32_t* bsq, int num_m, int num_n, int nchunks,
                             uint32_t* plan, cudaStream_t s);

// The largest sum of squares of the codes of one 1024-column chunk.
constexpr uint32_t kChunkSqMax = 1024u * 127u * 127u;

struct BwdGemmArgs {
  CUtensorMap tmW;    // fused schedule: CB int8 [N, K_pad] (inner K_pad, outer N), box 128 x 64, 128B swizzle
  CUtensorMap tmWT;   // materialized schedule: WdqT fp16 [K_pad, N_pad], box 64 x 128, 128B swizzle
  CUtensorMap tmG;    // G16 fp16 [M, N_pad], box 64 x 128, 128B swizzle
};

// D[r, m] = sum_c W(r, c) X[m, c], stored at out[m * K + r]: r < K output
// rows (the input features k of the int8 and 4-bit input gradients, the
// output features n of the 4-bit forward), c < N the reduction, m < M tokens.
struct BwdEpiArgs {
  int M, N, K;
  const float* SCB;      // int8: per weight row n, the absmax scale
  const void* addend;    // [M, K] in dt, or NULL
  void* grad_A;          // [M, K] in dt
  int dt;
  DevStatus* st;
  const void* bias;      // [K] in bias_dt, or NULL
  int bias_dt;
  uint32_t ab_fmt;       // instruction-descriptor bits of the operand type (0: fp16)
  const float* absmax;   // 4-bit: [weight rows, nblk] per-64-element scales
  int nblk;
  float lv[16];          // 4-bit: the code levels
  // grad_bias reduced inside the GEMM (the uncast X = G of the input-gradient
  // modes, row-major [M, N], N a multiple of 8, 16-byte aligned), or NULL:
  // the epilogue warps write partial[c, n] (kBiasChunkRows-row chunks c of
  // the tokens) for the 64-wide blocks n of the reduction that their tile
  // owns (block b belongs to the output tile row b % num_k)
  const void* gsum;
  int gsum_dt;           // DT_F16 or DT_BF16
  float* partial;        // [ceil(M / kBiasChunkRows), N]
};

// fused: the dequantized weight is rebuilt in shared memory from CB (tmW);
// otherwise it is read from WdqT (tmWT), written by launch_dequant_weight.
cudaError_t launch_bwd_gemm(const BwdGemmArgs& g, const BwdEpiArgs& e, bool fused, cudaStream_t s);

// 4-bit NormalFloat matmuls with the weight decoded per stage in shared memory
// (tmW: the packed codes [rows, row_bytes] uint8, no swizzle; box 64 x 64 for
// the input gradient, 32 x 128 for the forward; tmG: the 16-bit activations
// or output gradient, box 64 x 128, 128B swizzle).
// materialized: A operand read by TMA from a dequantized copy (tmWT: [R, C]
// 16-bit, box 64 x 128, 128B swizzle) instead of decoded per stage.
cudaError_t launch_nf4_gemm(const BwdGemmArgs& g, const BwdEpiArgs& e, bool input_grad, bool materialized,
                            cudaStream_t s);

// The 4-bit formats sharing the packed storage (two codes per byte, one fp32
// absmax per 64 elements of a row) and the table-driven decode of the
// matmuls: 4-bit NormalFloat and E2M1 floating point (i8lt_nf4.cu).
enum Fmt4 { kFmtNf4 = 0, kFmtFp4 = 1 };

// The 16 NF4 levels (ascending fp32), computed once on the host.
void nf4_levels(float out[16]);
// The 16 levels of a format, indexed by code, computed once on the host.
void fmt4_levels(int fmt, float out[16]);
// W [N, K] (dtype wt) -> packed [N, row_bytes] codes and absmax [N, ceil(K / 64)].
cudaError_t launch_nf4_quantize(const void* W, int wt, int64_t N, int64_t K, int64_t row_bytes, uint8_t* packed,
                                float* absmax, cudaStream_t s, int fmt = kFmtNf4);
// packed + absmax -> WdqT [K, N] (dtype dt, f16 or bf16; N a multiple of 8).
cudaError_t launch_nf4_dequantize_t(const uint8_t* packed, const float* absmax, int64_t N, int64_t K,
                                    int64_t row_bytes, void* WdqT, int dt, cudaStream_t s, int fmt = kFmtNf4);
// packed + absmax -> out [N, K] (dtype dt): lv[code] * absmax, rounded once.
cudaError_t launch_nf4_dequantize(const uint8_t* packed, const float* absmax, int64_t N, int64_t K,
                                  int64_t row_bytes, void* out, int dt, cudaStream_t s, int fmt = kFmtNf4);
// Double-quantized absmax: n fp32 values -> E4M3 codes q [n], absmax2
// [ceil(n / 256)], offset [1]; `buckets` is 256 u64 of scratch.
cudaError_t launch_absmax8_quantize(const float* absmax, int64_t n, uint8_t* q, float* absmax2, float* offset,
                                    unsigned long long* buckets, cudaStream_t s);
// ... and back to fp32 [n].
cudaError_t launch_absmax8_dequantize(const uint8_t* q, const float* absmax2, const float* offset, int64_t n,
                                      float* out, cudaStream_t s);

// Backward prepass of the materialized schedule: WdqT[k, n] =
// fp16_rn(fp32(CB[n, k]) * (SCB[n] * fp32(1/127))) for k < k_pad, n < N, and
// 0 for N <= n < n_pad (n_pad a multiple of 8, k_pad of 16).
cudaError_t launch_dequant_weight(const int8_t* CB, const float* SCB, int64_t N, int64_t k_pad, __half* WdqT,
                                  int64_t n_pad, cudaStream_t s);

// Raise a kernel's dynamic shared-memory limit to smem_bytes on the current
// device, once per (kernel, device): later calls, also those made while a
// stream is being captured, issue no CUDA call.
bool ensure_smem_attr(const void* fn, int smem_bytes);

// Persistent launch shape of a GEMM kernel (K_FWD_GEMM / K_BWD_GEMM).
cudaError_t gemm_launch_shape(int kernel_id, int* ctas, int* threads, int* smem_bytes);

// Kernel ids of the timing records (match i8lt_kernel_id in i8lt.h).
enum KernelId {
  K_QUANTIZE_WEIGHT = 0, K_COLMAX, K_OUTLIER_INDEX, K_ROW_QUANTIZE, K_SUBB, K_FWD_GEMM, K_GRADOUT_PREPASS,
  K_GRAD_BIAS_FINALIZE, K_BWD_GEMM, K_SILU, K_SILU_BACKWARD, K_WIDEN_CODES, K_DEQUANT_WEIGHT, K_COL_QUANTIZE,
  K_WGRAD_GEMM, K_UNIT_PLAN, K_NF4_QUANTIZE, K_NF4_DEQUANTIZE, K_NF4_GEMM_FWD, K_NF4_GEMM_BWD, K_ABSMAX8, K_COUNT
};

// Box sizes of the tensor maps (each CTA of a pair stages 128 rows of each
// operand per 64-deep stage).
constexpr int kBoxRows = 128;  // rows of A / CB / subA / subB / G16 boxes
constexpr int kBK = 64;        // reduction elements per pipeline stage
constexpr int kBoxK = 128;     // backward: output features per CB box row

}  // namespace i8lt
