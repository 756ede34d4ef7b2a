// Tensor-core GEMMs of the int8 quantized linear layer (sm_103a, tcgen05,
// CTA pairs).
//
// Forward (K5): out[m,n] = Cacc[m,n] * SCA[m] * SCB[n] / 127^2
//                          + sum_j subA[m,j] subB[n,j] + bias[n] (+ residual)
//   Cacc = sum_k Aq[m,k] CB[n,k] is the exact integer product of the int8
//   codes (bitsandbytes PR #33 "Memory efficient backward": the int8 matmul
//   of the forward, and the "Mixed-precision decomposition matmul" review
//   thread for the outlier part).  sm_103a has no int8 MMA (ptxas rejects
//   tcgen05.mma .kind::i8 for this target), so the codes enter the fp16
//   tensor cores as exact fp16 integers and accumulate in fp32 TMEM, exact
//   while every partial sum stays an integer below 2^24.  The reduction is cut
//   into groups of 1024-deep chunks chosen per tile pair by the accumulation
//   plan (launch_unit_plan: a Cauchy-Schwarz bound from the chunk sums of
//   squared codes; one chunk, <= 1024 * 127^2 < 2^24, always qualifies); each
//   group is drained from TMEM into an int32 running sum held in TMEM, so Cacc
//   is exact for any K <= 133144.  The outlier sub-GEMM subA x subB^T runs as
//   one more fp32 accumulation unit after the int8 groups.
//
// Backward (K6): grad_A[m,k] = sum_n fp16(G)[m,n] * Wdq[n,k],
//   Wdq[n,k] = fp16_rn(fp32(CB[n,k]) * (SCB[n] * fp32(1/127))), rebuilt per
//   stage in shared memory and never stored (PR description, backward bullet;
//   review thread on ".mul(1/127.0)").  Computed transposed,
//   D[k, m] = Wdq^T G16^T, so the converted operand is the A side, stored
//   MN-major (k contiguous, as CB's rows are); B = G16 via TMA, K-major.
//   The backward kernel also runs the 4-bit NormalFloat weight-only matmuls
//   (forward and input gradient of a frozen NF4 layer, see BwdMode).
//
// Both kernels run on CTA pairs (a cluster of 2, tcgen05 cta_group::2): the
// pair computes a 256 x 256 tile with M = 256 MMAs issued by the even CTA;
// each CTA stages its own 128 rows of A and its own 128 rows of B, so the
// per-SM shared-memory traffic is half of a single-CTA 128 x 256 tile.
// Persistent: each pair walks tiles cluster_id, cluster_id + #clusters, ...
// in a grouped raster.
//
// Operand hand-over between the CTAs of a pair.  The even CTA's MMA reads
// both CTAs' shared memory, so every operand tile of the odd CTA must be
// visible to it.  Forward: every operand arrives by TMA and both CTAs' copies
// complete on the even CTA's barrier (cta_group::2 loads): ordered by the
// hardware.  The weight codes are widened to fp16 once per call by a
// memory-bound prepass (the page's forward also re-lays the weight out on
// every call).  Backward: the fp16 weights are rebuilt per stage by converter
// warps and never stored; the odd CTA's converters arrive on a local barrier
// and four relay warps forward each stage to the even CTA with a
// cluster-scope release arrive (~1 us each, so four in flight).  The int8
// weight tiles have a ring of their own, so their copies run ahead of the
// operand stages they are converted into.
//
// Warp roles.  Forward (512 threads per CTA): warp 0 TMA producer; warp 1
// TMEM owner and, in the even CTA, the MMA issuer; warps 6-13 epilogue (warp
// w reads TMEM lanes 32 * (w % 4); warps 6-9 take columns 0-127, warps 10-13
// columns 128-255).  Backward (576 threads): warp 0 G16 producer; warp 1
// TMEM owner and MMA issuer (even CTA) or relay (odd CTA); warps 2-9
// converters; warps 10-13 epilogue (all 256 columns); warp 16 int8 producer;
// warps 14, 15, 17 relays (odd CTA).  Every wait is bounded (mbar_wait).
#include <algorithm>

#include "i8lt_internal.h"

namespace i8lt {

namespace {

constexpr int kThreads = 512;      // forward
constexpr int kBwdThreads = 704;   // backward: 22 warps
constexpr int kFwdStages = 6;      // 32 KB stages: fp16 A and B tiles
constexpr int kI8Stages = 4;       // backward, fused: 8 KB int8 weight tiles on their way to the converters
constexpr int kI8PrefetchAhead = 8;   // int8 weight tiles are fetched into L2 this many stages early
constexpr int kMaxStages = 6;
constexpr int kChunkKB = 16;   // K-blocks of 64 per exact fp32 chunk: 1024 products

constexpr int kWarpProducer = 0;
constexpr int kWarpMMA = 1;
constexpr int kWarpCvt0 = 2;   // backward: 2..9
constexpr int kWarpEpi0 = 6;   // forward: 6..13
constexpr int kBwdWarpEpi0 = 10; // backward: 10..13 and 18..21
constexpr int kBwdWarpEpi1 = 18;
constexpr int kWarpRelay0 = 14; // backward, odd CTA: 14, 15, 17 and warp 1
constexpr int kWarpI8Producer = 16;   // backward: TMA of the int8 weight tiles
constexpr int kWarpRelayLast = 17;
constexpr int kRelays = 4;
// The epilogue waits for a whole accumulation unit (microseconds): it polls
// with a back-off so that the converter warps on the same schedulers keep
// their issue slots.
constexpr unsigned kEpiSleepNs = 256;
constexpr int kCvtWarps = 8;       // backward: every converter warp works on every stage
constexpr int kEpiWarps = 8;      // forward
constexpr int kBwdEpiWarps = 8;   // backward: two per TMEM lane quadrant, each half of the columns
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kBarEpi = 2;     // named barrier id

constexpr int kPairM = 256;    // rows of the pair tile (MMA M)
constexpr int kPairN = 256;    // columns of the pair tile (MMA N)
constexpr int kCtaRows = 128;  // rows of A and of B that each CTA stages

// roles reported in the status word when a wait times out
enum { kWhereProducer = 1, kWhereCvt = 2, kWhereMMA = 3, kWhereEpi = 4, kWhereTeardown = 5 };

struct __align__(8) Barriers {
  uint64_t full[kMaxStages];      // forward and materialized backward, even CTA: both CTAs' copies of
                                  // stage s landed
  uint64_t ready[kMaxStages];     // fused backward, even CTA: both CTAs' operands of stage s in place
                                  // (the G16 copies and the converted tiles: the MMA's one wait a stage)
  uint64_t cvt_done[kMaxStages];  // backward, odd CTA: its converters finished stage s
  uint64_t empty[kMaxStages];     // the pair's MMAs finished reading stage s
  uint64_t i8_full[kI8Stages];    // backward: this CTA's int8 weight tile j landed
  uint64_t i8_empty[kI8Stages];   // backward: this CTA's converters read int8 tile j
  uint64_t acc_full[2];         // an accumulator unit / buffer is complete
  uint64_t acc_empty[2];        // even CTA: both CTAs' epilogues released it
  uint64_t teardown;            // even CTA: every MMA finished
  uint32_t tmem_base;
  int abort_flag;
};

// stage s of each CTA: [A operand 16 KB][B operand(s) 16 KB each] fp16,
// 128B-swizzled.
constexpr int kOpBytes = kCtaRows * kBK * 2;   // 16 KB
constexpr int kI8Bytes = kCtaRows * kBK;       // 8 KB
constexpr int kNf4Bytes = kCtaRows * kBK / 2;  // 4 KB: 4-bit weight tiles
constexpr int kFwdStageBytes = 2 * kOpBytes;
constexpr int kFwdSmemBytes = 1024 /*align slack*/ + kFwdStages * kFwdStageBytes + 3 * kPairN * 4 /*epilogue vectors*/ +
                              static_cast<int>(sizeof(Barriers));

// Backward geometry.  Materialized schedule: 256 (k) x 256 (tokens) pair
// tiles, 6 stages of [WdqT 16 KB][G16 16 KB], two 256-column accumulators so
// that the epilogue of one tile overlaps the next tile's main loop.  Fused
// schedule: 256 (k) x 512 (tokens) pair tiles -- every converted weight tile
// feeds two N = 256 MMAs, which halves the conversion and hand-over work per
// flop -- with 4 stages of [Wdq^T 16 KB][G16 2 x 16 KB], the 512 TMEM
// columns as one accumulator, and a separate ring of 4 int8 weight tiles
// after the operand stages: a weight tile is loaded while the operand stage
// it will be converted into is still being read by the tensor cores, so the
// copy latency and the conversion and hand-over latency overlap instead of
// adding up.
//
// The same kernel runs the 4-bit NormalFloat weight-only matmuls (QLoRA
// fine-tuning with frozen 4-bit weights): the converters decode 4-bit codes
// with per-64-element absmax scales instead of int8 rows with a row scale.
// kModeNf4T is the input gradient (D[k, m] = sum_n Wdq[n, k] G[m, n], the
// converted tile MN-major like the int8 one); kModeNf4 the forward
// (D[n, m] = sum_k Wdq[n, k] A[m, k], the converted tile K-major).
enum BwdMode { kModeMat = 0, kModeI8 = 1, kModeNf4T = 2, kModeNf4 = 3 };

template <int kMode>
struct BwdGeom {
  static constexpr bool kFused = kMode != kModeMat;
  static constexpr bool kNf4 = kMode == kModeNf4T || kMode == kModeNf4;
  static constexpr bool kAmn = kMode == kModeI8 || kMode == kModeNf4T;   // converted tile MN-major
  static constexpr int kRingBytes = kNf4 ? kNf4Bytes : kI8Bytes;
  static constexpr int kSub = kFused ? 2 : 1;                  // N = 256 MMAs per k step
  static constexpr int kTileTokens = kSub * kPairN;            // tokens per pair tile
  static constexpr int kStages = kFused ? 4 : 6;
  static constexpr int kStageBytes = (1 + kSub) * kOpBytes;
  static constexpr int kI8Offset = kStages * kStageBytes;
  static constexpr int kTiles = kI8Offset + (kFused ? kI8Stages * kRingBytes : 0);
  static constexpr int kAccBufs = kFused ? 1 : 2;
  static constexpr int kSmemBytes = 1024 /*align slack*/ + kTiles + static_cast<int>(sizeof(Barriers));
};
static_assert(BwdGeom<kModeI8>::kSmemBytes <= 232448 && BwdGeom<kModeMat>::kSmemBytes <= 232448 &&
                  BwdGeom<kModeNf4>::kSmemBytes <= 232448 && kFwdSmemBytes <= 232448,
              "shared memory per CTA");
static_assert(BwdGeom<kModeI8>::kStages <= kMaxStages && BwdGeom<kModeMat>::kStages <= kMaxStages, "barrier arrays");

__device__ __forceinline__ uint32_t f2i_rn(uint32_t fbits) {
  return static_cast<uint32_t>(__float2int_rn(__uint_as_float(fbits)));
}

// Exact int32 of 32 integer-valued fp32 chunk sums, added to r (or written
// when `first`).  `small`: every |x| < 2^22, so x + 1.5 * 2^23 lies in
// [2^23, 2^24) where fp32 steps by 1 and bits(x + 1.5 * 2^23) = 0x4B400000 + x
// exactly: one packed fp32 add and one integer add per element.  Otherwise
// the conversion instruction (1/8 of the fp32 rate on this SM).
template <int N>
__device__ __forceinline__ void chunk_to_int(const uint32_t (&x)[N], uint32_t (&r)[N], bool first, bool small) {
  if (small) {
#pragma unroll
    for (int j = 0; j < N; j += 2) {
      uint32_t t0, t1;
      asm("{\n .reg .b64 a, b;\n mov.b64 a, {%2, %3};\n"
          " add.rn.f32x2 b, a, %4;\n mov.b64 {%0, %1}, b;\n}"
          : "=r"(t0), "=r"(t1)
          : "r"(x[j]), "r"(x[j + 1]), "l"(0x4B4000004B400000ull));
      r[j] = (first ? 0u : r[j]) + t0 - 0x4B400000u;
      r[j + 1] = (first ? 0u : r[j + 1]) + t1 - 0x4B400000u;
    }
  } else {
#pragma unroll
    for (int j = 0; j < N; ++j) r[j] = (first ? 0u : r[j]) + f2i_rn(x[j]);
  }
}

// 4 signed int8 in a word -> 4 fp16 (exact): bytes biased to unsigned, placed
// in the low mantissa byte of 1024.0 (0x6400), minus 1152 = 1024 + 128.
__device__ __forceinline__ void i8x4_to_h4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t a = __byte_perm(u, 0x64646464u, 0x5140);
  const uint32_t b = __byte_perm(u, 0x64646464u, 0x7362);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));   // 1152
  __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
  __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
  lo = *reinterpret_cast<uint32_t*>(&ha);
  hi = *reinterpret_cast<uint32_t*>(&hb);
}

// 4 signed int8 -> fp16_rn(fp32(q) * f) for each byte.  fp32(q) is built
// exactly as (2^23 + q + 128) - (2^23 + 128); the subtraction and the
// multiply by f run as packed IEEE fp32 pairs (add/mul.rn.f32x2, the same
// rounding per element as the scalar operations), then cvt.rn.f16x2.f32.
__device__ __forceinline__ uint32_t i8x2_scale_to_h2(uint32_t x0, uint32_t x1, uint64_t negc2, uint64_t f2) {
  uint32_t out;
  asm("{\n .reg .b64 x, q, p;\n .reg .b32 plo, phi;\n"
      " mov.b64 x, {%1, %2};\n"
      " add.rn.f32x2 q, x, %3;\n"
      " mul.rn.f32x2 p, q, %4;\n"
      " mov.b64 {plo, phi}, p;\n"
      " cvt.rn.f16x2.f32 %0, phi, plo;\n}"
      : "=r"(out)
      : "r"(x0), "r"(x1), "l"(negc2), "l"(f2));
  return out;
}

__device__ __forceinline__ uint64_t f32x2_splat(float f) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "r"(__float_as_uint(f)));
  return r;
}

__device__ __forceinline__ void i8x4_scale_to_h4(uint32_t w, uint64_t negc2, uint64_t f2, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  lo = i8x2_scale_to_h2(__byte_perm(u, 0x4B000000u, 0x7540), __byte_perm(u, 0x4B000000u, 0x7541), negc2, f2);
  hi = i8x2_scale_to_h2(__byte_perm(u, 0x4B000000u, 0x7542), __byte_perm(u, 0x4B000000u, 0x7543), negc2, f2);
}

// Wait used in teardown only: bounded, ignores the abort flag.
__device__ __forceinline__ void mbar_wait_teardown(uint64_t* bar, uint32_t parity, DevStatus* st) {
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > kWaitTimeoutNs) {
      set_status(st, ST_TIMEOUT, kWhereTeardown);
      return;
    }
  }
}

template <typename T>
__device__ __forceinline__ float load_elem(const void* p, int64_t i) {
  return to_float(static_cast<const T*>(p)[i]);
}

__device__ __forceinline__ float load_any(const void* p, int dt, int64_t i) {
  switch (dt) {
    case DT_F16: return load_elem<__half>(p, i);
    case DT_BF16: return load_elem<__nv_bfloat16>(p, i);
    default: return load_elem<float>(p, i);
  }
}

// Grouped raster: consecutive tiles walk `group` M-tiles of one N-tile, so
// the pairs working at the same time share their A rows and B rows in L2.
__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int group, int& tm, int& tn) {
  const int per_group = group * num_n;
  const int g = t / per_group;
  const int first = g * group;
  const int gm = min(group, num_m - first);
  const int local = t - g * per_group;
  tm = first + local % gm;
  tn = local / gm;
}

// Tile t of the kernels with kTileTokens-token pair tiles (the fused
// backward and the 4-bit matmuls, 512 tokens).  The grouped raster's tiles
// [0, full) run whole; the remaining raster tiles, which would leave most
// pairs idle in the last round, run as two 256-token halves each: tiles
// full + 2 j and full + 2 j + 1 are the halves of raster tile full + j.
// Returns the tile's raster coordinates, its first token and its number of
// 256-token sub-tiles (1 or kTileTokens / 256).
template <int kTileTokens>
__device__ __forceinline__ void split_tile(int t, int full, int num_m, int num_k, int group, int& tm, int& tk,
                                           int& m_base, int& nsub) {
  int r = t, half = -1;
  if (t >= full) {
    r = full + ((t - full) >> 1);
    half = (t - full) & 1;
  }
  tile_coords(r, num_m, num_k, group, tm, tk);
  m_base = tm * kTileTokens + (half > 0 ? kTileTokens / 2 : 0);
  nsub = half >= 0 ? 1 : kTileTokens / 256;
}

__device__ __forceinline__ void init_barriers(Barriers* bars, int epi_warps) {
  for (int s = 0; s < kMaxStages; ++s) {
    mbar_init(&bars->full[s], 1);
    // backward, fused: the even CTA's converters, one relay arrival and the
    // producer's arrival with both CTAs' G16 bytes
    mbar_init(&bars->ready[s], kCvtWarps + 2);
    mbar_init(&bars->cvt_done[s], kCvtWarps);
    mbar_init(&bars->empty[s], 1);
  }
  for (int j = 0; j < kI8Stages; ++j) {
    mbar_init(&bars->i8_full[j], 1);
    mbar_init(&bars->i8_empty[j], kCvtWarps);
  }
  for (int b = 0; b < 2; ++b) {
    mbar_init(&bars->acc_full[b], 1);
    mbar_init(&bars->acc_empty[b], 2 * epi_warps);
  }
  mbar_init(&bars->teardown, 1);
  bars->abort_flag = 0;
  fence_mbar_init();
}

// ---------------------------------------------------------------------------
// Forward GEMM
// ---------------------------------------------------------------------------
template <typename OutT>
__device__ __forceinline__ void store16_to(void* base, int N, int64_t m, int n_base, const float (&v)[16], bool vec) {
  OutT* out = static_cast<OutT*>(base) + m * static_cast<int64_t>(N) + n_base;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int n = n_base + q * 8;
    if (n >= N) break;
    float f[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = v[q * 8 + i];
    store8(out + q * 8, N - n, vec && n + 8 <= N, f);
  }
}

// One halving step of a column-wise max over the lanes of a warp: c[0, 2H)
// holds this lane's values of 2H columns; partners `lane ^ off` split them, the
// lane with the `off` bit set keeping the upper H.
template <int H>
__device__ __forceinline__ void colmax_halve(uint32_t (&c)[16], int lane, int off) {
  const bool upper = (lane & off) != 0;
#pragma unroll
  for (int i = 0; i < H; ++i) {
    const uint32_t lo = c[i], hi = c[i + H];
    const uint32_t give = upper ? lo : hi;
    const uint32_t keep = upper ? hi : lo;
    c[i] = max(keep, __shfl_xor_sync(0xffffffffu, give, off));
  }
}

// MLP hidden layer: act = silu(out) as the standalone SiLU kernel computes it
// from the stored out, and the per-column maxima of |fp16(act)| over this
// warp's 32 rows raised in the tile's shared column maxima (cmax_s, the 16
// columns of this group), which go to act_colmax (the next layer's outlier
// detection) once per tile.
template <typename OutT>
__device__ __forceinline__ void silu_epilogue16(const FwdEpiArgs& e, int64_t m, int n_base, bool row_ok,
                                                const float (&v)[16], bool vec, int lane, uint32_t* cmax_s) {
  float a[16];
  uint32_t mag[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    a[j] = silu_f(to_float(from_float<OutT>(v[j])));
    const float ar = to_float(from_float<OutT>(a[j]));
    mag[j] = row_ok ? (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(ar))) & 0x7FFFu) : 0u;
  }
  if (row_ok) store16_to<OutT>(e.act, e.N, m, n_base, a, vec);
  // max over the 32 lanes (rows) of each of the 16 columns by a halving
  // exchange: each step a lane hands the partner the half of its columns it
  // gives up and keeps the maxima of the other half; after four steps lane
  // pairs (l, l ^ 1) hold column 8 b4 + 4 b3 + 2 b2 + b1 of their lane bits
  colmax_halve<8>(mag, lane, 16);
  colmax_halve<4>(mag, lane, 8);
  colmax_halve<2>(mag, lane, 4);
  colmax_halve<1>(mag, lane, 2);
  const uint32_t mx = max(mag[0], __shfl_xor_sync(0xffffffffu, mag[0], 1));
  const int j = ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
  if ((lane & 1) == 0 && mx != 0u) atomicMax(cmax_s + j, mx);
}

template <typename OutT>
__device__ __forceinline__ void fwd_store16(const FwdEpiArgs& e, int64_t m, int n_base, const float (&v)[16],
                                            bool vec) {
  store16_to<OutT>(e.out, e.N, m, n_base, v, vec);
}

template <typename OutT>
__device__ __forceinline__ void fwd_add_residual16(const FwdEpiArgs& e, int64_t m, int n_base, float (&v)[16],
                                                   bool vec) {
  const OutT* res = static_cast<const OutT*>(e.residual) + m * static_cast<int64_t>(e.N) + n_base;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int n = n_base + q * 8;
    if (n >= e.N) break;
    float f[8];
    load8_float(res + q * 8, e.N - n, vec && n + 8 <= e.N, f);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[q * 8 + i] += f[i];
  }
}

// kSilu: the MLP hidden-layer epilogue (also writes silu(out) and raises the
// per-column maxima of |fp16(silu(out))|).
template <bool kSilu>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    fwd_gemm_kernel(const __grid_constant__ FwdGemmArgs g, const FwdEpiArgs e, int num_m, int num_n, int group) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* scb_s = reinterpret_cast<float*>(smem + kFwdStages * kFwdStageBytes);
  float* bias_s = scb_s + kPairN;
  uint32_t* colmax_s = reinterpret_cast<uint32_t*>(bias_s + kPairN);   // fused SiLU: the tile's column maxima
  Barriers* bars = reinterpret_cast<Barriers*>(colmax_s + kPairN);
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cid = static_cast<int>(cluster_id_x()), ncl = static_cast<int>(num_clusters_x());
  const int num_tiles = num_m * num_n;

  const int KB = (e.K_pad + kBK - 1) / kBK;
  const int nchunks = (KB + kChunkKB - 1) / kChunkKB;
  const int used = e.use_outliers ? e.st->used : 0;
  const int OB = (used + kBK - 1) / kBK;
  const int blocks = KB + OB;                      // pipeline stages per tile
  // accumulation units of a tile: groups of `per` 1024-product chunks (the
  // tile's plan word), then the outlier unit
  auto tile_units = [&](uint32_t plan, int& per, int& n_int, bool& fast) {
    per = max(1, min(nchunks, static_cast<int>(plan & 0xFFFFu)));
    fast = ((plan >> 16) & 1u) != 0;
    n_int = (nchunks + per - 1) / per;
    return n_int + (OB > 0 ? 1 : 0);
  };

  if (threadIdx.x == 0) init_barriers(bars, kEpiWarps);
  if (warp == kWarpMMA) {
    tmem_alloc_pair(&bars->tmem_base, 512);
    tmem_relinquish_pair();
  }
  if (warp == kWarpProducer && lane == 0) {
    tma_prefetch_desc(&g.tmA);
    tma_prefetch_desc(&g.tmB);
    if (OB > 0) {
      tma_prefetch_desc(&g.tmSA);
      tma_prefetch_desc(&g.tmSB);
    }
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t tmem_R = tmem;          // int32 running sum, columns [0, 256)
  const uint32_t tmem_X = tmem + 256;    // fp32 accumulation unit, columns [256, 512)

  if (warp == kWarpProducer) {
    if (lane == 0) {
      const uint32_t full0 = mapa_shared(&bars->full[0], 0);   // the even CTA's barriers
      int it = 0;
      bool ok = true;
      for (int t = cid; t < num_tiles && ok; t += ncl) {
        int tm, tn;
        tile_coords(t, num_m, num_n, group, tm, tn);
        const int m_cta = tm * kPairM + static_cast<int>(rank) * kCtaRows;
        const int n_cta = tn * kPairN + static_cast<int>(rank) * kCtaRows;
        for (int b = 0; b < blocks; ++b, ++it) {
          const int s = it % kFwdStages;
          const uint32_t ph = (it / kFwdStages) & 1;
          if (!mbar_wait(&bars->empty[s], ph ^ 1, abort_flag, e.st, kWhereProducer)) { ok = false; break; }
          uint8_t* sa = smem + s * kFwdStageBytes;
          uint8_t* sb = sa + kOpBytes;
          const uint32_t full_s = full0 + static_cast<uint32_t>(s) * 8u;
          // the even CTA expects the bytes of both CTAs' copies
          if (rank == 0) mbar_arrive_expect_tx(&bars->full[s], 2 * 2 * kOpBytes);
          if (b < KB) {
            tma_load_2d_pair(sa, &g.tmA, b * kBK, m_cta, full_s);
            tma_load_2d_pair(sb, &g.tmB, b * kBK, n_cta, full_s);   // fp16 weight codes
          } else {
            tma_load_2d_pair(sa, &g.tmSA, (b - KB) * kBK, m_cta, full_s);
            tma_load_2d_pair(sb, &g.tmSB, (b - KB) * kBK, n_cta, full_s);
          }
        }
      }
      // teardown: every issued copy (of both CTAs) must have landed before the
      // pair passes its final cluster barrier
      if (rank == 0)
        for (int j = max(0, it - kFwdStages); j < it; ++j)
          mbar_wait_teardown(&bars->full[j % kFwdStages], (j / kFwdStages) & 1, e.st);
    }
  } else if (warp == kWarpMMA) {
    if (rank == 0 && lane == 0) {
      const uint32_t idesc = make_idesc_f16(kPairM, kPairN, false, false);
      const uint64_t desc0 = make_sdesc(smem_u32(smem), 16, 1024, kSwizzle128B);   // stage 0, A, k = 0
      int it = 0, u = 0, tl = 0;
      bool ok = true;
      for (int t = cid; t < num_tiles && ok; t += ncl, ++tl) {
        int tm, tn;
        tile_coords(t, num_m, num_n, group, tm, tn);
        int per, n_int;
        bool fast;
        const int units0 = tile_units(e.plan[tm * num_n + tn], per, n_int, fast);
        // one int8 unit and outliers: the outlier unit accumulates in R's
        // columns while the int8 unit stays in X, with no drain between them;
        // R must first be free of the previous tile's output values
        const bool r_out = OB > 0 && n_int == 1;
        const int units = r_out ? 1 : units0;
        for (int uu = 0; uu < units && ok; ++uu, ++u) {
          // the epilogues of both CTAs released the accumulator of unit u-1
          if (u > 0 && !mbar_wait_cluster(&bars->acc_empty[0], (u - 1) & 1, abort_flag, e.st, kWhereMMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const bool is_int = uu < n_int;
          const int b0 = r_out ? 0 : is_int ? uu * per * kChunkKB : KB;
          const int b1 = r_out ? KB : is_int ? min(KB, b0 + per * kChunkKB) : blocks;
          // one run of blocks into one accumulator, or (r_out) the int8 blocks
          // into X and then the outlier blocks into R; each run's loop is kept
          // free of per-block branches (the issuing thread's latency per block
          // shows directly in the tile time)
          for (int seg = 0; seg < (r_out ? 2 : 1) && ok; ++seg) {
            const int c0 = seg == 0 ? b0 : KB, c1 = seg == 0 ? b1 : blocks;
            const uint32_t dst = seg == 0 ? tmem_X : tmem_R;
            if (seg == 1 && tl > 0 &&
                !mbar_wait_cluster(&bars->acc_empty[1], (tl - 1) & 1, abort_flag, e.st, kWhereMMA)) {
              ok = false;
              break;
            }
            for (int b = c0; b < c1; ++b, ++it) {
              const int s = it % kFwdStages;
              const uint32_t ph = (it / kFwdStages) & 1;
              if (!mbar_wait(&bars->full[s], ph, abort_flag, e.st, kWhereMMA)) { ok = false; break; }
              tc_fence_after();
              const uint64_t ad0 = desc0 + static_cast<uint64_t>(s * (kFwdStageBytes >> 4));
#pragma unroll
              for (int k = 0; k < kBK / 16; ++k) {
                const uint64_t ad = ad0 + 2 * k;
                const uint64_t bd = ad0 + (kOpBytes >> 4) + 2 * k;
                umma_f16_pair(dst, ad, bd, idesc, (b > c0 || k > 0) ? 1u : 0u);
              }
              umma_commit_pair_mc(&bars->empty[s], 0x3);
            }
          }
          if (ok) umma_commit_pair_mc(&bars->acc_full[0], 0x3);
        }
      }
      umma_commit_pair(&bars->teardown);
      mbar_wait_teardown(&bars->teardown, 0, e.st);
    }
  } else if (warp >= kWarpEpi0 && warp < kWarpEpi0 + kEpiWarps) {
    // ---- epilogue: 8 warps; lanes = this CTA's 128 rows, two column halves
    const int et = threadIdx.x - kWarpEpi0 * 32;
    const int quad = warp & 3;
    const int col0 = ((warp - kWarpEpi0) >> 2) * 128;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t acc_empty0 = mapa_shared(&bars->acc_empty[0], 0);
    const uint32_t acc_empty1 = mapa_shared(&bars->acc_empty[1], 0);   // R free again, once per tile
    const bool vec = (e.N % 8) == 0;
    int u = 0;
    bool ok = true;
    int prev_n0 = -1;
    // fused SiLU: the column maxima of a tile, gathered in shared memory by
    // every epilogue warp, go out with one global atomic per column
    auto flush_colmax = [&]() {
      if constexpr (kSilu) {
        if (prev_n0 >= 0) {
          const int n = prev_n0 + et;
          const uint32_t v = colmax_s[et];
          if (n < e.N && v != 0u) atomicMax(e.act_colmax + n, v);
        }
        colmax_s[et] = 0u;
      }
    };
    for (int t = cid; t < num_tiles && ok; t += ncl) {
      int tm, tn;
      tile_coords(t, num_m, num_n, group, tm, tn);
      const int n0 = tn * kPairN;
      named_bar_sync(kBarEpi, kEpiThreads);   // the previous tile no longer reads the vectors
      flush_colmax();
      prev_n0 = n0;
      {
        const int n = n0 + et;
        scb_s[et] = (n < e.N) ? e.SCB[n] : 0.f;
        bias_s[et] = (n < e.N && e.bias != nullptr) ? load_any(e.bias, e.bias_dt, n) : 0.f;
      }
      named_bar_sync(kBarEpi, kEpiThreads);
      const int64_t m = static_cast<int64_t>(tm) * kPairM + static_cast<int64_t>(rank) * kCtaRows + quad * 32 + lane;
      const bool row_ok = m < e.M;
      int per, n_int;
      bool small;   // every partial sum of the tile's units below 2^22: the fast exact conversion
      const int units0 = tile_units(e.plan[tm * num_n + tn], per, n_int, small);
      const bool r_out = OB > 0 && n_int == 1;   // as the MMA: the int8 unit in X, the outliers in R
      const int units = r_out ? 1 : units0;
      for (int uu = 0; uu < units; ++uu, ++u) {
        // all 256 epilogue threads agree, so none is left at a named barrier
        if (!named_bar_and(kBarEpi, kEpiThreads,
                           mbar_wait(&bars->acc_full[0], u & 1, abort_flag, e.st, kWhereEpi, kEpiSleepNs))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (uu < units - 1) {
          // an int8 chunk followed by more units: X -> R (exact int32)
#pragma unroll 1
          for (int gc = 0; gc < 128; gc += 32) {
            uint32_t x[32], r[32];
            tmem_ld32_nowait(tmem_X + lane_off + col0 + gc, x);
            if (uu > 0) tmem_ld32_nowait(tmem_R + lane_off + col0 + gc, r);
            tmem_ld_wait_tie(x, r);
            chunk_to_int(x, r, uu == 0, small);
            tmem_st32_nowait(tmem_R + lane_off + col0 + gc, r);
          }
          tmem_st_wait();
        } else {
          // last unit of the tile, phase 1: the fp32 output values before the
          // residual, written into R (over the running sum, or over the
          // outlier unit's sums), so that X can be handed back to the MMA
          // before the slower stores of phase 2
          const bool has_o = OB > 0;
          const bool r_live = has_o ? (n_int > 0) : (n_int > 1);
          const float rs = row_ok ? __fmul_rn(e.SCA[m], 1.0f / 16129.0f) : 0.f;
#pragma unroll 1
          for (int gc = 0; gc < 128; gc += 16) {
            uint32_t r[16], x[16];
            if (r_out) {   // r: the int8 unit from X; x: the outlier unit from R
              uint32_t xi[16];
              tmem_ld16_nowait(tmem_X + lane_off + col0 + gc, xi);
              tmem_ld16_nowait(tmem_R + lane_off + col0 + gc, x);
              tmem_ld_wait_tie16(xi, x);
              chunk_to_int(xi, r, true, small);
            } else {
              tmem_ld16_nowait(tmem_X + lane_off + col0 + gc, x);
              if (r_live) tmem_ld16_nowait(tmem_R + lane_off + col0 + gc, r);
              tmem_ld_wait_tie16(x, r);
              if (!has_o) {
                chunk_to_int(x, r, !r_live, small);   // the last int8 chunk is still in X
#pragma unroll
                for (int j = 0; j < 16; ++j) x[j] = 0u;   // no outlier term
              } else if (!r_live) {
#pragma unroll
                for (int j = 0; j < 16; ++j) r[j] = 0;
              }
            }
            const int nb = n0 + col0 + gc;
            if (e.acc_i32 != nullptr && row_ok && nb < e.N) {
              int32_t* dst = e.acc_i32 + m * static_cast<int64_t>(e.N);
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (nb + j < e.N) dst[nb + j] = static_cast<int32_t>(r[j]);
            }
            uint32_t vb[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float sc = __fmul_rn(rs, scb_s[col0 + gc + j]);
              vb[j] = __float_as_uint(__fadd_rn(
                  __fmaf_rn(static_cast<float>(static_cast<int32_t>(r[j])), sc, __uint_as_float(x[j])),
                  bias_s[col0 + gc + j]));
            }
            tmem_st16_nowait(tmem_R + lane_off + col0 + gc, vb);
          }
          tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(acc_empty0);
        if (uu == units - 1) {
          // phase 2, while the MMA starts the next tile: residual, rounding,
          // stores (and the fused SiLU) from the values in R
#pragma unroll 1
          for (int gc = 0; gc < 128; gc += 16) {
            uint32_t vb[16];
            tmem_ld16(tmem_R + lane_off + col0 + gc, vb);
            const int nb = n0 + col0 + gc;
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = row_ok ? __uint_as_float(vb[j]) : 0.f;
            if (row_ok && nb < e.N) {
              if (e.residual != nullptr) {
                switch (e.out_dt) {
                  case DT_F16: fwd_add_residual16<__half>(e, m, nb, v, vec); break;
                  case DT_BF16: fwd_add_residual16<__nv_bfloat16>(e, m, nb, v, vec); break;
                  default: fwd_add_residual16<float>(e, m, nb, v, vec); break;
                }
              }
              switch (e.out_dt) {
                case DT_F16: fwd_store16<__half>(e, m, nb, v, vec); break;
                case DT_BF16: fwd_store16<__nv_bfloat16>(e, m, nb, v, vec); break;
                default: fwd_store16<float>(e, m, nb, v, vec); break;
              }
            }
            if constexpr (kSilu) {
              if (nb < e.N) {   // warp-uniform: every lane takes part in the column reduction
                switch (e.out_dt) {
                  case DT_F16: silu_epilogue16<__half>(e, m, nb, row_ok, v, vec, lane, colmax_s + col0 + gc); break;
                  case DT_BF16:
                    silu_epilogue16<__nv_bfloat16>(e, m, nb, row_ok, v, vec, lane, colmax_s + col0 + gc);
                    break;
                  default: silu_epilogue16<float>(e, m, nb, row_ok, v, vec, lane, colmax_s + col0 + gc); break;
                }
              }
            }
            __syncwarp();
          }
          // phase 2 has read R: the next tile's outlier unit may accumulate there
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(acc_empty1);
        }
      }
    }
    if constexpr (kSilu) {
      named_bar_sync(kBarEpi, kEpiThreads);   // every warp added the last tile's maxima
      flush_colmax();
    }
  }

  tc_fence_before();
  cluster_sync();
  if (warp == kWarpMMA) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

// Odd CTA of a backward pair: forward "stage s converted" to the even CTA's
// ready[s] with a cluster-scope release, so that the converted tiles (written
// by this CTA's threads) are visible to the even CTA's MMA.  Relay r takes
// the stages it % kRelays == r.
__device__ __noinline__ void relay_loop(Barriers* bars, int cid, int ncl, int num_tiles, int NB, int r, int stages,
                                        volatile int* abort_flag, DevStatus* st) {
  const uint32_t ready0 = mapa_shared(&bars->ready[0], 0);
  int it = 0;
  for (int t = cid; t < num_tiles; t += ncl) {
    for (int b = 0; b < NB; ++b, ++it) {
      if (it % kRelays != r) continue;
      const int s = it % stages;
      if (!mbar_wait(&bars->cvt_done[s], (it / stages) & 1, abort_flag, st, kWhereCvt)) return;
      mbar_arrive_remote_release_cluster(ready0 + static_cast<uint32_t>(s) * 8u);
    }
  }
}

// ---------------------------------------------------------------------------
// Backward GEMM (transposed): D[k, m] = sum_n Wdq[n, k] * G16[m, n]
// ---------------------------------------------------------------------------
template <typename OutT>
__device__ __forceinline__ void bwd_store16(const BwdEpiArgs& e, int64_t kk, int m_base, const uint32_t (&x)[16]) {
  OutT* out = static_cast<OutT*>(e.grad_A);
  const OutT* add = static_cast<const OutT*>(e.addend);
  const float bv = e.bias != nullptr ? load_any(e.bias, e.bias_dt, kk) : 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int64_t mm = m_base + j;
    if (mm < e.M) {
      float v = __uint_as_float(x[j]);
      if (add != nullptr) v = __fadd_rn(v, to_float(add[mm * e.K + kk]));
      if (e.bias != nullptr) v = __fadd_rn(v, bv);
      out[mm * e.K + kk] = from_float<OutT>(v);
    }
  }
}

// The 16 fp32 values x[j] (tokens m_base + j) of this lane's output feature,
// stored as 8-feature rows: within each group of 8 lanes (8 consecutive
// features) an 8 x 8 block of tokens x features is transposed in three
// exchange rounds, after which lane i of the group holds token 8 h + i of
// block h for the group's 8 features and stores them with one 16-byte store
// (two for fp32).  kg: the group's first feature; K % 8 == 0 and the output
// rows are 16-byte aligned, so a group is wholly in or out of range.  The
// addend, then the bias, are added after the exchange, in the order of the
// scalar path.  Every lane of the warp calls this (the exchange), whatever
// its range checks.
template <typename OutT>
__device__ __forceinline__ void bwd_store16_rows(const BwdEpiArgs& e, int64_t kg, int m_base, const uint32_t (&x)[16],
                                                 int lane) {
  OutT* out = static_cast<OutT*>(e.grad_A);
  const OutT* add = static_cast<const OutT*>(e.addend);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(x[8 * h + j]);
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) {
      const bool up = (lane & o) != 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j & o) continue;
        const float send = up ? v[j] : v[j + o];
        const float recv = __shfl_xor_sync(0xffffffffu, send, o);
        if (up)
          v[j] = recv;
        else
          v[j + o] = recv;
      }
    }
    const int64_t mm = m_base + 8 * h + (lane & 7);
    if (mm >= e.M || kg >= e.K) continue;
    OutT* dst = out + mm * e.K + kg;
    if (add != nullptr) {
      const OutT* src = add + mm * e.K + kg;
#pragma unroll
      for (int f = 0; f < 8; ++f) v[f] = __fadd_rn(v[f], to_float(src[f]));
    }
    if (e.bias != nullptr) {
#pragma unroll
      for (int f = 0; f < 8; ++f) v[f] = __fadd_rn(v[f], load_any(e.bias, e.bias_dt, kg + f));
    }
    if constexpr (sizeof(OutT) == 4) {
      reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
      reinterpret_cast<float4*>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
    } else {
      uint4 o;
      OutT* q = reinterpret_cast<OutT*>(&o);
#pragma unroll
      for (int f = 0; f < 8; ++f) q[f] = from_float<OutT>(v[f]);
      *reinterpret_cast<uint4*>(dst) = o;
    }
  }
}

// Two fp32 values times the splatted scale (one packed IEEE multiply, the
// same rounding as two scalar ones), rounded to a 16-bit pair; e0 in the low
// half.
template <bool kBf16>
__device__ __forceinline__ uint32_t mul2_to_16(float e0, float e1, uint64_t am2) {
  uint32_t out;
  if (kBf16) {
    asm("{\n .reg .b64 x, p;\n .reg .b32 lo, hi;\n mov.b64 x, {%1, %2};\n mul.rn.f32x2 p, x, %3;\n"
        " mov.b64 {lo, hi}, p;\n cvt.rn.bf16x2.f32 %0, hi, lo;\n}"
        : "=r"(out)
        : "f"(e0), "f"(e1), "l"(am2));
  } else {
    asm("{\n .reg .b64 x, p;\n .reg .b32 lo, hi;\n mov.b64 x, {%1, %2};\n mul.rn.f32x2 p, x, %3;\n"
        " mov.b64 {lo, hi}, p;\n cvt.rn.f16x2.f32 %0, hi, lo;\n}"
        : "=r"(out)
        : "f"(e0), "f"(e1), "l"(am2));
  }
  return out;
}

// 16 packed 4-bit codes (8 bytes, the even element of each pair in the high
// nibble) -> lv[code] * am rounded to the operand type; element 2i in the low
// half of word i.  The level table sits in shared memory at a fixed address:
// the byte offsets 4 * code are cut out of the packed bytes with two masks,
// and each lookup is one byte extract and one shared load.
template <bool kBf16>
__device__ __forceinline__ void nf4x16_decode(uint2 v, uint64_t am2, const float* lv_s, uint4& o0, uint4& o1) {
  uint32_t w[8];
  const char* base = reinterpret_cast<const char*>(lv_s);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t x = h ? v.y : v.x;
    const uint32_t hi4 = (x >> 2) & 0x3C3C3C3Cu;   // 4 * high nibble of each byte
    const uint32_t lo4 = (x << 2) & 0x3C3C3C3Cu;   // 4 * low nibble of each byte
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float e0 = *reinterpret_cast<const float*>(base + __byte_perm(hi4, 0u, 0x4440u + i));
      const float e1 = *reinterpret_cast<const float*>(base + __byte_perm(lo4, 0u, 0x4440u + i));
      w[4 * h + i] = mul2_to_16<kBf16>(e0, e1, am2);
    }
  }
  o0 = make_uint4(w[0], w[1], w[2], w[3]);
  o1 = make_uint4(w[4], w[5], w[6], w[7]);
}

// grad_bias partial sums of one kBiasChunkRows-row chunk c of G over the 64
// columns [n0, n0 + 64), by one warp, read from global memory (G is constant
// during the GEMM, so no stage of the pipeline is involved):
//   partial[c, n] = sum_{y=0..7} ( sum_{j=0..15} G[128 c + y + 8 j, n] ),
// each inner sum in increasing j from 0.f, the outer one in increasing y
// from 0.f -- the order of the grad_output prepass, so both give the same
// bits.  Lane (cg, yy) = (lane & 7, lane >> 3) loads 8 columns (16 bytes) of
// the rows of the two lanes y = yy and yy + 4; lanes cg then gather the
// eight sums in order with shuffles.  Rows past M add nothing; N is a
// multiple of 8, so a 16-byte group is all inside or all past N.
template <typename T>
__device__ __forceinline__ void bias_chunk_sums(const T* __restrict__ G, int M, int N, int c, int n0,
                                                float* __restrict__ partial, int lane) {
  const int cg = lane & 7, yy = lane >> 3;
  const int n = n0 + cg * 8;
  const bool col_ok = n < N;
  float p[2][8];
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int i = 0; i < 8; ++i) p[h][i] = 0.f;
  const int64_t r0 = static_cast<int64_t>(c) * kBiasChunkRows;
#pragma unroll 4
  for (int j = 0; j < kBiasChunkRows / 8; ++j) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t r = r0 + yy + 4 * h + 8 * j;
      if (col_ok && r < M) {
        float f[8];
        load8_float(G + r * N + n, 8, true, f);
#pragma unroll
        for (int i = 0; i < 8; ++i) p[h][i] += f[i];
      }
    }
  }
  float out[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float acc = 0.f;
#pragma unroll
    for (int y = 0; y < 8; ++y) acc += __shfl_sync(0xffffffffu, p[y >> 2][i], cg + 8 * (y & 3));
    out[i] = acc;
  }
  if (yy == 0 && col_ok) {
    float* dst = partial + static_cast<int64_t>(c) * N + n;
    reinterpret_cast<float4*>(dst)[0] = make_float4(out[0], out[1], out[2], out[3]);
    reinterpret_cast<float4*>(dst)[1] = make_float4(out[4], out[5], out[6], out[7]);
  }
}

// Fused modes: the A operand (the dequantized weight tile) is rebuilt per
// stage from the int8 or 4-bit weight tiles by the converter warps;
// kModeMat: it is loaded by TMA from the materialized WdqT (K-major, like
// G16) and the converter, weight-producer and relay warps stay idle.
template <int kMode>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kBwdThreads, 1)
    bwd_gemm_kernel(const __grid_constant__ BwdGemmArgs g, const BwdEpiArgs e, int num_k, int num_m, int group,
                    int split) {
  using Geo = BwdGeom<kMode>;
  constexpr bool kFused = Geo::kFused;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Barriers* bars = reinterpret_cast<Barriers*>(smem + Geo::kTiles);
  volatile int* abort_flag = &bars->abort_flag;
  uint8_t* i8_ring = smem + Geo::kI8Offset;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cid = static_cast<int>(cluster_id_x()), ncl = static_cast<int>(num_clusters_x());
  // `split` raster tiles at the end run as two 256-token halves each
  // (split_tile): num_tiles counts the tiles as run
  const int full_tiles = num_k * num_m - split;
  const int num_tiles = full_tiles + 2 * split;
  const int NB = (e.N + kBK - 1) / kBK;   // reduction blocks over n
  auto tile_of = [&](int t, int& tm, int& tk, int& m_base, int& nsub) {
    split_tile<Geo::kTileTokens>(t, full_tiles, num_m, num_k, group, tm, tk, m_base, nsub);
  };

  if (threadIdx.x == 0) init_barriers(bars, kBwdEpiWarps);
  __shared__ float lv_s[16];   // 4-bit modes: the code levels
  if (Geo::kNf4 && threadIdx.x < 16) lv_s[threadIdx.x] = e.lv[threadIdx.x];
  if (warp == kWarpMMA) {
    tmem_alloc_pair(&bars->tmem_base, 512);
    tmem_relinquish_pair();
  }
  if (warp == kWarpProducer && lane == 0) {
    tma_prefetch_desc(&g.tmG);
    if (!kFused) tma_prefetch_desc(&g.tmWT);
  }
  if (kFused && warp == kWarpI8Producer && lane == 0) tma_prefetch_desc(&g.tmW);
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;   // 512 columns: two 256-column accumulators, or one 512-column one

  if (warp == kWarpProducer) {
    // ---- G16 tiles (and WdqT tiles when materialized): both CTAs' copies
    // complete on the even CTA's barrier
    if (lane == 0) {
      // fused: the G16 copies complete on ready[s], the one barrier the MMA
      // waits on; materialized: on full[s]
      uint64_t* const land = kFused ? bars->ready : bars->full;
      const uint32_t full0 = mapa_shared(&land[0], 0);
      int it = 0;
      bool ok = true;
      for (int t = cid; t < num_tiles && ok; t += ncl) {
        int tm, tk, m_base, nsub;
        tile_of(t, tm, tk, m_base, nsub);
        const int m_cta = m_base + static_cast<int>(rank) * kCtaRows;
        const int k_cta = tk * kPairM + static_cast<int>(rank) * kCtaRows;
        for (int b = 0; b < NB; ++b, ++it) {
          const int s = it % Geo::kStages;
          const uint32_t ph = (it / Geo::kStages) & 1;
          if (!mbar_wait(&bars->empty[s], ph ^ 1, abort_flag, e.st, kWhereProducer)) { ok = false; break; }
          // the even CTA expects both CTAs' bytes of this stage
          if (rank == 0) mbar_arrive_expect_tx(&land[s], 2 * (kFused ? nsub : 2) * kOpBytes);
          const uint32_t full_s = full0 + static_cast<uint32_t>(s) * 8u;
          uint8_t* st_base = smem + s * Geo::kStageBytes;
          if (!kFused) tma_load_2d_pair(st_base, &g.tmWT, b * kBK, k_cta, full_s);   // WdqT[k:+128][n:+64]
#pragma unroll
          for (int u = 0; u < Geo::kSub; ++u)   // G16[m:+128][n:+64] of token sub-tile u
            if (u < nsub) tma_load_2d_pair(st_base + (1 + u) * kOpBytes, &g.tmG, b * kBK, m_cta + u * kPairN, full_s);
        }
      }
      if (rank == 0)
        for (int j = max(0, it - Geo::kStages); j < it; ++j)
          mbar_wait_teardown(&land[j % Geo::kStages], (j / Geo::kStages) & 1, e.st);
    }
  } else if (warp == kWarpI8Producer) {
    // ---- weight tiles, this CTA's own ring: int8 CB[n:+64][k:+128]; 4-bit,
    // input gradient: packed[n:+64][k:+128] (64 bytes a row); 4-bit, forward:
    // packed[n:+128][k:+64] (32 bytes a row)
    // (x = the byte column, y = the row of the weight)
    auto ring_xy = [&](int tk, int b, int& x, int& y) {
      const int r_cta = tk * kPairM + static_cast<int>(rank) * kCtaRows;
      if (kMode == kModeNf4) {
        x = b * (kBK / 2);
        y = r_cta;
      } else {
        x = Geo::kNf4 ? r_cta / 2 : r_cta;
        y = b * kBK;
      }
    };
    if (kFused && lane == 0) {
      int it = 0;
      bool ok = true;
      for (int t = cid; t < num_tiles && ok; t += ncl) {
        int tm, tk, m_base, nsub;
        tile_of(t, tm, tk, m_base, nsub);
        for (int b = 0; b < NB; ++b, ++it) {
          const int j = it % kI8Stages;
          const uint32_t ph = (it / kI8Stages) & 1;
          if (!mbar_wait(&bars->i8_empty[j], ph ^ 1, abort_flag, e.st, kWhereProducer)) { ok = false; break; }
          mbar_arrive_expect_tx(&bars->i8_full[j], Geo::kRingBytes);
          int x, y;
          ring_xy(tk, b, x, y);
          tma_load_2d(i8_ring + j * Geo::kRingBytes, &g.tmW, x, y, &bars->i8_full[j]);
          // the copy above waits on DRAM for about a microsecond; a tile a few
          // stages ahead is pulled into L2 now, so its own copy finds it there
          int bp = b + kI8PrefetchAhead, tp = t;
          while (bp >= NB && tp < num_tiles) {
            bp -= NB;
            tp += ncl;
          }
          if (tp < num_tiles) {
            int tmp, tkp, mbp, nsp;
            tile_of(tp, tmp, tkp, mbp, nsp);
            ring_xy(tkp, bp, x, y);
            tma_prefetch_l2_2d(&g.tmW, x, y);
          }
        }
      }
      for (int j = max(0, it - kI8Stages); j < it; ++j)
        mbar_wait_teardown(&bars->i8_full[j % kI8Stages], (j / kI8Stages) & 1, e.st);
    }
  } else if (warp == kWarpMMA) {
    if (rank == 0 && lane == 0) {
      // A, int8 and 4-bit input gradient: MN-major, 128B swizzle; MN atoms
      // (64 k) 1024 B apart, K atoms (8 n) 2048 B apart.  Materialized and
      // 4-bit forward: K-major like B.  ab_fmt: bf16 operands.
      const uint32_t idesc = make_idesc_f16(kPairM, kPairN, Geo::kAmn, false) | e.ab_fmt;
      // stage 0's descriptors at k = 0 (the start-address field, in 16-byte
      // units, then takes the offsets within shared memory below 256 KB)
      const uint32_t base0 = smem_u32(smem);
      const uint64_t adesc0 = Geo::kAmn ? make_sdesc(base0, 1024, 2048, kSwizzle128B)
                                        : make_sdesc(base0, 16, 1024, kSwizzle128B);
      const uint64_t bdesc0 = make_sdesc(base0 + kOpBytes, 16, 1024, kSwizzle128B);
      int it = 0, tl = 0;
      bool ok = true;
      for (int t = cid; t < num_tiles && ok; t += ncl, ++tl) {
        int tm, tk, m_base, nsub;
        tile_of(t, tm, tk, m_base, nsub);
        const int buf = tl % Geo::kAccBufs;
        const int use = tl / Geo::kAccBufs;
        if (use > 0 && !mbar_wait_cluster(&bars->acc_empty[buf], (use - 1) & 1, abort_flag, e.st, kWhereMMA)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(buf) * 256u;
        for (int b = 0; b < NB; ++b, ++it) {
          const int s = it % Geo::kStages;
          const uint32_t ph = (it / Geo::kStages) & 1;
          if (kFused ? !mbar_wait_cluster(&bars->ready[s], ph, abort_flag, e.st, kWhereMMA)
                     : !mbar_wait(&bars->full[s], ph, abort_flag, e.st, kWhereMMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t st16 = static_cast<uint64_t>(s * (Geo::kStageBytes >> 4));   // the stage, 16-byte units
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint64_t ad = adesc0 + st16 + (Geo::kAmn ? k * (4096 >> 4) : 2 * k);
#pragma unroll
            for (int u = 0; u < Geo::kSub; ++u) {   // token sub-tile u -> accumulator columns [256 u, 256 u + 256)
              if (u >= nsub) break;
              const uint64_t bd = bdesc0 + st16 + u * (kOpBytes >> 4) + 2 * k;
              umma_f16_pair(d + static_cast<uint32_t>(u) * 256u, ad, bd, idesc, (b > 0 || k > 0) ? 1u : 0u);
            }
          }
          umma_commit_pair_mc(&bars->empty[s], 0x3);
        }
        if (ok) umma_commit_pair_mc(&bars->acc_full[buf], 0x3);
      }
      umma_commit_pair(&bars->teardown);
      mbar_wait_teardown(&bars->teardown, 0, e.st);
    } else if (kFused && rank == 1 && lane == 0) {
      relay_loop(bars, cid, ncl, num_tiles, NB, 0, Geo::kStages, abort_flag, e.st);
    }
  } else if (warp == kWarpRelay0 || warp == kWarpRelay0 + 1 || warp == kWarpRelayLast) {
    if (kFused && rank == 1 && lane == 0)
      relay_loop(bars, cid, ncl, num_tiles, NB, warp == kWarpRelayLast ? 3 : 1 + (warp - kWarpRelay0), Geo::kStages,
                 abort_flag, e.st);
  } else if (warp < kBwdWarpEpi0) {
    if constexpr (kMode == kModeI8) {
      // ---- converters: CB int8 [64 n][128 k] (128B-swizzled rows) -> Wdq^T
      // fp16, MN-major 128B-swizzled.  All eight warps work on every stage: a
      // thread takes the 16-byte chunk q of rows nl0 and nl0 + 32 (16 k x 1 n
      // each).  The 8 lanes of a quarter warp take 8 consecutive rows of one
      // chunk column, so that with both tiles swizzled their 16-byte loads and
      // stores fall in 8 different bank groups.  The two row scales of a stage
      // are loaded one stage ahead, so that their L2 latency overlaps the wait
      // for the next tile.
      const int gt = threadIdx.x - kWarpCvt0 * 32;   // 0..255
      const uint64_t negc2 = f32x2_splat(-8388736.0f);   // -(2^23 + 128)
      const int r = gt & 7;                          // row within an 8-row atom
      const int q = (gt >> 3) & 7;                   // 16-byte chunk of the 128-byte int8 row
      const int nl0 = r + 8 * (gt >> 6);             // rows nl0 and nl0 + 32 of every int8 tile
      auto load_scb = [&](int b, float (&f)[2]) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int n = b * kBK + nl0 + 32 * j;
          f[j] = n < e.N ? __ldg(e.SCB + n) : 0.f;
        }
      };
      float scb_next[2];
      load_scb(0, scb_next);
      int it = 0;
      bool go = true;
      for (int t = cid; t < num_tiles && go; t += ncl) {
        for (int b = 0; b < NB; ++b, ++it) {
          const float scb_cur[2] = {scb_next[0], scb_next[1]};
          load_scb(b + 1 < NB ? b + 1 : 0, scb_next);
          const int s = it % Geo::kStages;
          const uint32_t ph = (it / Geo::kStages) & 1;
          const int j8 = it % kI8Stages;
          if (!__all_sync(0xffffffffu,
                          mbar_wait(&bars->i8_full[j8], (it / kI8Stages) & 1, abort_flag, e.st, kWhereCvt))) {
            go = false;
            break;
          }
          const uint8_t* src = i8_ring + j8 * kI8Bytes;
          uint4 v[2];
#pragma unroll
          for (int j = 0; j < 2; ++j) v[j] = ld_shared_v4(src + (nl0 + 32 * j) * 128 + ((q ^ r) << 4));
          // the operand slot is free once the pair's MMAs of its previous use completed
          if (!__all_sync(0xffffffffu, mbar_wait(&bars->empty[s], ph ^ 1, abort_flag, e.st, kWhereCvt))) {
            go = false;
            break;
          }
          uint8_t* sa = smem + s * Geo::kStageBytes;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const uint64_t f2 = f32x2_splat(__fmul_rn(scb_cur[j], 1.0f / 127.0f));
            const int i = (nl0 >> 3) + 4 * j;        // K atom (8 n) of row nl0 + 32 j
            const int ja = q >> 2;                   // MN atom (64 k)
            const int c0 = (q & 3) * 2;              // 16-byte chunk in the 128-byte row
            uint4 o0, o1;
            i8x4_scale_to_h4(v[j].x, negc2, f2, o0.x, o0.y);
            i8x4_scale_to_h4(v[j].y, negc2, f2, o0.z, o0.w);
            i8x4_scale_to_h4(v[j].z, negc2, f2, o1.x, o1.y);
            i8x4_scale_to_h4(v[j].w, negc2, f2, o1.z, o1.w);
            uint8_t* rowp = sa + i * 2048 + ja * 1024 + r * 128;
            st_shared_v4(rowp + ((c0 ^ r) << 4), o0);
            st_shared_v4(rowp + (((c0 + 1) ^ r) << 4), o1);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&bars->i8_empty[j8]);
            // the even CTA's MMA thread reads this CTA's tiles: local arrive there,
            // a relay (cluster-scope release) from the odd CTA
            mbar_arrive(rank == 0 ? &bars->ready[s] : &bars->cvt_done[s]);
          }
        }
      }
    } else if constexpr (Geo::kNf4) {
      // ---- converters, 4-bit codes -> Wdq = lv[code] * absmax in the operand
      // type.  Every thread takes two (row, 16-code segment) items of each
      // weight tile.  Input gradient: tile [64 n][128 k] -> Wdq^T MN-major,
      // rows nl0 and nl0 + 32, segment q, the thread layout of the int8
      // converters (same output positions).  Forward: tile [128 n][64 k] ->
      // Wdq K-major (8-row atoms of 128-byte rows, 16-byte chunks swizzled by
      // the row), rows rr0 and rr0 + 64, segment sg; a quarter warp reads 64
      // consecutive bytes and writes 8 distinct bank groups.  The absmax
      // values of a stage are loaded one stage ahead.
      const int gt = threadIdx.x - kWarpCvt0 * 32;   // 0..255
      const bool bf16 = e.ab_fmt != 0u;
      int row[2], seg;
      if (kMode == kModeNf4T) {
        seg = (gt >> 3) & 7;
        row[0] = (gt & 7) + 8 * (gt >> 6);
        row[1] = row[0] + 32;
      } else {
        seg = gt & 3;
        row[0] = gt >> 2;
        row[1] = row[0] + 64;
      }
      constexpr int kRowBytes = kMode == kModeNf4T ? 64 : 32;
      // first output row of this CTA in tile t
      auto cta_row0 = [&](int t) {
        int tm, tk, m_base, nsub;
        tile_of(t, tm, tk, m_base, nsub);
        return tk * kPairM + static_cast<int>(rank) * kCtaRows;
      };
      // the absmax values of stage b of a tile whose CTA rows start at r_cta
      auto load_am = [&](int r_cta, int b, float (&f)[2]) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          int n, kb;
          bool ok;
          if (kMode == kModeNf4T) {   // weight row n = reduction index, block of this CTA's k
            n = b * kBK + row[j];
            kb = (r_cta >> 6) + (seg >> 2);
            ok = n < e.N;
          } else {                    // weight row n = output row, block b of the reduction
            n = r_cta + row[j];
            kb = b;
            ok = n < e.K;
          }
          f[j] = ok && kb < e.nblk ? __ldg(e.absmax + static_cast<int64_t>(n) * e.nblk + kb) : 0.f;
        }
      };
      float am_next[2] = {0.f, 0.f};
      int r_next = cid < num_tiles ? cta_row0(cid) : 0;
      if (cid < num_tiles) load_am(r_next, 0, am_next);
      int it = 0;
      bool go = true;
      for (int t = cid; t < num_tiles && go; t += ncl) {
        const int r_cur = r_next;
        if (t + ncl < num_tiles) r_next = cta_row0(t + ncl);
        for (int b = 0; b < NB; ++b, ++it) {
          const float am[2] = {am_next[0], am_next[1]};
          if (b + 1 < NB) {
            load_am(r_cur, b + 1, am_next);
          } else if (t + ncl < num_tiles) {
            load_am(r_next, 0, am_next);
          }
          const int s = it % Geo::kStages;
          const uint32_t ph = (it / Geo::kStages) & 1;
          const int j8 = it % kI8Stages;
          if (!__all_sync(0xffffffffu,
                          mbar_wait(&bars->i8_full[j8], (it / kI8Stages) & 1, abort_flag, e.st, kWhereCvt))) {
            go = false;
            break;
          }
          const uint8_t* src = i8_ring + j8 * Geo::kRingBytes;
          uint2 v[2];
#pragma unroll
          for (int j = 0; j < 2; ++j) v[j] = ld_shared_v2(src + row[j] * kRowBytes + seg * 8);
          if (!__all_sync(0xffffffffu, mbar_wait(&bars->empty[s], ph ^ 1, abort_flag, e.st, kWhereCvt))) {
            go = false;
            break;
          }
          uint8_t* sa = smem + s * Geo::kStageBytes;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            uint4 o0, o1;
            const uint64_t am2 = f32x2_splat(am[j]);
            if (bf16) {
              nf4x16_decode<true>(v[j], am2, lv_s, o0, o1);
            } else {
              nf4x16_decode<false>(v[j], am2, lv_s, o0, o1);
            }
            const int r = row[j] & 7;
            int c0;
            uint8_t* rowp;
            if (kMode == kModeNf4T) {
              rowp = sa + (row[j] >> 3) * 2048 + (seg >> 2) * 1024 + r * 128;
              c0 = (seg & 3) * 2;
            } else {
              rowp = sa + (row[j] >> 3) * 1024 + r * 128;
              c0 = seg * 2;
            }
            st_shared_v4(rowp + ((c0 ^ r) << 4), o0);
            st_shared_v4(rowp + (((c0 + 1) ^ r) << 4), o1);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&bars->i8_empty[j8]);
            mbar_arrive(rank == 0 ? &bars->ready[s] : &bars->cvt_done[s]);
          }
        }
      }
    }
  } else {
    // ---- epilogue: lanes = this CTA's 128 output features k, columns = the
    // tile's tokens (column c of the accumulator is token m_base + c).
    // Warps 10-13 take the first half of the columns, warps 18-21 the second.
    const int quad = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t acc_empty_pair[2] = {mapa_shared(&bars->acc_empty[0], 0), mapa_shared(&bars->acc_empty[1], 0)};
    const int ew = (warp >= kBwdWarpEpi1 ? 4 : 0) + quad;   // epilogue warp 0..7
    // output rows of whole 16-byte groups of 8 features (and a 16-byte
    // aligned addend): the transposed 16-byte stores; else one scalar store
    // per element (2-byte stores scattered over 16 rows cost the epilogue
    // about 13 us per tile against 1 us for the transposed ones)
    const bool rows16 = (e.K % 8) == 0 && (reinterpret_cast<uintptr_t>(e.grad_A) & 15u) == 0 &&
                        (reinterpret_cast<uintptr_t>(e.addend) & 15u) == 0;
    int tl = 0;
    for (int t = cid; t < num_tiles; t += ncl, ++tl) {
      int tm, tk, m_base, nsub;
      tile_of(t, tm, tk, m_base, nsub);
      const int half_w = nsub * (kPairN / 2);              // this warp's columns
      const int col0 = warp >= kBwdWarpEpi1 ? half_w : 0;
      const int buf = tl % Geo::kAccBufs;
      if (e.partial != nullptr) {
        // while the tensor cores run this tile: the grad_bias partial sums of
        // the reduction blocks b = tk, tk + num_k, ... over this CTA's token
        // chunks of the tile (every (chunk, block) is owned by exactly one
        // tile), one (chunk, block) item per warp in turn
        int item = 0;
        for (int b = tk; b < NB; b += num_k) {
          for (int u = 0; u < nsub; ++u, ++item) {
            const int c = (m_base + u * kPairN) / kBiasChunkRows + static_cast<int>(rank);
            if (item % kBwdEpiWarps != ew || c * kBiasChunkRows >= e.M) continue;
            if (e.gsum_dt == DT_BF16)
              bias_chunk_sums(static_cast<const __nv_bfloat16*>(e.gsum), e.M, e.N, c, b * kBK, e.partial, lane);
            else
              bias_chunk_sums(static_cast<const __half*>(e.gsum), e.M, e.N, c, b * kBK, e.partial, lane);
          }
        }
      }
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->acc_full[buf], (tl / Geo::kAccBufs) & 1, abort_flag, e.st,
                                             kWhereEpi, kEpiSleepNs)))
        break;
      tc_fence_after();
      const int64_t kk = static_cast<int64_t>(tk) * kPairM + static_cast<int64_t>(rank) * kCtaRows + quad * 32 + lane;
      const int64_t kg = kk - (lane & 7);   // first feature of this lane's group of 8
      const uint32_t d = tmem + static_cast<uint32_t>(buf) * 256u + lane_off + static_cast<uint32_t>(col0);
      const int m0 = m_base + col0;
      auto store = [&](const uint32_t(&x)[16], int gc) {
        if (rows16) {   // 16-byte stores of 8 features (every lane takes part in the exchange)
          switch (e.dt) {
            case DT_F16: bwd_store16_rows<__half>(e, kg, m0 + gc, x, lane); break;
            case DT_BF16: bwd_store16_rows<__nv_bfloat16>(e, kg, m0 + gc, x, lane); break;
            default: bwd_store16_rows<float>(e, kg, m0 + gc, x, lane); break;
          }
        } else if (kk < e.K) {
          switch (e.dt) {
            case DT_F16: bwd_store16<__half>(e, kk, m0 + gc, x); break;
            case DT_BF16: bwd_store16<__nv_bfloat16>(e, kk, m0 + gc, x); break;
            default: bwd_store16<float>(e, kk, m0 + gc, x); break;
          }
        }
      };
      // two register buffers: the stores of one overlap the TMEM load of the other
      uint32_t xa[16], xb[16];
      tmem_ld16_nowait(d, xa);
      tmem_ld_wait_tie16(xa, xb);
#pragma unroll 1
      for (int gc = 0; gc < half_w; gc += 32) {
        tmem_ld16_nowait(d + gc + 16, xb);
        store(xa, gc);
        tmem_ld_wait_tie16(xa, xb);
        if (gc + 32 < half_w) tmem_ld16_nowait(d + gc + 32, xa);
        store(xb, gc + 16);
        tmem_ld_wait_tie16(xa, xb);
        __syncwarp();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(acc_empty_pair[buf]);
    }
  }

  tc_fence_before();
  cluster_sync();
  if (warp == kWarpMMA) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

// Forward prepass: CB int8 codes -> the same values as fp16 (exact).  One
// warp per (row, 1024-column chunk): four rounds in which lane l converts the
// 8 codes at 256 u + 8 l, so that every load (256 bytes) and every store (512
// bytes) of the warp is contiguous; the chunk's sum of squares of the codes
// (dp4a) raises the row tile's entry of bsq, the weight side of the
// accumulation plan.  Two work items per iteration, all their loads first.
__global__ void __launch_bounds__(256) widen_codes_kernel(const int8_t* __restrict__ CB, __half* __restrict__ CBh,
                                                          int64_t N, int64_t k_pad, int nchunks,
                                                          uint32_t* __restrict__ bsq) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * 8;
  const int64_t total = N * nchunks;
  // the bounds are uniform over the warp, so the shuffles below are safe
  for (int64_t w0 = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5); w0 < total; w0 += 2 * nwarps) {
    uint2 v[2][4];
    int64_t n[2];
    int c[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int64_t w = w0 + i * nwarps;
      n[i] = w < total ? w / nchunks : 0;
      c[i] = static_cast<int>(w - n[i] * nchunks);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t k = static_cast<int64_t>(c[i]) * 1024 + u * 256 + lane * 8;
        v[i][u] = (w < total && k < k_pad)   // k_pad is a multiple of 16: a group of 8 is all in or all out
                      ? __ldg(reinterpret_cast<const uint2*>(CB + n[i] * k_pad + k))
                      : make_uint2(0u, 0u);
      }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      if (w0 + i * nwarps >= total) break;
      int sq = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t k = static_cast<int64_t>(c[i]) * 1024 + u * 256 + lane * 8;
        if (k < k_pad) {
          const uint2 x = v[i][u];
          sq = __dp4a(static_cast<int>(x.x), static_cast<int>(x.x), sq);
          sq = __dp4a(static_cast<int>(x.y), static_cast<int>(x.y), sq);
          uint4 o;
          i8x4_to_h4(x.x, o.x, o.y);
          i8x4_to_h4(x.y, o.z, o.w);
          *reinterpret_cast<uint4*>(CBh + n[i] * k_pad + k) = o;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
      if (lane == 0 && sq != 0) atomicMax(bsq + (n[i] >> 8) * nchunks + c[i], static_cast<uint32_t>(sq));
    }
  }
}

// The accumulation plan (see launch_unit_plan): one block per row tile tm of
// the first operand, its chunk sums staged in shared memory, one thread per
// column tile tn.  L is searched downwards from all chunks; uniform data stop
// at the first candidate.
constexpr int kPlanMaxChunks = 160;   // K <= 163840
__global__ void __launch_bounds__(256) unit_plan_kernel(const uint32_t* __restrict__ asq,
                                                        const uint32_t* __restrict__ bsq, int num_n, int nchunks,
                                                        uint32_t* __restrict__ plan) {
  __shared__ uint32_t a_s[kPlanMaxChunks];
  const int tm = blockIdx.x;
  for (int c = threadIdx.x; c < nchunks; c += blockDim.x) a_s[c] = asq[static_cast<int64_t>(tm) * nchunks + c];
  __syncthreads();
  constexpr unsigned long long kExact = 1ull << 48, kFast = 1ull << 44;
  for (int tn = threadIdx.x; tn < num_n; tn += blockDim.x) {
    const uint32_t* b = bsq + static_cast<int64_t>(tn) * nchunks;
    int best = 1;
    bool fast = true;
    for (int L = nchunks; L >= 1; --L) {
      bool ok = true, f = true;
      for (int c0 = 0; c0 < nchunks && ok; c0 += L) {
        unsigned long long sa = 0, sb = 0;
        for (int c = c0; c < min(nchunks, c0 + L); ++c) {
          sa += a_s[c];
          sb += b[c];
        }
        const unsigned long long p = sa * sb;   // < 160^2 * 2^48: no overflow
        ok = p < kExact;
        f = f && p < kFast;
      }
      if (ok) {
        best = L;
        fast = f;
        break;
      }
    }
    plan[static_cast<int64_t>(tm) * num_n + tn] = static_cast<uint32_t>(best) | (fast ? 1u << 16 : 0u);
  }
}

int g_pairs_fwd[64] = {};   // resident pairs per device, per kernel
int g_pairs_fwd_silu[64] = {};
int g_pairs_bwd[4][64] = {};   // per BwdMode

// Backward prepass of the materialized schedule: WdqT[k][n] =
// fp16_rn(fp32(CB[n][k]) * (SCB[n] * fp32(1/127))) -- the page's per-call
// dequantization of the int8 weight for the fp16 backward matmul --
// transposed so that the reduction index n is contiguous (a K-major GEMM
// operand).  One CTA per 64 (n) x 128 (k) tile: coalesced 16-byte loads of
// the int8 rows into shared memory, then each thread converts 8 consecutive
// n of one k and writes them with one 16-byte store.
constexpr int kDqN = 64, kDqK = 128, kDqPitch = kDqK + 4;   // shared rows padded by one word
__global__ void __launch_bounds__(256) dequant_weight_kernel(const int8_t* __restrict__ CB,
                                                             const float* __restrict__ SCB, int N, int k_pad,
                                                             __half* __restrict__ WdqT, int n_pad) {
  __shared__ __align__(16) uint8_t tile[kDqN * kDqPitch];
  __shared__ float f_s[kDqN];
  const int n0 = blockIdx.x * kDqN;
  const int k0 = blockIdx.y * kDqK;
  for (int c = threadIdx.x; c < kDqN * 8; c += 256) {
    const int nl = c >> 3, q = c & 7;
    const int n = n0 + nl, k = k0 + q * 16;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (n < N && k < k_pad) v = __ldg(reinterpret_cast<const uint4*>(CB + static_cast<int64_t>(n) * k_pad + k));
    uint32_t* dst = reinterpret_cast<uint32_t*>(tile + nl * kDqPitch + q * 16);
    dst[0] = v.x;
    dst[1] = v.y;
    dst[2] = v.z;
    dst[3] = v.w;
  }
  if (threadIdx.x < kDqN) {
    const int n = n0 + static_cast<int>(threadIdx.x);
    f_s[threadIdx.x] = n < N ? __fmul_rn(SCB[n], 1.0f / 127.0f) : 0.f;
  }
  __syncthreads();
  for (int c = threadIdx.x; c < kDqK * 8; c += 256) {
    const int g8 = c & 7, kl = c >> 3;
    const int k = k0 + kl, n = n0 + g8 * 8;
    if (k >= k_pad || n >= n_pad) continue;
    uint32_t h[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int a = g8 * 8 + 2 * i;
      const float x0 = __fmul_rn(static_cast<float>(static_cast<int8_t>(tile[a * kDqPitch + kl])), f_s[a]);
      const float x1 = __fmul_rn(static_cast<float>(static_cast<int8_t>(tile[(a + 1) * kDqPitch + kl])), f_s[a + 1]);
      const __half2 p = __halves2half2(__float2half_rn(x0), __float2half_rn(x1));
      h[i] = *reinterpret_cast<const uint32_t*>(&p);
    }
    *reinterpret_cast<uint4*>(WdqT + static_cast<int64_t>(k) * n_pad + n) = make_uint4(h[0], h[1], h[2], h[3]);
  }
}

// Number of CTA pairs that fit on the device at once (each CTA needs most
// of an SM's shared memory), so that a persistent grid never has a second
// wave of pairs.
int resident_pairs(const void* fn, int threads, int smem_bytes, int* cached /* [64] */) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  int sms = 152;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * (sms / 2)), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = sms / 2;
  }
  n = std::max(1, std::min(n, sms / 2));
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}


}  // namespace


cudaError_t gemm_launch_shape(int kernel_id, int* ctas, int* threads, int* smem_bytes) {
  // the backward reports the schedule the workspace-sized default picks: fused
  const void* fn = nullptr;
  int nthreads = 0, smem = 0;
  int* cache = nullptr;
  if (kernel_id == K_FWD_GEMM) {
    fn = reinterpret_cast<const void*>(fwd_gemm_kernel<false>);
    nthreads = kThreads;
    smem = kFwdSmemBytes;
    cache = g_pairs_fwd;
  } else if (kernel_id == K_BWD_GEMM) {
    fn = reinterpret_cast<const void*>(bwd_gemm_kernel<kModeI8>);
    nthreads = kBwdThreads;
    smem = BwdGeom<kModeI8>::kSmemBytes;
    cache = g_pairs_bwd[kModeI8];
  } else {
    return cudaErrorInvalidValue;
  }
  if (!ensure_smem_attr(fn, smem)) return cudaGetLastError();
  if (ctas != nullptr) *ctas = 2 * resident_pairs(fn, nthreads, smem, cache);
  if (threads != nullptr) *threads = nthreads;
  if (smem_bytes != nullptr) *smem_bytes = smem;
  return cudaSuccess;
}

cudaError_t launch_widen_codes(const int8_t* CB, __half* CBh, int64_t N, int64_t k_pad, uint32_t* bsq,
                               cudaStream_t s) {
  if (N == 0 || k_pad == 0) return cudaSuccess;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int nchunks = static_cast<int>(ceil_div(k_pad, 1024));
  const int blocks = static_cast<int>(std::min<int64_t>(ceil_div(N * nchunks, 8), static_cast<int64_t>(sms) * 8));
  ProfScope ps(K_WIDEN_CODES, s);
  widen_codes_kernel<<<blocks, 256, 0, s>>>(CB, CBh, N, k_pad, nchunks, bsq);
  return cudaGetLastError();
}

cudaError_t launch_unit_plan(const uint32_t* asq, const uint32_t* bsq, int num_m, int num_n, int nchunks,
                             uint32_t* plan, cudaStream_t s) {
  if (num_m == 0 || num_n == 0) return cudaSuccess;
  if (nchunks > kPlanMaxChunks) return cudaErrorInvalidValue;
  ProfScope ps(K_UNIT_PLAN, s);
  unit_plan_kernel<<<num_m, 256, 0, s>>>(asq, bsq, num_n, nchunks, plan);
  return cudaGetLastError();
}

template <bool kSilu>
cudaError_t launch_fwd_variant(const FwdGemmArgs& g, const FwdEpiArgs& e, cudaStream_t s, int prof_id) {
  const int num_m = static_cast<int>(ceil_div(e.M, kPairM));
  const int num_n = static_cast<int>(ceil_div(e.N, kPairN));
  if (num_m == 0 || num_n == 0) return cudaSuccess;
  const void* fn = reinterpret_cast<const void*>(fwd_gemm_kernel<kSilu>);
  if (!ensure_smem_attr(fn, kFwdSmemBytes)) return cudaGetLastError();
  const int tiles = num_m * num_n;
  const int clusters = std::min(tiles, resident_pairs(fn, kThreads, kFwdSmemBytes, kSilu ? g_pairs_fwd_silu : g_pairs_fwd));
  const int group = std::min(num_m, 8);
  ProfScope ps(prof_id, s);
  fwd_gemm_kernel<kSilu><<<2 * clusters, kThreads, kFwdSmemBytes, s>>>(g, e, num_m, num_n, group);
  return cudaGetLastError();
}

cudaError_t launch_fwd_gemm(const FwdGemmArgs& g, const FwdEpiArgs& e, cudaStream_t s, int prof_id) {
  static_assert(K_FWD_GEMM == 5, "default profile id of launch_fwd_gemm");
  return e.act != nullptr ? launch_fwd_variant<true>(g, e, s, prof_id) : launch_fwd_variant<false>(g, e, s, prof_id);
}

// Raster tiles of the 512-token schedules to run as two 256-token halves:
// the R = tiles % pairs tiles of an incomplete last round, when their 2 R
// halves fit in one round (then that round takes half as long); with fewer
// tiles than pairs, every tile when the halves fit.
int tail_split(int tiles, int pairs) {
  const int r = tiles >= pairs ? tiles % pairs : tiles;
  return (r > 0 && 2 * r <= pairs) ? r : 0;
}

template <int kMode>
cudaError_t launch_bwd_schedule(const BwdGemmArgs& g, const BwdEpiArgs& e, cudaStream_t s, int prof_id) {
  using Geo = BwdGeom<kMode>;
  const int num_k = static_cast<int>(ceil_div(e.K, kPairM));
  const int num_m = static_cast<int>(ceil_div(e.M, Geo::kTileTokens));
  if (num_k == 0 || num_m == 0) return cudaSuccess;
  const void* fn = reinterpret_cast<const void*>(bwd_gemm_kernel<kMode>);
  if (!ensure_smem_attr(fn, Geo::kSmemBytes)) return cudaGetLastError();
  const int tiles = num_k * num_m;
  const int pairs = resident_pairs(fn, kBwdThreads, Geo::kSmemBytes, g_pairs_bwd[kMode]);
  const int split = Geo::kSub == 2 ? tail_split(tiles, pairs) : 0;
  const int clusters = std::min(tiles + split, pairs);
  const int group = std::min(num_m, 8);
  ProfScope ps(prof_id, s);
  bwd_gemm_kernel<kMode><<<2 * clusters, kBwdThreads, Geo::kSmemBytes, s>>>(g, e, num_k, num_m, group, split);
  return cudaGetLastError();
}

cudaError_t launch_bwd_gemm(const BwdGemmArgs& g, const BwdEpiArgs& e, bool fused, cudaStream_t s) {
  return fused ? launch_bwd_schedule<kModeI8>(g, e, s, K_BWD_GEMM) : launch_bwd_schedule<kModeMat>(g, e, s, K_BWD_GEMM);
}

cudaError_t launch_nf4_gemm(const BwdGemmArgs& g, const BwdEpiArgs& e, bool input_grad, bool materialized,
                            cudaStream_t s) {
  const int prof = input_grad ? K_NF4_GEMM_BWD : K_NF4_GEMM_FWD;
  if (materialized) return launch_bwd_schedule<kModeMat>(g, e, s, prof);
  return input_grad ? launch_bwd_schedule<kModeNf4T>(g, e, s, prof) : launch_bwd_schedule<kModeNf4>(g, e, s, prof);
}

cudaError_t launch_dequant_weight(const int8_t* CB, const float* SCB, int64_t N, int64_t k_pad, __half* WdqT,
                                  int64_t n_pad, cudaStream_t s) {
  if (N == 0 || k_pad == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(ceil_div(n_pad, kDqN)), static_cast<unsigned>(ceil_div(k_pad, kDqK)));
  ProfScope ps(K_DEQUANT_WEIGHT, s);
  dequant_weight_kernel<<<grid, 256, 0, s>>>(CB, SCB, static_cast<int>(N), static_cast<int>(k_pad), WdqT,
                                             static_cast<int>(n_pad));
  return cudaGetLastError();
}

}  // namespace i8lt
