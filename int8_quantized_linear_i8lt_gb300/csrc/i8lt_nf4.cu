// 4-bit NormalFloat (NF4) weight storage for the weight-only matmuls of
// QLoRA fine-tuning ("Support QLoRA 4-bit finetuning with bitsandbytes",
// lit-gpt PR #275: the bnb.nf4 quantize option; frozen 4-bit base weights,
// bf16 compute).  The page names the format without defining it; this file
// follows the published construction of QLoRA's 4-bit NormalFloat:
//   levels: 7 negated and 8 positive standard-normal quantiles of evenly
//           spaced probabilities between 1/2 and delta = ((1 - 1/30) +
//           (1 - 1/32)) / 2, plus 0, divided by the largest (so -1 .. 1);
//   blocks: 64 consecutive elements of a weight row share one fp32 absmax;
//   code:   the nearest level to x / absmax, decided in fp32 against the
//           midpoints of adjacent levels (strictly greater: the upper level);
//   packing: two codes per byte, the even element in the high nibble, rows
//           padded to a multiple of 64 elements with the zero level.
// Beside NF4, the same storage holds FP4 (the bnb.fp4 quantize option of the
// same page, also named there without a definition): the 4-bit floating-point
// format with 1 sign, 2 exponent and 1 mantissa bits (E2M1: magnitudes 0,
// 0.5, 1, 1.5, 2, 3, 4, 6 for the codes 0..7 of the exponent-mantissa bits,
// the sign in bit 3), the block's absmax mapped to 6:
//   levels: lv[code] = +-E2M1(code) / 6 in fp32 (code 8 is -0);
//   code:   the magnitude code of the level nearest to |x / absmax|, decided
//           in fp32 against the midpoints of adjacent magnitude levels, a tie
//           going to the code whose mantissa bit is 0 (round half to even);
//           the sign bit set for x < 0 unless the magnitude code is 0 (one
//           zero code, 0, also for padding and all-zero blocks).
// The matmuls that decode these codes inside the tensor-core pipeline are in
// i8lt_gemm.cu (kModeNf4, kModeNf4T): they look every code up in the
// 16-entry level table, so both formats run through them unchanged.
#include <algorithm>
#include <cmath>
#include <mutex>

#include <type_traits>

#include "i8lt_internal.h"

namespace i8lt {

namespace {

double normal_cdf(double x) { return 0.5 * std::erfc(-x / std::sqrt(2.0)); }

// Standard-normal quantile: bisection on the CDF down to adjacent doubles.
double normal_quantile(double p) {
  double lo = -10.0, hi = 10.0;
  for (int i = 0; i < 200; ++i) {
    const double mid = 0.5 * (lo + hi);
    if (mid == lo || mid == hi) break;
    if (normal_cdf(mid) < p) {
      lo = mid;
    } else {
      hi = mid;
    }
  }
  return 0.5 * (lo + hi);
}

// Level table and decision thresholds of a 4-bit format.  NF4: lv ascending
// with the code, mid[0..14] between adjacent levels.  FP4: lv by code
// (sign-magnitude), mid[0..6] between adjacent magnitude levels lv[0..7],
// bit j of tie_up set when a value equal to mid[j] takes the upper level.
struct Nf4Tables {
  float lv[16];
  float mid[15];
  uint32_t tie_up;
};

const Nf4Tables& fp4_tables() {
  static Nf4Tables t;
  static std::once_flag once;
  std::call_once(once, [] {
    t = Nf4Tables{};
    // E2M1 magnitude of the exponent-mantissa bits c = (e1 e0 m): e = 0 is
    // subnormal (m / 2), otherwise 2^(e - 1) (1 + m / 2)
    double mag[8];
    for (int c = 0; c < 8; ++c) {
      const int e = c >> 1, m = c & 1;
      mag[c] = e == 0 ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, e - 1);
    }
    for (int c = 0; c < 8; ++c) {
      t.lv[c] = static_cast<float>(mag[c] / mag[7]);
      t.lv[8 + c] = -t.lv[c];
    }
    for (int j = 0; j < 7; ++j) {
      t.mid[j] = static_cast<float>((static_cast<double>(t.lv[j]) + static_cast<double>(t.lv[j + 1])) / 2.0);
      if (((j + 1) & 1) == 0) t.tie_up |= 1u << j;   // the upper code's mantissa bit is 0
    }
  });
  return t;
}

const Nf4Tables& tables() {
  static Nf4Tables t;
  static std::once_flag once;
  std::call_once(once, [] {
    t.tie_up = 0;
    const double delta = ((1.0 - 1.0 / 30.0) + (1.0 - 1.0 / 32.0)) / 2.0;
    const double step_neg = (0.5 - delta) / 7.0, step_pos = (0.5 - delta) / 8.0;
    double v[16];
    int n = 0;
    for (int i = 0; i < 7; ++i) v[n++] = -normal_quantile(static_cast<double>(i) * step_neg + delta);
    v[n++] = 0.0;
    for (int i = 0; i < 8; ++i) v[n++] = normal_quantile(static_cast<double>(i) * step_pos + delta);
    std::sort(v, v + 16);
    for (int i = 0; i < 16; ++i) t.lv[i] = static_cast<float>(v[i] / v[15]);
    for (int i = 0; i < 15; ++i)
      t.mid[i] = static_cast<float>((static_cast<double>(t.lv[i]) + static_cast<double>(t.lv[i + 1])) / 2.0);
  });
  return t;
}

template <typename T>
__device__ __forceinline__ float load_w(const T* p, int64_t i) {
  return to_float(p[i]);
}

// One thread per 8 consecutive elements of a row (one 32-bit word of packed
// codes); the 8 threads of a 64-element block reduce its absmax with three
// shuffles.  Every thread of a block runs every iteration (the shuffles take
// the whole warp).
template <typename T, bool kFp4>
__global__ void __launch_bounds__(256) nf4_quantize_kernel(const T* __restrict__ W, int64_t N, int64_t K,
                                                           int64_t row_bytes, int nblk, Nf4Tables c,
                                                           uint8_t* __restrict__ packed,
                                                           float* __restrict__ absmax) {
  constexpr uint32_t kZero = kFp4 ? 0u : 7u;   // the code of the zero level
  // NF4: the 15 level midpoints in shared memory for a binary search (each
  // lane indexes its own midpoints)
  __shared__ float mid_s[16];
  if (threadIdx.x < 15) mid_s[threadIdx.x] = c.mid[threadIdx.x];
  __syncthreads();
  const int64_t gpr = row_bytes / 4;   // groups of 8 per row (a multiple of 8)
  const int64_t total = N * gpr;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x; base < total; base += stride) {
    const int64_t g = base + threadIdx.x;
    const bool act = g < total;
    const int64_t n = act ? g / gpr : 0;
    const int64_t kg = act ? g - n * gpr : 0;
    const int64_t k0 = kg * 8;
    float x[8];
    float am = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      x[i] = (act && k0 + i < K) ? load_w(W, n * K + k0 + i) : 0.f;
      am = fmaxf(am, fabsf(x[i]));
    }
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 4));
    if (!act) continue;
    if ((kg & 7) == 0) absmax[n * nblk + (kg >> 3)] = am;
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t code = kZero;   // padding and all-zero blocks
      if (k0 + i < K && am > 0.f) {
        const float xn = __fdiv_rn(x[i], am);
        code = 0u;
        if constexpr (kFp4) {
          const float a = fabsf(xn);
#pragma unroll
          for (int j = 0; j < 7; ++j) code += (a > c.mid[j] || (a == c.mid[j] && ((c.tie_up >> j) & 1u))) ? 1u : 0u;
          if (xn < 0.f && code != 0u) code |= 8u;
        } else {
          // the number of midpoints below xn (they ascend), by halving: the
          // same count as comparing with all fifteen
          code = xn > mid_s[7] ? 8u : 0u;
          code += xn > mid_s[code + 3] ? 4u : 0u;
          code += xn > mid_s[code + 1] ? 2u : 0u;
          code += xn > mid_s[code] ? 1u : 0u;
        }
      }
      // byte i / 2 holds elements (2j, 2j + 1) as (high, low) nibbles
      word |= code << (8 * (i >> 1) + ((i & 1) ? 0 : 4));
    }
    *reinterpret_cast<uint32_t*>(packed + n * row_bytes + kg * 4) = word;
  }
}

// Two fp32 levels times the block's absmax (one packed IEEE multiply: the
// same rounding as two scalar ones), rounded to a 16-bit pair, e0 in the low
// half.
template <bool kBf16>
__device__ __forceinline__ uint32_t levels_times_absmax(float e0, float e1, float am) {
  uint32_t out;
  if (kBf16) {
    asm("{\n .reg .b64 x, a, p;\n .reg .b32 lo, hi;\n mov.b64 x, {%1, %2};\n mov.b64 a, {%3, %3};\n"
        " mul.rn.f32x2 p, x, a;\n mov.b64 {lo, hi}, p;\n cvt.rn.bf16x2.f32 %0, hi, lo;\n}"
        : "=r"(out)
        : "f"(e0), "f"(e1), "f"(am));
  } else {
    asm("{\n .reg .b64 x, a, p;\n .reg .b32 lo, hi;\n mov.b64 x, {%1, %2};\n mov.b64 a, {%3, %3};\n"
        " mul.rn.f32x2 p, x, a;\n mov.b64 {lo, hi}, p;\n cvt.rn.f16x2.f32 %0, hi, lo;\n}"
        : "=r"(out)
        : "f"(e0), "f"(e1), "f"(am));
  }
  return out;
}

template <typename OutT>
__global__ void __launch_bounds__(256) nf4_dequantize_kernel(const uint8_t* __restrict__ packed,
                                                             const float* __restrict__ absmax, int64_t N, int64_t K,
                                                             int64_t row_bytes, int nblk, Nf4Tables c,
                                                             bool vec, OutT* __restrict__ out) {
  // the levels in shared memory: indexed by each lane's own code (a
  // parameter-space table indexed per lane would serialize the warp)
  __shared__ float lv_s[16];
  if (threadIdx.x < 16) lv_s[threadIdx.x] = c.lv[threadIdx.x];
  __syncthreads();
  const int64_t gpr = row_bytes / 4;
  const int64_t total = N * gpr;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < total; g += stride) {
    const int64_t n = g / gpr;
    const int64_t kg = g - n * gpr;
    const int64_t k0 = kg * 8;
    if (k0 >= K) continue;
    const uint32_t word = *reinterpret_cast<const uint32_t*>(packed + n * row_bytes + kg * 4);
    const float am = absmax[n * nblk + (kg >> 3)];
    OutT o[8];
    if constexpr (sizeof(OutT) == 2) {   // byte j: element 2j in the high nibble, 2j + 1 in the low
      uint32_t* w = reinterpret_cast<uint32_t*>(o);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t byte = (word >> (8 * j)) & 0xFFu;
        w[j] = levels_times_absmax<std::is_same<OutT, __nv_bfloat16>::value>(lv_s[byte >> 4], lv_s[byte & 15u], am);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t code = (word >> (8 * (i >> 1) + ((i & 1) ? 0 : 4))) & 15u;
        o[i] = from_float<OutT>(__fmul_rn(lv_s[code], am));
      }
    }
    OutT* dst = out + n * K + k0;
    if (vec && k0 + 8 <= K) {   // 16 or 32 bytes at an aligned address
      if constexpr (sizeof(OutT) == 2) {
        *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(o);
      } else {
        reinterpret_cast<uint4*>(dst)[0] = reinterpret_cast<const uint4*>(o)[0];
        reinterpret_cast<uint4*>(dst)[1] = reinterpret_cast<const uint4*>(o)[1];
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (k0 + i < K) dst[i] = o[i];
    }
  }
}

// Transposed dequantization for the materialized input gradient: WdqT[k, n]
// = Wdq[n, k], [K, N] with N a multiple of 8.  One block per 64 (n) x 128 (k)
// tile: the packed bytes (64 a row) and the two absmax values of each row
// are staged in shared memory, then each thread writes 8 consecutive n of one
// k with one 16-byte store.
constexpr int kTn = 64, kTk = 128, kTPitch = kTk / 2 + 4;
template <typename OutT>
__global__ void __launch_bounds__(256) nf4_dequantize_t_kernel(const uint8_t* __restrict__ packed,
                                                               const float* __restrict__ absmax, int64_t N, int64_t K,
                                                               int64_t row_bytes, int nblk, Nf4Tables c,
                                                               OutT* __restrict__ WdqT) {
  __shared__ __align__(16) uint8_t tile[kTn * kTPitch];
  __shared__ float am_s[kTn][2];
  __shared__ float lv_s[16];
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kTn;
  const int64_t k0 = static_cast<int64_t>(blockIdx.y) * kTk;
  {
    const int nl = threadIdx.x >> 2, q = threadIdx.x & 3;   // 64 rows x 4 chunks of 16 bytes
    const int64_t n = n0 + nl, byte = k0 / 2 + q * 16;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (n < N && byte < row_bytes) v = *reinterpret_cast<const uint4*>(packed + n * row_bytes + byte);
    uint32_t* dst = reinterpret_cast<uint32_t*>(tile + nl * kTPitch + q * 16);
    dst[0] = v.x;
    dst[1] = v.y;
    dst[2] = v.z;
    dst[3] = v.w;
  }
  if (threadIdx.x < 2 * kTn) {
    const int nl = threadIdx.x >> 1, b = threadIdx.x & 1;
    const int64_t n = n0 + nl, kb = k0 / 64 + b;
    am_s[nl][b] = (n < N && kb < nblk) ? absmax[n * nblk + kb] : 0.f;
  }
  if (threadIdx.x < 16) lv_s[threadIdx.x] = c.lv[threadIdx.x];
  __syncthreads();
  for (int it = threadIdx.x; it < kTk * (kTn / 8); it += 256) {
    const int g8 = it & 7, kl = it >> 3;
    const int64_t k = k0 + kl, n = n0 + g8 * 8;
    if (k >= K || n >= N) continue;
    OutT o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int nl = g8 * 8 + i;
      const uint32_t byte = tile[nl * kTPitch + (kl >> 1)];
      const uint32_t code = (kl & 1) ? (byte & 15u) : (byte >> 4);
      o[i] = from_float<OutT>(__fmul_rn(lv_s[code], am_s[nl][kl >> 6]));
    }
    *reinterpret_cast<uint4*>(WdqT + k * N + n) = *reinterpret_cast<const uint4*>(o);
  }
}

int grid_for(int64_t threads) {
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(ceil_div(threads, 256), static_cast<int64_t>(sms) * 8)));
}

}  // namespace

void nf4_levels(float out[16]) { fmt4_levels(kFmtNf4, out); }

void fmt4_levels(int fmt, float out[16]) {
  const Nf4Tables& t = fmt == kFmtFp4 ? fp4_tables() : tables();
  for (int i = 0; i < 16; ++i) out[i] = t.lv[i];
}

namespace {
template <bool kFp4>
void quantize_launch(const void* W, int wt, int64_t N, int64_t K, int64_t row_bytes, int nblk, int blocks,
                     const Nf4Tables& c, uint8_t* packed, float* absmax, cudaStream_t s) {
  switch (wt) {
    case DT_F16:
      nf4_quantize_kernel<__half, kFp4><<<blocks, 256, 0, s>>>(static_cast<const __half*>(W), N, K, row_bytes, nblk,
                                                               c, packed, absmax);
      break;
    case DT_BF16:
      nf4_quantize_kernel<__nv_bfloat16, kFp4><<<blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(W), N, K,
                                                                      row_bytes, nblk, c, packed, absmax);
      break;
    default:
      nf4_quantize_kernel<float, kFp4><<<blocks, 256, 0, s>>>(static_cast<const float*>(W), N, K, row_bytes, nblk,
                                                              c, packed, absmax);
      break;
  }
}
}  // namespace

cudaError_t launch_nf4_quantize(const void* W, int wt, int64_t N, int64_t K, int64_t row_bytes, uint8_t* packed,
                                float* absmax, cudaStream_t s, int fmt) {
  if (N == 0 || K == 0) return cudaSuccess;
  const int nblk = static_cast<int>(ceil_div(K, 64));
  const int blocks = grid_for(N * (row_bytes / 4));
  ProfScope ps(K_NF4_QUANTIZE, s);
  if (fmt == kFmtFp4) {
    quantize_launch<true>(W, wt, N, K, row_bytes, nblk, blocks, fp4_tables(), packed, absmax, s);
  } else {
    quantize_launch<false>(W, wt, N, K, row_bytes, nblk, blocks, tables(), packed, absmax, s);
  }
  return cudaGetLastError();
}

cudaError_t launch_nf4_dequantize(const uint8_t* packed, const float* absmax, int64_t N, int64_t K,
                                  int64_t row_bytes, void* out, int dt, cudaStream_t s, int fmt) {
  if (N == 0 || K == 0) return cudaSuccess;
  const int nblk = static_cast<int>(ceil_div(K, 64));
  const int blocks = grid_for(N * (row_bytes / 4));
  const Nf4Tables& c = fmt == kFmtFp4 ? fp4_tables() : tables();
  // rows of K elements start 16-byte aligned when K is a multiple of 8 and
  // the output is 16-byte aligned
  const bool vec = (K % 8) == 0 && (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
  ProfScope ps(K_NF4_DEQUANTIZE, s);
  switch (dt) {
    case DT_F16:
      nf4_dequantize_kernel<__half><<<blocks, 256, 0, s>>>(packed, absmax, N, K, row_bytes, nblk, c, vec,
                                                           static_cast<__half*>(out));
      break;
    case DT_BF16:
      nf4_dequantize_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(packed, absmax, N, K, row_bytes, nblk, c, vec,
                                                                  static_cast<__nv_bfloat16*>(out));
      break;
    default:
      nf4_dequantize_kernel<float><<<blocks, 256, 0, s>>>(packed, absmax, N, K, row_bytes, nblk, c, vec,
                                                          static_cast<float*>(out));
      break;
  }
  return cudaGetLastError();
}

cudaError_t launch_nf4_dequantize_t(const uint8_t* packed, const float* absmax, int64_t N, int64_t K,
                                    int64_t row_bytes, void* WdqT, int dt, cudaStream_t s, int fmt) {
  if (N == 0 || K == 0) return cudaSuccess;
  const int nblk = static_cast<int>(ceil_div(K, 64));
  const dim3 grid(static_cast<unsigned>(ceil_div(N, kTn)), static_cast<unsigned>(ceil_div(K, kTk)));
  const Nf4Tables& c = fmt == kFmtFp4 ? fp4_tables() : tables();
  ProfScope ps(K_NF4_DEQUANTIZE, s);
  if (dt == DT_BF16) {
    nf4_dequantize_t_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(packed, absmax, N, K, row_bytes, nblk, c,
                                                                 static_cast<__nv_bfloat16*>(WdqT));
  } else {
    nf4_dequantize_t_kernel<__half><<<grid, 256, 0, s>>>(packed, absmax, N, K, row_bytes, nblk, c,
                                                          static_cast<__half*>(WdqT));
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Double-quantized absmax (the "-dq" options of the 4-bit formats, lit-gpt PR
// #275 "Support QLoRA 4-bit finetuning with bitsandbytes"; QLoRA's double
// quantization): the fp32 absmax values c of the 64-element blocks are stored
// as FP8 E4M3 codes of d = c - offset in blocks of 256 with an fp32 scale
// each; offset is the mean of all c.
// ---------------------------------------------------------------------------
namespace {

constexpr int kAbs8Block = 256;
constexpr float kInv448 = 0x1.24924ap-9f;   // fp32(1 / 448), correctly rounded

// E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, exponent 0
// subnormal, largest finite 448) from its bit fields.  Codes 0x7F / 0xFF (NaN)
// are never produced by absmax8_encode.
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  const uint32_t e = (code >> 3) & 15u, m = code & 7u;
  const float mag = e == 0u ? static_cast<float>(m) * 0x1p-9f : __uint_as_float(((e + 120u) << 23) | (m << 20));
  return (code & 0x80u) ? -mag : mag;
}

// The E4M3 code nearest to y, ties to the even code (round half to even on
// the 3-bit mantissa), |y| >= 448 saturating to 448, the sign of y kept.
__device__ __forceinline__ uint32_t absmax8_encode(float y) {
  const uint32_t sign = (__float_as_uint(y) >> 24) & 0x80u;
  const float a = fabsf(y);
  if (!(a < 448.f)) return sign | 0x7Eu;
  if (a < 0x1p-6f) return sign | static_cast<uint32_t>(__float2int_rn(a * 512.f));   // subnormal: steps of 2^-9
  const int e = static_cast<int>(__float_as_uint(a) >> 23) - 127;                     // -6 .. 8
  // a * 2^(3 - e) in [8, 16): the mantissa with its leading bit, rounded;
  // 16 carries into the next exponent through the addition below
  const float scaled = a * __uint_as_float(static_cast<uint32_t>(127 + 3 - e) << 23);
  const int m = __float2int_rn(scaled);
  return sign | static_cast<uint32_t>(((e + 7) << 3) + (m - 8));
}

// Per-exponent integer sums of the significands (exact): bucket[e] gathers
// the 24-bit significands of the values with biased exponent e (subnormals
// in bucket 1), so sum(c) = sum_e bucket[e] * 2^(e - 150).  Lanes with the
// same exponent are combined first, then one shared atomic per group.
__global__ void __launch_bounds__(256) absmax8_sum_kernel(const float* __restrict__ c, int64_t n,
                                                           unsigned long long* __restrict__ buckets) {
  __shared__ unsigned long long b_s[256];
  for (int i = threadIdx.x; i < 256; i += blockDim.x) b_s[i] = 0ull;
  __syncthreads();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  // every lane of a warp runs the same number of rounds (the shuffles below)
  const int64_t rounds = (n + stride - 1) / stride;
  for (int64_t rd = 0; rd < rounds; ++rd) {
    const int64_t i = i0 + rd * stride;
    uint32_t e = 0u, m = 0u;
    if (i < n) {
      const uint32_t bits = __float_as_uint(c[i]) & 0x7FFFFFFFu;   // the values are non-negative
      const uint32_t be = bits >> 23;
      if (be != 255u && bits != 0u) {
        e = be == 0u ? 1u : be;
        m = (bits & 0x7FFFFFu) | (be == 0u ? 0u : 0x800000u);
      }
    }
    const unsigned grp = __match_any_sync(0xffffffffu, e);
    const unsigned sum = __reduce_add_sync(grp, m);   // <= 32 * 2^24
    if (m != 0u || e != 0u) {
      if ((threadIdx.x & 31) == static_cast<unsigned>(__ffs(grp) - 1) && sum != 0u)
        atomicAdd(&b_s[e], static_cast<unsigned long long>(sum));
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 256; i += blockDim.x)
    if (b_s[i] != 0ull) atomicAdd(&buckets[i], b_s[i]);
}

__device__ __forceinline__ double pow2d(int k) {   // 2^k for -1022 <= k <= 1023
  return __longlong_as_double(static_cast<long long>(1023 + k) << 52);
}

// offset = fp32(S / n): the exact sum S of the buckets as a 384-bit integer
// times 2^-149, rounded once to float64 (half to even), an IEEE float64
// division by n, one rounding to fp32.  One thread.
__global__ void absmax8_offset_kernel(const unsigned long long* __restrict__ buckets, int64_t n,
                                      float* __restrict__ offset) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  uint64_t w[6] = {0, 0, 0, 0, 0, 0};   // little-endian words of sum_e bucket[e] * 2^(e - 1)
  for (int e = 1; e < 255; ++e) {
    const uint64_t v = buckets[e];
    if (v == 0) continue;
    const int sh = e - 1, q = sh >> 6, r = sh & 63;
    const uint64_t lo = v << r, hi = r ? (v >> (64 - r)) : 0ull;
    uint64_t s0 = w[q] + lo;
    uint64_t carry = s0 < lo ? 1ull : 0ull;
    w[q] = s0;
    uint64_t s1 = w[q + 1] + hi;
    uint64_t c1 = s1 < hi ? 1ull : 0ull;
    s1 += carry;
    c1 += s1 < carry ? 1ull : 0ull;
    w[q + 1] = s1;
    for (int j = q + 2; j < 6 && c1 != 0ull; ++j) {
      w[j] += c1;
      c1 = w[j] == 0ull ? 1ull : 0ull;
    }
  }
  int top = -1;
  for (int j = 5; j >= 0 && top < 0; --j)
    if (w[j] != 0ull) top = 64 * j + 63 - __clzll(static_cast<long long>(w[j]));
  auto bit = [&](int b) -> uint64_t { return (w[b >> 6] >> (b & 63)) & 1ull; };
  double s64 = 0.0;
  if (top >= 0 && top < 53) {
    s64 = static_cast<double>(w[0]) * pow2d(-149);   // exact: fewer than 54 bits
  } else if (top >= 53) {
    uint64_t mant = 0;
    for (int b = top; b > top - 53; --b) mant = (mant << 1) | bit(b);
    const uint64_t rnd = bit(top - 53);
    bool sticky = false;
    for (int b = top - 54; b >= 0 && !sticky; --b) sticky = bit(b) != 0ull;
    int p = top;
    if (rnd && (sticky || (mant & 1ull))) {
      ++mant;
      if (mant == (1ull << 53)) {
        mant >>= 1;
        ++p;
      }
    }
    s64 = static_cast<double>(mant) * pow2d(p - 52 - 149);   // exact: 53 bits times a power of two
  }
  *offset = n > 0 ? __double2float_rn(__ddiv_rn(s64, static_cast<double>(n))) : 0.f;
}

// One warp per block of 256 values: d = c - offset, absmax2 = max |d|, codes
// of d * fp32(448 / absmax2).
__global__ void __launch_bounds__(256) absmax8_quant_kernel(const float* __restrict__ c, int64_t n,
                                                             const float* __restrict__ offset,
                                                             uint8_t* __restrict__ q, float* __restrict__ absmax2) {
  const int lane = threadIdx.x & 31;
  const int64_t blk = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (blk >= (n + kAbs8Block - 1) / kAbs8Block) return;   // uniform over the warp
  const float off = *offset;
  float d[8];
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int64_t i = blk * kAbs8Block + j * 32 + lane;
    d[j] = i < n ? __fsub_rn(c[i], off) : 0.f;
    m = fmaxf(m, fabsf(d[j]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float s2 = m > 0.f ? __fdiv_rn(448.f, m) : 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int64_t i = blk * kAbs8Block + j * 32 + lane;
    if (i < n) q[i] = static_cast<uint8_t>(absmax8_encode(__fmul_rn(d[j], s2)));
  }
  if (lane == 0) absmax2[blk] = m;
}

__global__ void __launch_bounds__(256) absmax8_dequant_kernel(const uint8_t* __restrict__ q,
                                                               const float* __restrict__ absmax2,
                                                               const float* __restrict__ offset, int64_t n,
                                                               float* __restrict__ out) {
  const float off = *offset;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float f2 = __fmul_rn(absmax2[i / kAbs8Block], kInv448);
    out[i] = __fadd_rn(__fmul_rn(e4m3_value(q[i]), f2), off);
  }
}

}  // namespace

cudaError_t launch_absmax8_quantize(const float* absmax, int64_t n, uint8_t* q, float* absmax2, float* offset,
                                    unsigned long long* buckets, cudaStream_t s) {
  ProfScope ps(K_ABSMAX8, s);
  if (n == 0) return cudaMemsetAsync(offset, 0, sizeof(float), s);
  cudaError_t err = cudaMemsetAsync(buckets, 0, 256 * sizeof(unsigned long long), s);
  if (err != cudaSuccess) return err;
  absmax8_sum_kernel<<<grid_for(n), 256, 0, s>>>(absmax, n, buckets);
  absmax8_offset_kernel<<<1, 32, 0, s>>>(buckets, n, offset);
  const int64_t warps = (n + kAbs8Block - 1) / kAbs8Block;
  absmax8_quant_kernel<<<static_cast<unsigned>(ceil_div(warps, 8)), 256, 0, s>>>(absmax, n, offset, q, absmax2);
  return cudaGetLastError();
}

cudaError_t launch_absmax8_dequantize(const uint8_t* q, const float* absmax2, const float* offset, int64_t n,
                                      float* out, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  ProfScope ps(K_ABSMAX8, s);
  absmax8_dequant_kernel<<<grid_for(n), 256, 0, s>>>(q, absmax2, offset, n, out);
  return cudaGetLastError();
}

}  // namespace i8lt
