// Memory-bound kernels of the int8 quantized linear layer (sm_103a):
//   K1 weight quantization, K2 outlier-column detection, the outlier index
//   build, K3 row-wise (vector-wise) activation quantization, K4 the fp16
//   outlier weight columns, K7 the grad_output prepass (grad_bias + fp16 cast)
//   and the SiLU between MLP layers.
//
// Method: bitsandbytes PR #33 "Memory efficient backward" (PR description and
// the review threads on bitsandbytes/autograd/_functions.py).  All loads and
// stores move 16 bytes per thread when rows are 16-byte aligned.
#include <algorithm>
#include <type_traits>

#include <mutex>

#include "i8lt_internal.h"

namespace i8lt {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = v;
  __syncthreads();
  float r = (threadIdx.x < (blockDim.x >> 5)) ? red[threadIdx.x] : 0.f;
  if (w == 0) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) r = fmaxf(r, __shfl_xor_sync(0xffffffffu, r, o));
    if (l == 0) red[0] = r;
  }
  __syncthreads();
  r = red[0];
  __syncthreads();
  return r;
}

// q = round_half_even(x * s) in IEEE fp32 (s = 127 / absmax), |q| <= 127.
__device__ __forceinline__ int quant_code(float x, float s) {
  int q = __float2int_rn(__fmul_rn(x, s));
  return max(-127, min(127, q));
}

// ---------------------------------------------------------------------------
// K1 (weights) and K3 (activations): row-wise absmax quantization.
// One block per row (grid-stride).  Pass 1: absmax of the fp16-cast row
// outside the outlier columns.  Pass 2: codes, zero for outlier columns and
// for the padding up to ld.  Activations also gather their outlier columns.
// ---------------------------------------------------------------------------
template <typename T, typename OutT>
__global__ void __launch_bounds__(kThreads) row_quantize_kernel(
    const T* __restrict__ A, int64_t M, int64_t K, int64_t ld, int vec, const uint32_t* __restrict__ mask,
    const int* __restrict__ idx, const DevStatus* __restrict__ st, int64_t cap_pad, float* __restrict__ scale,
    OutT* __restrict__ codes, __half* __restrict__ sub, uint32_t* __restrict__ asq) {
  __shared__ float red[32];
  __shared__ int chunk_sq[2];   // sum of code^2 of the two 1024-column chunks of one pass-2 step
  const int nchunks = static_cast<int>((ld + 1023) / 1024);
  const int used = (mask != nullptr) ? st->used : 0;
  const int used_pad = (used + 63) / 64 * 64;
  for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
    const T* row = A + m * K;
    float amax = 0.f;
    for (int64_t c = static_cast<int64_t>(threadIdx.x) * 8; c < K; c += kThreads * 8) {
      __half h[8];
      load8_half(row + c, K - c, vec != 0 && c + 8 <= K, h);
      const uint32_t bits = (mask != nullptr) ? ((mask[c >> 5] >> (c & 31)) & 0xFFu) : 0u;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (!((bits >> i) & 1u)) amax = fmaxf(amax, fabsf(__half2float(h[i])));
    }
    amax = block_max(amax, red);
    const float s = (amax > 0.f) ? __fdiv_rn(127.0f, amax) : 0.f;
    OutT* out = codes + m * ld;
    for (int64_t c0 = 0; c0 < ld; c0 += kThreads * 8) {
      const int64_t c = c0 + static_cast<int64_t>(threadIdx.x) * 8;
      if (asq != nullptr && threadIdx.x < 2) chunk_sq[threadIdx.x] = 0;
      if (asq != nullptr) __syncthreads();
      int sq = 0;
      if (c < ld) {
      __half h[8];
      if (c < K) {
        load8_half(row + c, K - c, vec != 0 && c + 8 <= K, h);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) h[i] = __float2half_rn(0.f);
      }
      const uint32_t bits = (mask != nullptr && c < K) ? ((mask[c >> 5] >> (c & 31)) & 0xFFu) : 0u;
      int q[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        q[i] = (amax > 0.f && !((bits >> i) & 1u)) ? quant_code(__half2float(h[i]), s) : 0;
        sq += q[i] * q[i];
      }
      if constexpr (sizeof(OutT) == 1) {
        uint2 u;
        u.x = (q[0] & 0xFF) | ((q[1] & 0xFF) << 8) | ((q[2] & 0xFF) << 16) | ((q[3] & 0xFF) << 24);
        u.y = (q[4] & 0xFF) | ((q[5] & 0xFF) << 8) | ((q[6] & 0xFF) << 16) | ((q[7] & 0xFF) << 24);
        *reinterpret_cast<uint2*>(out + c) = u;   // ld % 16 == 0, c % 8 == 0
      } else {
        uint4 u;
        __half* o = reinterpret_cast<__half*>(&u);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = __int2half_rn(q[i]);   // exact: |q| <= 127
        *reinterpret_cast<uint4*>(out + c) = u;
      }
      }
      if (asq != nullptr) {
        // threads 0-127 cover columns c0 .. c0+1023, threads 128-255 the next 1024
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
        if ((threadIdx.x & 31) == 0 && sq != 0) atomicAdd(&chunk_sq[threadIdx.x >> 7], sq);
        __syncthreads();
        const int64_t ck = (c0 >> 10) + threadIdx.x;
        if (threadIdx.x < 2 && ck < nchunks && chunk_sq[threadIdx.x] != 0)
          atomicMax(asq + (m >> 8) * nchunks + ck, static_cast<uint32_t>(chunk_sq[threadIdx.x]));
        __syncthreads();
      }
    }
    if (sub != nullptr) {
      for (int j = threadIdx.x; j < used_pad; j += kThreads)
        sub[m * cap_pad + j] = (j < used) ? to_half(row[idx[j]]) : __float2half_rn(0.f);
    }
    if (threadIdx.x == 0) scale[m] = amax;
  }
}

// ---------------------------------------------------------------------------
// K3 for rows that fit in shared memory (K_pad <= kStagedMaxLd): the same
// quantization as row_quantize_kernel<T, __half>, with the fp16-cast row
// staged in shared memory so that A is read from HBM once.  The codes are
// rounded with an IEEE fp32 add of 1.5 * 2^23 (round to nearest even, exact
// for |x * s| < 2^22; here |x * s| <= 127 + 2^-16), the same rounding as
// __float2int_rn, and stored two at a time with one fp32x2 -> fp16x2
// conversion (exact: integers of magnitude <= 127).  With `asq`, each row's
// sums of squared codes per 1024-column chunk raise its 256-row tile's entries
// (asq[(m / 256) * nchunks + chunk], the activation side of the GEMM's exact
// accumulation plan).
// ---------------------------------------------------------------------------
constexpr int kStagedMaxLd = 49152;   // 96 KB of fp16 per row
constexpr int kStagedMaxChunks = kStagedMaxLd / 1024;

__device__ __forceinline__ float rint_small(float y) {
  return __fsub_rn(__fadd_rn(y, 12582912.0f), 12582912.0f);
}

// OutT = __half: activation codes (K3); OutT = int8_t: weight codes (K1, with
// no outlier mask, no subA and no asq).
template <typename T, typename OutT>
__global__ void __launch_bounds__(kThreads) act_quantize_staged_kernel(
    const T* __restrict__ A, int64_t M, int64_t K, int64_t ld, int vec, const uint32_t* __restrict__ mask,
    const int* __restrict__ idx, const DevStatus* __restrict__ st, int64_t cap_pad, float* __restrict__ scale,
    OutT* __restrict__ codes, __half* __restrict__ sub, uint32_t* __restrict__ asq) {
  extern __shared__ uint4 srow4[];   // ld fp16 values of the current row
  __shared__ float red[32];
  __shared__ int chunk_sq[kStagedMaxChunks];
  const __half* srow = reinterpret_cast<const __half*>(srow4);
  const int used = (mask != nullptr) ? st->used : 0;
  const int used_pad = (used + 63) / 64 * 64;
  const int nchunks = static_cast<int>((ld + 1023) / 1024);
  for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
    const T* row = A + m * K;
    float amax = 0.f;
    for (int64_t c = static_cast<int64_t>(threadIdx.x) * 8; c < ld; c += kThreads * 8) {
      __half h[8];
      if (c < K) {
        load8_half(row + c, K - c, vec != 0 && c + 8 <= K, h);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) h[i] = __float2half_rn(0.f);
      }
      srow4[c >> 3] = *reinterpret_cast<const uint4*>(h);
      const uint32_t bits = (mask != nullptr && c < K) ? ((mask[c >> 5] >> (c & 31)) & 0xFFu) : 0u;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (!((bits >> i) & 1u)) amax = fmaxf(amax, fabsf(__half2float(h[i])));
    }
    if (asq != nullptr)
      for (int i = threadIdx.x; i < nchunks; i += kThreads) chunk_sq[i] = 0;
    amax = block_max(amax, red);   // its barriers also publish the staged row and the cleared sums
    const float s = (amax > 0.f) ? __fdiv_rn(127.0f, amax) : 0.f;
    OutT* out = codes + m * ld;
    // every thread runs every iteration (the shuffles below need all 32 lanes)
    for (int64_t c0 = 0; c0 < ld; c0 += kThreads * 8) {
      const int64_t c = c0 + static_cast<int64_t>(threadIdx.x) * 8;
      float sq = 0.f;
      if (c < ld) {
        const uint4 u = srow4[c >> 3];
        const __half* h = reinterpret_cast<const __half*>(&u);
        const uint32_t bits = (mask != nullptr && c < K) ? ((mask[c >> 5] >> (c & 31)) & 0xFFu) : 0u;
        float q[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float r = rint_small(__fmul_rn(__half2float(h[i]), s));
          q[i] = ((bits >> i) & 1u) ? 0.f : fminf(127.f, fmaxf(-127.f, r));
          sq += q[i] * q[i];
        }
        if constexpr (sizeof(OutT) == 1) {
          uint32_t b[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) b[i] = static_cast<uint32_t>(static_cast<int>(q[i])) & 0xFFu;
          *reinterpret_cast<uint2*>(out + c) = make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24),
                                                          b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
        } else {
          uint4 o;
          __half2* o2 = reinterpret_cast<__half2*>(&o);
#pragma unroll
          for (int i = 0; i < 4; ++i) o2[i] = __floats2half2_rn(q[2 * i], q[2 * i + 1]);
          *reinterpret_cast<uint4*>(out + c) = o;
        }
      }
      if (asq != nullptr) {
        // a warp's 256 columns lie in one 1024-column chunk; a warp past the
        // end of the row sums to 0 and adds nothing
        int v = static_cast<int>(sq);
#pragma unroll
        for (int k = 16; k > 0; k >>= 1) v += __shfl_xor_sync(0xffffffffu, v, k);
        const int64_t cw = c0 + static_cast<int64_t>(threadIdx.x & ~31) * 8;
        if ((threadIdx.x & 31) == 0 && v != 0) atomicAdd(&chunk_sq[cw >> 10], v);
      }
    }
    if (sub != nullptr) {
      for (int j = threadIdx.x; j < used_pad; j += kThreads)
        sub[m * cap_pad + j] = (j < used) ? srow[idx[j]] : __float2half_rn(0.f);
    }
    if (asq != nullptr) {
      __syncthreads();
      for (int i = threadIdx.x; i < nchunks; i += kThreads)
        if (chunk_sq[i] != 0) atomicMax(asq + (m >> 8) * nchunks + i, static_cast<uint32_t>(chunk_sq[i]));
    }
    __syncthreads();   // also: the staged row is no longer read
    if (threadIdx.x == 0) scale[m] = amax;
  }
}

// ---------------------------------------------------------------------------
// K2: per-column max of |fp16(A)|.  Block = 32 column groups of 8 x 8 row
// lanes; each block covers 256 columns x kColRows rows, then one atomicMax
// per column.  fp16 magnitudes compare as unsigned integers.
// ---------------------------------------------------------------------------
constexpr int kColRows = 256;

template <typename T>
__global__ void __launch_bounds__(kThreads) colmax_kernel(const T* __restrict__ A, int64_t M, int64_t K, int vec,
                                                          uint32_t* __restrict__ colmax) {
  __shared__ uint16_t red[8][256 + 8];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int64_t c0 = (static_cast<int64_t>(blockIdx.x) * 32 + tx) * 8;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kColRows;
  const int64_t r1 = min(M, r0 + kColRows);
  uint32_t mx[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) mx[i] = 0;
  if (c0 < K) {
    for (int64_t r = r0 + ty; r < r1; r += 8) {
      __half h[8];
      load8_half(A + r * K + c0, K - c0, vec != 0 && c0 + 8 <= K, h);
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = max(mx[i], static_cast<uint32_t>(__half_as_ushort(h[i]) & 0x7FFFu));
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) red[ty][tx * 8 + i] = static_cast<uint16_t>(mx[i]);
  __syncthreads();
  // 256 threads reduce 256 columns over the 8 row lanes
  const int col = threadIdx.x;
  uint32_t v = 0;
#pragma unroll
  for (int y = 0; y < 8; ++y) v = max(v, static_cast<uint32_t>(red[y][col]));
  const int64_t k = static_cast<int64_t>(blockIdx.x) * 256 + col;
  if (k < K && v != 0) atomicMax(colmax + k, v);
}

// ---------------------------------------------------------------------------
// Outlier index build (one block of 1024 threads): mask bit k set when
// fp16(colmax[k]) > thr; ascending idx[] by a block-wide exclusive scan.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) outlier_index_kernel(const uint32_t* __restrict__ colmax, int64_t K,
                                                             float thr, int64_t cap, int* __restrict__ idx,
                                                             uint32_t* __restrict__ mask, DevStatus* st) {
  __shared__ int wsum[32];
  const int t = threadIdx.x;
  const int64_t nwords = (K + 31) / 32;
  const int64_t wpt = (nwords + 1023) / 1024;
  const int64_t w0 = t * wpt, w1 = min(nwords, w0 + wpt);
  int count = 0;
  for (int64_t w = w0; w < w1; ++w) {
    uint32_t bits = 0;
    for (int b = 0; b < 32; ++b) {
      const int64_t k = w * 32 + b;
      if (k < K && __half2float(__ushort_as_half(static_cast<unsigned short>(colmax[k]))) > thr) bits |= 1u << b;
    }
    mask[w] = bits;
    count += __popc(bits);
  }
  // exclusive scan of count over the block
  int incl = count;
  const int lane = t & 31, w = t >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[w] = incl;
  __syncthreads();
  if (w == 0) {
    int v = wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    wsum[lane] = v;   // inclusive over warps
  }
  __syncthreads();
  const int offset = incl - count + (w > 0 ? wsum[w - 1] : 0);
  int j = offset;
  for (int64_t ww = w0; ww < w1; ++ww) {
    uint32_t bits = mask[ww];
    while (bits) {
      const int b = __ffs(bits) - 1;
      bits &= bits - 1;
      if (j < cap) idx[j] = static_cast<int>(ww * 32 + b);
      ++j;
    }
  }
  if (t == 1023) {
    const int total = wsum[31];
    st->found = total;
    st->used = static_cast<int>(min(static_cast<int64_t>(total), cap));
    if (total > cap) set_status(st, ST_OUTLIER_CAPACITY, 0);
  }
}

// ---------------------------------------------------------------------------
// K4: subB[n, j] = fp16_rn(fp32(CB[n, idx[j]]) * (SCB[n] * fp32(1/127))),
// zero for used <= j < used_pad.  One warp per row.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) build_subB_kernel(const int8_t* __restrict__ CB, int64_t ld,
                                                              const float* __restrict__ SCB, int64_t N,
                                                              const int* __restrict__ idx,
                                                              const DevStatus* __restrict__ st, int64_t cap_pad,
                                                              __half* __restrict__ subB) {
  const int used = st->used;
  const int used_pad = (used + 63) / 64 * 64;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
  const int lane = threadIdx.x & 31;
  for (int64_t n = warp; n < N; n += nwarps) {
    const float f = __fmul_rn(SCB[n], 1.0f / 127.0f);
    for (int j = lane; j < used_pad; j += 32)
      subB[n * cap_pad + j] =
          (j < used) ? __float2half_rn(__fmul_rn(static_cast<float>(CB[n * ld + idx[j]]), f)) : __float2half_rn(0.f);
  }
}

// ---------------------------------------------------------------------------
// K7: grad_output prepass.  Column sums of the uncast G in fp32 per chunk of
// kBiasChunkRows = 128 rows, optional G16 = fp16_rn(G) padded to N_pad
// columns.  Within a chunk the order is fixed: eight row lanes y = 0..7 each
// sum the rows y, y + 8, ..., y + 120 in increasing order, then the eight
// lane sums are added in the order y = 0..7 -- the same order as the
// backward GEMM's own grad_bias reduction (bias_chunk_sums in
// i8lt_gemm.cu), so that every path gives the same bits.  A finalize
// kernel then sums the chunks in order.
// ---------------------------------------------------------------------------
constexpr int kSumRows = kBiasChunkRows;

template <typename T>
__global__ void __launch_bounds__(kThreads) gradout_prepass_kernel(const T* __restrict__ G, int64_t M, int64_t N,
                                                                   int vec, __half* __restrict__ G16,
                                                                   int64_t N_pad, float* __restrict__ partial) {
  __shared__ float red[8][256 + 4];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int64_t c0 = (static_cast<int64_t>(blockIdx.x) * 32 + tx) * 8;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kSumRows;
  const int64_t r1 = min(M, r0 + kSumRows);
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  const int64_t width = (G16 != nullptr) ? N_pad : N;
  if (c0 < width) {
    for (int64_t r = r0 + ty; r < r1; r += 8) {
      float f[8];
      if (c0 < N) {
        load8_float(G + r * N + c0, N - c0, vec != 0 && c0 + 8 <= N, f);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += f[i];
      if (G16 != nullptr) {
        uint4 u;
        __half* o = reinterpret_cast<__half*>(&u);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = __float2half_rn(f[i]);
        *reinterpret_cast<uint4*>(G16 + r * N_pad + c0) = u;   // N_pad % 8 == 0
      }
    }
  }
  if (partial == nullptr) return;
#pragma unroll
  for (int i = 0; i < 8; ++i) red[ty][tx * 8 + i] = acc[i];
  __syncthreads();
  const int col = threadIdx.x;
  float s = 0.f;
#pragma unroll
  for (int y = 0; y < 8; ++y) s += red[y][col];
  const int64_t n = static_cast<int64_t>(blockIdx.x) * 256 + col;
  if (n < N) partial[static_cast<int64_t>(blockIdx.y) * N + n] = s;
}

template <typename BT>
__global__ void __launch_bounds__(kThreads) grad_bias_finalize_kernel(const float* __restrict__ partial,
                                                                      int64_t chunks, int64_t N,
                                                                      BT* __restrict__ grad_bias) {
  for (int64_t n = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; n < N;
       n += static_cast<int64_t>(gridDim.x) * kThreads) {
    float s = 0.f;
    for (int64_t c = 0; c < chunks; ++c) s += partial[c * N + n];
    grad_bias[n] = from_float<BT>(s);
  }
}

// ---------------------------------------------------------------------------
// SiLU between MLP layers: y = h * sigmoid(h); dh = g * s * (1 + h (1 - s)).
// ---------------------------------------------------------------------------

template <typename T>
__global__ void __launch_bounds__(kThreads) silu_kernel(const T* __restrict__ h, int64_t n, int vec,
                                                        T* __restrict__ out) {
  for (int64_t c = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) * 8; c < n;
       c += static_cast<int64_t>(gridDim.x) * kThreads * 8) {
    float x[8], y[8];
    const bool v = vec != 0 && c + 8 <= n;
    load8_float(h + c, n - c, v, x);
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = silu_f(x[i]);
    store8(out + c, n - c, v, y);
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) silu_backward_kernel(const T* __restrict__ g, const T* __restrict__ h,
                                                                 int64_t n, int vec, T* __restrict__ out) {
  for (int64_t c = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) * 8; c < n;
       c += static_cast<int64_t>(gridDim.x) * kThreads * 8) {
    float x[8], gg[8], y[8];
    const bool v = vec != 0 && c + 8 <= n;
    load8_float(h + c, n - c, v, x);
    load8_float(g + c, n - c, v, gg);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float s = sigmoid_f(x[i]);
      y[i] = gg[i] * (s * (1.0f + x[i] * (1.0f - s)));
    }
    store8(out + c, n - c, v, y);
  }
}

// ---------------------------------------------------------------------------
// Trainable-weight mode: column-wise (vector-wise along the tokens) absmax
// quantization of a token-major X [R, C], written transposed, Xt [C, R_pad]
// as exact fp16 codes (the K-major operand rows of the weight-gradient GEMM):
// scale[c] = max_r |fp16(X[r, c])| (the colmax kernel's bits), Xt[c, r] =
// rint(fp32(fp16(X[r, c])) * (127 / scale[c])), 0 for R <= r < R_pad.  One
// block per 64 (r) x 64 (c) tile: coalesced 16-byte loads of 8 columns, the
// codes transposed through shared memory, 16-byte stores of 8 tokens.  With
// `sq` it also adds the sum of squared codes of each column over the tile's
// rows to sq[c, r / 1024] (the GEMM's accumulation plan).
// ---------------------------------------------------------------------------
constexpr int kCqTile = 64;
constexpr int kCqPitch = kCqTile + 2;   // halves; a 132-byte row keeps the transposed writes at 2-way

template <typename T>
__global__ void __launch_bounds__(kThreads) col_quantize_kernel(const T* __restrict__ X, int64_t R, int64_t C, int vec,
                                                                const uint32_t* __restrict__ colmax, int64_t R_pad,
                                                                float* __restrict__ scale, __half* __restrict__ Xt,
                                                                int* __restrict__ sq, int64_t nchunks) {
  __shared__ __align__(16) __half tile[kCqTile * kCqPitch];   // [c][r]
  __shared__ float s_s[kCqTile];
  __shared__ int sq_s[kCqTile];
  const int t = threadIdx.x, lane = t & 31;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kCqTile;
  const int64_t c0 = static_cast<int64_t>(blockIdx.y) * kCqTile;
  if (t < kCqTile) {
    const int64_t c = c0 + t;
    const float am = c < C ? __half2float(__ushort_as_half(static_cast<unsigned short>(colmax[c]))) : 0.f;
    s_s[t] = am > 0.f ? __fdiv_rn(127.0f, am) : 0.f;
    sq_s[t] = 0;
    if (blockIdx.x == 0 && c < C) scale[c] = am;
  }
  __syncthreads();
  const int cg = (t & 7) * 8;              // 8 consecutive columns
  int sqc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int rl = (t >> 3) + 32 * i;
    const int64_t r = r0 + rl, c = c0 + cg;
    __half h[8];
    if (r < R && c < C) {
      load8_half(X + r * C + c, C - c, vec != 0 && c + 8 <= C, h);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) h[j] = __float2half_rn(0.f);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float q = fminf(127.f, fmaxf(-127.f, rint_small(__fmul_rn(__half2float(h[j]), s_s[cg + j]))));
      tile[(cg + j) * kCqPitch + rl] = __float2half_rn(q);   // exact: an integer of magnitude <= 127
      sqc[j] += static_cast<int>(q * q);
    }
  }
  if (sq != nullptr) {
    // lanes l, l ^ 8, l ^ 16, l ^ 24 hold the same 8 columns
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      sqc[j] += __shfl_xor_sync(0xffffffffu, sqc[j], 8);
      sqc[j] += __shfl_xor_sync(0xffffffffu, sqc[j], 16);
    }
    if (lane < 8)
#pragma unroll
      for (int j = 0; j < 8; ++j) atomicAdd(&sq_s[cg + j], sqc[j]);
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int idx = t + kThreads * i;
    const int cl = idx >> 3, rc = (idx & 7) * 8;
    const int64_t c = c0 + cl, r = r0 + rc;
    if (c < C && r < R_pad) {
      const uint32_t* src = reinterpret_cast<const uint32_t*>(tile + cl * kCqPitch + rc);
      *reinterpret_cast<uint4*>(Xt + c * R_pad + r) = make_uint4(src[0], src[1], src[2], src[3]);
    }
  }
  if (sq != nullptr && t < kCqTile && c0 + t < C && sq_s[t] != 0)
    atomicAdd(&sq[(c0 + t) * nchunks + (r0 >> 10)], sq_s[t]);
}

// tsq[(c / 256) * nchunks + k] = max over the 256 columns c of a tile of
// sq[c, k] (the per-tile chunk maxima of the accumulation plan).
__global__ void __launch_bounds__(kThreads) tile_sq_kernel(const int* __restrict__ sq, int64_t C, int64_t nchunks,
                                                           uint32_t* __restrict__ tsq) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < C * nchunks;
       i += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int64_t c = i / nchunks, k = i - c * nchunks;
    if (sq[i] != 0) atomicMax(tsq + (c >> 8) * nchunks + k, static_cast<uint32_t>(sq[i]));
  }
}

// Diagnostic: one block waits, through the same bounded wait as every
// pipeline of the library, on an mbarrier that nothing arrives on; after
// limit_ns it records ST_TIMEOUT (where = kWhereDiagnostic) and returns.
constexpr int kWhereDiagnostic = 9;
__global__ void __launch_bounds__(32) wait_limit_kernel(DevStatus* st, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  mbar_wait_limit(&bar, 0, &abort_flag, st, kWhereDiagnostic, 0, limit_ns);
}

int grid_rows(int64_t rows) {
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  return static_cast<int>(rows < cap ? (rows > 0 ? rows : 1) : cap);
}

template <typename F>
cudaError_t dispatch_dt(int dt, F&& f) {
  switch (dt) {
    case DT_F16: return f(static_cast<__half*>(nullptr));
    case DT_BF16: return f(static_cast<__nv_bfloat16*>(nullptr));
    case DT_F32: return f(static_cast<float*>(nullptr));
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// Row quantization with the rows streamed by bulk copies (16-bit input, K a
// multiple of 8): two row buffers in shared memory; while the block
// quantizes row i from one, a bulk copy brings row i + 1 into the other, so
// the HBM reads never wait for the arithmetic.  Same arithmetic as
// act_quantize_staged_kernel.  Waits are bounded: on a timeout the block
// records ST_TIMEOUT, lets its copy in flight land (bounded) and returns.
// ---------------------------------------------------------------------------
constexpr int kBulkMaxRowBytes = 100 * 1024;   // two buffers fit one block per SM

// 8 consecutive elements of a row staged in shared memory (16-byte aligned),
// cast to fp16 (RNE), with 16-byte loads.
template <typename T>
__device__ __forceinline__ void smem_load8_half(const T* p, __half (&h)[8]) {
  constexpr int kVec = 16 / static_cast<int>(sizeof(T));   // elements per 16-byte load
#pragma unroll
  for (int v = 0; v < 8 / kVec; ++v) {
    const uint4 u = *reinterpret_cast<const uint4*>(p + v * kVec);
    const T* x = reinterpret_cast<const T*>(&u);
#pragma unroll
    for (int j = 0; j < kVec; ++j) h[v * kVec + j] = to_half(x[j]);
  }
}
bool ensure_smem_attr(const void* fn, int smem_bytes) {
  struct Entry {
    const void* fn;
    int dev, smem;
  };
  static Entry done[128];
  static int used = 0;
  static std::mutex mu;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (done[i].fn == fn && done[i].dev == dev && done[i].smem >= smem_bytes) return true;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) != cudaSuccess) return false;
  if (used < 128) done[used++] = Entry{fn, dev, smem_bytes};
  return true;
}

// Blocks per SM of a kernel at a given dynamic shared-memory size, cached
// per (kernel, device, size) so that launches made while a stream is being
// captured into a CUDA graph query nothing.
int cached_blocks_per_sm(const void* fn, int threads, int smem) {
  struct Entry {
    const void* fn;
    int dev, threads, smem, per_sm;
  };
  static Entry cache[64];
  static int used = 0;
  static std::mutex mu;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (cache[i].fn == fn && cache[i].dev == dev && cache[i].threads == threads && cache[i].smem == smem)
      return cache[i].per_sm;
  int per_sm = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem) != cudaSuccess || per_sm < 1) {
    cudaGetLastError();
    per_sm = 1;
  }
  if (used < 64) cache[used++] = Entry{fn, dev, threads, smem, per_sm};
  return per_sm;
}

constexpr int kWhereQuantize = 6;               // status `where` of a timed-out row copy

template <typename T, typename OutT, int kBlock>
__global__ void __launch_bounds__(kBlock) row_quantize_bulk_kernel(
    const T* __restrict__ A, int64_t M, int64_t K, int64_t ld, const uint32_t* __restrict__ mask,
    const int* __restrict__ idx, DevStatus* st, int64_t cap_pad, float* __restrict__ scale,
    OutT* __restrict__ codes, __half* __restrict__ sub, uint32_t* __restrict__ asq, int row_bytes) {
  extern __shared__ __align__(16) uint8_t rowbuf[];   // two buffers of row_bytes (a multiple of 16)
  __shared__ float red[32];
  __shared__ int chunk_sq[kStagedMaxChunks];
  __shared__ __align__(8) uint64_t full[2];
  __shared__ int abort_flag;
  const int used = (mask != nullptr) ? st->used : 0;
  const int used_pad = (used + 63) / 64 * 64;
  const int nchunks = static_cast<int>((ld + 1023) / 1024);
  const uint32_t bytes = static_cast<uint32_t>(K * static_cast<int64_t>(sizeof(T)));
  if (threadIdx.x == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int64_t m0 = blockIdx.x;
  if (threadIdx.x == 0 && m0 < M) {
    mbar_arrive_expect_tx(&full[0], bytes);
    bulk_load(rowbuf, A + m0 * K, bytes, &full[0]);
  }
  int i = 0;
  for (int64_t m = m0; m < M; m += gridDim.x, ++i) {
    const int b = i & 1;
    const int64_t mn = m + gridDim.x;
    if (threadIdx.x == 0 && mn < M) {   // the other buffer was released at the end of the previous row
      mbar_arrive_expect_tx(&full[b ^ 1], bytes);
      bulk_load(rowbuf + (b ^ 1) * row_bytes, A + mn * K, bytes, &full[b ^ 1]);
    }
    volatile int* abort_p = &abort_flag;
    if (!__syncthreads_and(mbar_wait(&full[b], (i >> 1) & 1, abort_p, st, kWhereQuantize))) {
      // let the copy in flight into the other buffer land before the block exits
      if (threadIdx.x == 0 && mn < M) {
        *abort_p = 0;
        mbar_wait(&full[b ^ 1], ((i + 1) >> 1) & 1, abort_p, nullptr, 0);
      }
      return;
    }
    const T* row = reinterpret_cast<const T*>(rowbuf + b * row_bytes);
    float amax = 0.f;
    for (int64_t c = static_cast<int64_t>(threadIdx.x) * 8; c < K; c += kBlock * 8) {
      __half h[8];
      smem_load8_half(row + c, h);
      const uint32_t bits = (mask != nullptr) ? ((mask[c >> 5] >> (c & 31)) & 0xFFu) : 0u;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (!((bits >> j) & 1u)) amax = fmaxf(amax, fabsf(__half2float(h[j])));
    }
    if (asq != nullptr)
      for (int k = threadIdx.x; k < nchunks; k += kBlock) chunk_sq[k] = 0;
    amax = block_max(amax, red);
    const float s = (amax > 0.f) ? __fdiv_rn(127.0f, amax) : 0.f;
    OutT* out = codes + m * ld;
    for (int64_t c0 = 0; c0 < ld; c0 += kBlock * 8) {   // every thread runs every iteration
      const int64_t c = c0 + static_cast<int64_t>(threadIdx.x) * 8;
      float sq = 0.f;
      if (c < ld) {
        __half h[8];
        if (c < K) {
          smem_load8_half(row + c, h);
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) h[j] = __float2half_rn(0.f);
        }
        const uint32_t bits = (mask != nullptr && c < K) ? ((mask[c >> 5] >> (c & 31)) & 0xFFu) : 0u;
        float q[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float r = rint_small(__fmul_rn(__half2float(h[j]), s));
          q[j] = ((bits >> j) & 1u) ? 0.f : fminf(127.f, fmaxf(-127.f, r));
          sq += q[j] * q[j];
        }
        if constexpr (sizeof(OutT) == 1) {
          uint32_t w[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) w[j] = static_cast<uint32_t>(static_cast<int>(q[j])) & 0xFFu;
          *reinterpret_cast<uint2*>(out + c) = make_uint2(w[0] | (w[1] << 8) | (w[2] << 16) | (w[3] << 24),
                                                          w[4] | (w[5] << 8) | (w[6] << 16) | (w[7] << 24));
        } else {
          uint4 o;
          __half2* o2 = reinterpret_cast<__half2*>(&o);
#pragma unroll
          for (int j = 0; j < 4; ++j) o2[j] = __floats2half2_rn(q[2 * j], q[2 * j + 1]);
          *reinterpret_cast<uint4*>(out + c) = o;
        }
      }
      if (asq != nullptr) {
        int v = static_cast<int>(sq);
#pragma unroll
        for (int k = 16; k > 0; k >>= 1) v += __shfl_xor_sync(0xffffffffu, v, k);
        const int64_t cw = c0 + static_cast<int64_t>(threadIdx.x & ~31) * 8;
        if ((threadIdx.x & 31) == 0 && v != 0) atomicAdd(&chunk_sq[cw >> 10], v);
      }
    }
    if (sub != nullptr) {
      for (int j = threadIdx.x; j < used_pad; j += kBlock)
        sub[m * cap_pad + j] = (j < used) ? to_half(row[idx[j]]) : __float2half_rn(0.f);
    }
    if (asq != nullptr) {
      __syncthreads();
      for (int k = threadIdx.x; k < nchunks; k += kBlock)
        if (chunk_sq[k] != 0) atomicMax(asq + (m >> 8) * nchunks + k, static_cast<uint32_t>(chunk_sq[k]));
    }
    __syncthreads();   // also: this row buffer is no longer read
    if (threadIdx.x == 0) scale[m] = amax;
  }
}

template <typename T, typename OutT, int kBlock>
cudaError_t launch_bulk_block(int prof_id, const T* A, int64_t M, int64_t K, int64_t K_pad, const uint32_t* mask,
                              const int* idx, DevStatus* st, int64_t cap_pad, float* scale, OutT* codes, __half* sub,
                              uint32_t* asq, int row_bytes, int sms, cudaStream_t s) {
  const int smem = 2 * row_bytes;
  if (!ensure_smem_attr(reinterpret_cast<const void*>(row_quantize_bulk_kernel<T, OutT, kBlock>),
                        2 * kBulkMaxRowBytes))
    return cudaGetLastError();
  const int per_sm =
      cached_blocks_per_sm(reinterpret_cast<const void*>(row_quantize_bulk_kernel<T, OutT, kBlock>), kBlock, smem);
  const int grid = static_cast<int>(std::min<int64_t>(M, static_cast<int64_t>(sms) * per_sm));
  ProfScope ps(prof_id, s);
  row_quantize_bulk_kernel<T, OutT, kBlock><<<grid, kBlock, smem, s>>>(A, M, K, K_pad, mask, idx, st, cap_pad, scale,
                                                                       codes, sub, asq, row_bytes);
  return cudaGetLastError();
}

// Rows are streamed through two shared-memory buffers per block; the rows in
// flight per SM are the blocks that fit.  Short rows get small blocks (up to
// 7 of 256 threads per SM for 16 KB rows), long rows one or two blocks of
// 1024 threads.
template <typename T, typename OutT>
cudaError_t launch_bulk(int prof_id, const T* A, int64_t M, int64_t K, int64_t K_pad, const uint32_t* mask,
                        const int* idx, DevStatus* st, int64_t cap_pad, float* scale, OutT* codes, __half* sub,
                        uint32_t* asq, cudaStream_t s) {
  const int row_bytes = static_cast<int>(round_up(K * static_cast<int64_t>(sizeof(T)), 16));
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int fit = std::max(1, (220 * 1024) / (2 * row_bytes));   // blocks per SM that shared memory allows
  if (fit >= 6)
    return launch_bulk_block<T, OutT, 256>(prof_id, A, M, K, K_pad, mask, idx, st, cap_pad, scale, codes, sub, asq,
                                           row_bytes, sms, s);
  if (fit >= 3)
    return launch_bulk_block<T, OutT, 512>(prof_id, A, M, K, K_pad, mask, idx, st, cap_pad, scale, codes, sub, asq,
                                           row_bytes, sms, s);
  return launch_bulk_block<T, OutT, 1024>(prof_id, A, M, K, K_pad, mask, idx, st, cap_pad, scale, codes, sub, asq,
                                          row_bytes, sms, s);
}

// Launch of the staged row quantization (K_pad <= kStagedMaxLd): one row per
// block at a time, as many blocks as fit with the row in shared memory.
template <typename T, typename OutT>
cudaError_t launch_staged(int prof_id, const T* A, int64_t M, int64_t K, int64_t K_pad, bool vec, const uint32_t* mask,
                          const int* idx, const DevStatus* st, int64_t cap_pad, float* scale, OutT* codes,
                          __half* sub, uint32_t* asq, cudaStream_t s) {
  const int smem = static_cast<int>(K_pad * 2);
  if (!ensure_smem_attr(reinterpret_cast<const void*>(act_quantize_staged_kernel<T, OutT>), kStagedMaxLd * 2))
    return cudaGetLastError();
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int per_sm = cached_blocks_per_sm(reinterpret_cast<const void*>(act_quantize_staged_kernel<T, OutT>), kThreads,
                                          smem);
  const int grid = static_cast<int>(std::min<int64_t>(M, static_cast<int64_t>(sms) * per_sm));
  ProfScope ps(prof_id, s);
  act_quantize_staged_kernel<T, OutT><<<grid, kThreads, smem, s>>>(A, M, K, K_pad, vec ? 1 : 0, mask, idx, st, cap_pad,
                                                                   scale, codes, sub, asq);
  return cudaGetLastError();
}

cudaError_t launch_quantize_weight(const void* W, int wt, int64_t N, int64_t K, int64_t ld, bool vec, int8_t* CB,
                                   float* SCB, cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  // 16-bit weights with 16-byte rows that fit the ring: the row pass of the
  // fused activation quantization, each code row stored in bulk
  if (act_quant_fused_supported(wt, K) && ld == round_up(K, 16))
    return launch_quantize_weight_fused(W, wt, N, K, ld, CB, SCB, s);
  return dispatch_dt(wt, [&](auto* tag) {
    using T = std::remove_pointer_t<decltype(tag)>;
    if (vec && K * static_cast<int64_t>(sizeof(T)) <= kBulkMaxRowBytes)
      return launch_bulk<T, int8_t>(K_QUANTIZE_WEIGHT, static_cast<const T*>(W), N, K, ld, nullptr, nullptr, nullptr, 0,
                                    SCB, CB, nullptr, nullptr, s);
    if (ld <= kStagedMaxLd)
      return launch_staged<T, int8_t>(K_QUANTIZE_WEIGHT, static_cast<const T*>(W), N, K, ld, vec, nullptr, nullptr,
                                      nullptr, 0, SCB, CB, nullptr, nullptr, s);
    ProfScope ps(K_QUANTIZE_WEIGHT, s);
    row_quantize_kernel<T, int8_t><<<grid_rows(N), kThreads, 0, s>>>(
        static_cast<const T*>(W), N, K, ld, vec ? 1 : 0, nullptr, nullptr, nullptr, 0, SCB, CB, nullptr, nullptr);
    return cudaGetLastError();
  });
}

cudaError_t launch_colmax(const void* A, int at, int64_t M, int64_t K, bool vec, uint32_t* colmax,
                          cudaStream_t s) {
  if (M == 0 || K == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(ceil_div(K, 256)), static_cast<unsigned>(ceil_div(M, kColRows)));
  return dispatch_dt(at, [&](auto* tag) {
    using T = std::remove_pointer_t<decltype(tag)>;
    ProfScope ps(K_COLMAX, s);
    colmax_kernel<T><<<grid, kThreads, 0, s>>>(static_cast<const T*>(A), M, K, vec ? 1 : 0, colmax);
    return cudaGetLastError();
  });
}

cudaError_t launch_outlier_index(const uint32_t* colmax, int64_t K, float thr, int64_t cap, int* idx,
                                 uint32_t* mask, DevStatus* st, cudaStream_t s) {
  ProfScope ps(K_OUTLIER_INDEX, s);
  outlier_index_kernel<<<1, 1024, 0, s>>>(colmax, K, thr, cap, idx, mask, st);
  return cudaGetLastError();
}

cudaError_t launch_row_quantize(const void* A, int at, int64_t M, int64_t K, int64_t K_pad, bool vec,
                                const uint32_t* mask, const int* idx, DevStatus* st, int64_t cap_pad,
                                float* SCA, __half* Aq, __half* subA, uint32_t* asq, cudaStream_t s) {
  if (M == 0) return cudaSuccess;
  return dispatch_dt(at, [&](auto* tag) {
    using T = std::remove_pointer_t<decltype(tag)>;
    if (vec && K * static_cast<int64_t>(sizeof(T)) <= kBulkMaxRowBytes)
      return launch_bulk<T, __half>(K_ROW_QUANTIZE, static_cast<const T*>(A), M, K, K_pad, mask, idx, st, cap_pad,
                                    SCA, Aq, subA, asq, s);
    if (K_pad <= kStagedMaxLd)
      return launch_staged<T, __half>(K_ROW_QUANTIZE, static_cast<const T*>(A), M, K, K_pad, vec, mask, idx, st,
                                      cap_pad, SCA, Aq, subA, asq, s);
    ProfScope ps(K_ROW_QUANTIZE, s);
    row_quantize_kernel<T, __half><<<grid_rows(M), kThreads, 0, s>>>(
        static_cast<const T*>(A), M, K, K_pad, vec ? 1 : 0, mask, idx, st, cap_pad, SCA, Aq, subA, asq);
    return cudaGetLastError();
  });
}

cudaError_t launch_build_subB(const int8_t* CB, int64_t ld, const float* SCB, int64_t N, const int* idx,
                              const DevStatus* st, int64_t cap_pad, __half* subB, cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  const int blocks = static_cast<int>(std::min<int64_t>(ceil_div(N, kThreads / 32), 152 * 8));
  ProfScope ps(K_SUBB, s);
  build_subB_kernel<<<blocks, kThreads, 0, s>>>(CB, ld, SCB, N, idx, st, cap_pad, subB);
  return cudaGetLastError();
}

int64_t gradout_partial_chunks(int64_t M) { return ceil_div(M > 0 ? M : 1, kSumRows); }

cudaError_t launch_gradout_prepass(const void* G, int gt, int64_t M, int64_t N, bool vec, __half* G16,
                                   int64_t N_pad, void* grad_bias, int bt, float* partial, int64_t max_chunks,
                                   cudaStream_t s) {
  const int64_t chunks = gradout_partial_chunks(M);
  if (chunks > max_chunks) return cudaErrorInvalidValue;
  const int64_t width = (G16 != nullptr) ? N_pad : N;
  if (M > 0 && width > 0) {
    const dim3 grid(static_cast<unsigned>(ceil_div(width, 256)), static_cast<unsigned>(chunks));
    cudaError_t e = dispatch_dt(gt, [&](auto* tag) {
      using T = std::remove_pointer_t<decltype(tag)>;
      ProfScope ps(K_GRADOUT_PREPASS, s);
      gradout_prepass_kernel<T><<<grid, kThreads, 0, s>>>(static_cast<const T*>(G), M, N, vec ? 1 : 0, G16, N_pad,
                                                          grad_bias != nullptr ? partial : nullptr);
      return cudaGetLastError();
    });
    if (e != cudaSuccess) return e;
  }
  if (grad_bias == nullptr || N == 0) return cudaSuccess;
  return launch_grad_bias_finalize(partial, M, N, grad_bias, bt, s);
}

cudaError_t launch_grad_bias_finalize(const float* partial, int64_t M, int64_t N, void* grad_bias, int bt,
                                      cudaStream_t s) {
  if (grad_bias == nullptr || N == 0) return cudaSuccess;
  if (M == 0) return cudaMemsetAsync(grad_bias, 0, static_cast<size_t>(N) * (bt == DT_F32 ? 4 : 2), s);
  const int64_t chunks = gradout_partial_chunks(M);
  const int blocks = static_cast<int>(std::min<int64_t>(ceil_div(N, kThreads), 152 * 4));
  return dispatch_dt(bt, [&](auto* tag) {
    using BT = std::remove_pointer_t<decltype(tag)>;
    ProfScope ps(K_GRAD_BIAS_FINALIZE, s);
    grad_bias_finalize_kernel<BT><<<blocks, kThreads, 0, s>>>(partial, chunks, N, static_cast<BT*>(grad_bias));
    return cudaGetLastError();
  });
}

cudaError_t launch_col_quantize(const void* X, int xt, int64_t R, int64_t C, bool vec, const uint32_t* colmax,
                                int64_t R_pad, float* scale, __half* Xt, int* sq, uint32_t* tsq, cudaStream_t s) {
  if (R_pad == 0 || C == 0) return cudaSuccess;
  const int64_t nchunks = ceil_div(R_pad, 1024);
  const dim3 grid(static_cast<unsigned>(ceil_div(R_pad, kCqTile)), static_cast<unsigned>(ceil_div(C, kCqTile)));
  cudaError_t e = dispatch_dt(xt, [&](auto* tag) {
    using T = std::remove_pointer_t<decltype(tag)>;
    ProfScope ps(K_COL_QUANTIZE, s);
    col_quantize_kernel<T><<<grid, kThreads, 0, s>>>(static_cast<const T*>(X), R, C, vec ? 1 : 0, colmax, R_pad, scale,
                                                    Xt, sq, nchunks);
    return cudaGetLastError();
  });
  if (e != cudaSuccess || sq == nullptr) return e;
  ProfScope ps(K_COL_QUANTIZE, s);
  tile_sq_kernel<<<static_cast<unsigned>(std::min<int64_t>(ceil_div(C * nchunks, kThreads), 4096)), kThreads, 0, s>>>(
      sq, C, nchunks, tsq);
  return cudaGetLastError();
}

cudaError_t launch_wait_limit(DevStatus* st, unsigned long long limit_ns, cudaStream_t s) {
  wait_limit_kernel<<<1, 32, 0, s>>>(st, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_silu(const void* h, int dt, int64_t n, bool vec, void* out, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int blocks = static_cast<int>(std::min<int64_t>(ceil_div(n, kThreads * 8), 152 * 8));
  return dispatch_dt(dt, [&](auto* tag) {
    using T = std::remove_pointer_t<decltype(tag)>;
    ProfScope ps(K_SILU, s);
    silu_kernel<T><<<blocks, kThreads, 0, s>>>(static_cast<const T*>(h), n, vec ? 1 : 0, static_cast<T*>(out));
    return cudaGetLastError();
  });
}

cudaError_t launch_silu_backward(const void* g, const void* h, int dt, int64_t n, bool vec, void* out,
                                 cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int blocks = static_cast<int>(std::min<int64_t>(ceil_div(n, kThreads * 8), 152 * 8));
  return dispatch_dt(dt, [&](auto* tag) {
    using T = std::remove_pointer_t<decltype(tag)>;
    ProfScope ps(K_SILU_BACKWARD, s);
    silu_backward_kernel<T><<<blocks, kThreads, 0, s>>>(static_cast<const T*>(g), static_cast<const T*>(h), n,
                                                        vec ? 1 : 0, static_cast<T*>(out));
    return cudaGetLastError();
  });
}

}  // namespace i8lt
