// Tensor-core GEMMs of the int8 quantized linear layer (sm_103a, tcgen05).
//
// Forward (K5): out[m,n] = Cacc[m,n] * SCA[m] * SCB[n] / 127^2
//                          + sum_j subA[m,j] subB[n,j] + bias[n] (+ residual)
//   Cacc = sum_k Aq[m,k] CB[n,k] is the exact integer product of the int8
//   codes (bitsandbytes PR #33 "Memory efficient backward", the int8 matmul of
//   the forward and the "Mixed-precision decomposition matmul" review thread).
//   sm_103a has no int8 MMA (ptxas rejects tcgen05.mma .kind::i8 for this
//   target), so the codes enter the fp16 tensor cores as exact fp16 integers
//   and accumulate in fp32 TMEM.  Every partial sum of at most 1024 products
//   is an integer of magnitude <= 1024 * 127^2 < 2^24, hence exact in fp32;
//   every 1024-deep chunk is drained from TMEM into an int32 running sum held
//   in TMEM, so Cacc is exact for any K <= 133144.
//   Tile 128 (tokens) x 256 (features) x 64 per stage.  A = Aq via TMA
//   (128B swizzle); B = CB int8 via TMA, widened to fp16 in shared memory by
//   four converter warps (in place, 128B-swizzled K-major).  The outlier
//   sub-GEMM subA x subB^T runs as one more fp32 accumulation unit.
//
// Backward (K6): grad_A[m,k] = sum_n fp16(G)[m,n] * Wdq[n,k],
//   Wdq[n,k] = fp16_rn(fp32(CB[n,k]) * (SCB[n] * fp32(1/127))), rebuilt per
//   tile in shared memory and never stored (PR description, backward bullet;
//   review thread on ".mul(1/127.0)").  Computed transposed,
//   D[k, m] = Wdq^T G16^T, so the converted operand is the 128-row A side
//   (half the conversion work of a 256-row B side).  A = Wdq^T stored
//   MN-major (k contiguous, as CB's rows are), B = G16 via TMA, K-major.
//
// Warp roles (320 threads): warp 0 TMA producer, warp 1 MMA issuer and TMEM
// owner, warps 2-5 int8 -> fp16 converters, warps 6-9 epilogue (warp w reads
// TMEM lanes 32 * (w % 4) ...).  Every wait is bounded (see mbar_wait).
#include <algorithm>

#include "i8lt_internal.h"

namespace i8lt {

namespace {

constexpr int kThreads = 320;
constexpr int kStages = 4;
constexpr int kChunkKB = 16;   // K-blocks of 64 per exact fp32 chunk: 1024 products

constexpr int kWarpProducer = 0;
constexpr int kWarpMMA = 1;
constexpr int kWarpCvt0 = 2;   // 2..5
constexpr int kWarpEpi0 = 6;   // 6..9
constexpr int kCvtThreads = 128;
constexpr int kEpiThreads = 128;
constexpr int kBarCvt = 1;     // named barrier ids
constexpr int kBarEpi = 2;

// roles reported in the status word when a wait times out
enum { kWhereProducer = 1, kWhereCvt = 2, kWhereMMA = 3, kWhereEpi = 4, kWhereTeardown = 5 };

struct __align__(8) Barriers {
  uint64_t tma_full[kStages];
  uint64_t cvt_full[kStages];
  uint64_t empty[kStages];
  uint64_t acc_full;
  uint64_t acc_empty;
  uint64_t teardown;
  uint32_t tmem_base;
  int abort_flag;
};

// --- shared memory plan (identical for both GEMMs) --------------------------
// stage s: [A tile 16 KB][B tile 32 KB]; forward: A = Aq (TMA), B = CB int8
// (TMA into the first 16 KB, widened in place to 32 KB fp16); backward:
// A = Wdq^T (int8 TMA into the first 8 KB, widened in place to 16 KB),
// B = G16 (TMA).
constexpr int kATileBytes = 128 * kBK * 2;   // 16 KB
constexpr int kBTileBytes = 256 * kBK * 2;   // 32 KB
constexpr int kStageBytes = kATileBytes + kBTileBytes;
constexpr int kSmemTiles = kStages * kStageBytes;
constexpr int kSmemBytes = 1024 /*align slack*/ + kSmemTiles + 2 * 256 * 4 /*epilogue vectors*/ + sizeof(Barriers);

__device__ __forceinline__ uint32_t f2i_rn(uint32_t fbits) {
  return static_cast<uint32_t>(__float2int_rn(__uint_as_float(fbits)));
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
// exactly as (2^23 + q + 128) - (2^23 + 128).
__device__ __forceinline__ void i8x4_scale_to_h4(uint32_t w, float f, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const float c = 8388736.0f;   // 2^23 + 128
  const float q0 = __fsub_rn(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540)), c);
  const float q1 = __fsub_rn(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7541)), c);
  const float q2 = __fsub_rn(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7542)), c);
  const float q3 = __fsub_rn(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7543)), c);
  __half2 a = __floats2half2_rn(__fmul_rn(q0, f), __fmul_rn(q1, f));
  __half2 b = __floats2half2_rn(__fmul_rn(q2, f), __fmul_rn(q3, f));
  lo = *reinterpret_cast<uint32_t*>(&a);
  hi = *reinterpret_cast<uint32_t*>(&b);
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

// Grouped raster: consecutive CTAs walk `group` M-tiles of one N-tile, so a
// wave shares its A rows and B rows through L2.
__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int group, int& tm, int& tn) {
  const int per_group = group * num_n;
  const int g = t / per_group;
  const int first = g * group;
  const int gm = min(group, num_m - first);
  const int local = t - g * per_group;
  tm = first + local % gm;
  tn = local / gm;
}

// ---------------------------------------------------------------------------
// Forward GEMM
// ---------------------------------------------------------------------------
template <typename OutT>
__device__ __forceinline__ void fwd_store_row(const FwdEpiArgs& e, int64_t m, int n_base, const float (&v)[32],
                                              bool vec) {
  OutT* out = static_cast<OutT*>(e.out) + m * static_cast<int64_t>(e.N) + n_base;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int n = n_base + q * 8;
    if (n >= e.N) break;
    float f[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = v[q * 8 + i];
    store8(out + q * 8, e.N - n, vec && n + 8 <= e.N, f);
  }
}

template <typename OutT>
__device__ __forceinline__ void fwd_load_residual(const FwdEpiArgs& e, int64_t m, int n_base, float (&v)[32],
                                                  bool vec) {
  const OutT* res = static_cast<const OutT*>(e.residual) + m * static_cast<int64_t>(e.N) + n_base;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int n = n_base + q * 8;
    float f[8];
    if (n < e.N) {
      load8_float(res + q * 8, e.N - n, vec && n + 8 <= e.N, f);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) v[q * 8 + i] += f[i];
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    fwd_gemm_kernel(const __grid_constant__ FwdGemmArgs g, const FwdEpiArgs e, int num_m, int num_n, int group) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* scb_s = reinterpret_cast<float*>(smem + kSmemTiles);
  float* bias_s = scb_s + 256;
  Barriers* bars = reinterpret_cast<Barriers*>(bias_s + 256);
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int tm, tn;
  tile_coords(blockIdx.x, num_m, num_n, group, tm, tn);
  const int m0 = tm * kFwdBM, n0 = tn * kFwdBN;

  const int KB = (e.K_pad + kBK - 1) / kBK;
  const int nchunks = (KB + kChunkKB - 1) / kChunkKB;
  const int used = e.use_outliers ? e.st->used : 0;
  const int OB = (used + kBK - 1) / kBK;
  const int total_blocks = KB + OB;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->tma_full[s], 1);
      mbar_init(&bars->cvt_full[s], kCvtThreads);
      mbar_init(&bars->empty[s], 1);
    }
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, kEpiThreads / 32);
    mbar_init(&bars->teardown, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMMA) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
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
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t tmem_R = tmem;          // int32 running sum, columns [0, 256)
  const uint32_t tmem_X = tmem + 256;    // fp32 accumulation unit, columns [256, 512)

  if (warp == kWarpProducer) {
    if (lane == 0) {
      int issued = 0;
      for (int it = 0; it < total_blocks; ++it) {
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        if (!mbar_wait(&bars->empty[s], ph ^ 1, abort_flag, e.st, kWhereProducer)) break;
        uint8_t* sa = smem + s * kStageBytes;
        uint8_t* sb = sa + kATileBytes;
        if (it < KB) {
          mbar_arrive_expect_tx(&bars->tma_full[s], kATileBytes + kFwdBN * kBK);
          tma_load_2d(sa, &g.tmA, it * kBK, m0, &bars->tma_full[s]);
          tma_load_2d(sb, &g.tmB, it * kBK, n0, &bars->tma_full[s]);
        } else {
          const int ob = it - KB;
          mbar_arrive_expect_tx(&bars->tma_full[s], kATileBytes + kBTileBytes);
          tma_load_2d(sa, &g.tmSA, ob * kBK, m0, &bars->tma_full[s]);
          tma_load_2d(sb, &g.tmSB, ob * kBK, n0, &bars->tma_full[s]);
        }
        issued = it + 1;
      }
      // teardown: every issued copy must have landed before the CTA exits
      for (int it = max(0, issued - kStages); it < issued; ++it)
        mbar_wait_teardown(&bars->tma_full[it % kStages], (it / kStages) & 1, e.st);
    }
  } else if (warp == kWarpMMA) {
    if (lane == 0) {
      const uint32_t idesc = make_idesc_f16(kFwdBM, kFwdBN, false, false);
      const int units = nchunks + (OB > 0 ? 1 : 0);
      bool ok = true;
      for (int u = 0; u < units && ok; ++u) {
        if (u >= 1 && !mbar_wait(&bars->acc_empty, (u - 1) & 1, abort_flag, e.st, kWhereMMA)) break;
        tc_fence_after();
        const bool is_int = u < nchunks;
        const int b0 = is_int ? u * kChunkKB : KB;
        const int b1 = is_int ? min(KB, b0 + kChunkKB) : total_blocks;
        for (int it = b0; it < b1; ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!mbar_wait(&bars->tma_full[s], ph, abort_flag, e.st, kWhereMMA)) { ok = false; break; }
          if (is_int && !mbar_wait(&bars->cvt_full[s], ph, abort_flag, e.st, kWhereMMA)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_base = smem_u32(smem + s * kStageBytes);
          const uint32_t b_base = a_base + kATileBytes;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint64_t ad = make_sdesc(a_base + k * 32, 16, 1024, kSwizzle128B);
            const uint64_t bd = make_sdesc(b_base + k * 32, 16, 1024, kSwizzle128B);
            umma_f16(tmem_X, ad, bd, idesc, (it > b0 || k > 0) ? 1u : 0u);
          }
          umma_commit(&bars->empty[s]);
        }
        if (ok) umma_commit(&bars->acc_full);
      }
      umma_commit(&bars->teardown);
      mbar_wait_teardown(&bars->teardown, 0, e.st);
    }
  } else if (warp < kWarpEpi0) {
    // ---- converters: CB int8 [256 rows][64] -> fp16 128B-swizzled K-major
    const int ct = threadIdx.x - kWarpCvt0 * 32;
    for (int it = 0; it < KB; ++it) {
      const int s = it % kStages;
      const uint32_t ph = (it / kStages) & 1;
      const bool ok = mbar_wait(&bars->tma_full[s], ph, abort_flag, e.st, kWhereCvt);
      uint8_t* sb = smem + s * kStageBytes + kATileBytes;
      uint4 v[8];
      if (ok) {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = reinterpret_cast<const uint4*>(sb)[ct + kCvtThreads * j];
      }
      // all int8 read before the in-place widening; all converters agree to go on
      if (!named_bar_and(kBarCvt, kCvtThreads, ok)) break;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int item = ct + kCvtThreads * j;   // row = item / 4, 16-byte quarter q = item % 4
        const int row = item >> 2, q = item & 3;
        uint4 o0, o1;
        i8x4_to_h4(v[j].x, o0.x, o0.y);
        i8x4_to_h4(v[j].y, o0.z, o0.w);
        i8x4_to_h4(v[j].z, o1.x, o1.y);
        i8x4_to_h4(v[j].w, o1.z, o1.w);
        uint8_t* rowp = sb + row * 128;
        *reinterpret_cast<uint4*>(rowp + (((2 * q) ^ (row & 7)) << 4)) = o0;
        *reinterpret_cast<uint4*>(rowp + (((2 * q + 1) ^ (row & 7)) << 4)) = o1;
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars->cvt_full[s]);
    }
  } else {
    // ---- epilogue
    const int et = threadIdx.x - kWarpEpi0 * 32;
    const int quad = warp & 3;
    for (int i = et; i < 256; i += kEpiThreads) {
      const int n = n0 + i;
      scb_s[i] = (n < e.N) ? e.SCB[n] : 0.f;
      bias_s[i] = (n < e.N && e.bias != nullptr) ? load_any(e.bias, e.bias_dt, n) : 0.f;
    }
    named_bar_sync(kBarEpi, kEpiThreads);
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    bool ok = true;
    for (int u = 0; u < nchunks; ++u) {
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->acc_full, u & 1, abort_flag, e.st, kWhereEpi))) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int gcol = 0; gcol < 8; ++gcol) {
        uint32_t x[32], r[32];
        tmem_ld32(tmem_X + lane_off + gcol * 32, x);
        if (u > 0) {
          tmem_ld32(tmem_R + lane_off + gcol * 32, r);
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] += f2i_rn(x[j]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = f2i_rn(x[j]);
        }
        tmem_st32(tmem_R + lane_off + gcol * 32, r);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->acc_empty);
    }
    const bool has_o = OB > 0;
    if (ok && has_o && !__all_sync(0xffffffffu, mbar_wait(&bars->acc_full, nchunks & 1, abort_flag, e.st, kWhereEpi)))
      ok = false;
    if (ok) {
      tc_fence_after();
      const int64_t m = m0 + quad * 32 + lane;
      const bool row_ok = m < e.M;
      const float rs = row_ok ? __fmul_rn(e.SCA[m], 1.0f / 16129.0f) : 0.f;
      const bool vec = (e.N % 8) == 0;
#pragma unroll 1
      for (int gcol = 0; gcol < 8; ++gcol) {
        uint32_t r[32], o[32];
        if (nchunks > 0) {
          tmem_ld32(tmem_R + lane_off + gcol * 32, r);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = 0;
        }
        if (has_o) {
          tmem_ld32(tmem_X + lane_off + gcol * 32, o);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = 0;
        }
        const int nb = n0 + gcol * 32;
        if (!row_ok || nb >= e.N) continue;
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float sc = __fmul_rn(rs, scb_s[gcol * 32 + j]);
          v[j] = __fadd_rn(__fmaf_rn(static_cast<float>(static_cast<int32_t>(r[j])), sc, __uint_as_float(o[j])),
                           bias_s[gcol * 32 + j]);
        }
        if (e.residual != nullptr) {
          switch (e.out_dt) {
            case DT_F16: fwd_load_residual<__half>(e, m, nb, v, vec); break;
            case DT_BF16: fwd_load_residual<__nv_bfloat16>(e, m, nb, v, vec); break;
            default: fwd_load_residual<float>(e, m, nb, v, vec); break;
          }
        }
        switch (e.out_dt) {
          case DT_F16: fwd_store_row<__half>(e, m, nb, v, vec); break;
          case DT_BF16: fwd_store_row<__nv_bfloat16>(e, m, nb, v, vec); break;
          default: fwd_store_row<float>(e, m, nb, v, vec); break;
        }
        if (e.acc_i32 != nullptr) {
          int32_t* dst = e.acc_i32 + m * static_cast<int64_t>(e.N);
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (nb + j < e.N) dst[nb + j] = static_cast<int32_t>(r[j]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMMA) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// Backward GEMM (transposed): D[k, m] = sum_n Wdq[n, k] * G16[m, n]
// ---------------------------------------------------------------------------
template <typename OutT>
__device__ __forceinline__ void bwd_store(const BwdEpiArgs& e, int64_t kk, int m_base, const uint32_t (&x)[32]) {
  OutT* out = static_cast<OutT*>(e.grad_A);
  const OutT* add = static_cast<const OutT*>(e.addend);
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int64_t mm = m_base + j;
    if (mm < e.M) {
      float v = __uint_as_float(x[j]);
      if (add != nullptr) v = __fadd_rn(v, to_float(add[mm * e.K + kk]));
      out[mm * e.K + kk] = from_float<OutT>(v);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    bwd_gemm_kernel(const __grid_constant__ BwdGemmArgs g, const BwdEpiArgs e, int num_k, int num_m, int group) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Barriers* bars = reinterpret_cast<Barriers*>(smem + kSmemTiles + 2 * 256 * 4);
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int tk, tm;
  tile_coords(blockIdx.x, num_m, num_k, group, tm, tk);
  const int k0 = tk * kBwdBM, m0 = tm * kBwdBN;
  const int NB = (e.N + kBK - 1) / kBK;   // reduction blocks over n

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->tma_full[s], 1);
      mbar_init(&bars->cvt_full[s], kCvtThreads);
      mbar_init(&bars->empty[s], 1);
    }
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, kEpiThreads / 32);
    mbar_init(&bars->teardown, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMMA) {
    tmem_alloc(&bars->tmem_base, 256);
    tmem_relinquish();
  }
  if (warp == kWarpProducer && lane == 0) {
    tma_prefetch_desc(&g.tmW);
    tma_prefetch_desc(&g.tmG);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == kWarpProducer) {
    if (lane == 0) {
      int issued = 0;
      for (int it = 0; it < NB; ++it) {
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        if (!mbar_wait(&bars->empty[s], ph ^ 1, abort_flag, e.st, kWhereProducer)) break;
        uint8_t* sa = smem + s * kStageBytes;
        uint8_t* sb = sa + kATileBytes;
        mbar_arrive_expect_tx(&bars->tma_full[s], kBK * kBwdBM + kBTileBytes);
        tma_load_2d(sa, &g.tmW, k0, it * kBK, &bars->tma_full[s]);   // CB[n0:+64][k0:+128] int8
        tma_load_2d(sb, &g.tmG, it * kBK, m0, &bars->tma_full[s]);   // G16[m0:+256][n0:+64]
        issued = it + 1;
      }
      for (int it = max(0, issued - kStages); it < issued; ++it)
        mbar_wait_teardown(&bars->tma_full[it % kStages], (it / kStages) & 1, e.st);
    }
  } else if (warp == kWarpMMA) {
    if (lane == 0) {
      // A: MN-major, 128B swizzle; MN atoms (64 k) 1024 B apart, K atoms (8 n) 2048 B apart.
      const uint32_t idesc = make_idesc_f16(kBwdBM, kBwdBN, true, false);
      bool ok = true;
      for (int it = 0; it < NB; ++it) {
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        if (!mbar_wait(&bars->tma_full[s], ph, abort_flag, e.st, kWhereMMA)) { ok = false; break; }
        if (!mbar_wait(&bars->cvt_full[s], ph, abort_flag, e.st, kWhereMMA)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a_base = smem_u32(smem + s * kStageBytes);
        const uint32_t b_base = a_base + kATileBytes;
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k) {
          const uint64_t ad = make_sdesc(a_base + k * 4096, 1024, 2048, kSwizzle128B);
          const uint64_t bd = make_sdesc(b_base + k * 32, 16, 1024, kSwizzle128B);
          umma_f16(tmem, ad, bd, idesc, (it > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(&bars->empty[s]);
      }
      if (ok && NB > 0) umma_commit(&bars->acc_full);
      umma_commit(&bars->teardown);
      mbar_wait_teardown(&bars->teardown, 0, e.st);
    }
  } else if (warp < kWarpEpi0) {
    // ---- converters: CB int8 [64 n][128 k] -> Wdq^T fp16, MN-major 128B-swizzled
    const int ct = threadIdx.x - kWarpCvt0 * 32;
    for (int it = 0; it < NB; ++it) {
      const int s = it % kStages;
      const uint32_t ph = (it / kStages) & 1;
      const bool ok = mbar_wait(&bars->tma_full[s], ph, abort_flag, e.st, kWhereCvt);
      uint8_t* sa = smem + s * kStageBytes;
      uint4 v[4];
      float f[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int item = ct + kCvtThreads * j;   // n_local = item / 8, 16-byte group q = item % 8
        if (ok) v[j] = reinterpret_cast<const uint4*>(sa)[item];
        const int n = it * kBK + (item >> 3);
        f[j] = (n < e.N) ? __fmul_rn(__ldg(e.SCB + n), 1.0f / 127.0f) : 0.f;
      }
      if (!named_bar_and(kBarCvt, kCvtThreads, ok)) break;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int item = ct + kCvtThreads * j;
        const int nl = item >> 3, q = item & 7;
        const int r = nl & 7, i = nl >> 3;       // row in atom, K atom
        const int ja = q >> 2;                   // MN atom (64 k)
        const int c0 = (q & 3) * 2;              // 16-byte chunk in the 128-byte row
        uint4 o0, o1;
        i8x4_scale_to_h4(v[j].x, f[j], o0.x, o0.y);
        i8x4_scale_to_h4(v[j].y, f[j], o0.z, o0.w);
        i8x4_scale_to_h4(v[j].z, f[j], o1.x, o1.y);
        i8x4_scale_to_h4(v[j].w, f[j], o1.z, o1.w);
        uint8_t* rowp = sa + i * 2048 + ja * 1024 + r * 128;
        *reinterpret_cast<uint4*>(rowp + ((c0 ^ r) << 4)) = o0;
        *reinterpret_cast<uint4*>(rowp + (((c0 + 1) ^ r) << 4)) = o1;
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars->cvt_full[s]);
    }
  } else {
    // ---- epilogue: lane = output feature k, columns = tokens m
    const int quad = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    bool ok = NB > 0 && __all_sync(0xffffffffu, mbar_wait(&bars->acc_full, 0, abort_flag, e.st, kWhereEpi));
    if (ok) tc_fence_after();
    const int64_t kk = k0 + quad * 32 + lane;
#pragma unroll 1
    for (int gcol = 0; gcol < 8; ++gcol) {
      uint32_t x[32];
      if (ok) {
        tmem_ld32(tmem + lane_off + gcol * 32, x);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = 0;
      }
      if (NB > 0 && !ok) break;
      if (kk >= e.K) continue;
      const int mb = m0 + gcol * 32;
      switch (e.dt) {
        case DT_F16: bwd_store<__half>(e, kk, mb, x); break;
        case DT_BF16: bwd_store<__nv_bfloat16>(e, kk, mb, x); break;
        default: bwd_store<float>(e, kk, mb, x); break;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMMA) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace

cudaError_t launch_fwd_gemm(const FwdGemmArgs& g, const FwdEpiArgs& e, cudaStream_t s) {
  const int num_m = static_cast<int>(ceil_div(e.M, kFwdBM));
  const int num_n = static_cast<int>(ceil_div(e.N, kFwdBN));
  if (num_m == 0 || num_n == 0) return cudaSuccess;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t err = cudaFuncSetAttribute(fwd_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (err != cudaSuccess) return err;
    attr_set = true;
  }
  const int group = std::min(num_m, 16);
  ProfScope ps(K_FWD_GEMM, s);
  fwd_gemm_kernel<<<num_m * num_n, kThreads, kSmemBytes, s>>>(g, e, num_m, num_n, group);
  return cudaGetLastError();
}

cudaError_t launch_bwd_gemm(const BwdGemmArgs& g, const BwdEpiArgs& e, cudaStream_t s) {
  const int num_k = static_cast<int>(ceil_div(e.K, kBwdBM));
  const int num_m = static_cast<int>(ceil_div(e.M, kBwdBN));
  if (num_k == 0 || num_m == 0) return cudaSuccess;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t err = cudaFuncSetAttribute(bwd_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (err != cudaSuccess) return err;
    attr_set = true;
  }
  const int group = std::min(num_m, 8);
  ProfScope ps(K_BWD_GEMM, s);
  bwd_gemm_kernel<<<num_k * num_m, kThreads, kSmemBytes, s>>>(g, e, num_k, num_m, group);
  return cudaGetLastError();
}

}  // namespace i8lt
