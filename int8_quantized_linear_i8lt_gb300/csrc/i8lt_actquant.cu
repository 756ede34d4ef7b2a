// Fused activation quantization of the forward (K2 + K3 in one launch):
// outlier-column detection and row-wise (vector-wise) absmax int8
// quantization of a 16-bit activation A [M, K] (bitsandbytes PR #33 "Memory
// efficient backward": the double_quant of the cast fp16 input with its
// coo_tensorA of outlier columns, and the "Mixed-precision decomposition
// matmul" review thread for the outlier rule).
//
// One persistent launch (cooperative when it computes the column maxima).
// Block b owns the contiguous rows [M b / nb, M (b + 1) / nb); thread t owns
// the 8-column groups t + i NT (i < G) of every row, so that it keeps the same
// columns through all phases.  Rows stream through a ring of shared-memory
// buffers filled by bulk copies, several rows ahead, and every thread copies
// its groups of a row into registers once.
//   phase 1  column maxima of |fp16(A)| over the block's rows, in registers as
//            packed 16-bit magnitudes (fp16 magnitudes order as integers);
//            then a two-level reduction that never has two blocks reducing
//            into one address at once: each block stores its partial maxima
//            as one row of a scratch (the code region, written only in phase
//            3), a bounded grid-wide wait, block b reduces the columns of its
//            slice over all partial rows in shared memory and stores the final
//            maxima, a second bounded grid-wide wait (every block resident by
//            the cooperative launch; a wait that runs out records ST_TIMEOUT);
//   phase 2  every block reads the column maxima of its columns and derives
//            the outlier mask (max > threshold, strictly) and, by an ordered
//            block scan over (i, t) -- column order --, the ascending position
//            of each outlier column in subA; block 0 also writes the global
//            mask, idx and outlier counts for the later kernels;
//   phase 3  the block's rows in reverse order (the rows phase 1 read last are
//            the likeliest to be still in L2): the absmax outside the outlier
//            columns reduced over the block, then the codes rint(fp32(A16) *
//            (127 / absmax)) (IEEE fp32 divide and multiply, round half to
//            even) as exact fp16 integers with the outlier columns at 0,
//            written over the row's own ring buffer and sent to global memory
//            by one bulk store per row; the outlier columns' fp16 values go to
//            subA; the per-1024-column sums of squared codes raise the row
//            tile's asq entries.
// The same arithmetic as colmax_kernel + outlier_index_kernel +
// row_quantize_bulk_kernel (i8lt_quant.cu), so the results are bit-identical.
// Used for 16-bit A with K a multiple of 8 up to 32768 (16-byte rows that fit
// the ring); the other inputs take the separate kernels.
#include <algorithm>
#include <cstring>
#include <type_traits>

#include "i8lt_internal.h"

namespace i8lt {

namespace {

constexpr int kWhereActQuant = 7;   // status `where` of a timed-out grid-wide wait

struct ActQuantArgs {
  const void* A;         // [M, K] fp16 or bf16, K % 8 == 0, 16-byte aligned
  int64_t M;
  int K, k_pad;          // k_pad = round_up(K, 16): the leading dimension of Aq
  float thr;             // outlier threshold (used when `enabled`)
  int enabled;           // outlier decomposition on
  int do_colmax;         // phase 1: the column maxima of A's rows into colmax (zeroed)
  int64_t cap, cap_pad;  // outlier capacity and the leading dimension of subA
  int nch;               // 1024-column chunks of a code row (asq's second dimension)
  uint32_t* colmax;      // [K]
  uint32_t* mask;        // [ceil(K / 32)]
  int* idx;              // [cap_pad]
  DevStatus* st;
  unsigned* arrive;      // grid-wide wait counter (zeroed)
  float* SCA;            // [M]
  void* Aq;              // [M, k_pad] codes: exact fp16 integers (activations) or int8 (weights)
  __half* subA;          // [M, cap_pad]
  uint32_t* asq;         // [ceil(M / 256), nch]
  int nbuf;              // rows in the shared-memory ring
};

// 8 elements (16 bytes) as fp16 values in a uint4; bf16 cast to fp16 (RNE).
template <typename T>
__device__ __forceinline__ uint4 to_half8(uint4 v) {
  if constexpr (std::is_same<T, __half>::value) {
    return v;
  } else {
    const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(&v);
    uint4 o;
    __half* h = reinterpret_cast<__half*>(&o);
#pragma unroll
    for (int j = 0; j < 8; ++j) h[j] = to_half(b[j]);
    return o;
  }
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Every block of the grid arrives once per wait; returns false (after
// recording ST_TIMEOUT) when the counter has not reached `target` (the
// blocks times the waits so far) within the time limit.
__device__ bool grid_wait(unsigned* arrive, unsigned target, DevStatus* st,
                          unsigned long long limit_ns = kWaitTimeoutNs) {
  __shared__ int ok_s;
  __threadfence();   // this thread's column-maxima reductions, before the arrival
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(arrive, 1u);
    int ok = 1;
    const unsigned long long t0 = global_ns();
    while (ld_acquire_gpu(arrive) < target) {
      __nanosleep(256);
      if (global_ns() - t0 > limit_ns) {
        set_status(st, ST_TIMEOUT, kWhereActQuant);
        ok = 0;
        break;
      }
    }
    __threadfence();
    ok_s = ok;
  }
  __syncthreads();
  return ok_s != 0;
}

// Exclusive prefix sum of v over the block (threads in order) and the total.
__device__ __forceinline__ int block_exclusive_scan(int v, int& total, int* warp_s) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_s[w] = incl;
  __syncthreads();
  if (w == 0) {
    int x = lane < nw ? warp_s[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane < nw) warp_s[lane] = x;   // inclusive over warps
  }
  __syncthreads();
  const int before = w > 0 ? warp_s[w - 1] : 0;
  total = warp_s[nw - 1];
  __syncthreads();   // warp_s is reused by the next scan
  return before + incl - v;
}

// Sums x[i] over the warp for every i < G (G a power of two, 2..32) with
// G - 1 + log2(32 / G) shuffles instead of G * 5: each halving step
// exchanges half of the remaining values with the lane `o` apart, the lane
// with bit o clear keeping the lower half.  Returns, at lane l, the warp sum
// of x[l / (32 / G)].
template <int G>
__device__ __forceinline__ int warp_transpose_sum(int (&x)[G], int lane) {
#pragma unroll
  for (int n = G, o = 16; n > 1; n >>= 1, o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int j = 0; j < n / 2; ++j) {
      const int send = up ? x[j] : x[j + n / 2];
      const int keep = up ? x[j + n / 2] : x[j];
      x[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  int y = x[0];
#pragma unroll
  for (int o = 16 / G; o > 0; o >>= 1) y += __shfl_xor_sync(0xffffffffu, y, o);
  return y;
}

constexpr int kMaxBufs = 8;   // rows in the shared-memory ring

template <typename T, typename CodeT, int G, int NT, int MINB>
__global__ void __launch_bounds__(NT, MINB) act_quant_fused_kernel(const ActQuantArgs a) {
  // int8 codes: the weight quantization (no column maxima, no outliers, no
  // sums of squared codes); fp16 codes: the activations
  constexpr bool kI8 = std::is_same<CodeT, int8_t>::value;
  extern __shared__ __align__(128) uint8_t ring[];   // a.nbuf row buffers of K 16-bit elements
  __shared__ __align__(8) uint64_t full[kMaxBufs];
  __shared__ int abort_flag;
  __shared__ float red_s[2][32];
  __shared__ int chunk_s[2][64];
  __shared__ int warp_s[32];
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  constexpr int kWarps = NT / 32;
  const int ng = a.K / 8;            // 8-column groups holding data
  const int ng_pad = a.k_pad / 8;    // groups of a code row (with the zero padding)
  const int64_t r0 = a.M * blockIdx.x / gridDim.x, r1 = a.M * (blockIdx.x + 1) / gridDim.x;
  const int64_t nrows = r1 - r0;
  const T* A = static_cast<const T*>(a.A);
  const uint32_t row_bytes = static_cast<uint32_t>(a.K) * 2u;     // one input row
  const uint32_t buf_bytes = static_cast<uint32_t>(a.k_pad) * 2u; // one ring buffer: a row of fp16 codes
  const int nbuf = a.nbuf;
  volatile int* abort_p = &abort_flag;
  if (t == 0) {
    for (int b = 0; b < nbuf; ++b) mbar_init(&full[b], 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (t < 64) {
    chunk_s[0][t] = 0;
    chunk_s[1][t] = 0;
  }
  __syncthreads();

  // Rows stream through the ring of shared-memory buffers by bulk copies
  // (thread 0 issues them, nbuf rows ahead); the u-th row streamed by this
  // block goes to buffer u % nbuf.  Phase 1 streams rows r0, r0 + 1, ...,
  // phase 3 rows r1 - 1, r1 - 2, ... (u keeps counting across the phases).
  auto issue = [&](int64_t u, int64_t r) {
    const int b = static_cast<int>(u % nbuf);
    fence_proxy_async_smem();   // the buffer's last readers are past a block barrier
    mbar_arrive_expect_tx(&full[b], row_bytes);
    bulk_load(ring + static_cast<size_t>(b) * buf_bytes, A + r * a.K, row_bytes, &full[b]);
  };
  // wait for stream row u and copy this thread's groups of it into registers
  auto fetch = [&](int64_t u, uint4 (&v)[G]) -> bool {
    const int b = static_cast<int>(u % nbuf);
    const bool ok = mbar_wait(&full[b], static_cast<uint32_t>((u / nbuf) & 1), abort_p, a.st, kWhereActQuant);
    const uint4* src = reinterpret_cast<const uint4*>(ring + static_cast<size_t>(b) * buf_bytes);
#pragma unroll
    for (int i = 0; i < G; ++i) {
      const int gi = t + i * NT;
      v[i] = gi < ng ? to_half8<T>(src[gi]) : make_uint4(0u, 0u, 0u, 0u);
    }
    return ok;
  };
  // after a timeout at stream row u_fail: let the copies issued and not yet
  // consumed (rows u_fail .. u_issued - 1) land, each wait bounded, and the
  // bulk stores in flight finish, before the block leaves
  auto drain = [&](int64_t u_fail, int64_t u_issued) {
    if (t == 0) {
      *abort_p = 0;
      for (int64_t v = u_fail; v < u_issued; ++v)
        mbar_wait(&full[v % nbuf], static_cast<uint32_t>((v / nbuf) & 1), abort_p, nullptr, 0);
      bulk_wait_all();   // code rows still being stored from shared memory
    }
  };
  int64_t u = 0;   // rows streamed so far

  // ---- phase 1: column maxima of this block's rows
  if (a.do_colmax) {
    uint32_t cm[G][4];
#pragma unroll
    for (int i = 0; i < G; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) cm[i][j] = 0u;
    if (t == 0)
      for (int64_t k = 0; k < nrows && k < nbuf; ++k) issue(u + k, r0 + k);
    for (int64_t k = 0; k < nrows; ++k) {
      uint4 h[G];
      const bool ok = fetch(u + k, h);
      if (!__syncthreads_and(ok)) {   // every thread read its groups: the buffer is free
        drain(u + k, u + std::min<int64_t>(nrows, k + nbuf));
        return;
      }
      if (t == 0 && k + nbuf < nrows) issue(u + k + nbuf, r0 + k + nbuf);
#pragma unroll
      for (int i = 0; i < G; ++i) {
        cm[i][0] = __vmaxu2(cm[i][0], h[i].x & 0x7FFF7FFFu);
        cm[i][1] = __vmaxu2(cm[i][1], h[i].y & 0x7FFF7FFFu);
        cm[i][2] = __vmaxu2(cm[i][2], h[i].z & 0x7FFF7FFFu);
        cm[i][3] = __vmaxu2(cm[i][3], h[i].w & 0x7FFF7FFFu);
      }
    }
    u += nrows;
    // Two-level reduction, with no two blocks reducing into one address at
    // once: every block stores its partial maxima (8 packed 16-bit values a
    // group) as row b of a scratch in the Aq region (written only in phase
    // 3); after the wait, block b reduces the groups [g0, g1) over all the
    // partial rows in shared memory and stores the final column maxima.
    uint4* part = reinterpret_cast<uint4*>(a.Aq);   // [gridDim.x, ng]: M * k_pad >= gridDim.x * K
#pragma unroll
    for (int i = 0; i < G; ++i) {
      const int gi = t + i * NT;
      if (gi < ng) part[static_cast<int64_t>(blockIdx.x) * ng + gi] = make_uint4(cm[i][0], cm[i][1], cm[i][2], cm[i][3]);
    }
    if (!grid_wait(a.arrive, gridDim.x, a.st)) return;
    const int g0 = static_cast<int>(static_cast<int64_t>(ng) * blockIdx.x / gridDim.x);
    const int g1 = static_cast<int>(static_cast<int64_t>(ng) * (blockIdx.x + 1) / gridDim.x);
    const int S = g1 - g0;
    uint32_t* colm_s = reinterpret_cast<uint32_t*>(ring);   // 8 S values (the ring holds >= 3 K halves)
    for (int x = t; x < 8 * S; x += NT) colm_s[x] = 0u;
    __syncthreads();
    const int nparts = static_cast<int>(gridDim.x);
    for (int x = t; x < S * nparts; x += NT) {
      const int p = x / S, gl = x - p * S;
      const uint4 v = __ldcg(part + static_cast<int64_t>(p) * ng + g0 + gl);
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t m = (w4[j >> 1] >> (16 * (j & 1))) & 0xFFFFu;
        if (m != 0u) atomicMax(colm_s + 8 * gl + j, m);
      }
    }
    __syncthreads();
    for (int x = t; x < 8 * S; x += NT) a.colmax[8 * g0 + x] = colm_s[x];
    if (!grid_wait(a.arrive, 2 * gridDim.x, a.st)) return;
  }

  // ---- phase 2: the outlier columns among this thread's columns and their
  // ascending positions in subA (the same in every block)
  uint32_t mb[G];   // bit j: column 8 gi + j is an outlier
  int jb[G];        // position in subA of the first outlier column of group i
  int used = 0;
#pragma unroll
  for (int i = 0; i < G; ++i) {
    mb[i] = 0u;
    jb[i] = 0;
  }
  if (a.enabled) {
#pragma unroll
    for (int i = 0; i < G; ++i) {
      const int gi = t + i * NT;
      if (gi < ng) {
        const uint4 c0 = __ldcg(reinterpret_cast<const uint4*>(a.colmax + 8 * gi));
        const uint4 c1 = __ldcg(reinterpret_cast<const uint4*>(a.colmax + 8 * gi) + 1);
        const uint32_t cv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (__half2float(__ushort_as_half(static_cast<unsigned short>(cv[j]))) > a.thr) mb[i] |= 1u << j;
      }
    }
    int base = 0;
#pragma unroll
    for (int i = 0; i < G; ++i) {   // column order: group i of every thread, then group i + 1
      int total;
      jb[i] = base + block_exclusive_scan(__popc(mb[i]), total, warp_s);
      base += total;
    }
    used = static_cast<int>(min(static_cast<int64_t>(base), a.cap));
    if (blockIdx.x == 0) {
#pragma unroll
      for (int i = 0; i < G; ++i) {
        const int gi = t + i * NT;
        // four consecutive groups make one 32-bit mask word (NT % 4 == 0)
        const uint32_t m1 = __shfl_down_sync(0xffffffffu, mb[i], 1);
        const uint32_t m2 = __shfl_down_sync(0xffffffffu, mb[i], 2);
        const uint32_t m3 = __shfl_down_sync(0xffffffffu, mb[i], 3);
        if ((t & 3) == 0 && gi < ng) a.mask[gi >> 2] = mb[i] | (m1 << 8) | (m2 << 16) | (m3 << 24);
        int j = jb[i];
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          if ((mb[i] >> b) & 1u) {
            if (j < a.cap) a.idx[j] = 8 * gi + b;
            ++j;
          }
        }
      }
      if (t == 0) {
        a.st->found = base;
        a.st->used = used;
        if (base > a.cap) set_status(a.st, ST_OUTLIER_CAPACITY, 0);
      }
    }
  }
  const int used_pad = (used + 63) / 64 * 64;

  // ---- phase 3: the rows in reverse order (those phase 1 read last first).
  // A row's codes are written over its own ring buffer (each thread over the
  // groups it read) and leave as one bulk store, issued after the next row's
  // barrier; the buffer is refilled once that store has read it, so a buffer
  // goes: loaded -> read -> codes -> stored -> loaded, nbuf - 2 rows ahead.
  // (Refilling the buffer of row k - 2 instead, with more lookahead for the
  // store, made the 8192-column rows 30 % slower.)
  int64_t issued = std::min<int64_t>(nrows, nbuf);   // stream rows issued (uniform over the block)
  if (t == 0)
    for (int64_t k = 0; k < issued; ++k) issue(u + k, r1 - 1 - k);
  auto slot = [&](int64_t v) { return ring + static_cast<size_t>(v % nbuf) * buf_bytes; };
  const uint32_t code_bytes = static_cast<uint32_t>(a.k_pad) * sizeof(CodeT);   // a row of codes
  auto code_row = [&](int64_t r) { return static_cast<uint8_t*>(a.Aq) + r * code_bytes; };
  constexpr int kSpan = 32 / G;   // lanes that end up holding one group's warp sum (warp_transpose_sum)
  int par = 0;
  int64_t prev = -1;
  for (int64_t k = 0; k < nrows; ++k, par ^= 1) {
    const int64_t r = r1 - 1 - k;
    uint4 h[G];
    const bool ok = fetch(u + k, h);
    // the row's absmax outside the outlier columns: packed fp16 maxima of
    // magnitudes (exact) for groups without outlier columns
    __half2 m2 = __float2half2_rn(0.f);
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < G; ++i) {
      if (mb[i] == 0u) {
        const __half2* x2 = reinterpret_cast<const __half2*>(&h[i]);
#pragma unroll
        for (int j = 0; j < 4; ++j) m2 = __hmax2(m2, __habs2(x2[j]));
      } else {
        const __half* x = reinterpret_cast<const __half*>(&h[i]);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (!((mb[i] >> j) & 1u)) amax = fmaxf(amax, fabsf(__half2float(x[j])));
      }
    }
    amax = fmaxf(amax, fmaxf(__low2float(m2), __high2float(m2)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) red_s[par][w] = amax;
    // every thread has read its groups of this row and published its warp
    // maximum, and has written and fenced its codes of the previous row
    if (!__syncthreads_and(ok)) {
      drain(u + k, u + issued);
      return;
    }
    if (t == 0 && prev >= 0) {
      bulk_store(code_row(prev), slot(u + k - 1), code_bytes);
      bulk_commit();
    }
    // the previous row's chunk sums are complete: raise its tile's asq entries
    if (!kI8 && prev >= 0 && t < a.nch) {
      const int v = chunk_s[par ^ 1][t];
      if (v != 0) atomicMax(a.asq + (prev >> 8) * a.nch + t, static_cast<uint32_t>(v));
      chunk_s[par ^ 1][t] = 0;
    }
    amax = lane < kWarps ? red_s[par][lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = (amax > 0.f) ? __fdiv_rn(127.0f, amax) : 0.f;
    uint8_t* cbuf = slot(u + k);
    int sqi[G];
#pragma unroll
    for (int i = 0; i < G; ++i) {
      const int gi = t + i * NT;
      const __half* x = reinterpret_cast<const __half*>(&h[i]);
      // q = rint(x * s), round half to even by the exact add of 1.5 * 2^23;
      // |x| <= absmax outside the outlier columns, so |x * s| <= 127 (1 +
      // 2^-23) and no clamp is needed
      float q[8];
      float sq = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        q[j] = __fsub_rn(__fadd_rn(__fmul_rn(__half2float(x[j]), s), 12582912.0f), 12582912.0f);
        if (!kI8) sq = __fmaf_rn(q[j], q[j], sq);
      }
      if (mb[i] != 0u) {
        sq = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if ((mb[i] >> j) & 1u) q[j] = 0.f;
          sq = __fmaf_rn(q[j], q[j], sq);
        }
      }
      if (gi < ng_pad) {
        if constexpr (kI8) {   // 8 bytes: the codes as int8, element j in byte j
          uint32_t wd[2] = {0u, 0u};
#pragma unroll
          for (int j = 0; j < 8; ++j)
            wd[j >> 2] |= (static_cast<uint32_t>(static_cast<int>(q[j])) & 0xFFu) << (8 * (j & 3));
          *reinterpret_cast<uint2*>(cbuf + 8 * gi) = make_uint2(wd[0], wd[1]);
        } else {
          uint4 o;
          __half2* o2 = reinterpret_cast<__half2*>(&o);
#pragma unroll
          for (int j = 0; j < 4; ++j) o2[j] = __floats2half2_rn(q[2 * j], q[2 * j + 1]);
          st_shared_v4(cbuf + 16 * gi, o);
        }
      }
      sqi[i] = static_cast<int>(sq);
      if (mb[i] != 0u) {   // rare: the outlier columns of the group, in column order
        int j = jb[i];
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          if ((mb[i] >> b) & 1u) {
            if (j < a.cap) a.subA[r * a.cap_pad + j] = x[b];
            ++j;
          }
        }
      }
    }
    // the warp's sums of the G groups at once; group i of this warp lies in
    // the 1024-column chunk (32 w + i NT) / 128 (NT % 128 == 0)
    if constexpr (!kI8) {
      const int tot = warp_transpose_sum<G>(sqi, lane);
      if ((lane & (kSpan - 1)) == 0 && tot != 0) atomicAdd(&chunk_s[par][(32 * w + (lane / kSpan) * NT) >> 7], tot);
    }
    for (int j = used + t; j < used_pad; j += NT) a.subA[r * a.cap_pad + j] = __float2half_rn(0.f);
    if (t == 0) a.SCA[r] = amax;
    fence_proxy_async_smem();   // this thread's codes, for the bulk store
    // the buffer of the previous row: refill it once its store has read it
    if (k >= 1) {
      if (t == 0 && k - 1 + nbuf < nrows) {
        bulk_wait_read<0>();
        issue(u + k - 1 + nbuf, r1 - 1 - (k - 1 + nbuf));
      }
      issued = std::min<int64_t>(nrows, k + nbuf);
    }
    prev = r;
  }
  __syncthreads();   // the last row's codes are written and fenced; its chunk sums are complete
  if (t == 0) {
    if (prev >= 0) {
      bulk_store(code_row(prev), slot(u + nrows - 1), code_bytes);
      bulk_commit();
    }
    bulk_wait_all();
  }
  if (!kI8 && prev >= 0 && t < a.nch) {
    const int v = chunk_s[par ^ 1][t];
    if (v != 0) atomicMax(a.asq + (prev >> 8) * a.nch + t, static_cast<uint32_t>(v));
  }
}

// Blocks of NT threads, G groups each, MINB blocks per SM: a configuration
// that covers the row (256 x 2 groups up to 4096 columns and 256 x 4 up to
// 8192, four blocks per SM, when there are rows enough -- else 256 x 2 and
// 512 x 2, two; 256 x 8 up to 16384, two; else 1024 x 4, one).  More
// resident blocks hide each block's per-row barrier and bulk-copy waits
// behind the others' work.  The ring takes what shared memory the blocks of
// an SM leave, 3 to kMaxBufs rows.
constexpr int kRingBudget = 200 * 1024;

template <typename T, typename CodeT, int G, int NT, int MINB>
cudaError_t launch_cfg(ActQuantArgs a, bool cooperative, int sms, cudaStream_t s) {
  const void* fn = reinterpret_cast<const void*>(act_quant_fused_kernel<T, CodeT, G, NT, MINB>);
  const int target = MINB;
  const int64_t buf_bytes = static_cast<int64_t>(a.k_pad) * 2;   // a row of fp16 codes
  a.nbuf = static_cast<int>(std::max<int64_t>(3, std::min<int64_t>(kMaxBufs, kRingBudget / target / buf_bytes)));
  const int smem = static_cast<int>(a.nbuf * buf_bytes);
  if (!ensure_smem_attr(fn, kRingBudget)) return cudaGetLastError();
  const int per_sm = std::max(1, std::min(cached_blocks_per_sm(fn, NT, smem), target));
  const int nb = static_cast<int>(std::min<int64_t>(a.M, static_cast<int64_t>(sms) * per_sm));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(nb), 1, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = cooperative ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, act_quant_fused_kernel<T, CodeT, G, NT, MINB>, a);
}

template <typename T, typename CodeT>
cudaError_t launch_typed(const ActQuantArgs& a, bool cooperative, int sms, cudaStream_t s) {
  const int groups = a.k_pad / 8;
  // four blocks per SM only when every block still gets a few dozen rows
  // (with 2048 rows of 4096 columns they made the launch 24 % slower)
  const bool many_rows = a.M >= 32LL * sms;
  if (groups <= 256 * 2)
    return many_rows ? launch_cfg<T, CodeT, 2, 256, 4>(a, cooperative, sms, s) : launch_cfg<T, CodeT, 2, 256, 2>(a, cooperative, sms, s);
  if (groups <= 512 * 2)
    return many_rows ? launch_cfg<T, CodeT, 4, 256, 4>(a, cooperative, sms, s) : launch_cfg<T, CodeT, 2, 512, 2>(a, cooperative, sms, s);
  if (groups <= 256 * 8) return launch_cfg<T, CodeT, 8, 256, 2>(a, cooperative, sms, s);
  return launch_cfg<T, CodeT, 4, 1024, 1>(a, cooperative, sms, s);
}

// The failure path of the grid-wide wait without a fault: every block
// waits for one arrival more than the grid makes, so each one runs out of
// time, records ST_TIMEOUT and returns.
__global__ void grid_wait_probe_kernel(unsigned* arrive, DevStatus* st, unsigned long long limit_ns) {
  grid_wait(arrive, gridDim.x + 1, st, limit_ns);
}

}  // namespace

cudaError_t launch_grid_wait_probe(DevStatus* st, unsigned* arrive, unsigned long long limit_ns, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(32, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, grid_wait_probe_kernel, arrive, st, limit_ns);
}

// Rows up to 32768 columns (one block of 1024 threads, 4 groups of 8 each);
// longer rows take the separate kernels.
bool act_quant_fused_supported(int at, int64_t K) {
  return (at == DT_F16 || at == DT_BF16) && K > 0 && K % 8 == 0 && round_up(K, 16) <= 1024 * 4 * 8;
}

cudaError_t launch_act_quant_fused(const void* A, int at, int64_t M, int64_t K, int64_t k_pad, bool enabled,
                                   float thr, bool do_colmax, int64_t cap, int64_t cap_pad, uint32_t* colmax,
                                   uint32_t* mask, int* idx, DevStatus* st, unsigned* arrive, float* SCA,
                                   __half* Aq, __half* subA, uint32_t* asq, cudaStream_t s) {
  if (M == 0) return cudaSuccess;
  ActQuantArgs a;
  a.A = A;
  a.M = M;
  a.K = static_cast<int>(K);
  a.k_pad = static_cast<int>(k_pad);
  a.thr = thr;
  a.enabled = enabled ? 1 : 0;
  a.do_colmax = do_colmax ? 1 : 0;
  a.cap = cap;
  a.cap_pad = cap_pad;
  a.nch = static_cast<int>(ceil_div(k_pad, 1024));
  a.colmax = colmax;
  a.mask = mask;
  a.idx = idx;
  a.st = st;
  a.arrive = arrive;
  a.SCA = SCA;
  a.Aq = Aq;
  a.subA = subA;
  a.asq = asq;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const bool cooperative = do_colmax;   // the grid-wide waits need every block resident
  ProfScope ps(K_ROW_QUANTIZE, s);
  return at == DT_BF16 ? launch_typed<__nv_bfloat16, __half>(a, cooperative, sms, s)
                       : launch_typed<__half, __half>(a, cooperative, sms, s);
}


// The weight quantization through the same kernel: W [N, K] (16-bit, K % 8
// == 0, k_pad <= 32768) -> SCB[n] = max_k |fp16(W[n, k])| and CB [N, k_pad]
// int8 codes rint(fp32(W16) * (127 / SCB[n])), zero in the padding -- the
// row pass alone (no column maxima, no outliers), each code row stored in
// bulk from its ring buffer.
cudaError_t launch_quantize_weight_fused(const void* W, int wt, int64_t N, int64_t K, int64_t k_pad, int8_t* CB,
                                         float* SCB, cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  ActQuantArgs a;
  std::memset(&a, 0, sizeof(a));
  a.A = W;
  a.M = N;
  a.K = static_cast<int>(K);
  a.k_pad = static_cast<int>(k_pad);
  a.nch = static_cast<int>(ceil_div(k_pad, 1024));
  a.SCA = SCB;
  a.Aq = CB;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  ProfScope ps(K_QUANTIZE_WEIGHT, s);
  return wt == DT_BF16 ? launch_typed<__nv_bfloat16, int8_t>(a, false, sms, s)
                       : launch_typed<__half, int8_t>(a, false, sms, s);
}

}  // namespace i8lt
