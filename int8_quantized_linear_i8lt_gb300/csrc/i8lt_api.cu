// C ABI of libi8lt: argument checks, workspace layout, TMA descriptors and
// the launch sequence of the forward and backward of the int8 quantized
// linear layer (bitsandbytes PR #33 "Memory efficient backward").
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "i8lt.h"
#include "i8lt_internal.h"

using namespace i8lt;

namespace {

constexpr int kAbiVersion = 4;
constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool valid_dt(int dt) { return dt == DT_F16 || dt == DT_BF16 || dt == DT_F32; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool threshold_enabled(float t) { return std::isfinite(t) && t > 0.0f; }

int64_t cap_pad_of(int64_t cap) { return cap > 0 ? round_up(cap, 64) : 0; }

// Device check: the kernels are built for sm_103a only.
int check_device() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return I8LT_ERR_CUDA;
  if (dev < 0 || dev >= 64) return I8LT_ERR_DEVICE;
  int c = cached[dev].load();
  if (c == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return I8LT_ERR_CUDA;
    c = (major == 10 && minor == 3) ? 1 : 2;
    cached[dev].store(c);
  }
  return c == 1 ? I8LT_OK : I8LT_ERR_DEVICE;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D row-major tensor (inner x outer elements, row pitch in bytes) with a
// box of box_inner x box_outer elements.
bool make_tmap(CUtensorMap* tm, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
               uint64_t pitch, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(tm, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? I8LT_OK : I8LT_ERR_CUDA; }

i8lt_fwd_layout fwd_layout(int64_t M, int64_t K, int64_t N, int64_t cap) {
  i8lt_fwd_layout L;
  std::memset(&L, 0, sizeof(L));
  L.k_pad = round_up(K, 16);
  L.cap_pad = cap_pad_of(cap < K ? cap : K);
  const int64_t nch = ceil_div(L.k_pad, 1024);
  size_t off = 0;
  L.status = off;
  off += kAlign;
  L.asq = off;
  off += align_up(static_cast<size_t>(ceil_div(M, 256)) * nch * 4);
  L.bsq = off;
  off += align_up(static_cast<size_t>(ceil_div(N, 256)) * nch * 4);
  L.colmax = off;
  off += align_up(static_cast<size_t>(K) * 4);
  L.mask = off;
  off += align_up(static_cast<size_t>(ceil_div(K, 32)) * 4);
  L.idx = off;
  off += align_up(static_cast<size_t>(L.cap_pad) * 4);
  L.sca = off;
  off += align_up(static_cast<size_t>(M) * 4);
  L.plan = off;
  off += align_up(static_cast<size_t>(ceil_div(M, 256)) * ceil_div(N, 256) * 4);
  L.aq = off;
  off += align_up(static_cast<size_t>(M) * L.k_pad * 2);
  L.suba = off;
  off += align_up(static_cast<size_t>(M) * L.cap_pad * 2);
  L.subb = off;
  off += align_up(static_cast<size_t>(N) * L.cap_pad * 2);
  L.cbh = off;
  off += align_up(static_cast<size_t>(N) * L.k_pad * 2);
  L.total = off;
  return L;
}

bool needs_g16(int64_t N, int gt) { return gt != DT_F16 || (N % 8) != 0; }

// Backward workspace: [status][grad_bias partial sums][G16 when needed]
// = the fused schedule's minimum (`total`), then [WdqT, K_pad x N_pad fp16]
// for the materialized schedule (`total_dq`).
struct BwdLayout {
  size_t status, partial, g16, total, wdq, total_dq;
  int64_t n_pad, chunks;
};

BwdLayout bwd_layout(int64_t M, int64_t N, int64_t K, int gt) {
  BwdLayout L;
  L.n_pad = round_up(N, 8);
  L.chunks = gradout_partial_chunks(M);
  size_t off = 0;
  L.status = off;
  off += kAlign;
  L.partial = off;
  off += align_up(static_cast<size_t>(L.chunks) * N * 4);
  L.g16 = off;
  if (needs_g16(N, gt)) off += align_up(static_cast<size_t>(M) * L.n_pad * 2);
  L.total = off;
  L.wdq = off;
  off += align_up(static_cast<size_t>(round_up(K, 16)) * L.n_pad * 2);
  L.total_dq = off;
  return L;
}

// Weight-gradient workspace (trainable-weight mode):
// [status][colmax G, N][colmax A, K][scale G, N][scale A, K]
// [tile chunk maxima G, A][chunk sums G, N x chunks][chunk sums A, K x chunks]
// [plan][Gt fp16, N x R_pad][At fp16, K x R_pad], R_pad = M rounded up to 16
// (the reduction dimension of the GEMM).
struct WgradLayout {
  size_t status, colmax_g, colmax_a, scale_g, scale_a, tsq_g, tsq_a, sq_g, sq_a, plan, gt, at, total;
  int64_t r_pad, chunks;
};

WgradLayout wgrad_layout(int64_t M, int64_t N, int64_t K) {
  WgradLayout L;
  L.r_pad = round_up(M, 16);
  L.chunks = ceil_div(L.r_pad, 1024);
  size_t off = 0;
  L.status = off;
  off += kAlign;
  L.colmax_g = off;
  off += align_up(static_cast<size_t>(N) * 4);
  L.colmax_a = off;
  off += align_up(static_cast<size_t>(K) * 4);
  L.scale_g = off;
  off += align_up(static_cast<size_t>(N) * 4);
  L.scale_a = off;
  off += align_up(static_cast<size_t>(K) * 4);
  L.tsq_g = off;
  off += align_up(static_cast<size_t>(ceil_div(N, 256)) * L.chunks * 4);
  L.tsq_a = off;
  off += align_up(static_cast<size_t>(ceil_div(K, 256)) * L.chunks * 4);
  L.sq_g = off;
  off += align_up(static_cast<size_t>(N) * L.chunks * 4);
  L.sq_a = off;
  off += align_up(static_cast<size_t>(K) * L.chunks * 4);
  L.plan = off;
  off += align_up(static_cast<size_t>(ceil_div(N, 256)) * ceil_div(K, 256) * 4);
  L.gt = off;
  off += align_up(static_cast<size_t>(N) * L.r_pad * 2);
  L.at = off;
  off += align_up(static_cast<size_t>(K) * L.r_pad * 2);
  L.total = off;
  return L;
}

// ---- kernel timing --------------------------------------------------------
struct ProfRec {
  int id;
  cudaEvent_t a, b;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
int g_prof_max = 0;
int g_prof_count = 0;
std::vector<ProfRec> g_prof;
std::vector<cudaEvent_t> g_ev_pool;
int g_ev_next = 0;

cudaEvent_t pool_event() {
  if (g_ev_next == static_cast<int>(g_ev_pool.size())) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    g_ev_pool.push_back(e);
  }
  return g_ev_pool[g_ev_next++];
}

}  // namespace

namespace i8lt {
void prof_begin(int id, cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof_on) return;
  ++g_prof_count;
  if (static_cast<int>(g_prof.size()) >= g_prof_max) return;
  ProfRec r{id, pool_event(), pool_event()};
  if (r.a == nullptr || r.b == nullptr) return;
  cudaEventRecord(r.a, s);
  g_prof.push_back(r);
}
void prof_end(cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof_on || g_prof.empty()) return;
  cudaEventRecord(g_prof.back().b, s);
}
}  // namespace i8lt

namespace {

// The three forms of the forward: the whole call; only the column maxima of
// this call's rows (first half of a token-sharded forward); everything after
// the column maxima, which the caller has merged across the shards.
enum FwdMode { kFwdFull = 0, kFwdColmaxOnly = 1, kFwdFromColmax = 2 };

int forward_impl(FwdMode mode, const void* A, int at, int64_t M, int64_t K, const int8_t* CB, const float* SCB,
                 int64_t N, const void* bias, int bt, float threshold, const void* residual, void* out, void* ws,
                 size_t ws_bytes, int64_t max_outliers, const i8lt_fwd_debug* dbg, void* stream,
                 void* act = nullptr, uint32_t* act_colmax = nullptr) {
  const bool colmax_only = mode == kFwdColmaxOnly;
  if (!valid_dt(at) || (!colmax_only && bias != nullptr && !valid_dt(bt))) return I8LT_ERR_UNSUPPORTED_DTYPE;
  if (M < 0 || N <= 0 || K <= 0 || max_outliers < 0) return I8LT_ERR_INVALID_ARG;
  if (K > I8LT_MAX_K) return I8LT_ERR_K_TOO_LARGE;
  if (M > INT32_MAX / 2 || N > INT32_MAX / 2) return I8LT_ERR_INVALID_ARG;
  if (ws == nullptr || (!colmax_only && (CB == nullptr || SCB == nullptr))) return I8LT_ERR_INVALID_ARG;
  if (M > 0 && (A == nullptr || (!colmax_only && out == nullptr))) return I8LT_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(CB) || !aligned16(out) || !aligned16(residual)) return I8LT_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return I8LT_ERR_MISALIGNED;
  const i8lt_fwd_layout L = fwd_layout(M, K, N, max_outliers);
  if (ws_bytes < L.total) return I8LT_ERR_WORKSPACE;
  if (dbg != nullptr && dbg->acc_i32 != nullptr && !aligned16(dbg->acc_i32)) return I8LT_ERR_MISALIGNED;
  if ((act == nullptr) != (act_colmax == nullptr)) return I8LT_ERR_INVALID_ARG;
  if (!aligned16(act) || (reinterpret_cast<uintptr_t>(act_colmax) & 3u) != 0) return I8LT_ERR_MISALIGNED;
  if (int d = check_device()) return d;
  if (act_colmax != nullptr &&
      cudaMemsetAsync(act_colmax, 0, static_cast<size_t>(N) * 4, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return I8LT_ERR_CUDA;
  if (M == 0 && !colmax_only) return I8LT_OK;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  DevStatus* st = reinterpret_cast<DevStatus*>(w + L.status);
  uint32_t* colmax = reinterpret_cast<uint32_t*>(w + L.colmax);
  uint32_t* mask = reinterpret_cast<uint32_t*>(w + L.mask);
  int* idx = reinterpret_cast<int*>(w + L.idx);
  float* SCA = reinterpret_cast<float*>(w + L.sca);
  uint32_t* asq = reinterpret_cast<uint32_t*>(w + L.asq);
  uint32_t* bsq = reinterpret_cast<uint32_t*>(w + L.bsq);
  uint32_t* plan = reinterpret_cast<uint32_t*>(w + L.plan);
  __half* Aq = reinterpret_cast<__half*>(w + L.aq);
  __half* subA = reinterpret_cast<__half*>(w + L.suba);
  __half* subB = reinterpret_cast<__half*>(w + L.subb);
  __half* CBh = reinterpret_cast<__half*>(w + L.cbh);
  const bool enabled = threshold_enabled(threshold);
  const bool vec = (K % 8) == 0;

  // one memset clears the status word of this call (with the grid-wide wait
  // counter after it), the chunk maxima of the accumulation plan and (unless
  // they are given) the column maxima
  const bool own_colmax = (enabled || colmax_only) && mode != kFwdFromColmax;
  const size_t clear = own_colmax ? L.colmax + static_cast<size_t>(K) * 4 : L.colmax;
  if ((cudaMemsetAsync(w, 0, clear, s)) != cudaSuccess) return I8LT_ERR_CUDA;
  if (!colmax_only && act_quant_fused_supported(at, K)) {
    // 16-bit A, 16-byte rows: column maxima, outlier set and row quantization
    // in one launch
    unsigned* arrive = reinterpret_cast<unsigned*>(w + L.status + 64);
    if (launch_act_quant_fused(A, at, M, K, L.k_pad, enabled, threshold, own_colmax && M > 0, max_outliers,
                               L.cap_pad, colmax, mask, idx, st, arrive, SCA, Aq, enabled ? subA : nullptr, asq,
                               s) != cudaSuccess)
      return I8LT_ERR_CUDA;
  } else {
    if (own_colmax && M > 0) {
      if ((launch_colmax(A, at, M, K, vec, colmax, s)) != cudaSuccess) return I8LT_ERR_CUDA;
    }
    if (colmax_only) return I8LT_OK;
    if (enabled) {
      if ((launch_outlier_index(colmax, K, threshold, max_outliers, idx, mask, st, s)) != cudaSuccess)
        return I8LT_ERR_CUDA;
    }
    if ((launch_row_quantize(A, at, M, K, L.k_pad, vec, enabled ? mask : nullptr, idx, st, L.cap_pad, SCA, Aq,
                             enabled ? subA : nullptr, asq, s)) != cudaSuccess)
      return I8LT_ERR_CUDA;
  }
  const bool with_outliers = enabled && L.cap_pad > 0;
  if (with_outliers) {
    if ((launch_build_subB(CB, L.k_pad, SCB, N, idx, st, L.cap_pad, subB, s)) != cudaSuccess)
      return I8LT_ERR_CUDA;
  }

  if ((launch_widen_codes(CB, CBh, N, L.k_pad, bsq, s)) != cudaSuccess) return I8LT_ERR_CUDA;
  if ((launch_unit_plan(asq, bsq, static_cast<int>(ceil_div(M, 256)), static_cast<int>(ceil_div(N, 256)),
                            static_cast<int>(ceil_div(L.k_pad, 1024)), plan, s)) != cudaSuccess)
    return I8LT_ERR_CUDA;

  FwdGemmArgs g;
  std::memset(&g, 0, sizeof(g));
  if (!make_tmap(&g.tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, Aq, L.k_pad, M, L.k_pad * 2, kBK, kBoxRows,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap(&g.tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, CBh, L.k_pad, N, L.k_pad * 2, kBK, kBoxRows,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return I8LT_ERR_CUDA;
  if (with_outliers) {
    if (!make_tmap(&g.tmSA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, subA, L.cap_pad, M, L.cap_pad * 2, kBK, kBoxRows,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap(&g.tmSB, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, subB, L.cap_pad, N, L.cap_pad * 2, kBK, kBoxRows,
                   CU_TENSOR_MAP_SWIZZLE_128B))
      return I8LT_ERR_CUDA;
  }
  FwdEpiArgs ea;
  ea.M = static_cast<int>(M);
  ea.N = static_cast<int>(N);
  ea.K_pad = static_cast<int>(L.k_pad);
  ea.use_outliers = with_outliers ? 1 : 0;
  ea.SCA = SCA;
  ea.plan = plan;
  ea.SCB = SCB;
  ea.bias = bias;
  ea.bias_dt = bt;
  ea.residual = residual;
  ea.out = out;
  ea.out_dt = at;
  ea.acc_i32 = dbg != nullptr ? dbg->acc_i32 : nullptr;
  ea.act = act;
  ea.act_colmax = act_colmax;
  ea.st = st;
  return cuda_status(launch_fwd_gemm(g, ea, s));
}

}  // namespace

extern "C" {

int i8lt_abi_version(void) { return kAbiVersion; }

const char* i8lt_status_string(int s) {
  switch (s) {
    case I8LT_OK: return "ok";
    case I8LT_ERR_INVALID_ARG: return "invalid argument";
    case I8LT_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
    case I8LT_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case I8LT_ERR_WORKSPACE: return "workspace missing or too small";
    case I8LT_ERR_K_TOO_LARGE: return "in_features too large for exact int32 accumulation";
    case I8LT_ERR_OUTLIER_CAPACITY: return "more outlier columns than max_outliers";
    case I8LT_ERR_TIMEOUT: return "a device pipeline wait timed out";
    case I8LT_ERR_CUDA: return "CUDA error";
    case I8LT_ERR_DEVICE: return "device is not sm_103 (GB300)";
    case I8LT_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the no-alloc buffer holds";
    default: return "unknown status";
  }
}

int64_t i8lt_weight_ld(int64_t K) { return K < 0 ? -1 : round_up(K, 16); }

int i8lt_quantize_weight(const void* W, int wt, int64_t N, int64_t K, int8_t* CB, float* SCB, void* stream) {
  if (!valid_dt(wt)) return I8LT_ERR_UNSUPPORTED_DTYPE;
  if (N < 0 || K <= 0) return I8LT_ERR_INVALID_ARG;
  if (N == 0) return I8LT_OK;
  if (W == nullptr || CB == nullptr || SCB == nullptr) return I8LT_ERR_INVALID_ARG;
  if (!aligned16(W) || !aligned16(CB)) return I8LT_ERR_MISALIGNED;
  if (int d = check_device()) return d;
  const bool vec = (K % 8) == 0;
  return cuda_status(launch_quantize_weight(W, wt, N, K, round_up(K, 16), vec, CB, SCB,
                                            static_cast<cudaStream_t>(stream)));
}

size_t i8lt_forward_workspace_size(int64_t M, int64_t K, int64_t N, int64_t max_outliers) {
  if (M < 0 || K < 0 || N < 0 || max_outliers < 0) return 0;
  return fwd_layout(M, K, N, max_outliers).total;
}

int i8lt_forward_workspace_layout(int64_t M, int64_t K, int64_t N, int64_t max_outliers, i8lt_fwd_layout* out) {
  if (out == nullptr || M < 0 || K < 0 || N < 0 || max_outliers < 0) return I8LT_ERR_INVALID_ARG;
  *out = fwd_layout(M, K, N, max_outliers);
  return I8LT_OK;
}


int i8lt_forward(const void* A, int at, int64_t M, int64_t K, const int8_t* CB, const float* SCB, int64_t N,
                 const void* bias, int bt, float threshold, const void* residual, void* out, void* ws,
                 size_t ws_bytes, int64_t max_outliers, const i8lt_fwd_debug* dbg, void* stream) {
  return forward_impl(kFwdFull, A, at, M, K, CB, SCB, N, bias, bt, threshold, residual, out, ws, ws_bytes,
                      max_outliers, dbg, stream);
}

int i8lt_forward_silu(const void* A, int at, int64_t M, int64_t K, const int8_t* CB, const float* SCB, int64_t N,
                      const void* bias, int bt, float threshold, const void* residual, void* out, void* act,
                      uint32_t* act_colmax, void* ws, size_t ws_bytes, int64_t max_outliers,
                      const i8lt_fwd_debug* dbg, void* stream) {
  if (act == nullptr || act_colmax == nullptr) return I8LT_ERR_INVALID_ARG;
  return forward_impl(kFwdFull, A, at, M, K, CB, SCB, N, bias, bt, threshold, residual, out, ws, ws_bytes,
                      max_outliers, dbg, stream, act, act_colmax);
}

int i8lt_forward_colmax(const void* A, int at, int64_t M, int64_t K, int64_t N, void* ws, size_t ws_bytes,
                        int64_t max_outliers, void* stream) {
  return forward_impl(kFwdColmaxOnly, A, at, M, K, nullptr, nullptr, N, nullptr, 0, 1.0f, nullptr, nullptr, ws,
                      ws_bytes, max_outliers, nullptr, stream);
}

int i8lt_forward_from_colmax(const void* A, int at, int64_t M, int64_t K, const int8_t* CB, const float* SCB,
                             int64_t N, const void* bias, int bt, float threshold, const void* residual, void* out,
                             void* ws, size_t ws_bytes, int64_t max_outliers, const i8lt_fwd_debug* dbg,
                             void* stream) {
  return forward_impl(kFwdFromColmax, A, at, M, K, CB, SCB, N, bias, bt, threshold, residual, out, ws, ws_bytes,
                      max_outliers, dbg, stream);
}

size_t i8lt_backward_workspace_size(int64_t M, int64_t N, int gt) {
  if (M < 0 || N < 0 || !valid_dt(gt)) return 0;
  return bwd_layout(M, N, 0, gt).total;
}

size_t i8lt_backward_workspace_size_dq(int64_t M, int64_t N, int64_t K, int gt) {
  if (M < 0 || N < 0 || K < 0 || K > I8LT_MAX_K || !valid_dt(gt)) return 0;
  return bwd_layout(M, N, K, gt).total_dq;
}

int i8lt_backward_input(const void* G, int gt, int64_t M, int64_t N, const int8_t* CB, const float* SCB, int64_t K,
                        const void* addend, void* grad_A, void* grad_bias, int bt, void* ws, size_t ws_bytes,
                        void* stream) {
  if (!valid_dt(gt) || (grad_bias != nullptr && !valid_dt(bt))) return I8LT_ERR_UNSUPPORTED_DTYPE;
  if (M < 0 || N <= 0 || K <= 0) return I8LT_ERR_INVALID_ARG;
  if (K > I8LT_MAX_K) return I8LT_ERR_K_TOO_LARGE;
  if (M > INT32_MAX / 2 || N > INT32_MAX / 2) return I8LT_ERR_INVALID_ARG;
  if (ws == nullptr) return I8LT_ERR_WORKSPACE;
  if (grad_A != nullptr && (CB == nullptr || SCB == nullptr)) return I8LT_ERR_INVALID_ARG;
  if (M > 0 && G == nullptr) return I8LT_ERR_INVALID_ARG;
  if (!aligned16(G) || !aligned16(CB) || !aligned16(grad_A) || !aligned16(addend)) return I8LT_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return I8LT_ERR_MISALIGNED;
  const BwdLayout L = bwd_layout(M, N, K, gt);
  if (ws_bytes < L.total) return I8LT_ERR_WORKSPACE;
  const bool materialize = ws_bytes >= L.total_dq;   // else the fused schedule
  if (int d = check_device()) return d;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  DevStatus* st = reinterpret_cast<DevStatus*>(w + L.status);
  float* partial = reinterpret_cast<float*>(w + L.partial);
  const bool g16_needed = grad_A != nullptr && M > 0 && needs_g16(N, gt);
  __half* G16 = g16_needed ? reinterpret_cast<__half*>(w + L.g16) : nullptr;
  const bool vec = (N % 8) == 0;
  // fp16 G that the GEMM reads as it is: grad_bias is reduced inside the
  // GEMM (its epilogue warps, from the uncast G) and no pass of its own
  // reads G; otherwise the prepass casts G and sums it in the same order
  const bool bias_in_gemm = grad_bias != nullptr && grad_A != nullptr && M > 0 && !g16_needed;
  if (cudaMemsetAsync(st, 0, sizeof(DevStatus), s) != cudaSuccess) return I8LT_ERR_CUDA;

  if ((grad_bias != nullptr && !bias_in_gemm) || G16 != nullptr) {
    if (launch_gradout_prepass(G, gt, M, N, vec, G16, L.n_pad, bias_in_gemm ? nullptr : grad_bias, bt, partial,
                               L.chunks, s) != cudaSuccess)
      return I8LT_ERR_CUDA;
  }
  if (grad_A == nullptr || M == 0) return I8LT_OK;

  const int64_t k_pad = round_up(K, 16);
  BwdGemmArgs g;
  std::memset(&g, 0, sizeof(g));
  const void* gsrc = G16 != nullptr ? static_cast<const void*>(G16) : G;
  const int64_t gpitch = G16 != nullptr ? L.n_pad : N;
  if (!make_tmap(&g.tmG, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, gsrc, gpitch, M, gpitch * 2, kBK, kBoxRows,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return I8LT_ERR_CUDA;
  if (materialize) {
    __half* WdqT = reinterpret_cast<__half*>(w + L.wdq);
    if (!make_tmap(&g.tmWT, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, WdqT, L.n_pad, k_pad, L.n_pad * 2, kBK, kBoxRows,
                   CU_TENSOR_MAP_SWIZZLE_128B))
      return I8LT_ERR_CUDA;
    if (launch_dequant_weight(CB, SCB, N, k_pad, WdqT, L.n_pad, s) != cudaSuccess) return I8LT_ERR_CUDA;
  } else if (!make_tmap(&g.tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, CB, k_pad, N, k_pad, kBoxK, kBK,
                        CU_TENSOR_MAP_SWIZZLE_128B)) {
    return I8LT_ERR_CUDA;
  }
  BwdEpiArgs ea;
  std::memset(&ea, 0, sizeof(ea));
  ea.M = static_cast<int>(M);
  ea.N = static_cast<int>(N);
  ea.K = static_cast<int>(K);
  ea.SCB = SCB;
  ea.addend = addend;
  ea.grad_A = grad_A;
  ea.dt = gt;
  ea.st = st;
  if (bias_in_gemm) {
    ea.gsum = G;
    ea.gsum_dt = gt;
    ea.partial = partial;
  }
  if (launch_bwd_gemm(g, ea, !materialize, s) != cudaSuccess) return I8LT_ERR_CUDA;
  if (bias_in_gemm) return cuda_status(launch_grad_bias_finalize(partial, M, N, grad_bias, bt, s));
  return I8LT_OK;
}

size_t i8lt_grad_weight_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 0) return 0;
  return wgrad_layout(M, N, K).total;
}

int i8lt_grad_weight(const void* G, int gt, const void* A, int at, int64_t M, int64_t N, int64_t K, void* grad_W,
                     int wt, void* ws, size_t ws_bytes, void* stream) {
  if (!valid_dt(gt) || !valid_dt(at) || !valid_dt(wt)) return I8LT_ERR_UNSUPPORTED_DTYPE;
  if (M < 0 || N <= 0 || K <= 0) return I8LT_ERR_INVALID_ARG;
  if (round_up(M, 16) > I8LT_MAX_K) return I8LT_ERR_K_TOO_LARGE;   // the tokens are the reduction
  if (N > INT32_MAX / 2 || K > INT32_MAX / 2) return I8LT_ERR_INVALID_ARG;
  if (grad_W == nullptr || ws == nullptr || (M > 0 && (G == nullptr || A == nullptr))) return I8LT_ERR_INVALID_ARG;
  if (!aligned16(G) || !aligned16(A) || !aligned16(grad_W)) return I8LT_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return I8LT_ERR_MISALIGNED;
  const WgradLayout L = wgrad_layout(M, N, K);
  if (ws_bytes < L.total) return I8LT_ERR_WORKSPACE;
  if (int d = check_device()) return d;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  // one memset: status, both column maxima; another: the chunk sums and maxima
  if (cudaMemsetAsync(w, 0, L.scale_g, s) != cudaSuccess) return I8LT_ERR_CUDA;
  if (M == 0) {
    const size_t bytes = static_cast<size_t>(N) * K * (wt == DT_F32 ? 4 : 2);
    return cuda_status(cudaMemsetAsync(grad_W, 0, bytes, s));
  }
  if (cudaMemsetAsync(w + L.tsq_g, 0, L.plan - L.tsq_g, s) != cudaSuccess) return I8LT_ERR_CUDA;
  DevStatus* st = reinterpret_cast<DevStatus*>(w + L.status);
  uint32_t* cm_g = reinterpret_cast<uint32_t*>(w + L.colmax_g);
  uint32_t* cm_a = reinterpret_cast<uint32_t*>(w + L.colmax_a);
  float* sc_g = reinterpret_cast<float*>(w + L.scale_g);
  float* sc_a = reinterpret_cast<float*>(w + L.scale_a);
  uint32_t* tsq_g = reinterpret_cast<uint32_t*>(w + L.tsq_g);
  uint32_t* tsq_a = reinterpret_cast<uint32_t*>(w + L.tsq_a);
  int* sq_g = reinterpret_cast<int*>(w + L.sq_g);
  int* sq_a = reinterpret_cast<int*>(w + L.sq_a);
  uint32_t* plan = reinterpret_cast<uint32_t*>(w + L.plan);
  __half* Gt = reinterpret_cast<__half*>(w + L.gt);
  __half* At = reinterpret_cast<__half*>(w + L.at);
  if (launch_colmax(G, gt, M, N, (N % 8) == 0, cm_g, s) != cudaSuccess ||
      launch_colmax(A, at, M, K, (K % 8) == 0, cm_a, s) != cudaSuccess ||
      launch_col_quantize(G, gt, M, N, (N % 8) == 0, cm_g, L.r_pad, sc_g, Gt, sq_g, tsq_g, s) != cudaSuccess ||
      launch_col_quantize(A, at, M, K, (K % 8) == 0, cm_a, L.r_pad, sc_a, At, sq_a, tsq_a, s) != cudaSuccess ||
      launch_unit_plan(tsq_g, tsq_a, static_cast<int>(ceil_div(N, 256)), static_cast<int>(ceil_div(K, 256)),
                       static_cast<int>(L.chunks), plan, s) != cudaSuccess)
    return I8LT_ERR_CUDA;
  // grad_W[n, k] = sum_m Gt[n, m] At[k, m] * scale_g[n] * scale_a[k] / 127^2: the
  // forward GEMM with the tokens as its reduction dimension
  FwdGemmArgs g;
  std::memset(&g, 0, sizeof(g));
  if (!make_tmap(&g.tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, Gt, L.r_pad, N, L.r_pad * 2, kBK, kBoxRows,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap(&g.tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, At, L.r_pad, K, L.r_pad * 2, kBK, kBoxRows,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return I8LT_ERR_CUDA;
  FwdEpiArgs ea;
  std::memset(&ea, 0, sizeof(ea));
  ea.M = static_cast<int>(N);
  ea.N = static_cast<int>(K);
  ea.K_pad = static_cast<int>(L.r_pad);
  ea.use_outliers = 0;
  ea.SCA = sc_g;
  ea.plan = plan;
  ea.SCB = sc_a;
  ea.bias = nullptr;
  ea.bias_dt = 0;
  ea.residual = nullptr;
  ea.out = grad_W;
  ea.out_dt = wt;
  ea.acc_i32 = nullptr;
  ea.st = st;
  return cuda_status(launch_fwd_gemm(g, ea, s, K_WGRAD_GEMM));
}

int i8lt_nf4_levels(float* out) {
  if (out == nullptr) return I8LT_ERR_INVALID_ARG;
  nf4_levels(out);
  return I8LT_OK;
}

int i8lt_fp4_levels(float* out) {
  if (out == nullptr) return I8LT_ERR_INVALID_ARG;
  fmt4_levels(kFmtFp4, out);
  return I8LT_OK;
}

int64_t i8lt_nf4_row_bytes(int64_t K) { return K < 0 ? -1 : round_up(K, 64) / 2; }

int64_t i8lt_nf4_blocks(int64_t K) { return K < 0 ? -1 : ceil_div(K, 64); }

static int quantize_4bit(int fmt, const void* W, int wt, int64_t N, int64_t K, uint8_t* packed, float* absmax,
                  void* stream) {
  if (!valid_dt(wt)) return I8LT_ERR_UNSUPPORTED_DTYPE;
  if (N < 0 || K < 0 || N > INT32_MAX / 2 || K > INT32_MAX / 2) return I8LT_ERR_INVALID_ARG;
  if (N == 0 || K == 0) return I8LT_OK;
  if (W == nullptr || packed == nullptr || absmax == nullptr) return I8LT_ERR_INVALID_ARG;
  if (!aligned16(packed)) return I8LT_ERR_MISALIGNED;
  if (int d = check_device()) return d;
  return cuda_status(launch_nf4_quantize(W, wt, N, K, i8lt_nf4_row_bytes(K), packed, absmax,
                                         static_cast<cudaStream_t>(stream), fmt));
}

static int dequantize_4bit(int fmt, const uint8_t* packed, const float* absmax, int64_t N, int64_t K, void* out, int dt,
                    void* stream) {
  if (!valid_dt(dt)) return I8LT_ERR_UNSUPPORTED_DTYPE;
  if (N < 0 || K < 0 || N > INT32_MAX / 2 || K > INT32_MAX / 2) return I8LT_ERR_INVALID_ARG;
  if (N == 0 || K == 0) return I8LT_OK;
  if (packed == nullptr || absmax == nullptr || out == nullptr) return I8LT_ERR_INVALID_ARG;
  if (!aligned16(packed)) return I8LT_ERR_MISALIGNED;
  if (int d = check_device()) return d;
  return cuda_status(launch_nf4_dequantize(packed, absmax, N, K, i8lt_nf4_row_bytes(K), out, dt,
                                           static_cast<cudaStream_t>(stream), fmt));
}

int i8lt_nf4_quantize(const void* W, int wt, int64_t N, int64_t K, uint8_t* packed, float* absmax, void* stream) {
  return quantize_4bit(kFmtNf4, W, wt, N, K, packed, absmax, stream);
}

int i8lt_fp4_quantize(const void* W, int wt, int64_t N, int64_t K, uint8_t* packed, float* absmax, void* stream) {
  return quantize_4bit(kFmtFp4, W, wt, N, K, packed, absmax, stream);
}

int i8lt_nf4_dequantize(const uint8_t* packed, const float* absmax, int64_t N, int64_t K, void* out, int dt,
                        void* stream) {
  return dequantize_4bit(kFmtNf4, packed, absmax, N, K, out, dt, stream);
}

int i8lt_fp4_dequantize(const uint8_t* packed, const float* absmax, int64_t N, int64_t K, void* out, int dt,
                        void* stream) {
  return dequantize_4bit(kFmtFp4, packed, absmax, N, K, out, dt, stream);
}

int64_t i8lt_absmax8_blocks(int64_t count) { return count < 0 ? -1 : ceil_div(count, 256); }

size_t i8lt_absmax8_workspace_size(void) { return kAlign + 256 * sizeof(unsigned long long); }

int i8lt_absmax8_quantize(const float* absmax, int64_t count, uint8_t* q, float* absmax2, float* offset, void* ws,
                          size_t ws_bytes, void* stream) {
  if (count < 0 || count > (int64_t(1) << 40)) return I8LT_ERR_INVALID_ARG;
  if (offset == nullptr || (count > 0 && (absmax == nullptr || q == nullptr || absmax2 == nullptr)))
    return I8LT_ERR_INVALID_ARG;
  if (ws == nullptr || ws_bytes < i8lt_absmax8_workspace_size()) return I8LT_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return I8LT_ERR_MISALIGNED;
  if (int d = check_device()) return d;
  auto* buckets = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(ws) + kAlign);
  return cuda_status(
      launch_absmax8_quantize(absmax, count, q, absmax2, offset, buckets, static_cast<cudaStream_t>(stream)));
}

int i8lt_absmax8_dequantize(const uint8_t* q, const float* absmax2, const float* offset, int64_t count, float* out,
                            void* stream) {
  if (count < 0 || count > (int64_t(1) << 40)) return I8LT_ERR_INVALID_ARG;
  if (count == 0) return I8LT_OK;
  if (q == nullptr || absmax2 == nullptr || offset == nullptr || out == nullptr) return I8LT_ERR_INVALID_ARG;
  if (int d = check_device()) return d;
  return cuda_status(launch_absmax8_dequantize(q, absmax2, offset, count, out, static_cast<cudaStream_t>(stream)));
}

size_t i8lt_nf4_workspace_size(void) { return kAlign; }

size_t i8lt_nf4_workspace_size_dq(int64_t K, int64_t N) {
  if (K < 0 || N < 0 || K > INT32_MAX / 2 || N > INT32_MAX / 2) return 0;
  return kAlign + align_up(static_cast<size_t>(N) * static_cast<size_t>(K) * 2);
}

size_t i8lt_nf4_grad_bias_bytes(int64_t M, int64_t N) {
  if (M < 0 || N < 0 || M > INT32_MAX / 2 || N > INT32_MAX / 2) return 0;
  return align_up(static_cast<size_t>(gradout_partial_chunks(M)) * static_cast<size_t>(N) * 4);
}

}  // extern "C"

namespace {

// The two 4-bit matmuls: D[r, m] = sum_c Wdq(r, c) X[m, c] with the packed
// weight decoded per stage (input_grad: r = k, c = n; forward: r = n, c = k).
// Workspace: [status][grad_bias partial sums, input gradient with grad_bias]
// [the dequantized weight, materialized schedule].
int nf4_gemm(int fmt, bool input_grad, const void* X, int xt, int64_t M, int64_t C, int64_t R, const uint8_t* packed,
             const float* absmax, int64_t K, int64_t N, const void* bias, int bt, void* out, void* grad_bias,
             void* ws, size_t ws_bytes, void* stream) {
  if (xt != DT_F16 && xt != DT_BF16) return I8LT_ERR_UNSUPPORTED_DTYPE;
  if ((bias != nullptr || grad_bias != nullptr) && !valid_dt(bt)) return I8LT_ERR_UNSUPPORTED_DTYPE;
  if (M < 0 || K <= 0 || N <= 0) return I8LT_ERR_INVALID_ARG;
  if (M > INT32_MAX / 2 || K > INT32_MAX / 2 || N > INT32_MAX / 2) return I8LT_ERR_INVALID_ARG;
  if (C % 8 != 0) return I8LT_ERR_INVALID_ARG;   // 16-byte rows of X for the tensor copies
  if (ws == nullptr || packed == nullptr || absmax == nullptr) return I8LT_ERR_INVALID_ARG;
  if (M > 0 && (X == nullptr || (out == nullptr && (grad_bias == nullptr || !input_grad)))) return I8LT_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(packed) || !aligned16(out)) return I8LT_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return I8LT_ERR_MISALIGNED;
  const size_t base = kAlign + (grad_bias != nullptr ? i8lt_nf4_grad_bias_bytes(M, N) : 0);
  if (ws_bytes < base) return I8LT_ERR_WORKSPACE;
  if (int d = check_device()) return d;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DevStatus* st = static_cast<DevStatus*>(ws);
  float* partial = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kAlign);
  if (cudaMemsetAsync(st, 0, sizeof(DevStatus), s) != cudaSuccess) return I8LT_ERR_CUDA;
  if (M == 0 || out == nullptr) {
    // the bias gradient alone (or of an empty batch): the prepass reduction
    if (grad_bias == nullptr) return I8LT_OK;
    return cuda_status(launch_gradout_prepass(X, xt, M, N, true, nullptr, 0, grad_bias, bt, partial,
                                              gradout_partial_chunks(M), s));
  }
  const int64_t row_bytes = i8lt_nf4_row_bytes(K);
  const CUtensorMapDataType xdt = xt == DT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  BwdGemmArgs g;
  std::memset(&g, 0, sizeof(g));
  if (!make_tmap(&g.tmG, xdt, X, C, M, C * 2, kBK, kBoxRows, CU_TENSOR_MAP_SWIZZLE_128B)) return I8LT_ERR_CUDA;
  // a workspace with room for the dequantized weight selects the materialized
  // schedule: a prepass writes Wdq [N, K] (forward) or Wdq^T [K, N] (input
  // gradient) and the GEMM reads it by TMA; otherwise the weight is decoded
  // per stage inside the GEMM
  const size_t wdq_bytes = i8lt_nf4_workspace_size_dq(K, N) - kAlign;
  const bool materialize = ws_bytes >= base + wdq_bytes;
  if (materialize) {
    void* wdq = static_cast<uint8_t*>(ws) + base;
    cudaError_t e = input_grad ? launch_nf4_dequantize_t(packed, absmax, N, K, row_bytes, wdq, xt, s, fmt)
                               : launch_nf4_dequantize(packed, absmax, N, K, row_bytes, wdq, xt, s, fmt);
    if (e != cudaSuccess) return I8LT_ERR_CUDA;
    if (!make_tmap(&g.tmWT, xdt, wdq, C, R, C * 2, kBK, kBoxRows, CU_TENSOR_MAP_SWIZZLE_128B)) return I8LT_ERR_CUDA;
  } else if (!make_tmap(&g.tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, packed, row_bytes, N, row_bytes,
                        input_grad ? 64 : 32, input_grad ? kBK : kBoxRows, CU_TENSOR_MAP_SWIZZLE_NONE)) {
    // weight tiles: [64 n][128 k] (64 bytes a row) for the input gradient,
    // [128 n][64 k] (32 bytes a row) for the forward
    return I8LT_ERR_CUDA;
  }
  BwdEpiArgs ea;
  std::memset(&ea, 0, sizeof(ea));
  ea.M = static_cast<int>(M);
  ea.N = static_cast<int>(C);
  ea.K = static_cast<int>(R);
  ea.grad_A = out;
  ea.dt = xt;
  ea.st = st;
  ea.bias = bias;
  ea.bias_dt = bt;
  ea.ab_fmt = xt == DT_BF16 ? ((1u << 7) | (1u << 10)) : 0u;   // A and B format: bf16
  ea.absmax = absmax;
  ea.nblk = static_cast<int>(ceil_div(K, 64));
  fmt4_levels(fmt, ea.lv);
  if (grad_bias != nullptr) {   // input gradient: the GEMM reduces grad_bias from G (16-bit, N % 8 == 0)
    ea.gsum = X;
    ea.gsum_dt = xt;
    ea.partial = partial;
  }
  if (launch_nf4_gemm(g, ea, input_grad, materialize, s) != cudaSuccess) return I8LT_ERR_CUDA;
  if (grad_bias != nullptr) return cuda_status(launch_grad_bias_finalize(partial, M, N, grad_bias, bt, s));
  return I8LT_OK;
}

}  // namespace

extern "C" {

int i8lt_nf4_forward(const void* A, int at, int64_t M, int64_t K, const uint8_t* packed, const float* absmax,
                     int64_t N, const void* bias, int bt, void* out, void* ws, size_t ws_bytes, void* stream) {
  return nf4_gemm(kFmtNf4, false, A, at, M, K, N, packed, absmax, K, N, bias, bt, out, nullptr, ws, ws_bytes, stream);
}

int i8lt_fp4_forward(const void* A, int at, int64_t M, int64_t K, const uint8_t* packed, const float* absmax,
                     int64_t N, const void* bias, int bt, void* out, void* ws, size_t ws_bytes, void* stream) {
  return nf4_gemm(kFmtFp4, false, A, at, M, K, N, packed, absmax, K, N, bias, bt, out, nullptr, ws, ws_bytes, stream);
}

int i8lt_nf4_backward_input(const void* G, int gt, int64_t M, int64_t N, const uint8_t* packed, const float* absmax,
                            int64_t K, void* grad_A, void* grad_bias, int bt, void* ws, size_t ws_bytes,
                            void* stream) {
  return nf4_gemm(kFmtNf4, true, G, gt, M, N, K, packed, absmax, K, N, nullptr, bt, grad_A, grad_bias, ws, ws_bytes,
                  stream);
}

int i8lt_fp4_backward_input(const void* G, int gt, int64_t M, int64_t N, const uint8_t* packed, const float* absmax,
                            int64_t K, void* grad_A, void* grad_bias, int bt, void* ws, size_t ws_bytes,
                            void* stream) {
  return nf4_gemm(kFmtFp4, true, G, gt, M, N, K, packed, absmax, K, N, nullptr, bt, grad_A, grad_bias, ws, ws_bytes,
                  stream);
}

int i8lt_silu_forward(const void* h, int dt, int64_t n, void* out, void* stream) {
  if (!valid_dt(dt)) return I8LT_ERR_UNSUPPORTED_DTYPE;
  if (n < 0 || (n > 0 && (h == nullptr || out == nullptr))) return I8LT_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(out)) return I8LT_ERR_MISALIGNED;
  if (int d = check_device()) return d;
  return cuda_status(launch_silu(h, dt, n, true, out, static_cast<cudaStream_t>(stream)));
}

int i8lt_silu_backward(const void* g, const void* h, int dt, int64_t n, void* out, void* stream) {
  if (!valid_dt(dt)) return I8LT_ERR_UNSUPPORTED_DTYPE;
  if (n < 0 || (n > 0 && (g == nullptr || h == nullptr || out == nullptr))) return I8LT_ERR_INVALID_ARG;
  if (!aligned16(g) || !aligned16(h) || !aligned16(out)) return I8LT_ERR_MISALIGNED;
  if (int d = check_device()) return d;
  return cuda_status(launch_silu_backward(g, h, dt, n, true, out, static_cast<cudaStream_t>(stream)));
}

int i8lt_profile_start(int max_launches) {
  if (max_launches < 0) return I8LT_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof.clear();
  g_ev_next = 0;
  g_prof_count = 0;
  g_prof_max = max_launches;
  g_prof_on = true;
  return I8LT_OK;
}

int i8lt_profile_stop(i8lt_kernel_time* out, int cap, int* n_records, int* n_launches) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = false;
  int st = I8LT_OK;
  int k = 0;
  for (const ProfRec& r : g_prof) {
    float ms = -1.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) {
      st = I8LT_ERR_CUDA;
      ms = -1.f;
    }
    if (out != nullptr && k < cap) out[k++] = i8lt_kernel_time{r.id, ms};
  }
  if (n_records != nullptr) *n_records = k;
  if (n_launches != nullptr) *n_launches = g_prof_count;
  g_prof.clear();
  g_ev_next = 0;
  return st;
}

int i8lt_gemm_launch_info(int kernel, int* ctas, int* threads, int* smem_bytes) {
  if (kernel != I8LT_K_FWD_GEMM && kernel != I8LT_K_BWD_GEMM) return I8LT_ERR_INVALID_ARG;
  if (int d = check_device()) return d;
  return cuda_status(gemm_launch_shape(kernel, ctas, threads, smem_bytes));
}

const char* i8lt_kernel_name(int k) {
  static const char* names[] = {"quantize_weight", "colmax",          "outlier_index",      "row_quantize",
                                "build_subB",      "fwd_gemm",        "gradout_prepass",    "grad_bias_finalize",
                                "bwd_gemm",        "silu",            "silu_backward",      "widen_codes",
                                "dequant_weight",  "col_quantize",    "wgrad_gemm",         "unit_plan",
                                "nf4_quantize",    "nf4_dequantize",  "nf4_gemm_fwd",       "nf4_gemm_bwd",
                                "absmax8"};
  return (k >= 0 && k < K_COUNT) ? names[k] : "unknown";
}

int i8lt_debug_wait_timeout(int64_t limit_ns, void* ws, size_t ws_bytes, void* stream) {
  if (limit_ns <= 0 || limit_ns > 2000000000LL) return I8LT_ERR_INVALID_ARG;
  if (ws == nullptr || ws_bytes < kAlign) return I8LT_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return I8LT_ERR_MISALIGNED;
  if (int d = check_device()) return d;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, sizeof(DevStatus), s) != cudaSuccess) return I8LT_ERR_CUDA;
  return cuda_status(launch_wait_limit(static_cast<DevStatus*>(ws), static_cast<unsigned long long>(limit_ns), s));
}

int i8lt_debug_grid_wait_timeout(int64_t limit_ns, void* ws, size_t ws_bytes, void* stream) {
  if (limit_ns <= 0 || limit_ns > 2000000000LL) return I8LT_ERR_INVALID_ARG;
  if (ws == nullptr || ws_bytes < kAlign) return I8LT_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return I8LT_ERR_MISALIGNED;
  if (int d = check_device()) return d;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, kAlign, s) != cudaSuccess) return I8LT_ERR_CUDA;
  unsigned* arrive = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(ws) + 64);
  return cuda_status(launch_grid_wait_probe(static_cast<DevStatus*>(ws), arrive,
                                            static_cast<unsigned long long>(limit_ns), s));
}

int i8lt_read_device_status(void* ws, int32_t* status, int32_t* outliers, void* stream) {
  if (ws == nullptr) return I8LT_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DevStatus h;
  if (cudaMemcpyAsync(&h, ws, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess) return I8LT_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return I8LT_ERR_CUDA;
  if (h.status != 0 && cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) return I8LT_ERR_CUDA;
  if (status != nullptr) *status = h.status;
  if (outliers != nullptr) *outliers = h.found;
  return h.status;
}

}  // extern "C"
