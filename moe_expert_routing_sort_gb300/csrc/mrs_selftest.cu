// mrs_selftest.cu -- the proxy score's error bound, checked on the device; per-context host
// state; test hooks.
//
// The multi-CTA route kernels prune with a cheap score 0.5 * tanh.approx(0.5 x) + 0.5 whose
// distance from the exact sigmoid 1 / (1 + expf(-x)) must stay within kProxyTanhBound for every
// finite bf16 x.  That is a property of the hardware's tanh approximation, so the library checks
// it itself: the first call on each device context that would prune (outside stream capture)
// enqueues an exhaustive check of all 65,536 bf16 inputs ahead of its own kernels.  The check
// writes a state word in device memory; the route kernels read it and prune only when it says
// the bound holds (1), otherwise they take exact keys for every expert.  Nothing waits on the
// host for the result.
#include <atomic>
#include <mutex>

#include "mrs_internal.h"
#include "moe_route_sort.h"

namespace mrs {

// 0: not checked on this device yet; 1: bound verified; 2: bound failed (prune nothing).
static __device__ int32_t g_proxy_state;

// Largest |0.5 * tanh.approx(0.5 x) + 0.5 - exact score| over bf16 patterns [h0, h0 + n).
__device__ __forceinline__ float proxy_error(uint32_t h) {
  const float x = bf16_bits_to_float(h);
  if (!isfinite(x)) return 0.0f;
  const float t = tanh_approx(0.5f * x);
  const double approx = 0.5 * static_cast<double>(t) + 0.5;
  const double exact = static_cast<double>(exact_score(x));
  return static_cast<float>(fabs(approx - exact)) * 1.0000001f;  // round the error upward
}

__global__ void __launch_bounds__(256) mrs_proxy_selftest_kernel(unsigned int* max_err_bits,
                                                                  float* bound_out) {
  const uint32_t h = blockIdx.x * 256u + threadIdx.x;  // 65536 patterns
  if (h == 0) *bound_out = kProxyTanhBound;
  float err = proxy_error(h);
  for (int d = 16; d > 0; d >>= 1) err = fmaxf(err, __shfl_xor_sync(kFull, err, d));
  if ((threadIdx.x & 31) == 0) atomicMax(max_err_bits, __float_as_uint(err));
}

// The in-library check: one CTA of 1024 threads takes 64 patterns each, reduces the largest
// error and writes the state word (a bound below 0 forces a failure: a test hook).
constexpr int kCheckThreads = 1024;
__global__ void __launch_bounds__(kCheckThreads) mrs_proxy_check_kernel(float bound) {
  __shared__ float wmax[kCheckThreads / 32];
  const int tid = threadIdx.x;
  float err = 0.0f;
  for (uint32_t h = tid; h < 65536u; h += kCheckThreads) err = fmaxf(err, proxy_error(h));
  for (int d = 16; d > 0; d >>= 1) err = fmaxf(err, __shfl_xor_sync(kFull, err, d));
  if ((tid & 31) == 0) wmax[tid >> 5] = err;
  __syncthreads();
  if (tid < 32) {
    float m = wmax[tid];
    for (int d = 16; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, d));
    if (tid == 0) g_proxy_state = (m <= bound) ? 1 : 2;
  }
}

// ------------------------------------------------------------------- host state
namespace {

std::atomic<long long> g_wait_limit{-1};   // < 0: kWaitLimitNs
std::atomic<int> g_cluster_tokens{-1};     // < 0: the default reach
std::atomic<int> g_grid_tokens{-1};        // < 0: kDecodeGridTokens
std::atomic<int> g_warp_grid_tokens{-1};   // < 0: the default reach
std::atomic<int> g_force_proxy_fail{0};
std::atomic<int> g_proxy_generation{1};    // bumped when the forced failure changes

using CtxGetCurrentFn = int (*)(void**);
using CtxGetIdFn = int (*)(void*, unsigned long long*);

struct DriverFns {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

const DriverFns& driver_fns() {
  static DriverFns fns = [] {
    DriverFns f;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_id = reinterpret_cast<CtxGetIdFn>(p);
    cudaGetLastError();
    return f;
  }();
  return fns;
}

struct ProxyEntry {
  int dev = -1;
  unsigned long long ctx = 0;
  int generation = 0;   // generation of the check enqueued for this context (0: none)
  int32_t* state = nullptr;
};

std::mutex g_proxy_mu;
ProxyEntry g_proxy_entries[64];

}  // namespace

unsigned long long debug_wait_limit_ns() {
  const long long v = g_wait_limit.load(std::memory_order_relaxed);
  return v < 0 ? kWaitLimitNs : static_cast<unsigned long long>(v);
}

namespace {
long long padded_rows(int T, int E, int K, int B) {
  const long long N = static_cast<long long>(T) * K;
  return N + (N < E ? N : E) * static_cast<long long>(B - 1);
}
}  // namespace

bool cluster_reach(int T, int E, int K, int B) {
  const int v = g_cluster_tokens.load(std::memory_order_relaxed);
  if (v >= 0) return T <= v;
  return T <= kClusterMaxTokens && 2ll * static_cast<long long>(T) * E <= kClusterMaxLogitBytes &&
         padded_rows(T, E, K, B) <= kClusterMaxPadded;
}

bool decode_grid_reach(int T) {
  const int v = g_grid_tokens.load(std::memory_order_relaxed);
  if (T < 2 || T > kDecodeGridTokens) return false;
  return v < 0 ? T >= kDecodeGridMinTokens : T <= v;
}

bool warp_grid_reach(int T, int sms, int& per) {
  if (T < 2 || sms < 1) return false;
  const int v = g_warp_grid_tokens.load(std::memory_order_relaxed);
  if (v < 0 ? (T < kWarpGridMinTokens || T > kWarpGridTokens) : T <= v) return false;
  per = (T + sms - 1) / sms;
  return per <= 16;
}

bool cluster_reach_sort(int T, int E, int K, int B) {
  const int v = g_cluster_tokens.load(std::memory_order_relaxed);
  if (v >= 0) return T <= v;
  return static_cast<long long>(T) * K <= kClusterMaxSortRoutes &&
         padded_rows(T, E, K, B) <= kClusterMaxPadded;
}

bool current_context(int& dev, unsigned long long& ctx_id) {
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return false;
  }
  ctx_id = 0;
  const DriverFns& f = driver_fns();
  void* ctx = nullptr;
  if (f.get_current && f.get_id && f.get_current(&ctx) == 0 && ctx) {
    unsigned long long id = 0;
    if (f.get_id(ctx, &id) == 0) ctx_id = id + 1;  // 0 stays "unknown"
  }
  return true;
}

const int32_t* proxy_state_for_launch(cudaStream_t st) {
  int dev = 0;
  unsigned long long ctx = 0;
  if (!current_context(dev, ctx) || dev >= 64) return nullptr;
  const int gen = g_proxy_generation.load(std::memory_order_relaxed);
  std::lock_guard<std::mutex> lock(g_proxy_mu);
  ProxyEntry& en = g_proxy_entries[dev];
  if (en.dev != dev || en.ctx != ctx) {
    en = ProxyEntry{};
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_proxy_state) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    en.dev = dev;
    en.ctx = ctx;
    en.state = static_cast<int32_t*>(p);
  }
  if (en.generation != gen) {
    // enqueue the check unless the stream is being captured (a captured call would freeze
    // it into the graph); until a check has run, the route kernels take exact keys
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusActive;
    const bool free_stream =
        cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusNone;
    cudaGetLastError();
    if (free_stream) {
      const float bound = g_force_proxy_fail.load() ? -1.0f : kProxyTanhBound;
      mrs_proxy_check_kernel<<<1, kCheckThreads, 0, st>>>(bound);
      if (cudaGetLastError() != cudaSuccess) return nullptr;
      en.generation = gen;
    }
  }
  return en.state;
}

}  // namespace mrs

extern "C" int moe_route_sort_proxy_selftest(float* out2, cudaStream_t stream) {
  if (!out2) return MOE_RS_ERR_NULL_POINTER;
  if (reinterpret_cast<uintptr_t>(out2) % 4) return MOE_RS_ERR_MISALIGNED;
  if (cudaMemsetAsync(out2, 0, sizeof(float), stream) != cudaSuccess) return MOE_RS_ERR_LAUNCH;
  mrs::mrs_proxy_selftest_kernel<<<256, 256, 0, stream>>>(reinterpret_cast<unsigned int*>(out2),
                                                          out2 + 1);
  if (cudaGetLastError() != cudaSuccess) return MOE_RS_ERR_LAUNCH;
  return MOE_RS_OK;
}

extern "C" int moe_route_sort_proxy_state(int32_t* dst, cudaStream_t stream) {
  if (!dst) return MOE_RS_ERR_NULL_POINTER;
  if (reinterpret_cast<uintptr_t>(dst) % 4) return MOE_RS_ERR_MISALIGNED;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, mrs::g_proxy_state) != cudaSuccess) {
    cudaGetLastError();
    return MOE_RS_ERR_LAUNCH;
  }
  if (cudaMemcpyAsync(dst, p, sizeof(int32_t), cudaMemcpyDefault, stream) != cudaSuccess) {
    cudaGetLastError();
    return MOE_RS_ERR_LAUNCH;
  }
  return MOE_RS_OK;
}

extern "C" int moe_route_sort_debug_set(int knob, long long value) {
  switch (knob) {
    case MOE_RS_DEBUG_WAIT_LIMIT_NS:
      mrs::g_wait_limit.store(value < 0 ? -1 : value);
      return MOE_RS_OK;
    case MOE_RS_DEBUG_FORCE_PROXY_FAIL: {
      const int v = value != 0 ? 1 : 0;
      if (mrs::g_force_proxy_fail.exchange(v) != v) mrs::g_proxy_generation.fetch_add(1);
      return MOE_RS_OK;
    }
    case MOE_RS_DEBUG_CLUSTER_TOKENS:
    case MOE_RS_DEBUG_GRID_TOKENS:
    case MOE_RS_DEBUG_WARP_GRID_TOKENS: {
      const long long v = value < 0 ? -1 : (value > (1ll << 30) ? (1ll << 30) : value);
      (knob == MOE_RS_DEBUG_GRID_TOKENS
           ? mrs::g_grid_tokens
           : (knob == MOE_RS_DEBUG_CLUSTER_TOKENS ? mrs::g_cluster_tokens
                                                  : mrs::g_warp_grid_tokens))
          .store(static_cast<int>(v));
      return MOE_RS_OK;
    }
    default:
      return MOE_RS_ERR_BAD_DEBUG_KNOB;
  }
}
