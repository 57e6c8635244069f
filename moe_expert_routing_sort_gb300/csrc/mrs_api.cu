// mrs_api.cu -- C ABI of the MoE route-sort library: argument checks, sizes, dispatch.
//
// Everything here runs on the host and only enqueues kernels on the caller's stream; no
// call synchronises, allocates or keeps device state.  The operation is defined in
// include/moe_route_sort.h.
#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/moe_route_sort.h"
#include "mrs_internal.h"

namespace {

using namespace mrs;

constexpr int kMaxBlockM = 1024;

struct DeviceInfo {
  int sms = 0;
  int smem_optin = 0;
};

// Device attributes, cached per device on first use (host-only queries, no sync).
bool device_info(DeviceInfo& out) {
  static DeviceInfo cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return false;
  if (dev < 64 && cache[dev].sms > 0) {
    out = cache[dev];
    return true;
  }
  DeviceInfo d;
  if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return false;
  if (cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
      cudaSuccess)
    return false;
  if (dev < 64) cache[dev] = d;
  out = d;
  return true;
}

bool pow2_block_m(int B) { return B >= 1 && B <= kMaxBlockM && (B & (B - 1)) == 0; }

int64_t max_padded64(int T, int E, int K, int B) {
  const int64_t N = static_cast<int64_t>(T) * K;
  const int64_t nz = N < E ? N : E;
  return N + nz * (B - 1);
}

int check_sort_shape(int T, int E, int K, int B) {
  if (T < 0) return MOE_RS_ERR_BAD_TOKENS;
  if (E < 1 || E > kMaxExperts) return MOE_RS_ERR_BAD_EXPERTS;
  if (K < 1 || K > kMaxTopk) return MOE_RS_ERR_BAD_TOPK;
  if (!pow2_block_m(B)) return MOE_RS_ERR_BAD_BLOCK_M;
  if (static_cast<int64_t>(T) * K > INT32_MAX) return MOE_RS_ERR_OVERFLOW;
  if (max_padded64(T, E, K, B) > INT32_MAX) return MOE_RS_ERR_OVERFLOW;
  return MOE_RS_OK;
}

int check_route_shape(int T, int E, int G, int Kg, int K, float R) {
  if (T < 0) return MOE_RS_ERR_BAD_TOKENS;
  if (E < 1 || E > kMaxExperts) return MOE_RS_ERR_BAD_EXPERTS;
  if (G < 1 || G > kMaxGroups || E % G != 0 || Kg < 1 || Kg > G) return MOE_RS_ERR_BAD_GROUPS;
  if (K < 1 || K > kMaxTopk || static_cast<int64_t>(K) > static_cast<int64_t>(Kg) * (E / G))
    return MOE_RS_ERR_BAD_TOPK;
  if (!std::isfinite(R)) return MOE_RS_ERR_BAD_SCALE;
  if (static_cast<int64_t>(T) * K > INT32_MAX) return MOE_RS_ERR_OVERFLOW;
  return MOE_RS_OK;
}

struct Span {
  uintptr_t lo, hi;  // [lo, hi)
};

Span span(const void* p, size_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return Span{a, a + bytes};
}

bool overlap(const Span& a, const Span& b) {
  if (a.lo == a.hi || b.lo == b.hi) return false;
  return a.lo < b.hi && b.lo < a.hi;
}

// Outputs must not overlap each other or any input.
bool any_alias(const Span* outs, int nout, const Span* ins, int nin) {
  for (int i = 0; i < nout; ++i) {
    for (int j = i + 1; j < nout; ++j)
      if (overlap(outs[i], outs[j])) return true;
    for (int j = 0; j < nin; ++j)
      if (overlap(outs[i], ins[j])) return true;
  }
  return false;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

RouteShape make_shape(int E, int G, int Kg, int K, float R) {
  RouteShape sh{};
  sh.E = E;
  sh.G = G;
  sh.g = E / G;
  sh.Kg = Kg;
  sh.K = K;
  sh.R = R;
  int L = 1;
  if (G <= 32)
    while (L * 2 * G <= 32) L *= 2;
  sh.L = L;
  sh.log2L = 0;
  while ((1 << sh.log2L) < L) ++sh.log2L;
  sh.gpr = 32 / L;
  sh.rounds = (G + sh.gpr - 1) / sh.gpr;
  return sh;
}

int launch_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_RS_OK;
  cudaGetLastError();  // clear a non-sticky launch error
  return MOE_RS_ERR_LAUNCH;
}

// Warps per CTA of the route kernel that fit in shared memory.
int route_max_warps(int E, bool hist, const DeviceInfo& d) {
  int w = 16;
  while (w > 1 && route_smem_bytes(E, w, hist) > static_cast<size_t>(d.smem_optin)) --w;
  return w;
}

// Multi-CTA route step.  Units are contiguous token ranges; one CTA each.
int run_route(const void* logits, const float* bias, int T, const RouteShape& sh,
              int32_t* topk_ids, float* topk_w, int32_t* partial, int32_t* unit_flags,
              int U, const DeviceInfo& d, cudaStream_t st) {
  RouteArgs a{};
  a.logits = static_cast<const uint16_t*>(logits);
  a.bias = bias;
  a.T = T;
  a.U = U;
  const bool hist = partial != nullptr;
  const int maxw = route_max_warps(sh.E, hist, d);
  const int per_unit = (T + U - 1) / U;
  a.nwarps = per_unit < maxw ? per_unit : maxw;
  a.vec16 = (sh.E % 8) == 0;
  a.sh = sh;
  a.topk_ids = topk_ids;
  a.topk_w = topk_w;
  a.partial = partial;
  a.unit_flags = unit_flags;
  const size_t smem = route_smem_bytes(sh.E, a.nwarps, hist);
  if (smem > static_cast<size_t>(d.smem_optin)) return MOE_RS_ERR_LAUNCH;
  return launch_status(launch_route(a, smem, st));
}

int units_for(int T, const DeviceInfo& d) {
  int U = d.sms;
  if (U > kMaxUnits) U = kMaxUnits;
  if (U > T) U = T;
  return U < 1 ? 1 : U;
}

// Scan + scatter over the partial counts already in the workspace.
int run_sort_tail(const int32_t* ids, const float* w, int T, int E, int K, int B, int U,
                  int32_t* sorted_ids, float* sorted_w, int32_t* expert_ids, int32_t* npp,
                  unsigned char* ws, const WsLayout& l, cudaStream_t st) {
  ScanArgs s{};
  s.E = E;
  s.U = U;
  s.B = B;
  s.partial = reinterpret_cast<int32_t*>(ws + l.partial);
  s.cnt_tot = reinterpret_cast<int32_t*>(ws + l.cnt_tot);
  s.inchunk_off = reinterpret_cast<int32_t*>(ws + l.inchunk_off);
  s.chunk_tot = reinterpret_cast<int32_t*>(ws + l.chunk_tot);
  int rc = launch_status(launch_scan(s, st));
  if (rc) return rc;
  ScatterArgs c{};
  c.ids = ids;
  c.w = w;
  c.T = T;
  c.K = K;
  c.E = E;
  c.U = U;
  c.B = B;
  c.N = T * K;
  c.nchunk = (E + kChunk - 1) / kChunk;
  c.partial = s.partial;
  c.cnt_tot = s.cnt_tot;
  c.inchunk_off = s.inchunk_off;
  c.chunk_tot = s.chunk_tot;
  c.unit_flags = reinterpret_cast<const int32_t*>(ws + l.unit_flags);
  c.sorted_ids = sorted_ids;
  c.sorted_w = sorted_w;
  c.expert_ids = expert_ids;
  c.npp = npp;
  c.status = reinterpret_cast<int32_t*>(ws + l.status);
  return launch_status(launch_scatter(c, st));
}

// Single-CTA path: shared-memory layout for the largest wave that fits.
bool small_plan(int T, int E, int K, int B, bool sort_only, const DeviceInfo& d,
                SmallLayout& lay, int& wave, int& nb_max) {
  if (T > kSmallMaxTokens) return false;
  const int N = T * K;
  nb_max = static_cast<int>(max_padded64(T, E, K, B) / B);
  wave = sort_only ? 0 : (T < 32 ? T : 32);
  for (;;) {
    lay = small_layout(E, N, wave, nb_max, sort_only);
    if (lay.total <= d.smem_optin) return true;
    if (sort_only || wave <= 1) return false;
    --wave;
  }
}

}  // namespace

extern "C" {

size_t moe_sort_max_padded(int T, int E, int topk, int block_m) {
  if (T < 0 || E < 1 || topk < 1 || !pow2_block_m(block_m)) return 0;
  return static_cast<size_t>(max_padded64(T, E, topk, block_m));
}

size_t moe_sort_max_blocks(int T, int E, int topk, int block_m) {
  if (T < 0 || E < 1 || topk < 1 || !pow2_block_m(block_m)) return 0;
  return static_cast<size_t>(max_padded64(T, E, topk, block_m) / block_m);
}

size_t moe_route_sort_workspace_bytes(int T, int E, int topk, int block_m) {
  if (T < 0 || E < 1 || E > kMaxExperts || topk < 1 || !pow2_block_m(block_m)) return 0;
  return ws_layout(T, E).total;
}

const char* moe_route_sort_strerror(int status) {
  switch (status) {
    case MOE_RS_OK: return "success";
    case MOE_RS_ERR_NULL_POINTER: return "a required pointer is NULL";
    case MOE_RS_ERR_BAD_EXPERTS: return "number of experts E must be in [1, 4096]";
    case MOE_RS_ERR_BAD_GROUPS:
      return "n_group must be in [1, 64] and divide E; topk_group must be in [1, n_group]";
    case MOE_RS_ERR_BAD_TOPK:
      return "topk must be in [1, 32] and at most topk_group * (E / n_group)";
    case MOE_RS_ERR_BAD_BLOCK_M: return "block_m must be a power of two in [1, 1024]";
    case MOE_RS_ERR_BAD_TOKENS: return "number of tokens T must be >= 0";
    case MOE_RS_ERR_OVERFLOW: return "T*topk or the padded length does not fit in int32";
    case MOE_RS_ERR_MISALIGNED:
      return "logits/workspace must be 16-byte aligned, other buffers 4-byte aligned";
    case MOE_RS_ERR_ALIAS: return "an output buffer overlaps an input or another output";
    case MOE_RS_ERR_WORKSPACE: return "workspace is NULL or smaller than required";
    case MOE_RS_ERR_BAD_SCALE: return "routed_scale must be finite";
    case MOE_RS_ERR_LAUNCH: return "the CUDA runtime rejected a kernel launch";
    default: return "unknown status";
  }
}

int moe_topk(const void* logits_bf16, const float* bias, int T, int E, int n_group,
             int topk_group, int topk, float routed_scale, int32_t* topk_ids,
             float* topk_weights, cudaStream_t stream) {
  int rc = check_route_shape(T, E, n_group, topk_group, topk, routed_scale);
  if (rc) return rc;
  if (T == 0) return MOE_RS_OK;
  if (!logits_bf16 || !bias || !topk_ids || !topk_weights) return MOE_RS_ERR_NULL_POINTER;
  if (!aligned(logits_bf16, 16) || !aligned(bias, 4) || !aligned(topk_ids, 4) ||
      !aligned(topk_weights, 4))
    return MOE_RS_ERR_MISALIGNED;
  const size_t NK = static_cast<size_t>(T) * topk;
  const Span outs[] = {span(topk_ids, 4 * NK), span(topk_weights, 4 * NK)};
  const Span ins[] = {span(logits_bf16, 2 * static_cast<size_t>(T) * E), span(bias, 4 * (size_t)E)};
  if (any_alias(outs, 2, ins, 2)) return MOE_RS_ERR_ALIAS;
  DeviceInfo d;
  if (!device_info(d)) return MOE_RS_ERR_LAUNCH;
  const RouteShape sh = make_shape(E, n_group, topk_group, topk, routed_scale);
  return run_route(logits_bf16, bias, T, sh, topk_ids, topk_weights, nullptr, nullptr,
                   units_for(T, d), d, stream);
}

int moe_route_sort(const void* logits_bf16, const float* bias, int T, int E, int n_group,
                   int topk_group, int topk, float routed_scale, int block_m,
                   int32_t* topk_ids, float* topk_weights, int32_t* sorted_token_ids,
                   float* sorted_weights, int32_t* expert_ids,
                   int32_t* num_tokens_post_pad, void* workspace, size_t workspace_bytes,
                   cudaStream_t stream) {
  int rc = check_route_shape(T, E, n_group, topk_group, topk, routed_scale);
  if (rc) return rc;
  rc = check_sort_shape(T, E, topk, block_m);
  if (rc) return rc;
  if (!num_tokens_post_pad || !workspace) return workspace ? MOE_RS_ERR_NULL_POINTER
                                                           : MOE_RS_ERR_WORKSPACE;
  if (T > 0 && (!logits_bf16 || !bias || !topk_ids || !topk_weights || !sorted_token_ids ||
                !sorted_weights || !expert_ids))
    return MOE_RS_ERR_NULL_POINTER;
  const WsLayout l = ws_layout(T, E);
  if (workspace_bytes < l.total) return MOE_RS_ERR_WORKSPACE;
  if (!aligned(workspace, 16) || !aligned(num_tokens_post_pad, 4)) return MOE_RS_ERR_MISALIGNED;
  if (T > 0 && (!aligned(logits_bf16, 16) || !aligned(bias, 4) || !aligned(topk_ids, 4) ||
                !aligned(topk_weights, 4) || !aligned(sorted_token_ids, 4) ||
                !aligned(sorted_weights, 4) || !aligned(expert_ids, 4)))
    return MOE_RS_ERR_MISALIGNED;
  const size_t NK = static_cast<size_t>(T) * topk;
  const size_t P = static_cast<size_t>(max_padded64(T, E, topk, block_m));
  const size_t NB = P / block_m;
  const Span outs[] = {span(topk_ids, 4 * NK),         span(topk_weights, 4 * NK),
                       span(sorted_token_ids, 4 * P),  span(sorted_weights, 4 * P),
                       span(expert_ids, 4 * NB),       span(num_tokens_post_pad, 4),
                       span(workspace, workspace_bytes)};
  const Span ins[] = {span(logits_bf16, 2 * static_cast<size_t>(T) * E),
                      span(bias, T > 0 ? 4 * static_cast<size_t>(E) : 0)};
  if (any_alias(outs, 7, ins, 2)) return MOE_RS_ERR_ALIAS;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  int32_t* status = reinterpret_cast<int32_t*>(ws + l.status);
  if (T == 0) return launch_status(launch_empty(num_tokens_post_pad, status, stream));

  DeviceInfo d;
  if (!device_info(d)) return MOE_RS_ERR_LAUNCH;
  const RouteShape sh = make_shape(E, n_group, topk_group, topk, routed_scale);

  SmallLayout lay;
  int wave = 0, nb_max = 0;
  if (T <= kSmallMaxTokens && small_plan(T, E, topk, block_m, false, d, lay, wave, nb_max)) {
    SmallArgs a{};
    a.logits = static_cast<const uint16_t*>(logits_bf16);
    a.bias = bias;
    a.T = T;
    a.N = T * topk;
    a.B = block_m;
    a.wave = wave;
    a.nb_max = nb_max;
    a.sh = sh;
    a.lay = lay;
    a.topk_ids = topk_ids;
    a.topk_w = topk_weights;
    a.sorted_ids = sorted_token_ids;
    a.sorted_w = sorted_weights;
    a.expert_ids = expert_ids;
    a.npp = num_tokens_post_pad;
    a.status = status;
    return launch_status(launch_small(a, false, stream));
  }

  const int U = units_for(T, d);
  int32_t* partial = reinterpret_cast<int32_t*>(ws + l.partial);
  int32_t* unit_flags = reinterpret_cast<int32_t*>(ws + l.unit_flags);
  rc = run_route(logits_bf16, bias, T, sh, topk_ids, topk_weights, partial, unit_flags, U, d,
                 stream);
  if (rc) return rc;
  return run_sort_tail(topk_ids, topk_weights, T, E, topk, block_m, U, sorted_token_ids,
                       sorted_weights, expert_ids, num_tokens_post_pad, ws, l, stream);
}

int moe_sort(const int32_t* topk_ids, const float* topk_weights, int T, int E, int topk,
             int block_m, int32_t* sorted_token_ids, float* sorted_weights,
             int32_t* expert_ids, int32_t* num_tokens_post_pad, void* workspace,
             size_t workspace_bytes, cudaStream_t stream) {
  int rc = check_sort_shape(T, E, topk, block_m);
  if (rc) return rc;
  if (!num_tokens_post_pad || !workspace) return workspace ? MOE_RS_ERR_NULL_POINTER
                                                           : MOE_RS_ERR_WORKSPACE;
  if (T > 0 && (!topk_ids || !topk_weights || !sorted_token_ids || !sorted_weights ||
                !expert_ids))
    return MOE_RS_ERR_NULL_POINTER;
  const WsLayout l = ws_layout(T, E);
  if (workspace_bytes < l.total) return MOE_RS_ERR_WORKSPACE;
  if (!aligned(workspace, 16) || !aligned(num_tokens_post_pad, 4)) return MOE_RS_ERR_MISALIGNED;
  if (T > 0 && (!aligned(topk_ids, 4) || !aligned(topk_weights, 4) ||
                !aligned(sorted_token_ids, 4) || !aligned(sorted_weights, 4) ||
                !aligned(expert_ids, 4)))
    return MOE_RS_ERR_MISALIGNED;
  const size_t NK = static_cast<size_t>(T) * topk;
  const size_t P = static_cast<size_t>(max_padded64(T, E, topk, block_m));
  const size_t NB = P / block_m;
  const Span outs[] = {span(sorted_token_ids, 4 * P), span(sorted_weights, 4 * P),
                       span(expert_ids, 4 * NB), span(num_tokens_post_pad, 4),
                       span(workspace, workspace_bytes)};
  const Span ins[] = {span(topk_ids, 4 * NK), span(topk_weights, 4 * NK)};
  if (any_alias(outs, 5, ins, 2)) return MOE_RS_ERR_ALIAS;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  int32_t* status = reinterpret_cast<int32_t*>(ws + l.status);
  if (T == 0) return launch_status(launch_empty(num_tokens_post_pad, status, stream));

  DeviceInfo d;
  if (!device_info(d)) return MOE_RS_ERR_LAUNCH;
  SmallLayout lay;
  int wave = 0, nb_max = 0;
  if (T * topk <= 2048 && small_plan(T, E, topk, block_m, true, d, lay, wave, nb_max)) {
    SmallArgs a{};
    a.in_ids = topk_ids;
    a.in_w = topk_weights;
    a.T = T;
    a.N = T * topk;
    a.B = block_m;
    a.nb_max = nb_max;
    a.sh = make_shape(E, 1, 1, 1, 1.0f);
    a.sh.K = topk;
    a.lay = lay;
    a.sorted_ids = sorted_token_ids;
    a.sorted_w = sorted_weights;
    a.expert_ids = expert_ids;
    a.npp = num_tokens_post_pad;
    a.status = status;
    return launch_status(launch_small(a, true, stream));
  }
  const int U = units_for(T, d);
  CountArgs c{};
  c.ids = topk_ids;
  c.T = T;
  c.K = topk;
  c.E = E;
  c.U = U;
  c.partial = reinterpret_cast<int32_t*>(ws + l.partial);
  c.unit_flags = reinterpret_cast<int32_t*>(ws + l.unit_flags);
  rc = launch_status(launch_count(c, stream));
  if (rc) return rc;
  return run_sort_tail(topk_ids, topk_weights, T, E, topk, block_m, U, sorted_token_ids,
                       sorted_weights, expert_ids, num_tokens_post_pad, ws, l, stream);
}

}  // extern "C"
