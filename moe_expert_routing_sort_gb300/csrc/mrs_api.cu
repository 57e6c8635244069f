// mrs_api.cu -- C ABI of the MoE route-sort library: argument checks, sizes, dispatch.
//
// Everything here runs on the host and only enqueues kernels on the caller's stream; no
// call synchronises, allocates or keeps device state.  The operation is defined in
// include/moe_route_sort.h.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "moe_route_sort.h"
#include "mrs_internal.h"

namespace {

using namespace mrs;

constexpr int kMaxBlockM = 1024;

struct DeviceInfo {
  int sms = 0;
  int smem_optin = 0;
  int clusters = 0;  // kClusterCtas-CTA clusters of the segment kernel the device can hold
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
  // the limit covers static and dynamic shared memory together: keep room for the kernels'
  // own static variables, so that a planned dynamic size can always be granted
  d.smem_optin -= 1024;
  // at the largest shared-memory size: a launch that needs less fits wherever this one does
  d.clusters = seg_cluster_capacity(static_cast<size_t>(d.smem_optin));
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

// Shared-memory wavefronts of pass 1 (mrs_seg.cuh) over its first 16 unit steps (the pattern
// repeats after nu), for the start rule ((l * rot) >> rsh) % nu: lane l of a token loads 8
// bytes of its row at expert e0 = j g + q sl + 4 u (the tokens of a warp step sit in
// consecutive row buffers; half-warp phases) and the 16 bytes of bias at e0 (quarter-warp
// phases); a phase costs as many wavefronts as the most distinct words any bank serves.
int pass1_wavefronts(const SegShape& s, int lanes, int rot, int rsh) {
  int total = 0;
  for (int k = 0; k < (s.nu < 16 ? s.nu : 16); ++k) {
    for (int width = 16; width >= 8; width >>= 1) {  // 16: row loads, 8: bias loads
      const int bytes = (width == 16) ? 8 : 16;
      for (int p0 = 0; p0 < 32; p0 += width) {
        int words[32][16];
        int nw[32] = {0};
        int worst = 1;
        for (int lane = p0; lane < p0 + width; ++lane) {
          const int h = lane / lanes, ll = lane % lanes;
          const int j = ll >> s.log2L, q = ll & (s.L - 1);
          if (j >= s.G) continue;
          const int u = (((ll * rot) >> rsh) + k) % s.nu;
          const long e0 = static_cast<long>(j) * s.g + static_cast<long>(q) * s.sl + 4 * u;
          const long addr = (width == 16) ? (static_cast<long>(h) * s.E * 2 + 2 * e0) : 4 * e0;
          const int w = static_cast<int>(addr / bytes);
          for (int b = 0; b < bytes / 4; ++b) {
            const int bank = static_cast<int>((addr / 4 + b) % 32);
            bool seen = false;
            for (int i = 0; i < nw[bank]; ++i) seen |= (words[bank][i] == w);
            if (!seen && nw[bank] < 16) words[bank][nw[bank]++] = w;
            worst = nw[bank] > worst ? nw[bank] : worst;
          }
        }
        total += worst;
      }
    }
  }
  return total;
}

// The start rule of pass 1 with the fewest simulated wavefronts among rot 0 and rot 1 with a
// shift of 0 to 3 (ties keep the plain order, then the smaller shift); remembered per shape
// and thread.  The first call of a shape spends at most about 0.15 ms of host time on it.
void choose_unit_order(SegShape& s, int lanes) {
  struct Entry {
    int E, G, lanes, rot, rsh;
  };
  thread_local Entry cache[8] = {};
  thread_local int next = 0;
  for (const Entry& c : cache) {
    if (c.lanes == lanes && c.E == s.E && c.G == s.G) {
      s.rot = c.rot;
      s.rsh = c.rsh;
      return;
    }
  }
  int best_rot = 0, best_rsh = 0, best = pass1_wavefronts(s, lanes, 0, 0);
  for (int rsh = 0; rsh <= 3; ++rsh) {
    const int c = pass1_wavefronts(s, lanes, 1, rsh);
    if (c < best) {
      best = c;
      best_rot = 1;
      best_rsh = rsh;
    }
  }
  s.rot = best_rot;
  s.rsh = best_rsh;
  cache[next] = Entry{s.E, s.G, lanes, best_rot, best_rsh};
  next = (next + 1) % 8;
}

// Segment layout of the route step (see mrs_seg.cuh) for `lanes` lanes per token: groups
// split into L lanes of equal, 4-expert-aligned segments.  False when the shape does not
// allow it.
bool make_seg_shape(int E, int G, int Kg, int K, float R, int lanes, SegShape& s) {
  if (G > lanes) return false;
  int L = 1;
  while (L * 2 * G <= lanes) L *= 2;
  const int g = E / G;
  if (g % L != 0) return false;
  const int sl = g / L;
  if (sl % 4 != 0 || sl > 256) return false;  // units per lane fit a 64-bit mask
  s.E = E;
  s.G = G;
  s.g = g;
  s.Kg = Kg;
  s.K = K;
  s.L = L;
  s.log2L = 0;
  while ((1 << s.log2L) < L) ++s.log2L;
  s.sl = sl;
  s.nu = sl / 4;
  choose_unit_order(s, lanes);
  s.R = R;
  return true;
}

int launch_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_RS_OK;
  cudaGetLastError();  // clear a non-sticky launch error
  return MOE_RS_ERR_LAUNCH;
}

// Multi-CTA route step.  Units are contiguous token ranges, one CTA each; with `sort`,
// each CTA also runs phase 1 of the sort step into the workspace.
// With `co`, the grid is one cluster of U CTAs that also runs both sort phases into co
// (the segment kernel only; the caller checks that the shape has a segment layout).
int run_route(const void* logits, const float* bias, int T, const RouteShape& sh, bool sort,
              int32_t* topk_ids, float* topk_w, unsigned char* ws, const WsLayout& l, int U,
              int nslices, const DeviceInfo& d, cudaStream_t st,
              const ClusterOut* co = nullptr) {
  RouteArgs a{};
  const bool cluster = co != nullptr;
  a.logits = static_cast<const uint16_t*>(logits);
  a.bias = bias;
  a.T = T;
  a.U = U;
  a.sort = sort;
  const int tpu = (T + U - 1) / U;
  a.max_routes = tpu * sh.K;
  a.vec16 = (sh.E % 8) == 0;
  // Launch plan of the segment kernel for `lanes` lanes per token: the most warps (up to
  // one per step of the unit) whose shared memory fits, with the largest number of row
  // buffers (<= 2) that costs no warps.
  struct Plan {
    bool seg;
    SegShape shape;
    int lanes, nbuf, nwarps, want;
    size_t smem;
  };
  auto plan_for = [&](int lanes) {
    Plan p{};
    p.lanes = lanes;
    p.seg = a.vec16 && make_seg_shape(sh.E, sh.G, sh.Kg, sh.K, sh.R, lanes, p.shape);
    if (!p.seg) return p;
    const int tpw = 32 / lanes;
    const int steps = (tpu + tpw - 1) / tpw;
    const int cap = kSegThreads / 32;
    // (the cluster path keeps every warp for its sort step, whose exchange and scan are
    // spread over the CTA's threads)
    p.want = (steps < cap && !cluster) ? steps : cap;
    for (int nbuf = 2; nbuf >= 1; --nbuf) {
      int w = p.want;
      auto bytes = [&](int ww) {
        return seg_smem_bytes(sh.E, p.shape.nu, ww, a.max_routes, sort, tpw, nbuf, cluster);
      };
      while (w > 1 && bytes(w) > static_cast<size_t>(d.smem_optin)) --w;
      if (w > p.nwarps) {
        p.nwarps = w;
        p.nbuf = nbuf;
        p.smem = bytes(w);
      }
    }
    return p;
  };
  // Two tokens per warp (16 lanes each) share the per-token shuffle and scan work of the
  // route step: taken when K <= 16, the unit has tokens for every warp and all warps fit
  // with two row buffers each.  Otherwise one token per warp.
  Plan p{};
  if (sh.K <= 16 && tpu >= 2 * (kSegThreads / 32)) p = plan_for(16);
  if (!(p.seg && p.nwarps == p.want && p.nbuf == 2)) p = plan_for(32);
  a.use_seg = p.seg;
  if (cluster && !p.seg) return MOE_RS_ERR_LAUNCH;
  size_t smem;
  if (p.seg) {
    a.seg = p.shape;
    a.seg.softmax = sh.softmax;
    a.lanes = p.lanes;
    a.nbuf = p.nbuf;
    a.nwarps = p.nwarps;
    smem = p.smem;
  } else {
    int w = tpu < 16 ? tpu : 16;
    while (w > 1 && route_smem_bytes(sh.E, w, a.max_routes, sort) >
                        static_cast<size_t>(d.smem_optin))
      --w;
    a.nwarps = w;
    smem = route_smem_bytes(sh.E, w, a.max_routes, sort);
  }
  if (smem > static_cast<size_t>(d.smem_optin)) return MOE_RS_ERR_LAUNCH;
  a.sh = sh;
  a.wait_limit_ns = debug_wait_limit_ns();
  // the segment kernel prunes with proxy scores once their bound is verified on the device
  a.proxy_state = (a.use_seg && !sh.softmax) ? proxy_state_for_launch(st) : nullptr;
  a.topk_ids = topk_ids;
  a.topk_w = topk_w;
  if (sort) {
    a.uo.loc_off = reinterpret_cast<int32_t*>(ws + l.loc_off);
    a.uo.unit_buf = reinterpret_cast<int2*>(ws + l.unit_buf);
    a.uo.unit_e = reinterpret_cast<uint16_t*>(ws + l.unit_e);
    a.uo.slice_flags = reinterpret_cast<unsigned long long*>(ws + l.slice_flags);
    a.uo.unit_flags = reinterpret_cast<int32_t*>(ws + l.unit_flags);
    a.uo.status = reinterpret_cast<int32_t*>(ws + l.status);
    a.uo.nslices = nslices;
  }
  if (cluster) {
    a.cluster = true;
    a.co = *co;
  }
  return launch_status(launch_route(a, smem, st));
}

// Phase 2 of the sort step over the per-unit results in the workspace.
int run_slices(int T, int E, int K, int B, int U, int nslices, int32_t* sorted_ids,
               float* sorted_w, int32_t* expert_ids, int32_t* npp, unsigned char* ws,
               const WsLayout& l, cudaStream_t st) {
  SliceArgs c{};
  c.T = T;
  c.K = K;
  c.E = E;
  c.U = U;
  c.B = B;
  c.N = T * K;
  c.nslices = nslices;
  c.wait_limit_ns = debug_wait_limit_ns();
  c.loc_off = reinterpret_cast<const int32_t*>(ws + l.loc_off);
  c.unit_buf = reinterpret_cast<const int2*>(ws + l.unit_buf);
  c.unit_e = reinterpret_cast<const uint16_t*>(ws + l.unit_e);
  c.adj = reinterpret_cast<int32_t*>(ws + l.adj);
  c.slice_flags = reinterpret_cast<unsigned long long*>(ws + l.slice_flags);
  c.unit_flags = reinterpret_cast<const int32_t*>(ws + l.unit_flags);
  c.sorted_ids = sorted_ids;
  c.sorted_w = sorted_w;
  c.expert_ids = expert_ids;
  c.npp = npp;
  c.status = reinterpret_cast<int32_t*>(ws + l.status);
  int rc = launch_status(launch_slices(c, st));
  if (rc) return rc;
  return launch_status(launch_scatter(c, st));
}

// Single-CTA path: shared-memory layout for the largest wave that fits.
bool small_plan(int T, int E, int K, int B, bool sort_only, int nu, const DeviceInfo& d,
                SmallLayout& lay, int& wave, int& nb_max) {
  if (T > kSmallMaxTokens) return false;
  const int N = T * K;
  nb_max = static_cast<int>(max_padded64(T, E, K, B) / B);
  wave = sort_only ? 0 : (T < 16 ? T : 16);
  for (;;) {
    lay = small_layout(E, N, wave, nu, sort_only, false);
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
  if (T < 0 || E < 1 || E > kMaxExperts || topk < 1 || topk > kMaxTopk ||
      !pow2_block_m(block_m))
    return 0;
  return ws_layout(T, E, topk).total;
}

int moe_route_sort_map_host(const void* host_ptr, void** device_ptr) {
  if (!host_ptr || !device_ptr) return MOE_RS_ERR_NULL_POINTER;
  void* d = nullptr;
  if (cudaHostGetDevicePointer(&d, const_cast<void*>(host_ptr), 0) != cudaSuccess || !d) {
    cudaGetLastError();  // clear the non-sticky error
    return MOE_RS_ERR_NOT_MAPPED;
  }
  *device_ptr = d;
  return MOE_RS_OK;
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
    case MOE_RS_ERR_BAD_TOKENS:
      return "number of tokens T must be >= 0 (and at most 8 for moe_gate_route_sort)";
    case MOE_RS_ERR_OVERFLOW: return "T*topk or the padded length does not fit in int32";
    case MOE_RS_ERR_MISALIGNED:
      return "logits/workspace must be 16-byte aligned, other buffers 4-byte aligned";
    case MOE_RS_ERR_ALIAS: return "an output buffer overlaps an input or another output";
    case MOE_RS_ERR_WORKSPACE: return "workspace is NULL or smaller than required";
    case MOE_RS_ERR_BAD_SCALE: return "routed_scale must be finite";
    case MOE_RS_ERR_LAUNCH: return "the CUDA runtime rejected a kernel launch";
    case MOE_RS_ERR_TOO_LARGE:
      return "the shape needs more scratch than moe_route_sort_noalloc's static 32 MiB";
    case MOE_RS_ERR_BAD_HIDDEN:
      return "hidden size H must be a multiple of 8 in [8, 8192]";
    case MOE_RS_ERR_NOT_MAPPED:
      return "host memory is not pinned and mapped into the device address space";
    case MOE_RS_ERR_BAD_DEBUG_KNOB: return "unknown moe_route_sort_debug_set knob";
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
  const WsLayout none{};
  return run_route(logits_bf16, bias, T, sh, false, topk_ids, topk_weights, nullptr, none,
                   units_for_shape(T, topk, d.sms), 0, d, stream);
}

}  // extern "C"

namespace {

// Gate projection run ahead of the path (moe_gate_route_sort): it writes the logits the
// path then reads.  Checked by the caller except for what route_sort_impl checks itself.
struct GatePre {
  const void* hidden;
  const void* w_gate;
  int H;
};

// The whole path for both scorings: sigmoid + bias with grouped top-k (softmax == false), or
// softmax over the logits with plain top-k (softmax == true: n_group = topk_group = 1 and
// bias unused, may be NULL).  With `gate`, the gate projection producing logits_bf16 is
// launched first, once every argument has been accepted.
// Every host-side check of the whole path (shapes, pointers, workspace, alignment, aliasing),
// in the order the status codes are documented; MOE_RS_OK if the call may launch.
int validate_route_sort(const void* logits_bf16, const float* bias, int T, int E, int n_group,
                        int topk_group, int topk, float routed_scale, int block_m, bool softmax,
                        int32_t* topk_ids, float* topk_weights, int32_t* sorted_token_ids,
                        float* sorted_weights, int32_t* expert_ids,
                        int32_t* num_tokens_post_pad, void* workspace,
                        size_t workspace_bytes) {
  int rc = check_route_shape(T, E, n_group, topk_group, topk, routed_scale);
  if (rc) return rc;
  rc = check_sort_shape(T, E, topk, block_m);
  if (rc) return rc;
  if (!num_tokens_post_pad || !workspace) return workspace ? MOE_RS_ERR_NULL_POINTER
                                                           : MOE_RS_ERR_WORKSPACE;
  if (softmax) bias = nullptr;
  if (T > 0 && (!logits_bf16 || (!bias && !softmax) || !topk_ids || !topk_weights ||
                !sorted_token_ids || !sorted_weights || !expert_ids))
    return MOE_RS_ERR_NULL_POINTER;
  const WsLayout l = ws_layout(T, E, topk);
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
                      span(bias, (T > 0 && bias) ? 4 * static_cast<size_t>(E) : 0)};
  if (any_alias(outs, 7, ins, 2)) return MOE_RS_ERR_ALIAS;
  return MOE_RS_OK;
}

int route_sort_impl(const void* logits_bf16, const float* bias, int T, int E, int n_group,
                    int topk_group, int topk, float routed_scale, int block_m, bool softmax,
                    const GatePre* gate, int32_t* topk_ids, float* topk_weights,
                    int32_t* sorted_token_ids, float* sorted_weights, int32_t* expert_ids,
                    int32_t* num_tokens_post_pad, void* workspace, size_t workspace_bytes,
                    cudaStream_t stream) {
  int rc = validate_route_sort(logits_bf16, bias, T, E, n_group, topk_group, topk,
                               routed_scale, block_m, softmax, topk_ids, topk_weights,
                               sorted_token_ids, sorted_weights, expert_ids,
                               num_tokens_post_pad, workspace, workspace_bytes);
  if (rc) return rc;
  if (softmax) bias = nullptr;
  const WsLayout l = ws_layout(T, E, topk);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  int32_t* status = reinterpret_cast<int32_t*>(ws + l.status);
  if (T == 0) return launch_status(launch_empty(num_tokens_post_pad, status, stream));
  if (gate) {
    DeviceInfo gd;
    if (!device_info(gd)) return MOE_RS_ERR_LAUNCH;
    const GatePlan gp = gate_plan(E, gd.sms);
    GateArgs ga{};
    ga.hidden = static_cast<const uint16_t*>(gate->hidden);
    ga.w = static_cast<const uint16_t*>(gate->w_gate);
    ga.logits = static_cast<uint16_t*>(const_cast<void*>(logits_bf16));
    ga.T = T;
    ga.E = E;
    ga.H = gate->H;
    ga.rpc = gp.rpc;
    rc = launch_status(launch_gate(ga, gp, stream));
    if (rc) return rc;
  }

  // a few hundred tokens: the single-CTA kernel on a cooperative grid, one warp per token and
  // a contiguous range of at most 16 tokens per CTA
  DeviceInfo dw;
  int per = 0;
  if (device_info(dw) && warp_grid_reach(T, dw.sms, per)) {
    RouteShape wsh = make_shape(E, n_group, topk_group, topk, routed_scale);
    wsh.softmax = softmax ? 1 : 0;
    SegShape wseg{};
    const bool wuse_seg = make_seg_shape(E, n_group, topk_group, topk, routed_scale, 32, wseg);
    wseg.softmax = wsh.softmax;
    const SmallLayout wlay =
        small_layout(E, per * topk, per, wuse_seg ? wseg.nu : 0, false, true);
    if (wlay.total <= dw.smem_optin) {
      SmallArgs a{};
      a.use_seg = wuse_seg;
      a.seg = wseg;
      a.logits = static_cast<const uint16_t*>(logits_bf16);
      a.bias = bias;
      a.T = T;
      a.N = per * topk;
      a.B = block_m;
      a.wave = per;
      a.per = per;
      a.xchg = reinterpret_cast<int32_t*>(ws + l.unit_buf);  // T * K int32 fit in [T * K] int2
      a.bar = reinterpret_cast<unsigned*>(ws + l.status + 8);
      a.wait_limit_ns = debug_wait_limit_ns();
      a.sh = wsh;
      a.lay = wlay;
      a.topk_ids = topk_ids;
      a.topk_w = topk_weights;
      a.sorted_ids = sorted_token_ids;
      a.sorted_w = sorted_weights;
      a.expert_ids = expert_ids;
      a.npp = num_tokens_post_pad;
      a.status = status;
      rc = launch_status(launch_small_grid(a, stream));
      // a rejected launch (more CTAs than the device holds at once) enqueued at most the
      // zeroing kernel: the paths below take the call
      if (rc != MOE_RS_ERR_LAUNCH) return rc;
    }
  }

  DeviceInfo dg;
  if (decode_grid_reach(T) && device_info(dg) &&
      decode_grid_smem(E, T, topk) <= static_cast<size_t>(dg.smem_optin)) {
    // a few tokens: one CTA per token on a cooperative grid, both sort phases across the grid
    DecodeArgs a{};
    a.xchg = reinterpret_cast<int32_t*>(ws + l.unit_buf);  // T * K int32 fit in [T * K] int2
    a.bar = reinterpret_cast<unsigned*>(ws + l.status + 8);
    a.wait_limit_ns = debug_wait_limit_ns();
    a.logits = static_cast<const uint16_t*>(logits_bf16);
    a.bias = bias;
    a.E = E;
    a.G = n_group;
    a.g = E / n_group;
    a.Kg = topk_group;
    a.K = topk;
    a.B = block_m;
    a.R = routed_scale;
    a.softmax = softmax ? 1 : 0;
    a.topk_ids = topk_ids;
    a.topk_w = topk_weights;
    a.sorted_ids = sorted_token_ids;
    a.sorted_w = sorted_weights;
    a.expert_ids = expert_ids;
    a.npp = num_tokens_post_pad;
    a.status = status;
    a.T = T;
    rc = launch_status(launch_decode_grid(a, T < dg.sms ? T : dg.sms, stream));
    // a rejected launch (more CTAs than the device holds at once) enqueued nothing: the paths
    // below take the call
    if (rc != MOE_RS_ERR_LAUNCH) return rc;
  }

  if (T == 1) {
    DecodeArgs a{};
    a.logits = static_cast<const uint16_t*>(logits_bf16);
    a.bias = bias;
    a.E = E;
    a.G = n_group;
    a.g = E / n_group;
    a.Kg = topk_group;
    a.K = topk;
    a.B = block_m;
    a.R = routed_scale;
    a.softmax = softmax ? 1 : 0;
    a.topk_ids = topk_ids;
    a.topk_w = topk_weights;
    a.sorted_ids = sorted_token_ids;
    a.sorted_w = sorted_weights;
    a.expert_ids = expert_ids;
    a.npp = num_tokens_post_pad;
    a.status = status;
    return launch_status(launch_decode(a, stream));
  }
  DeviceInfo d;
  if (!device_info(d)) return MOE_RS_ERR_LAUNCH;
  RouteShape sh = make_shape(E, n_group, topk_group, topk, routed_scale);
  sh.softmax = softmax ? 1 : 0;

  SmallLayout lay;
  int wave = 0, nb_max = 0;
  SegShape seg{};
  const bool use_seg = make_seg_shape(E, n_group, topk_group, topk, routed_scale, 32, seg);
  seg.softmax = sh.softmax;
  if (T <= kSmallRouteTokens &&
      small_plan(T, E, topk, block_m, false, use_seg ? seg.nu : 0, d, lay, wave, nb_max)) {
    SmallArgs a{};
    a.use_seg = use_seg;
    a.seg = seg;
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

  // mid-sized calls: one cluster routes and sorts in a single launch
  if (use_seg && d.clusters > 0 && cluster_reach(T, E, topk, block_m) &&
      static_cast<int64_t>(T) * topk <= static_cast<int64_t>(kClusterCtas) * kUnitRouteCap) {
    ClusterOut co{};
    co.sorted_ids = sorted_token_ids;
    co.sorted_w = sorted_weights;
    co.expert_ids = expert_ids;
    co.npp = num_tokens_post_pad;
    co.status = status;
    co.B = block_m;
    co.N = T * topk;
    rc = run_route(logits_bf16, bias, T, sh, true, topk_ids, topk_weights, ws, l, kClusterCtas,
                   0, d, stream, &co);
    // a rejected cluster launch enqueued nothing: the three-kernel path below takes the call
    if (rc != MOE_RS_ERR_LAUNCH) return rc;
  }

  const int U = units_for_shape(T, topk, d.sms);
  const int nslices = slices_for(U, E);
  rc = run_route(logits_bf16, bias, T, sh, true, topk_ids, topk_weights, ws, l, U, nslices, d,
                 stream);
  if (rc) return rc;
  return run_slices(T, E, topk, block_m, U, nslices, sorted_token_ids, sorted_weights,
                    expert_ids, num_tokens_post_pad, ws, l, stream);
}

}  // namespace

extern "C" {

int moe_route_sort(const void* logits_bf16, const float* bias, int T, int E, int n_group,
                   int topk_group, int topk, float routed_scale, int block_m,
                   int32_t* topk_ids, float* topk_weights, int32_t* sorted_token_ids,
                   float* sorted_weights, int32_t* expert_ids,
                   int32_t* num_tokens_post_pad, void* workspace, size_t workspace_bytes,
                   cudaStream_t stream) {
  return route_sort_impl(logits_bf16, bias, T, E, n_group, topk_group, topk, routed_scale,
                         block_m, false, nullptr, topk_ids, topk_weights, sorted_token_ids,
                         sorted_weights, expert_ids, num_tokens_post_pad, workspace,
                         workspace_bytes, stream);
}

int moe_gate_route_sort(const void* hidden_bf16, const void* w_gate_bf16, const float* bias,
                        int T, int E, int H, int n_group, int topk_group, int topk,
                        float routed_scale, int block_m, void* logits_bf16, int32_t* topk_ids,
                        float* topk_weights, int32_t* sorted_token_ids, float* sorted_weights,
                        int32_t* expert_ids, int32_t* num_tokens_post_pad, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream) {
  if (T > kGateMaxTokens) return MOE_RS_ERR_BAD_TOKENS;
  if (H < 8 || H > kGateMaxHidden || H % 8 != 0) return MOE_RS_ERR_BAD_HIDDEN;
  int rc = check_route_shape(T, E, n_group, topk_group, topk, routed_scale);
  if (rc) return rc;
  if (T > 0) {
    if (!hidden_bf16 || !w_gate_bf16 || !logits_bf16) return MOE_RS_ERR_NULL_POINTER;
    if (!aligned(hidden_bf16, 16) || !aligned(w_gate_bf16, 16)) return MOE_RS_ERR_MISALIGNED;
    // the gate's inputs must not overlap anything the call writes
    const size_t NK = static_cast<size_t>(T) * topk;
    const size_t P = block_m >= 1 && (block_m & (block_m - 1)) == 0
                         ? static_cast<size_t>(max_padded64(T, E, topk, block_m))
                         : 0;
    const size_t NB = block_m >= 1 ? P / static_cast<size_t>(block_m) : 0;
    const Span outs[] = {span(logits_bf16, 2 * static_cast<size_t>(T) * E),
                         span(topk_ids, topk_ids ? 4 * NK : 0),
                         span(topk_weights, topk_weights ? 4 * NK : 0),
                         span(sorted_token_ids, sorted_token_ids ? 4 * P : 0),
                         span(sorted_weights, sorted_weights ? 4 * P : 0),
                         span(expert_ids, expert_ids ? 4 * NB : 0),
                         span(num_tokens_post_pad, num_tokens_post_pad ? 4 : 0),
                         span(workspace, workspace ? workspace_bytes : 0)};
    // (the bias, read by the route step, must not overlap the logits the gate writes either)
    const Span ins[] = {span(hidden_bf16, 2 * static_cast<size_t>(T) * H),
                        span(w_gate_bf16, 2 * static_cast<size_t>(E) * H),
                        span(bias, bias ? 4 * static_cast<size_t>(E) : 0)};
    for (const Span& o : outs)
      for (const Span& i : ins)
        if (overlap(o, i)) return MOE_RS_ERR_ALIAS;
  }
  const GatePre gate{hidden_bf16, w_gate_bf16, H};
  return route_sort_impl(logits_bf16, bias, T, E, n_group, topk_group, topk, routed_scale,
                         block_m, false, &gate, topk_ids, topk_weights, sorted_token_ids,
                         sorted_weights, expert_ids, num_tokens_post_pad, workspace,
                         workspace_bytes, stream);
}

int moe_route_sort_softmax(const void* logits_bf16, int T, int E, int topk, float routed_scale,
                           int block_m, int32_t* topk_ids, float* topk_weights,
                           int32_t* sorted_token_ids, float* sorted_weights,
                           int32_t* expert_ids, int32_t* num_tokens_post_pad,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return route_sort_impl(logits_bf16, nullptr, T, E, 1, 1, topk, routed_scale, block_m, true,
                         nullptr, topk_ids, topk_weights, sorted_token_ids, sorted_weights,
                         expert_ids, num_tokens_post_pad, workspace, workspace_bytes, stream);
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
  const WsLayout l = ws_layout(T, E, topk);
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
  if (T * topk <= kSmallSortRoutes &&
      small_plan(T, E, topk, block_m, true, 0, d, lay, wave, nb_max)) {
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
  // mid-sized calls: one cluster counts and places every route in a single launch
  if (d.clusters > 0 && cluster_reach_sort(T, E, topk, block_m) &&
      static_cast<int64_t>(T) * topk <= static_cast<int64_t>(kClusterCtas) * kUnitRouteCap) {
    UnitArgs c{};
    c.ids = topk_ids;
    c.w = topk_weights;
    c.T = T;
    c.K = topk;
    c.E = E;
    c.U = kClusterCtas;
    c.max_routes = ((T + kClusterCtas - 1) / kClusterCtas) * topk;
    c.cluster = true;
    c.co.sorted_ids = sorted_token_ids;
    c.co.sorted_w = sorted_weights;
    c.co.expert_ids = expert_ids;
    c.co.npp = num_tokens_post_pad;
    c.co.status = status;
    c.co.B = block_m;
    c.co.N = T * topk;
    rc = launch_status(launch_unit(c, stream));
    // a rejected cluster launch enqueued nothing: the three-kernel path below takes the call
    if (rc != MOE_RS_ERR_LAUNCH) return rc;
  }
  const int U = units_for_shape(T, topk, d.sms);
  const int nslices = slices_for(U, E);
  UnitArgs c{};
  c.ids = topk_ids;
  c.w = topk_weights;
  c.T = T;
  c.K = topk;
  c.E = E;
  c.U = U;
  c.max_routes = ((T + U - 1) / U) * topk;
  c.uo.loc_off = reinterpret_cast<int32_t*>(ws + l.loc_off);
  c.uo.unit_buf = reinterpret_cast<int2*>(ws + l.unit_buf);
  c.uo.unit_e = reinterpret_cast<uint16_t*>(ws + l.unit_e);
  c.uo.slice_flags = reinterpret_cast<unsigned long long*>(ws + l.slice_flags);
  c.uo.unit_flags = reinterpret_cast<int32_t*>(ws + l.unit_flags);
  c.uo.status = reinterpret_cast<int32_t*>(ws + l.status);
  c.uo.nslices = nslices;
  rc = launch_status(launch_unit(c, stream));
  if (rc) return rc;
  return run_slices(T, E, topk, block_m, U, nslices, sorted_token_ids, sorted_weights,
                    expert_ids, num_tokens_post_pad, ws, l, stream);
}

int moe_route_sort_from_host(const void* logits_host, void* logits_dev, const float* bias,
                             int T, int E, int n_group, int topk_group, int topk,
                             float routed_scale, int block_m, int32_t* topk_ids,
                             float* topk_weights, int32_t* sorted_token_ids,
                             float* sorted_weights, int32_t* expert_ids,
                             int32_t* num_tokens_post_pad, void* workspace,
                             size_t workspace_bytes, const void* result_dev, void* result_host,
                             size_t result_bytes, cudaStream_t stream) {
  if (T > 0 && (!logits_host || !logits_dev)) return MOE_RS_ERR_NULL_POINTER;
  if (result_bytes > 0 && (!result_dev || !result_host)) return MOE_RS_ERR_NULL_POINTER;
  // every check of moe_route_sort, on the device copy of the logits (which must not overlap an
  // output or the workspace), before anything is enqueued
  int rc = validate_route_sort(logits_dev, bias, T, E, n_group, topk_group, topk, routed_scale,
                               block_m, false, topk_ids, topk_weights, sorted_token_ids,
                               sorted_weights, expert_ids, num_tokens_post_pad, workspace,
                               workspace_bytes);
  if (rc) return rc;
  const size_t in_bytes = 2 * static_cast<size_t>(T) * static_cast<size_t>(E);
  if (in_bytes > 0 &&
      cudaMemcpyAsync(logits_dev, logits_host, in_bytes, cudaMemcpyHostToDevice, stream) !=
          cudaSuccess)
    return launch_status(cudaErrorInvalidValue);
  rc = moe_route_sort(logits_dev, bias, T, E, n_group, topk_group, topk, routed_scale, block_m,
                      topk_ids, topk_weights, sorted_token_ids, sorted_weights, expert_ids,
                      num_tokens_post_pad, workspace, workspace_bytes, stream);
  if (rc) return rc;
  if (result_bytes > 0 &&
      cudaMemcpyAsync(result_host, result_dev, result_bytes, cudaMemcpyDeviceToHost, stream) !=
          cudaSuccess)
    return launch_status(cudaErrorInvalidValue);
  return MOE_RS_OK;
}

int moe_sort_atomic(const int32_t* topk_ids, const float* topk_weights, int T, int E, int topk,
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
  const WsLayout l = ws_layout(T, E, topk);
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
  const size_t arr = align16(sizeof(int32_t) * static_cast<size_t>(E));
  AtomicSortArgs a{};
  a.ids = topk_ids;
  a.w = topk_weights;
  a.N = T * topk;
  a.E = E;
  a.B = block_m;
  a.cnt = reinterpret_cast<int32_t*>(ws + 16);
  a.cursor = reinterpret_cast<int32_t*>(ws + 16 + arr);
  a.offs = reinterpret_cast<int32_t*>(ws + 16 + 2 * arr);
  a.status = status;
  a.sorted_ids = sorted_token_ids;
  a.sorted_w = sorted_weights;
  a.expert_ids = expert_ids;
  a.npp = num_tokens_post_pad;
  const int nblk = atomic_sort_blocks(a.N, d.sms);
  a.chunk = (a.N + nblk - 1) / nblk;
  // the status word and the counts start at zero
  if (cudaMemsetAsync(ws, 0, 16 + sizeof(int32_t) * static_cast<size_t>(E), stream) !=
      cudaSuccess)
    return launch_status(cudaErrorInvalidValue);
  return launch_status(launch_atomic_sort(a, nblk, stream));
}

// ------------------------------------------------- allocation-free variant
// Scratch for moe_route_sort_noalloc: a fixed array in the library's device image, so the
// call itself allocates nothing.  Every GPU that loads the library keeps these bytes until
// the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MOE_RS_NOALLOC_SCRATCH_BYTES];

// Device address of the array in the current device's context, looked up once per context
// (with that device current) and cached: a context created again (after cudaDeviceReset, for
// example) gets a new id and a new lookup.  nullptr if the lookup fails.
static void* noalloc_scratch_ptr() {
  static std::mutex mu;
  struct Entry {
    int dev = -1;
    unsigned long long ctx = 0;
    void* ptr = nullptr;
  };
  static Entry cache[64];
  int dev = 0;
  unsigned long long ctx = 0;
  if (!current_context(dev, ctx) || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  Entry& en = cache[dev];
  if (en.ptr == nullptr || en.dev != dev || en.ctx != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    en.dev = dev;
    en.ctx = ctx;
    en.ptr = p;
  }
  return en.ptr;
}

int moe_route_sort_noalloc(const void* logits_bf16, const float* bias, int T, int E,
                           int n_group, int topk_group, int topk, float routed_scale,
                           int block_m, int32_t* topk_ids, float* topk_weights,
                           int32_t* sorted_token_ids, float* sorted_weights,
                           int32_t* expert_ids, int32_t* num_tokens_post_pad,
                           cudaStream_t stream) {
  // shapes first, so a rejected shape gets its own status and nothing is looked up
  int rc = check_route_shape(T, E, n_group, topk_group, topk, routed_scale);
  if (rc) return rc;
  rc = check_sort_shape(T, E, topk, block_m);
  if (rc) return rc;
  const size_t need = moe_route_sort_workspace_bytes(T, E, topk, block_m);
  if (need > MOE_RS_NOALLOC_SCRATCH_BYTES) return MOE_RS_ERR_TOO_LARGE;
  void* scratch = noalloc_scratch_ptr();
  if (scratch == nullptr) return MOE_RS_ERR_LAUNCH;
  return moe_route_sort(logits_bf16, bias, T, E, n_group, topk_group, topk, routed_scale,
                        block_m, topk_ids, topk_weights, sorted_token_ids, sorted_weights,
                        expert_ids, num_tokens_post_pad, scratch, MOE_RS_NOALLOC_SCRATCH_BYTES,
                        stream);
}

int moe_route_sort_noalloc_status(int32_t* dst, cudaStream_t stream) {
  if (!dst) return MOE_RS_ERR_NULL_POINTER;
  if (!aligned(dst, 4)) return MOE_RS_ERR_MISALIGNED;
  void* scratch = noalloc_scratch_ptr();
  if (scratch == nullptr) return MOE_RS_ERR_LAUNCH;
  // the status word is the first int32 of the workspace (offset 0 of the layout)
  if (cudaMemcpyAsync(dst, scratch, sizeof(int32_t), cudaMemcpyDefault, stream) !=
      cudaSuccess) {
    cudaGetLastError();
    return MOE_RS_ERR_LAUNCH;
  }
  return MOE_RS_OK;
}

}  // extern "C"
