// mrs_internal.h -- argument blocks and launchers shared by the C ABI and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <utility>

#include "mrs_device.cuh"
#include "mrs_seg.cuh"

namespace mrs {

// Largest T the single-CTA kernel can take (its ranks use one 64-bit token mask).
constexpr int kSmallMaxTokens = 64;
// Largest T (moe_route_sort) and T * K (moe_sort) that the dispatch gives the single-CTA
// kernel: it routes a wave of up to 16 tokens at a time, one per warp, and ranks given routes
// with one warp, so past these sizes the one-cluster or three-kernel paths are faster on a
// GB300 (measured: T = 8 12.1 against 12.6 µs on the cluster, T = 64 53.7 against 13.6;
// moe_sort, 64 routes 5.3 against 7.9, 256 routes 12.0 against 8.5).
constexpr int kSmallRouteTokens = 8;
constexpr int kSmallSortRoutes = 128;
constexpr int kSmallThreads = 512;
constexpr int kSegThreads = 512;
constexpr int kUnitThreads = 512;
constexpr int kSliceThreads = 512;
constexpr int kSliceWarps = kSliceThreads / 32;
// A unit (one CTA of the route step) holds at most this many routes in shared memory.
constexpr int kUnitRouteCap = 4096;

// Units of the multi-CTA path for T tokens: one per SM (counting at most kMaxUnitSms SMs),
// but no fewer than kUnitMinTokens tokens each (a unit's warps have a token each before the
// sort step has more units to join), and at most kUnitRouteCap routes each; `sms` is the
// device's SM count.
constexpr int kMaxUnitSms = 256;
constexpr int kUnitMinTokens = 16;
inline int units_for_shape(int T, int K, int sms) {
  const int tpu_cap = kUnitRouteCap / K > 0 ? kUnitRouteCap / K : 1;
  const int s = sms < kMaxUnitSms ? sms : kMaxUnitSms;
  const int by_tokens = (T + kUnitMinTokens - 1) / kUnitMinTokens;
  int U = by_tokens < s ? by_tokens : s;
  const int need = (T + tpu_cap - 1) / tpu_cap;
  if (need > U) U = need;
  return U < 1 ? 1 : U;
}
// The largest unit count of any device: the workspace is sized for it.
inline int units_bound(int T, int K) { return units_for_shape(T, K, kMaxUnitSms); }
// Expert slices of the sort step: one per unit, or more so that a slice holds at most 16
// experts; at most one per expert and kMaxSlices.
constexpr int kMaxSlices = 256;
inline int slices_for(int U, int E) {
  int n = (E + 15) / 16;
  if (n < U) n = U;
  if (n > E) n = E;
  return n < kMaxSlices ? n : kMaxSlices;
}

// Workspace layout (byte offsets), identical for every call with the same (T, E, K).
struct WsLayout {
  size_t status;       // int32 (bytes 8..11: the grid barrier word of the few-token path)
  size_t unit_flags;   // int32[U]
  size_t slice_flags;  // uint64[slices]  look-back words of the slice kernel
  size_t loc_off;      // int32[U][E + 1] per-unit exclusive offsets of each expert
  size_t unit_buf;     // int2[T * K]     per-unit routes sorted by expert: (flat index, weight)
  size_t unit_e;       // uint16[T * K]   the expert of each unit_buf entry
  size_t adj;          // int32[E][U]     final row of unit u's first route of expert e, minus
                       //                 that route's position in the unit's list
  size_t total;
};

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

inline WsLayout ws_layout(int T, int E, int K) {
  const int U = units_bound(T, K);
  WsLayout l{};
  size_t o = 0;
  l.status = o;
  o = align16(o + 16);
  l.unit_flags = o;
  o = align16(o + sizeof(int32_t) * U);
  l.slice_flags = o;
  o = align16(o + sizeof(unsigned long long) * slices_for(U, E));
  l.loc_off = o;
  o = align16(o + sizeof(int32_t) * static_cast<size_t>(U) * (E + 1));
  l.unit_buf = o;
  o = align16(o + 8 * static_cast<size_t>(T) * K);
  l.unit_e = o;
  o = align16(o + 2 * static_cast<size_t>(T) * K);
  l.adj = o;
  o = align16(o + sizeof(int32_t) * static_cast<size_t>(U) * E);
  // moe_sort_atomic uses the same workspace as status + three [E] arrays from offset 16
  const size_t atomic_need = 16 + 3 * align16(sizeof(int32_t) * static_cast<size_t>(E));
  if (o < atomic_need) o = atomic_need;
  l.total = o;
  return l;
}

// ------------------------------------------------------------- single-CTA path
struct SmallLayout {
  int bias, keys, svals, scratch, umax, rid, rw, rrank, cnt, off, masks, owner, misc, total;
};

struct SmallArgs {
  const uint16_t* logits;
  const float* bias;
  const int32_t* in_ids;  // sort-only mode
  const float* in_w;
  int T, N, B, wave, nb_max;
  int per;                          // grid: tokens per CTA (<= wave)
  int32_t* xchg;                    // grid: T * K selected ids exchanged through global memory
  unsigned* bar;                    // grid: barrier word, zeroed by mrs_grid_prep_kernel
  unsigned long long wait_limit_ns; // grid: limit of the barrier wait (0: give up at once)
  RouteShape sh;
  bool use_seg;  // route with the segment routine (SegShape valid)
  SegShape seg;
  SmallLayout lay;
  int32_t* topk_ids;
  float* topk_w;
  int32_t* sorted_ids;
  float* sorted_w;
  int32_t* expert_ids;
  int32_t* npp;
  int32_t* status;
};

// ------------------------------------------------------------- one token (decode)
struct DecodeArgs {
  int T;          // tokens (several tokens on a grid; 1 otherwise)
  int32_t* xchg;  // several tokens on a grid: T * K selected ids exchanged through global memory
  unsigned* bar;  // several tokens on a grid: the grid barrier's word (zeroed ahead of the call)
  unsigned long long wait_limit_ns;  // several tokens: bound of the grid barrier's wait
  const uint16_t* logits;
  const float* bias;
  int E, G, g, Kg, K, B;
  float R;
  int softmax;  // 1: softmax scoring (G == 1, bias unused)
  int32_t* topk_ids;
  float* topk_w;
  int32_t* sorted_ids;
  float* sorted_w;
  int32_t* expert_ids;
  int32_t* npp;
  int32_t* status;
};

// ------------------------------------------------------------- multi-CTA path
// Phase-1 outputs of a unit, written at the end of the route (or unit) kernel.
struct UnitOut {
  int32_t* loc_off;                 // [U][E + 1]
  int2* unit_buf;                   // [T * K]
  uint16_t* unit_e;                 // [T * K]
  unsigned long long* slice_flags;  // [nslices], cleared for the slice kernel
  int32_t* unit_flags;              // [U]
  int32_t* status;                  // cleared for the slice kernel
  int nslices;
};

// Outputs of the sort step when the route step runs as one thread-block cluster.
struct ClusterOut {
  int32_t* sorted_ids;
  float* sorted_w;
  int32_t* expert_ids;
  int32_t* npp;
  int32_t* status;
  int B, N;
};

// CTAs of the cluster that runs a mid-sized route-sort call (a non-portable cluster size,
// used only where the device can place such a cluster).
constexpr int kClusterCtas = 16;
// Default reach of the cluster paths.  The cluster sits on one GPC, so it reads its inputs
// through that GPC's share of the memory system, routes on 16 SMs and writes every padding row
// from those 16 SMs; past these sizes the three-kernel path, spread over the whole GPU, is
// faster on a GB300.  moe_route_sort: at most kClusterMaxTokens tokens and
// kClusterMaxLogitBytes of logits; moe_sort: at most kClusterMaxSortRoutes routes; both: at
// most kClusterMaxPadded rows of the worst-case padded length.
constexpr int kClusterMaxTokens = 256;
constexpr long long kClusterMaxLogitBytes = 512 << 10;
constexpr long long kClusterMaxSortRoutes = 8192;
constexpr long long kClusterMaxPadded = 65536;

struct RouteArgs {
  const uint16_t* logits;
  const float* bias;
  int T, U, nwarps, max_routes;
  bool vec16;    // rows are 16-byte aligned (E % 8 == 0)
  bool use_seg;  // segment shape valid and rows 16-byte aligned: TMA-staged segment kernel
  bool sort;     // run phase 1 of the sort step after routing (else route only)
  int lanes;     // segment kernel: lanes per token (32, or 16 for two tokens per warp)
  int nbuf;      // segment kernel: row buffers per warp (1 or 2)
  RouteShape sh;
  SegShape seg;
  unsigned long long wait_limit_ns;  // bound of the row-copy waits (0: give up at once)
  const int32_t* proxy_state;        // 1 once the proxy bound has been verified on the device
  int32_t* topk_ids;
  float* topk_w;
  UnitOut uo;
  bool cluster;   // the grid is one cluster that runs both sort phases itself (co)
  ClusterOut co;
};

struct UnitArgs {
  const int32_t* ids;
  const float* w;
  int T, K, E, U, max_routes;
  UnitOut uo;
  bool cluster;   // the grid is one cluster that runs both sort phases itself (co)
  ClusterOut co;
};

struct SliceArgs {
  int T, K, E, U, B, N, nslices;
  unsigned long long wait_limit_ns;  // bound of the look-back wait (0: give up at once)
  const int32_t* loc_off;
  const int2* unit_buf;
  const uint16_t* unit_e;
  int32_t* adj;
  unsigned long long* slice_flags;
  const int32_t* unit_flags;
  int32_t* sorted_ids;
  float* sorted_w;
  int32_t* expert_ids;
  int32_t* npp;
  int32_t* status;
};

// Launch with programmatic dependent launch allowed: the kernel may be scheduled while the
// previous kernel of the stream is finishing; every kernel launched this way executes
// griddepcontrol.wait (pdl_wait) before it reads or writes global memory, so stream order
// holds (an L2 prefetch of its own inputs, which changes no value a load observes, may come
// earlier).
template <class... Params, class... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ------------------------------------------------------- atomic-order sort step
struct AtomicSortArgs {
  const int32_t* ids;
  const float* w;
  int N, E, B, chunk;
  int32_t* cnt;     // [E] global counts (zeroed before the launch)
  int32_t* cursor;  // [E] reservation cursors
  int32_t* offs;    // [E] padded exclusive offsets
  int32_t* status;
  int32_t* sorted_ids;
  float* sorted_w;
  int32_t* expert_ids;
  int32_t* npp;
};
int atomic_sort_blocks(int N, int sms);
cudaError_t launch_atomic_sort(const AtomicSortArgs& a, int nblk, cudaStream_t st);

// ------------------------------------------------------ gate projection (GEMV)
constexpr int kGateMaxTokens = 8;     // tokens per call of the gate path
constexpr int kGateMaxHidden = 8192;  // hidden size limit (a multiple of 8)
struct GateArgs {
  const uint16_t* hidden;  // [T, H] bf16
  const uint16_t* w;       // [E, H] bf16, one gate row per expert
  uint16_t* logits;        // [T, E] bf16
  int T, E, H;
  int rpc;  // gate rows per CTA (<= 16)
};
// Launch plan for `sms` SMs: gate rows per CTA and the grid.
struct GatePlan {
  int rpc, grid;
};
GatePlan gate_plan(int E, int sms);
cudaError_t launch_gate(const GateArgs& a, const GatePlan& p, cudaStream_t st);
// A cooperative grid of `ctas` CTAs (no more than the device can hold at once: one CTA per SM)
// over a.T tokens (2 <= a.T <= kDecodeGridTokens), CTA b routing tokens b, b + ctas, ..., then
// both sort phases across the grid through a.xchg (T * K int32 of the workspace) and one
// bounded grid-wide barrier on a.bar; a one-thread kernel ahead of it zeroes a.bar and the
// status word.  decode_grid_smem: the grid kernel's dynamic shared memory.
constexpr int kDecodeGridTokens = 320;
// Default lower end of that path: up to four tokens the single-CTA kernel is faster
// (measured per call: T = 2 7.7 against 9.8 us, T = 4 8.9 against 9.6).
constexpr int kDecodeGridMinTokens = 5;
// Default reach of the warp-per-token grid path (launch_small_grid): kWarpGridMinTokens <= T <=
// kWarpGridTokens, below it the per-token grid.  Measured per call (E = 896, K = 16, graph of
// calls, L2 flushed): T = 64 9.1 against 8.9 us on the per-token grid, T = 128 9.4 against 9.4,
// T = 152 9.6 against 9.9; T = 512 10.3 against 16.9 on the three-kernel path, T = 1536 15.8
// against 19.0, T = 2048 18.9 against 19.1.
constexpr int kWarpGridMinTokens = 129;
constexpr int kWarpGridTokens = 2048;
cudaError_t launch_decode_grid(const DecodeArgs& a, int ctas, cudaStream_t st);
// One-thread kernel that zeroes a grid path's barrier and status words once the kernel ahead
// in the stream has completed.
cudaError_t launch_grid_prep(unsigned* bar, int32_t* status, cudaStream_t st);
// The single-CTA kernel as a cooperative grid of ceil(a.T / a.per) CTAs (a.per <= a.wave tokens
// each, one warp per token), both sort phases across the grid through a.xchg and one bounded
// grid-wide barrier on a.bar (zeroed, with the status word, by a one-thread kernel ahead of it).
// The layout is small_layout(E, a.per * K, a.wave, nu, false, true).
cudaError_t launch_small_grid(const SmallArgs& a, cudaStream_t st);
size_t decode_grid_smem(int E, int T, int K);

// ------------------------------------------------------------ per-context host state
// Test hooks set through moe_route_sort_debug_set (process-wide).
unsigned long long debug_wait_limit_ns();  // kWaitLimitNs unless lowered
// Whether a call of T tokens over E experts (K routes per token, blocks of B rows) takes the
// cluster path: the defaults above, or, once a test hook has set a token limit, T <= that
// limit (0: never).
bool cluster_reach(int T, int E, int K, int B);
// The same for moe_sort.
bool cluster_reach_sort(int T, int E, int K, int B);
// Whether the few-token grid path takes T tokens: kDecodeGridMinTokens <= T <=
// kDecodeGridTokens by default, 2 <= T <= min(kDecodeGridTokens, limit) once the grid test hook
// has set a token limit.
bool decode_grid_reach(int T);
// Whether a call of T tokens takes the warp-per-token grid path on a device of `sms` SMs, and
// with how many tokens per CTA (`per`, at most 16, so that ceil(T / per) <= sms): by default
// kWarpGridMinTokens <= T <= kWarpGridTokens; T > limit (and T >= 2) once the test hook has
// set a limit.
bool warp_grid_reach(int T, int sms, int& per);
// Identity of the current device and context (the context's unique id, 0 if the driver cannot
// tell): host caches of device addresses are keyed on it.
bool current_context(int& dev, unsigned long long& ctx_id);
// Device address of the proxy-bound state word on the current device (1: the bound has been
// verified there; see mrs_selftest.cu).  The first call on a context, outside stream capture,
// enqueues the exhaustive check on `st` ahead of the caller's kernels.  nullptr on failure.
const int32_t* proxy_state_for_launch(cudaStream_t st);

// Launchers return the cudaError_t of the launch.
cudaError_t launch_small(const SmallArgs& a, bool sort_only, cudaStream_t st);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_route(const RouteArgs& a, size_t smem, cudaStream_t st);
cudaError_t launch_unit(const UnitArgs& a, cudaStream_t st);
cudaError_t launch_slices(const SliceArgs& a, cudaStream_t st);
cudaError_t launch_scatter(const SliceArgs& a, cudaStream_t st);
cudaError_t launch_empty(int32_t* npp, int32_t* status, cudaStream_t st);

// Shared memory of the multi-CTA route kernels for a given warp count.
size_t route_smem_bytes(int E, int nwarps, int max_routes, bool sort);
size_t seg_smem_bytes(int E, int nu, int nwarps, int max_routes, bool sort, int tpw, int nbuf,
                      bool cluster);
int seg_cluster_capacity(size_t smem);
SmallLayout small_layout(int E, int N, int wave, int nu, bool sort_only, bool grid);

// Shared memory used by phase 1 of the sort step (mrs_unit.cuh) besides the routes.
__host__ __device__ inline size_t unit_scratch_bytes(int E) {
  return align16(sizeof(unsigned long long) * E) + align16(sizeof(int32_t) * E) +
         align16(sizeof(int32_t) * (E + 1)) + align16(sizeof(int32_t) * E) + 256;
}

// Shared memory the cluster sort step needs besides the routes and counts.
__host__ __device__ inline size_t cluster_scratch_bytes(int E) {
  return align16(sizeof(unsigned) * 2 * static_cast<size_t>(E)) +   // masks
         3 * align16(sizeof(int32_t) * static_cast<size_t>(E)) +    // run, pad, tot
         align16(sizeof(int32_t) * (static_cast<size_t>(E) + 1)) +  // base
         256;                                                       // scan, dup flags
}

}  // namespace mrs
