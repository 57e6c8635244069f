// mrs_internal.h -- argument blocks and launchers shared by the C ABI and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "mrs_device.cuh"

namespace mrs {

// Routes per unit-tile in the scatter step: one bit per token in a 64-bit mask.
constexpr int kTileTokens = 64;
// Largest number of units (CTAs of the multi-CTA path); sizes the workspace bound.
constexpr int kMaxUnits = 1024;
// Largest T that takes the single-CTA path (its ranks use one 64-bit token mask).
constexpr int kSmallMaxTokens = 64;
constexpr int kSmallThreads = 1024;
constexpr int kChunk = 32;  // experts per chunk of the padded scan
constexpr int kMaxChunks = kMaxExperts / kChunk;

// Workspace layout (byte offsets), identical for every call with the same (T, E).
struct WsLayout {
  size_t status;       // int32
  size_t unit_flags;   // int32[kMaxUnits]
  size_t cnt_tot;      // int32[E]   routes per expert
  size_t inchunk_off;  // int32[E]   padded offset inside its 32-expert chunk
  size_t chunk_tot;    // int32[kMaxChunks] padded rows per chunk
  size_t partial;      // int32[U_bound][E] per-unit counts, then exclusive prefix over units
  size_t total;
};

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

inline int units_bound(int T) { return T < kMaxUnits ? (T > 0 ? T : 1) : kMaxUnits; }

inline WsLayout ws_layout(int T, int E) {
  WsLayout l{};
  size_t o = 0;
  l.status = o;
  o = align16(o + 16);
  l.unit_flags = o;
  o = align16(o + sizeof(int32_t) * kMaxUnits);
  l.cnt_tot = o;
  o = align16(o + sizeof(int32_t) * E);
  l.inchunk_off = o;
  o = align16(o + sizeof(int32_t) * E);
  l.chunk_tot = o;
  o = align16(o + sizeof(int32_t) * kMaxChunks);
  l.partial = o;
  o = align16(o + sizeof(int32_t) * (size_t)units_bound(T) * E);
  l.total = o;
  return l;
}

// ------------------------------------------------------------- single-CTA path
struct SmallLayout {
  int bias, keys, svals, scratch, rid, rw, rrank, cnt, off, masks, owner, misc, total;
};

struct SmallArgs {
  const uint16_t* logits;
  const float* bias;
  const int32_t* in_ids;  // sort-only mode
  const float* in_w;
  int T, N, B, wave, nb_max;
  RouteShape sh;
  SmallLayout lay;
  int32_t* topk_ids;
  float* topk_w;
  int32_t* sorted_ids;
  float* sorted_w;
  int32_t* expert_ids;
  int32_t* npp;
  int32_t* status;
};

// ------------------------------------------------------------- multi-CTA path
struct RouteArgs {
  const uint16_t* logits;
  const float* bias;
  int T, U, nwarps;
  bool vec16;  // rows are 16-byte aligned (E % 8 == 0)
  RouteShape sh;
  int32_t* topk_ids;
  float* topk_w;
  int32_t* partial;     // [U][E] or null (route only)
  int32_t* unit_flags;  // [U] or null
};

struct CountArgs {
  const int32_t* ids;
  int T, K, E, U;
  int32_t* partial;
  int32_t* unit_flags;
};

struct ScanArgs {
  int E, U, B;
  int32_t* partial;
  int32_t* cnt_tot;
  int32_t* inchunk_off;
  int32_t* chunk_tot;
};

struct ScatterArgs {
  const int32_t* ids;
  const float* w;
  int T, K, E, U, B, N, nchunk;
  const int32_t* partial;
  const int32_t* cnt_tot;
  const int32_t* inchunk_off;
  const int32_t* chunk_tot;
  const int32_t* unit_flags;
  int32_t* sorted_ids;
  float* sorted_w;
  int32_t* expert_ids;
  int32_t* npp;
  int32_t* status;
};

// Launchers return the cudaError_t of the launch.
cudaError_t launch_small(const SmallArgs& a, bool sort_only, cudaStream_t st);
cudaError_t launch_route(const RouteArgs& a, size_t smem, cudaStream_t st);
cudaError_t launch_count(const CountArgs& a, cudaStream_t st);
cudaError_t launch_scan(const ScanArgs& a, cudaStream_t st);
cudaError_t launch_scatter(const ScatterArgs& a, cudaStream_t st);
cudaError_t launch_empty(int32_t* npp, int32_t* status, cudaStream_t st);

// Shared memory of the multi-CTA route kernel for a given warp count.
size_t route_smem_bytes(int E, int nwarps, bool with_hist);
SmallLayout small_layout(int E, int N, int wave, int nb_max, bool sort_only);

}  // namespace mrs
