// mrs_sort_atomic.cu -- the sort step with atomic slot reservation (moe_sort_atomic).
//
// The unordered counterpart of moe_sort, kept to measure what the deterministic order
// costs.  It follows the workgroup-histogram scheme of "Summary -- general gfx1250
// ordinary-TP route optimization" (Capacity and dispatch; Dispatch and contracts): per-block
// shared-memory counts, one global atomic interval reservation per nonempty (expert, block),
// then block-local atomic ranks inside the reserved interval.  Which route lands in which row
// of its expert's segment therefore depends on the order the atomics happen to run in; the
// segment boundaries, padding rows, expert_ids and npp are the same as moe_sort's.
//
//   hist     blocks count their chunk of routes in shared memory, add nonzero counts to the
//            global per-expert counts (zeroed by a memset before the launch)
//   scan     one block: padded exclusive scan over experts -> offsets, reservation cursors, npp
//   scatter  blocks recount their chunk, reserve one interval per nonempty expert (global
//            atomic on the cursor), place each route at interval start + local atomic rank;
//            block c also writes the padding rows and block owners of experts c, c + grid, ...
#include "mrs_internal.h"
#include "moe_route_sort.h"

namespace mrs {

constexpr int kAtomicThreads = 512;
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kAtomicThreads) mrs_atomic_hist_kernel(const AtomicSortArgs a) {
  extern __shared__ int32_t cnt_s[];  // [E]
  const int tid = threadIdx.x;
  pdl_trigger();
  pdl_wait();
  for (int e = tid; e < a.E; e += blockDim.x) cnt_s[e] = 0;
  __syncthreads();
  const int r0 = blockIdx.x * a.chunk, r1 = min(a.N, r0 + a.chunk);
  bool bad = false;
  for (int r = r0 + tid; r < r1; r += blockDim.x) {
    const int e = a.ids[r];
    if (e >= a.E) bad = true;
    else if (e >= 0) atomicAdd(&cnt_s[e], 1);
  }
  if (__syncthreads_or(bad) && tid == 0) atomicOr(a.status, MOE_RS_DEVICE_BAD_EXPERT_ID);
  for (int e = tid; e < a.E; e += blockDim.x)
    if (cnt_s[e] != 0) atomicAdd(&a.cnt[e], cnt_s[e]);
}

__global__ void __launch_bounds__(kScanThreads) mrs_atomic_scan_kernel(const AtomicSortArgs a) {
  __shared__ int32_t wtot[33];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kScanThreads / 32;
  pdl_trigger();
  pdl_wait();
  const int B = a.B;
  const int ept = (a.E + kScanThreads - 1) / kScanThreads;  // <= 4 (E <= 4096)
  int pad[4];
  int s = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = tid * ept + i;
    pad[i] = (i < ept && e < a.E) ? ((a.cnt[e] + B - 1) & ~(B - 1)) : 0;
    s += pad[i];
  }
  const int incl = warp_inclusive_sum(s, lane);
  if (lane == 31) wtot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int v = (lane < kWarps) ? wtot[lane] : 0;
    const int wi = warp_inclusive_sum(v, lane);
    __syncwarp();
    if (lane < kWarps) wtot[lane] = wi - v;
    if (lane == 31) wtot[32] = wi;
  }
  __syncthreads();
  int off = wtot[warp] + incl - s;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = tid * ept + i;
    if (i < ept && e < a.E) {
      a.offs[e] = off;
      a.cursor[e] = off;
      off += pad[i];
    }
  }
  if (tid == 0) *a.npp = wtot[32];
}

__global__ void __launch_bounds__(kAtomicThreads)
    mrs_atomic_scatter_kernel(const AtomicSortArgs a) {
  extern __shared__ int32_t sm[];  // cnt_s[E], base_s[E]
  int32_t* cnt_s = sm;
  int32_t* base_s = sm + a.E;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  pdl_wait();
  for (int e = tid; e < a.E; e += blockDim.x) cnt_s[e] = 0;
  __syncthreads();
  const int r0 = blockIdx.x * a.chunk, r1 = min(a.N, r0 + a.chunk);
  for (int r = r0 + tid; r < r1; r += blockDim.x) {
    const int e = a.ids[r];
    if (e >= 0 && e < a.E) atomicAdd(&cnt_s[e], 1);
  }
  __syncthreads();
  // one global reservation per nonempty expert of this block
  for (int e = tid; e < a.E; e += blockDim.x) {
    const int c = cnt_s[e];
    if (c != 0) base_s[e] = atomicAdd(&a.cursor[e], c);
    cnt_s[e] = 0;
  }
  __syncthreads();
  for (int r = r0 + tid; r < r1; r += blockDim.x) {
    const int e = a.ids[r];
    if (e >= 0 && e < a.E) {
      const int pos = base_s[e] + atomicAdd(&cnt_s[e], 1);
      a.sorted_ids[pos] = r;
      a.sorted_w[pos] = a.w[r];
    }
  }
  // padding rows and block owners of experts blockIdx.x, blockIdx.x + gridDim.x, ...
  for (int e = blockIdx.x * nwarps + warp; e < a.E; e += gridDim.x * nwarps) {
    const int c = a.cnt[e];
    if (c == 0) continue;
    const int o = a.offs[e];
    const int p = (c + a.B - 1) & ~(a.B - 1);
    for (int q = o + c + lane; q < o + p; q += 32) {
      a.sorted_ids[q] = a.N;
      a.sorted_w[q] = 0.0f;
    }
    for (int b = o / a.B + lane; b < (o + p) / a.B; b += 32) a.expert_ids[b] = e;
  }
}

int atomic_sort_blocks(int N, int sms) {
  const int by_routes = (N + 511) / 512;
  const int n = by_routes < sms ? by_routes : sms;
  return n < 1 ? 1 : n;
}

cudaError_t launch_atomic_sort(const AtomicSortArgs& a, int nblk, cudaStream_t st) {
  const size_t hist_smem = sizeof(int32_t) * a.E, scat_smem = 2 * sizeof(int32_t) * a.E;
  cudaError_t err = cudaFuncSetAttribute(mrs_atomic_scatter_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(scat_smem));
  if (err != cudaSuccess) return err;
  err = launch_pdl(mrs_atomic_hist_kernel, dim3(nblk), dim3(kAtomicThreads), hist_smem, st, a);
  if (err != cudaSuccess) return err;
  err = launch_pdl(mrs_atomic_scan_kernel, dim3(1), dim3(kScanThreads), 0, st, a);
  if (err != cudaSuccess) return err;
  return launch_pdl(mrs_atomic_scatter_kernel, dim3(nblk), dim3(kAtomicThreads), scat_smem, st,
                    a);
}

}  // namespace mrs
