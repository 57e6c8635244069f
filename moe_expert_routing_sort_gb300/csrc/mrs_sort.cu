// mrs_sort.cu -- both sort phases of the multi-CTA MoE route-sort path for sm_103a.
//
// Source: "perf(flydsl): Kimi-K3 B1 route-sort + prepared-MoE handoff (stack)", Summary
// ("both sort phases" feeding prepared metadata to GEMM1).  Dropped routes (negative ids)
// claim no slot: "Summary -- general gfx1250 ordinary-TP route optimization", Dispatch and
// contracts.
//
// Phase 1 runs at the end of the kernel that produced the routes of a unit (a contiguous
// token range, one CTA): unit_sort_tail() stable-sorts the unit's routes by expert in
// shared memory and stores, per unit, the exclusive per-expert offsets loc[u][0..E] and
// the sorted (flat index, weight, expert) list.  It also clears the look-back flags of
// phase 2.
//
// Phase 2a (mrs_slices_kernel) gives every CTA a slice of experts: a prefix over units of
// the slice's counts, the block_m-padded offsets inside the slice and a decoupled
// look-back for the slice's base row (every slice publishes its padded size and sums those
// of the slices before it).  It stores, for every (unit, expert) pair with routes, the
// final row of the pair's first route minus that route's position in the unit's list,
// and writes the padding rows and the per-block expert ids.
// Phase 2b (mrs_scatter_kernel), one CTA per unit, moves each route of the unit's list to
// its final row: work is proportional to the unit's routes, however skewed the experts.
// Entries of one expert stay in token-then-slot order by construction; no global atomics
// are used, and every wait is bounded.
#include "mrs_internal.h"
#include "mrs_cluster.cuh"
#include "mrs_unit.cuh"
#include "moe_route_sort.h"

namespace mrs {

// ------------------------------------------------- phase 1 for moe_sort (given routes)
// kCluster: the grid is one thread-block cluster that runs both sort phases itself
// (cluster_sort_tail) instead of phase 1 into the workspace.
template <bool kCluster>
__global__ void __launch_bounds__(kUnitThreads) mrs_unit_kernel(const UnitArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x;
  int t0, t1;
  unit_range(blockIdx.x, a.T, a.U, t0, t1);
  const int nr = (t1 - t0) * a.K;
  int32_t* rid = reinterpret_cast<int32_t*>(smem);
  float* rw = reinterpret_cast<float*>(smem + align16(sizeof(int32_t) * a.max_routes));
  int32_t* cnt = reinterpret_cast<int32_t*>(smem + 2 * align16(sizeof(int32_t) * a.max_routes));
  unsigned char* scratch = smem + 2 * align16(sizeof(int32_t) * a.max_routes) +
                           align16(sizeof(int32_t) * (a.E + 1));
  __shared__ int bad;
  pdl_trigger();
  pdl_wait();
  if (tid == 0) bad = 0;
  for (int e = tid; e < a.E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const size_t r0 = static_cast<size_t>(t0) * a.K;
  for (int i = tid; i < nr; i += blockDim.x) {
    const int e = a.ids[r0 + i];
    rid[i] = e;
    rw[i] = a.w[r0 + i];
    if (e >= a.E) bad = MOE_RS_DEVICE_BAD_EXPERT_ID;
    else if (e >= 0) atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  if (kCluster) {
    cluster_sort_tail(rid, rw, cnt, &bad, a.E, a.K, t0, t1, blockIdx.x,
                      static_cast<uint32_t>(a.U), scratch, a.co);
  } else {
    unit_sort_tail(rid, rw, cnt, a.E, a.K, blockIdx.x, t0, t1, scratch, a.uo, a.U);
    if (tid == 0) a.uo.unit_flags[blockIdx.x] = bad;
  }
}

size_t unit_kernel_smem(int E, int max_routes, bool cluster) {
  const size_t tail = cluster ? cluster_scratch_bytes(E) : unit_scratch_bytes(E);
  return 2 * align16(sizeof(int32_t) * max_routes) + align16(sizeof(int32_t) * (E + 1)) + tail;
}

cudaError_t launch_unit(const UnitArgs& a, cudaStream_t st) {
  const size_t smem = unit_kernel_smem(a.E, a.max_routes, a.cluster);
  auto* kern = a.cluster ? mrs_unit_kernel<true> : mrs_unit_kernel<false>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  if (!a.cluster) return launch_pdl(kern, dim3(a.U), dim3(kUnitThreads), smem, st, a);
  err = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.U);
  cfg.blockDim = dim3(kUnitThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = a.U;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

// ------------------------------------------------------------------ phase 2: slices
constexpr unsigned long long kFlagReady = 1ull << 32;  // low word = the slice's padded rows

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}


// Moves each placed route of unit u's sorted list to row = offset(expert, unit) + position.
__device__ __forceinline__ void scatter_unit(const SliceArgs& a, int u, int tid, int nthreads) {
  int t0, t1;
  unit_range(u, a.T, a.U, t0, t1);
  const size_t r0 = static_cast<size_t>(t0) * a.K;
  const int n = a.loc_off[static_cast<size_t>(u) * (a.E + 1) + a.E];  // routes placed
  for (int p = tid; p < n; p += nthreads) {
    const int2 v = a.unit_buf[r0 + p];
    const int dst = a.adj[static_cast<size_t>(a.unit_e[r0 + p]) * a.U + u] + p;
    a.sorted_ids[dst] = v.x;
    a.sorted_w[dst] = __int_as_float(v.y);
  }
}

size_t slices_smem_bytes(int U, int E, int nslices);

__global__ void __launch_bounds__(kSliceThreads) mrs_slices_kernel(const SliceArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int c = blockIdx.x;
  const int e0 = static_cast<int>(static_cast<long long>(c) * a.E / a.nslices);
  const int e1 = static_cast<int>(static_cast<long long>(c + 1) * a.E / a.nslices);
  const int ns = e1 - e0;
  const int U = a.U, B = a.B;
  const int SU = U | 1;  // row stride of locs and seg (odd: conflict-free columns)
  int32_t* locs = reinterpret_cast<int32_t*>(smem);                  // [ns + 1][SU] (by expert)
  int32_t* seg = locs + static_cast<size_t>(ns + 1) * SU;            // [ns][SU] starts
  int32_t* tot = seg + static_cast<size_t>(ns) * SU;                 // [ns + 1] unpadded prefix
  int32_t* soff = tot + ns + 1;                                       // [ns + 1] padded prefix
  __shared__ int32_t base_s, flags_s;

  // everything below reads what the previous kernel wrote
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid == 0) {
    base_s = 0;
    flags_s = 0;
  }
  // the slice's columns of the per-unit offsets, stored by expert: lane i reads column
  // e0 + i of units warp, warp + 16, ... with all its loads in flight at once
  for (int i0 = 0; i0 <= ns; i0 += 32) {
    const int i = i0 + lane;
    for (int ub = 0; ub < U; ub += 16 * kSliceWarps) {
      int v[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int u = ub + warp + k * kSliceWarps;
        if (i <= ns && u < U) v[k] = a.loc_off[static_cast<size_t>(u) * (a.E + 1) + e0 + i];
      }
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int u = ub + warp + k * kSliceWarps;
        if (i <= ns && u < U) locs[i * SU + u] = v[k];
      }
    }
  }
  __syncthreads();
  // per expert of the slice (warp per expert): exclusive prefix over units of its counts;
  // lane l sums a run of consecutive units, one warp scan joins the runs
  {
    const int per = (U + 31) / 32;
    const int ulo = min(U, lane * per), uhi = min(U, ulo + per);
    for (int i = warp; i < ns; i += nwarps) {
      const int* lo = locs + i * SU;
      const int* hi = locs + (i + 1) * SU;
      int sum = 0;
      for (int u = ulo; u < uhi; ++u) sum += hi[u] - lo[u];
      const int incl = warp_inclusive_sum(sum, lane);
      int r = incl - sum;
      for (int u = ulo; u < uhi; ++u) {
        seg[i * SU + u] = r;
        r += hi[u] - lo[u];
      }
      if (lane == 31) tot[i] = incl;  // the expert's count, for now
    }
  }
  __syncthreads();
  // unpadded and padded prefixes over the slice's experts (one warp)
  if (warp == 0) {
    int run = 0, prun = 0;
    for (int i0 = 0; i0 < ns; i0 += 32) {
      const int i = i0 + lane;
      const int cnt = (i < ns) ? tot[i] : 0;
      const int pad = (cnt + B - 1) & ~(B - 1);
      const int ci = warp_inclusive_sum(cnt, lane);
      const int pi = warp_inclusive_sum(pad, lane);
      __syncwarp();
      if (i < ns) {
        tot[i] = run + ci - cnt;
        soff[i] = prun + pi - pad;
      }
      run += __shfl_sync(kFull, ci, 31);
      prun += __shfl_sync(kFull, pi, 31);
    }
    if (lane == 0) {
      tot[ns] = run;
      soff[ns] = prun;
      // publish this slice's padded size for the slices after it (the word is all they
      // read from this slice, so no ordering with other memory is needed); an atomic
      // exchange is performed at L2 at once, where the polls look
      atomicExch(&a.slice_flags[c], kFlagReady | static_cast<uint32_t>(prun));
    }
  }
  // this slice's first row = sum of the padded sizes of all earlier slices: warp 0 polls
  // all their words at once (lane l holds slices l, l + 32, ...; bounded wait)
  // (a wait limit of 0, a test hook, gives up at once: every slice but the first reports a
  // timeout and sums nothing, so its rows start too low but stay inside the buffers)
  if (warp == 0) {
    const unsigned long long t_start = globaltimer_ns();
    unsigned long long f[kMaxSlices / 32];
    bool ok = true;
    if (a.wait_limit_ns == 0ull) {
#pragma unroll
      for (int k = 0; k < kMaxSlices / 32; ++k) f[k] = 0ull;
      ok = (c == 0);
    } else {
      for (;;) {
        bool missing = false;
#pragma unroll
        for (int k = 0; k < kMaxSlices / 32; ++k) {
          const int p = lane + 32 * k;
          f[k] = (p < c) ? ld_relaxed_u64(&a.slice_flags[p]) : kFlagReady;
          missing |= (f[k] & kFlagReady) == 0ull;
        }
        if (!__any_sync(kFull, missing)) break;
        if (globaltimer_ns() - t_start > a.wait_limit_ns) {
          ok = false;
          break;
        }
      }
    }
    int v = 0;
#pragma unroll
    for (int k = 0; k < kMaxSlices / 32; ++k)
      v += (lane + 32 * k < c && (f[k] & kFlagReady)) ? static_cast<int>(f[k] & 0xffffffffull)
                                                       : 0;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(kFull, v, d);
    if (lane == 0) {
      base_s = v;
      flags_s = ok ? 0 : MOE_RS_DEVICE_WAIT_TIMEOUT;
    }
  }
  __syncthreads();
  const int base = base_s;
  // (expert, unit) pairs with routes: final row of the first one, minus its list position
  for (int i = warp; i < ns; i += nwarps) {
    int32_t* adj = a.adj + static_cast<size_t>(e0 + i) * U;
    const int b_i = base + soff[i];
    for (int u = lane; u < U; u += 32) {
      const int l0 = locs[i * SU + u];
      if (locs[(i + 1) * SU + u] > l0) adj[u] = b_i + seg[i * SU + u] - l0;
    }
  }
  // padding rows and block owners
  for (int i = warp; i < ns; i += nwarps) {
    const int cnt = tot[i + 1] - tot[i];
    if (cnt == 0) continue;
    const int off = base + soff[i];
    const int pad = (cnt + B - 1) & ~(B - 1);
    for (int p = off + cnt + lane; p < off + pad; p += 32) {
      a.sorted_ids[p] = a.N;
      a.sorted_w[p] = 0.0f;
    }
    for (int b = off / B + lane; b < (off + pad) / B; b += 32) a.expert_ids[b] = e0 + i;
  }
  if (c == a.nslices - 1 && warp == 0) {
    int f = 0;
    for (int v = lane; v < U; v += 32) f |= a.unit_flags[v];
    f = __reduce_or_sync(kFull, f);
    if (lane == 0) {
      *a.npp = base + soff[ns];
      if (f) atomicOr(a.status, f);
    }
  }
  if (flags_s != 0 && tid == 0) atomicOr(a.status, flags_s);
}

// ------------------------------------------------------------------ phase 2b: scatter
__global__ void __launch_bounds__(kSliceThreads) mrs_scatter_kernel(const SliceArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  scatter_unit(a, blockIdx.x, threadIdx.x, blockDim.x);
}



size_t slices_smem_bytes(int U, int E, int nslices) {
  const int ns = (E + nslices - 1) / nslices;
  const size_t SU = static_cast<size_t>(U | 1);
  return sizeof(int32_t) * ((ns + 1) * SU + ns * SU + 2 * static_cast<size_t>(ns) + 2);
}

cudaError_t launch_slices(const SliceArgs& a, cudaStream_t st) {
  const size_t smem = slices_smem_bytes(a.U, a.E, a.nslices);
  cudaError_t err = cudaFuncSetAttribute(mrs_slices_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.nslices);
  cfg.blockDim = dim3(kSliceThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mrs_slices_kernel, a);
}

cudaError_t launch_scatter(const SliceArgs& a, cudaStream_t st) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.U);
  cfg.blockDim = dim3(kSliceThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mrs_scatter_kernel, a);
}

// ------------------------------------------------------------------ empty call
__global__ void mrs_empty_kernel(int32_t* npp, int32_t* status) {
  pdl_wait();
  *npp = 0;
  if (status) *status = 0;
}

cudaError_t launch_empty(int32_t* npp, int32_t* status, cudaStream_t st) {
  return launch_pdl(mrs_empty_kernel, dim3(1), dim3(1), 0, st, npp, status);
}

}  // namespace mrs
