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
#include "mrs_unit.cuh"
#include "moe_route_sort.h"

namespace mrs {

// ------------------------------------------------- phase 1 for moe_sort (given routes)
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
  unit_sort_tail(rid, rw, cnt, a.E, a.K, blockIdx.x, t0, t1, scratch, a.uo, a.U);
  if (tid == 0) a.uo.unit_flags[blockIdx.x] = bad;
}

size_t unit_kernel_smem(int E, int max_routes) {
  return 2 * align16(sizeof(int32_t) * max_routes) + align16(sizeof(int32_t) * (E + 1)) +
         unit_scratch_bytes(E);
}

cudaError_t launch_unit(const UnitArgs& a, cudaStream_t st) {
  const size_t smem = unit_kernel_smem(a.E, a.max_routes);
  cudaError_t err = cudaFuncSetAttribute(mrs_unit_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  mrs_unit_kernel<<<a.U, kUnitThreads, smem, st>>>(a);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ phase 2: slices
constexpr unsigned long long kFlagReady = 1ull << 32;  // low word = the slice's padded rows

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__global__ void __launch_bounds__(kSliceThreads) mrs_slices_kernel(const SliceArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int c = blockIdx.x;
  const int e0 = static_cast<int>(static_cast<long long>(c) * a.E / a.nslices);
  const int e1 = static_cast<int>(static_cast<long long>(c + 1) * a.E / a.nslices);
  const int ns = e1 - e0;
  const int U = a.U, B = a.B;
  int32_t* locs = reinterpret_cast<int32_t*>(smem);                  // [U][ns + 1]
  int32_t* seg = locs + static_cast<size_t>(U) * (ns + 1);            // [ns][U + 1] starts
  int32_t* tot = seg + static_cast<size_t>(ns) * (U + 1);             // [ns + 1] unpadded prefix
  int32_t* soff = tot + ns + 1;                                       // [ns + 1] padded prefix
  __shared__ int32_t base_s, flags_s;

  // everything below reads what the previous kernel wrote
  asm volatile("griddepcontrol.wait;" ::: "memory");

  for (int idx = tid; idx < U * (ns + 1); idx += blockDim.x) {
    const int u = idx / (ns + 1), i = idx - u * (ns + 1);
    locs[idx] = a.loc_off[static_cast<size_t>(u) * (a.E + 1) + e0 + i];
  }
  __syncthreads();
  // per expert of the slice: exclusive prefix over units of its counts (warp per expert)
  for (int i = warp; i < ns; i += nwarps) {
    const int per = (U + 31) / 32;
    const int ulo = min(U, lane * per), uhi = min(U, ulo + per);
    int sum = 0;
    for (int u = ulo; u < uhi; ++u) sum += locs[u * (ns + 1) + i + 1] - locs[u * (ns + 1) + i];
    const int incl = warp_inclusive_sum(sum, lane);
    int r = incl - sum;
    for (int u = ulo; u < uhi; ++u) {
      seg[i * (U + 1) + u] = r;
      r += locs[u * (ns + 1) + i + 1] - locs[u * (ns + 1) + i];
    }
    if (lane == 31) seg[i * (U + 1) + U] = incl;
  }
  __syncthreads();
  // unpadded and padded prefixes over the slice's experts (one warp)
  if (warp == 0) {
    int run = 0, prun = 0;
    for (int i0 = 0; i0 < ns; i0 += 32) {
      const int i = i0 + lane;
      const int cnt = (i < ns) ? seg[i * (U + 1) + U] : 0;
      const int pad = (cnt + B - 1) & ~(B - 1);
      const int ci = warp_inclusive_sum(cnt, lane);
      const int pi = warp_inclusive_sum(pad, lane);
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
      flags_s = 0;
    }
  }
  __syncthreads();
  // this slice's first row = sum of the padded sizes of all earlier slices: publish mine,
  // then read every earlier slice's word in parallel (one warp; bounded wait)
  if (warp == 0) {
    if (lane == 0) st_release_u64(&a.slice_flags[c], kFlagReady | static_cast<uint32_t>(soff[ns]));
    int base = 0;
    bool ok = true;
    const unsigned long long t_start = globaltimer_ns();
    for (int p0 = 0; p0 < c; p0 += 32) {
      const int p = p0 + lane;
      unsigned long long f = 0ull;
      for (;;) {
        f = (p < c) ? ld_acquire_u64(&a.slice_flags[p]) : kFlagReady;
        const bool missing = (f & kFlagReady) == 0ull;
        if (!__any_sync(kFull, missing)) break;
        if (globaltimer_ns() - t_start > kWaitLimitNs) {
          ok = false;
          break;
        }
      }
      if (!ok) break;
      int v = (p < c) ? static_cast<int>(f & 0xffffffffull) : 0;
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(kFull, v, d);
      base += v;
    }
    if (lane == 0) {
      base_s = base;
      flags_s = ok ? 0 : MOE_RS_DEVICE_WAIT_TIMEOUT;
    }
  }
  __syncthreads();
  const int base = base_s;
  // (unit, expert) pairs with routes: final row of the first one, minus its list position
  for (int idx = tid; idx < U * ns; idx += blockDim.x) {
    const int u = idx / ns, i = idx - u * ns;
    const int l0 = locs[u * (ns + 1) + i];
    if (locs[u * (ns + 1) + i + 1] > l0)
      a.adj[static_cast<size_t>(u) * a.E + e0 + i] = base + soff[i] + seg[i * (U + 1) + u] - l0;
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
    f = __reduce_or_sync(kFull, f) | flags_s;
    if (lane == 0) {
      *a.npp = base + soff[ns];
      *a.status = f;
    }
  }
}

// ------------------------------------------------------------------ phase 2b: scatter
__global__ void __launch_bounds__(kSliceThreads) mrs_scatter_kernel(const SliceArgs a) {
  const int u = blockIdx.x;
  int t0, t1;
  unit_range(u, a.T, a.U, t0, t1);
  const size_t r0 = static_cast<size_t>(t0) * a.K;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int n = a.loc_off[static_cast<size_t>(u) * (a.E + 1) + a.E];  // routes placed
  const int32_t* adj = a.adj + static_cast<size_t>(u) * a.E;
  for (int p = threadIdx.x; p < n; p += blockDim.x) {
    const int2 v = a.unit_buf[r0 + p];
    const int dst = adj[a.unit_e[r0 + p]] + p;
    a.sorted_ids[dst] = v.x;
    a.sorted_w[dst] = __int_as_float(v.y);
  }
}

size_t slices_smem_bytes(int U, int E, int nslices) {
  const int ns = (E + nslices - 1) / nslices;
  return sizeof(int32_t) * (static_cast<size_t>(U) * (ns + 1) +
                            static_cast<size_t>(ns) * (U + 1) + 2 * static_cast<size_t>(ns) + 2);
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
  *npp = 0;
  if (status) *status = 0;
}

cudaError_t launch_empty(int32_t* npp, int32_t* status, cudaStream_t st) {
  mrs_empty_kernel<<<1, 1, 0, st>>>(npp, status);
  return cudaGetLastError();
}

}  // namespace mrs
