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
// the sorted (flat index, weight) list.  It also clears the look-back flags of phase 2.
//
// Phase 2 (mrs_slices_kernel) gives every CTA a slice of experts: a prefix over units of
// the slice's counts, the block_m-padded offsets inside the slice, a decoupled look-back
// over slices for the slice's base row, then a copy of every (unit, expert) segment to its
// final rows, the padding rows and the per-block expert ids.  Entries of one expert stay in
// token-then-slot order by construction; no global atomics are used, and every wait is
// bounded.
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
  unit_sort_tail(rid, rw, cnt, a.E, a.K, blockIdx.x, t0, t1, scratch, a.loc_off, a.unit_buf,
                 a.slice_flags, a.nslices, a.U);
  if (tid == 0) a.unit_flags[blockIdx.x] = bad;
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
constexpr unsigned long long kFlagAgg = 1ull << 32;  // value = the slice's padded rows
constexpr unsigned long long kFlagInc = 2ull << 32;  // value = rows up to and including it
constexpr unsigned long long kFlagErr = 1ull << 40;  // a wait before this slice gave up
constexpr unsigned long long kFlagState = 3ull << 32;

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
  const int U = a.U, K = a.K, B = a.B;
  int32_t* locs = reinterpret_cast<int32_t*>(smem);                      // [U][ns + 1]
  int32_t* ex = locs + static_cast<size_t>(U) * (ns + 1);                 // [U][ns]
  int32_t* tot = ex + static_cast<size_t>(U) * ns;                        // [ns]
  int32_t* soff = tot + ns;                                               // [ns + 1]
  __shared__ int32_t base_s, flags_s;

  // everything below reads what the previous kernel wrote
  asm volatile("griddepcontrol.wait;" ::: "memory");

  for (int idx = tid; idx < U * (ns + 1); idx += blockDim.x) {
    const int u = idx / (ns + 1), i = idx - u * (ns + 1);
    locs[idx] = a.loc_off[static_cast<size_t>(u) * (a.E + 1) + e0 + i];
  }
  if (tid == 0) flags_s = 0;
  __syncthreads();
  // prefix over units of each expert's counts: warp per expert, lanes over runs of units
  for (int i = warp; i < ns; i += nwarps) {
    const int per = (U + 31) / 32;
    const int ulo = min(U, lane * per), uhi = min(U, ulo + per);
    int s = 0;
    for (int u = ulo; u < uhi; ++u) s += locs[u * (ns + 1) + i + 1] - locs[u * (ns + 1) + i];
    const int incl = warp_inclusive_sum(s, lane);
    int r = incl - s;
    for (int u = ulo; u < uhi; ++u) {
      ex[u * ns + i] = r;
      r += locs[u * (ns + 1) + i + 1] - locs[u * (ns + 1) + i];
    }
    if (lane == 31) tot[i] = incl;
  }
  __syncthreads();
  // padded offsets inside the slice (one warp; slices hold few experts)
  if (warp == 0) {
    int run = 0;
    for (int i0 = 0; i0 < ns; i0 += 32) {
      const int i = i0 + lane;
      const int p = (i < ns) ? ((tot[i] + B - 1) & ~(B - 1)) : 0;
      const int incl = warp_inclusive_sum(p, lane);
      if (i < ns) soff[i] = run + incl - p;
      run += __shfl_sync(kFull, incl, 31);
    }
    if (lane == 0) soff[ns] = run;
  }
  __syncthreads();
  // decoupled look-back over slices for this slice's first row, one warp reading 32
  // predecessor flags per round: the nearest inclusive prefix ends the walk, aggregates in
  // front of it are added.  A timed-out wait marks the flag this slice publishes, so the
  // error reaches the last slice (the status word's writer).
  if (warp == 0) {
    const uint32_t mine = static_cast<uint32_t>(soff[ns]);
    int base = 0;
    unsigned long long err = 0ull;
    if (c == 0) {
      if (lane == 0) st_release_u64(&a.slice_flags[0], kFlagInc | mine);
    } else {
      if (lane == 0) st_release_u64(&a.slice_flags[c], kFlagAgg | mine);
      const unsigned long long t_start = globaltimer_ns();
      int hi = c - 1;  // next predecessor to read
      while (hi >= 0) {
        const int p = hi - lane;
        const unsigned long long f = (p >= 0) ? ld_acquire_u64(&a.slice_flags[p]) : kFlagAgg;
        const unsigned long long state = f & kFlagState;
        const unsigned inc = __ballot_sync(kFull, p >= 0 && state == kFlagInc);
        const unsigned none = __ballot_sync(kFull, p >= 0 && state == 0ull);
        // lanes up to the nearest inclusive flag are the ones that count this round
        const int stop = inc ? __ffs(inc) - 1 : 31;
        const unsigned upto = (stop == 31) ? kFull : ((2u << stop) - 1u);
        if ((none & upto) != 0u) {  // a needed predecessor has not published yet
          if (globaltimer_ns() - t_start > kWaitLimitNs) {
            err = kFlagErr;
            break;
          }
          continue;
        }
        const bool take = p >= 0 && lane <= stop;
        int v = take ? static_cast<int>(f & 0xffffffffull) : 0;
        unsigned long long ev = take ? (f & kFlagErr) : 0ull;
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
          v += __shfl_xor_sync(kFull, v, d);
          ev |= __shfl_xor_sync(kFull, ev, d);
        }
        base += v;
        err |= ev;
        if (inc) break;
        hi -= 32;
      }
      if (lane == 0)
        st_release_u64(&a.slice_flags[c], kFlagInc | err | static_cast<uint32_t>(base + mine));
    }
    if (lane == 0) {
      base_s = base;
      flags_s = err ? MOE_RS_DEVICE_WAIT_TIMEOUT : 0;
    }
  }
  __syncthreads();
  const int base = base_s;
  // copy every (unit, expert) segment to its rows
  for (int idx = tid; idx < U * ns; idx += blockDim.x) {
    const int u = idx / ns, i = idx - u * ns;
    const int lo = locs[u * (ns + 1) + i], n = locs[u * (ns + 1) + i + 1] - lo;
    if (n == 0) continue;
    int t0, t1;
    unit_range(u, a.T, U, t0, t1);
    const int2* __restrict__ src = a.unit_buf + static_cast<size_t>(t0) * K + lo;
    int32_t* __restrict__ dids = a.sorted_ids + base + soff[i] + ex[idx];
    float* __restrict__ dw = a.sorted_w + base + soff[i] + ex[idx];
#pragma unroll 4
    for (int k = 0; k < n; ++k) {
      const int2 v = src[k];
      dids[k] = v.x;
      dw[k] = __int_as_float(v.y);
    }
  }
  // padding rows and block owners
  for (int i = warp; i < ns; i += nwarps) {
    const int cnt = tot[i];
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

size_t slices_smem_bytes(int U, int E, int nslices) {
  const int ns = (E + nslices - 1) / nslices;
  return sizeof(int32_t) * (static_cast<size_t>(U) * (ns + 1) + static_cast<size_t>(U) * ns +
                            2 * static_cast<size_t>(ns) + 1);
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
