// mrs_sort.cu -- sort phases of the multi-CTA MoE route-sort path for sm_103a.
//
// Both sort phases ("perf(flydsl): Kimi-K3 B1 route-sort + prepared-MoE handoff (stack)",
// Summary) over units: unit u = the routes of a contiguous token range, one CTA each.
//   count   (moe_sort only) per-unit histogram in shared memory -> partial[u][e]
//   scan    per 32-expert chunk: exclusive prefix of partial over units (in place), the
//           expert totals, block_m-padded offsets inside the chunk and the chunk totals
//   scatter per unit: global offsets = prefix of chunk totals + in-chunk offset + the unit's
//           prefix; stable ranks inside the unit from 64-token bitmasks; padding rows and
//           per-block expert ids for a slice of the experts; npp and the status word
// Order inside each expert segment is token-then-slot, independent of scheduling: no
// global atomics anywhere.  Dropped routes (negative ids) claim no slot ("Summary --
// general gfx1250 ordinary-TP route optimization", Dispatch and contracts).
#include "mrs_internal.h"
#include "../../include/moe_route_sort.h"

namespace mrs {

__device__ __forceinline__ void unit_range(int u, int T, int U, int& t0, int& t1) {
  t0 = static_cast<int>(static_cast<long long>(u) * T / U);
  t1 = static_cast<int>(static_cast<long long>(u + 1) * T / U);
}

// ------------------------------------------------------------------------ count
__global__ void __launch_bounds__(512) mrs_count_kernel(const CountArgs a) {
  extern __shared__ __align__(16) int32_t cnts[];  // [E] + flag
  const int tid = threadIdx.x;
  int32_t* flag = cnts + a.E;
  for (int e = tid; e < a.E; e += blockDim.x) cnts[e] = 0;
  if (tid == 0) *flag = 0;
  __syncthreads();
  int t0, t1;
  unit_range(blockIdx.x, a.T, a.U, t0, t1);
  const size_t r0 = static_cast<size_t>(t0) * a.K, r1 = static_cast<size_t>(t1) * a.K;
  for (size_t r = r0 + tid; r < r1; r += blockDim.x) {
    const int e = a.ids[r];
    if (e >= a.E) {
      *flag = MOE_RS_DEVICE_BAD_EXPERT_ID;
    } else if (e >= 0) {
      atomicAdd(&cnts[e], 1);
    }
  }
  __syncthreads();
  for (int e = tid; e < a.E; e += blockDim.x)
    a.partial[static_cast<size_t>(blockIdx.x) * a.E + e] = cnts[e];
  if (tid == 0) a.unit_flags[blockIdx.x] = *flag;
}

cudaError_t launch_count(const CountArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(int32_t) * (a.E + 1);
  mrs_count_kernel<<<a.U, 512, smem, st>>>(a);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------- scan
// Block of 32 warps; lane = expert inside the chunk, warp w = a contiguous run of units.
__global__ void __launch_bounds__(1024) mrs_scan_kernel(const ScanArgs a) {
  __shared__ int32_t part[32][33];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e = blockIdx.x * kChunk + lane;
  const bool valid = e < a.E;
  const int u0 = static_cast<int>(static_cast<long long>(warp) * a.U / 32);
  const int u1 = static_cast<int>(static_cast<long long>(warp + 1) * a.U / 32);
  int sum = 0;
  if (valid)
    for (int u = u0; u < u1; ++u) sum += a.partial[static_cast<size_t>(u) * a.E + e];
  part[warp][lane] = sum;
  __syncthreads();
  if (warp == 0) {
    int run = 0;
    for (int w = 0; w < 32; ++w) {
      const int v = part[w][lane];
      part[w][lane] = run;
      run += v;
    }
    const int pad = valid ? ((run + a.B - 1) & ~(a.B - 1)) : 0;
    const int incl = warp_inclusive_sum(pad, lane);
    if (valid) {
      a.cnt_tot[e] = run;
      a.inchunk_off[e] = incl - pad;
    }
    if (lane == 31) a.chunk_tot[blockIdx.x] = incl;
  }
  __syncthreads();
  if (valid) {
    int run = part[warp][lane];
    for (int u = u0; u < u1; ++u) {
      const size_t i = static_cast<size_t>(u) * a.E + e;
      const int v = a.partial[i];
      a.partial[i] = run;
      run += v;
    }
  }
}

cudaError_t launch_scan(const ScanArgs& a, cudaStream_t st) {
  const int nchunk = (a.E + kChunk - 1) / kChunk;
  mrs_scan_kernel<<<nchunk, 1024, 0, st>>>(a);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------- scatter
__global__ void __launch_bounds__(512) mrs_scatter_kernel(const ScatterArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int E = a.E, K = a.K, B = a.B;
  unsigned long long* masks = reinterpret_cast<unsigned long long*>(smem);  // [E]
  int32_t* base = reinterpret_cast<int32_t*>(smem + align16(sizeof(unsigned long long) * E));
  int32_t* cpre = base + E;              // [kMaxChunks + 1]
  int32_t* flag = cpre + kMaxChunks + 1;  // [1]

  // global chunk offsets: exclusive prefix of the chunk totals (<= 128 chunks)
  if (warp == 0) {
    int v[4];
    int s = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = lane * 4 + i;
      v[i] = (c < a.nchunk) ? a.chunk_tot[c] : 0;
      s += v[i];
    }
    const int incl = warp_inclusive_sum(s, lane);
    int run = incl - s;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      cpre[lane * 4 + i] = run;
      run += v[i];
    }
    if (lane == 31) cpre[kMaxChunks] = incl;
  }
  if (tid == 0) *flag = 0;
  __syncthreads();
  const int u = blockIdx.x;
  for (int e = tid; e < E; e += blockDim.x) {
    base[e] = cpre[e / kChunk] + a.inchunk_off[e] + a.partial[static_cast<size_t>(u) * E + e];
    masks[e] = 0ull;
  }
  __syncthreads();

  int t0, t1;
  unit_range(u, a.T, a.U, t0, t1);
  for (int tt = t0; tt < t1; tt += kTileTokens) {
    const int nt = min(kTileTokens, t1 - tt);
    const int nr = nt * K;
    const size_t r0 = static_cast<size_t>(tt) * K;
    for (int i = tid; i < nr; i += blockDim.x) {
      const int e = a.ids[r0 + i];
      if (e < 0 || e >= E) continue;
      const unsigned long long bit = 1ull << (i / K);
      const unsigned long long old = atomicOr(&masks[e], bit);
      if (old & bit) *flag = 1;  // the same expert twice in one token
    }
    __syncthreads();
    if (*flag == 0) {
      for (int i = tid; i < nr; i += blockDim.x) {
        const size_t r = r0 + i;
        const int e = a.ids[r];
        if (e < 0 || e >= E) continue;
        const int tl = i / K;
        const int pos = base[e] + __popcll(masks[e] & ((1ull << tl) - 1ull));
        a.sorted_ids[pos] = static_cast<int32_t>(r);
        a.sorted_w[pos] = a.w[r];
      }
      __syncthreads();
      for (int i = tid; i < nr; i += blockDim.x) {
        const int e = a.ids[r0 + i];
        if (e < 0 || e >= E) continue;
        const unsigned long long m = masks[e];
        if ((m >> (i / K)) == 1ull) {  // last token of the tile routed to e
          base[e] += __popcll(m);
          masks[e] = 0ull;
        }
      }
      __syncthreads();
    } else {
      // repeated ids inside a token: rank this tile's routes in flat order, 32 at a time
      for (int i = tid; i < nr; i += blockDim.x) {
        const int e = a.ids[r0 + i];
        if (e >= 0 && e < E) masks[e] = 0ull;
      }
      __syncthreads();
      if (warp == 0) {
        for (int b0 = 0; b0 < nr; b0 += 32) {
          const int i = b0 + lane;
          const size_t r = r0 + i;
          const int e = (i < nr) ? a.ids[r] : -1;
          const bool valid = (e >= 0) && (e < E);
          const unsigned peers = __match_any_sync(kFull, valid ? e : -1 - lane);
          int p0 = 0;
          if (valid) {
            p0 = base[e];
            const int pos = p0 + __popc(peers & lanemask_lt(lane));
            a.sorted_ids[pos] = static_cast<int32_t>(r);
            a.sorted_w[pos] = a.w[r];
          }
          __syncwarp();
          if (valid && (peers >> lane) == 1u) base[e] = p0 + __popc(peers);
          __syncwarp();
        }
      }
      __syncthreads();
      if (tid == 0) *flag = 0;
      __syncthreads();
    }
  }

  // padding rows and block owners for this unit's slice of the experts
  const int e0 = static_cast<int>(static_cast<long long>(u) * E / a.U);
  const int e1 = static_cast<int>(static_cast<long long>(u + 1) * E / a.U);
  for (int e = e0 + warp; e < e1; e += nwarps) {
    const int c = a.cnt_tot[e];
    if (c == 0) continue;
    const int off = cpre[e / kChunk] + a.inchunk_off[e];
    const int pad = (c + B - 1) & ~(B - 1);
    for (int p = off + c + lane; p < off + pad; p += 32) {
      a.sorted_ids[p] = a.N;
      a.sorted_w[p] = 0.0f;
    }
    for (int b = off / B + lane; b < (off + pad) / B; b += 32) a.expert_ids[b] = e;
  }
  if (u == 0 && warp == 0) {
    int f = 0;
    for (int v = lane; v < a.U; v += 32) f |= a.unit_flags[v];
    f = __reduce_or_sync(kFull, f);
    if (lane == 0) {
      *a.npp = cpre[kMaxChunks];
      *a.status = f;
    }
  }
}

cudaError_t launch_scatter(const ScatterArgs& a, cudaStream_t st) {
  const size_t smem = align16(sizeof(unsigned long long) * a.E) +
                      sizeof(int32_t) * (a.E + kMaxChunks + 2);
  cudaError_t err = cudaFuncSetAttribute(
      mrs_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  mrs_scatter_kernel<<<a.U, 512, smem, st>>>(a);
  return cudaGetLastError();
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
