// mrs_route.cu -- route step kernels of MoE route-sort for sm_103a.
//
//  * mrs_small_kernel: the whole path (route step + both sort phases) in one CTA, for
//    decode-sized calls (T <= 64).  Scores of a wave of tokens are computed by the whole
//    CTA, each warp routes one token, then the CTA counts, scans and scatters in shared
//    memory.  No global atomics, one launch.
//  * mrs_route_kernel: the route step of the multi-CTA path.  CTA u owns a contiguous range
//    of tokens (its "unit"); each warp routes one token at a time and, when asked, the CTA
//    counts its routes per expert in shared memory and stores the unit's histogram.
//
// Source: "perf(flydsl): Kimi-K3 B1 route-sort + prepared-MoE handoff (stack)", Summary
// (FP32 logit conversion + correction bias, grouped top-k, both sort phases in one kernel).
#include "mrs_internal.h"
#include "../../include/moe_route_sort.h"

namespace mrs {

// Exclusive prefix sum of the block_m-padded counts over experts, by a 1024-thread block
// (4 consecutive experts per thread).  Returns the total; off[e] receives the prefix.
__device__ __forceinline__ int block_scan_padded(const int* cnt, int* off, int E, int B,
                                                 int* wtot) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int loc[4];
  int s = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = tid * 4 + i;
    const int p = (e < E) ? ((cnt[e] + B - 1) & ~(B - 1)) : 0;
    loc[i] = s;
    s += p;
  }
  const int incl = warp_inclusive_sum(s, lane);
  if (lane == 31) wtot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int v = wtot[lane];
    const int wi = warp_inclusive_sum(v, lane);
    __syncwarp();
    wtot[lane] = wi - v;
    if (lane == 31) wtot[32] = wi;
  }
  __syncthreads();
  const int base = wtot[warp] + incl - s;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = tid * 4 + i;
    if (e < E) off[e] = base + loc[i];
  }
  const int total = wtot[32];
  __syncthreads();
  return total;
}

template <bool kSortOnly>
__global__ void __launch_bounds__(kSmallThreads, 1) mrs_small_kernel(const SmallArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const RouteShape sh = a.sh;
  const int E = sh.E, K = sh.K, N = a.N, B = a.B;
  int32_t* rid = reinterpret_cast<int32_t*>(smem + a.lay.rid);
  float* rw = reinterpret_cast<float*>(smem + a.lay.rw);
  int32_t* cnt = reinterpret_cast<int32_t*>(smem + a.lay.cnt);
  int32_t* off = reinterpret_cast<int32_t*>(smem + a.lay.off);
  int32_t* owner = reinterpret_cast<int32_t*>(smem + a.lay.owner);
  int32_t* misc = reinterpret_cast<int32_t*>(smem + a.lay.misc);  // [0] flags, [4..37] scan

  // ------------------------------------------------------------ route step
  if (!kSortOnly) {
    float* bias_s = reinterpret_cast<float*>(smem + a.lay.bias);
    float* keys = reinterpret_cast<float*>(smem + a.lay.keys);
    float* svals = reinterpret_cast<float*>(smem + a.lay.svals);
    WarpScratch* scr = reinterpret_cast<WarpScratch*>(smem + a.lay.scratch);
    for (int e = tid; e < E; e += blockDim.x) bias_s[e] = a.bias[e];
    __syncthreads();
    for (int t0 = 0; t0 < a.T; t0 += a.wave) {
      const int nt = min(a.wave, a.T - t0);
      for (int tl = 0; tl < nt; ++tl) {
        const uint16_t* row = a.logits + static_cast<size_t>(t0 + tl) * E;
        for (int e = tid; e < E; e += blockDim.x) {
          const float s = exact_score(bf16_bits_to_float(row[e]));
          svals[tl * E + e] = s;
          keys[tl * E + e] = __fadd_rn(s, bias_s[e]);
        }
      }
      __syncthreads();
      if (warp < nt) {
        const SmemExactSrc src{keys + warp * E, svals + warp * E};
        int id;
        float w;
        route_token(src, sh, scr[warp], lane, id, w);
        if (lane < K) {
          const int r = (t0 + warp) * K + lane;
          a.topk_ids[r] = id;
          a.topk_w[r] = w;
          rid[r] = id;
          rw[r] = w;
        }
      }
      __syncthreads();
    }
  } else {
    for (int r = tid; r < N; r += blockDim.x) {
      rid[r] = a.in_ids[r];
      rw[r] = a.in_w[r];
    }
  }

  // ------------------------------------------------------- sort phase 1: counts, ranks
  if (tid == 0) misc[0] = 0;
  for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
  if (!kSortOnly) {
    unsigned long long* masks = reinterpret_cast<unsigned long long*>(smem + a.lay.masks);
    for (int e = tid; e < E; e += blockDim.x) masks[e] = 0ull;
    __syncthreads();
    // experts are distinct within a token: one bit per token gives count and stable rank
    for (int r = tid; r < N; r += blockDim.x) {
      const int e = rid[r];
      if (e >= 0 && e < E) atomicOr(&masks[e], 1ull << (r / K));
    }
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) cnt[e] = __popcll(masks[e]);
  } else {
    int32_t* rrank = reinterpret_cast<int32_t*>(smem + a.lay.rrank);
    __syncthreads();
    if (warp == 0) {
      // ids may repeat inside a token: rank routes in flat order, 32 at a time
      bool bad = false;
      for (int base = 0; base < N; base += 32) {
        const int r = base + lane;
        const int e = (r < N) ? rid[r] : -1;
        const bool valid = (e >= 0) && (e < E);
        bad |= (e >= E);
        const unsigned peers = __match_any_sync(kFull, valid ? e : -1 - lane);
        int c0 = 0;
        if (valid) {
          c0 = cnt[e];
          rrank[r] = c0 + __popc(peers & lanemask_lt(lane));
        }
        __syncwarp();
        if (valid && (peers >> lane) == 1u) cnt[e] = c0 + __popc(peers);
        __syncwarp();
      }
      if (__any_sync(kFull, bad) && lane == 0) misc[0] = MOE_RS_DEVICE_BAD_EXPERT_ID;
    }
  }
  __syncthreads();

  // --------------------------------------------- sort phase 2: padded scan and scatter
  const int total = block_scan_padded(cnt, off, E, B, misc + 4);
  for (int r = tid; r < N; r += blockDim.x) {
    const int e = rid[r];
    if (e < 0 || e >= E) continue;
    int rank;
    if (!kSortOnly) {
      const unsigned long long* masks =
          reinterpret_cast<const unsigned long long*>(smem + a.lay.masks);
      rank = __popcll(masks[e] & ((1ull << (r / K)) - 1ull));
    } else {
      rank = reinterpret_cast<const int32_t*>(smem + a.lay.rrank)[r];
    }
    const int pos = off[e] + rank;
    a.sorted_ids[pos] = r;
    a.sorted_w[pos] = rw[r];
  }
  for (int e = tid; e < E; e += blockDim.x) {
    const int c = cnt[e];
    if (c == 0) continue;
    const int p = (c + B - 1) & ~(B - 1);
    for (int b = off[e] / B; b < (off[e] + p) / B; ++b) owner[b] = e;
  }
  __syncthreads();
  for (int p = tid; p < total; p += blockDim.x) {
    const int e = owner[p / B];
    if (p - off[e] >= cnt[e]) {
      a.sorted_ids[p] = N;
      a.sorted_w[p] = 0.0f;
    }
  }
  for (int b = tid; b < total / B; b += blockDim.x) a.expert_ids[b] = owner[b];
  if (tid == 0) {
    *a.npp = total;
    *a.status = misc[0];
  }
}

SmallLayout small_layout(int E, int N, int wave, int nb_max, bool sort_only) {
  SmallLayout l{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const int at = static_cast<int>(o);
    o = align16(o + bytes);
    return at;
  };
  l.bias = sort_only ? 0 : take(sizeof(float) * E);
  l.keys = sort_only ? 0 : take(sizeof(float) * (size_t)wave * E);
  l.svals = sort_only ? 0 : take(sizeof(float) * (size_t)wave * E);
  l.scratch = sort_only ? 0 : take(sizeof(WarpScratch) * (size_t)wave);
  l.rid = take(sizeof(int32_t) * N);
  l.rw = take(sizeof(float) * N);
  l.rrank = sort_only ? take(sizeof(int32_t) * N) : 0;
  l.cnt = take(sizeof(int32_t) * E);
  l.off = take(sizeof(int32_t) * E);
  l.masks = sort_only ? 0 : take(sizeof(unsigned long long) * E);
  l.owner = take(sizeof(int32_t) * (nb_max > 0 ? nb_max : 1));
  l.misc = take(sizeof(int32_t) * 40);
  l.total = static_cast<int>(o);
  return l;
}

cudaError_t launch_small(const SmallArgs& a, bool sort_only, cudaStream_t st) {
  const size_t smem = static_cast<size_t>(a.lay.total);
  cudaError_t err;
  if (sort_only) {
    err = cudaFuncSetAttribute(mrs_small_kernel<true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    mrs_small_kernel<true><<<1, kSmallThreads, smem, st>>>(a);
  } else {
    err = cudaFuncSetAttribute(mrs_small_kernel<false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    mrs_small_kernel<false><<<1, kSmallThreads, smem, st>>>(a);
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------------ multi-CTA route
size_t route_smem_bytes(int E, int nwarps, bool with_hist) {
  const size_t per_warp = align16(sizeof(float) * 2 * (size_t)E) + sizeof(WarpScratch);
  return align16(sizeof(float) * E) + (with_hist ? align16(sizeof(int32_t) * E) : 0) +
         per_warp * nwarps;
}

template <bool kHist>
__global__ void __launch_bounds__(512) mrs_route_kernel(const RouteArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const RouteShape sh = a.sh;
  const int E = sh.E, K = sh.K;
  float* bias_s = reinterpret_cast<float*>(smem);
  size_t o = align16(sizeof(float) * E);
  int32_t* counts = reinterpret_cast<int32_t*>(smem + o);
  if (kHist) o += align16(sizeof(int32_t) * E);
  const size_t per_warp = align16(sizeof(float) * 2 * (size_t)E) + sizeof(WarpScratch);
  unsigned char* mine = smem + o + per_warp * warp;
  float* key = reinterpret_cast<float*>(mine);
  float* sv = key + E;
  WarpScratch& scr =
      *reinterpret_cast<WarpScratch*>(mine + align16(sizeof(float) * 2 * (size_t)E));

  for (int e = tid; e < E; e += blockDim.x) {
    bias_s[e] = a.bias[e];
    if (kHist) counts[e] = 0;
  }
  __syncthreads();

  const int u = blockIdx.x;
  const int t0 = static_cast<int>(static_cast<long long>(u) * a.T / a.U);
  const int t1 = static_cast<int>(static_cast<long long>(u + 1) * a.T / a.U);
  for (int t = t0 + warp; t < t1; t += a.nwarps) {
    const uint16_t* row = a.logits + static_cast<size_t>(t) * E;
    if (a.vec16) {
      const uint4* r4 = reinterpret_cast<const uint4*>(row);
      const int nv = E >> 3;
      for (int v = lane; v < nv; v += 32) {
        const uint4 q = __ldcs(r4 + v);
        const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int e = v * 8 + 2 * j;
          const float s0 = exact_score(__uint_as_float(wd[j] << 16));
          const float s1 = exact_score(__uint_as_float(wd[j] & 0xffff0000u));
          sv[e] = s0;
          sv[e + 1] = s1;
          key[e] = __fadd_rn(s0, bias_s[e]);
          key[e + 1] = __fadd_rn(s1, bias_s[e + 1]);
        }
      }
    } else {
      for (int e = lane; e < E; e += 32) {
        const float s = exact_score(bf16_bits_to_float(row[e]));
        sv[e] = s;
        key[e] = __fadd_rn(s, bias_s[e]);
      }
    }
    __syncwarp();
    int id;
    float w;
    route_token(SmemExactSrc{key, sv}, sh, scr, lane, id, w);
    if (lane < K) {
      a.topk_ids[static_cast<size_t>(t) * K + lane] = id;
      a.topk_w[static_cast<size_t>(t) * K + lane] = w;
      if (kHist && id >= 0 && id < E) atomicAdd(&counts[id], 1);
    }
  }
  if (kHist) {
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) a.partial[static_cast<size_t>(u) * E + e] = counts[e];
    if (tid == 0) a.unit_flags[u] = 0;
  }
}

cudaError_t launch_route(const RouteArgs& a, size_t smem, cudaStream_t st) {
  cudaError_t err;
  const int threads = a.nwarps * 32;
  if (a.partial) {
    err = cudaFuncSetAttribute(mrs_route_kernel<true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    mrs_route_kernel<true><<<a.U, threads, smem, st>>>(a);
  } else {
    err = cudaFuncSetAttribute(mrs_route_kernel<false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    mrs_route_kernel<false><<<a.U, threads, smem, st>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace mrs
