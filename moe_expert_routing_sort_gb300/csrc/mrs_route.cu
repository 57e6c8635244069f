// mrs_route.cu -- route step kernels of MoE route-sort for sm_103a.
//
//  * mrs_small_kernel: the whole path (route step + both sort phases) in one CTA for
//    decode-sized calls (T <= 64): one launch, no global atomics, shared-memory histogram.
//    The CTA computes the exact scores of a wave of tokens (one DRAM round trip: 16-byte
//    logit vectors and bias together), each warp routes one token, and the CTA counts,
//    scans and scatters in shared memory.
//  * mrs_route_seg_kernel: route step of the multi-CTA path for shapes whose groups split
//    into equal 4-expert-aligned lane segments (see mrs_seg.cuh).  CTA u owns a contiguous
//    token range (its "unit"); each warp streams its tokens' rows into shared memory with
//    bulk copies (TMA) and routes them with cheap proxy scores plus exact refinement, one
//    or two tokens per warp; the CTA counts its routes per expert for the sort step.
//  * mrs_route_kernel: the same step for any other shape: exact scores of a row into
//    shared memory, then the warp-level route step over them.
//
// Source: "perf(flydsl): Kimi-K3 B1 route-sort + prepared-MoE handoff (stack)", Summary
// (FP32 logit conversion + correction bias, grouped top-k, both sort phases in one kernel).
#include "mrs_internal.h"
#include "mrs_seg.cuh"
#include "mrs_cluster.cuh"
#include "mrs_unit.cuh"
#include "moe_route_sort.h"

namespace mrs {

// Exclusive prefix sum of the block_m-padded counts over experts by the whole block
// (ept = ceil(E / threads) consecutive experts per thread, at most 8).  off[e] receives the
// prefix; returns the total.
template <int kThreads>
__device__ __forceinline__ int block_scan_padded(const int* cnt, int* off, int E, int B,
                                                 int* wtot) {
  constexpr int kWarps = kThreads / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ept = (E + kThreads - 1) / kThreads;
  int loc[8];
  int s = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = tid * ept + i;
    const int p = (i < ept && e < E) ? ((cnt[e] + B - 1) & ~(B - 1)) : 0;
    loc[i] = s;
    s += p;
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
  const int base = wtot[warp] + incl - s;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = tid * ept + i;
    if (i < ept && e < E) off[e] = base + loc[i];
  }
  const int total = wtot[32];
  __syncthreads();  // every off[] is read by other threads next
  return total;
}

// Exact scores and keys of `nt` rows starting at row t0, by the whole block.
__device__ __forceinline__ void small_scores(const SmallArgs& a, int t0, int nt, float* keys,
                                             float* svals) {
  const int E = a.sh.E;
  const bool sm = a.sh.softmax != 0;  // no bias with softmax scoring
  if ((E & 7) == 0) {
    // 16-byte vectors of 8 logits; the matching 8 biases come from global alongside
    const int nv = E >> 3;
    const int total = nt * nv;
    // a 16-byte aligned bias (the usual case) comes as two 16-byte vectors per chunk
    const bool b16 = !sm && (reinterpret_cast<uintptr_t>(a.bias) & 15u) == 0u;
    for (int base = threadIdx.x; base < total; base += kSmallThreads * 4) {
      uint4 q[4];
      float bb[4][8];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int idx = base + u * kSmallThreads;
        if (idx < total) {
          const int tl = idx / nv, v = idx - tl * nv;
          q[u] = reinterpret_cast<const uint4*>(a.logits + static_cast<size_t>(t0 + tl) * E)[v];
          if (b16) {
            const float4 b0 = reinterpret_cast<const float4*>(a.bias)[2 * v];
            const float4 b1 = reinterpret_cast<const float4*>(a.bias)[2 * v + 1];
            bb[u][0] = b0.x;
            bb[u][1] = b0.y;
            bb[u][2] = b0.z;
            bb[u][3] = b0.w;
            bb[u][4] = b1.x;
            bb[u][5] = b1.y;
            bb[u][6] = b1.z;
            bb[u][7] = b1.w;
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) bb[u][j] = sm ? 0.0f : a.bias[8 * v + j];
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int idx = base + u * kSmallThreads;
        if (idx < total) {
          const int tl = idx / nv, v = idx - tl * nv;
          const uint32_t wd[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
          float k8[8], s8[8];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            k8[2 * j] = score_key(__uint_as_float(wd[j] << 16), bb[u][2 * j], sm, s8[2 * j]);
            k8[2 * j + 1] = score_key(__uint_as_float(wd[j] & 0xffff0000u), bb[u][2 * j + 1],
                                      sm, s8[2 * j + 1]);
          }
          // 16-byte stores (E % 8 == 0 keeps every row's 8-key chunks 32-byte aligned): a
          // warp's scalar stores 32 bytes apart would hit only 4 banks
          float4* kr = reinterpret_cast<float4*>(keys + tl * E + 8 * v);
          float4* sr = reinterpret_cast<float4*>(svals + tl * E + 8 * v);
          kr[0] = make_float4(k8[0], k8[1], k8[2], k8[3]);
          kr[1] = make_float4(k8[4], k8[5], k8[6], k8[7]);
          sr[0] = make_float4(s8[0], s8[1], s8[2], s8[3]);
          sr[1] = make_float4(s8[4], s8[5], s8[6], s8[7]);
        }
      }
    }
  } else {
    const int total = nt * E;
    for (int base = threadIdx.x; base < total; base += kSmallThreads * 4) {
      uint16_t x[4];
      float b[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int idx = base + u * kSmallThreads;
        if (idx < total) {
          const int tl = idx / E, e = idx - tl * E;
          x[u] = a.logits[static_cast<size_t>(t0 + tl) * E + e];
          b[u] = sm ? 0.0f : a.bias[e];
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int idx = base + u * kSmallThreads;
        if (idx < total) {
          keys[idx] = score_key(bf16_bits_to_float(x[u]), b[u], sm, svals[idx]);
        }
      }
    }
  }
}

static_assert(sizeof(SegScratch) <= sizeof(WarpScratch), "segment scratch reuses WarpScratch");

// The sort step of a grid-wide call (kGrid below), after this CTA has routed its tokens
// [g0, g0 + gn): rid/rw hold their routes (index (t - g0) * K + k), masks[e] bit t - g0 is set
// for each of them routed to e, and every CTA has written its ids to a.xchg.  After the
// grid-wide barrier (bounded; on a timeout the CTA reports MOE_RS_DEVICE_WAIT_TIMEOUT and
// writes nothing more) each CTA reads all T * K ids, counts them per expert (cnt) and those of
// tokens before g0 (bef), forms the block_m-padded prefix over experts (off), and writes its own
// routes to row off[e] + bef[e] + (its earlier tokens routed to e): token-then-slot order, as a
// token holds each expert at most once.  CTA b of n writes the padding rows and block owners
// of experts [b E / n, (b + 1) E / n), CTA 0 npp; the status word is zeroed by
// mrs_grid_prep_kernel and only ever ORed here.
__device__ __forceinline__ void small_grid_sort(const SmallArgs& a, int g0, int gn,
                                                const int32_t* rid, const float* rw,
                                                const unsigned* masks, int32_t* cnt,
                                                int32_t* bef, int32_t* off, int32_t* misc) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = a.sh.E, K = a.sh.K, B = a.B;
  const int b = static_cast<int>(blockIdx.x), n = static_cast<int>(gridDim.x);
  const int N = a.T * K, nb = g0 * K;
  for (int e = tid; e < E; e += kSmallThreads) {
    cnt[e] = 0;
    bef[e] = 0;
  }
  if (!grid_barrier_bounded(a.bar, static_cast<unsigned>(n), a.wait_limit_ns, misc + 2)) {
    if (tid == 0) atomicOr(a.status, MOE_RS_DEVICE_WAIT_TIMEOUT);
    return;
  }
  // four 16-byte loads per thread in flight (the exchange buffer is 16-byte aligned)
  for (int x0 = 4 * tid; x0 < N; x0 += 16 * kSmallThreads) {
    int v[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int x = x0 + 4 * kSmallThreads * u;
      if (x + 3 < N) {
        const int4 q = __ldcg(reinterpret_cast<const int4*>(a.xchg + x));
        v[u][0] = q.x;
        v[u][1] = q.y;
        v[u][2] = q.z;
        v[u][3] = q.w;
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) v[u][j] = (x + j < N) ? __ldcg(a.xchg + x + j) : -1;
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int x = x0 + 4 * kSmallThreads * u;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = v[u][j];
        if (e >= 0 && e < E) {
          atomicAdd(&cnt[e], 1);
          if (x + j < nb) atomicAdd(&bef[e], 1);
        }
      }
    }
  }
  __syncthreads();
  const int total = block_scan_padded<kSmallThreads>(cnt, off, E, B, misc + 4);
  for (int r = tid; r < gn * K; r += kSmallThreads) {
    const int e = rid[r];
    if (e < 0 || e >= E) continue;
    const int tl = r / K;
    const int pos = off[e] + bef[e] + __popc(masks[e] & ((1u << tl) - 1u));
    a.sorted_ids[pos] = nb + r;
    a.sorted_w[pos] = rw[r];
  }
  const int e0 = static_cast<int>(static_cast<long long>(b) * E / n);
  const int e1 = static_cast<int>(static_cast<long long>(b + 1) * E / n);
  for (int e = e0 + warp; e < e1; e += kSmallThreads / 32) {
    const int c = cnt[e];
    if (c == 0) continue;
    const int o = off[e];
    const int end = o + ((c + B - 1) & ~(B - 1));
    for (int p = o + c + lane; p < end; p += 32) {
      a.sorted_ids[p] = N;
      a.sorted_w[p] = 0.0f;
    }
    for (int q = o / B + lane; q < end / B; q += 32) a.expert_ids[q] = e;
  }
  if (b == 0 && tid == 0) *a.npp = total;
}

// kSeg (route step only): route with the segment routine (a.use_seg), else the generic one;
// one instance per routine, so that a launch fetches and holds only the code it runs.
// kGrid: one CTA of a cooperative grid over a.T tokens; CTA b routes tokens [b * a.per,
// (b + 1) * a.per) (at most one wave), then the grid sorts all routes (small_grid_sort).
template <bool kSortOnly, bool kSeg, bool kGrid>
__global__ void __launch_bounds__(kSmallThreads, 1) mrs_small_kernel(const SmallArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const RouteShape sh = a.sh;
  const int E = sh.E, K = sh.K, N = a.N, B = a.B;
  // the tokens this CTA routes: [g0, g0 + gT)
  const int g0 = kGrid ? static_cast<int>(blockIdx.x) * a.per : 0;
  const int gT = kGrid ? min(a.per, a.T - g0) : a.T;
  int32_t* rid = reinterpret_cast<int32_t*>(smem + a.lay.rid);
  float* rw = reinterpret_cast<float*>(smem + a.lay.rw);
  int32_t* cnt = reinterpret_cast<int32_t*>(smem + a.lay.cnt);
  int32_t* off = reinterpret_cast<int32_t*>(smem + a.lay.off);
  int32_t* misc = reinterpret_cast<int32_t*>(smem + a.lay.misc);  // [0] flags, [4..37] scan
  unsigned* masks = reinterpret_cast<unsigned*>(smem + a.lay.masks);  // [2][E]: tokens 0-31, 32-63
  pdl_trigger();
  // the inputs start towards L2 while the kernel ahead in the stream finishes
  if (!kSortOnly) {
    if (tid < 384)
      prefetch_l2_range(a.logits + static_cast<size_t>(g0) * E, 2 * static_cast<size_t>(gT) * E,
                        tid, 384);
    else if (a.bias)
      prefetch_l2_range(a.bias, 4 * static_cast<size_t>(E), tid - 384, 128);
  }
  pdl_wait();

  if (!kSortOnly) {
    // -------------------------------------------------------------- route step
    float* keys = reinterpret_cast<float*>(smem + a.lay.keys);
    float* svals = reinterpret_cast<float*>(smem + a.lay.svals);
    WarpScratch* scr = reinterpret_cast<WarpScratch*>(smem + a.lay.scratch);
    for (int e = tid; e < (kGrid ? E : 2 * E); e += kSmallThreads) masks[e] = 0u;
    if (kSeg && warp < a.wave)
      ub_init_pads(reinterpret_cast<unsigned short*>(smem + a.lay.umax + ub_bytes(a.seg.nu) * warp),
                   lane, a.seg.nu);
    for (int t0 = 0; t0 < gT; t0 += a.wave) {
      const int nt = min(a.wave, gT - t0);
      small_scores(a, g0 + t0, nt, keys, svals);
      __syncthreads();
      for (int tl = warp; tl < nt; tl += kSmallThreads / 32) {
        int id;
        float w;
        if (kSeg) {
          unsigned short* umax = reinterpret_cast<unsigned short*>(
              smem + a.lay.umax + ub_bytes(a.seg.nu) * warp);
          const ExactKeyRow row{keys + tl * E, svals + tl * E};
          const LaneTop top = seg_pass1<32, 1>(row, a.seg, umax, lane, true);
          seg_select<32, 1>(row, a.seg, *reinterpret_cast<SegScratch*>(&scr[warp]), umax, lane,
                            0.0f, true, top, [] {}, id, w);
        } else {
          route_token(SmemExactSrc{keys + tl * E, svals + tl * E}, sh, scr[warp], lane, id, w);
        }
        if (lane < K) {
          const int t = t0 + tl;  // of this CTA's tokens
          const int r = t * K + lane;
          const int rg = (g0 + t) * K + lane;
          a.topk_ids[rg] = id;
          a.topk_w[rg] = w;
          rid[r] = id;
          rw[r] = w;
          if (kGrid) a.xchg[rg] = id;
          // experts are distinct within a token: one bit per token gives count and rank
          if (id >= 0 && id < E) atomicOr(&masks[(t >> 5) * E + id], 1u << (t & 31));
        }
      }
      __syncthreads();
    }
    if constexpr (kGrid) {
      small_grid_sort(a, g0, gT, rid, rw, masks, cnt,
                      reinterpret_cast<int32_t*>(smem + a.lay.owner), off, misc);
    } else {
      for (int e = tid; e < E; e += kSmallThreads)
        cnt[e] = __popc(masks[e]) + __popc(masks[E + e]);
      if (tid == 0) misc[0] = 0;
      __syncthreads();
    }
  } else {
    // ---------------------------------------- sort step only: ranks in flat route order
    for (int r = tid; r < N; r += kSmallThreads) {
      rid[r] = a.in_ids[r];
      rw[r] = a.in_w[r];
    }
    for (int e = tid; e < E; e += kSmallThreads) cnt[e] = 0;
    __syncthreads();
    if (warp == 0) {
      int32_t* rrank = reinterpret_cast<int32_t*>(smem + a.lay.rrank);
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
      const bool any_bad = __any_sync(kFull, bad);
      if (lane == 0) misc[0] = any_bad ? MOE_RS_DEVICE_BAD_EXPERT_ID : 0;
    }
    __syncthreads();
  }

  if constexpr (!kGrid) {
    // ------------------------------------------------ padded scan, scatter, padding
    const int total = block_scan_padded<kSmallThreads>(cnt, off, E, B, misc + 4);
    for (int r = tid; r < N; r += kSmallThreads) {
      const int e = rid[r];
      if (e < 0 || e >= E) continue;
      int rank;
      if (!kSortOnly) {
        const int t = r / K;
        rank = (t < 32) ? __popc(masks[e] & ((1u << t) - 1u))
                        : __popc(masks[e]) + __popc(masks[E + e] & ((1u << (t - 32)) - 1u));
      } else {
        rank = reinterpret_cast<const int32_t*>(smem + a.lay.rrank)[r];
      }
      const int pos = off[e] + rank;
      a.sorted_ids[pos] = r;
      a.sorted_w[pos] = rw[r];
    }
    for (int e = tid; e < E; e += kSmallThreads) {
      const int c = cnt[e];
      if (c == 0) continue;
      const int o = off[e];
      const int p = (c + B - 1) & ~(B - 1);
      for (int q = o + c; q < o + p; ++q) {
        a.sorted_ids[q] = N;
        a.sorted_w[q] = 0.0f;
      }
      for (int b = o / B; b < (o + p) / B; ++b) a.expert_ids[b] = e;
    }
    if (tid == 0) {
      *a.npp = total;
      *a.status = misc[0];
    }
  }
}

SmallLayout small_layout(int E, int N, int wave, int nu, bool sort_only, bool grid) {
  SmallLayout l{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const int at = static_cast<int>(o);
    o = align16(o + bytes);
    return at;
  };
  l.bias = 0;
  l.keys = sort_only ? 0 : take(sizeof(float) * (size_t)wave * E);
  l.svals = sort_only ? 0 : take(sizeof(float) * (size_t)wave * E);
  const int warps = wave < kSmallThreads / 32 ? wave : kSmallThreads / 32;
  l.scratch = sort_only ? 0 : take(sizeof(WarpScratch) * (size_t)warps);
  l.umax = (sort_only || nu == 0) ? 0 : take(ub_bytes(nu) * warps);
  l.rid = take(sizeof(int32_t) * N);
  l.rw = take(sizeof(float) * N);
  l.rrank = sort_only ? take(sizeof(int32_t) * N) : 0;
  l.cnt = take(sizeof(int32_t) * E);
  l.off = take(sizeof(int32_t) * E);
  l.masks = sort_only ? 0 : take(sizeof(unsigned) * (grid ? 1 : 2) * E);
  l.owner = grid ? take(sizeof(int32_t) * E) : 0;  // grid: routes of earlier CTAs per expert
  l.misc = take(sizeof(int32_t) * 40);
  l.total = static_cast<int>(o);
  return l;
}

cudaError_t launch_small(const SmallArgs& a, bool sort_only, cudaStream_t st) {
  const size_t smem = static_cast<size_t>(a.lay.total);
  auto* kern = sort_only ? mrs_small_kernel<true, false, false>
                         : (a.use_seg ? mrs_small_kernel<false, true, false>
                                      : mrs_small_kernel<false, false, false>);
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  return launch_pdl(kern, dim3(1), dim3(kSmallThreads), smem, st, a);
}

cudaError_t launch_small_grid(const SmallArgs& a, cudaStream_t st) {
  const int ctas = (a.T + a.per - 1) / a.per;
  if (a.T < 2 || a.per < 1 || a.per > a.wave || a.wave > kSmallThreads / 32 ||
      a.xchg == nullptr || a.bar == nullptr)
    return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(a.lay.total);
  auto* kern = a.use_seg ? mrs_small_kernel<false, true, true> : mrs_small_kernel<false, false, true>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  err = launch_grid_prep(a.bar, a.status, st);
  if (err != cudaSuccess) return err;
  // a cooperative launch: all CTAs are resident together (the launch fails otherwise), which
  // the grid-wide barrier needs
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kSmallThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

// --------------------------------------------------------- multi-CTA route, any shape
// Shared memory: bias[E], counts[E], the unit's routes (ids, weights), then per warp the
// exact keys and scores of one row and the route scratch; after routing, the per-warp
// region is reused by phase 1 of the sort step.
struct GenCtaLayout {
  size_t bias, counts, rid, rw, warps, per_warp, total;
};

__host__ __device__ inline GenCtaLayout gen_cta_layout(int E, int nwarps, int max_routes,
                                                       bool sort) {
  GenCtaLayout l{};
  size_t o = 0;
  l.bias = o;
  o = align16(o + sizeof(float) * E);
  l.counts = o;
  o = align16(o + sizeof(int32_t) * E);
  l.rid = o;
  o = align16(o + (sort ? sizeof(int32_t) * max_routes : 0));
  l.rw = o;
  o = align16(o + (sort ? sizeof(float) * max_routes : 0));
  l.warps = o;
  l.per_warp = align16(sizeof(float) * 2 * (size_t)E) + sizeof(WarpScratch);
  size_t region = l.per_warp * nwarps;
  if (sort && region < unit_scratch_bytes(E)) region = unit_scratch_bytes(E);
  l.total = o + region;
  return l;
}

size_t route_smem_bytes(int E, int nwarps, int max_routes, bool sort) {
  return gen_cta_layout(E, nwarps, max_routes, sort).total;
}

template <bool kSort>
__global__ void __launch_bounds__(512) mrs_route_kernel(const RouteArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const RouteShape sh = a.sh;
  const int E = sh.E, K = sh.K;
  const GenCtaLayout lay = gen_cta_layout(E, a.nwarps, a.max_routes, kSort);
  float* bias_s = reinterpret_cast<float*>(smem + lay.bias);
  int32_t* counts = reinterpret_cast<int32_t*>(smem + lay.counts);
  int32_t* rid = reinterpret_cast<int32_t*>(smem + lay.rid);
  float* rw = reinterpret_cast<float*>(smem + lay.rw);
  unsigned char* mine = smem + lay.warps + lay.per_warp * warp;
  float* key = reinterpret_cast<float*>(mine);
  float* sv = key + E;
  WarpScratch& scr =
      *reinterpret_cast<WarpScratch*>(mine + align16(sizeof(float) * 2 * (size_t)E));
  pdl_trigger();
  pdl_wait();

  const bool sm = sh.softmax != 0;  // no bias with softmax scoring
  for (int e = tid; e < E; e += blockDim.x) {
    bias_s[e] = sm ? 0.0f : a.bias[e];
    counts[e] = 0;
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
        // 16-byte shared-memory accesses (the bias and the per-warp key and score rows are
        // 16-byte aligned, E % 8 == 0): scalar ones 32 bytes apart would hit 4 banks
        const float4 b0 = reinterpret_cast<const float4*>(bias_s)[2 * v];
        const float4 b1 = reinterpret_cast<const float4*>(bias_s)[2 * v + 1];
        const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
        float k8[8], s8[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          k8[2 * j] = score_key(__uint_as_float(wd[j] << 16), bb[2 * j], sm, s8[2 * j]);
          k8[2 * j + 1] =
              score_key(__uint_as_float(wd[j] & 0xffff0000u), bb[2 * j + 1], sm, s8[2 * j + 1]);
        }
        float4* kr = reinterpret_cast<float4*>(key + 8 * v);
        float4* sr = reinterpret_cast<float4*>(sv + 8 * v);
        kr[0] = make_float4(k8[0], k8[1], k8[2], k8[3]);
        kr[1] = make_float4(k8[4], k8[5], k8[6], k8[7]);
        sr[0] = make_float4(s8[0], s8[1], s8[2], s8[3]);
        sr[1] = make_float4(s8[4], s8[5], s8[6], s8[7]);
      }
    } else {
      for (int e = lane; e < E; e += 32) {
        key[e] = score_key(bf16_bits_to_float(row[e]), bias_s[e], sm, sv[e]);
      }
    }
    __syncwarp();
    int id;
    float w;
    route_token(SmemExactSrc{key, sv}, sh, scr, lane, id, w);
    if (lane < K) {
      a.topk_ids[static_cast<size_t>(t) * K + lane] = id;
      a.topk_w[static_cast<size_t>(t) * K + lane] = w;
      if (kSort) {
        rid[(t - t0) * K + lane] = id;
        rw[(t - t0) * K + lane] = w;
        if (id >= 0 && id < E) atomicAdd(&counts[id], 1);
      }
    }
  }
  if (kSort) {
    __syncthreads();
    unit_sort_tail(rid, rw, counts, E, K, u, t0, t1, smem + lay.warps, a.uo, a.U);
    if (tid == 0) a.uo.unit_flags[u] = 0;
  }
}


// ------------------------------------------------- multi-CTA route, TMA-staged segments
// Shared memory: bias[E], counts[E], the unit's routes (ids, weights), then per warp: nbuf
// row buffers of tpw rows each, two mbarriers, one route scratch per token of a step and the
// unit bounds; after routing, the per-warp region is reused by phase 1.
struct SegCtaLayout {
  size_t bias, counts, rid, rw, warps, per_warp, rows, mbar, scratch, umax, total;
};

__host__ __device__ inline SegCtaLayout seg_cta_layout(int E, int nu, int nwarps,
                                                       int max_routes, bool sort, int tpw,
                                                       int nbuf, bool cluster) {
  SegCtaLayout l{};
  size_t o = 0;
  l.bias = o;
  o = align16(o + sizeof(float) * E);
  l.counts = o;
  o = align16(o + sizeof(int32_t) * E);
  l.rid = o;
  o = align16(o + (sort ? sizeof(int32_t) * max_routes : 0));
  l.rw = o;
  o = align16(o + (sort ? sizeof(float) * max_routes : 0));
  l.warps = o;
  size_t w = 0;
  l.rows = w;
  w = align16(w + static_cast<size_t>(nbuf) * tpw * sizeof(uint16_t) * E);
  l.mbar = w;
  w = align16(w + 2 * sizeof(unsigned long long));
  l.scratch = w;
  w = align16(w + static_cast<size_t>(tpw) * sizeof(SegScratch));
  l.umax = w;
  w = align16(w + ub_bytes(nu));
  l.per_warp = w;
  size_t region = w * nwarps;
  const size_t tail = cluster ? cluster_scratch_bytes(E) : unit_scratch_bytes(E);
  if (sort && region < tail) region = tail;
  l.total = o + region;
  return l;
}

size_t seg_smem_bytes(int E, int nu, int nwarps, int max_routes, bool sort, int tpw,
                      int nbuf, bool cluster) {
  return seg_cta_layout(E, nu, nwarps, max_routes, sort, tpw, nbuf, cluster).total;
}

// Warp w of unit u takes steps w, w + nwarps, ...; step i covers the 32 / LT consecutive
// tokens t0 + i * (32 / LT) + h, token h routed by lanes [h * LT, (h + 1) * LT).  The rows
// of a step are contiguous, so one bulk copy brings them in.  A buffer goes back to the copy
// engine (for the warp's step nbuf further on) as soon as the selection stops reading it.
// kSoftmax: softmax scoring, selection on the logits themselves (LogitRow, no bias, exact).
// kCluster: the grid is one thread-block cluster and runs both sort phases itself
// (cluster_sort_tail) instead of phase 1 into the workspace.
template <bool kSort, int LT, bool kSoftmax, bool kCluster>
__global__ void __launch_bounds__(kSegThreads, 1) mrs_route_seg_kernel(const RouteArgs a) {
  constexpr int kTpw = 32 / LT;
  constexpr int kParts = (LT == 16) ? 2 : 1;
  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = lane / LT, ll = lane & (LT - 1);
  const SegShape sh = a.seg;
  const int E = sh.E, K = sh.K, nbuf = a.nbuf;
  const SegCtaLayout lay =
      seg_cta_layout(E, sh.nu, a.nwarps, a.max_routes, kSort, kTpw, nbuf, kCluster);
  float* bias_s = reinterpret_cast<float*>(smem + lay.bias);
  int32_t* counts = reinterpret_cast<int32_t*>(smem + lay.counts);
  int32_t* rid = reinterpret_cast<int32_t*>(smem + lay.rid);
  float* rw = reinterpret_cast<float*>(smem + lay.rw);
  unsigned char* mine = smem + lay.warps + lay.per_warp * warp;
  uint16_t* rows = reinterpret_cast<uint16_t*>(mine + lay.rows);
  unsigned long long* mbar = reinterpret_cast<unsigned long long*>(mine + lay.mbar);
  SegScratch* scr = reinterpret_cast<SegScratch*>(mine + lay.scratch);
  unsigned short* umax = reinterpret_cast<unsigned short*>(mine + lay.umax);
  __shared__ int cta_flags;
  __shared__ unsigned int cta_bmax_bits;

  const int u = blockIdx.x;
  const int t0 = static_cast<int>(static_cast<long long>(u) * a.T / a.U);
  const int t1 = static_cast<int>(static_cast<long long>(u + 1) * a.T / a.U);
  const int n_steps = (t1 - t0 + kTpw - 1) / kTpw;
  const int n_mine = (n_steps - warp + a.nwarps - 1) / a.nwarps;  // steps of this warp
  auto step_t = [&](int k) { return t0 + (warp + k * a.nwarps) * kTpw; };
  auto issue = [&](int k, int b) {
    const int ts = step_t(k);
    const int n = min(kTpw, t1 - ts);
    tma_load_1d(rows + static_cast<size_t>(b) * kTpw * E,
                a.logits + static_cast<size_t>(ts) * E,
                static_cast<uint32_t>(n) * static_cast<uint32_t>(E) * 2u, &mbar[b]);
  };

  // the sort kernel that follows may take SMs as this grid's blocks exit (it waits for all)
  pdl_trigger();
  pdl_wait();
  // start this warp's first copies before anything else
  if (lane == 0) {
    mbar_init(&mbar[0], 1);
    mbar_init(&mbar[1], 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (lane == 0)
    for (int k = 0; k < nbuf && k < n_mine; ++k) issue(k, k);
  ub_init_pads(umax, lane, sh.nu);
  if (tid == 0) {
    cta_flags = 0;
    cta_bmax_bits = 0u;
  }
  // routes of tokens that never get routed (a timed-out copy) stay dropped
  if (kSort)
    for (int i = tid; i < (t1 - t0) * K; i += blockDim.x) rid[i] = -1;
  __syncthreads();
  float bmax = 0.0f;  // largest |bias|, NaN-propagating (NaN fails the limit test below)
  for (int e = tid; e < E; e += blockDim.x) {
    if (!kSoftmax) {
      const float b = a.bias[e];
      bias_s[e] = b;
      const float ab = fabsf(b);
      bmax = (ab > bmax || ab != ab) ? ab : bmax;
    }
    counts[e] = 0;
  }
  for (int d = 16; d > 0; d >>= 1) {
    const float o = __shfl_xor_sync(kFull, bmax, d);
    bmax = (o > bmax || o != o) ? o : bmax;
  }
  if (lane == 0) atomicMax(&cta_bmax_bits, (bmax != bmax) ? 0x7fffffffu : __float_as_uint(bmax));
  __syncthreads();
  // the proxy bound holds for |bias| <= kProxyBiasLimit once it has been verified on this
  // device; otherwise every step is exact
  const float bm = __uint_as_float(cta_bmax_bits);
  const bool proxy_ok = a.proxy_state != nullptr && *a.proxy_state == 1;
  const float delta = kSoftmax ? 0.0f
                      : (bm <= kProxyBiasLimit && proxy_ok) ? proxy_delta(bm) : INFINITY;

  uint32_t phase = 0u;  // bit b = parity to wait for on buffer b
  int issued = n_mine < nbuf ? n_mine : nbuf;
  int consumed = 0;
  bool ok = true;
  for (int k = 0; k < n_mine; ++k) {
    const int b = (nbuf == 2) ? (k & 1) : 0;
    if (!mbar_wait_bounded(&mbar[b], (phase >> b) & 1u, a.wait_limit_ns)) {
      ok = false;
      break;
    }
    consumed = k + 1;
    phase ^= 1u << b;
    const int t = step_t(k) + h;
    const bool valid = t < t1;
    const uint16_t* row_s = rows + static_cast<size_t>(b * kTpw + h) * E;
    const auto row = [&] {
      if constexpr (kSoftmax) return LogitRow{row_s};
      else return ProxyRow{row_s, bias_s};
    }();
    const LaneTop top = seg_pass1<LT, kParts>(row, sh, umax, lane, valid);
    auto release = [&] {
      __syncwarp();  // every lane is done with the buffer
      if (k + nbuf < n_mine) {
        if (lane == 0) {
          fence_proxy_async_smem();
          issue(k + nbuf, b);
        }
        ++issued;
      }
    };
    int id;
    float w;
    seg_select<LT, kParts>(row, sh, scr[h], umax, lane, delta, valid, top, release, id, w);
    if (valid && ll < K) {
      a.topk_ids[static_cast<size_t>(t) * K + ll] = id;
      a.topk_w[static_cast<size_t>(t) * K + ll] = w;
      if (kSort) {
        rid[(t - t0) * K + ll] = id;
        rw[(t - t0) * K + ll] = w;
        if (id >= 0 && id < E) atomicAdd(&counts[id], 1);
      }
    }
  }
  bool drained = true;
  if (!ok) {
    // a copy did not complete in time: report it, then give the copies still in flight a
    // bounded chance to land before their buffers are reused or the CTA exits
    if (lane == 0) atomicOr(&cta_flags, MOE_RS_DEVICE_WAIT_TIMEOUT);
    for (int k = consumed; k < issued; ++k) {
      const int b = (nbuf == 2) ? (k & 1) : 0;
      drained &= mbar_wait_bounded(&mbar[b], (phase >> b) & 1u, kWaitLimitNs);
      phase ^= 1u << b;
    }
  }
  // the barriers' memory is reused by the sort step below
  if (drained && lane == 0) {
    mbar_inval(&mbar[0]);
    mbar_inval(&mbar[1]);
  }
  if (kSort) {
    __syncthreads();
    if (kCluster) {
      if (tid == 0) cta_flags &= MOE_RS_DEVICE_WAIT_TIMEOUT;
      __syncthreads();
      cluster_sort_tail(rid, rw, counts, &cta_flags, E, K, t0, t1, static_cast<uint32_t>(u),
                        static_cast<uint32_t>(a.U), smem + lay.warps, a.co);
    } else {
      unit_sort_tail(rid, rw, counts, E, K, u, t0, t1, smem + lay.warps, a.uo, a.U);
      if (tid == 0) a.uo.unit_flags[u] = cta_flags & MOE_RS_DEVICE_WAIT_TIMEOUT;
    }
  }
}

template <bool kSort, int LT, bool kSoftmax, bool kCluster>
static cudaError_t launch_seg_h(const RouteArgs& a, size_t smem, cudaStream_t st) {
  auto* kern = mrs_route_seg_kernel<kSort, LT, kSoftmax, kCluster>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  if (!kCluster) return launch_pdl(kern, dim3(a.U), dim3(a.nwarps * 32), smem, st, a);
  err = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.U);
  cfg.blockDim = dim3(a.nwarps * 32);
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

template <bool kSort, bool kSoftmax, bool kCluster>
static cudaError_t launch_seg(const RouteArgs& a, size_t smem, cudaStream_t st) {
  return a.lanes == 16 ? launch_seg_h<kSort, 16, kSoftmax, kCluster>(a, smem, st)
                       : launch_seg_h<kSort, 32, kSoftmax, kCluster>(a, smem, st);
}

// Clusters of kClusterCtas CTAs of the segment kernel (one per SM: 512 threads of up to 128
// registers) that the device can hold at once; 0 when it cannot place one (the cluster path
// is then not taken).
int seg_cluster_capacity(size_t smem) {
  auto* kern = mrs_route_seg_kernel<true, 16, false, true>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
          cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(kClusterCtas);
  cfg.blockDim = dim3(kSegThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kClusterCtas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_route(const RouteArgs& a, size_t smem, cudaStream_t st) {
  if (a.use_seg) {
    // softmax scoring only comes with the sort step (moe_route_sort_softmax)
    if (a.cluster) {
      if (!a.sort) return cudaErrorInvalidValue;
      return a.seg.softmax ? launch_seg<true, true, true>(a, smem, st)
                           : launch_seg<true, false, true>(a, smem, st);
    }
    if (a.seg.softmax)
      return a.sort ? launch_seg<true, true, false>(a, smem, st) : cudaErrorInvalidValue;
    return a.sort ? launch_seg<true, false, false>(a, smem, st)
                  : launch_seg<false, false, false>(a, smem, st);
  }
  cudaError_t err;
  const int threads = a.nwarps * 32;
  if (a.sort) {
    err = cudaFuncSetAttribute(mrs_route_kernel<true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    err = launch_pdl(mrs_route_kernel<true>, dim3(a.U), dim3(threads), smem, st, a);
  } else {
    err = cudaFuncSetAttribute(mrs_route_kernel<false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    err = launch_pdl(mrs_route_kernel<false>, dim3(a.U), dim3(threads), smem, st, a);
  }
  return err;
}

}  // namespace mrs
