// mrs_decode.cu -- the whole route-sort path for one token (decode), one CTA, one launch.
//
// Latency-oriented: four block barriers from the logits to the outputs; the serial steps run
// in one warp while the others wait, so they do not share the schedulers with copies of
// themselves.
//   rows      group j is held by TPG consecutive threads (TPG = the largest power of two
//             with TPG * G <= 512): thread i of the group owns experts j*g + i + TPG*r;
//             one DRAM round trip brings logits and bias, exact scores stay in registers
//   groups    a shuffle tree over each group's threads gives, at the 8-thread level, the
//             top-2 of every 8-thread segment (threshold samples) and, at the top, the
//             group's top-2 (one partial per warp when a group spans several warps)
//   ---- barrier
//   kept      warp 0 alone merges the partials and ranks the G group scores (the other warps
//             wait at the next barrier, so the serial steps run at one warp's full issue rate)
//   threshold warp 0: at least ceil(K/2) kept segments hold two keys >= t2, so at least K
//             kept keys are >= t2 (and the K-th best segment maximum is also such a bound);
//             the kept-group masks and the threshold go to shared memory
//   ---- barrier
//   survivors every thread compacts its kept keys at or above the threshold (warp-aggregated
//             slots)
//   ---- barrier
//   rank      four threads per survivor count the better survivors (rank by counting)
//   ---- barrier
//   finish    warp 0 forms the weights and writes the K slots
//   sort      one token: each selected expert gets one route, so expert id_k owns block
//             (number of selected ids below id_k), its row 0 is route k and rows 1..B-1 are
//             padding (written at the start, as they depend on nothing); npp = K * B
// With softmax scoring (G = 1, no bias) the keys are the logits and the weight step turns the
// selected logits into softmax terms.
// Source: "perf(flydsl): Kimi-K3 B1 route-sort + prepared-MoE handoff (stack)", Summary --
// the B1 (batch-one) route-sort: FP32 logits, correction bias, grouped top-k, both sort
// phases, in one kernel.
#include "mrs_internal.h"
#include "mrs_unit.cuh"
#include "moe_route_sort.h"

namespace mrs {

constexpr int kDecodeThreads = 512;
constexpr int kDecodeWarps = kDecodeThreads / 32;
constexpr int kDecodeEpt = 16;   // experts per thread, at most (g <= TPG * kDecodeEpt)
constexpr int kDecodeCap = 128;  // survivors kept for ranking
constexpr int kDecodeSamples = kDecodeThreads / 8;
// Tokens one CTA of the grid path routes at most: ceil(kDecodeGridTokens / 152 SMs) with room.
constexpr int kDecodeGridOwn = 4;

struct DecodeSmem {
  float samp1[kDecodeSamples], samp2[kDecodeSamples];  // 8-thread segments' top-2
  float part1[64], part2[64];                          // per-group partial top-2
  unsigned long long cand[kDecodeCap];
  float cand_s[kDecodeCap];
  unsigned long long wbest[kDecodeWarps];
  float wbest_s[kDecodeWarps];
  alignas(16) int sel_id[kMaxTopk];
  alignas(16) float sel_s[kMaxTopk];
  alignas(16) float own_w[kDecodeGridOwn][kMaxTopk];  // several tokens: this CTA's weights
  int count;
  float tau;            // selection threshold (warp 0)
  unsigned kept[2];     // kept-group masks, groups 0-31 and 32-63 (warp 0)
};

__device__ __forceinline__ void top2_merge_xor(float& m1, float& m2, int d) {
  const float o1 = __shfl_xor_sync(kFull, m1, d);
  const float o2 = __shfl_xor_sync(kFull, m2, d);
  m2 = fmaxf(fmaxf(m2, o2), fminf(m1, o1));
  m1 = fmaxf(m1, o1);
}

// Threads per group for G groups: the largest power of two with TPG * G <= 512 (>= 8).
__host__ __device__ inline int decode_tpg(int G) {
  int t = 512;
  while (t * G > kDecodeThreads) t >>= 1;
  return t;
}

__device__ void decode_grid_sort(const DecodeArgs& a, const DecodeSmem& sm, int T);

// kSoftmax: softmax scoring (keys are the logits, no bias).
// kEpt: experts per thread the code is unrolled for (>= ceil(g / TPG)); the smallest fitting
// instance is launched, so that a launch fetches only the instructions it runs (the kernel
// usually lands on an SM whose instruction cache has never held it).
// The route step of token t by the whole CTA (and, with one token, both sort phases).
// kMulti: one of several tokens of a cooperative grid: no sort here (decode_grid_sort).
template <bool kSoftmax, int kEpt, bool kMulti>
__device__ __forceinline__ void decode_token(const DecodeArgs& a, DecodeSmem& sm, int t) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint16_t* logits = a.logits + static_cast<size_t>(t) * a.E;
  const int G = a.G, g = a.g, Kg = a.Kg, K = a.K, B = a.B;
  const int TPG = decode_tpg(G);
  const int P = TPG > 32 ? TPG / 32 : 1;  // partials per group
  const int j = tid / TPG, i = tid - j * TPG;
  const bool in_group = j < G;
  // experts per thread: 2 * 256 / G < TPG, so g = E / G <= 4096 / G < 16 * TPG
  const int R = (g + TPG - 1) / TPG;

  // ---- loads (one DRAM round trip); rows that depend on nothing meanwhile
  float key[kEpt], sv[kEpt];
  {
    uint16_t x[kEpt];
    float b[kEpt];
#pragma unroll
    for (int r = 0; r < kEpt; ++r) {
      if (r >= R) break;
      const int li = i + TPG * r;
      if (in_group && li < g) {
        x[r] = logits[j * g + li];
        b[r] = kSoftmax ? 0.0f : a.bias[j * g + li];
      }
    }
    if (!kMulti) {
      for (int p = tid; p < K * B; p += kDecodeThreads) {
        if ((p & (B - 1)) != 0) {
          a.sorted_ids[p] = K;  // sentinel T * K with T = 1
          a.sorted_w[p] = 0.0f;
        }
      }
    }
    if (tid == 0) {
      if (!kMulti) {
        *a.npp = K * B;
        *a.status = 0;
      }
      sm.count = 0;
    }
    float t1 = -INFINITY, t2 = -INFINITY;
#pragma unroll
    for (int r = 0; r < kEpt; ++r) {
      const int li = i + TPG * r;
      key[r] = -INFINITY;
      sv[r] = 0.0f;
      if (r < R && in_group && li < g) {
        key[r] = score_key(bf16_bits_to_float(x[r]), b[r], kSoftmax, sv[r]);
        t2 = fmaxf(t2, fminf(t1, key[r]));
        t1 = fmaxf(t1, key[r]);
      }
    }
    // ---- shuffle tree: 8-thread segments (samples), then the group (partials)
    top2_merge_xor(t1, t2, 1);
    top2_merge_xor(t1, t2, 2);
    top2_merge_xor(t1, t2, 4);
    if ((tid & 7) == 0) {
      sm.samp1[tid >> 3] = t1;
      sm.samp2[tid >> 3] = t2;
    }
    for (int d = 8; d < 32 && d < TPG; d <<= 1) top2_merge_xor(t1, t2, d);
    if (in_group && (i & 31 & (TPG - 1)) == 0) {
      const int p = (TPG > 32) ? (i >> 5) : 0;
      sm.part1[j * P + p] = t1;
      sm.part2[j * P + p] = t2;
    }
  }
  __syncthreads();

  if (warp == 0) {
    // ---- group scores and kept groups (lane l holds groups l and l + 32)
    unsigned km0 = 0xffffffffu, km1 = 0xffffffffu;
    if (Kg < G) {
      float gs[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int l = lane + 32 * h;
        gs[h] = -INFINITY;
        if (l < G) {
          float m1 = -INFINITY, m2 = -INFINITY;
          for (int p = 0; p < P; ++p) {
            const float o1 = sm.part1[l * P + p], o2 = sm.part2[l * P + p];
            m2 = fmaxf(fmaxf(m2, o2), fminf(m1, o1));
            m1 = fmaxf(m1, o1);
          }
          gs[h] = (g >= 2) ? __fadd_rn(m1, m2) : m1;
        }
      }
      int rk0 = 0, rk1 = 0;
      for (int m = 0; m < G; ++m) {
        const float o = __shfl_sync(kFull, (m < 32) ? gs[0] : gs[1], m & 31);
        rk0 += (o > gs[0] || (o == gs[0] && m < lane)) ? 1 : 0;
        rk1 += (o > gs[1] || (o == gs[1] && m < lane + 32)) ? 1 : 0;
      }
      km0 = __ballot_sync(kFull, lane < G && rk0 < Kg);
      km1 = __ballot_sync(kFull, lane + 32 < G && rk1 < Kg);
    }
    // ---- threshold from the kept segments' samples (segment q covers threads 8q .. 8q+7)
    const int q0 = lane, q1 = lane + 32;
    const int g0 = (8 * q0) / TPG, g1 = (8 * q1) / TPG;
    const bool k0 = g0 < G && (((g0 < 32 ? (km0 >> g0) : (km1 >> (g0 - 32))) & 1u) != 0u);
    const bool k1 = g1 < G && (((g1 < 32 ? (km0 >> g1) : (km1 >> (g1 - 32))) & 1u) != 0u);
    const float ninf = -INFINITY;
    float tau = seg_kth_desc2<32>(k0 ? sm.samp2[q0] : ninf, k1 ? sm.samp2[q1] : ninf, lane,
                                  (K - 1) >> 1);
    if (__any_sync(kFull, tau == -INFINITY))
      tau = fmaxf(tau, seg_kth_desc2<32>(k0 ? sm.samp1[q0] : ninf, k1 ? sm.samp1[q1] : ninf,
                                         lane, K - 1));
    if (lane == 0) {
      sm.tau = tau;
      sm.kept[0] = km0;
      sm.kept[1] = km1;
    }
  }
  __syncthreads();
  const float tau = sm.tau;
  const unsigned km0 = sm.kept[0], km1 = sm.kept[1];
  auto kept_group = [&](int grp) {
    return ((grp < 32 ? (km0 >> grp) : (km1 >> (grp - 32))) & 1u) != 0u;
  };

  // ---- survivors: kept keys >= tau, compacted (warp-aggregated slots)
  const bool mine_kept = in_group && kept_group(j);
#pragma unroll
  for (int r = 0; r < kEpt; ++r) {
    if (r >= R) break;
    const bool s_ok = mine_kept && key[r] >= tau;
    const unsigned bl = __ballot_sync(kFull, s_ok);
    if (bl) {
      int base = 0;
      if (lane == 0) base = atomicAdd(&sm.count, __popc(bl));
      base = __shfl_sync(kFull, base, 0);
      if (s_ok) {
        const int pos = base + __popc(bl & lanemask_lt(lane));
        if (pos < kDecodeCap) {
          sm.cand[pos] = composite(key[r], j * g + i + TPG * r);
          sm.cand_s[pos] = sv[r];
        }
      }
    }
  }
  __syncthreads();
  const int total = sm.count;

  if (total <= kDecodeCap) {
    // ---- rank by counting (composites are distinct): four threads per survivor, each
    // counting the better composites in a quarter of the list
    static_assert(4 * kDecodeCap <= kDecodeThreads, "four threads per survivor");
    const int c = tid >> 2, q = tid & 3;
    int rk = 0;
    unsigned long long me = 0ull;
    if (c < total) {
      me = sm.cand[c];
      for (int p = q; p < total; p += 4) rk += (sm.cand[p] > me) ? 1 : 0;
    }
    rk += __shfl_xor_sync(kFull, rk, 1);
    rk += __shfl_xor_sync(kFull, rk, 2);
    if (c < total && q == 0 && rk < K) {
      sm.sel_id[rk] = composite_expert(me);
      sm.sel_s[rk] = sm.cand_s[c];
    }
    __syncthreads();
    if (!kMulti && warp != 0) return;
  } else {
    // very many survivors (wide exact ties): K rounds of a block-wide maximum
    unsigned long long prev = ~0ull;
    for (int k = 0; k < K; ++k) {
      unsigned long long best = 0ull;
      float best_s = 0.0f;
#pragma unroll
      for (int r = 0; r < kEpt; ++r) {
        if (mine_kept && key[r] >= tau) {
          const unsigned long long c = composite(key[r], j * g + i + TPG * r);
          if (c < prev && c > best) {
            best = c;
            best_s = sv[r];
          }
        }
      }
      unsigned long long wb = best;
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) {
        const unsigned long long o = __shfl_xor_sync(kFull, wb, d);
        wb = (o > wb) ? o : wb;
      }
      const unsigned own = __ballot_sync(kFull, best == wb && wb != 0ull);
      const float ws = __shfl_sync(kFull, best_s, own ? __ffs(own) - 1 : 0);
      if (lane == 0) {
        sm.wbest[warp] = wb;
        sm.wbest_s[warp] = ws;
      }
      __syncthreads();
      unsigned long long all = 0ull;
      float all_s = 0.0f;
      for (int w = 0; w < kDecodeWarps; ++w) {
        if (sm.wbest[w] > all) {
          all = sm.wbest[w];
          all_s = sm.wbest_s[w];
        }
      }
      if (tid == 0) {
        sm.sel_id[k] = composite_expert(all);
        sm.sel_s[k] = all_s;
      }
      prev = all;
      __syncthreads();
    }
    if (!kMulti && warp != 0) return;
  }

  // ---- warp 0: weights, outputs and the one-token sort
  if (!kMulti || warp == 0) {
    if (kSoftmax) softmax_terms(sm.sel_s, lane, K);
    const bool mine = lane < K;
    const int id = mine ? sm.sel_id[lane] : 0x7fffffff;
    const float s = mine ? sm.sel_s[lane] : 0.0f;
    float sum = 0.0f;
    if (lane == 0) {  // slot order
      float4 q4[kMaxTopk / 4];
      const float4* s4 = reinterpret_cast<const float4*>(sm.sel_s);
#pragma unroll
      for (int h = 0; h < kMaxTopk / 4; ++h)
        q4[h] = (4 * h < K) ? s4[h] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
      for (int h = 0; h < kMaxTopk / 4; ++h) {
        if (4 * h < K) sum = __fadd_rn(sum, q4[h].x);
        if (4 * h + 1 < K) sum = __fadd_rn(sum, q4[h].y);
        if (4 * h + 2 < K) sum = __fadd_rn(sum, q4[h].z);
        if (4 * h + 3 < K) sum = __fadd_rn(sum, q4[h].w);
      }
    }
    sum = __shfl_sync(kFull, sum, 0);
    const float w = __fmul_rn(__fdiv_rn(s, sum), a.R);
    if (kMulti) {
      if (mine) {
        a.topk_ids[t * K + lane] = id;
        a.topk_w[t * K + lane] = w;
        a.xchg[t * K + lane] = id;
        sm.own_w[(t - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x)][lane] = w;
      }
    } else {
      int blk = 0;  // number of selected ids below mine
#pragma unroll
      for (int m = 0; m < 32; ++m) blk += (__shfl_sync(kFull, id, m) < id) ? 1 : 0;
      if (mine) {
        a.topk_ids[lane] = id;
        a.topk_w[lane] = w;
        a.sorted_ids[blk * B] = lane;
        a.sorted_w[blk * B] = w;
        a.expert_ids[blk] = id;
      }
    }
  }
}

// kSoftmax: softmax scoring (keys are the logits, no bias).
// kEpt: experts per thread the code is unrolled for (>= ceil(g / TPG)); the smallest fitting
// instance is launched, so that a launch fetches only the instructions it runs (the kernel
// usually lands on an SM whose instruction cache has never held it).
// kGrid: 0 for one token; otherwise a.T tokens (2 <= a.T <= kDecodeGridTokens) on a cooperative
// grid, CTA b routing tokens b, b + gridDim.x, ... (1: exactly one token per CTA, 2: several),
// after which the CTAs sort all T * K routes together (decode_grid_sort).
template <bool kSoftmax, int kEpt, int kGrid>
__global__ void __launch_bounds__(kDecodeThreads, 1) mrs_decode_kernel(const DecodeArgs a) {
  constexpr bool kMulti = kGrid != 0;
  __shared__ DecodeSmem sm;
  const int tid = threadIdx.x;
  const int t0 = kMulti ? static_cast<int>(blockIdx.x) : 0;
  const int T = kMulti ? a.T : 1;
  const int step = kMulti ? static_cast<int>(gridDim.x) : 1;
  pdl_trigger();
  // the inputs start towards L2 while the kernel ahead in the stream finishes
  if (tid < 64)
    prefetch_l2_range(a.logits + static_cast<size_t>(t0) * a.E, 2 * static_cast<size_t>(a.E),
                      tid, 64);
  else if (!kSoftmax && tid < 192)
    prefetch_l2_range(a.bias, 4 * static_cast<size_t>(a.E), tid - 64, 128);
  pdl_wait();
  if constexpr (kGrid == 0) {
    decode_token<kSoftmax, kEpt, false>(a, sm, 0);
  } else if constexpr (kGrid == 1) {
    decode_token<kSoftmax, kEpt, true>(a, sm, t0);
    decode_grid_sort(a, sm, T);
  } else {
    for (int t = t0; t < T; t += step) {
      if (t + step < T && tid < 64)  // the CTA's next row starts towards L2
        prefetch_l2_range(a.logits + static_cast<size_t>(t + step) * a.E,
                          2 * static_cast<size_t>(a.E), tid, 64);
      decode_token<kSoftmax, kEpt, true>(a, sm, t);
      __syncthreads();  // the token's scratch is reused by the next one
    }
    decode_grid_sort(a, sm, T);
  }
}

// Both sort phases for T tokens on a cooperative grid (kMulti), every thread of every CTA:
// after a grid-wide barrier (bounded; on a timeout the CTA reports MOE_RS_DEVICE_WAIT_TIMEOUT
// and writes nothing more) each CTA reads all T * K selected ids from the exchange buffer,
// counts them per expert (with a token bit mask per expert) and forms the same block_m-padded
// prefix; the routes of its own tokens go to row base(e) + (tokens before t routed to e), which
// is the token-then-slot order because a token holds each expert at most once; CTA b of n
// writes the padding rows and block owners of experts [b E / n, (b + 1) E / n), CTA 0 npp (the
// status word is zeroed by mrs_grid_prep_kernel and only ever ORed here).  Dynamic shared
// memory: decode_grid_smem(E, T).
__device__ void decode_grid_sort(const DecodeArgs& a, const DecodeSmem& sm, int T) {
  extern __shared__ __align__(16) int32_t dsm[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = static_cast<int>(blockIdx.x), n = static_cast<int>(gridDim.x);
  const int E = a.E, K = a.K, B = a.B, N = T * K;
  const int W = (T + 31) >> 5;                         // token mask words per expert
  int32_t* cnt = dsm;                                  // [E]
  int32_t* padv = cnt + E;                             // [E]
  int32_t* base = padv + E;                            // [E + 1]
  unsigned* tmask = reinterpret_cast<unsigned*>(base + E + 1);  // [E][W]
  int32_t* all_id = reinterpret_cast<int32_t*>(tmask + static_cast<size_t>(E) * W);  // [N]
  int32_t* misc = all_id + N;                                                          // [64]
  for (int e = tid; e < E; e += kDecodeThreads) cnt[e] = 0;
  for (int x = tid; x < E * W; x += kDecodeThreads) tmask[x] = 0u;
  // every CTA's ids are in the exchange buffer once the whole grid has arrived (the barrier
  // orders the writes before it with the reads after it)
  if (!grid_barrier_bounded(a.bar, static_cast<unsigned>(n), a.wait_limit_ns, misc + 48)) {
    if (tid == 0) atomicOr(a.status, MOE_RS_DEVICE_WAIT_TIMEOUT);
    return;
  }
  for (int x = tid; x < N; x += kDecodeThreads) {
    const int e = __ldcg(a.xchg + x);
    all_id[x] = e;
    if (e >= 0 && e < E) {
      atomicAdd(&cnt[e], 1);
      const int tt = x / K;
      atomicOr(&tmask[e * W + (tt >> 5)], 1u << (tt & 31));
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += kDecodeThreads) padv[e] = (cnt[e] + B - 1) & ~(B - 1);
  __syncthreads();
  block_exclusive_scan(padv, base, E, misc);  // base[E] = the padded total
  // the routes of this CTA's tokens b, b + n, ...: thread x takes own token x / K, slot x % K
  const int own = (T - b + n - 1) / n;
  for (int x = tid; x < own * K; x += kDecodeThreads) {
    const int jj = x / K, k = x - jj * K;
    const int t = b + jj * n;
    const int r = t * K + k;
    const int e = all_id[r];
    const unsigned* m = tmask + e * W;
    int rank = __popc(m[t >> 5] & ((1u << (t & 31)) - 1u));
    for (int w = 0; w < (t >> 5); ++w) rank += __popc(m[w]);
    const int dst = base[e] + rank;
    a.sorted_ids[dst] = r;
    a.sorted_w[dst] = sm.own_w[jj][k];
  }
  const int e0 = static_cast<int>(static_cast<long long>(b) * E / n);
  const int e1 = static_cast<int>(static_cast<long long>(b + 1) * E / n);
  for (int e = e0 + warp; e < e1; e += kDecodeWarps) {
    const int c = cnt[e];
    if (c == 0) continue;
    const int off = base[e];
    const int end = off + padv[e];
    for (int p = off + c + lane; p < end; p += 32) {
      a.sorted_ids[p] = N;
      a.sorted_w[p] = 0.0f;
    }
    for (int q = off / B + lane; q < end / B; q += 32) a.expert_ids[q] = e;
  }
  if (b == 0 && tid == 0) *a.npp = base[E];
}

// Ahead of a grid-path call: zero its barrier word and status word, once the kernel ahead in the
// stream (possibly the previous grid-path call on the same workspace) has completed.
__global__ void mrs_grid_prep_kernel(unsigned* bar, int32_t* status) {
  pdl_trigger();
  pdl_wait();
  *bar = 0u;
  *status = 0;
}

cudaError_t launch_grid_prep(unsigned* bar, int32_t* status, cudaStream_t st) {
  return launch_pdl(mrs_grid_prep_kernel, dim3(1), dim3(1), 0, st, bar, status);
}

size_t decode_grid_smem(int E, int T, int K) {
  const size_t W = static_cast<size_t>(T + 31) / 32;
  return sizeof(int32_t) *
         (3 * static_cast<size_t>(E) + 1 + W * E + static_cast<size_t>(T) * K + 64);
}

template <int kEpt, int kGrid>
static cudaError_t launch_decode_ept(const DecodeArgs& a, int T, cudaStream_t st) {
  auto* kern = a.softmax ? mrs_decode_kernel<true, kEpt, kGrid>
                         : mrs_decode_kernel<false, kEpt, kGrid>;
  if (kGrid == 0) return launch_pdl(kern, dim3(1), dim3(kDecodeThreads), 0, st, a);
  const size_t smem = decode_grid_smem(a.E, a.T, a.K);
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  // a cooperative launch: all T CTAs are resident together (the launch fails otherwise), which
  // the grid-wide barrier needs
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(T);  // CTAs of the grid (<= a.T tokens)
  cfg.blockDim = dim3(kDecodeThreads);
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

template <int kGrid>
static cudaError_t launch_decode_any(const DecodeArgs& a, int T, cudaStream_t st) {
  const int tpg = decode_tpg(a.G);
  const int r = (a.g + tpg - 1) / tpg;  // <= kDecodeEpt (g <= 4096 / G < 16 * TPG)
  if (r <= 2) return launch_decode_ept<2, kGrid>(a, T, st);
  if (r <= 4) return launch_decode_ept<4, kGrid>(a, T, st);
  if (r <= 8) return launch_decode_ept<8, kGrid>(a, T, st);
  return launch_decode_ept<kDecodeEpt, kGrid>(a, T, st);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
  return launch_decode_any<0>(a, 1, st);
}

cudaError_t launch_decode_grid(const DecodeArgs& a, int ctas, cudaStream_t st) {
  if (a.T < 2 || a.T > kDecodeGridTokens || ctas < 1 || ctas > a.T ||
      (a.T + ctas - 1) / ctas > kDecodeGridOwn || a.xchg == nullptr || a.bar == nullptr)
    return cudaErrorInvalidValue;
  cudaError_t err = launch_grid_prep(a.bar, a.status, st);
  if (err != cudaSuccess) return err;
  return ctas == a.T ? launch_decode_any<1>(a, ctas, st) : launch_decode_any<2>(a, ctas, st);
}

}  // namespace mrs
