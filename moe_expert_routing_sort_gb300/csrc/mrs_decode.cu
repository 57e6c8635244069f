// mrs_decode.cu -- the whole route-sort path for one token (decode), one CTA, one launch.
//
// Latency-oriented: every step uses the whole CTA and the sort needs no scan over experts.
//   scores    thread t owns experts t, t + 512, ...; one DRAM round trip (logits and bias)
//   groups    warp j scores group j (sum of its two best keys) from shared memory
//   kept      every warp ranks the G group scores itself (no barrier needed)
//   threshold each warp's two best candidates are samples; the K-th best sample is a lower
//             bound on the K-th best candidate key
//   survivors candidates at or above it are compacted and ranked in parallel by counting
//   sort      one token: each selected expert gets one route, so expert id_k owns block
//             (number of selected ids below id_k), its row 0 is route k and rows 1..B-1 are
//             padding; npp = K * B
// Source: "perf(flydsl): Kimi-K3 B1 route-sort + prepared-MoE handoff (stack)", Summary --
// the B1 (batch-one) route-sort: FP32 logits, correction bias, grouped top-k, both sort
// phases, in one kernel.
#include "mrs_internal.h"
#include "moe_route_sort.h"

namespace mrs {

constexpr int kDecodeThreads = 512;
constexpr int kDecodeWarps = kDecodeThreads / 32;
constexpr int kDecodeEpt = kMaxExperts / kDecodeThreads;  // experts per thread, at most
constexpr int kDecodeCap = 128;                            // survivors kept for ranking

struct DecodeSmem {
  float key[kMaxExperts];
  float s[kMaxExperts];
  float gs[kMaxGroups];
  float samples[2 * kDecodeWarps];
  unsigned long long cand[kDecodeCap];
  float cand_s[kDecodeCap];
  unsigned long long wbest[kDecodeWarps];
  float wbest_s[kDecodeWarps];
  int sel_id[kMaxTopk];
  float sel_s[kMaxTopk];
  int count;
};

__device__ __forceinline__ void warp_top2_merge(float& m1, float& m2) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    const float o1 = __shfl_xor_sync(kFull, m1, d);
    const float o2 = __shfl_xor_sync(kFull, m2, d);
    m2 = fmaxf(fmaxf(m2, o2), fminf(m1, o1));
    m1 = fmaxf(m1, o1);
  }
}

__global__ void __launch_bounds__(kDecodeThreads, 1) mrs_decode_kernel(const DecodeArgs a) {
  __shared__ DecodeSmem sm;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_trigger();
  pdl_wait();
  const int E = a.E, G = a.G, g = a.g, Kg = a.Kg, K = a.K, B = a.B;
  const bool grouped = Kg < G;

  // ---- exact scores and keys (one DRAM round trip)
  float key[kDecodeEpt], sv[kDecodeEpt];
  {
    uint16_t x[kDecodeEpt];
    float b[kDecodeEpt];
#pragma unroll
    for (int i = 0; i < kDecodeEpt; ++i) {
      const int e = tid + kDecodeThreads * i;
      if (e < E) {
        x[i] = a.logits[e];
        b[i] = a.bias[e];
      }
    }
#pragma unroll
    for (int i = 0; i < kDecodeEpt; ++i) {
      const int e = tid + kDecodeThreads * i;
      key[i] = -INFINITY;
      sv[i] = 0.0f;
      if (e < E) {
        sv[i] = exact_score(bf16_bits_to_float(x[i]));
        key[i] = __fadd_rn(sv[i], b[i]);
        sm.key[e] = key[i];
        sm.s[e] = sv[i];
      }
    }
  }
  if (tid == 0) sm.count = 0;
  __syncthreads();

  // ---- group scores (warp per group), then every warp ranks the groups itself
  if (grouped) {
    for (int j = warp; j < G; j += kDecodeWarps) {
      float m1 = -INFINITY, m2 = -INFINITY;
      for (int i = lane; i < g; i += 32) {
        const float v = sm.key[j * g + i];
        m2 = fmaxf(m2, fminf(m1, v));
        m1 = fmaxf(m1, v);
      }
      warp_top2_merge(m1, m2);
      if (lane == 0) sm.gs[j] = (g >= 2) ? __fadd_rn(m1, m2) : m1;
    }
    __syncthreads();
  }
  unsigned km0 = 0xffffffffu, km1 = 0xffffffffu;
  if (grouped) {
    bool k0 = false, k1 = false;
    if (lane < G) {
      const float v = sm.gs[lane];
      int r = 0;
      for (int jj = 0; jj < G; ++jj) {
        const float o = sm.gs[jj];
        r += (o > v || (o == v && jj < lane)) ? 1 : 0;
      }
      k0 = r < Kg;
    }
    if (lane + 32 < G) {
      const float v = sm.gs[lane + 32];
      int r = 0;
      for (int jj = 0; jj < G; ++jj) {
        const float o = sm.gs[jj];
        r += (o > v || (o == v && jj < lane + 32)) ? 1 : 0;
      }
      k1 = r < Kg;
    }
    km0 = __ballot_sync(kFull, k0);
    km1 = __ballot_sync(kFull, k1);
  }

  // ---- candidates; each warp's two best are threshold samples
  bool cand[kDecodeEpt];
  float t1 = -INFINITY, t2 = -INFINITY;
#pragma unroll
  for (int i = 0; i < kDecodeEpt; ++i) {
    const int e = tid + kDecodeThreads * i;
    bool c = e < E;
    if (c && grouped) {
      const int j = e / g;
      c = ((j < 32 ? (km0 >> j) : (km1 >> (j - 32))) & 1u) != 0u;
    }
    cand[i] = c;
    if (c) {
      t2 = fmaxf(t2, fminf(t1, key[i]));
      t1 = fmaxf(t1, key[i]);
    }
  }
  warp_top2_merge(t1, t2);
  if (lane == 0) {
    sm.samples[2 * warp] = t1;
    sm.samples[2 * warp + 1] = t2;
  }
  __syncthreads();
  // every warp: the K-th best of the 32 samples (distinct candidates); -inf if fewer
  float tau;
  {
    const float v = sm.samples[lane];
    int r = 0;
#pragma unroll
    for (int m = 0; m < 2 * kDecodeWarps; ++m) {
      const float o = sm.samples[m];
      r += (o > v || (o == v && m < lane)) ? 1 : 0;
    }
    const unsigned hit = __ballot_sync(kFull, r == K - 1);
    tau = __shfl_sync(kFull, v, __ffs(hit) - 1);
    if (!(tau > -INFINITY)) tau = -INFINITY;
  }

  // ---- survivors: candidates with key >= tau, compacted (warp-aggregated slots)
#pragma unroll
  for (int i = 0; i < kDecodeEpt; ++i) {
    const bool sv_ok = cand[i] && key[i] >= tau;
    const unsigned b = __ballot_sync(kFull, sv_ok);
    if (b) {
      int base = 0;
      if (lane == 0) base = atomicAdd(&sm.count, __popc(b));
      base = __shfl_sync(kFull, base, 0);
      if (sv_ok) {
        const int pos = base + __popc(b & lanemask_lt(lane));
        if (pos < kDecodeCap) {
          const int e = tid + kDecodeThreads * i;
          sm.cand[pos] = composite(key[i], e);
          sm.cand_s[pos] = sv[i];
        }
      }
    }
  }
  __syncthreads();
  const int total = sm.count;
  if (total <= kDecodeCap) {
    for (int q = tid; q < total; q += kDecodeThreads) {
      const unsigned long long me = sm.cand[q];
      int r = 0;
#pragma unroll 8
      for (int p = 0; p < total; ++p) r += (sm.cand[p] > me) ? 1 : 0;
      if (r < K) {
        sm.sel_id[r] = composite_expert(me);
        sm.sel_s[r] = sm.cand_s[q];
      }
    }
  } else {
    // very many survivors (wide exact ties): K rounds of a block-wide maximum
    unsigned long long prev = ~0ull;
    for (int k = 0; k < K; ++k) {
      unsigned long long best = 0ull;
      float best_s = 0.0f;
#pragma unroll
      for (int i = 0; i < kDecodeEpt; ++i) {
        if (cand[i] && key[i] >= tau) {
          const unsigned long long c = composite(key[i], tid + kDecodeThreads * i);
          if (c < prev && c > best) {
            best = c;
            best_s = sv[i];
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
  }
  __syncthreads();

  // ---- weights, outputs and the one-token sort (warp 0)
  if (warp == 0) {
    const bool mine = lane < K;
    const int id = mine ? sm.sel_id[lane] : 0x7fffffff;
    const float s = mine ? sm.sel_s[lane] : 0.0f;
    float sum = 0.0f;
    for (int k = 0; k < K; ++k) sum = __fadd_rn(sum, sm.sel_s[k]);  // slot order
    const float w = __fmul_rn(__fdiv_rn(s, sum), a.R);
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
    for (int p = lane; p < K * B; p += 32) {
      if ((p & (B - 1)) != 0) {
        a.sorted_ids[p] = K;  // sentinel T * K with T = 1
        a.sorted_w[p] = 0.0f;
      }
    }
    if (lane == 0) {
      *a.npp = K * B;
      *a.status = 0;
    }
  }
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
  return launch_pdl(mrs_decode_kernel, dim3(1), dim3(kDecodeThreads), 0, st, a);
}

}  // namespace mrs
