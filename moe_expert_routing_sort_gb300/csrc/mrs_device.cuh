// mrs_device.cuh -- device helpers and the warp-level route step of MoE route-sort.
//
// One warp routes one token: group scores -> kept groups -> top-K inside the kept groups ->
// renormalised weights.  Source of the step: "perf(flydsl): Kimi-K3 B1 route-sort +
// prepared-MoE handoff (stack)", Summary (FP32 logits, correction bias, grouped top-k).
//
// The selection reads keys through a "key source" with two views of expert e:
//   proxy(e)        a value within kDelta of the exact key (equal to it when kDelta == 0)
//   exact(e, s)     the exact key s_e + bias_e, and the exact score s_e through s
// Every decision is taken on exact keys: proxies only prune, with windows widened by
// 2*kDelta so that no element that can still win is pruned (see topk_in_kept).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace mrs {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxExperts = 4096;
constexpr int kMaxGroups = 64;
constexpr int kMaxTopk = 32;
constexpr int kCandCap = 64;  // survivors kept for the exact ranking before the fallback

// ------------------------------------------------------------------ scalar helpers
__device__ __forceinline__ float bf16_bits_to_float(uint32_t h16) {
  return __uint_as_float(h16 << 16);
}

// Sigmoid score with CUDA's full-precision expf and a correctly rounded reciprocal (the
// same value as the IEEE quotient 1.0f / (1.0f + e)).  Built without fast-math.
__device__ __forceinline__ float exact_score(float x) {
  return __frcp_rn(__fadd_rn(1.0f, expf(-x)));
}

// Order-preserving map of a float onto uint32 (for non-NaN values; -0 sorts below +0,
// which never matters here because keys are never -0).
__device__ __forceinline__ uint32_t ordered_bits(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// (key desc, expert asc) as one integer: larger composite = better route.
__device__ __forceinline__ unsigned long long composite(float key, int e) {
  return (static_cast<unsigned long long>(ordered_bits(key)) << 32) |
         static_cast<unsigned long long>(0xffffffffu - static_cast<uint32_t>(e));
}

__device__ __forceinline__ int composite_expert(unsigned long long c) {
  return static_cast<int>(0xffffffffu - static_cast<uint32_t>(c & 0xffffffffull));
}

__device__ __forceinline__ unsigned lanemask_lt(int lane) { return (1u << lane) - 1u; }

__device__ __forceinline__ int warp_inclusive_sum(int v, int lane) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(kFull, v, d);
    if (lane >= d) v += o;
  }
  return v;
}

// K-th largest of one float per lane (1 <= k <= 32), by counting for each lane how many
// lanes beat it (larger value, or equal value and lower lane).  32 independent shuffles:
// short dependency chains, for latency-bound callers.
__device__ __forceinline__ float warp_kth_largest(float v, int k, int lane) {
  int rank = 0;
#pragma unroll
  for (int m = 0; m < 32; ++m) {
    const float o = __shfl_sync(kFull, v, m);
    rank += ((o > v) || (o == v && m < lane)) ? 1 : 0;
  }
  const unsigned b = __ballot_sync(kFull, rank == k - 1);
  return __shfl_sync(kFull, v, __ffs(b) - 1);
}

// Programmatic dependent launch: wait until the previous kernel of the stream has completed
// and its memory is visible (returns at once when there is none), and let the next kernel
// of the stream be scheduled early (it waits the same way).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Ask L2 for the line that holds byte p of global memory.  A prefetch is only a hint: it
// changes no value that any load observes (L2 is where the device's writes become
// coherent), so it may be issued before pdl_wait, while the kernel ahead in the stream is
// still running, for inputs that kernel does not produce.
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Prefetch bytes [0, n) of the buffer at p into L2, one line per thread and step; threads
// [t0, t0 + nt) of the block take part.
__device__ __forceinline__ void prefetch_l2_range(const void* p, size_t n, int t, int nt) {
  const char* c = static_cast<const char*>(p);
  for (size_t o = static_cast<size_t>(t) * 128u; o < n; o += static_cast<size_t>(nt) * 128u)
    prefetch_l2(c + o);
}

// ------------------------------------------------------------------ proxy score
// Cheap stand-in for the selection key, shifted by the constant -0.5 that every expert
// shares: p = 0.5 * tanh.approx(0.5 x) + bias.  0.5 + 0.5 tanh(x / 2) is the logistic
// function, so p + 0.5 differs from the exact key s + bias by the hardware tanh
// approximation plus the roundings of p and of the exact key (values below max|bias| + 1
// in magnitude); proxy_delta() bounds the total for biases up to kProxyBiasLimit.  The
// selection only compares proxies with each other and uses them to discard experts that
// are worse than a proven bound by more than 2 * delta.
//
// kProxyTanhBound bounds |0.5 * tanh.approx(0.5 x) + 0.5 - s(x)| over all 65,536 bf16 x.
// The instruction's documented relative error (about 2^-11) would allow 2^-12; the sm_103a
// hardware is far closer (3.6e-6 over every bf16 input).  The bound used, 2^-16, keeps a
// 4x margin over that measurement, and moe_route_sort_proxy_selftest (run by the GPU tests)
// re-checks it exhaustively on the device: every decision's exactness rests on it.
constexpr float kProxyTanhBound = 1.0f / 65536.0f;
constexpr float kProxyBiasLimit = 1024.0f;

// Bound on |proxy + 0.5 - exact key| for biases of magnitude <= max_abs_bias: the tanh
// bound plus four half-ulp roundings of values below max_abs_bias + 1.5 (two are needed).
__host__ __device__ inline float proxy_delta(float max_abs_bias) {
  return kProxyTanhBound + (max_abs_bias + 2.0f) * 2.384185791e-7f;  // 2 * 2^-23
}

__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Half of each bf16 of the pair w (low half -> lo), as fp32: one bf16-operand FMA each,
// x * 0.5 + (-0), whose product is exact and unrounded, so the result equals 0.5f * x bit for
// bit (the argument of tanh.approx in the proxy score 0.5 * tanh.approx(0.5 x) + bias, the form
// the in-library check verifies) without a separate unpack.
__device__ __forceinline__ void half_bf16x2(uint32_t w, float& lo, float& hi) {
  asm("{ .reg .b16 l, u, c; mov.b16 c, 0x3F00; mov.b32 {l, u}, %2;\n"
      " fma.rn.f32.bf16 %0, l, c, 0f80000000; fma.rn.f32.bf16 %1, u, c, 0f80000000; }"
      : "=f"(lo), "=f"(hi)
      : "r"(w));
}

// Exact key and score of one logit: key = s + bias with s the exact score.
__device__ __forceinline__ float exact_key(float x, float bias, float& s) {
  s = exact_score(x);
  return __fadd_rn(s, bias);
}

// Softmax-scored routing selects on the logit itself.  Adding +0 turns a -0 logit into +0,
// so that the two zeros, equal as floats, also tie in the composite order (lower index wins).
__device__ __forceinline__ float logit_key(float x) { return __fadd_rn(x, 0.0f); }

// Score and selection key of one logit: the sigmoid score and score + bias, or with softmax
// scoring the logit for both (the weight step turns it into a softmax term).
__device__ __forceinline__ float score_key(float x, float bias, bool softmax, float& s) {
  if (softmax) {
    s = x;
    return logit_key(x);
  }
  return exact_key(x, bias, s);
}

// Softmax-scored routing: the logits x_k of the K selected slots (sel_s[0..K), slot 0 the
// largest) become the terms exp(x_k - x_0).  Renormalising them gives the softmax over all
// experts restricted to the selection (the common factor cancels), and no term exceeds 1.
// Called by every lane of the warp; lane slot `k` (< K) converts its own slot.
__device__ __forceinline__ void softmax_terms(float* sel_s, int k, int K) {
  const float x0 = sel_s[0];
  const float t = (k < K) ? expf(__fsub_rn(sel_s[k], x0)) : 0.0f;
  __syncwarp();
  if (k < K) sel_s[k] = t;
  __syncwarp();
}

// ------------------------------------------------------------------ route shape
struct RouteShape {
  int E, G, g, Kg, K;
  int L;       // lanes per group in the group pass (power of two)
  int log2L;
  int gpr;     // groups per round = 32 / L
  int rounds;  // ceil(G / gpr)
  float R;     // routed_scale
  int softmax; // 1: keys are the logits, weights the renormalised softmax (no bias)
};

// Per-warp shared scratch of the route step.
struct __align__(16) WarpScratch {
  unsigned long long cand[kCandCap];
  float cand_s[kCandCap];
  float gs[kMaxGroups];
  float p2[kMaxGroups];
  int kept[kMaxGroups];
  unsigned kept_mask[2];  // bit j of group j (groups 0..31, 32..63)
  int count;              // survivors appended so far
  int sel_id[kMaxTopk];
  float sel_s[kMaxTopk];
};

// ----------------------------------------------------------- step 1: group scores
// Group score = sum of the two largest keys of the group (the one key when g == 1).
// Lanes are split into 32/L slots of L lanes; slot i of round r owns group r*(32/L) + i.
template <class Src>
__device__ __forceinline__ void group_scores_proxy(const Src& src, const RouteShape& sh,
                                                   WarpScratch& ws, int lane) {
  const int q = lane & (sh.L - 1);
  const int slot = lane >> sh.log2L;
  for (int r = 0; r < sh.rounds; ++r) {
    const int j = r * sh.gpr + slot;
    float m1 = -INFINITY, m2 = -INFINITY;
    if (j < sh.G) {
      const int base = j * sh.g;
      for (int i = q; i < sh.g; i += sh.L) {
        const float v = src.proxy(base + i);
        m2 = fmaxf(m2, fminf(m1, v));
        m1 = fmaxf(m1, v);
      }
    }
    for (int d = 1; d < sh.L; d <<= 1) {
      const float o1 = __shfl_xor_sync(kFull, m1, d);
      const float o2 = __shfl_xor_sync(kFull, m2, d);
      m2 = fmaxf(fmaxf(m2, o2), fminf(m1, o1));
      m1 = fmaxf(m1, o1);
    }
    if (j < sh.G && q == 0) {
      ws.gs[j] = (sh.g >= 2) ? __fadd_rn(m1, m2) : m1;
      ws.p2[j] = (sh.g >= 2) ? m2 : m1;
    }
  }
  __syncwarp();
}

// Exact group scores: the exact top-2 of group j lie in the window proxy >= p2_j - 2*delta
// (order statistics of the proxies are within delta of those of the keys).
template <class Src>
__device__ __forceinline__ void group_scores_exact(const Src& src, const RouteShape& sh,
                                                   WarpScratch& ws, int lane) {
  const int q = lane & (sh.L - 1);
  const int slot = lane >> sh.log2L;
  for (int r = 0; r < sh.rounds; ++r) {
    const int j = r * sh.gpr + slot;
    float m1 = -INFINITY, m2 = -INFINITY;
    if (j < sh.G) {
      const int base = j * sh.g;
      const float lo = ws.p2[j] - 2.0f * Src::kDelta;
      for (int i = q; i < sh.g; i += sh.L) {
        if (src.proxy(base + i) >= lo) {
          float s;
          const float v = src.exact(base + i, s);
          m2 = fmaxf(m2, fminf(m1, v));
          m1 = fmaxf(m1, v);
        }
      }
    }
    for (int d = 1; d < sh.L; d <<= 1) {
      const float o1 = __shfl_xor_sync(kFull, m1, d);
      const float o2 = __shfl_xor_sync(kFull, m2, d);
      m2 = fmaxf(fmaxf(m2, o2), fminf(m1, o1));
      m1 = fmaxf(m1, o1);
    }
    if (j < sh.G && q == 0) ws.gs[j] = (sh.g >= 2) ? __fadd_rn(m1, m2) : m1;
  }
  __syncwarp();
}

// --------------------------------------------------------- step 2: kept groups
// Rank of group j = number of groups that beat it (higher score, or equal score and lower
// index); kept iff rank < Kg.  Writes the kept groups in ascending order to ws.kept.
// Returns false when `margin` >= 0 and the Kg-th and (Kg+1)-th scores are within `margin`
// (approximate scores cannot decide the kept set).
__device__ __forceinline__ bool rank_groups(const RouteShape& sh, WarpScratch& ws, int lane,
                                            float margin) {
  int r0 = 0x7fffffff, r1 = 0x7fffffff;
  float v0 = 0.0f, v1 = 0.0f;
  if (lane < sh.G) {
    v0 = ws.gs[lane];
    r0 = 0;
    for (int j = 0; j < sh.G; ++j) {
      const float o = ws.gs[j];
      r0 += (o > v0) || (o == v0 && j < lane);
    }
  }
  if (lane + 32 < sh.G) {
    v1 = ws.gs[lane + 32];
    r1 = 0;
    for (int j = 0; j < sh.G; ++j) {
      const float o = ws.gs[j];
      r1 += (o > v1) || (o == v1 && j < lane + 32);
    }
  }
  bool certain = true;
  if (margin >= 0.0f) {
    const unsigned ha = __ballot_sync(kFull, r0 == sh.Kg - 1 || r1 == sh.Kg - 1);
    const unsigned hb = __ballot_sync(kFull, r0 == sh.Kg || r1 == sh.Kg);
    const float va = __shfl_sync(kFull, r0 == sh.Kg - 1 ? v0 : v1, __ffs(ha) - 1);
    const float vb = __shfl_sync(kFull, r0 == sh.Kg ? v0 : v1, __ffs(hb) - 1);
    certain = (va - vb) > margin;  // Kg < G, so both ranks exist
  }
  __syncwarp();
  const bool k0 = r0 < sh.Kg, k1 = r1 < sh.Kg;
  const unsigned b0 = __ballot_sync(kFull, k0);
  const unsigned b1 = __ballot_sync(kFull, k1);
  if (k0) ws.kept[__popc(b0 & lanemask_lt(lane))] = lane;
  if (k1) ws.kept[__popc(b0) + __popc(b1 & lanemask_lt(lane))] = lane + 32;
  if (lane == 0) {
    ws.kept_mask[0] = b0;
    ws.kept_mask[1] = b1;
  }
  __syncwarp();
  return certain;
}

// Slots of the K best of ws.cand[0..total): rank = number of better composites (all
// composites are distinct, so ranks are 0..total-1).
__device__ __forceinline__ void rank_candidates(WarpScratch& ws, int total, int K, int lane) {
  for (int a = lane; a < total; a += 32) {
    const unsigned long long me = ws.cand[a];
    int rank = 0;
#pragma unroll 4
    for (int b = 0; b < total; ++b) rank += (ws.cand[b] > me) ? 1 : 0;
    if (rank < K) {
      ws.sel_id[rank] = composite_expert(me);
      ws.sel_s[rank] = ws.cand_s[a];
    }
  }
}

// Renormalised weights of the K selected experts: sum of scores in slot order, then
// (s_k / sum) * R; with `softmax` the scores are first the terms of softmax_terms.  Lane
// k < K returns slot k.
__device__ __forceinline__ void finish_weights(WarpScratch& ws, int K, float R, bool softmax,
                                               int lane, int& id, float& w) {
  if (softmax) softmax_terms(ws.sel_s, lane, K);
  const bool mine = lane < K;
  const float s = mine ? ws.sel_s[lane] : 0.0f;
  id = mine ? ws.sel_id[lane] : -1;
  float sum = 0.0f;
  if (lane == 0)
    for (int k = 0; k < K; ++k) sum = __fadd_rn(sum, ws.sel_s[k]);  // slot order
  sum = __shfl_sync(kFull, sum, 0);
  w = mine ? __fmul_rn(__fdiv_rn(s, sum), R) : 0.0f;
  __syncwarp();
}

// --------------------------------------------- step 3: top-K inside the kept groups
// tau = K-th largest of the 32 per-lane maxima of the proxies: at least K candidates have
// a proxy >= tau, so the K-th best exact key is >= tau - delta and every member of the
// exact top-K has proxy >= tau - 2*delta.  Those survivors get exact keys and are ranked
// by (key desc, expert asc); more than kCandCap survivors take a slower exact path.
template <class Src>
__device__ __forceinline__ void topk_in_kept(const Src& src, const RouteShape& sh,
                                             WarpScratch& ws, int lane) {
  const int g = sh.g;
  const bool all_kept = (sh.Kg == sh.G);
  // every slot gets a value even if non-finite keys leave fewer than K survivors
  if (lane < sh.K) {
    ws.sel_id[lane] = -1;
    ws.sel_s[lane] = 0.0f;
  }
  __syncwarp();
  float M = -INFINITY;
  for (int i = 0; i < sh.Kg; ++i) {
    const int base = (all_kept ? i : ws.kept[i]) * g;
    for (int c = lane; c < g; c += 32) M = fmaxf(M, src.proxy(base + c));
  }
  const float tau = warp_kth_largest(M, sh.K, lane);
  const float theta = (Src::kDelta > 0.0f) ? tau - 2.0f * Src::kDelta : tau;

  int cnt = 0;
  for (int i = 0; i < sh.Kg; ++i) {
    const int base = (all_kept ? i : ws.kept[i]) * g;
    for (int c = lane; c < g; c += 32) cnt += (src.proxy(base + c) >= theta) ? 1 : 0;
  }
  const int total = __reduce_add_sync(kFull, cnt);

  if (total <= kCandCap) {
    int w = warp_inclusive_sum(cnt, lane) - cnt;
    for (int i = 0; i < sh.Kg; ++i) {
      const int base = (all_kept ? i : ws.kept[i]) * g;
      for (int c = lane; c < g; c += 32) {
        const int e = base + c;
        if (src.proxy(e) >= theta) {
          float s;
          const float k = src.exact(e, s);
          ws.cand[w] = composite(k, e);
          ws.cand_s[w] = s;
          ++w;
        }
      }
    }
    __syncwarp();
    rank_candidates(ws, total, sh.K, lane);
  } else {
    // K rounds: the best exact composite strictly below the previous winner.
    unsigned long long prev = ~0ull;
    for (int k = 0; k < sh.K; ++k) {
      unsigned long long best = 0ull;
      float best_s = 0.0f;
      for (int i = 0; i < sh.Kg; ++i) {
        const int base = (all_kept ? i : ws.kept[i]) * g;
        for (int c = lane; c < g; c += 32) {
          const int e = base + c;
          if (src.proxy(e) >= theta) {
            float s;
            const float key = src.exact(e, s);
            const unsigned long long cc = composite(key, e);
            if (cc < prev && cc > best) {
              best = cc;
              best_s = s;
            }
          }
        }
      }
      unsigned long long wb = best;
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) {
        const unsigned long long o = __shfl_xor_sync(kFull, wb, d);
        wb = (o > wb) ? o : wb;
      }
      const unsigned owner = __ballot_sync(kFull, best == wb);
      const float ws_s = __shfl_sync(kFull, best_s, __ffs(owner) - 1);
      if (lane == 0) {
        ws.sel_id[k] = composite_expert(wb);
        ws.sel_s[k] = ws_s;
      }
      prev = wb;
    }
  }
  __syncwarp();
}

// --------------------------------------------------------------- the whole route step
// On return lane k < K holds the k-th selected expert in `id` and its weight in `w`
// (lanes >= K get id = -1, w = 0).
template <class Src>
__device__ __forceinline__ void route_token(const Src& src, const RouteShape& sh,
                                            WarpScratch& ws, int lane, int& id, float& w) {
  if (sh.Kg < sh.G) {
    group_scores_proxy(src, sh, ws, lane);
    if (Src::kDelta > 0.0f) {
      // approximate scores are within 2*delta (+ two roundings) of the exact ones
      const float margin = 2.0f * (2.0f * Src::kDelta + 1e-6f);
      if (!rank_groups(sh, ws, lane, margin)) {
        group_scores_exact(src, sh, ws, lane);
        rank_groups(sh, ws, lane, -1.0f);
      }
    } else {
      rank_groups(sh, ws, lane, -1.0f);
    }
  }
  topk_in_kept(src, sh, ws, lane);
  finish_weights(ws, sh.K, sh.R, sh.softmax != 0, lane, id, w);
}

// Key source over exact keys and scores already in shared memory.
struct SmemExactSrc {
  static constexpr float kDelta = 0.0f;
  const float* key;
  const float* s;
  __device__ __forceinline__ float proxy(int e) const { return key[e]; }
  __device__ __forceinline__ float exact(int e, float& se) const {
    se = s[e];
    return key[e];
  }
};

// ------------------------------------------------------- TMA bulk copies, mbarriers
// A device wait gives up after this long (an error bit is raised instead of hanging).  The
// launch argument `wait_limit_ns` carries it (a test hook can lower it to 0); waits for copies
// still in flight before a CTA exits always use this value.
constexpr unsigned long long kWaitLimitNs = 200ull * 1000ull * 1000ull;

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barrier of a cooperative launch over the word at bar (zeroed ahead of the launch
// by mrs_grid_prep_kernel): thread 0 of each CTA publishes the CTA's earlier writes and
// arrives, then waits, at most limit_ns (0: not at all, a test hook), until all n CTAs have
// arrived.  ok_s: one int of the CTA's shared memory.  Every thread of the CTA calls this;
// returns false on a timeout.
__device__ __forceinline__ bool grid_barrier_bounded(unsigned* bar, unsigned n,
                                                     unsigned long long limit_ns, int* ok_s) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(bar, 1u);
    bool ok = limit_ns != 0ull;
    if (ok) {
      const unsigned long long t0 = globaltimer_ns();
      while (ld_acquire_u32(bar) < n) {
        if (globaltimer_ns() - t0 > limit_ns) {
          ok = false;
          break;
        }
      }
    }
    *ok_s = ok ? 1 : 0;
  }
  __syncthreads();
  return *ok_s != 0;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(unsigned long long* mbar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(mbar)), "r"(count)
               : "memory");
}

// Ends the life of an mbarrier (no arrivals or copies pending on it) so that its shared
// memory can be used for something else.
__device__ __forceinline__ void mbar_inval(unsigned long long* mbar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(mbar)) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from global memory
// into shared memory, completing a transaction count of `bytes` on `mbar`.
__device__ __forceinline__ void tma_load_1d(void* dst, const void* src, uint32_t bytes,
                                            unsigned long long* mbar) {
  const uint32_t m = smem_u32(mbar);
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(m), "r"(bytes)
               : "memory");
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(m)
      : "memory");
}

// Orders this thread's earlier generic-proxy accesses to shared memory before later
// async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ bool mbar_try_wait(unsigned long long* mbar, uint32_t phase) {
  uint32_t done;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
      "selp.u32 %0, 1, 0, p; }"
      : "=r"(done)
      : "r"(smem_u32(mbar)), "r"(phase)
      : "memory");
  return done != 0u;
}

// Wait for phase `phase` of `mbar` to complete, at most `limit_ns` (0: report a timeout at
// once without looking, a test hook).  Every lane waits (each gets the acquire); the result
// is made warp-uniform.
__device__ __forceinline__ bool mbar_wait_bounded(unsigned long long* mbar, uint32_t phase,
                                                  unsigned long long limit_ns) {
  if (limit_ns == 0ull) return __all_sync(kFull, false);
  bool ok = mbar_try_wait(mbar, phase);
  if (!ok) {
    const unsigned long long t0 = globaltimer_ns();
    while (!(ok = mbar_try_wait(mbar, phase))) {
      if (globaltimer_ns() - t0 > limit_ns) break;
    }
  }
  return __all_sync(kFull, ok);
}

}  // namespace mrs
