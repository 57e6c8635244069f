// mrs_filter.cuh -- route step of one token by a logit threshold table: exact selection from
// a small candidate set, with a proof that nothing outside the set could have been selected.
//
// For a bound theta and expert e with bias b_e, filter_threshold() gives the bf16 value X_e
// such that every bf16 logit x < X_e has exact key s(x) + b_e < theta (exact_key as the path
// computes it: CUDA expf, correctly rounded reciprocal, one fp32 add).  Comparing a row with
// the table (two bf16 values per instruction) therefore yields a candidate set C that holds
// every expert whose key reaches theta.  Exact keys of the candidates then decide, per token:
//   groups  a group is complete when its two best keys (its best, when a group has one
//           expert) reach theta: those are then its true top two, since every expert left out
//           is below theta.  An incomplete group's score is bounded above by best + theta
//           (or 2 theta).  The kept groups are the Kg best under these scores/bounds (equal
//           values: lower group first); the selection is certain when all of them are
//           complete, since a bound that ranks below a group ranks the true score below it
//   top-K   the K best candidates of kept groups (key desc, expert asc), certain when the K-th
//           of them reaches theta: every expert left out is below it
// When a check fails (or the candidates overflow the scratch), filter_route() returns false
// and the caller routes the token another way; its results are then never used.  Nothing
// here depends on how theta was chosen: a poor theta only costs fallbacks.
// Source of the step: "perf(flydsl): Kimi-K3 B1 route-sort + prepared-MoE handoff (stack)",
// Summary (FP32 logit conversion + correction bias, grouped top-k).
#pragma once

#include <cuda_bf16.h>

#include "mrs_device.cuh"
#include "mrs_seg.cuh"

namespace mrs {

constexpr int kFilterCap = 128;            // candidates one token may have
constexpr float kFilterBiasLimit = 1.0f;   // |bias| up to which the table bound is proven

struct __align__(16) FilterScratch {
  unsigned long long comp[kFilterCap];   // composite (key desc, expert asc) of candidate j
  unsigned long long kcomp[kFilterCap];  // composites of the kept groups' candidates
  float s[kFilterCap];                   // exact score of candidate j
  float ks[kFilterCap];                  // scores of the kept groups' candidates
  uint32_t rec[kFilterCap];              // (bf16 bits << 16) | expert, as found
  unsigned long long gbest1[kMaxGroups], gbest2[kMaxGroups];  // best two composites per group
  int sel_id[kMaxTopk];
  float sel_s[kMaxTopk];
};

// The smallest bf16 value that is >= v (v finite).
__device__ __forceinline__ uint16_t bf16_round_up(float v) {
  const uint32_t u = __float_as_uint(v);
  if ((u & 0xffffu) == 0u) return static_cast<uint16_t>(u >> 16);
  if (u & 0x80000000u) return static_cast<uint16_t>(u >> 16);  // negative: toward zero
  return static_cast<uint16_t>((u >> 16) + 1u);
}

// X_e for bound theta and bias b (|b| <= kFilterBiasLimit, |theta| <= 2): every bf16 x < X_e
// has exact_key(x, b) < theta.  Let p = theta - b - 2e-6, rounded down.  If x < logit(p) then
// s(x) < p, the computed score is within 2.4e-7 of s(x), and key = RN(score + b) is below
// theta - 2e-6 + 2.4e-7 + ulp/2 < theta.  logit(p) = log(p) - log1p(-p) is evaluated with
// CUDA's logf/log1pf (1 ulp each) and lowered by far more than their error before rounding up
// to bf16.  p <= 0: every x may reach theta (-inf); p >= 1: none can (+inf).
__device__ __forceinline__ uint16_t filter_threshold(float theta, float b) {
  const float p = __fsub_rd(__fsub_rd(theta, b), 2.0e-6f);
  if (!(p > 0.0f)) return 0xff80u;  // -inf
  if (p >= 1.0f) return 0x7f80u;    // +inf
  const float lp = logf(p), lq = log1pf(-p);
  const float L = __fsub_rd(__fsub_rd(lp, lq), 1.0e-5f * (1.0f + fabsf(lp) + fabsf(lq)));
  return bf16_round_up(L);
}

// Bits b (0..7) of the result: element b of the 8 bf16 values in v is >= the matching
// threshold in th (element 2i is the low half of word i).  __hge2_mask gives 0xffff in each
// half where the comparison holds (false for NaN).
__device__ __forceinline__ unsigned ge_mask8(const uint4& v, const uint4& th) {
  const __nv_bfloat162* a = reinterpret_cast<const __nv_bfloat162*>(&v);
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&th);
  const unsigned m0 = __hge2_mask(a[0], b[0]), m1 = __hge2_mask(a[1], b[1]);
  const unsigned m2 = __hge2_mask(a[2], b[2]), m3 = __hge2_mask(a[3], b[3]);
  return (m0 & 1u) | ((m0 >> 15) & 2u) | ((m1 & 1u) << 2) | ((m1 >> 13) & 8u) |
         ((m2 & 1u) << 4) | ((m2 >> 11) & 32u) | ((m3 & 1u) << 6) | ((m3 >> 9) & 128u);
}

__device__ __forceinline__ uint4 ld_stream_u4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Brings `bytes` (multiple of 16, 16-byte aligned) from global memory into L2 ahead of use.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// The key of a composite (inverse of ordered_bits on its upper half).
__device__ __forceinline__ float composite_key(unsigned long long c) {
  const uint32_t u = static_cast<uint32_t>(c >> 32);
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

// bf16 bits of element b (0..7) of a 16-byte vector.
__device__ __forceinline__ uint32_t vec_bits(const uint4& v, int b) {
  const uint32_t w = (b < 2) ? v.x : (b < 4) ? v.y : (b < 6) ? v.z : v.w;
  return (b & 1) ? (w >> 16) : (w & 0xffffu);
}

// The route step of one token by the whole warp (see the file comment).  row: the token's
// bf16 logits (global, 16-byte aligned, E % 8 == 0); table, bias: shared memory.  Returns
// false if the selection could not be proven (id and w are then meaningless).  On true, lane
// k < K holds slot k in (id, w).
__device__ __forceinline__ bool filter_route(const uint16_t* row, const uint16_t* table,
                                             const float* bias, float theta, const SegShape& sh,
                                             FilterScratch& fs, int lane, int& id, float& w) {
  const int E = sh.E, G = sh.G, g = sh.g, Kg = sh.Kg, K = sh.K;
  const int nv = E >> 3;
  const uint4* r4 = reinterpret_cast<const uint4*>(row);
  const uint4* t4 = reinterpret_cast<const uint4*>(table);
  const unsigned lt = lanemask_lt(lane);
  // ---- candidates: elements at or above their expert's threshold.  Eight vectors per lane
  // in flight; their candidates are appended together (one warp scan per eight vectors).
  int total = 0;
  for (int c0 = 0; c0 < nv; c0 += 8 * 32) {
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = c0 + lane + 32 * i;
      v[i] = (c < nv) ? ld_stream_u4(r4 + c) : make_uint4(0u, 0u, 0u, 0u);
    }
    unsigned m[8];
    int n = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = c0 + lane + 32 * i;
      m[i] = (c < nv) ? ge_mask8(v[i], t4[c]) : 0u;
      n += __popc(m[i]);
    }
    if (__any_sync(kFull, n != 0)) {
      const int incl = warp_inclusive_sum(n, lane);
      int pos = total + incl - n;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        for (unsigned mm = m[i]; mm != 0u; mm &= mm - 1u) {
          const int b = __ffs(mm) - 1;
          if (pos < kFilterCap)
            fs.rec[pos] = (vec_bits(v[i], b) << 16) | (8 * (c0 + lane + 32 * i) + b);
          ++pos;
        }
      }
      total += __shfl_sync(kFull, incl, 31);
    }
  }
  if (total > kFilterCap || total < K) return false;
  if (lane < G) fs.gbest1[lane] = fs.gbest2[lane] = 0ull;  // 0: no candidate (worst)
  if (lane + 32 < G) fs.gbest1[lane + 32] = fs.gbest2[lane + 32] = 0ull;
  __syncwarp();
  // ---- exact keys of the candidates; the best composite of every group
  for (int j = lane; j < total; j += 32) {
    const uint32_t r = fs.rec[j];
    const int e = static_cast<int>(r & 0xffffu);
    float s;
    const float k = exact_key(bf16_bits_to_float(r >> 16), bias[e], s);
    const unsigned long long c = composite(k, e);
    fs.comp[j] = c;
    fs.s[j] = s;
    if (Kg < G) atomicMax(&fs.gbest1[e / g], c);
  }
  __syncwarp();
  unsigned long long kept = ~0ull;  // bit j: group j kept
  if (Kg < G) {
    // ---- the second best composite of every group
    for (int j = lane; j < total; j += 32) {
      const unsigned long long c = fs.comp[j];
      const int grp = composite_expert(c) / g;
      if (c != fs.gbest1[grp]) atomicMax(&fs.gbest2[grp], c);
    }
    __syncwarp();
    // ---- kept groups: scores of complete groups, upper bounds of the others
    float ub[2];
    bool complete[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int m = lane + 32 * h;
      ub[h] = -INFINITY;
      complete[h] = true;
      if (m < G) {
        const unsigned long long c1 = fs.gbest1[m], c2 = fs.gbest2[m];
        const float t1 = c1 ? composite_key(c1) : -INFINITY;
        const float t2 = c2 ? composite_key(c2) : -INFINITY;
        if (g >= 2) {
          complete[h] = t2 >= theta;
          ub[h] = complete[h] ? __fadd_rn(t1, t2)
                              : (t1 >= theta ? __fadd_rn(t1, theta) : __fadd_rn(theta, theta));
        } else {
          complete[h] = t1 >= theta;
          ub[h] = complete[h] ? t1 : theta;
        }
      }
    }
    int rk0 = 0, rk1 = 0;
    for (int m = 0; m < G; ++m) {
      const float o = __shfl_sync(kFull, (m < 32) ? ub[0] : ub[1], m & 31);
      rk0 += (o > ub[0] || (o == ub[0] && m < lane)) ? 1 : 0;
      rk1 += (o > ub[1] || (o == ub[1] && m < lane + 32)) ? 1 : 0;
    }
    const bool k0 = lane < G && rk0 < Kg, k1 = lane + 32 < G && rk1 < Kg;
    if (!__all_sync(kFull, (!k0 || complete[0]) && (!k1 || complete[1]))) return false;
    kept = static_cast<unsigned long long>(__ballot_sync(kFull, k0)) |
           (static_cast<unsigned long long>(__ballot_sync(kFull, k1)) << 32);
  }
  // ---- the kept groups' candidates, compacted
  int nk = 0;
  for (int j0 = 0; j0 < total; j0 += 32) {
    const int j = j0 + lane;
    const unsigned long long c = (j < total) ? fs.comp[j] : 0ull;
    const bool mine = j < total && ((kept >> (composite_expert(c) / g)) & 1ull);
    const unsigned b = __ballot_sync(kFull, mine);
    if (mine) {
      const int pos = nk + __popc(b & lt);
      fs.kcomp[pos] = c;
      fs.ks[pos] = fs.s[j];
    }
    nk += __popc(b);
  }
  if (nk < K) return false;
  __syncwarp();
  // ---- the K best of them by rank (composites are distinct); the K-th must reach theta
  bool cert = false;
  for (int a0 = lane; a0 < nk; a0 += 32) {
    const unsigned long long me = fs.kcomp[a0];
    int rk = 0;
#pragma unroll 4
    for (int b0 = 0; b0 < nk; ++b0) rk += (fs.kcomp[b0] > me) ? 1 : 0;
    if (rk < K) {
      fs.sel_id[rk] = composite_expert(me);
      fs.sel_s[rk] = fs.ks[a0];
    }
    cert |= (rk == K - 1) && composite_key(me) >= theta;
  }
  if (!__any_sync(kFull, cert)) return false;
  __syncwarp();
  // ---- renormalised weights: sum of the scores in slot order, then (s_k / sum) * R
  const bool mine = lane < K;
  const float s = mine ? fs.sel_s[lane] : 0.0f;
  id = mine ? fs.sel_id[lane] : -1;
  float4 q4[kMaxTopk / 4];
  const float4* s4 = reinterpret_cast<const float4*>(fs.sel_s);
#pragma unroll
  for (int i = 0; i < kMaxTopk / 4; ++i)
    q4[i] = (4 * i < K) ? s4[i] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  float sum = 0.0f;
#pragma unroll
  for (int i = 0; i < kMaxTopk / 4; ++i) {
    if (4 * i < K) sum = __fadd_rn(sum, q4[i].x);
    if (4 * i + 1 < K) sum = __fadd_rn(sum, q4[i].y);
    if (4 * i + 2 < K) sum = __fadd_rn(sum, q4[i].z);
    if (4 * i + 3 < K) sum = __fadd_rn(sum, q4[i].w);
  }
  w = mine ? __fmul_rn(__fdiv_rn(s, sum), sh.R) : 0.0f;
  __syncwarp();
  return true;
}

// A rough, cheap estimate for choosing theta from one token (the warp's pass-1 summary of it,
// lanes of 32 per token): the smaller of the K-th best sample of the kept groups and the
// second-best value of the Kg + 1 best groups, in key units.  No bound rests on it.
__device__ __forceinline__ float filter_calibrate(const SegShape& sh, const LaneTop& top,
                                                  int lane) {
  const int j = lane >> sh.log2L;
  const bool active = j < sh.G;
  float g1 = top.m1(), g2 = top.m2();
  for (int d = 1; d < sh.L; d <<= 1) {
    const float o1 = __shfl_xor_sync(kFull, g1, d);
    const float o2 = __shfl_xor_sync(kFull, g2, d);
    g2 = max3f(g2, o2, fminf(g1, o1));
    g1 = fmaxf(g1, o1);
  }
  const float gs = active ? __fadd_rn(g1, g2) : -INFINITY;
  int rank = 0;
  for (int i = 0; i < sh.G; ++i) {
    const float o = __shfl_sync(kFull, gs, i << sh.log2L);
    rank += (o > gs || (o == gs && i < j)) ? 1 : 0;
  }
  const bool kept = active && rank < sh.Kg;
  const bool near = active && rank <= sh.Kg;  // the kept groups and the next one
  const float ninf = -INFINITY;
  const float tau = seg_kth_desc2<32>(kept ? top.a1 : ninf, kept ? top.a2 : ninf, lane, sh.K - 1);
  float g2min = near ? g2 : INFINITY;
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) g2min = fminf(g2min, __shfl_xor_sync(kFull, g2min, d));
  return fminf(tau, g2min) + 0.5f;  // proxies are keys shifted by -0.5
}

}  // namespace mrs
