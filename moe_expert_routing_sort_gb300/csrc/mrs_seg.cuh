// mrs_seg.cuh -- warp-level route step over contiguous per-lane segments of a group.
//
// A token is routed by LT consecutive lanes of a warp (LT = 32, or 16 for two tokens per
// warp).  Inside those, lane ll owns group j = ll / L and the contiguous segment
// [j*g + q*sl, j*g + (q+1)*sl) of it (q = ll % L, sl = g / L), read as units of 4 experts.
//   seg_pass1   the only step that reads the whole row: the lane's top-2 (in V interleaved
//               parts) and an upper bound of the best value of every unit (fp16, rounded up)
//   seg_select  the rest, from those summaries: group scores are a shuffle merge over the
//               L lanes of a group, the K-th-best threshold comes from the parts' top-2, and
//               only units whose bound reaches the threshold are read again
// The selection reads the row only up to the survivor step; after that it calls the
// caller's release(), so the row buffer can take the next row while the token finishes.
// Source of the step: "perf(flydsl): Kimi-K3 B1 route-sort + prepared-MoE handoff
// (stack)", Summary (correction bias, grouped top-k).
//
// A row source provides
//   unit(e0, v[4])          selection values (proxies or exact keys) of e0..e0+3
//   late_words(e0)          the raw bf16 words of e0..e0+3
//   values(e0, words, v[4]) the selection values from those words
//   exact(e, bits, s)       exact key of expert e (logit bits `bits`), score through s
//                           (for softmax scoring the logit, converted at the weight step)
// Selection values are the exact keys minus a constant shift common to all experts, up to
// `delta` (0 for exact sources).  Decisions are exact: values only discard experts proven
// worse than a bound by more than 2 * delta, and only differences of values are used.
#pragma once

#include <cuda_fp16.h>

#include "mrs_device.cuh"

namespace mrs {

struct SegShape {
  int E, G, g, Kg, K;
  int L, log2L;  // lanes per group (power of two); G * L <= lanes per token
  int sl;        // experts per lane segment (multiple of 4, at most 256)
  int nu;        // units of 4 experts per segment (at most 64)
  int rot, rsh;  // unit order of lane l (of its token) starts at ((l * rot) >> rsh) % nu:
                 // spreads pass 1's shared-memory loads over the banks (chosen per shape)
  float R;
  int softmax;   // 1: values are the logits (LogitRow), weights the renormalised softmax
};

// Hot units listed for the compacted survivor scan (the list reuses SegScratch::cand_s).
constexpr int kHotCap = 2 * kCandCap;

// Route scratch of one token (shared memory).
struct __align__(16) SegScratch {
  unsigned long long cand[kCandCap];
  float cand_s[kCandCap];
  int sel_id[kMaxTopk];
  float sel_s[kMaxTopk];
};

__device__ __forceinline__ void top2_insert(float& m1, float& m2, float v) {
  m2 = fmaxf(m2, fminf(m1, v));
  m1 = fmaxf(m1, v);
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Best of 4 values; the running top-2 absorbs them.
__device__ __forceinline__ float top2_unit(const float (&v)[4], float& m1, float& m2) {
  const float h0 = fmaxf(v[0], v[1]), l0 = fminf(v[0], v[1]);
  const float h1 = fmaxf(v[2], v[3]), l1 = fminf(v[2], v[3]);
  const float a1 = fmaxf(h0, h1);
  const float a2 = max3f(fminf(h0, h1), l0, l1);
  m2 = max3f(m2, fminf(m1, a1), a2);
  m1 = fmaxf(m1, a1);
  return a1;
}

// Unit bounds are kept as fp16 rounded towards +inf: still upper bounds, half the space.
__device__ __forceinline__ unsigned short ub_half(float v) {
  return __half_as_ushort(__float2half_ru(v));
}
__device__ __forceinline__ float ub_float(unsigned short h) {
  return __half2float(__ushort_as_half(h));
}

// ------------------------------------------------------------------ row sources
// Exact keys and scores already in shared memory (single-CTA path).
struct ExactKeyRow {
  const float* key;
  const float* s;
  __device__ __forceinline__ void unit(int e0, float (&v)[4]) const {
    const float4 q = *reinterpret_cast<const float4*>(key + e0);
    v[0] = q.x;
    v[1] = q.y;
    v[2] = q.z;
    v[3] = q.w;
  }
  __device__ __forceinline__ uint2 late_words(int) const { return make_uint2(0u, 0u); }
  __device__ __forceinline__ void values(int e0, uint2, float (&v)[4]) const { unit(e0, v); }
  __device__ __forceinline__ float exact(int e, uint32_t, float& se) const {
    se = s[e];
    return key[e];
  }
};

// A bf16 logit row staged in shared memory; values are the shifted proxies
// 0.5 * tanh.approx(0.5 x) + bias (the exact key minus 0.5, up to delta).
struct ProxyRow {
  const uint16_t* row;  // [E] bf16 bit patterns, shared memory
  const float* bias;    // [E] shared memory
  __device__ __forceinline__ void values(int e0, uint2 w, float (&v)[4]) const {
    const float4 bb = *reinterpret_cast<const float4*>(bias + e0);
    float h[4];
    half_bf16x2(w.x, h[0], h[1]);
    half_bf16x2(w.y, h[2], h[3]);
    v[0] = fmaf(0.5f, tanh_approx(h[0]), bb.x);
    v[1] = fmaf(0.5f, tanh_approx(h[1]), bb.y);
    v[2] = fmaf(0.5f, tanh_approx(h[2]), bb.z);
    v[3] = fmaf(0.5f, tanh_approx(h[3]), bb.w);
  }
  __device__ __forceinline__ uint2 late_words(int e0) const {
    return *reinterpret_cast<const uint2*>(row + e0);
  }
  __device__ __forceinline__ void unit(int e0, float (&v)[4]) const {
    values(e0, late_words(e0), v);
  }
  __device__ __forceinline__ float exact(int e, uint32_t bits, float& se) const {
    return exact_key(bf16_bits_to_float(static_cast<uint16_t>(bits)), bias[e], se);
  }
};

// A bf16 logit row staged in shared memory, selected on the logits themselves (softmax
// scoring): values are exact, so delta = 0; the score handed on is the logit, turned into a
// softmax term by the weight step.
struct LogitRow {
  const uint16_t* row;  // [E] bf16 bit patterns, shared memory
  __device__ __forceinline__ void values(int, uint2 w, float (&v)[4]) const {
    v[0] = __uint_as_float(w.x << 16);
    v[1] = __uint_as_float(w.x & 0xffff0000u);
    v[2] = __uint_as_float(w.y << 16);
    v[3] = __uint_as_float(w.y & 0xffff0000u);
  }
  __device__ __forceinline__ uint2 late_words(int e0) const {
    return *reinterpret_cast<const uint2*>(row + e0);
  }
  __device__ __forceinline__ void unit(int e0, float (&v)[4]) const {
    values(e0, late_words(e0), v);
  }
  __device__ __forceinline__ float exact(int, uint32_t bits, float& se) const {
    se = bf16_bits_to_float(bits);
    return logit_key(se);
  }
};

// bf16 bits of expert e0 + t from the two words of a unit.
__device__ __forceinline__ uint32_t unit_bits(uint2 w, int t) {
  const uint32_t word = (t < 2) ? w.x : w.y;
  return (t & 1) ? (word >> 16) : (word & 0xffffu);
}

// ------------------------------------------------------------------ unit bounds
// A warp's unit bounds live in shared memory as fp16 quads: the bound of unit u of lane l
// is half (u & 3) of the 8-byte word (u >> 2) * 32 + l; slots of units >= nu hold -inf.
__device__ __forceinline__ int ub_index(int lane, int u) {
  return ((((u >> 2) << 5) + lane) << 2) + (u & 3);
}

__device__ __forceinline__ float unit_ub(const unsigned short* umax, int lane, int u) {
  return ub_float(umax[ub_index(lane, u)]);
}

// Bytes of a warp's unit bounds.
__host__ __device__ inline size_t ub_bytes(int nu) {
  return static_cast<size_t>((nu + 3) >> 2) * 32 * 8;
}

// The pad slots of a lane's last quad; once per kernel (pass 1 never writes them).
__device__ __forceinline__ void ub_init_pads(unsigned short* umax, int lane, int nu) {
  for (int u = nu; u < ((nu + 3) & ~3); ++u) umax[ub_index(lane, u)] = 0xfc00u;  // -inf
}

// Bit u set for each unit (u < nu <= 64) whose bound may reach theta: bounds are compared
// in fp16 against theta rounded down, which can only add units.
__device__ __forceinline__ unsigned long long hot_units(const unsigned short* umax, int lane,
                                                        int nu, float theta) {
  const __half th = __float2half_rd(theta);
  const __half2 th2 = __halves2half2(th, th);
  const uint2* q = reinterpret_cast<const uint2*>(umax) + lane;
  unsigned long long hot = 0ull;
  const int nq = (nu + 3) >> 2;
#pragma unroll 4
  for (int i = 0; i < nq; ++i) {
    const uint2 x = q[i * 32];
    const unsigned ma = __hge2_mask(*reinterpret_cast<const __half2*>(&x.x), th2);
    const unsigned mb = __hge2_mask(*reinterpret_cast<const __half2*>(&x.y), th2);
    const unsigned nib = (ma & 1u) | ((ma >> 15) & 2u) | ((mb & 1u) << 2) | ((mb >> 13) & 8u);
    hot |= static_cast<unsigned long long>(nib) << (4 * i);
  }
  return hot;
}

// ------------------------------------------------------- helpers over LT-lane segments
template <int LT>
__device__ __forceinline__ unsigned seg_lanes(int lane) {
  return (LT == 32) ? kFull : (((1u << LT) - 1u) << (lane & ~(LT - 1)));
}

// Descending rank k (0-based) among two values per lane of my LT-lane segment (2 * LT
// values; element 2 * ll + r is register r of lane ll): bitonic sort over the segment.
template <int LT>
__device__ __forceinline__ float seg_kth_desc2(float v0, float v1, int ll, int k) {
#pragma unroll
  for (int kk = 2; kk <= 2 * LT; kk <<= 1) {
#pragma unroll
    for (int j = kk >> 1; j > 0; j >>= 1) {
      const bool desc = ((2 * ll) & kk) == 0;
      if (j == 1) {  // partners are the lane's own two registers
        const float hi = fmaxf(v0, v1), lo = fminf(v0, v1);
        v0 = desc ? hi : lo;
        v1 = desc ? lo : hi;
      } else {
        const int d = j >> 1;
        const bool lower = (ll & d) == 0;
        const float o0 = __shfl_xor_sync(kFull, v0, d);
        const float o1 = __shfl_xor_sync(kFull, v1, d);
        v0 = (desc == lower) ? fmaxf(v0, o0) : fminf(v0, o0);
        v1 = (desc == lower) ? fmaxf(v1, o1) : fminf(v1, o1);
      }
    }
  }
  const float a0 = __shfl_sync(kFull, v0, k >> 1, LT);
  const float a1 = __shfl_sync(kFull, v1, k >> 1, LT);
  return (k & 1) ? a1 : a0;
}

// Descending rank k (0-based) among four values per lane of my LT-lane segment (4 * LT values;
// element 4 * ll + r is register r of lane ll): bitonic sort over the segment, the two lowest
// index bits inside the lane.
template <int LT>
__device__ __forceinline__ float seg_kth_desc4(float v0, float v1, float v2, float v3, int ll,
                                               int k) {
  float v[4] = {v0, v1, v2, v3};
#pragma unroll
  for (int kk = 2; kk <= 4 * LT; kk <<= 1) {
#pragma unroll
    for (int j = kk >> 1; j > 0; j >>= 1) {
      if (j < 4) {  // partners are registers r and r ^ j of the lane
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          if ((r & j) == 0) {
            const bool desc = ((4 * ll + r) & kk) == 0;
            const float hi = fmaxf(v[r], v[r ^ j]), lo = fminf(v[r], v[r ^ j]);
            v[r] = desc ? hi : lo;
            v[r ^ j] = desc ? lo : hi;
          }
        }
      } else {
        const int d = j >> 2;  // lane distance
        const bool lower = (ll & d) == 0;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const bool desc = ((4 * ll + r) & kk) == 0;
          const float o = __shfl_xor_sync(kFull, v[r], d);
          v[r] = (desc == lower) ? fmaxf(v[r], o) : fminf(v[r], o);
        }
      }
    }
  }
  const int src = k >> 2;
  const float a0 = __shfl_sync(kFull, v[0], src, LT);
  const float a1 = __shfl_sync(kFull, v[1], src, LT);
  const float a2 = __shfl_sync(kFull, v[2], src, LT);
  const float a3 = __shfl_sync(kFull, v[3], src, LT);
  const int r = k & 3;
  return r == 0 ? a0 : (r == 1 ? a1 : (r == 2 ? a2 : a3));
}

// Pass-1 summary of a lane: with one part, the top-2 values of its segment; with two
// interleaved parts (part = unit step modulo 2), in each part the largest and second-largest
// unit maximum, which are values of two distinct experts (of two units).  s2 is the lane's
// true second-largest value over its whole segment either way.  The parts cover disjoint
// experts, so V parts give the threshold of the selection twice V samples per lane.
struct LaneTop {
  float a1, a2;  // part 0
  float b1, b2;  // part 1 (-inf when V == 1)
  float s2;      // second-largest value of the segment (= m1() when the largest occurs twice)
  __device__ __forceinline__ float m1() const { return fmaxf(a1, b1); }
  __device__ __forceinline__ float m2() const { return s2; }
};

// Second-largest of 4 values.
__device__ __forceinline__ float second_of4(const float (&v)[4]) {
  const float h0 = fmaxf(v[0], v[1]), l0 = fminf(v[0], v[1]);
  const float h1 = fmaxf(v[2], v[3]), l1 = fminf(v[2], v[3]);
  return max3f(fminf(h0, h1), l0, l1);
}

// A unit's maximum enters its part's top-2 of unit maxima (best unit in ubest).
__device__ __forceinline__ void unit_max_insert(float mx, int u, float& m1, float& m2,
                                                int& ubest) {
  ubest = (mx > m1) ? u : ubest;
  m2 = fmaxf(m2, fminf(m1, mx));
  m1 = fmaxf(m1, mx);
}

// ------------------------------------------------------------------------ pass 1
// umax: the warp's unit bounds.  Lanes of an invalid token (or beyond the groups) return
// -inf and write nothing.
template <int LT, int V, class Row>
__device__ __forceinline__ LaneTop seg_pass1(const Row& row, const SegShape& sh,
                                             unsigned short* umax, int lane, bool token_valid) {
  static_assert(V == 1 || V == 2, "one or two parts per lane");
  const int ll = lane & (LT - 1);
  const int j = ll >> sh.log2L;
  LaneTop r{-INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY};
  if (!token_valid || j >= sh.G) return r;
  const int seg0 = j * sh.g + (ll & (sh.L - 1)) * sh.sl;
  int u = ((ll * sh.rot) >> sh.rsh) % sh.nu;
  if constexpr (V == 1) {
    // one part: the exact top-2 of every unit enters the running top-2
#pragma unroll 4
    for (int k = 0; k < sh.nu; ++k) {
      float v[4];
      row.unit(seg0 + 4 * u, v);
      umax[ub_index(lane, u)] = ub_half(top2_unit(v, r.a1, r.a2));
      u = (u + 1 == sh.nu) ? 0 : u + 1;
    }
    r.s2 = r.a2;
  } else {
    // two parts: only each unit's maximum enters its part's top-2 (fewer operations per
    // unit); the segment's second value is then the other part's best, a runner-up unit
    // maximum, or the second value inside the unit that holds the largest
    int ua = u, ub = u;  // unit holding a1 / b1
    int k = 0;
#pragma unroll 2
    for (; k + 2 <= sh.nu; k += 2) {
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        float v[4];
        row.unit(seg0 + 4 * u, v);
        const float mx = max3f(v[0], v[1], fmaxf(v[2], v[3]));
        if (p == 0)
          unit_max_insert(mx, u, r.a1, r.a2, ua);
        else
          unit_max_insert(mx, u, r.b1, r.b2, ub);
        umax[ub_index(lane, u)] = ub_half(mx);
        u = (u + 1 == sh.nu) ? 0 : u + 1;
      }
    }
    if (k < sh.nu) {  // odd unit count
      float v[4];
      row.unit(seg0 + 4 * u, v);
      const float mx = max3f(v[0], v[1], fmaxf(v[2], v[3]));
      unit_max_insert(mx, u, r.a1, r.a2, ua);
      umax[ub_index(lane, u)] = ub_half(mx);
    }
    float v[4];
    row.unit(seg0 + 4 * ((r.a1 >= r.b1) ? ua : ub), v);
    r.s2 = max3f(fminf(r.a1, r.b1), fmaxf(r.a2, r.b2), second_of4(v));
  }
  return r;
}

// --------------------------------------------------------------------- selection
// Everything after pass 1 for the token of my segment; ws is that token's scratch.
// Every branch that holds a shuffle is uniform over the warp; release() is called once, by
// the whole warp, as soon as the row is no longer read.  Lane ll < K of the segment returns
// slot ll in (id, w).
template <int LT, int V, class Row, class Release>
__device__ __forceinline__ void seg_select(const Row& row, const SegShape& sh, SegScratch& ws,
                                           const unsigned short* umax, int lane, float delta,
                                           bool token_valid, const LaneTop& top,
                                           const Release& release, int& id, float& w) {
  const float m1 = top.m1(), m2 = top.m2();
  const int ll = lane & (LT - 1);
  const int j = ll >> sh.log2L;  // my group
  const int q = ll & (sh.L - 1);
  const bool active = token_valid && j < sh.G;
  const int seg0 = j * sh.g + q * sh.sl;
  const unsigned lanes = seg_lanes<LT>(lane);

  // ---- group score: merge the L lanes of the group
  float g1 = m1, g2 = m2;
  for (int d = 1; d < sh.L; d <<= 1) {
    const float o1 = __shfl_xor_sync(kFull, g1, d);
    const float o2 = __shfl_xor_sync(kFull, g2, d);
    g2 = max3f(g2, o2, fminf(g1, o1));
    g1 = fmaxf(g1, o1);
  }
  bool kept = active;
  if (sh.Kg < sh.G) {
    const float gs = active ? __fadd_rn(g1, g2) : -INFINITY;
    int rank = 0;  // groups that beat mine (group i's first lane is lane i * L)
#pragma unroll 4
    for (int i = 0; i < sh.G; ++i) {
      const float o = __shfl_sync(kFull, gs, i << sh.log2L, LT);
      rank += (o > gs || (o == gs && i < j)) ? 1 : 0;
    }
    kept = active && rank < sh.Kg;
    const float eta = 2.0f * delta + 1e-6f;  // |approximate - exact group score| bound
    bool certain = true;
    float A = 0.0f, B = 0.0f;
    if (delta > 0.0f) {
      const unsigned ha = __ballot_sync(kFull, active && rank == sh.Kg - 1) & lanes;
      const unsigned hb = __ballot_sync(kFull, active && rank == sh.Kg) & lanes;
      A = __shfl_sync(kFull, gs, ha ? __ffs(ha) - 1 : 0);
      B = __shfl_sync(kFull, gs, hb ? __ffs(hb) - 1 : 0);
      certain = !(ha && hb) || (A - B) > 2.0f * eta;
    }
    if (__any_sync(kFull, !certain)) {
      // groups within 2*eta of the boundary get exact scores; the others keep their side
      const bool surely_in = certain ? kept : (active && gs > B + 2.0f * eta);
      const bool unsure = !certain && active && !surely_in && gs >= A - 2.0f * eta;
      float x1 = -INFINITY, x2 = -INFINITY;
      if (unsure) {
        const float lo = g2 - 2.0f * delta;  // the exact top-2 of the group lie above this
        for (int u = 0; u < sh.nu; ++u) {
          if (unit_ub(umax, lane, u) >= lo) {
            const uint2 wd = row.late_words(seg0 + 4 * u);
            float v[4];
            row.values(seg0 + 4 * u, wd, v);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              if (v[t] >= lo) {
                float s;
                top2_insert(x1, x2, row.exact(seg0 + 4 * u + t, unit_bits(wd, t), s));
              }
            }
          }
        }
      }
      for (int d = 1; d < sh.L; d <<= 1) {
        const float o1 = __shfl_xor_sync(kFull, x1, d);
        const float o2 = __shfl_xor_sync(kFull, x2, d);
        x2 = max3f(x2, o2, fminf(x1, o1));
        x1 = fmaxf(x1, o1);
      }
      const float xs = unsure ? __fadd_rn(x1, x2) : -INFINITY;
      const unsigned in_mask = __ballot_sync(kFull, surely_in && q == 0) & lanes;
      const int slots = sh.Kg - __popc(in_mask);
      int xr = 0;
      for (int i = 0; i < sh.G; ++i) {
        const int src = i << sh.log2L;
        const float o = __shfl_sync(kFull, xs, src, LT);
        const bool ou = __shfl_sync(kFull, unsure ? 1 : 0, src, LT) != 0;
        xr += (ou && (o > xs || (o == xs && i < j))) ? 1 : 0;
      }
      if (!certain) kept = surely_in || (unsure && xr < slots);
    }
  }

  // ---- top-K threshold from the pass-1 samples of kept groups: the top-2 values of the
  // parts are values of distinct experts, so the K-th best of all of them has at least K
  // values at or above it.  -inf when the kept parts hold fewer than K samples.
  float tau;
  const float ninf = -INFINITY;
  if (V == 1) {
    tau = seg_kth_desc2<LT>(kept ? top.a1 : ninf, kept ? top.a2 : ninf, ll, sh.K - 1);
  } else {
    tau = seg_kth_desc4<LT>(kept ? top.a1 : ninf, kept ? top.a2 : ninf, kept ? top.b1 : ninf,
                            kept ? top.b2 : ninf, ll, sh.K - 1);
  }
  const float theta = tau - 2.0f * delta;

  // ---- survivors: values >= theta in units whose bound may reach theta.  The segment's hot
  // units are first compacted into one list (first expert of each unit, in lane order), so a
  // round reads LT of them whichever lanes own them; the next round's words are loaded
  // ahead.  Hits are appended as records (bf16 bits << 16) | expert at a segment-wide
  // running count.  (A list longer than kHotCap falls back to each lane walking its own.)
  if (ll < sh.K) {
    ws.sel_id[ll] = -1;
    ws.sel_s[ll] = 0.0f;
  }
  const bool scan_mine = kept && m1 >= theta;
  unsigned long long hot = scan_mine ? hot_units(umax, lane, sh.nu, theta) : 0ull;
  const unsigned lt = lanemask_lt(lane) & lanes;
  const int nh = __popcll(static_cast<long long>(hot));
  int incl = nh;  // inclusive prefix of the hot-unit counts over the segment
#pragma unroll
  for (int d = 1; d < LT; d <<= 1) {
    const int o = __shfl_up_sync(kFull, incl, d, LT);
    if (ll >= d) incl += o;
  }
  const int htot = __shfl_sync(kFull, incl, LT - 1, LT);
  int total = 0;
  // one record round: lane's unit at e0 (if have) with words wd
  auto round = [&](bool have, int e0, uint2 wd) {
    unsigned hits = 0u;
    if (have) {
      float v[4];
      row.values(e0, wd, v);
#pragma unroll
      for (int t = 0; t < 4; ++t) hits |= (v[t] >= theta) ? (1u << t) : 0u;
    }
    const int n = __popc(hits);
    const unsigned b0 = __ballot_sync(kFull, n & 1) & lanes;
    const unsigned b1 = __ballot_sync(kFull, n & 2) & lanes;
    const unsigned b2 = __ballot_sync(kFull, n & 4) & lanes;
    int pos = total + __popc(b0 & lt) + 2 * __popc(b1 & lt) + 4 * __popc(b2 & lt);
    total += __popc(b0) + 2 * __popc(b1) + 4 * __popc(b2);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      if ((hits >> t) & 1u) {
        if (pos < kCandCap)
          ws.cand[pos] = (unit_bits(wd, t) << 16) | static_cast<uint32_t>(e0 + t);
        ++pos;
      }
    }
  };
  if (__all_sync(kFull, htot <= kHotCap)) {
    unsigned short* list = reinterpret_cast<unsigned short*>(ws.cand_s);  // free until the
    for (int i = incl - nh; hot != 0ull; ++i) {                           // exact evaluation
      list[i] = static_cast<unsigned short>(seg0 + 4 * (__ffsll(static_cast<long long>(hot)) - 1));
      hot &= hot - 1ull;
    }
    __syncwarp();
    bool have = ll < htot;
    int e0 = have ? list[ll] : 0;
    uint2 wd = have ? row.late_words(e0) : make_uint2(0u, 0u);
    for (int r = 0; __any_sync(kFull, r < htot); r += LT) {
      const bool have_n = r + LT + ll < htot;
      const int e0_n = have_n ? list[r + LT + ll] : 0;
      const uint2 wd_n = have_n ? row.late_words(e0_n) : make_uint2(0u, 0u);
      round(have, e0, wd);
      have = have_n;
      e0 = e0_n;
      wd = wd_n;
    }
    __syncwarp();  // the list is overwritten by the exact scores below
  } else {
    bool have = hot != 0ull;
    int u = 0;
    uint2 wd = make_uint2(0u, 0u);
    if (have) {
      u = __ffsll(static_cast<long long>(hot)) - 1;
      hot &= hot - 1ull;
      wd = row.late_words(seg0 + 4 * u);
    }
    while (__any_sync(kFull, have)) {
      const bool have_n = hot != 0ull;
      int u_n = 0;
      uint2 wd_n = make_uint2(0u, 0u);
      if (have_n) {
        u_n = __ffsll(static_cast<long long>(hot)) - 1;
        hot &= hot - 1ull;
        wd_n = row.late_words(seg0 + 4 * u_n);
      }
      round(have, seg0 + 4 * u, wd);
      have = have_n;
      u = u_n;
      wd = wd_n;
    }
  }
  const bool fits = __all_sync(kFull, total <= kCandCap);
  if (fits) release();  // the records hold the logit bits; the row is not read again
  __syncwarp();
  if (fits) {
    for (int a = ll; a < total; a += LT) {
      const uint32_t r = static_cast<uint32_t>(ws.cand[a]);
      const int e = static_cast<int>(r & 0xffffu);
      float s;
      const float k = row.exact(e, r >> 16, s);
      ws.cand[a] = composite(k, e);
      ws.cand_s[a] = s;
    }
    __syncwarp();
    // slot = number of better composites (composites are distinct); two per lane at once
    for (int a0 = ll; a0 < total; a0 += 2 * LT) {
      const int a1 = a0 + LT;
      const unsigned long long me0 = ws.cand[a0];
      const unsigned long long me1 = (a1 < total) ? ws.cand[a1] : ~0ull;
      int r0 = 0, r1 = 0;
#pragma unroll 4
      for (int b = 0; b < total; ++b) {
        const unsigned long long c = ws.cand[b];
        r0 += (c > me0) ? 1 : 0;
        r1 += (c > me1) ? 1 : 0;
      }
      if (r0 < sh.K) {
        ws.sel_id[r0] = composite_expert(me0);
        ws.sel_s[r0] = ws.cand_s[a0];
      }
      if (a1 < total && r1 < sh.K) {
        ws.sel_id[r1] = composite_expert(me1);
        ws.sel_s[r1] = ws.cand_s[a1];
      }
    }
  } else {
    // very many survivors (wide ties): K rounds of the best exact composite below the last
    unsigned long long prev = ~0ull;
    for (int k = 0; k < sh.K; ++k) {
      unsigned long long best = 0ull;
      float best_s = 0.0f;
      if (scan_mine) {
        for (int uu = 0; uu < sh.nu; ++uu) {
          if (unit_ub(umax, lane, uu) >= theta) {
            const uint2 w2 = row.late_words(seg0 + 4 * uu);
            float v[4];
            row.values(seg0 + 4 * uu, w2, v);
            for (int t = 0; t < 4; ++t) {
              if (v[t] >= theta) {
                const int e = seg0 + 4 * uu + t;
                float s;
                const unsigned long long c = composite(row.exact(e, unit_bits(w2, t), s), e);
                if (c < prev && c > best) {
                  best = c;
                  best_s = s;
                }
              }
            }
          }
        }
      }
      unsigned long long wbest = best;
#pragma unroll
      for (int d = LT >> 1; d > 0; d >>= 1) {
        const unsigned long long o = __shfl_xor_sync(kFull, wbest, d);
        wbest = (o > wbest) ? o : wbest;
      }
      const unsigned owner = __ballot_sync(kFull, best == wbest && wbest != 0ull) & lanes;
      const float owner_s = __shfl_sync(kFull, best_s, owner ? __ffs(owner) - 1 : 0);
      if (ll == 0 && wbest != 0ull) {
        ws.sel_id[k] = composite_expert(wbest);
        ws.sel_s[k] = owner_s;
      }
      prev = wbest;
    }
    release();
  }
  __syncwarp();
  // ---- renormalised weights: sum of the scores in slot order, then (s_k / sum) * R
  if (sh.softmax) softmax_terms(ws.sel_s, ll, sh.K);
  const bool mine = ll < sh.K;
  const float s = mine ? ws.sel_s[ll] : 0.0f;
  id = mine ? ws.sel_id[ll] : -1;
  // every lane forms the same sum from the slot scores in shared memory, slot 0 first
  float4 q4[kMaxTopk / 4];
  const float4* s4 = reinterpret_cast<const float4*>(ws.sel_s);
#pragma unroll
  for (int i = 0; i < kMaxTopk / 4; ++i)
    q4[i] = (4 * i < sh.K) ? s4[i] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  float sum = 0.0f;
#pragma unroll
  for (int i = 0; i < kMaxTopk / 4; ++i) {
    if (4 * i < sh.K) sum = __fadd_rn(sum, q4[i].x);
    if (4 * i + 1 < sh.K) sum = __fadd_rn(sum, q4[i].y);
    if (4 * i + 2 < sh.K) sum = __fadd_rn(sum, q4[i].z);
    if (4 * i + 3 < sh.K) sum = __fadd_rn(sum, q4[i].w);
  }
  w = mine ? __fmul_rn(__fdiv_rn(s, sum), sh.R) : 0.0f;
  __syncwarp();
}

}  // namespace mrs
