// mrs_seg.cuh -- warp-level route step over contiguous per-lane segments of a group.
//
// Lane l of the warp owns group j = l / L and, inside it, the contiguous segment
// [j*g + q*sl, j*g + (q+1)*sl) with q = l % L and sl = g / L, read as units of 4 experts.
// One pass over the segment gives the lane's top-2 (and the best of every unit); the group
// score is a shuffle merge over the L lanes of the group; the K-th-best threshold comes from
// the lanes' own top-2; survivors are found by rescanning only units whose best can reach
// the threshold.  Source of the step: "perf(flydsl): Kimi-K3 B1 route-sort + prepared-MoE
// handoff (stack)", Summary (correction bias, grouped top-k).
//
// The row is read through a source with
//   unit(e0, v[4])   the 4 selection values (proxies, or exact keys) of experts e0..e0+3
//   exact(e, s)      the exact key of expert e, and its exact score through s
// and `delta` bounds |value - exact key| (0 for exact sources).  Decisions are exact:
// proxies only discard experts proven worse than a bound by more than 2 * delta.
#pragma once

#include "mrs_device.cuh"

namespace mrs {

struct SegShape {
  int E, G, g, Kg, K;
  int L, log2L;  // lanes per group (power of two); G * L <= 32
  int sl;        // experts per lane segment (multiple of 4)
  int nu;        // units of 4 experts per segment
  int rot;       // unit order of lane l starts at (l * rot) % nu (spreads smem banks)
  float R;
};

__device__ __forceinline__ void top2_insert(float& m1, float& m2, float v) {
  m2 = fmaxf(m2, fminf(m1, v));
  m1 = fmaxf(m1, v);
}

// Best of 4 values and the running top-2 after them.
__device__ __forceinline__ float top2_unit(const float (&v)[4], float& m1, float& m2) {
  const float h0 = fmaxf(v[0], v[1]), l0 = fminf(v[0], v[1]);
  const float h1 = fmaxf(v[2], v[3]), l1 = fminf(v[2], v[3]);
  const float a1 = fmaxf(h0, h1);
  float a2;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(a2) : "f"(fminf(h0, h1)), "f"(l0), "f"(l1));
  // merge (a1, a2) into (m1, m2)
  float n2;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(n2) : "f"(m2), "f"(fminf(m1, a1)), "f"(a2));
  m2 = n2;
  m1 = fmaxf(m1, a1);
  return a1;
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
  __device__ __forceinline__ float exact(int e, float& se) const {
    se = s[e];
    return key[e];
  }
};

// A bf16 logit row in shared memory; values are proxies (multi-CTA path).
struct ProxyRow {
  const uint16_t* row;  // [E] bf16 bit patterns
  const float* c;       // [E] 0.5 + bias
  const float* bias;    // [E]
  __device__ __forceinline__ void unit(int e0, float (&v)[4]) const {
    const uint2 w = *reinterpret_cast<const uint2*>(row + e0);
    const float4 cc = *reinterpret_cast<const float4*>(c + e0);
    v[0] = proxy_key(__uint_as_float(w.x << 16), cc.x);
    v[1] = proxy_key(__uint_as_float(w.x & 0xffff0000u), cc.y);
    v[2] = proxy_key(__uint_as_float(w.y << 16), cc.z);
    v[3] = proxy_key(__uint_as_float(w.y & 0xffff0000u), cc.w);
  }
  __device__ __forceinline__ float exact(int e, float& se) const {
    return exact_key(bf16_bits_to_float(row[e]), bias[e], se);
  }
};

// --------------------------------------------------------------- the route step
// umax: this warp's scratch of 32 * nu floats, unit-major (umax[u * 32 + lane]), holding the
// best value of every unit of the lane's segment.  Lane k < K returns slot k in (id, w).
template <class Row>
__device__ __forceinline__ void route_token_seg(const Row& row, const SegShape& sh,
                                                WarpScratch& ws, float* umax, int lane,
                                                float delta, int& id, float& w) {
  const int j = lane >> sh.log2L;          // my group
  const int q = lane & (sh.L - 1);
  const bool active = j < sh.G;
  const int seg0 = j * sh.g + q * sh.sl;   // first expert of my segment
  float* my_umax = umax + lane;  // unit u of my segment at my_umax[u * 32]

  // ---- pass 1: top-2 of my segment, best of each unit
  float m1 = -INFINITY, m2 = -INFINITY;
  if (active) {
    int u = (lane * sh.rot) % sh.nu;
#pragma unroll 4
    for (int k = 0; k < sh.nu; ++k) {
      float v[4];
      row.unit(seg0 + 4 * u, v);
      my_umax[u * 32] = top2_unit(v, m1, m2);
      u = (u + 1 == sh.nu) ? 0 : u + 1;
    }
  }
  // ---- group score: merge the L lanes of the group
  float g1 = m1, g2 = m2;
  for (int d = 1; d < sh.L; d <<= 1) {
    const float o1 = __shfl_xor_sync(kFull, g1, d);
    const float o2 = __shfl_xor_sync(kFull, g2, d);
    float n2;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(n2) : "f"(g2), "f"(o2), "f"(fminf(g1, o1)));
    g2 = n2;
    g1 = fmaxf(g1, o1);
  }
  bool kept = active;
  if (sh.Kg < sh.G) {
    float gs = active ? __fadd_rn(g1, g2) : -INFINITY;
    // rank of my group among the G groups (leaders are lanes i * L)
    int rank = 0;
    for (int i = 0; i < sh.G; ++i) {
      const float o = __shfl_sync(kFull, gs, i << sh.log2L);
      rank += (o > gs || (o == gs && i < j)) ? 1 : 0;
    }
    const float eta = 2.0f * delta + 1e-6f;  // |approximate - exact group score| bound
    bool certain = true;
    float A = 0.0f, B = 0.0f;
    if (delta > 0.0f) {
      const unsigned ha = __ballot_sync(kFull, active && rank == sh.Kg - 1);
      const unsigned hb = __ballot_sync(kFull, active && rank == sh.Kg);
      A = __shfl_sync(kFull, gs, __ffs(ha) - 1);
      B = __shfl_sync(kFull, gs, __ffs(hb) - 1);
      certain = (A - B) > 2.0f * eta;
    }
    if (certain) {
      kept = active && rank < sh.Kg;
    } else {
      // groups within 2*eta of the boundary get exact scores; the others keep their side
      const bool surely_in = active && gs > B + 2.0f * eta;
      const bool unsure = active && !surely_in && gs >= A - 2.0f * eta;
      float x1 = -INFINITY, x2 = -INFINITY;
      if (unsure) {
        const float lo = g2 - 2.0f * delta;  // exact top-2 of the group lie in this window
        for (int u = 0; u < sh.nu; ++u) {
          if (my_umax[u * 32] >= lo) {
            float v[4];
            row.unit(seg0 + 4 * u, v);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              if (v[t] >= lo) {
                float s;
                top2_insert(x1, x2, row.exact(seg0 + 4 * u + t, s));
              }
            }
          }
        }
      }
      for (int d = 1; d < sh.L; d <<= 1) {
        const float o1 = __shfl_xor_sync(kFull, x1, d);
        const float o2 = __shfl_xor_sync(kFull, x2, d);
        float n2;
        asm("max.f32 %0, %1, %2, %3;" : "=f"(n2) : "f"(x2), "f"(o2), "f"(fminf(x1, o1)));
        x2 = n2;
        x1 = fmaxf(x1, o1);
      }
      const float xs = unsure ? __fadd_rn(x1, x2) : -INFINITY;
      const unsigned in_mask = __ballot_sync(kFull, surely_in && q == 0);
      const int slots = sh.Kg - __popc(in_mask);
      int xr = 0;
      for (int i = 0; i < sh.G; ++i) {
        const int src = i << sh.log2L;
        const float o = __shfl_sync(kFull, xs, src);
        const bool ou = __shfl_sync(kFull, unsure ? 1 : 0, src) != 0;
        xr += (ou && (o > xs || (o == xs && i < j))) ? 1 : 0;
      }
      kept = surely_in || (unsure && xr < slots);
    }
  }

  // ---- top-K threshold from the lanes' own top-2 (lanes of kept groups only): at least
  // ceil(K/2) lanes hold two values >= t2, so at least K values are >= t2; when fewer lanes
  // are kept, t1 = the K-th best lane maximum is the bound
  const float k2 = kept ? m2 : -INFINITY;
  float tau = __shfl_sync(kFull, warp_sort_desc(k2, lane), (sh.K - 1) >> 1);
  if (tau == -INFINITY) {
    const float k1 = kept ? m1 : -INFINITY;
    tau = __shfl_sync(kFull, warp_sort_desc(k1, lane), sh.K - 1);
  }
  const float theta = tau - 2.0f * delta;

  // ---- survivors: my units whose best reaches theta, compacted without atomics: count,
  // warp scan for each lane's first slot, then write (the few surviving units are read twice)
  if (lane < sh.K) {
    ws.sel_id[lane] = -1;
    ws.sel_s[lane] = 0.0f;
  }
  const bool scan_mine = kept && m1 >= theta;
  int found = 0;
  if (scan_mine) {
    for (int u = 0; u < sh.nu; ++u) {
      if (my_umax[u * 32] >= theta) {
        float v[4];
        row.unit(seg0 + 4 * u, v);
#pragma unroll
        for (int t = 0; t < 4; ++t) found += (v[t] >= theta) ? 1 : 0;
      }
    }
  }
  const int incl = warp_inclusive_sum(found, lane);
  const int total = __shfl_sync(kFull, incl, 31);
  if (total <= kCandCap && found > 0) {
    int pos = incl - found;
    for (int u = 0; u < sh.nu; ++u) {
      if (my_umax[u * 32] >= theta) {
        float v[4];
        row.unit(seg0 + 4 * u, v);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          if (v[t] >= theta) ws.cand[pos++] = static_cast<unsigned long long>(seg0 + 4 * u + t);
        }
      }
    }
  }
  __syncwarp();
  if (total <= kCandCap) {
    for (int a = lane; a < total; a += 32) {
      const int e = static_cast<int>(ws.cand[a]);
      float s;
      const float k = row.exact(e, s);
      ws.cand[a] = composite(k, e);
      ws.cand_s[a] = s;
    }
    __syncwarp();
    rank_candidates(ws, total, sh.K, lane);
  } else {
    // many survivors (wide ties): K rounds of the best exact composite below the last one
    unsigned long long prev = ~0ull;
    for (int k = 0; k < sh.K; ++k) {
      unsigned long long best = 0ull;
      float best_s = 0.0f;
      if (scan_mine) {
        for (int u = 0; u < sh.nu; ++u) {
          if (my_umax[u * 32] >= theta) {
            float v[4];
            row.unit(seg0 + 4 * u, v);
            for (int t = 0; t < 4; ++t) {
              if (v[t] >= theta) {
                const int e = seg0 + 4 * u + t;
                float s;
                const unsigned long long c = composite(row.exact(e, s), e);
                if (c < prev && c > best) {
                  best = c;
                  best_s = s;
                }
              }
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
      const unsigned owner = __ballot_sync(kFull, best == wb && wb != 0ull);
      const float ws_s = __shfl_sync(kFull, best_s, owner ? __ffs(owner) - 1 : 0);
      if (lane == 0 && wb != 0ull) {
        ws.sel_id[k] = composite_expert(wb);
        ws.sel_s[k] = ws_s;
      }
      prev = wb;
    }
  }
  __syncwarp();
  finish_weights(ws, sh.K, sh.R, lane, id, w);
}

}  // namespace mrs
