// mrs_unit.cuh -- phase 1 of the sort step for one unit (a contiguous token range): the
// unit's routes stable-sorted by expert in shared memory, with per-unit expert offsets.
// Shared by the route kernels (which run it after routing) and the moe_sort unit kernel.
// Source: "perf(flydsl): Kimi-K3 B1 route-sort + prepared-MoE handoff (stack)", Summary
// ("both sort phases").
#pragma once

#include "mrs_internal.h"

namespace mrs {

__device__ __forceinline__ void unit_range(int u, int T, int U, int& t0, int& t1) {
  t0 = static_cast<int>(static_cast<long long>(u) * T / U);
  t1 = static_cast<int>(static_cast<long long>(u + 1) * T / U);
}

// Exclusive prefix sum of v[0..n) by the whole block into out[0..n], out[n] = total.
// Warp w owns the contiguous chunk [w * per, (w + 1) * per) and reads it in rows of 32
// consecutive elements (conflict-free): one pass for the chunk total, then, after the
// cross-warp prefix, each row's warp scan plus the running carry.  scan_tmp: 33 ints.
// Ends with a block barrier.
__device__ __forceinline__ void block_exclusive_scan(const int32_t* v, int32_t* out, int n,
                                                     int32_t* scan_tmp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int per = (n + nwarps - 1) / nwarps;
  const int w0 = min(n, warp * per), w1 = min(n, w0 + per);
  int s = 0;
  for (int i = w0 + lane; i < w1; i += 32) s += v[i];
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) s += __shfl_xor_sync(kFull, s, d);
  if (lane == 0) scan_tmp[warp] = s;
  __syncthreads();
  if (warp == 0) {
    const int x = (lane < nwarps) ? scan_tmp[lane] : 0;
    const int xi = warp_inclusive_sum(x, lane);
    __syncwarp();
    if (lane < nwarps) scan_tmp[lane] = xi - x;
    if (lane == 31) scan_tmp[32] = xi;
  }
  __syncthreads();
  int carry = scan_tmp[warp];
#pragma unroll 4
  for (int i0 = w0; i0 < w1; i0 += 32) {
    const int i = i0 + lane;
    const int x = (i < w1) ? v[i] : 0;
    const int incl = warp_inclusive_sum(x, lane);
    if (i < w1) out[i] = carry + incl - x;
    carry += __shfl_sync(kFull, incl, 31);
  }
  if (tid == 0) out[n] = scan_tmp[32];
  __syncthreads();
}


// Places the routes of tokens [t0, t1) (rid/rw: shared memory, index (t - t0) * K + k; an id
// outside [0, E) is not placed) in expert order, stable by token then slot: route r of
// expert e goes to position run[e] + (number of earlier routes of e), and place(pos, r, e)
// stores it.  run[e] must hold each expert's first position; masks (2 * E words, zero on
// entry) and dup (two ints, zero on entry) are scratch.  All threads of the CTA call this;
// it ends with a block barrier.
//
// Tiles of 32 tokens: warp w takes tokens w, w + nwarps, ... of the tile, lane k slot k.
// Per tile: mark (bit of the token in its experts' masks), place (rank = earlier tokens of
// the tile in the mask, plus the expert's running count), advance (the tile's last token of
// an expert adds the mask's count and clears it).  Tile j uses mask buffer j & 1, so the
// next tile is marked in the same phase as this one advances: two barriers per tile.
template <class Place>
__device__ __forceinline__ void place_unit_routes(const int32_t* rid, int E, int K, int t0,
                                                  int t1, unsigned* masks, int32_t* run,
                                                  int32_t* dup2, const Place& place) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int nt_all = t1 - t0;
  auto mark = [&](int tb, unsigned* m, int32_t* dup) {
    const int nt = min(32, nt_all - tb);
    for (int tl = warp; tl < nt; tl += nwarps) {
      const int e = (lane < K) ? rid[(tb + tl) * K + lane] : -1;
      if (e >= 0 && e < E) {
        const unsigned bit = 1u << tl;
        if (atomicOr(&m[e], bit) & bit) *dup = 1;  // an expert twice in one token
      }
    }
  };
  if (nt_all > 0) mark(0, masks, &dup2[0]);
  __syncthreads();
  for (int tb = 0, j = 0; tb < nt_all; tb += 32, ++j) {
    const int nt = min(32, nt_all - tb);
    unsigned* m = masks + (j & 1) * E;
    unsigned* m_next = masks + ((j + 1) & 1) * E;
    int32_t* dup = &dup2[j & 1];
    int32_t* dup_next = &dup2[(j + 1) & 1];
    const bool more = tb + 32 < nt_all;
    if (*dup == 0) {
      for (int tl = warp; tl < nt; tl += nwarps) {
        const int r = (tb + tl) * K + lane;
        const int e = (lane < K) ? rid[r] : -1;
        if (e >= 0 && e < E) place(run[e] + __popc(m[e] & ((1u << tl) - 1u)), r, e);
      }
      __syncthreads();
      for (int tl = warp; tl < nt; tl += nwarps) {
        const int e = (lane < K) ? rid[(tb + tl) * K + lane] : -1;
        if (e >= 0 && e < E) {
          const unsigned mm = m[e];
          if ((mm >> tl) == 1u) {  // the tile's last token routed to e
            run[e] += __popc(mm);
            m[e] = 0u;
          }
        }
      }
      if (more) mark(tb + 32, m_next, dup_next);
      __syncthreads();
    } else {
      // repeated ids inside a token: place this tile's routes in flat order, 32 at a time
      const int nr = nt * K;
      const int r0 = tb * K;
      for (int i = tid; i < nr; i += blockDim.x) {
        const int e = rid[r0 + i];
        if (e >= 0 && e < E) m[e] = 0u;
      }
      __syncthreads();
      if (warp == 0) {
        for (int b0 = 0; b0 < nr; b0 += 32) {
          const int i = b0 + lane;
          const int e = (i < nr) ? rid[r0 + i] : -1;
          const bool valid = (e >= 0) && (e < E);
          const unsigned peers = __match_any_sync(kFull, valid ? e : -1 - lane);
          int p0 = 0;
          if (valid) {
            p0 = run[e];
            place(p0 + __popc(peers & lanemask_lt(lane)), r0 + i, e);
          }
          __syncwarp();
          if (valid && (peers >> lane) == 1u) run[e] = p0 + __popc(peers);
          __syncwarp();
        }
      }
      if (more) mark(tb + 32, m_next, dup_next);
      __syncthreads();
    }
    if (tid == 0) *dup = 0;  // read by every thread before this tile's first barrier
  }
}

// Phase 1 for unit u (see the file comment).  rid/rw: the unit's routes in shared memory,
// index (t - t0) * K + k; an id outside [0, E) is not placed.  cnt: the unit's per-expert
// counts of placed routes (shared memory, may be overwritten).  scratch: shared memory of
// unit_scratch_bytes(E), free for use.  Writes the unit's offsets, its sorted routes and
// their experts to uo.  All threads of the CTA call this.
__device__ __forceinline__ void unit_sort_tail(const int32_t* rid, const float* rw, int32_t* cnt,
                                               int E, int K, int u, int t0, int t1,
                                               unsigned char* scratch, const UnitOut& uo,
                                               int U) {
  unsigned long long* slice_flags = uo.slice_flags;
  const int nslices = uo.nslices;
  const int tid = threadIdx.x;
  // one bit per token of a 32-token tile, two buffers (tiles alternate)
  unsigned* masks = reinterpret_cast<unsigned*>(scratch);
  size_t o = align16(sizeof(unsigned long long) * E);
  int32_t* run = reinterpret_cast<int32_t*>(scratch + o);
  o += align16(sizeof(int32_t) * E);
  int32_t* loc = reinterpret_cast<int32_t*>(scratch + o);
  o += align16(sizeof(int32_t) * (E + 1));
  o += align16(sizeof(int32_t) * E);
  int32_t* misc = reinterpret_cast<int32_t*>(scratch + o);  // [0..32] scan, [40..41] dup flags

  // clear the look-back words and the status word for the slice kernel
  for (int c = u + tid * U; c < nslices; c += blockDim.x * U) slice_flags[c] = 0ull;
  if (u == 0 && tid == 0) *uo.status = 0;

  block_exclusive_scan(cnt, loc, E, misc);
  int32_t* loc_g = uo.loc_off + static_cast<size_t>(u) * (E + 1);
  for (int e = tid; e <= E; e += blockDim.x) loc_g[e] = loc[e];
  for (int e = tid; e < E; e += blockDim.x) {
    run[e] = loc[e];
    masks[e] = 0u;
    masks[E + e] = 0u;
  }
  if (tid == 0) {
    misc[40] = 0;
    misc[41] = 0;
  }
  __syncthreads();
  int2* out = uo.unit_buf + static_cast<size_t>(t0) * K;
  uint16_t* out_e = uo.unit_e + static_cast<size_t>(t0) * K;
  place_unit_routes(rid, E, K, t0, t1, masks, run, &misc[40], [&](int pos, int r, int e) {
    out[pos] = make_int2(t0 * K + r, __float_as_int(rw[r]));
    out_e[pos] = static_cast<uint16_t>(e);
  });
}

}  // namespace mrs
