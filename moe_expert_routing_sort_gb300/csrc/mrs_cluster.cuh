// mrs_cluster.cuh -- both sort phases for a route step that one thread-block cluster runs.
//
// For mid-sized token counts the route step of the segment kernel runs as a single cluster
// of kClusterCtas CTAs (one contiguous token range each).  Once every CTA has its routes and
// per-expert counts in shared memory, the CTAs read each other's counts through distributed
// shared memory, so each knows, for every expert e,
//   total(e)   = the routes of e in the whole call, and
//   before(e)  = the routes of e in the CTAs of lower rank (earlier tokens),
// and computes the same block_m-padded exclusive prefix over experts, base(e).  Route k of
// token t routed to e then goes straight to its final row
//   base(e) + before(e) + (routes of e in this CTA from earlier tokens or slots),
// which keeps every expert's rows in token-then-slot order.  The CTA of rank c writes the
// padding rows and block owners of the experts [c E / n, (c + 1) E / n); rank 0 writes npp and
// the status word.  One launch, no workspace traffic and no global waits: the only waits are
// the two hardware cluster barriers, which every CTA reaches on every path.
// Source: "perf(flydsl): Kimi-K3 B1 route-sort + prepared-MoE handoff (stack)", Summary (both
// sort phases in the same kernel as the routing); dropped routes (ids < 0) claim no row:
// "Summary -- general gfx1250 ordinary-TP route optimization", Dispatch and contracts.
#pragma once

#include "mrs_unit.cuh"

namespace mrs {

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The int32 at the shared-memory address that p has in this CTA, read from CTA `rank` of the
// cluster (every CTA of the kernel has the same shared-memory layout).
__device__ __forceinline__ int32_t ld_cluster_s32(const int32_t* p, uint32_t rank) {
  const uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  int32_t v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
  return v;
}

// The same for the four int32 at p (16-byte aligned).
__device__ __forceinline__ int4 ld_cluster_v4(const int32_t* p, uint32_t rank) {
  const uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  int4 v;
  asm volatile("ld.shared::cluster.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(remote)
               : "memory");
  return v;
}

// The sort step of CTA `rank` of an n-CTA cluster (n <= kClusterCtas) that routed tokens
// [t0, t1).  rid/rw: its routes (shared memory, index (t - t0) * K + k; ids outside [0, E) are
// not placed); cnt: its per-expert counts of placed routes (16-byte aligned); flag: its device
// status bits.  rid, cnt and flag must sit at the same shared-memory offsets in every CTA and
// stay unchanged until every CTA has passed the second cluster barrier arrival of this
// routine; they are not written here.  scratch: cluster_scratch_bytes(E) of free shared
// memory.  All threads of every CTA call this.
__device__ __forceinline__ void cluster_sort_tail(const int32_t* rid, const float* rw,
                                                  const int32_t* cnt, const int32_t* flag,
                                                  int E, int K, int t0, int t1, uint32_t rank,
                                                  uint32_t n, unsigned char* scratch,
                                                  const ClusterOut& co) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int B = co.B;
  unsigned* masks = reinterpret_cast<unsigned*>(scratch);
  size_t o = align16(sizeof(unsigned) * 2 * static_cast<size_t>(E));
  int32_t* run = reinterpret_cast<int32_t*>(scratch + o);
  o += align16(sizeof(int32_t) * static_cast<size_t>(E));
  int32_t* pad = reinterpret_cast<int32_t*>(scratch + o);
  o += align16(sizeof(int32_t) * static_cast<size_t>(E));
  int32_t* tot = reinterpret_cast<int32_t*>(scratch + o);
  o += align16(sizeof(int32_t) * static_cast<size_t>(E));
  int32_t* base = reinterpret_cast<int32_t*>(scratch + o);
  o += align16(sizeof(int32_t) * (static_cast<size_t>(E) + 1));
  int32_t* misc = reinterpret_cast<int32_t*>(scratch + o);  // [0..32] scan, [40..41] dup flags

  // every CTA's counts and flags are final and visible once all have arrived
  cluster_arrive();
  cluster_wait();
  // four experts per thread and step, the counts of all n <= kClusterCtas CTAs requested at
  // once (cnt is 16-byte aligned; a quad reaching past E is cut off below)
  for (int q = tid; 4 * q < E; q += blockDim.x) {
    int4 v[kClusterCtas];
#pragma unroll
    for (int c = 0; c < kClusterCtas; ++c)
      v[c] = (static_cast<uint32_t>(c) < n) ? ld_cluster_v4(cnt + 4 * q, c)
                                            : make_int4(0, 0, 0, 0);
    int4 before = make_int4(0, 0, 0, 0), total = make_int4(0, 0, 0, 0);
#pragma unroll
    for (int c = 0; c < kClusterCtas; ++c) {
      if (static_cast<uint32_t>(c) < rank) {
        before.x += v[c].x;
        before.y += v[c].y;
        before.z += v[c].z;
        before.w += v[c].w;
      }
      total.x += v[c].x;
      total.y += v[c].y;
      total.z += v[c].z;
      total.w += v[c].w;
    }
    const int bq[4] = {before.x, before.y, before.z, before.w};
    const int tq[4] = {total.x, total.y, total.z, total.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int e = 4 * q + k;
      if (e < E) {
        run[e] = bq[k];
        tot[e] = tq[k];
        pad[e] = (tq[k] + B - 1) & ~(B - 1);
        masks[e] = 0u;
        masks[E + e] = 0u;
      }
    }
  }
  int flags = 0;
  if (rank == 0 && warp == 0) {
    for (uint32_t c = lane; c < n; c += 32) flags |= ld_cluster_s32(flag, c);
    flags = __reduce_or_sync(kFull, flags);
  }
  if (tid == 0) {
    misc[40] = 0;
    misc[41] = 0;
  }
  // this CTA reads no other CTA's shared memory after this point; the matching wait before
  // the end keeps every CTA's shared memory alive until all have read it
  cluster_arrive();
  __syncthreads();
  block_exclusive_scan(pad, base, E, misc);  // base[E] = the padded total
  for (int e = tid; e < E; e += blockDim.x) run[e] += base[e];
  __syncthreads();
  const int n0 = t0 * K;
  place_unit_routes(rid, E, K, t0, t1, masks, run, &misc[40], [&](int pos, int r, int) {
    co.sorted_ids[pos] = n0 + r;
    co.sorted_w[pos] = rw[r];
  });
  // padding rows and block owners of this CTA's experts
  const int e0 = static_cast<int>(static_cast<long long>(rank) * E / n);
  const int e1 = static_cast<int>(static_cast<long long>(rank + 1) * E / n);
  for (int e = e0 + warp; e < e1; e += nwarps) {
    const int c = tot[e];
    if (c == 0) continue;
    const int off = base[e];
    const int end = off + pad[e];
    for (int p = off + c + lane; p < end; p += 32) {
      co.sorted_ids[p] = co.N;
      co.sorted_w[p] = 0.0f;
    }
    for (int b = off / B + lane; b < end / B; b += 32) co.expert_ids[b] = e;
  }
  if (rank == 0 && tid == 0) {
    *co.npp = base[E];
    *co.status = flags;
  }
  cluster_wait();
}

}  // namespace mrs
