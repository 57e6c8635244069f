// mrs_gate.cu -- the router gate projection ahead of the path, for a few tokens (a GEMV).
//
// logits[t, e] = bf16(sum over h of hidden[t, h] * w_gate[e, h]) for T <= 8 tokens.  At these
// sizes the projection is bound by one read of the E x H bf16 gate matrix (12.8 MB for the
// Kimi-K3 shape, E = 896, H = 7168), so the kernel is built around keeping enough of it in
// flight:
//   rows     CTA c owns the gate rows [c * rpc, (c + 1) * rpc), rpc = ceil(E / SMs): one CTA per
//            SM, each streaming a contiguous part of the matrix.  It takes them 8 at a time (a
//            row group: the N = 8 side of an m16n8k16 bf16 MMA with fp32 accumulation; the
//            tokens are its M side, rows T..15 zero)
//   stream   a row group's columns are cut into chunks of kChunk columns.  One thread issues,
//            per chunk, one bulk copy (TMA) per row into a ring of shared-memory stages that
//            complete on their own mbarriers.  The ring has as many stages as the CTA has chunks
//            (all of them in flight at once: at E = 896 a CTA streams 6 rows, 84 KB) or as fit
//            in shared memory; rows are padded by 64 bytes so that the fragment loads below are
//            conflict-free.  The hidden rows are copied once per CTA the same way
//   compute  warp w takes the 32-column steps w, w + 8, ... of each chunk, two MMAs per step.
//            Lane (g, q) (g = lane / 4, q = lane % 4) loads 16 contiguous bytes, columns
//            8q..8q+7 of the step, of hidden row g and of gate row g of the group, and hands
//            words 0-1 to the first MMA's k slots {2q, 2q+1, 2q+8, 2q+9} and words 2-3 to the
//            second's: the sum over k does not care which column feeds which slot as long as A
//            and B agree, and every load is one conflict-free 16-byte vector
//   combine  after a group's last chunk each warp parks its 8 x 8 partial tile in shared
//            memory; the CTA adds the warps' partials in warp order and rounds once to bf16
// The fp32 result therefore does not depend on scheduling, and it is exact (so its rounding to
// bf16 is that of the exact dot product) whenever the partial sums are exactly representable.
// Every wait is bounded; a CTA that gives up records MOE_RS_DEVICE_WAIT_TIMEOUT in its own
// word of `flags`, which the route kernel that follows folds into the call's status word.  The
// route kernels are programmatic dependents: they are launched while this grid runs and wait
// (griddepcontrol.wait) for its completion before reading the logits.
// Source: "perf(flydsl): Kimi-K3 B1 route-sort + prepared-MoE handoff (stack)", Summary -- the
// stack specialises the Kimi-K3 batch-one gate projection that feeds the route-sort.
#include <cuda_bf16.h>

#include "mrs_internal.h"
#include "moe_route_sort.h"

namespace mrs {

constexpr int kGateThreads = 256;
constexpr int kGateWarps = kGateThreads / 32;
constexpr int kGateGroup = 8;    // gate rows per MMA (the N side)
constexpr int kChunk = 1024;     // columns per stage and row
constexpr int kMaxStages = 16;   // stages of the ring, at most (one mbarrier each)
// Row pitches in shared memory, in bf16: padded by 64 bytes, so that the two rows one quarter
// of a warp reads with its 16-byte loads land in opposite halves of the banks.
constexpr int kChunkPitch = kChunk + 32;
__host__ __device__ inline int hid_pitch(int H) { return H + 32; }

struct GateSmem {
  size_t hid, ring, part, mbar, total;
};

__host__ __device__ inline GateSmem gate_smem(int T, int H, int stages) {
  GateSmem l{};
  size_t o = 0;
  l.hid = o;
  o = align16(o + static_cast<size_t>(T) * hid_pitch(H) * 2);
  l.part = o;
  o = align16(o + sizeof(float) * kGateWarps * kGateMaxTokens * kGateGroup);
  l.mbar = o;
  o = align16(o + sizeof(unsigned long long) * (kMaxStages + 1));
  l.ring = o;
  o = align16(o + static_cast<size_t>(stages) * kGateGroup * kChunkPitch * 2);
  l.total = o;
  return l;
}

// D += A * B for one m16n8k16 bf16 MMA with fp32 accumulation (A row-major, B column-major).
// A rows 8..15 are zero here (at most 8 tokens), so their two registers are 0 and the
// accumulators d[2], d[3] stay 0.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a2,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) completing on `mbar`,
// whose expected transaction count the issuing thread has raised beforehand.
__device__ __forceinline__ void tma_copy_1d(void* dst, const void* src, uint32_t bytes,
                                            unsigned long long* mbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(mbar))
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect(unsigned long long* mbar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(mbar)),
               "r"(bytes)
               : "memory");
}

__global__ void __launch_bounds__(kGateThreads, 1) mrs_gate_kernel(const GateArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int T = a.T, H = a.H;
  const int stages = a.stages;
  const GateSmem lay = gate_smem(T, H, stages);
  uint16_t* hid = reinterpret_cast<uint16_t*>(smem + lay.hid);    // [T][hid_pitch(H)]
  uint16_t* ring = reinterpret_cast<uint16_t*>(smem + lay.ring);  // [stages][8][kChunkPitch]
  float* part = reinterpret_cast<float*>(smem + lay.part);        // [warps][8 tokens][8 rows]
  unsigned long long* mbar = reinterpret_cast<unsigned long long*>(smem + lay.mbar);
  unsigned long long* mbar_hid = mbar + stages;
  __shared__ int timed_out;

  const int r0 = blockIdx.x * a.rpc;
  const int nrows = min(a.rpc, a.E - r0);
  const int ngroups = (nrows + kGateGroup - 1) / kGateGroup;
  const int nchunks = (H + kChunk - 1) / kChunk;
  const int total = ngroups * nchunks;  // chunks of this CTA, group-major
  pdl_trigger();
  pdl_wait();

  // chunk k: group k / nchunks, columns [c0, c0 + cols) of its (up to 8) rows, into stage s
  auto issue = [&](int k) {
    const int grp = k / nchunks, c0 = (k - grp * nchunks) * kChunk;
    const int cols = min(kChunk, H - c0);
    const int rows = min(kGateGroup, nrows - grp * kGateGroup);
    const int s = k % stages;
    mbar_arrive_expect(&mbar[s], static_cast<uint32_t>(rows * cols * 2));
    for (int r = 0; r < rows; ++r)
      tma_copy_1d(ring + (static_cast<size_t>(s) * kGateGroup + r) * kChunkPitch,
                  a.w + static_cast<size_t>(r0 + grp * kGateGroup + r) * H + c0,
                  static_cast<uint32_t>(cols * 2), &mbar[s]);
  };
  if (tid == 0) {
    timed_out = 0;
    for (int s = 0; s <= stages; ++s) mbar_init(&mbar[s], 1);
    fence_mbar_init();
    mbar_arrive_expect(mbar_hid, static_cast<uint32_t>(T * H * 2));
    for (int t = 0; t < T; ++t)
      tma_copy_1d(hid + static_cast<size_t>(t) * hid_pitch(H), a.hidden + static_cast<size_t>(t) * H,
                  static_cast<uint32_t>(H * 2), mbar_hid);
    for (int k = 0; k < stages && k < total; ++k) issue(k);
  }
  __syncthreads();
  const int issued0 = min(stages, total);
  // every decision to give up is made for the whole CTA at once (the stages are shared)
  bool ok = __syncthreads_and(mbar_wait_bounded(mbar_hid, 0u, a.wait_limit_ns)) != 0;

  float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  int consumed = 0;
  const bool tok = g < T;
  const uint16_t* hrow = hid + static_cast<size_t>(tok ? g : 0) * hid_pitch(H);
  for (int k = 0; ok && k < total; ++k) {
    const int s = k % stages;
    const bool got =
        mbar_wait_bounded(&mbar[s], static_cast<uint32_t>((k / stages) & 1), a.wait_limit_ns);
    const int grp = k / nchunks, c0 = (k - grp * nchunks) * kChunk;
    const int cols = min(kChunk, H - c0);
    const int rows = min(kGateGroup, nrows - grp * kGateGroup);
    if (got) {
      const uint16_t* wrow = ring + (static_cast<size_t>(s) * kGateGroup + g) * kChunkPitch;
      for (int st = warp; st * 32 < cols; st += kGateWarps) {
        const int col = st * 32 + 8 * q;  // H % 8 == 0: a lane's 8 columns are all in or out
        const bool in = col < cols;
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        const uint4 hv = (in && tok) ? *reinterpret_cast<const uint4*>(hrow + c0 + col) : z;
        const uint4 wv = (in && g < rows) ? *reinterpret_cast<const uint4*>(wrow + col) : z;
        mma_bf16_16816(d, hv.x, hv.y, wv.x, wv.y);
        mma_bf16_16816(d, hv.z, hv.w, wv.z, wv.w);
      }
    }
    // every warp is done with stage s (and, at a group's end, with part); all or none go on
    if (!__syncthreads_and(got)) {
      ok = false;
      break;
    }
    consumed = k + 1;
    if (tid == 0 && k + stages < total) {
      fence_proxy_async_smem();
      issue(k + stages);
    }
    if (k - grp * nchunks == nchunks - 1) {
      // group done: d[0], d[1] = token g, group rows 2q, 2q + 1
      float* pw = part + (warp * kGateMaxTokens + g) * kGateGroup;
      pw[2 * q] = d[0];
      pw[2 * q + 1] = d[1];
      d[0] = d[1] = 0.0f;
      __syncthreads();
      if (tid < T * kGateGroup) {
        const int t = tid / kGateGroup, r = tid - t * kGateGroup;
        if (r < rows) {
          float sum = part[t * kGateGroup + r];
#pragma unroll
          for (int w = 1; w < kGateWarps; ++w)
            sum = __fadd_rn(sum, part[(w * kGateMaxTokens + t) * kGateGroup + r]);
          a.logits[static_cast<size_t>(t) * a.E + r0 + grp * kGateGroup + r] =
              __bfloat16_as_ushort(__float2bfloat16_rn(sum));
        }
      }
      // part is written again only after the next group's first barrier
    }
  }
  if (!ok) {
    // a copy did not complete in time: report it, then give every copy still in flight a
    // bounded chance to land before the CTA exits
    if (lane == 0) atomicOr(&timed_out, MOE_RS_DEVICE_WAIT_TIMEOUT);
    mbar_wait_bounded(mbar_hid, 0u, kWaitLimitNs);
    const int issued = min(total, max(issued0, consumed + stages));
    for (int k = consumed; k < issued; ++k)
      mbar_wait_bounded(&mbar[k % stages], static_cast<uint32_t>((k / stages) & 1),
                        kWaitLimitNs);
  }
  __syncthreads();
  if (tid == 0) a.flags[blockIdx.x] = timed_out;
}

GatePlan gate_plan(int T, int E, int H, int sms, int smem_optin) {
  GatePlan p{};
  const int n = sms > 0 ? sms : 1;
  p.rpc = (E + n - 1) / n;
  p.grid = (E + p.rpc - 1) / p.rpc;
  // as many stages as the busiest CTA has chunks, or as fit (at least 2)
  const int chunks = ((p.rpc + kGateGroup - 1) / kGateGroup) * ((H + kChunk - 1) / kChunk);
  int st = chunks < kMaxStages ? chunks : kMaxStages;
  while (st > 2 && gate_smem(T, H, st).total > static_cast<size_t>(smem_optin)) --st;
  if (st < 2) st = 2;
  p.stages = st;
  p.smem = gate_smem(T, H, st).total;
  return p;
}

cudaError_t launch_gate(const GateArgs& a, const GatePlan& p, cudaStream_t st) {
  cudaError_t err = cudaFuncSetAttribute(mrs_gate_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(p.smem));
  if (err != cudaSuccess) return err;
  return launch_pdl(mrs_gate_kernel, dim3(p.grid), dim3(kGateThreads), p.smem, st, a);
}

}  // namespace mrs
