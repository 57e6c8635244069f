// mrs_gate.cu -- the router gate projection ahead of the path, for a few tokens (a GEMV).
//
// logits[t, e] = bf16(sum over h of hidden[t, h] * w_gate[e, h]) for T <= 8 tokens.  At these
// sizes the projection is bound by one read of the E x H bf16 gate matrix.  One token takes
// mrs_gate1_kernel (below).  For 2..8 tokens the arithmetic goes to the tensor cores so that
// it never competes with the loads for issue slots:
//   tile     CTA c owns gate rows [c * rpc, c * rpc + nr), nr <= 16: the M side of an
//            m16n8k16 bf16 MMA (fp32 accumulate); the tokens are its N = 8 side
//   k split  the hidden dimension is cut into steps of 32 columns; warp w takes steps
//            w, w + warps, ... and accumulates its two MMAs per step in order
//   k order  the sum over k does not care how columns are assigned to the MMA's k slots, as
//            long as A and B agree: lane (g, q) (g = lane / 4, q = lane % 4) loads the 16
//            bytes of columns [32 s + 8 q, 32 s + 8 q + 8) of gate rows g and g + 8 and of
//            hidden row g, and hands words 0-1 to the first MMA's k slots {2q, 2q+1, 2q+8,
//            2q+9} and words 2-3 to the second's: every load is a contiguous 16 bytes
//   combine  each warp parks its 16 x 8 partial tile in shared memory; the CTA adds the
//            warps' partials in warp order and rounds once to bf16
// The fp32 result therefore does not depend on scheduling, and it is exact (so its rounding to
// bf16 is that of the exact dot product) whenever the partial sums are exactly representable.
// The route kernels that follow are programmatic dependents: they are launched while this grid
// runs and wait (griddepcontrol.wait) for its completion before reading the logits.
// Source: "perf(flydsl): Kimi-K3 B1 route-sort + prepared-MoE handoff (stack)", Summary -- the
// stack specialises the Kimi-K3 batch-one gate projection that feeds the route-sort.
#include <cuda_bf16.h>

#include "mrs_internal.h"

namespace mrs {

constexpr int kGateThreads = 256;
constexpr int kGateWarps = kGateThreads / 32;
constexpr int kGateRows = 16;  // M of the MMA tile: gate rows per CTA, at most
constexpr int kGateWin = 4;    // steps whose loads a warp keeps in flight

// D += A * B for one m16n8k16 bf16 MMA with fp32 accumulation (A row-major, B column-major).
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(kGateThreads, 2) mrs_gate_kernel(const GateArgs a) {
  __shared__ float part[kGateWarps][kGateRows][kGateMaxTokens];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int T = a.T, H = a.H;
  const int r0 = blockIdx.x * a.rpc;
  const int nr = min(a.rpc, a.E - r0);
  const int steps = (H + 31) >> 5;
  const int mine = (steps - warp + kGateWarps - 1) / kGateWarps;  // steps w, w + warps, ...
  pdl_trigger();
  // the CTA's gate rows (contiguous; weights, which the kernel ahead in the stream does not
  // normally write) start towards L2 while that kernel finishes
  prefetch_l2_range(a.w + static_cast<size_t>(r0) * H, 2 * static_cast<size_t>(nr) * H, tid,
                    kGateThreads);
  pdl_wait();

  const bool row_lo = g < nr, row_hi = g + 8 < nr, tok = g < T;
  const uint16_t* wlo = a.w + static_cast<size_t>(r0 + (row_lo ? g : 0)) * H;
  const uint16_t* whi = a.w + static_cast<size_t>(r0 + (row_hi ? g + 8 : 0)) * H;
  const uint16_t* hrow = a.hidden + static_cast<size_t>(tok ? g : 0) * H;
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  uint4 wl[kGateWin], wh[kGateWin], hv[kGateWin];
  auto load = [&](int k, int slot) {
    const int col = 32 * (warp + k * kGateWarps) + 8 * q;
    const bool in = k < mine && col < H;  // H is a multiple of 8: 8 columns all in or all out
    wl[slot] = (in && row_lo) ? __ldg(reinterpret_cast<const uint4*>(wlo + col)) : zero;
    wh[slot] = (in && row_hi) ? __ldg(reinterpret_cast<const uint4*>(whi + col)) : zero;
    hv[slot] = (in && tok) ? __ldg(reinterpret_cast<const uint4*>(hrow + col)) : zero;
  };
#pragma unroll
  for (int k = 0; k < kGateWin; ++k) load(k, k);
  float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int k0 = 0; k0 < mine; k0 += kGateWin) {
#pragma unroll
    for (int b = 0; b < kGateWin; ++b) {
      if (k0 + b >= mine) break;  // uniform over the warp
      const uint4 x = wl[b], y = wh[b], z = hv[b];
      mma_bf16_16816(d, x.x, y.x, x.y, y.y, z.x, z.y);
      mma_bf16_16816(d, x.z, y.z, x.w, y.w, z.z, z.w);
      load(k0 + b + kGateWin, b);  // refill the slot (nothing past the warp's steps)
    }
  }
  // d[0], d[1]: row g, tokens 2q, 2q + 1; d[2], d[3]: row g + 8, the same tokens
  part[warp][g][2 * q] = d[0];
  part[warp][g][2 * q + 1] = d[1];
  part[warp][g + 8][2 * q] = d[2];
  part[warp][g + 8][2 * q + 1] = d[3];
  __syncthreads();
  for (int i = tid; i < nr * T; i += kGateThreads) {
    const int r = i / T, t = i - r * T;
    float sum = part[0][r][t];
#pragma unroll
    for (int w = 1; w < kGateWarps; ++w) sum = __fadd_rn(sum, part[w][r][t]);
    a.logits[static_cast<size_t>(t) * a.E + r0 + r] =
        __bfloat16_as_ushort(__float2bfloat16_rn(sum));
  }
}

// One token (T = 1): the same sum with every load of a row group in flight at once, and the
// arithmetic on the FMA pipes (an MMA would leave 7 of its 8 token columns empty).  Thread t
// of the CTA takes the 16-byte column chunks t, t + 256, ... (at most four: H <= 8192) of
// each gate row and of the hidden row; it accumulates a row's products in fp32 in chunk
// order, the warp adds its 32 partial sums in a fixed shuffle tree, and the CTA adds the
// warps' sums in warp order and rounds once to bf16.  The rows of a group of kGate1Rows are
// requested together (up to 4 x 4 loads of 16 bytes per thread).
constexpr int kGate1Chunks = 4;  // chunks of a row per thread: 4 * 256 * 8 >= 8192 columns
constexpr int kGate1Rows = 4;

__global__ void __launch_bounds__(kGateThreads, 2) mrs_gate1_kernel(const GateArgs a) {
  __shared__ float part[kGateWarps][kGateRows];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = a.H, nch = H >> 3;  // 16-byte chunks of a row
  const int r0 = blockIdx.x * a.rpc;
  const int nr = min(a.rpc, a.E - r0);
  pdl_trigger();
  // the CTA's gate rows (contiguous; weights, which the kernel ahead in the stream does not
  // normally write) start towards L2 while that kernel finishes
  prefetch_l2_range(a.w + static_cast<size_t>(r0) * H, 2 * static_cast<size_t>(nr) * H, tid,
                    kGateThreads);
  pdl_wait();

  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  uint4 hv[kGate1Chunks];
#pragma unroll
  for (int i = 0; i < kGate1Chunks; ++i) {
    const int c = tid + kGateThreads * i;
    hv[i] = (c < nch) ? __ldg(reinterpret_cast<const uint4*>(a.hidden) + c) : zero;
  }
  const uint4* wrow = reinterpret_cast<const uint4*>(a.w + static_cast<size_t>(r0) * H);
  for (int j0 = 0; j0 < nr; j0 += kGate1Rows) {
    uint4 wv[kGate1Rows][kGate1Chunks];
#pragma unroll
    for (int jj = 0; jj < kGate1Rows; ++jj) {
#pragma unroll
      for (int i = 0; i < kGate1Chunks; ++i) {
        const int c = tid + kGateThreads * i;
        wv[jj][i] = (j0 + jj < nr && c < nch)
                        ? __ldg(wrow + static_cast<size_t>(j0 + jj) * nch + c)
                        : zero;
      }
    }
#pragma unroll
    for (int jj = 0; jj < kGate1Rows; ++jj) {
      float acc = 0.0f;
#pragma unroll
      for (int i = 0; i < kGate1Chunks; ++i) {
        const uint32_t wq[4] = {wv[jj][i].x, wv[jj][i].y, wv[jj][i].z, wv[jj][i].w};
        const uint32_t hq[4] = {hv[i].x, hv[i].y, hv[i].z, hv[i].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc = fmaf(__uint_as_float(wq[q] << 16), __uint_as_float(hq[q] << 16), acc);
          acc = fmaf(__uint_as_float(wq[q] & 0xffff0000u), __uint_as_float(hq[q] & 0xffff0000u),
                     acc);
        }
      }
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(kFull, acc, d));
      if (lane == 0 && j0 + jj < nr) part[warp][j0 + jj] = acc;
    }
  }
  __syncthreads();
  if (tid < nr) {
    float sum = part[0][tid];
#pragma unroll
    for (int w = 1; w < kGateWarps; ++w) sum = __fadd_rn(sum, part[w][tid]);
    a.logits[r0 + tid] = __bfloat16_as_ushort(__float2bfloat16_rn(sum));
  }
}

GatePlan gate_plan(int E, int sms) {
  GatePlan p{};
  const int slots = 2 * (sms > 0 ? sms : 1);  // two CTAs per SM
  int rpc = (E + slots - 1) / slots;
  if (rpc > kGateRows) rpc = kGateRows;
  p.rpc = rpc;
  p.grid = (E + rpc - 1) / rpc;
  return p;
}

cudaError_t launch_gate(const GateArgs& a, const GatePlan& p, cudaStream_t st) {
  if (a.T == 1) return launch_pdl(mrs_gate1_kernel, dim3(p.grid), dim3(kGateThreads), 0, st, a);
  return launch_pdl(mrs_gate_kernel, dim3(p.grid), dim3(kGateThreads), 0, st, a);
}

}  // namespace mrs
