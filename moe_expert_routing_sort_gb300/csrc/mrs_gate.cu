// mrs_gate.cu -- the router gate projection ahead of the path, for a few tokens (a GEMV).
//
// logits[t, e] = bf16(sum over h of hidden[t, h] * w_gate[e, h]) for T <= 8 tokens.  At these
// sizes the projection is a matrix-vector product bound by one read of the E x H bf16 gate
// matrix, so it runs on CUDA-core FMAs: a tensor-core tile would be at most 8/128 full.
//   rows     CTA c owns gate rows [c * rpc, (c + 1) * rpc), rpc = ceil(E / SMs): one wave
//   hidden   the T hidden rows are staged in shared memory once per CTA
//   chunks   a row is cut into chunks of 32 lanes x kGateVec 16-byte vectors (coalesced
//            512-byte warp loads); warps take the CTA's (row, chunk) items in a fixed order,
//            reduce each over the lanes with a fixed butterfly and park the partial in
//            shared memory; a row's partials are then added in chunk order
// The fp32 result therefore does not depend on scheduling, and it is exact (so its single
// rounding to bf16 is that of the exact dot product) whenever the products and partial sums
// are exactly representable.  The route kernels that follow are programmatic dependents:
// they are launched while this grid runs and wait (griddepcontrol.wait) for its completion
// before reading the logits, which are still in L2.
// Source: "perf(flydsl): Kimi-K3 B1 route-sort + prepared-MoE handoff (stack)", Summary --
// the stack specialises the Kimi-K3 batch-one gate projection that feeds the route-sort.
#include <cuda_bf16.h>

#include "mrs_internal.h"

namespace mrs {

constexpr int kGateThreads = 512;
constexpr int kGateWarps = kGateThreads / 32;
constexpr int kGateVec = 4;  // 16-byte vectors per lane per chunk

__device__ __forceinline__ void bf16x8_to_float(const uint4& q, float (&f)[8]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__global__ void __launch_bounds__(kGateThreads, 1) mrs_gate_kernel(const GateArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = a.T, H8 = a.H >> 3, nch = a.nch, rpc = a.rpc;
  uint4* hs = reinterpret_cast<uint4*>(smem);  // [T][H8]
  float* part = reinterpret_cast<float*>(smem + align16(sizeof(uint4) * T * H8));  // [T][rpc][nch]
  const int r0 = blockIdx.x * rpc;
  const int nr = min(rpc, a.E - r0);
  pdl_trigger();
  pdl_wait();

  const uint4* h4 = reinterpret_cast<const uint4*>(a.hidden);
  for (int i = tid; i < T * H8; i += kGateThreads) hs[i] = h4[i];
  __syncthreads();

  const uint4* w4 = reinterpret_cast<const uint4*>(a.w);
  const int items = nr * nch;
  for (int it = warp; it < items; it += kGateWarps) {
    const int r = it / nch, c = it - r * nch;
    const uint4* wrow = w4 + static_cast<size_t>(r0 + r) * H8;
    uint4 wv[kGateVec];
#pragma unroll
    for (int v = 0; v < kGateVec; ++v) {  // all of the item's loads in flight at once
      const int j = (c * kGateVec + v) * 32 + lane;
      wv[v] = (j < H8) ? __ldg(wrow + j) : make_uint4(0u, 0u, 0u, 0u);
    }
    float acc[kGateMaxTokens];
#pragma unroll
    for (int t = 0; t < kGateMaxTokens; ++t) acc[t] = 0.0f;
#pragma unroll
    for (int v = 0; v < kGateVec; ++v) {
      const int j = (c * kGateVec + v) * 32 + lane;
      if (j < H8) {
        float wf[8];
        bf16x8_to_float(wv[v], wf);
#pragma unroll
        for (int t = 0; t < kGateMaxTokens; ++t) {
          if (t < T) {
            float hf[8];
            bf16x8_to_float(hs[t * H8 + j], hf);
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[t] = fmaf(wf[q], hf[q], acc[t]);
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kGateMaxTokens; ++t) {
      if (t < T) {  // uniform over the warp
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) acc[t] = __fadd_rn(acc[t], __shfl_xor_sync(kFull, acc[t], d));
        if (lane == 0) part[(t * rpc + r) * nch + c] = acc[t];
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < T * nr; i += kGateThreads) {
    const int t = i / nr, r = i - t * nr;
    const float* p = part + (t * rpc + r) * nch;
    float s = p[0];
    for (int c = 1; c < nch; ++c) s = __fadd_rn(s, p[c]);
    a.logits[static_cast<size_t>(t) * a.E + r0 + r] = __bfloat16_as_ushort(__float2bfloat16_rn(s));
  }
}

GatePlan gate_plan(int T, int E, int H, int sms) {
  GatePlan p{};
  const int s = sms > 0 ? sms : 1;
  p.rpc = (E + s - 1) / s;
  p.grid = (E + p.rpc - 1) / p.rpc;
  const int H8 = H / 8;
  p.nch = (H8 + 32 * kGateVec - 1) / (32 * kGateVec);
  p.smem = align16(sizeof(uint4) * static_cast<size_t>(T) * H8) +
           sizeof(float) * static_cast<size_t>(T) * p.rpc * p.nch;
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
