// mrs_selftest.cu -- exhaustive device check of the proxy score's error bound.
//
// For every finite bf16 logit x, compares 0.5 * tanh.approx(0.5 x) + 0.5 (the proxy's
// score part, as the route kernels compute it) with the exact score 1 / (1 + expf(-x)) in
// double precision, and reports the largest difference next to the bound the selection
// assumes (kProxyTanhBound).
#include "mrs_internal.h"
#include "moe_route_sort.h"

namespace mrs {

__global__ void __launch_bounds__(256) mrs_proxy_selftest_kernel(unsigned int* max_err_bits,
                                                                  float* bound_out) {
  const uint32_t h = blockIdx.x * 256u + threadIdx.x;  // 65536 patterns
  if (h == 0) *bound_out = kProxyTanhBound;
  const float x = bf16_bits_to_float(h);
  float err = 0.0f;
  if (isfinite(x)) {
    const float t = tanh_approx(0.5f * x);
    const double approx = 0.5 * static_cast<double>(t) + 0.5;
    const double exact = static_cast<double>(exact_score(x));
    err = static_cast<float>(fabs(approx - exact)) * 1.0000001f;  // round the error upward
  }
  for (int d = 16; d > 0; d >>= 1) err = fmaxf(err, __shfl_xor_sync(kFull, err, d));
  if ((threadIdx.x & 31) == 0) atomicMax(max_err_bits, __float_as_uint(err));
}

}  // namespace mrs

extern "C" int moe_route_sort_proxy_selftest(float* out2, cudaStream_t stream) {
  if (!out2) return MOE_RS_ERR_NULL_POINTER;
  if (reinterpret_cast<uintptr_t>(out2) % 4) return MOE_RS_ERR_MISALIGNED;
  if (cudaMemsetAsync(out2, 0, sizeof(float), stream) != cudaSuccess) return MOE_RS_ERR_LAUNCH;
  mrs::mrs_proxy_selftest_kernel<<<256, 256, 0, stream>>>(reinterpret_cast<unsigned int*>(out2),
                                                          out2 + 1);
  if (cudaGetLastError() != cudaSuccess) return MOE_RS_ERR_LAUNCH;
  return MOE_RS_OK;
}
