// Router-weighted combine (step 5 of the block), sm_103a.
// zwxr.cn news/242664, section "一次路由的完整旅程": moe_combine adds the routed experts' outputs
// weighted by this layer's router weights: out[t] = sum_k w[t][k] * parts[t][k], here in fixed k
// order, then (residual layers) the layer input is added back.
#include "common.cuh"

namespace strata {
namespace {

__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ parts,
                                                      const float* __restrict__ weights, int T,
                                                      const float* residual, float* out) {
  const int64_t i4 = (int64_t)blockIdx.x * 256 + threadIdx.x;  // float4 index
  if (i4 >= (int64_t)T * (H / 4)) return;
  const int t = (int)(i4 / (H / 4));
  const int h4 = (int)(i4 % (H / 4));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const float w = __ldg(weights + t * K + k);
    const float4 p = __ldg(reinterpret_cast<const float4*>(parts + ((size_t)t * K + k) * H) + h4);
    acc.x = fmaf(w, p.x, acc.x);
    acc.y = fmaf(w, p.y, acc.y);
    acc.z = fmaf(w, p.z, acc.z);
    acc.w = fmaf(w, p.w, acc.w);
  }
  if (residual) {
    const float4 r = reinterpret_cast<const float4*>(residual + (size_t)t * H)[h4];
    acc.x = r.x + acc.x;
    acc.y = r.y + acc.y;
    acc.z = r.z + acc.z;
    acc.w = r.w + acc.w;
  }
  reinterpret_cast<float4*>(out + (size_t)t * H)[h4] = acc;
}

}  // namespace

cudaError_t launch_combine(const float* parts, const float* weights, int T, const float* residual, float* out,
                           cudaStream_t s) {
  const int64_t n4 = (int64_t)T * (H / 4);
  STRATA_LAUNCH(KID_COMBINE, s,
                combine_kernel<<<(unsigned)((n4 + 255) / 256), 256, 0, s>>>(parts, weights, T, residual, out));
  return cudaGetLastError();
}

}  // namespace strata
