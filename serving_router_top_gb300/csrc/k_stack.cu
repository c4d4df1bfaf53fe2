// Residual stream and RMS normalisation between the layers of a decode stack.
//
// The pages give the model as 48 MoE layers in sequence; the decode-stack
// workload wraps each layer as x_{l+1} = x_l + MoE_l(RMSNorm(x_l)) with an fp32
// residual stream, bf16 layer input/output and unit RMSNorm weight.  One
// kernel per layer boundary: add the previous layer's output into the stream
// and write the next layer's normalised bf16 input.
#include "internal.h"

namespace moe {

constexpr int kNormThreads = 256;
constexpr int kNormMaxPer = 4;  // float4 per thread: H <= 4096

// One CTA per token row.
__global__ void __launch_bounds__(kNormThreads) k_residual_rmsnorm(float* __restrict__ x, const uint16_t* __restrict__ y,
                                                                  uint16_t* __restrict__ xn, int H, float eps) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x, n4 = H / 4;
  float4* xr = reinterpret_cast<float4*>(x + size_t(t) * H);
  float4 v[kNormMaxPer];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < kNormMaxPer; ++j) {
    const int c4 = threadIdx.x + j * kNormThreads;
    v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c4 < n4) {
      v[j] = xr[c4];
      if (y) {
        const uint2 yb = reinterpret_cast<const uint2*>(y + size_t(t) * H)[c4];
        v[j].x += bf16_bits_to_f32(uint16_t(yb.x & 0xffffu));
        v[j].y += bf16_bits_to_f32(uint16_t(yb.x >> 16));
        v[j].z += bf16_bits_to_f32(uint16_t(yb.y & 0xffffu));
        v[j].w += bf16_bits_to_f32(uint16_t(yb.y >> 16));
        xr[c4] = v[j];
      }
      ss += v[j].x * v[j].x + v[j].y * v[j].y + v[j].z * v[j].z + v[j].w * v[j].w;
    }
  }
  __shared__ float red[kNormThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kNormThreads / 32; ++w) tot += red[w];
  const float inv = 1.0f / sqrtf(tot / float(H) + eps);
#pragma unroll
  for (int j = 0; j < kNormMaxPer; ++j) {
    const int c4 = threadIdx.x + j * kNormThreads;
    if (c4 < n4) {
      const __nv_bfloat162 p0 = __floats2bfloat162_rn(v[j].x * inv, v[j].y * inv);
      const __nv_bfloat162 p1 = __floats2bfloat162_rn(v[j].z * inv, v[j].w * inv);
      uint2 u;
      u.x = *reinterpret_cast<const uint32_t*>(&p0);
      u.y = *reinterpret_cast<const uint32_t*>(&p1);
      reinterpret_cast<uint2*>(xn + size_t(t) * H)[c4] = u;
    }
  }
}

}  // namespace moe

extern "C" int moe_residual_rmsnorm(float* x_res, const uint16_t* y_prev, uint16_t* xn_out, int T, int H, float eps,
                                    moe_stream_t stream) {
  using namespace moe;
  if (!x_res || !xn_out || T < 0 || H <= 0 || H % 4 || H > 4 * kNormThreads * kNormMaxPer || !(eps > 0.f))
    return MOE_EINVAL;
  if ((reinterpret_cast<uintptr_t>(x_res) & 15) || (reinterpret_cast<uintptr_t>(xn_out) & 7) ||
      (reinterpret_cast<uintptr_t>(y_prev) & 7))
    return MOE_EINVAL;
  if (T == 0) return MOE_OK;
  if (launch_pdl(k_residual_rmsnorm, dim3(T), dim3(kNormThreads), 0, reinterpret_cast<cudaStream_t>(stream), x_res,
                 y_prev, xn_out, H, eps) != cudaSuccess)
    return MOE_ECUDA;
  return MOE_OK;
}
