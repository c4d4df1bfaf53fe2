// Router logits, shared-expert gate logit and top-k.
//
// Strata expert paths, "显存里缓存的是什么？": the router decides which experts
// a token uses and the merge weights of their outputs.  Top-k with
// renormalised weights: the k largest logits (ties to the lower expert id),
// w_r = exp(l_r - l_0) / sum_j exp(l_j - l_0) over the chosen k -- equal to a
// softmax over all E renormalised over the k.
#include "topk.cuh"

namespace moe {

// ------------------------------------------------------------------ router
// One warp per (row, token tile): row e < E is a router row, row E the
// shared-expert gate vector.  Each lane issues every 16-byte load of its part
// of the weight row first -- before waiting for the previous kernel, since no
// kernel writes the weights -- then stages the tile's bf16 activations in
// shared memory and accumulates in fp32 (bf16 x bf16 products are exact).
constexpr int kRouterTokTile = 8;
constexpr int kRouterMaxChunksPerLane = 16;  // H <= 4096

__global__ void __launch_bounds__(128) k_router(const uint16_t* __restrict__ x, const uint16_t* __restrict__ w_router,
                                                const float* __restrict__ bias, const uint16_t* __restrict__ w_gate,
                                                float* __restrict__ logits, float* __restrict__ gate_logit, int T,
                                                int H, int E, int rows, __half* __restrict__ x16,
                                                float* __restrict__ xscale) {
  extern __shared__ uint4 smem_x4[];  // [kRouterTokTile][H/8]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.y * kRouterTokTile;
  const int nt = min(kRouterTokTile, T - t0);
  const int chunks = H / 8;
  const int row = blockIdx.x * (blockDim.x >> 5) + warp;
  const bool live = row < rows;
  const uint16_t* wrow = live ? (row < E ? w_router + size_t(row) * H : w_gate) : nullptr;
  uint4 wv[kRouterMaxChunksPerLane];
#pragma unroll
  for (int i = 0; i < kRouterMaxChunksPerLane; ++i) {
    const int c = lane + 32 * i;
    wv[i] = (live && c < chunks) ? __ldg(reinterpret_cast<const uint4*>(wrow) + c) : make_uint4(0, 0, 0, 0);
  }
  pdl_wait();
  {
    // the tile's rows are contiguous: up to 8 independent loads in flight per thread, then the stores
    const uint4* xt = reinterpret_cast<const uint4*>(x + size_t(t0) * H);
    const int n = nt * chunks;
    for (int base = 0; base < n; base += 8 * blockDim.x) {
      uint4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = base + j * blockDim.x + threadIdx.x;
        if (i < n) v[j] = xt[i];
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = base + j * blockDim.x + threadIdx.x;
        if (i < n) smem_x4[i] = v[j];
      }
    }
  }
  if (x16) {
    // the blocks of a token tile also write its activations as f16 times a
    // per-token power of two (max|x_t| lands in [2^12, 2^13)); every block finds
    // the scales from its own copy and converts one slice of the columns
    __shared__ float s_scale[kRouterTokTile];
    __syncthreads();
    const uint16_t* xs = reinterpret_cast<const uint16_t*>(smem_x4);
    for (int t = warp; t < nt; t += blockDim.x >> 5) {
      float mx[4] = {0.f, 0.f, 0.f, 0.f};  // four independent chains
      for (int i = lane; i < H; i += 128)
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (i + 32 * u < H) mx[u] = fmaxf(mx[u], fabsf(bf16_bits_to_f32(xs[t * H + i + 32 * u])));
      float m = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) s_scale[t] = pow2_scale_for(m);
    }
    __syncthreads();
    if (blockIdx.x == 0 && threadIdx.x < nt) xscale[t0 + threadIdx.x] = s_scale[threadIdx.x];
    const int per = ((H + gridDim.x - 1) / gridDim.x + 7) & ~7;
    const int c0 = blockIdx.x * per, c1 = min(H, c0 + per);
    const int wcols = c1 - c0;
    for (int i = threadIdx.x; wcols > 0 && i < nt * wcols; i += blockDim.x) {
      const int t = i / wcols, c = c0 + (i - t * wcols);
      x16[size_t(t0 + t) * H + c] = __float2half_rn(bf16_bits_to_f32(xs[t * H + c]) * s_scale[t]);
    }
  }
  __syncthreads();
  float acc[kRouterTokTile];
#pragma unroll
  for (int t = 0; t < kRouterTokTile; ++t) acc[t] = 0.f;
#pragma unroll
  for (int i = 0; i < kRouterMaxChunksPerLane; ++i) {
    const int c = lane + 32 * i;
    if (c < chunks) {
      const uint32_t wu[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
#pragma unroll
      for (int t = 0; t < kRouterTokTile; ++t) {
        if (t < nt) {
          const uint4 xv = smem_x4[t * chunks + c];
          const uint32_t xu[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            acc[t] = fmaf(__uint_as_float(wu[j] << 16), __uint_as_float(xu[j] << 16), acc[t]);
            acc[t] = fmaf(__uint_as_float(wu[j] & 0xffff0000u), __uint_as_float(xu[j] & 0xffff0000u), acc[t]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kRouterTokTile; ++t) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
  }
  // the next kernel's blocks are launched only now: launched at the start, they
  // slowed this kernel down by a third while they waited
  pdl_trigger();
  if (live && lane < nt) {
    float v = acc[0];
#pragma unroll
    for (int t = 1; t < kRouterTokTile; ++t)
      if (lane == t) v = acc[t];
    if (row < E)
      logits[size_t(t0 + lane) * E + row] = bias ? __fadd_rn(v, bias[row]) : v;
    else
      gate_logit[t0 + lane] = v;
  }
}

int launch_router(const uint16_t* x, const uint16_t* w_router, const float* bias, const uint16_t* w_gate,
                  float* logits, float* gate_logit, int T, int H, int E, cudaStream_t s, __half* x16,
                  float* xscale) {
  if (T <= 0) return MOE_OK;
  if (H / 8 > 32 * kRouterMaxChunksPerLane) return MOE_EINVAL;
  // rows 0..E-1 are router rows, row E the gate vector; without a router only the gate row runs
  const int E_eff = w_router ? E : 0;
  const int rows = E_eff + (w_gate ? 1 : 0);
  if (rows == 0) return MOE_OK;
  const int tok_tiles = (T + kRouterTokTile - 1) / kRouterTokTile;
  const size_t smem = size_t(kRouterTokTile) * H * 2;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(k_router, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
    return MOE_ECUDA;
  dim3 grid((rows + 3) / 4, tok_tiles);
  if (launch_pdl(k_router, grid, dim3(128), smem, s, x, w_router ? w_router : w_gate, bias, w_gate, logits,
                 gate_logit, T, H, E_eff, rows, x16, xscale) != cudaSuccess)
    return MOE_ECUDA;
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

template <int KPER>
__global__ void __launch_bounds__(256) k_topk(const float* __restrict__ logits, int T, int E, int k,
                                              int32_t* __restrict__ ids, float* __restrict__ w, int32_t* err) {
  pdl_trigger();
  pdl_wait();
  const int tok = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (tok >= T) return;
  topk_token<KPER>(logits + size_t(tok) * E, E, k, lane, ids + size_t(tok) * k, w + size_t(tok) * k, err);
}

int launch_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w, int32_t* err, cudaStream_t s) {
  if (T <= 0) return MOE_OK;
  const int blocks = (T * 32 + 255) / 256;
  const int per = (E + 31) / 32;
  cudaError_t rc = cudaSuccess;
  if (per <= 1) rc = launch_pdl(k_topk<1>, dim3(blocks), dim3(256), 0, s, logits, T, E, k, ids, w, err);
  else if (per <= 2) rc = launch_pdl(k_topk<2>, dim3(blocks), dim3(256), 0, s, logits, T, E, k, ids, w, err);
  else if (per <= 4) rc = launch_pdl(k_topk<4>, dim3(blocks), dim3(256), 0, s, logits, T, E, k, ids, w, err);
  else if (per <= 8) rc = launch_pdl(k_topk<8>, dim3(blocks), dim3(256), 0, s, logits, T, E, k, ids, w, err);
  else if (per <= 16) rc = launch_pdl(k_topk<16>, dim3(blocks), dim3(256), 0, s, logits, T, E, k, ids, w, err);
  else if (per <= 32) rc = launch_pdl(k_topk<32>, dim3(blocks), dim3(256), 0, s, logits, T, E, k, ids, w, err);
  else return MOE_EINVAL;
  if (rc != cudaSuccess) return MOE_ECUDA;
  return MOE_OK;
}

}  // namespace moe
