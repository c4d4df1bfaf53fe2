// Router logits, shared-expert gate logit, activation prep and top-k.
//
// Strata expert paths, "显存里缓存的是什么？": the router decides which experts
// a token uses and the merge weights of their outputs.  Top-k with
// renormalised weights: the k largest logits (ties to the lower expert id),
// w_r = exp(l_r - l_0) / sum_j exp(l_j - l_0) over the chosen k -- equal to a
// softmax over all E renormalised over the k.
#include "internal.h"

namespace moe {

// ------------------------------------------------------------------ router
// One warp per (row, token tile): row e < E is a router row, row E the
// shared-expert gate vector.  The token tile's bf16 activations sit in shared
// memory; each lane streams 16-byte chunks of the weight row.  fp32
// accumulate (bf16 x bf16 products are exact in fp32).
constexpr int kRouterTokTile = 8;

__global__ void __launch_bounds__(256) k_router(const uint16_t* __restrict__ x, const uint16_t* __restrict__ w_router,
                                                const float* __restrict__ bias, const uint16_t* __restrict__ w_gate,
                                                float* __restrict__ logits, float* __restrict__ gate_logit, int T,
                                                int H, int E, int rows, int tok_tiles) {
  extern __shared__ uint4 smem_x4[];  // [kRouterTokTile][H] bf16
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.y;
  const int t0 = tile * kRouterTokTile;
  const int nt = min(kRouterTokTile, T - t0);
  const int chunks = H / 8;  // 16-byte chunks of 8 bf16
  // stage the token tile
  for (int i = threadIdx.x; i < nt * chunks; i += blockDim.x) {
    int t = i / chunks, c = i % chunks;
    smem_x4[t * chunks + c] = reinterpret_cast<const uint4*>(x + size_t(t0 + t) * H)[c];
  }
  __syncthreads();
  const int row = blockIdx.x * (blockDim.x >> 5) + warp;
  if (row >= rows) return;
  const uint16_t* wrow = row < E ? w_router + size_t(row) * H : w_gate;
  float acc[kRouterTokTile];
#pragma unroll
  for (int t = 0; t < kRouterTokTile; ++t) acc[t] = 0.f;
  for (int c = lane; c < chunks; c += 32) {
    uint4 wv = reinterpret_cast<const uint4*>(wrow)[c];
    const uint32_t wu[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
    for (int t = 0; t < kRouterTokTile; ++t) {
      if (t < nt) {
        uint4 xv = smem_x4[t * chunks + c];
        const uint32_t xu[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[t] = fmaf(__uint_as_float(wu[j] << 16), __uint_as_float(xu[j] << 16), acc[t]);
          acc[t] = fmaf(__uint_as_float(wu[j] & 0xffff0000u), __uint_as_float(xu[j] & 0xffff0000u), acc[t]);
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kRouterTokTile; ++t) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
  }
  if (lane == 0) {
    for (int t = 0; t < nt; ++t) {
      if (row < E)
        logits[size_t(t0 + t) * E + row] = bias ? __fadd_rn(acc[t], bias[row]) : acc[t];
      else
        gate_logit[t0 + t] = acc[t];
    }
  }
}

int launch_router(const uint16_t* x, const uint16_t* w_router, const float* bias, const uint16_t* w_gate,
                  float* logits, float* gate_logit, int T, int H, int E, cudaStream_t s) {
  if (T <= 0) return MOE_OK;
  int rows = (w_router ? E : 0) + (w_gate ? 1 : 0);
  if (rows == 0) return MOE_OK;
  if (!w_router) {
    // gate row only: place it at index E with a zero-row router skipped
    rows = 1;
  }
  int tok_tiles = (T + kRouterTokTile - 1) / kRouterTokTile;
  size_t smem = size_t(kRouterTokTile) * H * 2;
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(k_router, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
      return MOE_ECUDA;
  }
  dim3 grid((rows + 7) / 8, tok_tiles);
  if (w_router) {
    k_router<<<grid, 256, smem, s>>>(x, w_router, bias, w_gate, logits, gate_logit, T, H, E, rows, tok_tiles);
  } else {
    // only the gate row: row index E selects w_gate
    k_router<<<grid, 256, smem, s>>>(x, w_gate, nullptr, w_gate, logits, gate_logit, T, H, /*E=*/0, 1, tok_tiles);
  }
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

// ------------------------------------------------------------ activations
// x (bf16) -> x16 = f16(x * 2^s_t) with a per-token power-of-two scale that
// puts max|x_t| in [2^12, 2^13); exact for every bf16 value above 2^-14 * 2^-s.
__global__ void __launch_bounds__(256) k_prep_act(const uint16_t* __restrict__ x, __half* __restrict__ x16,
                                                  float* __restrict__ scale, int H) {
  const int t = blockIdx.x;
  const uint16_t* xr = x + size_t(t) * H;
  float m = 0.f;
  for (int i = threadIdx.x; i < H; i += blockDim.x) m = fmaxf(m, fabsf(bf16_bits_to_f32(xr[i])));
  __shared__ float red[8];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (threadIdx.x == 0) red[0] = m;
  }
  __syncthreads();
  const float sc = pow2_scale_for(red[0]);
  if (threadIdx.x == 0) scale[t] = sc;
  for (int i = threadIdx.x; i < H; i += blockDim.x) x16[size_t(t) * H + i] = __float2half_rn(bf16_bits_to_f32(xr[i]) * sc);
}

int launch_prep_act(const uint16_t* x, __half* x16, float* scale, int T, int H, cudaStream_t s) {
  if (T <= 0) return MOE_OK;
  k_prep_act<<<T, 256, 0, s>>>(x, x16, scale, H);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

// ------------------------------------------------------------------- top-k
// One warp per token; lane j holds logits j, j+32, ... (up to kMaxE/32).
// Each of the k rounds takes the warp-wide best not-yet-taken entry by
// (value desc, id asc).  NaN logits record MOE_ENAN and rank as -inf.
__device__ __forceinline__ bool better(float a, int ia, float b, int ib) { return a > b || (a == b && ia < ib); }

__global__ void __launch_bounds__(256) k_topk(const float* __restrict__ logits, int T, int E, int k,
                                              int32_t* __restrict__ ids, float* __restrict__ w, int32_t* err) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= T) return;
  const float* lr = logits + size_t(warp) * E;
  constexpr int kPer = kMaxE / 32;
  float v[kPer];
  uint32_t avail = 0;  // bit j: entry lane+32j exists and is not taken
  bool nan_seen = false;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    int e = lane + 32 * j;
    float x = -INFINITY;
    if (e < E) {
      x = lr[e];
      if (x != x) { nan_seen = true; x = -INFINITY; }
      avail |= 1u << j;
    }
    v[j] = x;
  }
  if (__any_sync(0xffffffffu, nan_seen) && lane == 0) set_error(err, MOE_ENAN);
  float sel_v[kMaxK];
  int sel_i[kMaxK];
  for (int r = 0; r < k; ++r) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    int bj = -1;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      if (((avail >> j) & 1u) && better(v[j], lane + 32 * j, bv, bi)) { bv = v[j]; bi = lane + 32 * j; bj = j; }
    }
    float wv = bv;
    int wi = bi;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      float ov = __shfl_xor_sync(0xffffffffu, wv, o);
      int oi = __shfl_xor_sync(0xffffffffu, wi, o);
      if (better(ov, oi, wv, wi)) { wv = ov; wi = oi; }
    }
    sel_v[r] = wv;
    sel_i[r] = wi;
    if (bj >= 0 && bi == wi) avail &= ~(1u << bj);
  }
  if (lane == 0) {
    const float m = sel_v[0];
    float den = 0.f;
    float p[kMaxK];
    for (int r = 0; r < k; ++r) {
      p[r] = expf(sel_v[r] - m);
      den += p[r];
    }
    for (int r = 0; r < k; ++r) {
      ids[size_t(warp) * k + r] = sel_i[r];
      w[size_t(warp) * k + r] = p[r] / den;
    }
  }
}

int launch_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w, int32_t* err, cudaStream_t s) {
  if (T <= 0) return MOE_OK;
  int blocks = (T * 32 + 255) / 256;
  k_topk<<<blocks, 256, 0, s>>>(logits, T, E, k, ids, w, err);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

}  // namespace moe
