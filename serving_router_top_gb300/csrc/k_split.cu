// Activations as sums of NVFP4 terms, for the block-scaled FP4 tensor-core path.
//
// A block-scaled FP4 MMA takes both operands in the weights' format (PLE
// offload page, "NVFP4 code 和 scale 如何反量化": value = E2M1 code x FP8-E4M3
// scale per 16 values x FP32 global scale).  An activation row v (bf16 x, or
// the fp32 intermediate h) is written as R terms q_1 = Q(v), q_2 = Q(v - q_1),
// ..., each its own operand row; the product of the R terms summed (with each
// term's global scale) approaches the product of v.  Q per term:
//   G: the power of two with max|v| / (6 G) <= 448, the smallest such;
//   s: per 16 values, the smallest non-negative E4M3 value with 6 s G >= max|v|
//      of the block (so no code saturates);
//   code: the E2M1 value nearest to v / (s G), ties to the even code.
// The residual is kept in fp32: exact for bf16 rows (the few bits of every term
// fit), within one fp32 rounding per term for fp32 rows.
#include "internal.h"

namespace moe {
namespace split {

// fp32 pair -> two E2M1 codes in one byte (lo in the low nibble), round to nearest even.
__device__ __forceinline__ uint32_t e2m1x2_of(float lo, float hi) {
  uint32_t d;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(d)
      : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ float e4m3_value_of(uint32_t b) {
  uint32_t h2 = e4m3x2_to_f16x2(b);
  return __low2float(*reinterpret_cast<__half2*>(&h2));
}

// The smallest non-negative E4M3 byte s (0x00..0x7E) with 6 * value(s) * G >= bmax; every
// product involved is exact in fp32 (value(s) has 4 significant bits, 6 two, G is a
// power of two), so the test is exact.
__device__ __forceinline__ uint32_t e4m3_ceil_byte(float bmax, float G) {
  if (!(bmax > 0.f)) return 0u;
  uint32_t s;
  {
    uint16_t t;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(t) : "f"(0.f), "f"(bmax / (6.0f * G)));
    s = t & 0xffu;
  }
  s &= 0x7fu;
  if (s > 0x7eu) s = 0x7eu;
  while (s < 0x7eu && 6.0f * e4m3_value_of(s) * G < bmax) ++s;
  while (s > 0u && 6.0f * e4m3_value_of(s - 1) * G >= bmax) --s;
  return s;
}

// One warp per row; lane l owns the row's 16-value blocks l, l + 32, ... (VPL values).
template <int VPL, bool SRC32>
__global__ void __launch_bounds__(256) k_split(const void* __restrict__ src, int rows, int K, int ld, int R,
                                               uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                                               float* __restrict__ gscale) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= rows) return;
  constexpr int BPL = VPL / 16;  // blocks per lane
  const int nblk = K / 16;
  float v[VPL];
#pragma unroll
  for (int b = 0; b < BPL; ++b) {
    const int blk = lane + 32 * b;
#pragma unroll
    for (int j = 0; j < 16; j += 8) {
      if (blk < nblk) {
        if (SRC32) {
          const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(src) + size_t(warp) * ld +
                                                            blk * 16 + j);
          const float4 a = p[0], c = p[1];
          v[b * 16 + j + 0] = a.x; v[b * 16 + j + 1] = a.y; v[b * 16 + j + 2] = a.z; v[b * 16 + j + 3] = a.w;
          v[b * 16 + j + 4] = c.x; v[b * 16 + j + 5] = c.y; v[b * 16 + j + 6] = c.z; v[b * 16 + j + 7] = c.w;
        } else {
          const uint4 q = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(src) + size_t(warp) * ld +
                                                          blk * 16 + j);
          const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            v[b * 16 + j + 2 * i] = __uint_as_float(u[i] << 16);
            v[b * 16 + j + 2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[b * 16 + j + i] = 0.f;
      }
    }
  }
  for (int r = 0; r < R; ++r) {
    const size_t orow = size_t(warp) * R + r;
    float bm[BPL];
    float am = 0.f;
#pragma unroll
    for (int b = 0; b < BPL; ++b) {
      float m = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) m = fmaxf(m, fabsf(v[b * 16 + j]));
      bm[b] = m;
      am = fmaxf(am, m);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    // G: the smallest power of two with am / (6 G) <= 448
    float G = 1.0f;
    if (am > 0.f) {
      int e;
      frexpf(am / (6.0f * 448.0f), &e);
      G = ldexpf(1.0f, e);
      // settled with exact tests (2688 G is exact): 2688 G >= am > 1344 G
      while (2688.0f * G * 0.5f >= am) G *= 0.5f;
      while (2688.0f * G < am) G *= 2.0f;
    }
    if (lane == 0) gscale[orow] = G;
#pragma unroll
    for (int b = 0; b < BPL; ++b) {
      const int blk = lane + 32 * b;
      const uint32_t sb = e4m3_ceil_byte(bm[b], G);
      const float sG = e4m3_value_of(sb) * G;
      uint32_t packed[2] = {0u, 0u};
#pragma unroll
      for (int j = 0; j < 16; j += 2) {
        // correctly rounded quotients: for bf16 rows (and their few-bit residuals) a quotient
        // that is not itself a tie of the E2M1 grid never rounds onto one
        const uint32_t c = sb ? e2m1x2_of(__fdiv_rn(v[b * 16 + j], sG), __fdiv_rn(v[b * 16 + j + 1], sG)) : 0u;
        packed[j >> 3] |= c << (4 * (j & 7));
        const float2 q = f16x2_to_f32x2(e2m1x2_to_f16x2(c));
        v[b * 16 + j] -= q.x * sG;
        v[b * 16 + j + 1] -= q.y * sG;
      }
      if (blk < nblk) {
        *reinterpret_cast<uint2*>(codes + orow * (K / 2) + blk * 8) = make_uint2(packed[0], packed[1]);
        scales[orow * (K / 16) + blk] = uint8_t(sb);
      }
    }
  }
}

}  // namespace split

int launch_split_nvfp4(const void* src, int src_is_fp32, int rows, int K, int ld, int R, uint8_t* codes,
                       uint8_t* scales, float* gscale, cudaStream_t s) {
  if (rows <= 0) return MOE_OK;
  const int vpl = K / 32;  // values per lane
  const dim3 grid((rows * 32 + 255) / 256), block(256);
  cudaError_t rc;
#define MOE_SPLIT_CASE(V)                                                                                   \
  if (vpl <= V)                                                                                             \
    rc = src_is_fp32 ? (split::k_split<V, true><<<grid, block, 0, s>>>(src, rows, K, ld, R, codes, scales,   \
                                                                      gscale), cudaGetLastError())         \
                     : (split::k_split<V, false><<<grid, block, 0, s>>>(src, rows, K, ld, R, codes, scales,  \
                                                                       gscale), cudaGetLastError());       \
  else
  MOE_SPLIT_CASE(16) MOE_SPLIT_CASE(32) MOE_SPLIT_CASE(64) MOE_SPLIT_CASE(128) return MOE_EINVAL;
#undef MOE_SPLIT_CASE
  return rc == cudaSuccess ? MOE_OK : MOE_ECUDA;
}

}  // namespace moe

extern "C" int moe_nvfp4_split(const void* src, int src_is_fp32, int rows, int K, int ld, int R, uint8_t* codes,
                               uint8_t* scales, float* gscale, moe_stream_t stream) {
  using namespace moe;
  if (!src || !codes || !scales || !gscale || rows < 0 || K < 64 || K > 4096 || (K & (K - 1)) || ld < K || R < 1 ||
      R > 8 || (ld % 8) || (reinterpret_cast<uintptr_t>(src) & 15) || (reinterpret_cast<uintptr_t>(codes) & 7))
    return MOE_EINVAL;
  return launch_split_nvfp4(src, src_is_fp32, rows, K, ld, R, codes, scales, gscale,
                            reinterpret_cast<cudaStream_t>(stream));
}
