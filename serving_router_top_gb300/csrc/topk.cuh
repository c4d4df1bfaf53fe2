// Top-k of one token by one warp: the device routine shared by the top-k
// kernel and the fused small-window top-k + grouping kernel.
//
// Strata expert paths, "显存里缓存的是什么？": the k largest logits (ties to the
// lower expert id), w_r = exp(l_r - l_0) / sum_j exp(l_j - l_0) over the chosen
// k -- equal to a softmax over all E renormalised over the k.
#pragma once
#include "internal.h"

namespace moe {

// ------------------------------------------------------------------- top-k
// One warp per token; lane j holds logits j, j+32, ... (KPER per lane).
// Each lane keeps its best untaken entry; a round takes the warp-wide best by
// (value desc, id asc) with a shuffle reduction and only the owning lane
// rescans.  Lane r keeps the r-th selection.  NaN logits record MOE_ENAN and
// rank as -inf.
// fp32 -> uint32 whose unsigned order is the float order (-inf lowest).
__device__ __forceinline__ unsigned ordered_key(float f) {
  const unsigned b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// The float whose order_key is k (exact inverse).
__device__ __forceinline__ float float_of_key(unsigned k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Top-k of one token by one warp.  Lane l holds logits l, l+32, ... (KPER per
// lane) as order-preserving keys (0 below every real key for entries past E),
// sorted once per lane by (key desc, id asc) with a register bitonic network;
// each round then takes the warp-wide best head -- the largest key, ties to
// the lowest id -- and the winning lane shifts its list.  Lane r writes the
// r-th selection; weights are exp(l - l_0) / sum over the chosen.  NaN logits
// record MOE_ENAN and rank as -inf.
template <int KPER>
__device__ __forceinline__ void topk_token(const float* lr, int E, int k, int lane, int32_t* ids, float* w,
                                           int32_t* err) {
  unsigned u[KPER];
  int jj[KPER];
  bool nan_seen = false;
#pragma unroll
  for (int j = 0; j < KPER; ++j) {
    const int e = lane + 32 * j;
    unsigned key = 0u;
    if (e < E) {
      float x = lr[e];
      if (x != x) { nan_seen = true; x = -INFINITY; }
      key = ordered_key(x);
    }
    u[j] = key;
    jj[j] = j;
  }
  if (__any_sync(0xffffffffu, nan_seen) && lane == 0) set_error(err, MOE_ENAN);
  // (key desc, j asc): j orders like the expert id within a lane
  auto first = [](unsigned ka, int ja, unsigned kb, int jb) { return ka > kb || (ka == kb && ja < jb); };
#pragma unroll
  for (int size = 2; size <= KPER; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
      for (int i = 0; i < KPER; ++i) {
        const int l = i ^ stride;
        if (l > i) {
          const bool desc = (i & size) == 0;
          const bool sw = desc ? first(u[l], jj[l], u[i], jj[i]) : first(u[i], jj[i], u[l], jj[l]);
          if (sw) {
            const unsigned tu = u[i];
            u[i] = u[l];
            u[l] = tu;
            const int tj = jj[i];
            jj[i] = jj[l];
            jj[l] = tj;
          }
        }
      }
    }
  }
  int my_id = 0;
  float my_p = 0.f, m = 0.f, den = 0.f;
  for (int r = 0; r < k; ++r) {
    const unsigned kmax = __reduce_max_sync(0xffffffffu, u[0]);
    const unsigned id = unsigned(lane + 32 * jj[0]);
    const int wi = int(__reduce_min_sync(0xffffffffu, u[0] == kmax ? id : 0x7fffffffu));
    const float wv = float_of_key(kmax);
    if (r == 0) m = wv;
    const float p = expf(wv - m);
    den += p;
    if (lane == r) { my_id = wi; my_p = p; }
    if (lane == (wi & 31)) {
#pragma unroll
      for (int i = 0; i + 1 < KPER; ++i) {
        u[i] = u[i + 1];
        jj[i] = jj[i + 1];
      }
      u[KPER - 1] = 0u;
      jj[KPER - 1] = KPER;
    }
  }
  if (lane < k) {
    ids[lane] = my_id;
    w[lane] = my_p / den;
  }
}

}  // namespace moe

namespace moe {

// Top-k of up to 32 tokens by one CTA, G warps per token (warps tok*G ..
// tok*G + G - 1; G*k <= 128).  Warp wg of a token takes the k best of its
// slice of ceil(E/G) experts by selection rounds (KP1 logits per lane; the
// lane's best by value desc, id asc, then the warp's best key and, among equal
// keys, the lowest id), writing them to cand as (key << 32 | ~id); after a CTA
// barrier the token's first warp takes the k best of the G*k candidates the
// same way.  Ids and weights equal topk_token's: the same order (value desc,
// id asc) and the weights' terms summed in rank order.  Every thread of the CTA
// must call this (it holds one __syncthreads).
template <int KP1>
__device__ __forceinline__ void topk_tokens_cta(const float* __restrict__ logits, int T, int E, int k, int G,
                                                int32_t* __restrict__ ids, float* __restrict__ w, int32_t* err,
                                                unsigned long long* cand) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tok = warp / G, wg = warp - tok * G;
  const int nslice = (E + G - 1) / G;
  if (tok < T) {
    const float* lr = logits + size_t(tok) * E;
    const int e0 = wg * nslice, e1 = min(E, e0 + nslice);
    unsigned key[KP1];
    bool nan_seen = false;
#pragma unroll
    for (int j = 0; j < KP1; ++j) {
      const int e = e0 + lane + 32 * j;
      unsigned kk = 0u;
      if (e < e1) {
        float x = lr[e];
        if (x != x) {
          nan_seen = true;
          x = -INFINITY;
        }
        kk = ordered_key(x);
      }
      key[j] = kk;
    }
    if (__any_sync(0xffffffffu, nan_seen) && lane == 0) set_error(err, MOE_ENAN);
    unsigned long long* out = cand + size_t(tok * G + wg) * k;
    for (int r = 0; r < k; ++r) {
      unsigned bk = key[0];
      int bj = 0;
#pragma unroll
      for (int j = 1; j < KP1; ++j)
        if (key[j] > bk) {  // strict: an equal key at a higher j has a higher id
          bk = key[j];
          bj = j;
        }
      const unsigned kmax = __reduce_max_sync(0xffffffffu, bk);
      const unsigned mine = unsigned(e0 + lane + 32 * bj);
      const unsigned wid = __reduce_min_sync(0xffffffffu, bk == kmax ? mine : 0xffffffffu);
      if (lane == 0) out[r] = (static_cast<unsigned long long>(kmax) << 32) | (0xffffffffu - wid);
      if (bk == kmax && mine == wid) {
#pragma unroll
        for (int j = 0; j < KP1; ++j)
          if (j == bj) key[j] = 0u;
      }
    }
  }
  __syncthreads();
  if (tok < T && wg == 0) {
    const int nc = G * k;
    const unsigned long long* cc = cand + size_t(tok) * G * k;
    unsigned long long c[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = lane + 32 * q;
      c[q] = i < nc ? cc[i] : 0ull;
    }
    int my_id = 0;
    float m = 0.f, den = 0.f, my_p = 0.f;
    for (int r = 0; r < k; ++r) {
      unsigned long long b = c[0];
      int bq = 0;
#pragma unroll
      for (int q = 1; q < 4; ++q)
        if (c[q] > b) {
          b = c[q];
          bq = q;
        }
      const unsigned hi = __reduce_max_sync(0xffffffffu, unsigned(b >> 32));
      const unsigned lo = __reduce_max_sync(0xffffffffu, unsigned(b >> 32) == hi ? unsigned(b) : 0u);
      const unsigned long long best = (static_cast<unsigned long long>(hi) << 32) | lo;
      if (b == best) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (q == bq) c[q] = 0ull;
      }
      const float wv = float_of_key(hi);
      if (r == 0) m = wv;
      const float p = expf(wv - m);
      den += p;
      if (lane == r) {
        my_id = int(0xffffffffu - lo);
        my_p = p;
      }
    }
    if (lane < k) {
      ids[size_t(tok) * k + lane] = my_id;
      w[size_t(tok) * k + lane] = my_p / den;
    }
  }
}

}  // namespace moe
