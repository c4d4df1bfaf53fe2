// Adaptive expert-cache policy on the device.
//
// Strata expert paths, "哪些专家能长期留在显存？": accumulate how often each
// expert is routed to and decay the history periodically; within a layer,
// pair hot experts outside the cache with cold experts inside it and swap
// only when the heat difference reaches the threshold (default 1.5); sort all
// candidates by the difference and cap them per round (default 96); after an
// adjustment multiply the old heats by the decay (default 0.7); new weights
// become visible only after their copy completes, and an old slot is reused
// only after earlier reads of it have finished.
//
// The counters are fp32 and the policy is defined on them, so every step uses
// explicitly rounded single operations (__fadd_rn, __fsub_rn, __fmul_rn): no
// contraction into fused multiply-adds, identical results on every run.
#include "internal.h"

namespace moe {

// ------------------------------------------------------------- heat update
__global__ void __launch_bounds__(1024) k_heat(float* __restrict__ heat, const int32_t* __restrict__ ids, int n, int E,
                                               int layer, int32_t* err) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ int cnt[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  bool bad = false;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int e = ids[i];
    if (e < 0 || e >= E) { bad = true; continue; }
    atomicAdd(&cnt[e], 1);
  }
  if (bad) set_error(err, MOE_ERANGE);
  __syncthreads();
  float* row = heat + size_t(layer) * E;
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (cnt[e]) row[e] = __fadd_rn(row[e], float(cnt[e]));
}

int launch_heat_update(moe_cache* c, const int32_t* ids, int T, int k, int layer, int32_t* err, cudaStream_t s) {
  if (T <= 0) return MOE_OK;
  if (launch_pdl(k_heat, dim3(1), dim3(1024), size_t(c->E) * 4, s, c->heat, ids, T * k, c->E, layer, err) !=
      cudaSuccess)
    return MOE_ECUDA;
  return MOE_OK;
}

// ------------------------------------------------------------ sort helpers
// fp32 -> uint32 whose unsigned order is the float order.
__device__ __forceinline__ uint32_t ordered_bits(float f) {
  uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// In-place ascending bitonic sort of n (power of two) keys in shared memory.
__device__ void bitonic_sort(unsigned long long* key, int n) {
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int j = i ^ stride;
        if (j > i) {
          const bool up = (i & size) == 0;
          unsigned long long a = key[i], b = key[j];
          if ((a > b) == up) { key[i] = b; key[j] = a; }
        }
      }
      __syncthreads();
    }
  }
}

// ------------------------------------------------------------ plan: layer
// One CTA per layer.  Non-resident experts by (heat desc, id asc) and resident
// ones by (heat asc, id asc); the i-th pair is a candidate while
// fl32(h_hot - h_cold) >= threshold (the differences are non-increasing in i,
// so the candidates are a prefix).  Then the layer's heats decay.
__global__ void __launch_bounds__(1024) k_plan_layer(float* __restrict__ heat, const int32_t* __restrict__ resid, int E,
                                                     int P, float threshold, float decay,
                                                     unsigned long long* __restrict__ cand, int cand_stride,
                                                     int32_t* __restrict__ cand_count, int32_t* __restrict__ cold_of) {
  extern __shared__ unsigned long long sk[];
  unsigned long long* hot = sk;       // [P]
  unsigned long long* cold = sk + P;  // [P]
  __shared__ int s_nhot, s_ncold, s_ncand;
  const int l = blockIdx.x;
  float* hrow = heat + size_t(l) * E;
  const int32_t* rrow = resid + size_t(l) * E;
  if (threadIdx.x == 0) { s_nhot = 0; s_ncold = 0; s_ncand = 0; }
  __syncthreads();
  for (int i = threadIdx.x; i < P; i += blockDim.x) {
    unsigned long long kh = ~0ull, kc = ~0ull;
    if (i < E) {
      const uint32_t ob = ordered_bits(hrow[i]);
      if (rrow[i] < 0) { kh = (static_cast<unsigned long long>(~ob) << 32) | uint32_t(i); atomicAdd(&s_nhot, 1); }
      else { kc = (static_cast<unsigned long long>(ob) << 32) | uint32_t(i); atomicAdd(&s_ncold, 1); }
    }
    hot[i] = kh;
    cold[i] = kc;
  }
  __syncthreads();
  bitonic_sort(hot, P);
  bitonic_sort(cold, P);
  // Pairing stops at the first pair whose difference fails the test: with finite heats
  // the differences never increase along i, but a NaN (or inf - inf) fails the test
  // wherever it sits, so the candidates are the prefix before the first failure.
  const int npair = min(s_nhot, s_ncold);
  if (threadIdx.x == 0) s_ncand = npair;
  __syncthreads();
  for (int i = threadIdx.x; i < npair; i += blockDim.x) {
    const int a = int(hot[i] & 0xffffffffu), b = int(cold[i] & 0xffffffffu);
    if (!(__fsub_rn(hrow[a], hrow[b]) >= threshold)) atomicMin(&s_ncand, i);
  }
  __syncthreads();
  const int ncand = s_ncand;
  for (int i = threadIdx.x; i < ncand; i += blockDim.x) {
    const int a = int(hot[i] & 0xffffffffu), b = int(cold[i] & 0xffffffffu);
    const float d = __fsub_rn(hrow[a], hrow[b]);
    // global order: diff desc, layer asc, hot id asc (d >= threshold > 0, so its bits order like d)
    cand[size_t(l) * cand_stride + i] = (static_cast<unsigned long long>(0xffffffffu - __float_as_uint(d)) << 32) |
                                        (static_cast<unsigned long long>(l) << 16) | uint32_t(a);
    cold_of[size_t(l) * E + a] = b;
  }
  if (threadIdx.x == 0) cand_count[l] = ncand;
  __syncthreads();  // every thread has read the heats it compared before any is decayed
  for (int e = threadIdx.x; e < E; e += blockDim.x) hrow[e] = __fmul_rn(hrow[e], decay);
}

// ------------------------------------------------------------ plan: merge
__global__ void __launch_bounds__(1024) k_plan_merge(const unsigned long long* __restrict__ cand, int cand_stride,
                                                     const int32_t* __restrict__ cand_count, int L, int E, int P,
                                                     const int32_t* __restrict__ resid,
                                                     const int32_t* __restrict__ cold_of, int max_swaps,
                                                     moe_swap* __restrict__ plan, int32_t* __restrict__ n_out) {
  extern __shared__ unsigned long long keys[];  // [P]
  __shared__ int s_off[1024 + 1];
  if (threadIdx.x == 0) {
    int o = 0;
    for (int l = 0; l < L; ++l) { s_off[l] = o; o += cand_count[l]; }
    s_off[L] = o;
  }
  __syncthreads();
  const int total = s_off[L];
  for (int i = threadIdx.x; i < P; i += blockDim.x) keys[i] = ~0ull;
  __syncthreads();
  for (int l = 0; l < L; ++l) {
    const int n = s_off[l + 1] - s_off[l];
    for (int i = threadIdx.x; i < n; i += blockDim.x) keys[s_off[l] + i] = cand[size_t(l) * cand_stride + i];
  }
  __syncthreads();
  bitonic_sort(keys, P);
  const int n = min(total, max_swaps);
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const unsigned long long key = keys[i];
    const int l = int((key >> 16) & 0xffffu), a = int(key & 0xffffu);
    moe_swap sw;
    sw.layer = -1;  // an entry that fails the checks below is one the swap execution rejects
    sw.hot_expert = a;
    sw.cold_expert = -1;
    sw.slot = -1;
    sw.diff = __uint_as_float(0xffffffffu - uint32_t(key >> 32));
    if (l < L && a < E) {  // every key read was written by this round (a guard, not a path)
      const int b = cold_of[size_t(l) * E + a];
      if (b >= 0 && b < E) {
        sw.layer = l;
        sw.cold_expert = b;
        sw.slot = resid[size_t(l) * E + b];
      }
    }
    plan[i] = sw;
  }
  if (threadIdx.x == 0) *n_out = n;
}

static int pow2_at_least(int n) {
  int p = 1;
  while (p < n) p <<= 1;
  return p;
}

int launch_plan_swaps(moe_cache* c, const moe_policy_cfg* p, moe_swap* plan, int32_t* n, cudaStream_t s) {
  const int L = c->L, E = c->E;
  const int P = pow2_at_least(E);
  const int stride = (E + 1) / 2;
  auto* cand = reinterpret_cast<unsigned long long*>(c->plan_scratch);
  int32_t* cnt = reinterpret_cast<int32_t*>(cand + size_t(L) * stride);
  int32_t* cold_of = cnt + L;
  const size_t smem1 = size_t(2) * P * 8;
  if (smem1 > 48 * 1024 &&
      cudaFuncSetAttribute(k_plan_layer, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem1)) != cudaSuccess)
    return MOE_ECUDA;
  k_plan_layer<<<L, 1024, smem1, s>>>(c->heat, c->resid, E, P, p->threshold, p->decay, cand, stride, cnt, cold_of);
  MOE_LAUNCH_CHECK();
  const int PM = pow2_at_least(L * stride > 1 ? L * stride : 2);
  const size_t smem2 = size_t(PM) * 8;
  if (smem2 > 48 * 1024 &&
      cudaFuncSetAttribute(k_plan_merge, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem2)) != cudaSuccess)
    return MOE_ECUDA;
  k_plan_merge<<<1, 1024, smem2, s>>>(cand, stride, cnt, L, E, PM, c->resid, cold_of, p->max_swaps, plan, n);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

// ----------------------------------------------------------- apply swaps
// flat_cold: cold_expert is layer * E + expert of the evicted expert, or -1
// when the slot is empty (global LRU plans, whose victims may be in any layer).
__global__ void k_swap_unmap(const moe_swap* __restrict__ plan, const int32_t* __restrict__ n, int32_t* resid,
                             int32_t* slot_owner, int E, int L, int nslots, int32_t* err, int flat_cold) {
  const int cnt = *n;
  for (int i = threadIdx.x; i < cnt; i += blockDim.x) {
    const moe_swap sw = plan[i];
    if (sw.layer < 0 || sw.layer >= L || sw.slot < 0 || sw.slot >= nslots) { set_error(err, MOE_ERANGE); continue; }
    if (flat_cold) {
      if (sw.cold_expert < -1 || sw.cold_expert >= L * E) { set_error(err, MOE_ERANGE); continue; }
      if (sw.cold_expert < 0) {  // an empty slot: nothing to unmap
        if (slot_owner[sw.slot] != -1) set_error(err, MOE_ERANGE);
        continue;
      }
      if (resid[sw.cold_expert] != sw.slot) { set_error(err, MOE_ERANGE); continue; }
      resid[sw.cold_expert] = -1;
      slot_owner[sw.slot] = -1;
      continue;
    }
    if (sw.cold_expert < 0 || sw.cold_expert >= E) { set_error(err, MOE_ERANGE); continue; }
    const size_t f = size_t(sw.layer) * E + sw.cold_expert;
    if (resid[f] != sw.slot) { set_error(err, MOE_ERANGE); continue; }
    resid[f] = -1;
    slot_owner[sw.slot] = -1;
  }
}

// Fixed-shape copy: blockIdx.y is the swap index; blocks beyond the
// device-side count return at once (FreeToken notes, section 4: one
// fixed-shape launch with a valid-count mask).
__global__ void __launch_bounds__(256) k_swap_copy(const moe_swap* __restrict__ plan, const int32_t* __restrict__ n,
                                                   const uint8_t* __restrict__ backing, uint8_t* __restrict__ slots,
                                                   size_t blob_bytes, int E, int L, int nslots) {
  const int i = blockIdx.y;
  if (i >= *n) return;
  const moe_swap sw = plan[i];
  if (sw.layer < 0 || sw.layer >= L || sw.hot_expert < 0 || sw.hot_expert >= E || sw.slot < 0 || sw.slot >= nslots)
    return;
  const uint4* src = reinterpret_cast<const uint4*>(backing + (size_t(sw.layer) * E + sw.hot_expert) * blob_bytes);
  uint4* dst = reinterpret_cast<uint4*>(slots + size_t(sw.slot) * blob_bytes);
  const size_t n16 = blob_bytes / 16;
  for (size_t j = size_t(blockIdx.x) * blockDim.x + threadIdx.x; j < n16; j += size_t(gridDim.x) * blockDim.x)
    dst[j] = src[j];
}

__global__ void k_swap_publish(const moe_swap* __restrict__ plan, const int32_t* __restrict__ n, int32_t* resid,
                               int32_t* slot_owner, int E, int L, int nslots) {
  const int cnt = *n;
  for (int i = threadIdx.x; i < cnt; i += blockDim.x) {
    const moe_swap sw = plan[i];
    if (sw.layer < 0 || sw.layer >= L || sw.hot_expert < 0 || sw.hot_expert >= E || sw.slot < 0 || sw.slot >= nslots)
      continue;
    const int f = sw.layer * E + sw.hot_expert;
    resid[f] = sw.slot;
    slot_owner[sw.slot] = f;
  }
}

int launch_apply_swaps(moe_cache* c, const moe_swap* plan, const int32_t* n, int max_swaps, cudaStream_t compute,
                       cudaStream_t copy, bool flat_cold) {
  k_swap_unmap<<<1, 256, 0, compute>>>(plan, n, c->resid, c->slot_owner, c->E, c->L, c->nslots, nullptr,
                                       flat_cold ? 1 : 0);
  MOE_LAUNCH_CHECK();
  MOE_CUDA_TRY(cudaEventRecord(c->ev_unmapped, compute));
  MOE_CUDA_TRY(cudaStreamWaitEvent(copy, c->ev_unmapped, 0));
  if (max_swaps > 0) {
    dim3 grid(16, max_swaps);
    k_swap_copy<<<grid, 256, 0, copy>>>(plan, n, reinterpret_cast<const uint8_t*>(c->backing), c->slots,
                                        c->blob_bytes, c->E, c->L, c->nslots);
    MOE_LAUNCH_CHECK();
  }
  MOE_CUDA_TRY(cudaEventRecord(c->ev_copied, copy));
  MOE_CUDA_TRY(cudaStreamWaitEvent(compute, c->ev_copied, 0));
  k_swap_publish<<<1, 256, 0, compute>>>(plan, n, c->resid, c->slot_owner, c->E, c->L, c->nslots);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

}  // namespace moe
