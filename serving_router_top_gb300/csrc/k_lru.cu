// Global LRU over the cache slots.
//
// FreeToken reading notes, section 3.3: one LRU shared by every layer, over
// (layer, expert): a hit refreshes the expert's recency, a fill admits the
// newly chosen expert, eviction removes the least recently used.  Section 4:
// victims are not found by a scan per eviction -- one pass yields K
// candidates and the misses take the first q <= K, so the cost does not grow
// with the number of misses.
//
// Recency is a per-slot tick: the value of the cache's LRU clock (one count
// per planned layer call) at the slot's last use.  One CTA per call:
//   1. advance the clock; the call's resident groups mark their slots;
//   2. one pass over the slots: each warp keeps the 32 smallest victim keys of
//      its share in a lane-sorted list (lane i the i-th smallest), merging each
//      sorted batch of 32 into it; then a tree of merges across the warps;
//   3. the call's misses in group order take the first victims.
// A victim key orders empty slots first, then (tick, slot) ascending; a slot
// the call used is no candidate.
#include "internal.h"

namespace moe {
namespace {

constexpr int kLruWarps = 32;
constexpr unsigned long long kNoKey = ~0ull;
constexpr int kSlotBits = 24;  // slots < 2^24

__device__ __forceinline__ unsigned long long lru_key(int slot, uint32_t tick, int owner, uint32_t clock) {
  if (tick >= clock) return kNoKey;  // used by this call
  const unsigned long long rank = owner < 0 ? 0ull : static_cast<unsigned long long>(tick) + 1ull;
  return (rank << kSlotBits) | static_cast<unsigned long long>(slot);
}

// Bitonic sort of one key per lane, ascending across the lanes.
__device__ __forceinline__ unsigned long long warp_sort_asc(unsigned long long v, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, stride);
      const bool up = (lane & size) == 0, lower = (lane & stride) == 0;
      v = (lower == up) ? (v < o ? v : o) : (v > o ? v : o);
    }
  return v;
}

// The 32 smallest of two lane-sorted lists, lane-sorted: the pairwise smaller
// of a and b reversed is a bitonic sequence holding exactly them.
__device__ __forceinline__ unsigned long long merge_lowest(unsigned long long a, unsigned long long b, int lane) {
  const unsigned long long br = __shfl_sync(0xffffffffu, b, 31 - lane);
  unsigned long long c = a < br ? a : br;
#pragma unroll
  for (int stride = 16; stride > 0; stride >>= 1) {
    const unsigned long long o = __shfl_xor_sync(0xffffffffu, c, stride);
    c = (lane & stride) == 0 ? (c < o ? c : o) : (c > o ? c : o);
  }
  return c;
}

__global__ void __launch_bounds__(kLruWarps * 32) k_lru_plan(uint32_t* __restrict__ tick, uint32_t* __restrict__ clock_dev,
                                                            const int32_t* __restrict__ slot_owner, int nslots,
                                                            const int32_t* __restrict__ num_groups,
                                                            const int32_t* __restrict__ grp_expert,
                                                            const int32_t* __restrict__ grp_src,
                                                            const int32_t* __restrict__ grp_slot, int layer, int K,
                                                            moe_swap* __restrict__ plan, int32_t* __restrict__ n_out,
                                                            int32_t* err) {
  __shared__ uint32_t s_clock;
  __shared__ unsigned long long s_list[kLruWarps][32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = *num_groups;
  if (tid == 0) {
    const uint32_t c = *clock_dev + 1u;
    if (c == 0xffffffffu) set_error(err, MOE_ERANGE);  // the next call would wrap
    *clock_dev = c;
    s_clock = c;
  }
  __syncthreads();
  const uint32_t clock = s_clock;
  // 1. the call's hits are used now
  for (int g = tid; g < G; g += blockDim.x)
    if (grp_src[g] == MOE_SRC_RESIDENT) {
      const int s = grp_slot[g];
      if (s >= 0 && s < nslots) tick[s] = clock;
    }
  __syncthreads();
  // 2. one pass: the 32 smallest keys of each warp's share of the slots
  unsigned long long best = kNoKey;
  const int per = (nslots + kLruWarps - 1) / kLruWarps;
  const int s0 = warp * per, s1 = min(nslots, s0 + per);
  for (int b = s0; b < s1; b += 32) {
    const int s = b + lane;
    const unsigned long long key = s < s1 ? lru_key(s, __ldcg(tick + s), slot_owner[s], clock) : kNoKey;
    if (__all_sync(0xffffffffu, key == kNoKey)) continue;
    best = merge_lowest(best, warp_sort_asc(key, lane), lane);
  }
  s_list[warp][lane] = best;
  __syncthreads();
  for (int half = kLruWarps / 2; half > 0; half >>= 1) {
    if (warp < half) s_list[warp][lane] = merge_lowest(s_list[warp][lane], s_list[warp + half][lane], lane);
    __syncthreads();
  }
  // 3. the i-th miss of the call (group order) takes the i-th victim
  if (warp == 0) {
    const unsigned long long v = s_list[0][lane];
    const int nv = __popc(__ballot_sync(0xffffffffu, v != kNoKey));
    const int q = min(K, nv);
    int m = 0;
    for (int g0 = 0; g0 < G && m < q; g0 += 32) {
      const int g = g0 + lane;
      const int src = g < G ? grp_src[g] : MOE_SRC_RESIDENT;
      const bool miss = src == MOE_SRC_STAGED || src == MOE_SRC_MISSING;
      const unsigned bal = __ballot_sync(0xffffffffu, miss);
      const int idx = m + __popc(bal & ((1u << lane) - 1u));
      const unsigned long long vk = __shfl_sync(0xffffffffu, v, idx & 31);
      if (miss && idx < q) {
        const int slot = int(vk & ((1ull << kSlotBits) - 1ull));
        moe_swap sw;
        sw.layer = layer;
        sw.hot_expert = grp_expert[g];
        sw.cold_expert = slot_owner[slot];
        sw.slot = slot;
        sw.diff = 0.f;
        plan[idx] = sw;
        tick[slot] = clock;
      }
      m += __popc(bal);
    }
    if (lane == 0) *n_out = min(m, q);
  }
}

}  // namespace

int launch_lru_plan(moe_cache* c, const moe_ws* ws, int layer, int K, moe_swap* plan, int32_t* n, cudaStream_t s) {
  k_lru_plan<<<1, kLruWarps * 32, 0, s>>>(c->lru_tick, c->lru_clock, c->slot_owner, c->nslots, ws->num_groups,
                                          ws->grp_expert, ws->grp_src, ws->grp_slot, layer, K, plan, n, ws->error);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

}  // namespace moe
