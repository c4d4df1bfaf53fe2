// Dedupe of one layer's selections into expert groups, with the residency lookup.
//
// Strata expert paths, "路由以后，专家怎样分工？": repeated experts of one layer
// and window form one group that records its input and output positions;
// "哪些专家能长期留在显存？": the residency table maps (layer, expert) to a slot
// or a "not resident" value.  FreeToken notes, section 4: the dedupe, the
// classification against the residency table and the id -> slot rewrite stay
// on the device (no host round trip), so the step can be captured in a graph.
//
// Canonical output: groups by ascending expert id; within a group, entries by
// ascending token; an entry's output position is t*k + r.
//
// One CTA (1024 threads): a shared-memory histogram, a block scan over the E
// experts, then placement in token chunks -- within a chunk each expert keeps
// a bitmap of the tokens that chose it, and an entry's rank in its group is
// the experts' running count plus the popcount of the bits below its token.
#include "topk.cuh"

namespace moe {

__device__ __forceinline__ int block_excl_scan(int v, int* warp_sums, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  total = warp_sums[nw - 1];
  int before = warp ? warp_sums[warp - 1] : 0;
  __syncthreads();
  return before + x - v;
}

// Group g is expert e with entries from off on: its slot from the residency
// table, else the staging table, else MISSING; counts resident/staged/missing.
// tail: every entry of the group ranks at or past the tail-skip threshold
// (Strata page, "跳过尾部专家"), so a non-resident expert is dropped instead:
// no staging slot, no blob, no MISSING error.
__device__ __forceinline__ void resolve_group(int g, int e, int off, int layer, int E, const int32_t* resid,
                                              const int32_t* stage, const uint8_t* slots, const uint8_t* staging,
                                              size_t blob_bytes, int nslots, int nstaging, int32_t* grp_expert,
                                              int32_t* grp_off, int32_t* grp_slot, int32_t* grp_src,
                                              const uint8_t** grp_blob, int32_t* err, int* s_hit, int* s_stg,
                                              int* s_miss, bool tail, int* s_skip) {
  grp_expert[g] = e;
  grp_off[g] = off;
  const int flat = layer * E + e;
  // no residency table: the groups are bound to staging slots later (streamed prefill)
  if (!resid) {
    grp_slot[g] = -1;
    grp_src[g] = MOE_SRC_STAGED;
    grp_blob[g] = nullptr;
    atomicAdd(s_stg, 1);
    return;
  }
  int slot = resid[flat];
  const int st = stage ? stage[flat] : -1;  // read with the residency entry: one round trip, not two
  int src = MOE_SRC_MISSING;
  const uint8_t* blob = nullptr;
  if (slot >= 0) {
    if (slot < nslots) { src = MOE_SRC_RESIDENT; blob = slots + size_t(slot) * blob_bytes; }
    else { set_error(err, MOE_ERANGE); slot = -1; }
  }
  if (src == MOE_SRC_MISSING && tail) {
    grp_slot[g] = -1;
    grp_src[g] = MOE_SRC_SKIPPED;
    grp_blob[g] = nullptr;
    atomicAdd(s_skip, 1);
    return;
  }
  if (src == MOE_SRC_MISSING) {
    if (st >= 0 && st < nstaging) { slot = st; src = MOE_SRC_STAGED; blob = staging + size_t(st) * blob_bytes; }
    else if (st >= nstaging) set_error(err, MOE_ERANGE);
  }
  if (src == MOE_SRC_MISSING) { slot = -1; set_error(err, MOE_EMISSING); }
  grp_slot[g] = slot;
  grp_src[g] = src;
  grp_blob[g] = blob;
  atomicAdd(src == MOE_SRC_RESIDENT ? s_hit : src == MOE_SRC_STAGED ? s_stg : s_miss, 1);
}

// The single-CTA grouping of T*k <= 4096 entries (the CTA's threads, sm: its
// dynamic shared memory of 4E + E*W ints): counts (and, with the tail skip,
// each expert's lowest rank; with heat_row, the heat update of the window),
// scans, group table with the lookup, stable placement in token order.
__device__ __forceinline__ void group_body(int* sm, const int32_t* __restrict__ ids, int T, int k, int E, int layer,
                                           const int32_t* __restrict__ resid, const int32_t* __restrict__ stage,
                                           const uint8_t* slots, const uint8_t* staging, size_t blob_bytes, int nslots,
                                           int nstaging, int32_t* __restrict__ num_groups,
                                           int32_t* __restrict__ grp_expert, int32_t* __restrict__ grp_off,
                                           int32_t* __restrict__ grp_slot, int32_t* __restrict__ grp_src,
                                           const uint8_t** __restrict__ grp_blob, int32_t* __restrict__ ent_tok,
                                           int32_t* __restrict__ ent_pos, unsigned long long* stats, int32_t* err, int W,
                                           float* __restrict__ hmax, int maxTk, int skip_rank,
                                           float* __restrict__ heat_row) {
  int* cnt = sm;                                       // [E]
  int* off = cnt + E;                                  // [E]
  int* base = off + E;                                 // [E]
  int* minr = base + E;                                // [E] lowest rank choosing each expert
  uint32_t* bits = reinterpret_cast<uint32_t*>(minr + E);  // [E][W]
  __shared__ int warp_sums[32];
  __shared__ int s_hit, s_stg, s_miss, s_skip;
  const int n = T * k;
  const int chunk = W * 32;

  for (int e = threadIdx.x; e < E; e += blockDim.x) { cnt[e] = 0; base[e] = 0; minr[e] = k; }
  // the expert kernels of this call accumulate max|h| per row into hmax
  if (hmax) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) hmax[i] = 0.f;
    for (int i = threadIdx.x; i < T; i += blockDim.x) hmax[maxTk + i] = 0.f;
  }
  if (threadIdx.x == 0) { s_hit = 0; s_stg = 0; s_miss = 0; s_skip = 0; }
  __syncthreads();
  bool bad = false;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    int e = ids[i];
    if (e < 0 || e >= E) { bad = true; continue; }
    atomicAdd(&cnt[e], 1);
    if (skip_rank > 0) atomicMin(&minr[e], i % k);
  }
  if (bad) set_error(err, MOE_ERANGE);
  __syncthreads();

  // scan counts and presence (E <= blockDim.x)
  const int e = threadIdx.x;
  const int c = e < E ? cnt[e] : 0;
  if (heat_row && c > 0) heat_row[e] = __fadd_rn(heat_row[e], float(c));  // as the heat-update kernel
  int total_entries, total_groups;
  const int ex_c = block_excl_scan(c, warp_sums, total_entries);
  const int ex_g = block_excl_scan(c > 0 ? 1 : 0, warp_sums, total_groups);
  if (e < E) off[e] = ex_c;
  if (e < E && c > 0)
    resolve_group(ex_g, e, ex_c, layer, E, resid, stage, slots, staging, blob_bytes, nslots, nstaging, grp_expert,
                  grp_off, grp_slot, grp_src, grp_blob, err, &s_hit, &s_stg, &s_miss,
                  skip_rank > 0 && minr[e] >= skip_rank, &s_skip);
  __syncthreads();
  if (threadIdx.x == 0) {
    *num_groups = total_groups;
    grp_off[total_groups] = total_entries;
    if (stats) add_stats(stats + size_t(layer) * kStats, total_groups, s_hit, s_stg, s_miss, s_skip);
  }

  // stable placement, one token chunk at a time
  for (int t0 = 0; t0 < T; t0 += chunk) {
    const int t1 = min(T, t0 + chunk);
    for (int i = threadIdx.x; i < E * W; i += blockDim.x) bits[i] = 0u;
    __syncthreads();
    for (int i = t0 * k + threadIdx.x; i < t1 * k; i += blockDim.x) {
      const int ex = ids[i];
      if (ex < 0 || ex >= E) continue;
      const int lt = i / k - t0;
      uint32_t old = atomicOr(&bits[ex * W + (lt >> 5)], 1u << (lt & 31));
      if (old & (1u << (lt & 31))) set_error(err, MOE_ERANGE);  // an expert chosen twice by one token
    }
    __syncthreads();
    for (int i = t0 * k + threadIdx.x; i < t1 * k; i += blockDim.x) {
      const int ex = ids[i];
      if (ex < 0 || ex >= E) continue;
      const int t = i / k, lt = t - t0, wd = lt >> 5;
      const uint32_t* row = bits + ex * W;
      int rank = base[ex] + __popc(row[wd] & ((1u << (lt & 31)) - 1u));
      for (int w = 0; w < wd; ++w) rank += __popc(row[w]);
      const int pos = off[ex] + rank;
      ent_tok[pos] = t;
      ent_pos[pos] = i;
    }
    __syncthreads();
    for (int ex = threadIdx.x; ex < E; ex += blockDim.x) {
      int s = 0;
      for (int w = 0; w < W; ++w) s += __popc(bits[ex * W + w]);
      base[ex] += s;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(1024) k_group(const int32_t* __restrict__ ids, int T, int k, int E, int layer,
                                                const int32_t* __restrict__ resid, const int32_t* __restrict__ stage,
                                                const uint8_t* slots, const uint8_t* staging, size_t blob_bytes, int nslots,
                                                int nstaging, int32_t* __restrict__ num_groups,
                                                int32_t* __restrict__ grp_expert, int32_t* __restrict__ grp_off,
                                                int32_t* __restrict__ grp_slot, int32_t* __restrict__ grp_src,
                                                const uint8_t** __restrict__ grp_blob, int32_t* __restrict__ ent_tok,
                                                int32_t* __restrict__ ent_pos, unsigned long long* stats, int32_t* err, int W,
                                                float* __restrict__ hmax, int maxTk, int skip_rank,
                                                float* __restrict__ heat_row) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ int sm[];
  group_body(sm, ids, T, k, E, layer, resid, stage, slots, staging, blob_bytes, nslots, nstaging, num_groups, grp_expert, grp_off,
             grp_slot, grp_src, grp_blob, ent_tok, ent_pos, stats, err, W, hmax, maxTk, skip_rank, heat_row);
}

// Top-k of every token (G warps per token) and then the grouping, in one CTA:
// for decode windows, where each would otherwise be a launch of its own.
template <int KP1>
__global__ void __launch_bounds__(1024) k_topk_group(int G, const float* __restrict__ logits, float* __restrict__ topk_w,
                                                     int32_t* __restrict__ ids, int T, int k, int E, int layer,
                                                     const int32_t* __restrict__ resid, const int32_t* __restrict__ stage,
                                                     const uint8_t* slots, const uint8_t* staging, size_t blob_bytes, int nslots,
                                                     int nstaging, int32_t* __restrict__ num_groups,
                                                     int32_t* __restrict__ grp_expert, int32_t* __restrict__ grp_off,
                                                     int32_t* __restrict__ grp_slot, int32_t* __restrict__ grp_src,
                                                     const uint8_t** __restrict__ grp_blob, int32_t* __restrict__ ent_tok,
                                                     int32_t* __restrict__ ent_pos, unsigned long long* stats, int32_t* err, int W,
                                                     float* __restrict__ hmax, int maxTk, int skip_rank,
                                                     float* __restrict__ heat_row) {
  // the layer's residency, staging and heat rows do not depend on the previous
  // kernel: they travel to L2 while it finishes
  {
    const int lines = (E + 31) / 32, i = threadIdx.x;
    if (resid && i < lines) prefetch_l2(resid + size_t(layer) * E + 32 * i);
    else if (stage && i >= 32 && i - 32 < lines) prefetch_l2(stage + size_t(layer) * E + 32 * (i - 32));
    else if (heat_row && i >= 64 && i - 64 < lines) prefetch_l2(heat_row + 32 * (i - 64));
  }
  pdl_wait();
  extern __shared__ int sm[];
  __shared__ unsigned long long cand[32 * 128];  // per token: G*k <= 128 candidates
  topk_tokens_cta<KP1>(logits, T, E, k, G, ids, topk_w, err, cand);
  pdl_trigger();    // the expert kernels launch while the groups are built
  __syncthreads();  // the ids written above are read by other threads of the CTA
  group_body(sm, ids, T, k, E, layer, resid, stage, slots, staging, blob_bytes, nslots, nstaging, num_groups, grp_expert, grp_off,
             grp_slot, grp_src, grp_blob, ent_tok, ent_pos, stats, err, W, hmax, maxTk, skip_rank, heat_row);
}

// ------------------------------------------------------------------
// Long windows (prefill chunks): the same grouping in three passes over tiles
// of kGrpTok tokens.  (1) each CTA counts its tile's entries per expert; (2)
// one CTA turns the counts into, per expert, the entries before each tile and
// the group offsets, and resolves the groups as above; (3) each CTA places its
// tile's entries: group offset + entries of earlier tiles + the popcount of
// the tile's token bitmap below the token (ascending tokens, as above).
constexpr int kGrpTok = 256;

// A tile's count of an expert (at most kGrpTok) in the low 24 bits, the lowest
// rank choosing it in the tile (kMaxK when none) above them.
constexpr int kCntBits = 24;
constexpr int kCntMask = (1 << kCntBits) - 1;

__global__ void __launch_bounds__(256) k_group_count(const int32_t* __restrict__ ids, int T, int k, int E,
                                                     int32_t* __restrict__ cnt, int32_t* err) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ int sc[];  // [E] counts, then [E] lowest ranks
  int* smin = sc + E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) { sc[e] = 0; smin[e] = kMaxK; }
  __syncthreads();
  const int t0 = blockIdx.x * kGrpTok, t1 = min(T, t0 + kGrpTok);
  bool bad = false;
  for (int i = t0 * k + threadIdx.x; i < t1 * k; i += blockDim.x) {
    const int e = ids[i];
    if (e < 0 || e >= E) { bad = true; continue; }
    atomicAdd(&sc[e], 1);
    atomicMin(&smin[e], i % k);
  }
  if (bad) set_error(err, MOE_ERANGE);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[size_t(blockIdx.x) * E + e] = sc[e] | (smin[e] << kCntBits);
}

__global__ void __launch_bounds__(1024) k_group_scan(int ntile, int T, int k, int E, int layer,
                                                     const int32_t* __restrict__ resid, const int32_t* __restrict__ stage,
                                                     const uint8_t* slots, const uint8_t* staging, size_t blob_bytes,
                                                     int nslots, int nstaging, int32_t* __restrict__ cnt,
                                                     int32_t* __restrict__ eoff, int32_t* __restrict__ num_groups,
                                                     int32_t* __restrict__ grp_expert, int32_t* __restrict__ grp_off,
                                                     int32_t* __restrict__ grp_slot, int32_t* __restrict__ grp_src,
                                                     const uint8_t** __restrict__ grp_blob, unsigned long long* stats,
                                                     int32_t* err, float* __restrict__ hmax, int maxTk, int skip_rank,
                                                     float* __restrict__ heat_row) {
  pdl_trigger();
  pdl_wait();
  __shared__ int warp_sums[32];
  __shared__ int s_hit, s_stg, s_miss, s_skip;
  if (threadIdx.x == 0) { s_hit = 0; s_stg = 0; s_miss = 0; s_skip = 0; }
  const int n = T * k;
  if (hmax) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) hmax[i] = 0.f;
    for (int i = threadIdx.x; i < T; i += blockDim.x) hmax[maxTk + i] = 0.f;
  }
  // per expert: entries before each tile (in place), the total and the lowest
  // rank; loads eight tiles at a time
  const int e = threadIdx.x;
  int total = 0, low = kMaxK;
  if (e < E) {
    for (int c0 = 0; c0 < ntile; c0 += 8) {
      int v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = c0 + j < ntile ? cnt[size_t(c0 + j) * E + e] : 0;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (c0 + j < ntile) {
          cnt[size_t(c0 + j) * E + e] = total;
          total += v[j] & kCntMask;
          low = min(low, v[j] >> kCntBits);
        }
    }
  }
  if (heat_row && total > 0) heat_row[e] = __fadd_rn(heat_row[e], float(total));  // as the heat-update kernel
  __syncthreads();
  int total_entries, total_groups;
  const int ex_c = block_excl_scan(total, warp_sums, total_entries);
  const int ex_g = block_excl_scan(total > 0 ? 1 : 0, warp_sums, total_groups);
  if (e < E) eoff[e] = ex_c;
  if (e < E && total > 0)
    resolve_group(ex_g, e, ex_c, layer, E, resid, stage, slots, staging, blob_bytes, nslots, nstaging, grp_expert,
                  grp_off, grp_slot, grp_src, grp_blob, err, &s_hit, &s_stg, &s_miss,
                  skip_rank > 0 && low >= skip_rank, &s_skip);
  __syncthreads();
  if (threadIdx.x == 0) {
    *num_groups = total_groups;
    grp_off[total_groups] = total_entries;
    if (stats) add_stats(stats + size_t(layer) * kStats, total_groups, s_hit, s_stg, s_miss, s_skip);
  }
}

__global__ void __launch_bounds__(256) k_group_place(const int32_t* __restrict__ ids, int T, int k, int E,
                                                     const int32_t* __restrict__ cnt, const int32_t* __restrict__ eoff,
                                                     int32_t* __restrict__ ent_tok, int32_t* __restrict__ ent_pos,
                                                     int32_t* err) {
  pdl_trigger();
  pdl_wait();
  constexpr int W = kGrpTok / 32;
  extern __shared__ uint32_t bits[];  // [E][W] tokens of this tile that chose each expert
  for (int i = threadIdx.x; i < E * W; i += blockDim.x) bits[i] = 0u;
  __syncthreads();
  const int t0 = blockIdx.x * kGrpTok, t1 = min(T, t0 + kGrpTok);
  for (int i = t0 * k + threadIdx.x; i < t1 * k; i += blockDim.x) {
    const int ex = ids[i];
    if (ex < 0 || ex >= E) continue;
    const int lt = i / k - t0;
    const uint32_t old = atomicOr(&bits[ex * W + (lt >> 5)], 1u << (lt & 31));
    if (old & (1u << (lt & 31))) set_error(err, MOE_ERANGE);  // an expert chosen twice by one token
  }
  __syncthreads();
  const int32_t* before = cnt + size_t(blockIdx.x) * E;
  for (int i = t0 * k + threadIdx.x; i < t1 * k; i += blockDim.x) {
    const int ex = ids[i];
    if (ex < 0 || ex >= E) continue;
    const int t = i / k, lt = t - t0, wd = lt >> 5;
    const uint32_t* row = bits + ex * W;
    int rank = __popc(row[wd] & ((1u << (lt & 31)) - 1u));
#pragma unroll
    for (int w = 0; w < W; ++w)
      if (w < wd) rank += __popc(row[w]);
    const int pos = eoff[ex] + before[ex] + rank;
    ent_tok[pos] = t;
    ent_pos[pos] = i;
  }
}

int launch_group(const int32_t* ids, int T, int k, int E, int layer, moe_cache* c, moe_ws* ws, cudaStream_t s,
                 bool lookup) {
  const int32_t* resid = c && lookup ? c->resid : nullptr;
  const int32_t* stage = c && lookup ? c->stage : nullptr;
  const int skip_rank = lookup ? ws->tail_skip : 0;
  float* heat_row = c && ws->fused_heat ? c->heat + size_t(layer) * E : nullptr;
  if (E > 1024 || E <= 0) return MOE_EINVAL;
  if (T * k > 4096 && ws->grp_scratch) {
    const int ntile = (T + kGrpTok - 1) / kGrpTok;
    int32_t* cnt = ws->grp_scratch;              // [ntile][E]
    int32_t* eoff = cnt + size_t(ntile) * E;     // [E]
    const size_t smem3 = size_t(E) * (kGrpTok / 32) * 4;
    static bool attr3 = false;
    if (!attr3) {
      if (cudaFuncSetAttribute(k_group_place, cudaFuncAttributeMaxDynamicSharedMemorySize, 128 * 1024) != cudaSuccess)
        return MOE_ECUDA;
      attr3 = true;
    }
    if (launch_pdl(k_group_count, dim3(ntile), dim3(256), size_t(2 * E) * 4, s, ids, T, k, E, cnt, ws->error) !=
        cudaSuccess)
      return MOE_ECUDA;
    if (launch_pdl(k_group_scan, dim3(1), dim3(1024), 0, s, ntile, T, k, E, layer, resid, stage, c ? c->slots : nullptr, c ? c->staging : nullptr, c ? c->blob_bytes : 0,
                   c ? c->nslots : 0, c ? c->nstaging : 0, cnt, eoff, ws->num_groups, ws->grp_expert, ws->grp_off,
                   ws->grp_slot, ws->grp_src, ws->grp_blob, c ? c->stats : nullptr, ws->error, ws->hmax,
                   ws->maxT * ws->s.k, skip_rank, heat_row) != cudaSuccess)
      return MOE_ECUDA;
    if (launch_pdl(k_group_place, dim3(ntile), dim3(256), smem3, s, ids, T, k, E, cnt, eoff, ws->ent_tok,
                   ws->ent_pos, ws->error) != cudaSuccess)
      return MOE_ECUDA;
    return MOE_OK;
  }
  // bitmap words per expert: as many as fit 64 KB, at most 32 (1024 tokens per chunk)
  int W = 16384 / E;
  if (W > 32) W = 32;
  if (W < 1) W = 1;
  const int needW = (T + 31) / 32;
  if (W > needW) W = needW > 0 ? needW : 1;
  size_t smem = size_t(4 * E) * 4 + size_t(E) * W * 4;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(k_group, cudaFuncAttributeMaxDynamicSharedMemorySize, 100 * 1024) != cudaSuccess)
      return MOE_ECUDA;
    attr_set = true;
  }
  const cudaError_t rc = launch_pdl(k_group, dim3(1), dim3(1024), smem, s, ids, T, k, E, layer, resid, stage,
                                c ? c->slots : nullptr, c ? c->staging : nullptr, c ? c->blob_bytes : 0,
                                c ? c->nslots : 0, c ? c->nstaging : 0, ws->num_groups, ws->grp_expert, ws->grp_off,
                                ws->grp_slot, ws->grp_src, ws->grp_blob, ws->ent_tok, ws->ent_pos,
                                c ? c->stats : nullptr, ws->error, W, ws->hmax, ws->maxT * ws->s.k, skip_rank,
                                heat_row);
  if (rc != cudaSuccess) return MOE_ECUDA;
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

}  // namespace moe

namespace moe {

// Top-k and grouping in one launch for windows of at most 32 tokens; the same
// results as launch_topk followed by launch_group.  kNotFused when the window
// is larger (the caller then launches them apart).
int launch_topk_group(const float* logits, int T, int k, int E, int layer, moe_cache* c, moe_ws* ws, cudaStream_t s) {
  if (T > 32 || T * k > 4096 || E > 1024 || E <= 0) return kNotFused;
  int W = 16384 / E;  // bitmap words per expert, as launch_group chooses them
  if (W > 32) W = 32;
  if (W < 1) W = 1;
  const int needW = (T + 31) / 32;
  if (W > needW) W = needW > 0 ? needW : 1;
  const size_t smem = size_t(4 * E) * 4 + size_t(E) * W * 4;
  // G warps per token: a power of two with T*G <= 32 and G*k <= 128
  int Tp = 1;
  while (Tp < T) Tp <<= 1;
  int G = 32 / Tp;
  while (G > 1 && G * k > 128) G >>= 1;
  const int per = ((E + G - 1) / G + 31) / 32;  // logits per lane of a warp's slice
  // one shared-memory opt-in per instantiation: the instantiations share one
  // function-pointer type, so a flag in this lambda would be set by the first alone
  static bool attr[6] = {false, false, false, false, false, false};
  auto args = [&](auto kern, int which) {
    if (!attr[which]) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 100 * 1024) != cudaSuccess)
        return cudaErrorInvalidValue;
      attr[which] = true;
    }
    return launch_pdl(kern, dim3(1), dim3(1024), smem, s, G, logits, ws->topk_w, ws->topk_ids, T, k, E, layer,
                      c ? c->resid : nullptr, c ? c->stage : nullptr, c ? c->slots : nullptr,
                      c ? c->staging : nullptr, c ? c->blob_bytes : 0, c ? c->nslots : 0, c ? c->nstaging : 0,
                      ws->num_groups, ws->grp_expert, ws->grp_off, ws->grp_slot, ws->grp_src, ws->grp_blob,
                      ws->ent_tok, ws->ent_pos, c ? c->stats : nullptr, ws->error, W, ws->hmax, ws->maxT * ws->s.k,
                      c ? ws->tail_skip : 0, c && ws->fused_heat ? c->heat + size_t(layer) * E : nullptr);
  };
  cudaError_t rc;
  if (per <= 1) rc = args(k_topk_group<1>, 0);
  else if (per <= 2) rc = args(k_topk_group<2>, 1);
  else if (per <= 4) rc = args(k_topk_group<4>, 2);
  else if (per <= 8) rc = args(k_topk_group<8>, 3);
  else if (per <= 16) rc = args(k_topk_group<16>, 4);
  else rc = args(k_topk_group<32>, 5);
  return rc == cudaSuccess ? MOE_OK : MOE_ECUDA;
}

}  // namespace moe
