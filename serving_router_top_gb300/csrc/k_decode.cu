// The decode forward of one MoE layer in a single cooperative kernel.
//
// Strata expert paths: "显存里缓存的是什么？" (the router picks each token's
// experts and merge weights), "路由以后，专家怎样分工？" (repeated experts of a
// window form one group with input and output positions; outputs are weighted,
// summed, and the gated shared expert is added), "哪些专家能长期留在显存？"
// (the residency table maps (layer, expert) to a slot), "CPU 怎样把剩下的专家
// 算完？" (gate/up, the activation, then the down projection).
//
// A decode window of a few tokens touches tens of experts but moves only a few
// tens of megabytes, so a chain of dependent launches spends more time between
// and inside the prologues of its kernels than streaming weights.  Here one CTA
// per SM runs every step, the CTAs meeting at three grid barriers:
//
//   A  router logits and the shared-gate logit: CTA c owns rows c, c + ncta, ...
//      (row E is the gate vector), each row cut into 512-element slices, one
//      slice per warp, fp32 sums of exact bf16 products; the CTA meanwhile
//      prefetches its slice of the shared expert's blob into L2 and stages x,
//      then x as f16 times a per-token power of two (exact for bf16 values).
//   -- grid barrier --
//   B  every CTA reads all T x E logits and runs the same top-k (a threshold
//      from the 32-expert chunk maxima, then ranks by counting) and the same
//      grouping on them, so every CTA holds the same groups without another
//      barrier; CTA 0 writes them, with the top-k, lookups, statistics and the
//      heat update, to the workspace.  As soon as the top-k's candidates are
//      known (a superset of the selections), CTA c requests its share of their
//      gate/up bytes into L2, so the stream from HBM starts before the grouping.
//   C  gate/up: tasks are (group, 16-row block of I), CTA c owns a contiguous
//      range of them, and the (task, 256-column chunk) units go round-robin to
//      the 16 warps, two units in flight per warp in registers (the first two
//      requested right after grouping); mma.sync m16n8k16 f16 -> f32 with the
//      weights dequantised exactly into f16 (E2M1 code x E4M3 scale) as A and up
//      to 8 of the group's token rows as B; partial tiles are summed in chunk
//      order and the epilogue writes h = SiLU(gs_g g) * gs_u u (fp32) and max|h|
//      per row.  One lane meanwhile issues bulk L2 prefetches of the CTA's later
//      gate/up weights and of all its down weights.
//   -- grid barrier --
//   D  down: tasks are (group, 16-row block of H), CTA c owns a contiguous
//      range; the h rows of its groups are staged once as f16 times a per-row
//      power of two (exact to 11 bits), the units run as in C (three in flight
//      per warp, from L2), each task's chunks summed in order into o (by output
//      position).
//   -- grid barrier --
//   combine: y = sum_r w[t,r] o[t,r] + sigmoid(gl_t) s_t in rank order with the
//      shared term last, each CTA a slice of the T x H outputs -- deterministic,
//      no atomics.
//
// The first two barriers are split: a CTA arrives, does work that no other CTA's
// results feed (x into f16; the first down units' weight loads), then waits.
// Every wait is bounded: the grid barriers give up after the workspace's wait limit,
// record MOE_ETIMEOUT, and the CTAs skip the remaining phases.
#include "dequant.cuh"
#include "topk.cuh"

namespace moe {
namespace dec {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kGuDepth = 2;  // gate/up units in flight per warp (in registers)
constexpr int kChunk = 256;        // columns per unit: a lane's 64 columns, one 32-byte load per row
constexpr int kMaxT = 16;          // tokens (two 8-row tiles of the MMA's N)
constexpr int kXVec = (kMaxT * 2048 / 8 + kThreads - 1) / kThreads;  // 16-byte pieces of x per thread, at most
constexpr int kEVec = (1024 + kThreads - 1) / kThreads;          // residency entries per thread, at most
constexpr int kMaxEnt = 256;       // T * k
constexpr int kMaxGroups = kMaxEnt + 1;
constexpr int kSlice = 512;        // router row elements per warp pair
constexpr int kMaxPairs = 32;      // router slices per CTA at most (each warp takes every kWarps-th)
constexpr int kPadH = 32;          // f16 elements after each activation row: a row stride of 64 mod 128 bytes
constexpr int kMaxUnits = 64;      // gate/up partial tiles held per round (8 floats per lane)
constexpr int kMaxUnitsD = 128;    // down partial tiles held per round (4 floats per lane)

struct Args {
  const uint16_t* x;         // bf16 [T, H]
  const uint16_t* w_router;  // bf16 [E, H]
  const float* bias;         // [E] or null
  const uint16_t* w_sg;      // bf16 [H] or null
  const uint8_t* shared_blob;
  int T, H, I, E, k, layer, has_shared;
  DevBlobLayout lay;
  // the cache
  const int32_t* resid;
  const int32_t* stage;
  const uint8_t* slots;
  const uint8_t* staging;
  size_t blob_bytes, shared_bytes;
  int nslots, nstaging, tail_skip;
  unsigned long long* stats;
  float* heat_row;
  // the workspace
  float* logits;
  float* gate_logit;
  int32_t* topk_ids;
  float* topk_w;
  int32_t* num_groups;
  int32_t* grp_expert;
  int32_t* grp_off;
  int32_t* grp_slot;
  int32_t* grp_src;
  const uint8_t** grp_blob;
  int32_t* ent_tok;
  int32_t* ent_pos;
  float* h;
  float* hmax;
  float* o;                  // [(maxTk + maxT), H] expert outputs by position, then the shared rows
  int Imax, maxTk;
  void* y;
  int y_fp32;
  int32_t* err;
  unsigned long long* bar;   // grid-barrier arrivals (a multiple of the grid between launches)
  unsigned bar_extra;        // arrivals a barrier waits for beyond the grid (0; a test hook)
  unsigned long long wait_ns;
  // shared-memory carve (byte offsets); capc: top-k candidates per token; hrows: h rows
  // the down phase stages at once
  int o_x16, o_xs, o_lg, o_cb, o_cand, o_sel, o_pr, o_part, o_red, o_h16, o_small;
  int capc, hrows;
};

// Small tables, at the end of shared memory.
struct Small {
  int32_t ids[kMaxEnt];
  float w[kMaxEnt];
  uint32_t key[kMaxEnt];
  uint32_t srt[kMaxEnt];
  int32_t ent_tok[kMaxEnt];
  int32_t ent_pos[kMaxEnt];
  unsigned long long tau[kMaxT];  // top-k per token: threshold, best entry, candidates
  unsigned long long top[kMaxT];
  int32_t ncand[kMaxT];
  uint32_t cbits[32];  // candidate experts of the window (bit e)
  int32_t gexp[kMaxGroups];
  int32_t goff[kMaxGroups + 1];
  const uint8_t* gblob[kMaxGroups];
  float xinv[kMaxT];
  float bias_r[kMaxPairs];  // the router bias of the CTA's rows
  float gl[kMaxT];
  float hs_inv[kMaxEnt + kMaxT];
  int32_t resid[1024];  // the layer's residency and staging rows
  int32_t stage[1024];
  __align__(16) float gs[kMaxGroups][4];  // each group's global scales (gate, up, down) and a pad
  unsigned long long bar_base;  // the grid-barrier counter at the CTA's start, rounded down to the grid
  unsigned long long bar_idx;   // barriers passed
  int ok, cnt[4];
};

__device__ __forceinline__ unsigned long long ld_acquire_gpu(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void red_add_release_gpu(unsigned long long* p, unsigned long long v) {
  asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_gpu(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Grid barrier on a monotonic arrival counter: every barrier of every launch adds one
// arrival per CTA, so between launches the counter is a multiple of the grid.  Each CTA
// reads it once at its start (other CTAs may have arrived at the first barrier by then,
// but fewer than the grid) and rounds down to that multiple, its base; barrier i is
// complete when the counter reaches base + i * grid (+ the test hook's phantom arrivals,
// which never come).  An arrival is a release add whose result nobody waits for; then
// acquire loads until the count is reached -- at most wait_ns, after which the wait
// records MOE_ETIMEOUT and every later phase of the CTA is skipped (the host resets the
// counter with the error word).  (A two-level tree of counters was measured slower: its
// last arrival pays two dependent atomic round trips; an acquire-release add that returns
// the count costs every CTA a round trip before it starts polling; so were four staggered
// pollers per CTA.)  grid_arrive and grid_wait are the two halves: between them a CTA may
// do work that reads nothing another CTA writes before the barrier.  grid_wait returns
// whether the barrier was passed.  Every thread of the CTA calls both.
__device__ void grid_arrive(const Args& a, Small& sm) {
  __syncthreads();
  if (threadIdx.x == 0 && sm.ok) red_add_release_gpu(a.bar, 1ull);
}
__device__ bool grid_wait(const Args& a, Small& sm) {
  if (threadIdx.x == 0) {
    int ok = sm.ok;
    if (ok) {
      const unsigned long long target = sm.bar_base + (++sm.bar_idx) * gridDim.x + a.bar_extra;
      const unsigned long long t0 = globaltimer_ns();
      while (ld_acquire_gpu(a.bar) < target) {
        if (globaltimer_ns() - t0 > a.wait_ns) {
          set_error(a.err, MOE_ETIMEOUT);
          ok = 0;
          break;
        }
      }
    }
    sm.ok = ok;
  }
  __syncthreads();
  return *reinterpret_cast<volatile int*>(&sm.ok) != 0;
}
__device__ bool grid_barrier(const Args& a, Small& sm) {
  grid_arrive(a, sm);
  return grid_wait(a, sm);
}

// Column c of an activation row is stored where lane (., t4) finds its eight
// columns 8q..8q+7 of each 256-column chunk as one 16-byte load: chunk-major,
// then (q, t4), then the eight values.  Four lanes of a row read 64
// consecutive bytes; with the row stride 64 mod 128 bytes, two rows' quarter
// warps touch disjoint banks.
__device__ __forceinline__ int perm_col(int c) {
  const int cc = c & (kChunk - 1);
  return (c - cc) + (((cc & 63) >> 3) * 4 + (cc >> 6)) * 8 + (c & 7);
}

// L2 eviction policies: the router weights (read by every step) kept, the expert weights
// (read once per step) first to go
__device__ __forceinline__ unsigned long long policy_evict_last() {
  unsigned long long p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ unsigned long long policy_evict_first() {
  unsigned long long p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint4 ld_keep16(const void* p, unsigned long long pol) {
  uint4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}
__device__ __forceinline__ void ld_once32(const void* p, uint32_t (&r)[8], unsigned long long pol) {
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "l"(p), "l"(pol));
}
__device__ __forceinline__ uint32_t ld_once_u32(const void* p, unsigned long long pol) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.u32 %0, [%1], %2;" : "=r"(v) : "l"(p), "l"(pol));
  return v;
}

// One unit as loaded by a lane: rows g8 and g8 + 8 of each matrix, the lane's
// 64 columns (32 code bytes per row) and their four block scales.
template <int NM>
struct UnitRegs {
  uint32_t c[NM][2][8];
  uint32_t s[NM][2];
};

template <int NM>
__device__ __forceinline__ void load_unit(const uint8_t* blob, const DevBlobLayout& lay, int mat0, int K, int row,
                                          int ch, int t4, UnitRegs<NM>& R) {
#pragma unroll
  for (int m = 0; m < NM; ++m) {
    const uint8_t* cp = blob + lay.code_off[mat0 + m] + size_t(row) * (K / 2) + ch * 128 + 32 * t4;
    const unsigned long long pol = policy_evict_first();
    ld_once32(cp, R.c[m][0], pol);
    ld_once32(cp + size_t(8) * (K / 2), R.c[m][1], pol);
    const uint8_t* sp = blob + lay.scale_off[mat0 + m] + size_t(row) * (K / 16) + ch * 16 + 4 * t4;
    R.s[m][0] = ld_once_u32(sp, pol);
    R.s[m][1] = ld_once_u32(sp + size_t(8) * (K / 16), pol);
  }
}

// The same unit from a copy of 16 weight rows in shared memory: matrix m's code rows at
// base + m * mstride (K / 2 bytes each), its scale rows at base + soff + m * K (K / 16 each).
template <int NM>
__device__ __forceinline__ void load_unit_smem(const uint8_t* base, int mstride, int soff, int K, int row, int ch,
                                               int t4, UnitRegs<NM>& R) {
#pragma unroll
  for (int m = 0; m < NM; ++m) {
    const uint8_t* cp = base + m * mstride + row * (K / 2) + ch * 128 + 32 * t4;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const uint4 lo = *reinterpret_cast<const uint4*>(cp + r * 8 * (K / 2));
      const uint4 hi = *reinterpret_cast<const uint4*>(cp + r * 8 * (K / 2) + 16);
      R.c[m][r][0] = lo.x; R.c[m][r][1] = lo.y; R.c[m][r][2] = lo.z; R.c[m][r][3] = lo.w;
      R.c[m][r][4] = hi.x; R.c[m][r][5] = hi.y; R.c[m][r][6] = hi.z; R.c[m][r][7] = hi.w;
    }
    const uint8_t* sp = base + soff + m * K + row * (K / 16) + ch * 16 + 4 * t4;
    R.s[m][0] = *reinterpret_cast<const uint32_t*>(sp);
    R.s[m][1] = *reinterpret_cast<const uint32_t*>(sp + 8 * (K / 16));
  }
}

// The lane's 64 columns of chunk ch: dq(W rows) . B.  NT = 1: one tile of 8 B rows
// (brow0 = the lane's row), acc[m][0] and acc[m][1] the even and odd MMAs of each code
// word (two accumulation chains, summed by the caller).  NT = 2: two tiles (brow0 for
// rows 0..7, brow1 for rows 8..15 of the group), acc[m][tile]; the dequantised A
// fragments serve both.  A null B row reads zeros.
template <int NM, int NT>
__device__ __forceinline__ void mma_unit(const UnitRegs<NM>& R, const __half* brow0, const __half* brow1, int ch,
                                         int t4, float (&acc)[NM][2][4]) {
  const uint4* xp0 = brow0 ? reinterpret_cast<const uint4*>(brow0 + ch * kChunk) + t4 : nullptr;
  const uint4* xp1 = (NT == 2 && brow1) ? reinterpret_cast<const uint4*>(brow1 + ch * kChunk) + t4 : nullptr;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const uint4 xq = xp0 ? xp0[q * 4] : make_uint4(0u, 0u, 0u, 0u);
    uint4 xr = make_uint4(0u, 0u, 0u, 0u);
    if (NT == 2 && xp1) xr = xp1[q * 4];
    const int blk = q >> 1;
#pragma unroll
    for (int m = 0; m < NM; ++m) {
      const uint32_t sa = scale_pair((R.s[m][0] >> (8 * blk)) & 0xffu);
      const uint32_t sb = scale_pair((R.s[m][1] >> (8 * blk)) & 0xffu);
      const uint32_t w0 = R.c[m][0][q], w1 = R.c[m][1][q];
      uint32_t a0, a1, a2, a3;
      e2m1_pair2(w0, a0, a2);
      e2m1_pair2(w1, a1, a3);
      const uint32_t p0 = hmul2(a0, sa), p1 = hmul2(a1, sb), p2 = hmul2(a2, sa), p3 = hmul2(a3, sb);
      mma16816(acc[m][0], p0, p1, p2, p3, xq.x, xq.y);
      if (NT == 2) mma16816(acc[m][1], p0, p1, p2, p3, xr.x, xr.y);
      e2m1_pair2(w0 >> 16, a0, a2);
      e2m1_pair2(w1 >> 16, a1, a3);
      const uint32_t r0 = hmul2(a0, sa), r1 = hmul2(a1, sb), r2 = hmul2(a2, sa), r3 = hmul2(a3, sb);
      mma16816(acc[m][NT == 2 ? 0 : 1], r0, r1, r2, r3, xq.z, xq.w);
      if (NT == 2) mma16816(acc[m][1], r0, r1, r2, r3, xr.z, xr.w);
    }
  }
}

// An entry's place in the top-k order: the order-preserving key of its logit above, the
// complement of its id below -- a larger value is a better entry, equal logits going to the
// lower id (the order of the top-k kernel).
__device__ __forceinline__ unsigned long long rank_key(float x, int e) {
  return (static_cast<unsigned long long>(ordered_key(x)) << 32) | (0xffffffffu - unsigned(e));
}

// Top-k of the T tokens by the whole CTA from the logits in shared memory (lg [T, E]):
//   1. the best entry of each 32-expert chunk of a token (two warp reductions);
//   2. tau_t, the k-th best of the token's chunk bests (0 when it has fewer than k
//      chunks): k entries reach tau_t, so each of the token's k best does too;
//   3. the entries that reach tau_t -- those of the k chunks whose best does, at most
//      min(E, 32 k), usually a few more than k -- are compacted (their experts, over all
//      tokens, also as bits of sm.cbits), then on_cands runs;
//   4. each candidate takes as its rank the number of candidates above it; rank r < k is
//      the token's selection r, whose term p_r = exp(l_r - l_0) is taken at once (l_0,
//      the token's best entry, is its best chunk best).
// No step is a chain of warp-wide selections, which a decode step cannot afford (nor one
// warp per token: its chain of dependent shared-memory and shuffle steps was measured
// slower than the CTA-wide steps and their barriers); a warp takes its items of steps 1 and
// 3 four at a time, their loads, reductions and atomics side by side.  Ids and weights equal the top-k
// kernel's: the same order, and w_r = p_r / sum_j p_j summed in rank order.  NaN logits
// rank as -inf and record MOE_ENAN.  Leaves key[i] = id << 16 | i for the grouping.  Every
// thread of the CTA calls this; it holds four __syncthreads and ends without one.
template <typename OnCands>
__device__ void topk_ranked(const float* __restrict__ lg, int T, int E, int k, Small& sm, int32_t* err,
                            unsigned long long* __restrict__ cbest, unsigned long long* __restrict__ cand, int capc,
                            unsigned long long* __restrict__ sel, float* __restrict__ pr, OnCands on_cands) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NCH = (E + 31) >> 5;
  bool nan_seen = false;
  // a warp's items four at a time: every load first, then the reductions
  for (int it0 = warp; it0 < T * NCH; it0 += 4 * kWarps) {
    unsigned long long ck[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int it = it0 + q * kWarps, t = it / NCH, e = (it - t * NCH) * 32 + lane;
      ck[q] = 0ull;
      if (it < T * NCH && e < E) {
        float x = lg[t * E + e];
        if (x != x) {
          nan_seen = true;
          x = -INFINITY;
        }
        ck[q] = rank_key(x, e);
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int it = it0 + q * kWarps;
      if (it < T * NCH) {
        const unsigned hi = __reduce_max_sync(0xffffffffu, unsigned(ck[q] >> 32));
        const unsigned lo = __reduce_max_sync(0xffffffffu, unsigned(ck[q] >> 32) == hi ? unsigned(ck[q]) : 0u);
        if (lane == 0) cbest[it] = (static_cast<unsigned long long>(hi) << 32) | lo;
      }
    }
  }
  if (nan_seen) set_error(err, MOE_ENAN);
  if (tid < T) sm.ncand[tid] = 0;
  __syncthreads();
  if (warp < T) {
    const unsigned long long* cb = cbest + warp * NCH;
    const unsigned long long mine = lane < NCH ? cb[lane] : 0ull;
    int r = 0;
    for (int c = 0; c < NCH; ++c) r += cb[c] > mine ? 1 : 0;
    if (NCH < k) {
      if (lane == 0) sm.tau[warp] = 0ull;
    } else if (lane < NCH && r == k - 1) {
      sm.tau[warp] = mine;
    }
    if (lane < NCH && r == 0) sm.top[warp] = mine;
  }
  __syncthreads();
  // four items at a time again: the loads, the ballots, the four atomics (independent),
  // then the stores
  for (int it0 = warp; it0 < T * NCH; it0 += 4 * kWarps) {
    unsigned long long ck[4];
    unsigned b[4];
    int base[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int it = it0 + q * kWarps, t = it / NCH, e = (it - t * NCH) * 32 + lane;
      ck[q] = 0ull;
      bool take = false;
      if (it < T * NCH && e < E) {
        float x = lg[t * E + e];
        if (x != x) x = -INFINITY;
        ck[q] = rank_key(x, e);
        take = ck[q] >= sm.tau[t];
      }
      b[q] = __ballot_sync(0xffffffffu, take);
    }
    if (lane == 0) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int it = it0 + q * kWarps, t = it / NCH;
        base[q] = 0;
        if (b[q]) {
          base[q] = atomicAdd(&sm.ncand[t], __popc(b[q]));
          atomicOr(&sm.cbits[it - t * NCH], b[q]);  // the candidate experts of all tokens
        }
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int it = it0 + q * kWarps, t = it / NCH;
      const int pos = __shfl_sync(0xffffffffu, base[q], 0) + __popc(b[q] & ((1u << lane) - 1u));
      if ((b[q] >> lane) & 1u) {
        if (pos < capc) cand[t * capc + pos] = ck[q];
        else set_error(err, MOE_ERANGE);  // unreachable: at most min(E, 32 k) entries reach tau
      }
    }
  }
  __syncthreads();
  on_cands();
  {
    const int S = kThreads / T, t = tid / S;
    if (t < T) {
      const int C = min(sm.ncand[t], capc);
      const unsigned long long* cc = cand + t * capc;
      for (int i = tid - t * S; i < C; i += S) {
        const unsigned long long me = cc[i];
        int r = 0;
#pragma unroll 4
        for (int j = 0; j < C; ++j) r += cc[j] > me ? 1 : 0;
        if (r < k) {
          sm.ids[t * k + r] = int(0xffffffffu - unsigned(me));
          pr[t * k + r] = expf(float_of_key(unsigned(me >> 32)) - float_of_key(unsigned(sm.top[t] >> 32)));
        }
      }
    }
  }
  __syncthreads();
  const int n = T * k;
  for (int i = tid; i < n; i += kThreads) {
    const float* p = pr + (i / k) * k;
    float den = 0.f;
    for (int r = 0; r < k; ++r) den += p[r];
    sm.w[i] = pr[i] / den;
    sm.key[i] = (uint32_t(sm.ids[i]) << 16) | uint32_t(i);
  }
}

// TP: T rounded up to a power of two (the router's unrolled token loops); above 8 tokens
// the expert units run two 8-row tiles of B on the same dequantised weights.
template <int TP>
__global__ void __launch_bounds__(kThreads, 1) k_decode_fused(const Args a) {
  constexpr int kNT = TP > 8 ? 2 : 1;  // 8-row tiles of B per unit
  constexpr int kGD = TP > 8 ? 1 : kGuDepth;  // gate/up units in flight per warp (two tiles: registers)
  constexpr int kUnitsGU = kMaxUnits / kNT, kUnitsDN = kMaxUnitsD / kNT;  // partial tiles of one round
  extern __shared__ __align__(128) uint8_t smem[];
  __half* x16 = reinterpret_cast<__half*>(smem + a.o_x16);
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem + a.o_xs);
  float* lg = reinterpret_cast<float*>(smem + a.o_lg);
  unsigned long long* cbest = reinterpret_cast<unsigned long long*>(smem + a.o_cb);
  unsigned long long* cand = reinterpret_cast<unsigned long long*>(smem + a.o_cand);
  unsigned long long* sel = reinterpret_cast<unsigned long long*>(smem + a.o_sel);
  float* pr = reinterpret_cast<float*>(smem + a.o_pr);
  float* part = reinterpret_cast<float*>(smem + a.o_part);
  __half* h16 = reinterpret_cast<__half*>(smem + a.o_h16);
  float* red = reinterpret_cast<float*>(smem + a.o_red);
  Small& sm = *reinterpret_cast<Small*>(smem + a.o_small);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g8 = lane >> 2, t4 = lane & 3;
  const int cta = blockIdx.x, ncta = gridDim.x;
  const int T = a.T, H = a.H, I = a.I, E = a.E, k = a.k;
  const int n = T * k;
  const int XR = H + kPadH, HR = I + kPadH;
  const bool lead = cta == 0;
  int32_t* err = lead ? a.err : nullptr;

  // ================================================================ A: router
  if (tid == 0) {
    sm.ok = 1;
    sm.cnt[0] = sm.cnt[1] = sm.cnt[2] = sm.cnt[3] = 0;
    sm.bar_base = ld_relaxed_gpu(a.bar) / gridDim.x * gridDim.x;  // before this CTA's first arrival
    sm.bar_idx = 0;
  }
  if (tid < 32) sm.cbits[tid] = 0u;
  // this CTA's slice of the shared expert's blob into L2 (its gate/up tasks run in C)
  if (a.has_shared && tid == 0) {
    const size_t slice = ((a.shared_bytes + ncta - 1) / ncta + 15) & ~size_t(15);
    const size_t b0 = size_t(cta) * slice;
    if (b0 < a.shared_bytes) {
      const size_t nb = (a.shared_bytes - b0 < slice ? a.shared_bytes - b0 : slice) & ~size_t(15);
      if (nb) prefetch_bulk_l2(a.shared_blob + b0, uint32_t(nb));
    }
  }
  // router rows of this CTA: row E is the shared gate vector
  const int rows_total = E + (a.w_sg ? 1 : 0);
  const int nrows = cta < rows_total ? (rows_total - 1 - cta) / ncta + 1 : 0;
  const int QS = H / kSlice;
  const int npairs = nrows * QS;
  // the first of the warp's slices into registers now (no kernel writes the router weights);
  // later slices (more than 16 per CTA) are loaded when their turn comes
  auto router_row = [&](int p) {
    const int j = p / QS, q = p - j * QS, row = cta + j * ncta;
    return reinterpret_cast<const uint4*>(row < E ? a.w_router + size_t(row) * H : a.w_sg) + q * (kSlice / 8);
  };
  uint4 wv0 = make_uint4(0u, 0u, 0u, 0u), wv1 = wv0;
  if (warp < npairs) {
    const uint4* wr = router_row(warp);
    wv0 = ld_keep16(wr + lane, policy_evict_last());
    wv1 = ld_keep16(wr + 32 + lane, policy_evict_last());
  }
  // x into shared memory (all loads of a thread in flight together), and the
  // layer's residency and staging rows for the lookups of phase B
  {
    const uint4* src = reinterpret_cast<const uint4*>(a.x);
    uint4* dst = reinterpret_cast<uint4*>(xs);
    const int n16 = T * H / 8;
    uint4 v[kXVec];
#pragma unroll
    for (int j = 0; j < kXVec; ++j) {
      const int i = tid + j * kThreads;
      if (i < n16) v[j] = src[i];
    }
    // the router bias of this CTA's rows, with the other loads (the logits add it at the end)
    const int brow = cta + tid * ncta;
    const float bv = (tid < nrows && brow < E && a.bias) ? __ldg(a.bias + brow) : 0.f;
    int32_t rv[kEVec], sv[kEVec];
#pragma unroll
    for (int j = 0; j < kEVec; ++j) {
      const int e = tid + j * kThreads;
      rv[j] = e < E ? a.resid[size_t(a.layer) * E + e] : -1;
      sv[j] = (e < E && a.stage) ? a.stage[size_t(a.layer) * E + e] : -1;
    }
#pragma unroll
    for (int j = 0; j < kXVec; ++j) {
      const int i = tid + j * kThreads;
      if (i < n16) dst[i] = v[j];
    }
#pragma unroll
    for (int j = 0; j < kEVec; ++j) {
      const int e = tid + j * kThreads;
      if (e < E) {
        sm.resid[e] = rv[j];
        sm.stage[e] = sv[j];
      }
    }
    if (tid < nrows) sm.bias_r[tid] = bv;
  }
  // the expert kernels accumulate max|h| per row with atomicMax from phase C on
  if (lead) {
    for (int i = tid; i < n; i += kThreads) a.hmax[i] = 0.f;
    for (int i = tid; i < T; i += kThreads) a.hmax[a.maxTk + i] = 0.f;
  }
  __syncthreads();
  // per-token power of two, and x as f16 in the permuted layout
  if (warp < T) {
    float m = 0.f;
    for (int i = lane; i < H / 8; i += 32) {
      const uint4 q = reinterpret_cast<const uint4*>(xs + warp * H)[i];
      const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        m = fmaxf(m, fmaxf(fabsf(__uint_as_float(u[j] << 16)), fabsf(__uint_as_float(u[j] & 0xffff0000u))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) sm.xinv[warp] = pow2_scale_for(m);
  }
  // router partial sums: the lane's 16 elements of the slice, each token
#pragma unroll 1
  for (int p = warp; p < npairs; p += kWarps) {
    if (p != warp) {
      const uint4* wr = router_row(p);
      wv0 = ld_keep16(wr + lane, policy_evict_last());
      wv1 = ld_keep16(wr + 32 + lane, policy_evict_last());
    }
    const int q = p % QS;
    float pacc[TP];
#pragma unroll
    for (int t = 0; t < TP; ++t) pacc[t] = 0.f;
#pragma unroll
    for (int hv = 0; hv < 2; ++hv) {
      const uint4 w4 = hv ? wv1 : wv0;
      const uint32_t wu[4] = {w4.x, w4.y, w4.z, w4.w};
      const int c0 = q * kSlice + (hv * 32 + lane) * 8;
#pragma unroll
      for (int t = 0; t < TP; ++t) {
        if (t < T) {
          const uint4 xv = *reinterpret_cast<const uint4*>(xs + t * H + c0);
          const uint32_t xu[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            pacc[t] = fmaf(__uint_as_float(wu[j] << 16), __uint_as_float(xu[j] << 16), pacc[t]);
            pacc[t] = fmaf(__uint_as_float(wu[j] & 0xffff0000u), __uint_as_float(xu[j] & 0xffff0000u), pacc[t]);
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < TP; ++t) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) pacc[t] += __shfl_xor_sync(0xffffffffu, pacc[t], o);
    }
    if (lane < T) {
      float v = pacc[0];
#pragma unroll
      for (int t = 1; t < TP; ++t)
        if (lane == t) v = pacc[t];
      part[p * kMaxT + lane] = v;
    }
  }
  __syncthreads();
  // slices summed in order, plus the bias: the logits of this CTA's rows
  for (int i = tid; i < nrows * T; i += kThreads) {
    const int j = i / T, t = i - j * T, row = cta + j * ncta;
    float v = 0.f;
    for (int q = 0; q < QS; ++q) v += part[(j * QS + q) * kMaxT + t];
    if (row < E)
      a.logits[size_t(t) * E + row] = a.bias ? __fadd_rn(v, sm.bias_r[j]) : v;
    else
      a.gate_logit[t] = v;
  }
  grid_arrive(a, sm);
  // x as f16 times the token's power of two (read by every gate/up unit), eight
  // consecutive columns -- one 16-byte group of the permuted layout -- per item, while the
  // other CTAs arrive
  for (int i = tid; i < T * H / 8; i += kThreads) {
    const int t = (i * 8) / H, c = i * 8 - t * H;
    const uint4 q = reinterpret_cast<const uint4*>(xs)[i];
    const uint32_t u[4] = {q.x, q.y, q.z, q.w};
    const float sc = sm.xinv[t];
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __half2 hh = __floats2half2_rn(__uint_as_float(u[j] << 16) * sc, __uint_as_float(u[j] & 0xffff0000u) * sc);
      o[j] = *reinterpret_cast<uint32_t*>(&hh);
    }
    *reinterpret_cast<uint4*>(x16 + t * XR + perm_col(c)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (!grid_wait(a, sm)) return;

  // ============================================================ B: top-k, groups
  {
    float glv = 0.f;
    if (tid < T && a.has_shared) glv = __ldcg(a.gate_logit + tid);  // in the same round trip
    for (int i0 = 0; i0 < T * E; i0 += 8 * kThreads) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = i0 + tid + j * kThreads;
        if (i < T * E) v[j] = __ldcg(a.logits + i);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = i0 + tid + j * kThreads;
        if (i < T * E) lg[i] = v[j];
      }
    }
    if (tid < T) {
      sm.gl[tid] = glv;
      sm.xinv[tid] = 1.0f / sm.xinv[tid];
    }
  }
  __syncthreads();
  // The candidate experts' gate/up bytes (codes, then scales: two contiguous ranges of each
  // blob) requested into L2 as soon as the candidates are known, before the ranks and the
  // grouping: the candidates hold every selection.  The experts' bytes are taken as one
  // range, expert after expert, of which CTA c requests the c-th share -- a few large
  // requests per CTA -- from the last warp, which the ranks of up to 8 tokens leave idle.
  topk_ranked(lg, T, E, k, sm, err, cbest, cand, a.capc, sel, pr, [&]() {
    if (warp != kWarps - 1) return;
    const uint32_t gu_c = a.lay.code_off[2] - a.lay.code_off[0], gu_s = a.lay.scale_off[2] - a.lay.scale_off[0];
    const size_t per = size_t(gu_c) + gu_s;
    const unsigned word = lane < ((E + 31) >> 5) ? sm.cbits[lane] : 0u;
    const int cnt = __popc(word);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const size_t V = size_t(__shfl_sync(0xffffffffu, incl, 31)) * per;
    const size_t share = ((V + ncta - 1) / ncta + 15) & ~size_t(15);
    const size_t b0 = size_t(cta) * share, b1 = min(V, b0 + share);
    for (size_t x = b0 / per; b0 < b1 && x * per < b1; ++x) {
      const unsigned m = __ballot_sync(0xffffffffu, size_t(incl) > x);
      const int L = __ffs(m) - 1;
      const int nb = int(x) - __shfl_sync(0xffffffffu, incl - cnt, L);
      const unsigned w = __shfl_sync(0xffffffffu, word, L);
      if (lane == 0) {
        const int e = L * 32 + int(__fns(w, 0, nb + 1));
        const int slot = sm.resid[e], st = sm.stage[e];
        const uint8_t* blob = (slot >= 0 && slot < a.nslots) ? a.slots + size_t(slot) * a.blob_bytes
                              : (st >= 0 && st < a.nstaging) ? a.staging + size_t(st) * a.blob_bytes : nullptr;
        const size_t s0 = max(b0, x * per) - x * per, s1 = min(b1, (x + 1) * per) - x * per;
        if (blob && s0 < gu_c) prefetch_bulk_l2(blob + a.lay.code_off[0] + s0, uint32_t(min(s1, size_t(gu_c)) - s0));
        if (blob && s1 > gu_c) {
          const size_t c0 = max(s0, size_t(gu_c)) - gu_c;
          prefetch_bulk_l2(blob + a.lay.scale_off[0] + c0, uint32_t(s1 - gu_c - c0));
        }
      }
    }
  });
  __syncthreads();
  // groups: the n selections sorted by (expert, position); position t*k + r orders like the
  // token.  n <= 256 < the CTA's threads: one entry per thread.
  if (tid < n) {
    const uint32_t kk = sm.key[tid];
    int r = 0;
#pragma unroll 4
    for (int j = 0; j < n; ++j) r += sm.key[j] < kk ? 1 : 0;
    sm.srt[r] = kk;
  }
  __syncthreads();
  // the entries that start a group, as ballots over rounds of 32 that every warp takes
  // (the same masks in every warp); a start's group is the number of starts before it
  int G = 0, before = 0;
  unsigned mine = 0u;
  for (int r0 = 0; r0 < n; r0 += 32) {
    const int j = r0 + lane;
    const bool st = j < n && (j == 0 || (sm.srt[j - 1] >> 16) != (sm.srt[j] >> 16));
    const unsigned m = __ballot_sync(0xffffffffu, st);
    if (r0 < warp * 32) before += __popc(m);
    else if (r0 == warp * 32) mine = m;
    G += __popc(m);
  }
  if (tid < n) {
    const uint32_t kk = sm.srt[tid];
    const int pos = int(kk & 0xffffu);
    sm.ent_pos[tid] = pos;
    sm.ent_tok[tid] = pos / k;
    if ((mine >> lane) & 1u) {
      const int g = before + __popc(mine & ((1u << lane) - 1u));
      sm.gexp[g] = int(kk >> 16);
      sm.goff[g] = tid;
    }
  }
  const int Gt = G + a.has_shared;
  if (tid == 0) sm.goff[G] = n;
  __syncthreads();
  // lookup of each routed group (the same tables in every CTA: the same result)
  for (int g = tid; g < G; g += kThreads) {
    const int e = sm.gexp[g], e0 = sm.goff[g], e1 = (g + 1 < G) ? sm.goff[g + 1] : n;
    int slot = sm.resid[e];
    const int st = sm.stage[e];
    int src = MOE_SRC_MISSING;
    const uint8_t* blob = nullptr;
    if (slot >= 0) {
      if (slot < a.nslots) { src = MOE_SRC_RESIDENT; blob = a.slots + size_t(slot) * a.blob_bytes; }
      else { set_error(err, MOE_ERANGE); slot = -1; }
    }
    bool tail = false;
    if (a.tail_skip > 0 && src != MOE_SRC_RESIDENT) {
      int mr = k;
      for (int i = e0; i < e1; ++i) mr = min(mr, sm.ent_pos[i] % k);
      tail = mr >= a.tail_skip;
    }
    if (tail) {
      src = MOE_SRC_SKIPPED;
      slot = -1;
    } else if (src == MOE_SRC_MISSING) {
      if (st >= 0 && st < a.nstaging) { slot = st; src = MOE_SRC_STAGED; blob = a.staging + size_t(st) * a.blob_bytes; }
      else if (st >= a.nstaging) set_error(err, MOE_ERANGE);
      if (src == MOE_SRC_MISSING) { slot = -1; set_error(err, MOE_EMISSING); }
    }
    sm.gblob[g] = blob;
    if (lead) {
      a.grp_expert[g] = e;
      a.grp_off[g] = e0;
      a.grp_slot[g] = slot;
      a.grp_src[g] = src;
      a.grp_blob[g] = blob;
      atomicAdd(&sm.cnt[src == MOE_SRC_RESIDENT ? 0 : src == MOE_SRC_STAGED ? 1 : src == MOE_SRC_SKIPPED ? 3 : 2], 1);
      // as the heat-update kernel: one rounded add per expert (each is in one group), here a
      // reduction that no thread waits for
      if (a.heat_row) atomicAdd(a.heat_row + e, float(e1 - e0));
    }
  }
  if (a.has_shared && tid == 0) {
    sm.gblob[G] = a.shared_blob;
    sm.goff[G + 1] = n + T;  // the shared expert's entries are the T tokens, after the routed ones
  }
  __syncthreads();
  if (lead) {
    for (int i = tid; i < n; i += kThreads) {
      a.topk_ids[i] = sm.ids[i];
      a.topk_w[i] = sm.w[i];
      a.ent_tok[i] = sm.ent_tok[i];
      a.ent_pos[i] = sm.ent_pos[i];
    }
    if (tid == 0) {
      *a.num_groups = G;
      a.grp_off[G] = n;
      if (a.stats) add_stats(a.stats + size_t(a.layer) * kStats, G, sm.cnt[0], sm.cnt[1], sm.cnt[2], sm.cnt[3]);
    }
  }
  // Work of phases C and D: gate/up tasks (group, 16-row block of I) and down tasks
  // (group, 16-row block of H), each list group-major; CTA c owns a contiguous range of each.
  const int TPG = I / 16, NRB = H / 16;
  const int NT = Gt * TPG, ND = Gt * NRB;
  const int t0 = int((long long)cta * NT / ncta), t1 = int((long long)(cta + 1) * NT / ncta);
  const int d0 = int((long long)cta * ND / ncta), d1 = int((long long)(cta + 1) * ND / ncta);
  const int NCH = H / kChunk, NCD = I / kChunk;
  // H and I are powers of two here: the unit arithmetic of the hot loops in shifts
  const int lNCH = __ffs(NCH) - 1, lTPG = __ffs(TPG) - 1, lNRB = __ffs(NRB) - 1, lNCD = __ffs(NCD) - 1;

  // ============================================================ C: gate/up
  const int U = (t1 - t0) * NCH;
  int r0 = 0, nu = min(kUnitsGU, U);
  auto unit_at = [&](int u, int& gi, int& tb, int& ch) {
    const int task = t0 + (u >> lNCH);
    ch = u & (NCH - 1);
    gi = task >> lTPG;
    tb = task & (TPG - 1);
  };
  auto load = [&](int u, UnitRegs<2>& R) {
    if (u >= r0 + nu) return;
    int gi, tb, ch;
    unit_at(u, gi, tb, ch);
    const uint8_t* blob = sm.gblob[gi];
    if (blob) load_unit<2>(blob, a.lay, 0, H, tb * 16 + g8, ch, t4, R);
  };
  auto run = [&](int u, const UnitRegs<2>& R) {
    if (u >= r0 + nu) return;
    int gi, tb, ch;
    unit_at(u, gi, tb, ch);
    const int e0 = sm.goff[gi], nv = sm.goff[gi + 1] - e0;
    float acc[2][2][4];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[m][q >> 2][q & 3] = 0.f;
    if (sm.gblob[gi]) {
      const __half* b0 = nullptr;
      const __half* b1 = nullptr;
      if (g8 < nv) b0 = x16 + size_t(gi == G ? g8 : sm.ent_tok[e0 + g8]) * XR;
      if (kNT == 2 && g8 + 8 < nv) b1 = x16 + size_t(gi == G ? g8 + 8 : sm.ent_tok[e0 + g8 + 8]) * XR;
      mma_unit<2, kNT>(R, b0, b1, ch, t4, acc);
    }
    float4* dst = reinterpret_cast<float4*>(red + (size_t(u - r0) * 32 + lane) * 8 * kNT);
    if (kNT == 1) {
      dst[0] = make_float4(acc[0][0][0] + acc[0][1][0], acc[0][0][1] + acc[0][1][1], acc[0][0][2] + acc[0][1][2],
                           acc[0][0][3] + acc[0][1][3]);
      dst[1] = make_float4(acc[1][0][0] + acc[1][1][0], acc[1][0][1] + acc[1][1][1], acc[1][0][2] + acc[1][1][2],
                           acc[1][0][3] + acc[1][1][3]);
    } else {  // per tile: gate, then up
#pragma unroll
      for (int tl = 0; tl < kNT; ++tl) {
        dst[2 * tl] = make_float4(acc[0][tl][0], acc[0][tl][1], acc[0][tl][2], acc[0][tl][3]);
        dst[2 * tl + 1] = make_float4(acc[1][tl][0], acc[1][tl][1], acc[1][tl][2], acc[1][tl][3]);
      }
    }
  };
  // kGD units in flight per warp: the first ones are requested before anything else
  UnitRegs<2> rr[kGD];
#pragma unroll
  for (int d = 0; d < kGD; ++d) load(warp + d * kWarps, rr[d]);
  if (tid == kThreads - 32) {
    // every weight byte of the CTA's down tasks into L2 -- one bulk prefetch per group and
    // region, the rows of consecutive tasks of a group being contiguous
    for (int gi = d0 / NRB; d1 > d0 && gi <= (d1 - 1) / NRB; ++gi) {
      const uint8_t* blob = sm.gblob[gi];
      if (!blob) continue;
      const int ra_ = max(d0, gi * NRB) - gi * NRB, rbb = min(d1, (gi + 1) * NRB) - gi * NRB;
      prefetch_bulk_l2(blob + a.lay.code_off[2] + size_t(ra_) * 8 * I, uint32_t((rbb - ra_) * 8 * I));
      prefetch_bulk_l2(blob + a.lay.scale_off[2] + size_t(ra_) * I, uint32_t((rbb - ra_) * I));
    }
  }
  // the groups' global scales (the 16 header bytes at offset 16 of each blob) by
  // asynchronous copies, waited for only before the first epilogue
  for (int g = tid; g < Gt; g += kThreads) {
    if (sm.gblob[g]) cp16(&sm.gs[g][0], sm.gblob[g] + 16);
    else sm.gs[g][0] = sm.gs[g][1] = sm.gs[g][2] = 0.f;
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  for (; r0 < U; r0 += kUnitsGU) {
    nu = min(kUnitsGU, U - r0);
    if (r0 > 0) {
#pragma unroll
      for (int d = 0; d < kGD; ++d) load(r0 + warp + d * kWarps, rr[d]);
    }
    for (int u = r0 + warp; u < r0 + nu; u += kGD * kWarps) {
#pragma unroll
      for (int d = 0; d < kGD; ++d) {
        run(u + d * kWarps, rr[d]);
        load(u + (d + kGD) * kWarps, rr[d]);
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    // each task's chunks summed in order; epilogue h = SiLU(gs_g g / s_x) * (gs_u u / s_x)
    const int ntk = nu / NCH;
    for (int idx = tid; idx < ntk * 32; idx += kThreads) {
      const int tl = idx >> 5;
      const int task = t0 + (r0 >> lNCH) + tl, gi = task >> lTPG, tb = task & (TPG - 1);
      float v[8 * kNT];  // per tile: gate (4), up (4)
#pragma unroll
      for (int j = 0; j < 8 * kNT; ++j) v[j] = 0.f;
      for (int c = 0; c < NCH; ++c) {
        const float4* src = reinterpret_cast<const float4*>(red + (size_t(tl * NCH + c) * 32 + lane) * 8 * kNT);
#pragma unroll
        for (int j = 0; j < 2 * kNT; ++j) {
          const float4 pj = src[j];
          v[4 * j] += pj.x; v[4 * j + 1] += pj.y; v[4 * j + 2] += pj.z; v[4 * j + 3] += pj.w;
        }
      }
      const bool shared = gi == G;
      const bool has_blob = sm.gblob[gi] != nullptr;
      const int e0 = sm.goff[gi], nv = sm.goff[gi + 1] - e0;
      const float gs0 = sm.gs[gi][0], gs1 = sm.gs[gi][1];
#pragma unroll
      for (int tt = 0; tt < kNT; ++tt) {
        float hm[2] = {0.f, 0.f};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int jloc = 8 * tt + 2 * t4 + (q & 1);
          const int r = tb * 16 + g8 + 8 * (q >> 1);
          if (jloc < nv) {
            const int tok = shared ? jloc : sm.ent_tok[e0 + jloc];
            const float inv = sm.xinv[tok];
            const float hv =
                has_blob ? silu_f32(v[8 * tt + q] * inv * gs0) * (v[8 * tt + 4 + q] * inv * gs1) : 0.f;
            const int hrow = shared ? a.maxTk + jloc : e0 + jloc;
            a.h[size_t(hrow) * a.Imax + r] = hv;
            hm[q & 1] = fmaxf(hm[q & 1], fabsf(hv));
          }
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          hm[0] = fmaxf(hm[0], __shfl_xor_sync(0xffffffffu, hm[0], o));
          hm[1] = fmaxf(hm[1], __shfl_xor_sync(0xffffffffu, hm[1], o));
        }
        if (g8 == 0)
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int jloc = 8 * tt + 2 * t4 + q;
            if (jloc < nv)
              atomicMax(reinterpret_cast<unsigned int*>(a.hmax) + (shared ? a.maxTk + jloc : e0 + jloc),
                        __float_as_uint(hm[q]));
          }
      }
    }
    __syncthreads();
  }
  grid_arrive(a, sm);

  // ============================================================ D: down
  // The CTA's tasks [d0, d1) in group order.  The h rows of every group of its range --
  // entries goff[gA] .. goff[gB + 1], the shared expert's T rows counted as entries n ..
  // n + T - 1 -- are staged in ONE batch of loads with their max|h|, as f16 times the
  // power of two of each row's max|h| (11 significant bits); the (task, 256-column chunk)
  // units then run as in C, their weights already in L2, and each task's chunks are
  // summed in order into o (fp32, by output position t*k + r; the shared expert's rows
  // after).
  {
    const int gA = d1 > d0 ? d0 / NRB : 0, gB = d1 > d0 ? (d1 - 1) / NRB : -1;
    const int rbase = d1 > d0 ? sm.goff[gA] : 0, nrows = d1 > d0 ? sm.goff[gB + 1] - rbase : 0;
    const bool fits = nrows <= a.hrows;  // always, by the launch's row bound
    if (!fits) set_error(a.err, MOE_ERANGE);
    const int ud = fits ? (d1 - d0) * NCD : 0;
    auto unit_of = [&](int u, int& gi, int& rb, int& ch) {
      const int task = d0 + (u >> lNCD);
      ch = u & (NCD - 1);
      gi = task >> lNRB;
      rb = task & (NRB - 1);
    };
    // three units in flight per warp (a unit is half a gate/up unit); the first ones (their
    // weights in L2 by now, and no other CTA writes them) are requested between this CTA's
    // arrival at the barrier and its wait, the h rows staged after the wait
    auto load_d = [&](int u, int lim, UnitRegs<1>& R) {
      if (u >= lim) return;
      int gi, rb, ch;
      unit_of(u, gi, rb, ch);
      if (sm.gblob[gi]) load_unit<1>(sm.gblob[gi], a.lay, 2, I, rb * 16 + g8, ch, t4, R);
    };
    UnitRegs<1> da, db, dc;
    load_d(warp, min(kUnitsDN, ud), da);
    load_d(warp + kWarps, min(kUnitsDN, ud), db);
    load_d(warp + 2 * kWarps, min(kUnitsDN, ud), dc);
    if (!grid_wait(a, sm)) return;
    for (int q0 = 0; q0 < ud; q0 += kUnitsDN) {
      const int nq = min(kUnitsDN, ud - q0);
      if (q0 == 0) {
        const int per = I / 4, lper = __ffs(per) - 1;
        constexpr int kB = 4;  // 16 rows of 512 in one batch
        for (int i0 = 0; i0 < nrows * per; i0 += kB * kThreads) {
          float4 f[kB];
          float hmx[kB];
#pragma unroll
          for (int j = 0; j < kB; ++j) {
            const int i = i0 + tid + j * kThreads;
            if (i < nrows * per) {
              const int R = i >> lper, q4 = i & (per - 1), e = rbase + R;
              const size_t grow = e < n ? size_t(e) : size_t(a.maxTk + e - n);
              f[j] = __ldcg(reinterpret_cast<const float4*>(a.h + grow * a.Imax) + q4);
              hmx[j] = __ldcg(a.hmax + grow);
            }
          }
#pragma unroll
          for (int j = 0; j < kB; ++j) {
            const int i = i0 + tid + j * kThreads;
            if (i < nrows * per) {
              const int R = i >> lper, q4 = i & (per - 1);
              const float sc = pow2_scale_for(hmx[j]);
              __half2 p0 = __floats2half2_rn(f[j].x * sc, f[j].y * sc), p1 = __floats2half2_rn(f[j].z * sc, f[j].w * sc);
              uint2 w2;
              w2.x = *reinterpret_cast<uint32_t*>(&p0);
              w2.y = *reinterpret_cast<uint32_t*>(&p1);
              *reinterpret_cast<uint2*>(h16 + size_t(R) * HR + perm_col(4 * q4)) = w2;
              if (q4 == 0) sm.hs_inv[R] = 1.0f / sc;
            }
          }
        }
        __syncthreads();  // the staged rows are complete
      }
      if (q0 > 0) {
        load_d(q0 + warp, q0 + nq, da);
        load_d(q0 + warp + kWarps, q0 + nq, db);
        load_d(q0 + warp + 2 * kWarps, q0 + nq, dc);
      }
      auto run_d = [&](int u, const UnitRegs<1>& R) {
        if (u >= q0 + nq) return;
        int gi, rb, ch;
        unit_of(u, gi, rb, ch);
        const int nv = sm.goff[gi + 1] - sm.goff[gi];
        float acc[1][2][4];
#pragma unroll
        for (int x = 0; x < 8; ++x) acc[0][x >> 2][x & 3] = 0.f;
        if (sm.gblob[gi]) {
          const __half* hb = h16 + size_t(sm.goff[gi] - rbase) * HR;
          mma_unit<1, kNT>(R, g8 < nv ? hb + size_t(g8) * HR : nullptr,
                          (kNT == 2 && g8 + 8 < nv) ? hb + size_t(g8 + 8) * HR : nullptr, ch, t4, acc);
        }
        float4* dst = reinterpret_cast<float4*>(red + (size_t(u - q0) * 32 + lane) * 4 * kNT);
        if (kNT == 1)
          dst[0] = make_float4(acc[0][0][0] + acc[0][1][0], acc[0][0][1] + acc[0][1][1], acc[0][0][2] + acc[0][1][2],
                               acc[0][0][3] + acc[0][1][3]);
        else
#pragma unroll
          for (int tl = 0; tl < kNT; ++tl) dst[tl] = make_float4(acc[0][tl][0], acc[0][tl][1], acc[0][tl][2], acc[0][tl][3]);
      };
      for (int u = q0 + warp; u < q0 + nq; u += 3 * kWarps) {
        run_d(u, da);
        load_d(u + 3 * kWarps, q0 + nq, da);
        run_d(u + kWarps, db);
        load_d(u + 4 * kWarps, q0 + nq, db);
        run_d(u + 2 * kWarps, dc);
        load_d(u + 5 * kWarps, q0 + nq, dc);
      }
      __syncthreads();
      for (int idx = tid; idx < (nq / NCD) * 32; idx += kThreads) {
        const int tl = idx >> 5, task = d0 + (q0 >> lNCD) + tl, gi = task >> lNRB, rbk = task & (NRB - 1);
        float v[4 * kNT];
#pragma unroll
        for (int j = 0; j < 4 * kNT; ++j) v[j] = 0.f;
        for (int c = 0; c < NCD; ++c) {
          const float4* pp = reinterpret_cast<const float4*>(red + (size_t(tl * NCD + c) * 32 + lane) * 4 * kNT);
#pragma unroll
          for (int tt = 0; tt < kNT; ++tt) {
            const float4 f = pp[tt];
            v[4 * tt] += f.x; v[4 * tt + 1] += f.y; v[4 * tt + 2] += f.z; v[4 * tt + 3] += f.w;
          }
        }
        const bool shared = gi == G, has_blob = sm.gblob[gi] != nullptr;
        const int e0 = sm.goff[gi], nv = sm.goff[gi + 1] - e0;
        const float gsd = sm.gs[gi][2];
#pragma unroll
        for (int x = 0; x < 4 * kNT; ++x) {
          const int jloc = 8 * (x >> 2) + 2 * t4 + (x & 1);
          if (jloc < nv) {
            const int pos = shared ? a.maxTk + jloc : sm.ent_pos[e0 + jloc];
            a.o[size_t(pos) * H + rbk * 16 + g8 + 8 * ((x >> 1) & 1)] =
                has_blob ? v[x] * sm.hs_inv[e0 - rbase + jloc] * gsd : 0.f;
          }
        }
      }
      __syncthreads();
    }
  }
  if (!grid_barrier(a, sm)) return;

  // ============================================================ combine
  // y[t] = sum_r w[t,r] o[t*k + r] + sigmoid(gl_t) o[shared t], rank order, the shared
  // term last; CTA c owns a contiguous range of the T x H/4 four-column items.
  const int NI = T * (H / 4);
  const int i0 = int((long long)cta * NI / ncta), i1 = int((long long)(cta + 1) * NI / ncta);
  for (int i = i0 + tid; i < i1; i += kThreads) {
    const int t = i >> (__ffs(H) - 3), c4 = i & (H / 4 - 1);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const int nrow = k + a.has_shared;
    for (int r0 = 0; r0 < nrow; r0 += 16) {  // one round trip for k <= 15
      float4 v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int r = r0 + j;
        if (r < nrow) {
          const size_t row = r < k ? size_t(t * k + r) : size_t(a.maxTk + t);
          v[j] = __ldcg(reinterpret_cast<const float4*>(a.o + row * H) + c4);
        }
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int r = r0 + j;
        if (r < nrow) {
          const float cf = r < k ? sm.w[t * k + r] : sigmoid_f32(sm.gl[t]);
          acc.x = fmaf(cf, v[j].x, acc.x);
          acc.y = fmaf(cf, v[j].y, acc.y);
          acc.z = fmaf(cf, v[j].z, acc.z);
          acc.w = fmaf(cf, v[j].w, acc.w);
        }
      }
    }
    if (a.y_fp32) {
      reinterpret_cast<float4*>(a.y)[i] = acc;
    } else {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo);
      pk.y = *reinterpret_cast<uint32_t*>(&hi);
      reinterpret_cast<uint2*>(a.y)[i] = pk;
    }
  }
}

}  // namespace dec

// ----------------------------------------------------------------- host
namespace {

int sm_count_dec() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

bool pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

int align128(int v) { return (v + 127) & ~127; }

}  // namespace

// Shared-memory layout of one launch; false when the shapes do not fit the kernel.
static bool decode_fused_layout(const moe_layer_shape& sh, int T, int ncta, dec::Args& a, size_t& smem) {
  using namespace dec;
  const int H = sh.H, I = sh.I, k = sh.k, E = sh.E;
  // x as f16 (phases A..C); the partial tiles (C: 8 floats per lane and unit, D: 4); the
  // staged h rows (D): as many as a CTA's range of down tasks can reach -- the groups it
  // spans times T, at most every entry's and the shared expert's
  a.o_x16 = 0;
  const int nrb = H / 16, tasks = ((T * k + 1) * nrb + ncta - 1) / ncta;
  a.hrows = ((tasks + nrb - 1) / nrb + 1) * T;
  if (a.hrows > T * k + T) a.hrows = T * k + T;
  a.o_red = align128(T * (H + kPadH) * 2);
  a.o_h16 = a.o_red + kMaxUnits * 32 * 8 * 4;
  const int end_cd = a.o_h16 + align128(a.hrows * (I + kPadH) * 2);
  // over the tiles and the rows (unused until C): phase A's x (bf16) and router partial
  // sums, then, over those (dead after the first barrier), phase B's logits and the
  // top-k's chunk bests, candidates, selections and terms
  a.capc = E < 32 * k ? E : 32 * k;
  a.o_xs = a.o_red;
  a.o_part = a.o_xs + align128(T * H * 2);
  const int end_a = a.o_part + align128(kMaxPairs * dec::kMaxT * 4);
  a.o_lg = a.o_red;
  a.o_cb = a.o_lg + align128(T * E * 4);
  a.o_cand = a.o_cb + align128(T * 32 * 8);
  a.o_sel = a.o_cand + align128(T * a.capc * 8);
  a.o_pr = a.o_sel + align128(T * k * 8);
  const int end_b = a.o_pr + align128(T * k * 4);
  const int end_ab = end_a > end_b ? end_a : end_b;
  a.o_small = align128(end_ab > end_cd ? end_ab : end_cd);
  smem = size_t(a.o_small) + sizeof(Small);
  return smem <= 227 * 1024;
}

// The fused decode forward when the shapes allow it, else kNotFused.
int launch_decode_fused(const moe_layer_desc* d, moe_cache* c, const uint16_t* x, void* y, int y_is_fp32, int T,
                        moe_ws* ws, cudaStream_t s) {
  using namespace dec;
  const moe_layer_shape& sh = d->s;
  const bool has_shared = sh.I_shared > 0 && d->shared_blob;
  if (T < 1 || T > dec::kMaxT || T * sh.k > dec::kMaxEnt || sh.E > 1024) return kNotFused;
  if (!pow2(sh.H) || sh.H < kSlice || sh.H > 2048 || !pow2(sh.I) || sh.I < kChunk || sh.I > 1024) return kNotFused;
  if (has_shared && sh.I_shared != sh.I) return kNotFused;
  if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(y) & 15) ||
      (reinterpret_cast<uintptr_t>(d->w_router) & 15) ||
      (has_shared && ((reinterpret_cast<uintptr_t>(d->shared_blob) & 31) ||
                      (reinterpret_cast<uintptr_t>(d->w_shared_gate) & 15))))
    return kNotFused;
  const int ncta = sm_count_dec();
  const int rows_total = sh.E + (has_shared && d->w_shared_gate ? 1 : 0);
  if ((rows_total + ncta - 1) / ncta * (sh.H / kSlice) > kMaxPairs) return kNotFused;
  Args a = {};
  size_t smem = 0;
  if (!decode_fused_layout(sh, T, ncta, a, smem)) return kNotFused;
  const int tp = T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : T <= 8 ? 8 : 16;
  void (*kern)(const Args) = tp == 1 ? k_decode_fused<1> : tp == 2 ? k_decode_fused<2>
                           : tp == 4 ? k_decode_fused<4> : tp == 8 ? k_decode_fused<8> : k_decode_fused<16>;
  static bool attr[5] = {false, false, false, false, false};
  const int ti = tp == 1 ? 0 : tp == 2 ? 1 : tp == 4 ? 2 : tp == 8 ? 3 : 4;
  if (!attr[ti]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) != cudaSuccess)
      return MOE_ECUDA;
    attr[ti] = true;
  }
  a.x = x;
  a.w_router = d->w_router;
  a.bias = d->bias;
  a.w_sg = has_shared ? d->w_shared_gate : nullptr;
  a.shared_blob = has_shared ? static_cast<const uint8_t*>(d->shared_blob) : nullptr;
  a.T = T;
  a.H = sh.H;
  a.I = sh.I;
  a.E = sh.E;
  a.k = sh.k;
  a.layer = d->layer;
  a.has_shared = has_shared ? 1 : 0;
  a.lay = dev_layout(sh.H, sh.I);
  a.resid = c->resid;
  a.stage = c->stage;
  a.slots = c->slots;
  a.staging = c->staging;
  a.blob_bytes = c->blob_bytes;
  a.shared_bytes = has_shared ? blob_layout(sh.H, sh.I_shared).bytes : 0;
  a.nslots = c->nslots;
  a.nstaging = c->nstaging;
  a.tail_skip = ws->tail_skip;
  a.stats = c->stats;
  a.heat_row = ws->fused_heat ? c->heat + size_t(d->layer) * sh.E : nullptr;
  a.logits = ws->logits;
  a.gate_logit = ws->gate_logit;
  a.topk_ids = ws->topk_ids;
  a.topk_w = ws->topk_w;
  a.num_groups = ws->num_groups;
  a.grp_expert = ws->grp_expert;
  a.grp_off = ws->grp_off;
  a.grp_slot = ws->grp_slot;
  a.grp_src = ws->grp_src;
  a.grp_blob = ws->grp_blob;
  a.ent_tok = ws->ent_tok;
  a.ent_pos = ws->ent_pos;
  a.h = ws->h;
  a.hmax = ws->hmax;
  a.o = ws->o;
  a.Imax = ws->s.I > ws->s.I_shared ? ws->s.I : ws->s.I_shared;
  a.maxTk = ws->maxT * ws->s.k;
  a.y = y;
  a.y_fp32 = y_is_fp32;
  a.err = ws->error;
  a.bar = ws->bar;
  a.bar_extra = ws->bar_extra;
  a.wait_ns = ws->wait_ns;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ncta);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeCooperative;
  attrs[0].val.cooperative = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ECUDA;
  }
  return MOE_OK;
}

}  // namespace moe
