// Decode expert GEMVs for windows of at most 8 tokens: weights streamed from HBM
// straight into registers by every warp of the CTA.
//
// Strata expert paths, "CPU 怎样把剩下的专家算完？" (gate/up, activation, down)
// and "路由以后，专家怎样分工？" (outputs by position, then weighted and summed).
// The arithmetic is that of k_expert.cu: mma.sync m16n8k16 f16 -> f32 with the
// weights (E2M1 code x E4M3 block scale, exact in f16) as A and up to 8
// activation vectors (f16 after a per-vector power-of-two scale) as B, with the
// same lane-local K permutation (a lane reads 16 contiguous columns of one
// scale block per 64-column segment).
//
// Streaming.  A task is RB consecutive 16-row blocks of one group's matrix
// (gate/up: the gate rows and the matching up rows) over the full K range,
// cut into 128-column chunks.  Each CTA owns a contiguous range of tasks; its
// 16 warps split every task (row block x chunk), so each warp walks its own
// sequence of units and never waits for another warp while it streams: each
// lane owns 64 contiguous columns of a 256-column chunk (32 code bytes per
// row, one 256-bit load, so four lanes fetch a whole 128-byte line; four scale
// blocks) and loads them from HBM straight into a ring of registers a few
// units ahead, and the activations (x, or the groups' h rows as f16)
// sit in shared memory with the same lane-local K permutation.  Partial tiles
// go to shared memory; only when a round of tasks is complete do the warps
// meet, and each (task, row block) is then summed in warp order by one warp,
// which writes its rows -- no split crosses CTAs and the results do not depend
// on scheduling.
#include "dequant.cuh"

namespace moe {
namespace gemv {

constexpr int kWarps = 16;
constexpr int kChunk = 256;        // columns per chunk (a lane's 64 columns = one 32-byte load per row)
constexpr int kXPadH = 8;          // f16 elements after each activation row
constexpr int kDownGroups = 4;     // down: groups whose h rows a CTA keeps in shared memory
constexpr int kMaxRound = 16;      // tasks per round at most
constexpr size_t kSmemBudget = 226 * 1024;  // leaves room for static shared variables

// Geometry shared by host and device (the logged quantities are powers of two).
struct Geo {
  int K;         // contraction length of every matrix of this launch
  int rows;      // rows of one matrix (gate/up: I per matrix; down: H)
  int KPW, RB;   // warps per row block, row blocks per task (RB * KPW <= kWarps)
  int CPW;       // chunks per warp per task = K / kChunk / KPW
  int TPG;       // tasks per group = rows / (16 RB)
  int l_cpw, l_tpg, l_rb, l_per;
  int R;         // tasks per round (partial tiles held in shared memory)
  int xrow;      // activation row stride in f16 elements
  int TPC;       // tasks per CTA at most (scale buffer)
  int srow;      // scale row stride in shared memory: K/16 + 16 bytes
  int l_sq;      // log2 of the 16-byte scale chunks per row (K/256)
  int x_b, red_b, tab_b, sc_b;
};

struct Args {
  const int32_t* num_groups;
  const int32_t* grp_off;
  const uint8_t* const* grp_blob;
  const int32_t* ent_tok;
  const int32_t* ent_pos;
  float* h;              // [(maxTk + maxT) * Imax]
  float* hmax;           // [maxTk + maxT]
  float* o;              // [(maxTk + maxT) * H]
  const uint8_t* shared_blob;
  int T, H, I, Imax, maxTk, Tk;
  DevBlobLayout lay;     // routed and shared blobs share H and I here
  Geo geo;
  int32_t* err;
  const __half* x16;     // gate/up: [T, H] f16, x times a per-token power of two
  const float* xscale;   // gate/up: [T] that power of two
};

struct Smem {
  uint8_t* sc;           // [TPC][NM*16*RB rows][srow] scale rows of the CTA's tasks
  __half* xs;            // gate/up: [T][xrow] x16; down: [kDownGroups][8][xrow] h16 of the CTA's groups
  float* red;            // [R][kWarps][32][NM*4] partial tiles of a round
  int32_t* goff;         // [Tk + 2]
  int32_t* idx;          // [Tk] token (gate/up) or output position (down) of each entry
  const uint8_t** blob;  // [Tk + 1]
  float* vinv;           // gate/up: [8] 1/xscale per token; down: [kDownGroups][8] 1/(h scale) per entry
  float* gs;             // [Tk + 1][2] global scales of each group's matrices
};

__device__ __forceinline__ Smem carve(uint8_t* base, const Geo& g, int Tk) {
  Smem s;
  s.sc = base;
  base += g.sc_b;
  s.xs = reinterpret_cast<__half*>(base);
  s.red = reinterpret_cast<float*>(base + g.x_b);
  s.goff = reinterpret_cast<int32_t*>(base + g.x_b + g.red_b);
  s.idx = s.goff + (Tk + 2);
  uintptr_t q = reinterpret_cast<uintptr_t>(s.idx + Tk);
  q = (q + 7) & ~uintptr_t(7);
  s.blob = reinterpret_cast<const uint8_t**>(q);
  s.vinv = reinterpret_cast<float*>(s.blob + (Tk + 1));
  s.gs = s.vinv + kDownGroups * 8;
  return s;
}

// One chunk of one warp's rows, as loaded: rows g8 and g8+8 of each matrix.
template <int NM>
struct Unit {
  uint32_t c[NM][2][8];  // 32 code bytes per row (the lane's 64 columns)
};

// GATEUP: x (f16 rows of the tokens) -> h[entry row][r] = SiLU(gs_g <Wg_r,x>) * gs_u <Wu_r,x>, max|h| per row.
// !GATEUP: h (fp32 rows, to f16 with a per-row power of two) -> o[position][r] = gs_d <Wd_r,h>.
// Group G (after the routed groups) is the shared expert, whose entries are the T tokens.
template <bool GATEUP, int D>
__global__ void __launch_bounds__(kWarps * 32, 1) k_gemv(Args a) {
  pdl_wait();
  constexpr int NM = GATEUP ? 2 : 1;
  extern __shared__ __align__(128) uint8_t smem[];
  const Geo g = a.geo;
  const Smem S = carve(smem, g, a.Tk);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g8 = lane >> 2, t4 = lane & 3;

  // ---- tables: every load independent of the group count, so one latency
  const int G = *a.num_groups;
  for (int i = tid; i <= a.Tk + 1; i += blockDim.x) {
    const int off = i <= a.Tk ? a.grp_off[i] : 0;
    const uint8_t* b = i < a.Tk ? a.grp_blob[i] : nullptr;
    S.goff[i] = i <= G ? off : a.Tk + a.T;  // entry G+1 closes the shared expert's T entries
    if (i <= a.Tk) S.blob[i] = i < G ? b : (i == G ? a.shared_blob : nullptr);
  }
  for (int i = tid; i < a.Tk; i += blockDim.x) S.idx[i] = GATEUP ? a.ent_tok[i] : a.ent_pos[i];
  const int ngr = G + (a.shared_blob ? 1 : 0);
  const int NT = ngr * g.TPG;
  const int t_begin = int((long long)blockIdx.x * NT / gridDim.x);
  const int t_end = int((long long)(blockIdx.x + 1) * NT / gridDim.x);
  __syncthreads();
  if (t_begin >= t_end) return;  // uniform across the CTA (and not counted by the combine below)

  const int rbw = warp / g.KPW, kc = warp - rbw * g.KPW;
  const bool computes = rbw < g.RB;
  const int NU = (t_end - t_begin) << g.l_cpw;
  const int g_first = t_begin >> g.l_tpg, g_last = (t_end - 1) >> g.l_tpg;

  auto load_unit = [&](int u, Unit<NM>& R) {
    if (!computes || u >= NU) return;
    const int tl = u >> g.l_cpw, c = u & (g.CPW - 1);
    const int task = t_begin + tl, gi = task >> g.l_tpg, tb = task & (g.TPG - 1);
    const uint8_t* blob = S.blob[gi];
    if (!blob) return;  // a missing expert: its rows are written as zeros
    const int ch = kc + c * g.KPW;
    const int r = (tb * g.RB + rbw) * 16 + g8;
#pragma unroll
    for (int m = 0; m < NM; ++m) {
      const int mat = GATEUP ? m : 2;
      const uint8_t* cp = blob + a.lay.code_off[mat] + size_t(r) * (g.K / 2) + ch * 128 + 32 * t4;
      ld_stream32(cp, R.c[m][0]);
      ld_stream32(cp + size_t(8) * (g.K / 2), R.c[m][1]);
    }
  };
  // ---- the small operands first, as cp.async, so that they travel ahead of the weights:
  // scale rows of all the CTA's tasks (whole 16-byte chunks into padded rows), then
  // x rows (gate/up) or the groups' fp32 h rows and their max|h| (down)
  {
    const int rows_m = 16 * g.RB, nrow = NM * rows_m, sq = 1 << g.l_sq;
    const int total = ((t_end - t_begin) * nrow) << g.l_sq;
    for (int c = tid; c < total; c += blockDim.x) {
      const int q = c & (sq - 1), rr0 = c >> g.l_sq;
      const int tl = rr0 / nrow, r = rr0 - tl * nrow;
      const int task = t_begin + tl, gi = task >> g.l_tpg, tb = task & (g.TPG - 1);
      const uint8_t* blob = S.blob[gi];
      if (!blob) continue;
      const int m = r / rows_m, rr = r - m * rows_m;
      const uint8_t* src = blob + a.lay.scale_off[GATEUP ? m : 2] + size_t(tb * rows_m + rr) * (g.K / 16) + q * 16;
      cp16(S.sc + size_t(rr0) * g.srow + q * 16, src);
    }
  }
  float* hst = S.red;  // down: fp32 h rows [slot][8][I], staged before the partial tiles use the space
  if (GATEUP) {
    const int cpr = a.H / 8;
    for (int c = tid; c < a.T * cpr; c += blockDim.x) {
      const int t = c / cpr, q = c - t * cpr;
      cp16(S.xs + size_t(t) * g.xrow + q * 8, a.x16 + size_t(t) * a.H + q * 8);
    }
    if (tid < a.T) cp4(S.vinv + tid, a.xscale + tid);
  } else {
    const int per = a.I / 4;
    for (int gi = g_first; gi <= g_last; ++gi) {
      const int e0 = S.goff[gi], nv = S.goff[gi + 1] - e0, slot = gi - g_first;
      for (int c = tid; c < nv * per; c += blockDim.x) {
        const int j = c >> g.l_per, q4 = c & (per - 1);
        const int rowh = gi == G ? a.maxTk + j : e0 + j;
        cp16(hst + (size_t(slot) * 8 + j) * a.I + q4 * 4, a.h + size_t(rowh) * a.Imax + q4 * 4);
        if (q4 == 0) cp4(S.vinv + slot * 8 + j, a.hmax + rowh);
      }
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  float gsr[NM];  // global scales of group g_first + tid
#pragma unroll
  for (int m = 0; m < NM; ++m) gsr[m] = 0.f;
  if (g_first + tid <= g_last) {
    const uint8_t* b = S.blob[g_first + tid];
#pragma unroll
    for (int m = 0; m < NM; ++m) gsr[m] = b ? reinterpret_cast<const BlobHeader*>(b)->gscale[GATEUP ? m : 2] : 0.f;
  }

  if (g_first + tid <= g_last)
#pragma unroll
    for (int m = 0; m < NM; ++m) S.gs[2 * (g_first + tid) + m] = gsr[m];
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  // ---- then the weight stream, once the small operands have landed (issued
  // together, they queued behind the weights and arrived last)
  Unit<NM> ring[D];
#pragma unroll
  for (int d = 0; d < D; ++d) load_unit(d, ring[d]);
  // the codes of the tasks beyond the ring's first D units go to L2 now, so
  // that their loads, issued when the ring turns over, find them there
  {
    const int t_first = (D + g.CPW - 1) >> g.l_cpw, ntl = t_end - t_begin;
    if (t_first < ntl && tid < (ntl - t_first) * NM) {
      const int tl = t_first + tid / NM, m = tid - (tid / NM) * NM;
      const int task = t_begin + tl, gi = task >> g.l_tpg, tb = task & (g.TPG - 1);
      const uint8_t* blob = S.blob[gi];
      if (blob)
        prefetch_bulk_l2(blob + a.lay.code_off[GATEUP ? m : 2] + size_t(tb * g.RB * 16) * (g.K / 2),
                         uint32_t(g.RB * 16) * uint32_t(g.K / 2));
    }
  }
  if (GATEUP) {
    if (tid < a.T) S.vinv[tid] = 1.0f / S.vinv[tid];
    __syncthreads();
  } else {
    // h -> f16 times the power of two chosen from max|h| of its row
    const int per = a.I / 4;
    for (int gi = g_first; gi <= g_last; ++gi) {
      const int e0 = S.goff[gi], nv = S.goff[gi + 1] - e0, slot = gi - g_first;
      for (int c = tid; c < nv * per; c += blockDim.x) {
        const int j = c >> g.l_per, q4 = c & (per - 1);
        const float sc = pow2_scale_for(S.vinv[slot * 8 + j]);
        const float4 f = *reinterpret_cast<const float4*>(hst + (size_t(slot) * 8 + j) * a.I + q4 * 4);
        __half2 p0 = __floats2half2_rn(f.x * sc, f.y * sc), p1 = __floats2half2_rn(f.z * sc, f.w * sc);
        uint2 w2;
        w2.x = *reinterpret_cast<uint32_t*>(&p0);
        w2.y = *reinterpret_cast<uint32_t*>(&p1);
        *reinterpret_cast<uint2*>(S.xs + (size_t(slot) * 8 + j) * g.xrow + q4 * 4) = w2;
      }
    }
    __syncthreads();
    for (int i = tid; i < kDownGroups * 8; i += blockDim.x) S.vinv[i] = 1.0f / pow2_scale_for(S.vinv[i]);
    __syncthreads();
  }

  float acc[NM][2][4];  // two chains per matrix (even and odd MMAs), summed at the end of a task
#pragma unroll
  for (int m = 0; m < NM; ++m)
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[m][q >> 2][q & 3] = 0.f;

  auto compute_unit = [&](int u, const Unit<NM>& R) {
    const int tl = u >> g.l_cpw, c = u & (g.CPW - 1);
    const int gi = (t_begin + tl) >> g.l_tpg;
    const int e0 = S.goff[gi], nv = S.goff[gi + 1] - e0;
    const int ch = kc + c * g.KPW;
    // this lane's four scale bytes of rows g8 and g8 + 8 of each matrix
    uint32_t scw[NM][2];
#pragma unroll
    for (int m = 0; m < NM; ++m) {
      const int r = m * 16 * g.RB + rbw * 16 + g8;
      const uint8_t* sp = S.sc + (size_t(tl) * (NM * 16 * g.RB) + r) * g.srow + ch * 16 + 4 * t4;
      scw[m][0] = *reinterpret_cast<const uint32_t*>(sp);
      scw[m][1] = *reinterpret_cast<const uint32_t*>(sp + 8 * g.srow);
    }
    const bool has_vec = g8 < nv;
    const int row = has_vec ? (GATEUP ? (gi == G ? g8 : S.idx[e0 + g8]) : (gi - g_first) * 8 + g8) : 0;
    const uint4* xp = reinterpret_cast<const uint4*>(S.xs + size_t(row) * g.xrow + ch * kChunk + 64 * t4);
#pragma unroll
    for (int q = 0; q < 8; ++q) {  // lane columns 8q..8q+7: MMAs 2q and 2q+1
      const uint4 xq = has_vec ? xp[q] : make_uint4(0u, 0u, 0u, 0u);
      const int blk = q >> 1;      // scale block of these columns
#pragma unroll
      for (int m = 0; m < NM; ++m) {
        const uint32_t sa = scale_pair((scw[m][0] >> (8 * blk)) & 0xffu);
        const uint32_t sb = scale_pair((scw[m][1] >> (8 * blk)) & 0xffu);
        const uint32_t w0 = R.c[m][0][q], w1 = R.c[m][1][q];
        uint32_t a0, a1, a2, a3;
        e2m1_pair2(w0, a0, a2);  // row g8, columns 8q..8q+3
        e2m1_pair2(w1, a1, a3);  // row g8 + 8
        mma16816(acc[m][0], hmul2(a0, sa), hmul2(a1, sb), hmul2(a2, sa), hmul2(a3, sb), xq.x, xq.y);
        e2m1_pair2(w0 >> 16, a0, a2);  // columns 8q+4..8q+7
        e2m1_pair2(w1 >> 16, a1, a3);
        mma16816(acc[m][1], hmul2(a0, sa), hmul2(a1, sb), hmul2(a2, sa), hmul2(a3, sb), xq.z, xq.w);
      }
    }
  };

  // tasks [first, last] of the round (CTA-local indices): each (task, row block)
  // summed over its KPW warps in order by one warp, which writes the rows
  auto reduce_round = [&](int first, int last) {
    const int npair = (last - first + 1) << g.l_rb;
    for (int pi = warp; pi < npair; pi += kWarps) {
      const int tr = pi >> g.l_rb, rb = pi & (g.RB - 1);
      const int task = t_begin + first + tr, gi = task >> g.l_tpg, tb = task & (g.TPG - 1);
      const bool shared = gi == G;
      const int e0 = S.goff[gi], nv = S.goff[gi + 1] - e0;
      float v[NM][4];
#pragma unroll
      for (int m = 0; m < NM; ++m)
#pragma unroll
        for (int q = 0; q < 4; ++q) v[m][q] = 0.f;
      for (int p = 0; p < g.KPW; ++p) {
        const float4* src =
            reinterpret_cast<const float4*>(S.red + ((size_t(tr) * kWarps + rb * g.KPW + p) * 32 + lane) * NM * 4);
#pragma unroll
        for (int m = 0; m < NM; ++m) {
          const float4 f = src[m];
          v[m][0] += f.x;
          v[m][1] += f.y;
          v[m][2] += f.z;
          v[m][3] += f.w;
        }
      }
      const bool has_blob = S.blob[gi] != nullptr;
      const float gs0 = S.gs[2 * gi], gs1 = S.gs[2 * gi + (NM - 1)];
      const int row0 = (tb * g.RB + rb) * 16 + g8;
      float hm[2] = {0.f, 0.f};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int jloc = 2 * t4 + (q & 1);
        const int r = row0 + 8 * (q >> 1);
        if (jloc < nv) {
          const int rowh = shared ? a.maxTk + jloc : e0 + jloc;
          if (GATEUP) {
            const float inv = S.vinv[shared ? jloc : S.idx[e0 + jloc]];
            const float hv = has_blob ? silu_f32(v[0][q] * inv * gs0) * (v[NM - 1][q] * inv * gs1) : 0.f;
            a.h[size_t(rowh) * a.Imax + r] = hv;
            hm[q & 1] = fmaxf(hm[q & 1], fabsf(hv));
          } else {
            const int pos = shared ? a.maxTk + jloc : S.idx[e0 + jloc];
            a.o[size_t(pos) * a.H + r] = has_blob ? v[0][q] * S.vinv[(gi - g_first) * 8 + jloc] * gs0 : 0.f;
          }
        }
      }
      if (GATEUP) {
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          hm[0] = fmaxf(hm[0], __shfl_xor_sync(0xffffffffu, hm[0], o));
          hm[1] = fmaxf(hm[1], __shfl_xor_sync(0xffffffffu, hm[1], o));
        }
        if (g8 == 0)
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int jloc = 2 * t4 + q;
            if (jloc < nv)
              atomicMax(reinterpret_cast<unsigned int*>(a.hmax) + (shared ? a.maxTk + jloc : e0 + jloc),
                        __float_as_uint(hm[q]));
          }
      }
    }
  };

  int round_first = 0;
  for (int base = 0; base < NU; base += D) {
#pragma unroll
    for (int d = 0; d < D; ++d) {
      const int u = base + d;
      if (u < NU) {  // uniform across the CTA
        // the next kernel's blocks launch when this CTA enters its last D units
        // (launched at the start, waiting blocks slowed the running kernels)
        if (u == (NU > D ? NU - D : 0)) pdl_trigger();
        if (computes) compute_unit(u, ring[d]);
        load_unit(u + D, ring[d]);
        const int tl = u >> g.l_cpw;
        if ((u & (g.CPW - 1)) == g.CPW - 1) {  // the warp's last chunk of task tl
          if (computes)
#pragma unroll
            for (int m = 0; m < NM; ++m)
              reinterpret_cast<float4*>(S.red + ((size_t(tl - round_first) * kWarps + warp) * 32 + lane) * NM * 4)[m] =
                  make_float4(acc[m][0][0] + acc[m][1][0], acc[m][0][1] + acc[m][1][1],
                              acc[m][0][2] + acc[m][1][2], acc[m][0][3] + acc[m][1][3]);
#pragma unroll
          for (int m = 0; m < NM; ++m)
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[m][q >> 2][q & 3] = 0.f;
          if (tl - round_first == g.R - 1 || u == NU - 1) {
            __syncthreads();  // the round's partial tiles are written
            reduce_round(round_first, tl);
            __syncthreads();  // and read
            round_first = tl + 1;
          }
        }
      }
    }
  }

}

}  // namespace gemv

// ----------------------------------------------------------------- host
namespace {

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
int log2_of(int v) {
  int l = 0;
  while ((1 << (l + 1)) <= v) ++l;
  return l;
}

int sm_count_gemv() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

// Geometry of one launch; false when the shapes do not fit this kernel.
bool make_geo(bool gateup, const moe_layer_shape& sh, int T, int Tk, int grid, gemv::Geo& g, size_t& smem) {
  using namespace gemv;
  const int NM = gateup ? 2 : 1;
  g.K = gateup ? sh.H : sh.I;
  g.rows = gateup ? sh.I : sh.H;
  if (g.K < kChunk || g.rows < 16) return false;
  const int chunks = g.K / kChunk;
  g.KPW = chunks < kWarps ? chunks : kWarps;
  g.RB = kWarps / g.KPW;
  if (g.RB > g.rows / 16) g.RB = g.rows / 16;
  g.CPW = chunks / g.KPW;
  g.TPG = g.rows / (16 * g.RB);
  g.l_cpw = log2_of(g.CPW);
  g.l_tpg = log2_of(g.TPG);
  g.l_rb = log2_of(g.RB);
  g.l_per = log2_of(sh.I / 4);
  if (!gateup) {
    // the groups a CTA's task range can span must fit the h buffer
    const long long nt_max = (long long)(Tk + 1) * g.TPG;
    const long long per_cta = (nt_max + grid - 1) / grid;
    const long long span = (per_cta + g.TPG - 2) / g.TPG + 1;
    if (span > kDownGroups) return false;
  }
  g.TPC = int(((long long)(Tk + 1) * g.TPG + grid - 1) / grid);
  g.srow = g.K / 16 + 16;
  g.l_sq = log2_of(g.K / 256);
  g.sc_b = int(round_up(size_t(g.TPC) * NM * 16 * g.RB * g.srow, 128));
  g.xrow = (gateup ? sh.H : sh.I) + kXPadH;
  g.x_b = int(round_up(size_t(gateup ? T : kDownGroups * 8) * g.xrow * 2, 128));
  const size_t tab = round_up(size_t(Tk + 2) * 4 + size_t(Tk) * 4, 8) + size_t(Tk + 1) * 8 + kDownGroups * 8 * 4 +
                     size_t(Tk + 1) * 2 * 4;
  g.tab_b = int(round_up(tab, 128));
  const size_t per_task = size_t(kWarps) * 32 * NM * 16;
  const size_t fixed = size_t(g.sc_b) + g.x_b + g.tab_b;
  if (fixed + per_task > kSmemBudget) return false;
  size_t R = (kSmemBudget - fixed) / per_task;
  g.R = int(R > size_t(kMaxRound) ? kMaxRound : R);
  g.red_b = int(per_task * g.R);
  if (!gateup) {  // the fp32 h rows of the CTA's groups are staged in the partial-tile space
    const long long nt_max = (long long)(Tk + 1) * g.TPG;
    const long long per_cta = (nt_max + grid - 1) / grid;
    const long long span = (per_cta + g.TPG - 2) / g.TPG + 1;
    if (size_t(span) * 8 * sh.I * 4 > size_t(g.red_b)) return false;
  }
  smem = fixed + g.red_b;
  return smem <= kSmemBudget;
}

}  // namespace

bool gemv_decode_applicable(bool gateup, const moe_layer_desc* d, int T) {
  using namespace gemv;
  const moe_layer_shape& sh = d->s;
  const bool has_shared = sh.I_shared > 0 && d->shared_blob;
  if (T < 1 || T > 8 || (has_shared && sh.I_shared != sh.I) ||
      (has_shared && (reinterpret_cast<uintptr_t>(d->shared_blob) & 31)))
    return false;
  Geo g;
  size_t smem = 0;
  return make_geo(gateup, sh, T, T * sh.k, sm_count_gemv(), g, smem);
}

// Decode GEMV for windows of at most 8 tokens; returns kGemvNotApplicable when
// the shapes call for the general kernel.
int launch_gemv_decode(bool gateup, const moe_layer_desc* d, int T, moe_ws* ws, cudaStream_t s) {
  using namespace gemv;
  const moe_layer_shape& sh = d->s;
  const bool has_shared = sh.I_shared > 0 && d->shared_blob;
  if (!gemv_decode_applicable(gateup, d, T)) return kGemvNotApplicable;
  const int Tk = T * sh.k;
  const int grid = sm_count_gemv();
  Args a;
  size_t smem = 0;
  if (!make_geo(gateup, sh, T, Tk, grid, a.geo, smem)) return kGemvNotApplicable;
  a.num_groups = ws->num_groups;
  a.grp_off = ws->grp_off;
  a.grp_blob = ws->grp_blob;
  a.ent_tok = ws->ent_tok;
  a.ent_pos = ws->ent_pos;
  a.h = ws->h;
  a.hmax = ws->hmax;
  a.o = ws->o;
  a.shared_blob = has_shared ? reinterpret_cast<const uint8_t*>(d->shared_blob) : nullptr;
  a.T = T;
  a.H = sh.H;
  a.I = sh.I;
  a.Imax = ws->s.I > ws->s.I_shared ? ws->s.I : ws->s.I_shared;
  a.maxTk = ws->maxT * ws->s.k;
  a.Tk = Tk;
  a.lay = dev_layout(sh.H, sh.I);
  a.err = ws->error;
  a.x16 = ws->x16;
  a.xscale = ws->xscale;
  auto kern = gateup ? k_gemv<true, 2> : k_gemv<false, 3>;
  static bool attr_set[2] = {false, false};
  if (!attr_set[gateup]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBudget)) != cudaSuccess)
      return MOE_ECUDA;
    attr_set[gateup] = true;
  }
  if (launch_pdl(kern, dim3(grid), dim3(kWarps * 32), smem, s, a) != cudaSuccess) return MOE_ECUDA;
  return MOE_OK;
}

}  // namespace moe
