// Decode expert path: GEMVs over the slot blobs on the tensor cores, and the combine.
//
// Strata expert paths, "CPU 怎样把剩下的专家算完？": an expert computes gate and
// up, the activation, then the down projection; "路由以后，专家怎样分工？": each
// expert output is multiplied by its routing weight and summed, then the gated
// shared-expert contribution (same input) is added.  Qwen3.8-Flash-Next DGX
// Spark notes, "NVFP4 code 和 scale 如何反量化": weight = E2M1 code x E4M3 block
// scale (per 16) x FP32 global scale.
//
// Arithmetic.  A group's tokens (at most 8 at a time) form the N side of
// mma.sync m16n8k16 (f16 in, fp32 accumulate): A = code x block scale, which
// is exact in f16 (at most 6 significant bits, magnitude 2^-10 .. 2688);
// B = the activations in f16 after a power-of-two per-vector scale (the x
// input is bf16 and lands in f16 exactly; the down input h is fp32 and is
// rounded to f16, relative error <= 2^-11).  Within each 64-column segment a
// lane's K slots map to 16 contiguous physical columns (the sum over K is
// order-free when A and B use the same map), so a lane reads 8 contiguous code
// bytes per row, all of one scale block.  On CUDA cores the same dequantised
// dot product costs 2-5 instructions per weight, above the issue budget at HBM
// speed; here it is about one.
//
// Streaming.  A task is one 16-row block of one group's matrix (gate/up: the
// gate rows and the matching up rows) for one block of 8 activation vectors
// over one K slice; its K range is cut into units of UC columns.  Every warp
// runs its own pipeline over the units of its tasks: each unit's code bytes,
// scale bytes and activation slice are copied by the warp's lanes into a
// private ring of shared-memory stages with cp.async (rows padded so the
// fragment reads are free of bank conflicts), three units ahead of the one
// being computed.  No barrier spans more than one warp.  With K slices, the
// slices' 16x8 partial tiles go to a scratch buffer and the last warp to finish
// a row block (arrival counter) adds them in slice order, so results do not
// depend on scheduling.
#include "internal.h"

namespace moe {

// ---------------------------------------------------------------- helpers
// 16 bits = codes of K slots (2t, 2t+1) in the low byte and (2t+8, 2t+9) in the
// high byte -> the two f16 pairs (exact).
__device__ __forceinline__ void e2m1_pair2(uint32_t two_bytes, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(two_bytes));
}
// One E4M3 scale byte -> the f16 pair (s, s) (exact).
__device__ __forceinline__ uint32_t scale_pair(uint32_t byte) { return e4m3x2_to_f16x2(byte | (byte << 8)); }
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_small(void* dst, const void* src) {  // N = 4 or 8
  asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src), "n"(N)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

struct DecodeArgs {
  const int32_t* num_groups;
  const int32_t* grp_off;
  const uint8_t* const* grp_blob;
  const int32_t* ent_tok;
  const int32_t* ent_pos;
  const __half* x16;     // [T, H] f16, x * xscale
  const float* xscale;   // [T]
  float* h;              // [(maxTk + maxT) * Imax]
  float* hmax;           // [maxTk + maxT] max|h| per row (float bits, atomicMax)
  float* o;              // [(maxTk + maxT) * H]
  const uint8_t* shared_blob;
  int T, H, I, I_s, Imax, maxTk;
  DevBlobLayout lay_r, lay_s;
  int l_nrb_r, l_nrb_s;  // log2 of the 16-row blocks of a routed / the shared matrix
  int l_ks_r, l_ks_s;    // log2 of the K slices per row block
  int l_nbp;             // log2 of the vector blocks per row block (ceil(T/8) rounded up to a power of two)
  int maxG;              // upper bound of the group count (scratch geometry)
  float* part;           // split-K partial tiles [row block][kMaxSlices][32 lanes][8]
  int* cnt;              // per row block arrival counters (zero between calls)
  int32_t* err;
};

constexpr int kWarpsPerCta = 8;
constexpr int kStages = 4;
constexpr int kMaxSlices = 8;
constexpr int kCodePad = 32;  // bytes after each code row of a stage
constexpr int kXPad = 16;     // bytes after each activation vector of a stage

// What the computing lanes need to know about the unit in a stage.  Written by
// the issuing lanes, read three units later.
struct __align__(16) UnitMeta {
  const uint8_t* blob;
  int task;  // -1: no unit
  int u, units, shared, g, rb, ks, e0, nv, jbase;
  int idx[8];  // per vector: token (gate/up) or output position (down)
};

template <bool GATEUP, int UC>
struct StageGeo {
  static constexpr int NM = GATEUP ? 2 : 1;
  static constexpr int XSZ = GATEUP ? 2 : 4;         // bytes per activation element
  static constexpr int CPR = UC / 32;                 // 16-byte code chunks per row
  static constexpr int CROW = UC / 2 + kCodePad;      // code row stride
  static constexpr int SROW = UC / 16;                // scale bytes per row
  static constexpr int XROW = UC * XSZ + kXPad;       // activation vector stride
  static constexpr int XCP = UC * XSZ / 16;           // 16-byte chunks per vector
  static constexpr int SCALES = NM * 16 * CROW;       // offset of the scales
  static constexpr int XS = SCALES + NM * 16 * SROW;  // offset of the activations
  static constexpr int BYTES = (XS + 8 * XROW + 127) / 128 * 128;
};

// GATEUP: input x (f16 [T,H]) -> h[entry row][r] = SiLU(gs_g*<Wg_r,x>) * gs_u*<Wu_r,x>, and max|h| per row
// !GATEUP: input h (fp32 rows, to f16 with a per-row power-of-two scale) -> o[position][r] = gs_d*<Wd_r,h>
// Task index = ((nbk * G + g) * NRB + rb) * KS + ks with power-of-two NRB and
// KS: the vector block outermost, so that the tasks of the first block -- the
// only non-empty one of a group of at most 8 vectors -- are consecutive and
// spread over every warp (warps take every nw-th task).  The shared expert's
// tasks, ((nbk * NRB_s + rb) * KS_s + ks), follow the routed ones.  A task
// covers C/KS columns in units of UC.
template <bool GATEUP, int UC>
__global__ void __launch_bounds__(kWarpsPerCta * 32, 1) k_expert_stream(DecodeArgs a) {
  pdl_trigger();
  pdl_wait();
  using SG = StageGeo<GATEUP, UC>;
  constexpr int NM = SG::NM;
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31, g8 = lane >> 2, t4 = lane & 3, wib = threadIdx.x >> 5;
  const int gw = blockIdx.x * kWarpsPerCta + wib, nw = gridDim.x * kWarpsPerCta;
  uint8_t* wbase = smem + size_t(wib) * (kStages * (SG::BYTES + sizeof(UnitMeta)));
  UnitMeta* meta = reinterpret_cast<UnitMeta*>(wbase + kStages * SG::BYTES);
  const int G = *a.num_groups;
  const int lgs_r = a.l_nrb_r + a.l_ks_r, lgs_s = a.l_nrb_s + a.l_ks_s;  // tasks per (block, group)
  const int per_block = G << lgs_r;                                     // routed tasks per vector block
  const int routed = per_block << a.l_nbp;
  const int ntask = routed + (a.shared_blob ? (1 << (lgs_s + a.l_nbp)) : 0);

  // ---- issue side: the warp's cursor over (task, unit); tasks without vectors are skipped
  int cur = gw, cu = 0;
  const uint8_t* i_blob = nullptr;
  int i_shared = 0, i_g = 0, i_rb = 0, i_ks = 0, i_e0 = 0, i_nv = 0, i_jbase = 0, i_units = 0, i_C = 0, i_idx = 0;
  auto load_task = [&]() {
    for (; cur < ntask; cur += nw) {
      int n, r;
      if (cur < routed) {
        const int nbk = cur / per_block;
        r = cur - nbk * per_block;
        i_shared = 0;
        i_g = r >> lgs_r;
        const int rest = r & ((1 << lgs_r) - 1);
        i_rb = rest >> a.l_ks_r;
        i_ks = rest & ((1 << a.l_ks_r) - 1);
        i_jbase = nbk * 8;
        i_e0 = a.grp_off[i_g];
        n = a.grp_off[i_g + 1] - i_e0;
        i_C = GATEUP ? a.H : a.I;
        i_units = (i_C >> a.l_ks_r) / UC;
      } else {
        r = cur - routed;
        i_shared = 1;
        i_g = G;
        const int rest = r & ((1 << lgs_s) - 1);
        i_rb = rest >> a.l_ks_s;
        i_ks = rest & ((1 << a.l_ks_s) - 1);
        i_jbase = (r >> lgs_s) * 8;
        i_e0 = 0;
        n = a.T;
        i_C = GATEUP ? a.H : a.I_s;
        i_units = (i_C >> a.l_ks_s) / UC;
      }
      if (i_jbase >= n) continue;
      i_nv = min(8, n - i_jbase);
      i_blob = i_shared ? a.shared_blob : a.grp_blob[i_g];
      // lanes 0..7 hold the index of vector `lane`: its token (gate/up) or output position (down)
      i_idx = 0;
      if (lane < i_nv) {
        const int jj = i_jbase + lane;
        i_idx = i_shared ? (GATEUP ? jj : a.maxTk + jj) : (GATEUP ? a.ent_tok[i_e0 + jj] : a.ent_pos[i_e0 + jj]);
      }
      return;
    }
  };
  load_task();

  auto issue = [&](int s) {
    uint8_t* st = wbase + s * SG::BYTES;
    UnitMeta& mt = meta[s];
    if (cur < ntask) {
      const int kcol = (i_ks * (i_C >> (i_shared ? a.l_ks_s : a.l_ks_r))) + cu * UC;
      const int code_row = i_C >> 1, scale_row = i_C >> 4;
      if (i_blob) {
        const DevBlobLayout& lay = i_shared ? a.lay_s : a.lay_r;
#pragma unroll
        for (int c = lane; c < NM * 16 * SG::CPR; c += 32) {
          const int m = c / (16 * SG::CPR), rr = (c / SG::CPR) % 16, q = c % SG::CPR;
          cp_async16(st + (m * 16 + rr) * SG::CROW + q * 16,
                     i_blob + lay.code_off[GATEUP ? m : 2] + size_t(i_rb * 16 + rr) * code_row + kcol / 2 + q * 16);
        }
        if (lane < NM * 16) {
          const int m = lane >> 4, rr = lane & 15;
          const uint8_t* src = i_blob + lay.scale_off[GATEUP ? m : 2] + size_t(i_rb * 16 + rr) * scale_row + kcol / 16;
          uint8_t* dst = st + SG::SCALES + (m * 16 + rr) * SG::SROW;
          if (SG::SROW == 8) cp_async_small<8>(dst, src);
          else cp_async_small<4>(dst, src);
        }
      }
#pragma unroll
      for (int c = lane; c < 8 * SG::XCP; c += 32) {
        const int v = c / SG::XCP, q = c % SG::XCP;
        const int idx = __shfl_sync(0xffffffffu, i_idx, v);
        if (v < i_nv) {
          const void* src;
          if (GATEUP) src = a.x16 + size_t(idx) * a.H + kcol + q * 8;
          else src = a.h + size_t(i_shared ? a.maxTk + i_jbase + v : i_e0 + i_jbase + v) * a.Imax + kcol + q * 4;
          cp_async16(st + SG::XS + v * SG::XROW + q * 16, src);
        }
      }
      if (lane == 0) {
        mt.blob = i_blob;
        mt.task = cur;
        mt.u = cu;
        mt.units = i_units;
        mt.shared = i_shared;
        mt.g = i_g;
        mt.rb = i_rb;
        mt.ks = i_ks;
        mt.e0 = i_e0;
        mt.nv = i_nv;
        mt.jbase = i_jbase;
      }
      if (lane < 8) mt.idx[lane] = i_idx;
      if (++cu == i_units) {
        cu = 0;
        cur += nw;
        load_task();
      }
    } else if (lane == 0) {
      mt.task = -1;
    }
    cp_async_commit();
  };

#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) issue(s);

  float acc[NM][4];
#pragma unroll
  for (int m = 0; m < NM; ++m)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[m][q] = 0.f;
  for (int i = 0;; ++i) {
    issue((i + kStages - 1) % kStages);
    cp_async_wait<kStages - 1>();
    __syncwarp();
    const int s = i % kStages;
    const UnitMeta& mt = meta[s];
    if (mt.task < 0) break;
    const int nv = mt.nv;
    const uint8_t* st = wbase + s * SG::BYTES;
    if (mt.blob) {
      float bsc = 1.f;  // down: power-of-two scale of this lane's vector
      if (!GATEUP && g8 < nv) bsc = pow2_scale_for(a.hmax[mt.shared ? a.maxTk + mt.jbase + g8 : mt.e0 + mt.jbase + g8]);
#pragma unroll
      for (int seg = 0; seg < UC / 64; ++seg) {
        // B fragments: vector g8, K slots of this lane = 16 contiguous columns
        uint32_t bx[8];
        if (g8 < nv) {
          if (GATEUP) {
            const uint4* p = reinterpret_cast<const uint4*>(st + SG::XS + g8 * SG::XROW + (seg * 64 + 16 * t4) * 2);
            const uint4 v0 = p[0], v1 = p[1];
            bx[0] = v0.x; bx[1] = v0.y; bx[2] = v0.z; bx[3] = v0.w;
            bx[4] = v1.x; bx[5] = v1.y; bx[6] = v1.z; bx[7] = v1.w;
          } else {
            const float4* p = reinterpret_cast<const float4*>(st + SG::XS + g8 * SG::XROW + (seg * 64 + 16 * t4) * 4);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const float4 f = p[v];
              __half2 h0 = __floats2half2_rn(f.x * bsc, f.y * bsc);
              __half2 h1 = __floats2half2_rn(f.z * bsc, f.w * bsc);
              bx[2 * v] = *reinterpret_cast<uint32_t*>(&h0);
              bx[2 * v + 1] = *reinterpret_cast<uint32_t*>(&h1);
            }
          }
        } else {
#pragma unroll
          for (int v = 0; v < 8; ++v) bx[v] = 0u;
        }
#pragma unroll
        for (int m = 0; m < NM; ++m) {
          const uint8_t* c0p = st + (m * 16 + g8) * SG::CROW + seg * 32 + 8 * t4;
          const uint2 c0 = *reinterpret_cast<const uint2*>(c0p);
          const uint2 c1 = *reinterpret_cast<const uint2*>(c0p + 8 * SG::CROW);
          const uint8_t* sp = st + SG::SCALES + (m * 16 + g8) * SG::SROW + seg * 4 + t4;
          const uint32_t sc0 = scale_pair(sp[0]), sc1 = scale_pair(sp[8 * SG::SROW]);
          const uint32_t w0[2] = {c0.x, c0.y}, w1[2] = {c1.x, c1.y};
#pragma unroll
          for (int kb = 0; kb < 4; ++kb) {
            uint32_t a0, a1, a2, a3;
            e2m1_pair2(w0[kb >> 1] >> (16 * (kb & 1)), a0, a2);  // row g: K slots 2t,2t+1 / 2t+8,2t+9
            e2m1_pair2(w1[kb >> 1] >> (16 * (kb & 1)), a1, a3);  // row g+8
            mma16816(acc[m], hmul2(a0, sc0), hmul2(a1, sc1), hmul2(a2, sc0), hmul2(a3, sc1), bx[2 * kb],
                     bx[2 * kb + 1]);
          }
        }
      }
    }
    const int u = mt.u, units = mt.units, shared = mt.shared, g = mt.g, rb = mt.rb, ks = mt.ks, e0 = mt.e0;
    const int jbase = mt.jbase;
    const uint8_t* blob = mt.blob;
    const int myidx0 = mt.idx[(2 * t4) & 7], myidx1 = mt.idx[(2 * t4 + 1) & 7];
    __syncwarp();  // the stage and its metadata are free for a later issue
    if (u != units - 1) continue;

    // ---- the task's last unit: split-K hand-off, then the rows
    const int KS = 1 << (shared ? a.l_ks_s : a.l_ks_r);
    bool finish = true;
    if (KS > 1) {
      const int grb = shared ? a.maxG * (1 << a.l_nrb_r) + rb : g * (1 << a.l_nrb_r) + rb;
      float* pp = a.part + ((size_t(grb) * kMaxSlices + ks) * 32 + lane) * 8;
#pragma unroll
      for (int m = 0; m < NM; ++m)
        reinterpret_cast<float4*>(pp)[m] = make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
      __threadfence();
      int old = 0;
      if (lane == 0) old = atomicAdd(a.cnt + grb, 1);
      old = __shfl_sync(0xffffffffu, old, 0);
      finish = old == KS - 1;
      if (finish) {
        __threadfence();
#pragma unroll
        for (int m = 0; m < NM; ++m)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[m][q] = 0.f;
        for (int k2 = 0; k2 < KS; ++k2) {
          const float* qp = a.part + ((size_t(grb) * kMaxSlices + k2) * 32 + lane) * 8;
#pragma unroll
          for (int m = 0; m < NM; ++m) {
            const float4 f = __ldcg(reinterpret_cast<const float4*>(qp) + m);
            acc[m][0] += f.x;
            acc[m][1] += f.y;
            acc[m][2] += f.z;
            acc[m][3] += f.w;
          }
        }
        if (lane == 0) a.cnt[grb] = 0;  // ready for the next call
      }
    }
    if (finish) {
      float gsc[NM];
#pragma unroll
      for (int m = 0; m < NM; ++m)
        gsc[m] = blob ? reinterpret_cast<const BlobHeader*>(blob)->gscale[GATEUP ? m : 2] : 0.f;
      const int row0 = rb * 16 + g8;
      float hm[2] = {0.f, 0.f};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int jloc = 2 * t4 + (q & 1);
        const int r = row0 + 8 * (q >> 1);
        if (jloc < nv) {
          const int jj = jbase + jloc;
          const int rowh = shared ? a.maxTk + jj : e0 + jj;  // h row of this vector
          const int idx = (q & 1) ? myidx1 : myidx0;
          if (GATEUP) {
            const float inv = 1.0f / a.xscale[idx];
            const float hv = blob ? silu_f32(acc[0][q] * inv * gsc[0]) * (acc[NM - 1][q] * inv * gsc[NM - 1]) : 0.f;
            a.h[size_t(rowh) * a.Imax + r] = hv;
            hm[q & 1] = fmaxf(hm[q & 1], fabsf(hv));
          } else {
            const float inv = 1.0f / pow2_scale_for(a.hmax[rowh]);
            a.o[size_t(idx) * a.H + r] = blob ? acc[0][q] * inv * gsc[0] : 0.f;
          }
        }
      }
      if (GATEUP) {
        // max|h| over the block's 16 rows per vector: one atomic per vector
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          hm[0] = fmaxf(hm[0], __shfl_xor_sync(0xffffffffu, hm[0], o));
          hm[1] = fmaxf(hm[1], __shfl_xor_sync(0xffffffffu, hm[1], o));
        }
        if (g8 == 0) {
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int jloc = 2 * t4 + q;
            if (jloc < nv) {
              const int jj = jbase + jloc;
              atomicMax(reinterpret_cast<unsigned int*>(a.hmax) + (shared ? a.maxTk + jj : e0 + jj),
                        __float_as_uint(hm[q]));
            }
          }
        }
      }
    }
#pragma unroll
    for (int m = 0; m < NM; ++m)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[m][q] = 0.f;
  }
  cp_async_wait_all();
}

// ----------------------------------------------------------------- combine
// y[t] = sigmoid(gate_logit_t) * s_t + sum_r w[t,r] * o[t*k + r], rank order.
__global__ void __launch_bounds__(256) k_combine(const float* __restrict__ o, const float* __restrict__ w,
                                                 const float* __restrict__ gate_logit, int has_shared, int T, int H,
                                                 int k, int maxTk, void* y, int y_is_fp32) {
  pdl_trigger();
  pdl_wait();
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  const int per_tok = H / 4;
  if (idx >= T * per_tok) return;
  const int t = idx / per_tok, c4 = idx - t * per_tok;
  const float4 acc = combine4<false>(o, w, gate_logit, has_shared != 0, t, c4, H, k, maxTk);
  if (y_is_fp32) {
    reinterpret_cast<float4*>(y)[size_t(t) * per_tok + c4] = acc;
  } else {
    __nv_bfloat162 p0 = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 p1 = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&p0);
    u.y = *reinterpret_cast<uint32_t*>(&p1);
    reinterpret_cast<uint2*>(y)[size_t(t) * per_tok + c4] = u;
  }
}

// ----------------------------------------------------------------- launchers
static int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

static DecodeArgs decode_args(const moe_layer_desc* d, int T, moe_ws* ws) {
  const moe_layer_shape& sh = d->s;
  DecodeArgs a;
  a.num_groups = ws->num_groups;
  a.grp_off = ws->grp_off;
  a.grp_blob = ws->grp_blob;
  a.ent_tok = ws->ent_tok;
  a.ent_pos = ws->ent_pos;
  a.x16 = ws->x16;
  a.xscale = ws->xscale;
  a.h = ws->h;
  a.hmax = ws->hmax;
  a.o = ws->o;
  const bool has_shared = sh.I_shared > 0 && d->shared_blob;
  a.shared_blob = has_shared ? reinterpret_cast<const uint8_t*>(d->shared_blob) : nullptr;
  a.T = T;
  a.H = sh.H;
  a.I = sh.I;
  a.I_s = has_shared ? sh.I_shared : 0;
  a.Imax = ws->s.I > ws->s.I_shared ? ws->s.I : ws->s.I_shared;
  a.maxTk = ws->maxT * ws->s.k;
  a.lay_r = dev_layout(sh.H, sh.I);
  a.lay_s = dev_layout(sh.H, has_shared ? sh.I_shared : sh.I);
  a.err = ws->error;
  a.part = ws->part;
  a.cnt = ws->cnt;
  return a;
}

static int log2i(int v) {
  int l = 0;
  while ((1 << (l + 1)) <= v) ++l;
  return l;
}

// K slices: only when every group fits one block of 8 vectors (T <= 8), then
// one slice per 512 columns (at most kMaxSlices).
static int slices_for(int C, int T) {
  if (T > 8) return 1;
  int ks = C / 512;
  if (ks > kMaxSlices) ks = kMaxSlices;
  return ks < 1 ? 1 : ks;
}

template <bool GATEUP, int UC>
static int launch_stream_uc(DecodeArgs a, cudaStream_t s) {
  using SG = StageGeo<GATEUP, UC>;
  const size_t smem = size_t(kWarpsPerCta) * kStages * (SG::BYTES + sizeof(UnitMeta));
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(k_expert_stream<GATEUP, UC>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
        cudaSuccess)
      return MOE_ECUDA;
    attr = true;
  }
  if (launch_pdl(k_expert_stream<GATEUP, UC>, dim3(num_sms()), dim3(kWarpsPerCta * 32), smem, s, a) != cudaSuccess)
    return MOE_ECUDA;
  return MOE_OK;
}

template <bool GATEUP>
static int launch_stream(const moe_layer_desc* d, int T, moe_ws* ws, cudaStream_t s) {
  DecodeArgs a = decode_args(d, T, ws);
  const int rows_r = GATEUP ? a.I : a.H, rows_s = GATEUP ? a.I_s : a.H;
  const int C_r = GATEUP ? a.H : a.I, C_s = GATEUP ? a.H : (a.I_s ? a.I_s : a.I);
  a.l_nrb_r = log2i(rows_r / 16);
  a.l_nrb_s = a.shared_blob ? log2i(rows_s / 16) : 0;
  int nbp = 1;
  while (nbp * 8 < T) nbp *= 2;
  a.l_nbp = log2i(nbp);
  a.maxG = T * d->s.k < d->s.E ? T * d->s.k : d->s.E;
  const int ks_r = slices_for(C_r, T), ks_s = slices_for(C_s, T);
  a.l_ks_r = log2i(ks_r);
  a.l_ks_s = log2i(ks_s);
  // one unit width per launch: 128 columns, or 64 when a matrix slice is narrower
  const int uc = (C_r / ks_r >= 128 && C_s / ks_s >= 128) ? 128 : 64;
  if ((ks_r > 1 || ks_s > 1) && size_t(a.maxG) * (size_t(1) << a.l_nrb_r) + (rows_s / 16) > ws->split_blocks)
    return MOE_EINVAL;
  return uc == 128 ? launch_stream_uc<GATEUP, 128>(a, s) : launch_stream_uc<GATEUP, 64>(a, s);
}

int launch_gateup_decode(const moe_layer_desc* d, int T, moe_ws* ws, cudaStream_t s) {
  const int rc = launch_gemv_decode(true, d, T, ws, s);
  return rc == kGemvNotApplicable ? launch_stream<true>(d, T, ws, s) : rc;
}

int launch_down_decode(const moe_layer_desc* d, int T, moe_ws* ws, cudaStream_t s) {
  const int rc = launch_gemv_decode(false, d, T, ws, s);
  return rc == kGemvNotApplicable ? launch_stream<false>(d, T, ws, s) : rc;
}

int launch_combine(const moe_layer_desc* d, void* y, int y_is_fp32, int T, moe_ws* ws, cudaStream_t s) {
  if (T <= 0) return MOE_OK;
  const moe_layer_shape& sh = d->s;
  const int has_shared = sh.I_shared > 0 && d->shared_blob ? 1 : 0;
  const int n = T * (sh.H / 4);
  if (launch_pdl(k_combine, dim3((n + 255) / 256), dim3(256), 0, s, ws->o, ws->topk_w, ws->gate_logit, has_shared, T,
                 sh.H, sh.k, ws->maxT * ws->s.k, y, y_is_fp32) != cudaSuccess)
    return MOE_ECUDA;
  return MOE_OK;
}

}  // namespace moe
