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
// dot product costs 2-5 instructions per weight, above the issue budget at
// HBM speed; here it is about one.
#include "internal.h"

namespace moe {

// ---------------------------------------------------------------- helpers
// Two E2M1 codes (one byte, low nibble first) -> f16 pair (exact).
__device__ __forceinline__ uint32_t cvt_e2m1x2(uint32_t byte) {
  uint32_t out;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(out) : "r"(byte));
  return out;
}
// 16 bits = codes of K slots (2t, 2t+1) in the low byte and (2t+8, 2t+9) in the
// high byte -> the two f16 pairs.
__device__ __forceinline__ void e2m1_pair2(uint32_t two_bytes, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(two_bytes));
}
__device__ __forceinline__ uint2 ldg_stream_u2(const void* p) {
  uint2 v;
  asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldg_u8(const void* p) {
  unsigned short v;
  asm("ld.global.nc.u8 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
constexpr int kMaxSlices = 8;
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
  int nrb_r, nrb_s;      // 16-row blocks of a routed / the shared matrix
  int ks_r, ks_s;        // K slices per row block
  int ks_max, maxG;      // scratch geometry
  float* part;           // split-K partial tiles
  int* cnt;              // per row block arrival counters (zero between calls)
  int32_t* err;
};

// Work split.  A task is one 16-row block of one group's matrix (gate/up: the
// gate rows and the matching up rows) over one K slice of C/KS columns; warps
// take tasks independently (grid-stride).  Each lane loads its 8 code bytes
// of rows g and g+8 per 64-column segment straight from the slot blob (64-bit
// loads; the four lanes of a row read 32 contiguous bytes), four segments at
// a time before any math.  With KS > 1 the slices' 16x8 partial tiles go to a
// scratch buffer and the last warp to finish a row block (arrival counter)
// adds them in slice order and writes the rows, so results do not depend on
// scheduling.
struct GemvTask {
  const uint8_t* blob;
  int shared, g, rb, ks, KS, C, n, e0;
};

__device__ __forceinline__ bool gemv_task(const DecodeArgs& a, bool gateup, int task, int G, GemvTask& t) {
  const int routed = G * a.nrb_r * a.ks_r;
  if (task < routed) {
    t.shared = 0;
    t.ks = task % a.ks_r;
    const int grb = task / a.ks_r;
    t.g = grb / a.nrb_r;
    t.rb = grb - t.g * a.nrb_r;
    t.KS = a.ks_r;
    t.blob = a.grp_blob[t.g];
    t.C = gateup ? a.H : a.I;
    t.e0 = a.grp_off[t.g];
    t.n = a.grp_off[t.g + 1] - t.e0;
    return true;
  }
  const int st = task - routed;
  if (st >= a.nrb_s * a.ks_s) return false;
  t.shared = 1;
  t.ks = st % a.ks_s;
  t.rb = st / a.ks_s;
  t.g = G;
  t.KS = a.ks_s;
  t.blob = a.shared_blob;
  t.C = gateup ? a.H : a.I_s;
  t.e0 = 0;
  t.n = a.T;
  return true;
}

constexpr int kSegUnroll = 4;

// GATEUP: input x (f16 [T,H]) -> h[entry row][r] = SiLU(gs_g*<Wg_r,x>) * gs_u*<Wu_r,x>, and max|h| per row
// !GATEUP: input h (fp32 rows, to f16 with a per-row power-of-two scale) -> o[position][r] = gs_d*<Wd_r,h>
template <bool GATEUP>
__global__ void __launch_bounds__(256, 2) k_expert_gemv(DecodeArgs a) {
  constexpr int NM = GATEUP ? 2 : 1;
  const int lane = threadIdx.x & 31, g8 = lane >> 2, t4 = lane & 3;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const int G = *a.num_groups;
  const int total = G * a.nrb_r * a.ks_r + a.nrb_s * a.ks_s;
  for (int task = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; task < total; task += nwarps) {
    GemvTask tk;
    if (!gemv_task(a, GATEUP, task, G, tk)) break;
    const DevBlobLayout& lay = tk.shared ? a.lay_s : a.lay_r;
    const int code_row = tk.C / 2, scale_row = tk.C / 16;
    const int segs = tk.C / (64 * tk.KS), seg0 = tk.ks * segs;
    const int row0 = tk.rb * 16 + g8;  // this lane's rows: row0 and row0 + 8
    const uint8_t* cp[NM];
    const uint8_t* sp[NM];
    float gsc[NM];
#pragma unroll
    for (int m = 0; m < NM; ++m) {
      const int mi = GATEUP ? m : 2;
      cp[m] = tk.blob ? tk.blob + lay.code_off[mi] + size_t(row0) * code_row + 8 * t4 : nullptr;
      sp[m] = tk.blob ? tk.blob + lay.scale_off[mi] + size_t(row0) * scale_row + t4 : nullptr;
      gsc[m] = tk.blob ? reinterpret_cast<const BlobHeader*>(tk.blob)->gscale[mi] : 0.f;
    }
    const int nblocks = (tk.n + 7) >> 3;
    for (int nb = 0; nb < nblocks; ++nb) {
      const int nv = min(8, tk.n - nb * 8);
      // the activation vector this lane feeds to B: vector nb*8 + g8 of the group
      const bool bvalid = g8 < nv;
      const void* brow = nullptr;
      float bscale = 1.f;
      if (bvalid) {
        const int jj = nb * 8 + g8;
        if (GATEUP) {
          const int tok = tk.shared ? jj : a.ent_tok[tk.e0 + jj];
          brow = a.x16 + size_t(tok) * a.H;
        } else {
          const int hr = tk.shared ? a.maxTk + jj : tk.e0 + jj;
          brow = a.h + size_t(hr) * a.Imax;
          bscale = pow2_scale_for(a.hmax[hr]);
        }
      }
      float acc[NM][4];
#pragma unroll
      for (int m = 0; m < NM; ++m)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[m][q] = 0.f;
      if (tk.blob) {
        for (int s0 = 0; s0 < segs; s0 += kSegUnroll) {
          uint2 cw[kSegUnroll][NM][2];
          uint32_t sw[kSegUnroll][NM][2];
          uint32_t bx[kSegUnroll][8];
#pragma unroll
          for (int u = 0; u < kSegUnroll; ++u) {
            const int seg = seg0 + s0 + u;
            const bool ok = s0 + u < segs;
#pragma unroll
            for (int m = 0; m < NM; ++m) {
              cw[u][m][0] = ok ? ldg_stream_u2(cp[m] + seg * 32) : make_uint2(0, 0);
              cw[u][m][1] = ok ? ldg_stream_u2(cp[m] + size_t(8) * code_row + seg * 32) : make_uint2(0, 0);
              sw[u][m][0] = ok ? ldg_u8(sp[m] + seg * 4) : 0u;
              sw[u][m][1] = ok ? ldg_u8(sp[m] + size_t(8) * scale_row + seg * 4) : 0u;
            }
            if (ok && bvalid) {
              if (GATEUP) {
                const uint4* p = reinterpret_cast<const uint4*>(static_cast<const __half*>(brow) + seg * 64 + 16 * t4);
                const uint4 v0 = p[0], v1 = p[1];
                bx[u][0] = v0.x; bx[u][1] = v0.y; bx[u][2] = v0.z; bx[u][3] = v0.w;
                bx[u][4] = v1.x; bx[u][5] = v1.y; bx[u][6] = v1.z; bx[u][7] = v1.w;
              } else {
                const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(brow) + seg * 64 + 16 * t4);
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                  const float4 f = p[v];
                  __half2 h0 = __floats2half2_rn(f.x * bscale, f.y * bscale);
                  __half2 h1 = __floats2half2_rn(f.z * bscale, f.w * bscale);
                  bx[u][2 * v] = *reinterpret_cast<uint32_t*>(&h0);
                  bx[u][2 * v + 1] = *reinterpret_cast<uint32_t*>(&h1);
                }
              }
            } else {
#pragma unroll
              for (int v = 0; v < 8; ++v) bx[u][v] = 0u;
            }
          }
#pragma unroll
          for (int u = 0; u < kSegUnroll; ++u) {
            if (s0 + u < segs) {
#pragma unroll
              for (int m = 0; m < NM; ++m) {
                const uint32_t sc0 = scale_pair(sw[u][m][0]), sc1 = scale_pair(sw[u][m][1]);
                const uint32_t w0[2] = {cw[u][m][0].x, cw[u][m][0].y}, w1[2] = {cw[u][m][1].x, cw[u][m][1].y};
#pragma unroll
                for (int kb = 0; kb < 4; ++kb) {
                  uint32_t a0, a1, a2, a3;
                  e2m1_pair2(w0[kb >> 1] >> (16 * (kb & 1)), a0, a2);  // row g: K slots 2t,2t+1 / 2t+8,2t+9
                  e2m1_pair2(w1[kb >> 1] >> (16 * (kb & 1)), a1, a3);  // row g+8
                  mma16816(acc[m], hmul2(a0, sc0), hmul2(a1, sc1), hmul2(a2, sc0), hmul2(a3, sc1), bx[u][2 * kb],
                           bx[u][2 * kb + 1]);
                }
              }
            }
          }
        }
      }
      // ---- split-K: leave the partial, the last slice of the row block finishes it
      bool finish = true;
      if (tk.KS > 1) {
        const int grb = tk.shared ? a.maxG * a.nrb_r + tk.rb : tk.g * a.nrb_r + tk.rb;
        float* pp = a.part + ((size_t(grb) * a.ks_max + tk.ks) * 32 + lane) * 8;
#pragma unroll
        for (int m = 0; m < NM; ++m)
          reinterpret_cast<float4*>(pp)[m] = make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
        __threadfence();
        int old = 0;
        if (lane == 0) old = atomicAdd(a.cnt + grb, 1);
        old = __shfl_sync(0xffffffffu, old, 0);
        finish = old == tk.KS - 1;
        if (finish) {
          __threadfence();
#pragma unroll
          for (int m = 0; m < NM; ++m)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[m][q] = 0.f;
          for (int s = 0; s < tk.KS; ++s) {
            const float* qp = a.part + ((size_t(grb) * a.ks_max + s) * 32 + lane) * 8;
#pragma unroll
            for (int m = 0; m < NM; ++m) {
              const float4 f = __ldcg(reinterpret_cast<const float4*>(qp) + m);
              acc[m][0] += f.x; acc[m][1] += f.y; acc[m][2] += f.z; acc[m][3] += f.w;
            }
          }
          if (lane == 0) a.cnt[grb] = 0;  // ready for the next call
        }
      }
      if (!finish) continue;
      // ---- epilogue: lane holds rows row0, row0+8 x vectors nb*8 + 2*t4 + {0, 1}
      float hm[2] = {0.f, 0.f};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int jloc = 2 * t4 + (q & 1);
        const int r = row0 + 8 * (q >> 1);
        if (jloc < nv) {
          const int jj = nb * 8 + jloc;
          if (GATEUP) {
            const int tok = tk.shared ? jj : a.ent_tok[tk.e0 + jj];
            const float inv = 1.0f / a.xscale[tok];
            const int hrow = tk.shared ? a.maxTk + jj : tk.e0 + jj;
            const float hv = tk.blob ? silu_f32(acc[0][q] * inv * gsc[0]) * (acc[NM - 1][q] * inv * gsc[NM - 1]) : 0.f;
            a.h[size_t(hrow) * a.Imax + r] = hv;
            hm[q & 1] = fmaxf(hm[q & 1], fabsf(hv));
          } else {
            const int hr = tk.shared ? a.maxTk + jj : tk.e0 + jj;
            const float inv = 1.0f / pow2_scale_for(a.hmax[hr]);
            const int orow = tk.shared ? a.maxTk + jj : a.ent_pos[tk.e0 + jj];
            a.o[size_t(orow) * a.H + r] = tk.blob ? acc[0][q] * inv * gsc[0] : 0.f;
          }
        }
      }
      if (GATEUP) {
        // max|h| over the 16 rows of the block per vector, one atomic per vector
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
              const int jj = nb * 8 + jloc;
              const int hrow = tk.shared ? a.maxTk + jj : tk.e0 + jj;
              atomicMax(reinterpret_cast<unsigned int*>(a.hmax) + hrow, __float_as_uint(hm[q]));
            }
          }
        }
      }
    }
  }
}

// ----------------------------------------------------------------- combine
// y[t] = sigmoid(gate_logit_t) * s_t + sum_r w[t,r] * o[t*k + r], rank order.
__global__ void __launch_bounds__(256) k_combine(const float* __restrict__ o, const float* __restrict__ w,
                                                 const float* __restrict__ gate_logit, int has_shared, int T, int H,
                                                 int k, int maxTk, void* y, int y_is_fp32) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  const int per_tok = H / 4;
  if (idx >= T * per_tok) return;
  const int t = idx / per_tok, c4 = idx - t * per_tok;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int r = 0; r < k; ++r) {
    const float wr = w[t * k + r];
    const float4 v = reinterpret_cast<const float4*>(o + size_t(t * k + r) * H)[c4];
    acc.x = fmaf(wr, v.x, acc.x);
    acc.y = fmaf(wr, v.y, acc.y);
    acc.z = fmaf(wr, v.z, acc.z);
    acc.w = fmaf(wr, v.w, acc.w);
  }
  if (has_shared) {
    const float gm = sigmoid_f32(gate_logit[t]);
    const float4 s = reinterpret_cast<const float4*>(o + size_t(maxTk + t) * H)[c4];
    acc.x = fmaf(gm, s.x, acc.x);
    acc.y = fmaf(gm, s.y, acc.y);
    acc.z = fmaf(gm, s.z, acc.z);
    acc.w = fmaf(gm, s.w, acc.w);
  }
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
  return a;
}

static int pow2_floor(int v) {
  int p = 1;
  while (p * 2 <= v) p *= 2;
  return p;
}

// Slices per row block: enough tasks for about four per warp, each slice at
// least 256 columns.
static int pick_ks(int C, int row_blocks, int nwarps) {
  int ks = pow2_floor((4 * nwarps) / (row_blocks > 0 ? row_blocks : 1));
  const int cap = C / 256 > 0 ? C / 256 : 1;
  if (ks > cap) ks = cap;
  if (ks > kMaxSlices) ks = kMaxSlices;
  return ks < 1 ? 1 : ks;
}

template <bool GATEUP>
static int launch_gemv(const moe_layer_desc* d, int T, moe_ws* ws, cudaStream_t s) {
  DecodeArgs a = decode_args(d, T, ws);
  const int rows_r = GATEUP ? a.I : a.H, rows_s = GATEUP ? a.I_s : a.H;
  a.nrb_r = rows_r / 16;
  a.nrb_s = a.shared_blob ? rows_s / 16 : 0;
  a.maxG = T * d->s.k < d->s.E ? T * d->s.k : d->s.E;
  const int blocks = num_sms() * 2;
  const int nwarps = blocks * 8;
  const int C_r = GATEUP ? a.H : a.I, C_s = GATEUP ? a.H : (a.I_s ? a.I_s : a.I);
  // K is split only when every group fits one block of 8 vectors (T <= 8): the
  // partial scratch and counters are per row block, not per vector block
  a.ks_r = T <= 8 ? pick_ks(C_r, a.maxG * a.nrb_r + a.nrb_s, nwarps) : 1;
  a.ks_s = T <= 8 && a.shared_blob ? pick_ks(C_s, a.maxG * a.nrb_r + a.nrb_s, nwarps) : 1;
  a.ks_max = kMaxSlices;
  // slices only exist when row blocks are few (at most two per warp), so the
  // scratch sized for that bound always holds them
  if ((a.ks_r > 1 || a.ks_s > 1) && size_t(a.maxG * a.nrb_r + a.nrb_s) > ws->split_blocks) return MOE_EINVAL;
  a.part = ws->part;
  a.cnt = ws->cnt;
  k_expert_gemv<GATEUP><<<blocks, 256, 0, s>>>(a);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

int launch_gateup_decode(const moe_layer_desc* d, int T, moe_ws* ws, cudaStream_t s) {
  return launch_gemv<true>(d, T, ws, s);
}

int launch_down_decode(const moe_layer_desc* d, int T, moe_ws* ws, cudaStream_t s) {
  return launch_gemv<false>(d, T, ws, s);
}

int launch_combine(const moe_layer_desc* d, void* y, int y_is_fp32, int T, moe_ws* ws, cudaStream_t s) {
  if (T <= 0) return MOE_OK;
  const moe_layer_shape& sh = d->s;
  const int has_shared = sh.I_shared > 0 && d->shared_blob ? 1 : 0;
  const int n = T * (sh.H / 4);
  k_combine<<<(n + 255) / 256, 256, 0, s>>>(ws->o, ws->topk_w, ws->gate_logit, has_shared, T, sh.H, sh.k,
                                           ws->maxT * ws->s.k, y, y_is_fp32);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

}  // namespace moe
