// Decode expert path: memory-bound GEMVs over the slot blobs, and the combine.
//
// Strata expert paths, "CPU 怎样把剩下的专家算完？": an expert computes gate and
// up, the activation, then the down projection; "路由以后，专家怎样分工？": each
// expert output is multiplied by its routing weight and summed, then the gated
// shared-expert contribution (same input) is added.  Qwen3.8-Flash-Next DGX
// Spark notes, "NVFP4 code 和 scale 如何反量化": weight = E2M1 code x E4M3 block
// scale (per 16) x FP32 global scale.
//
// Work unit: a warp owns a tile of rows of one group (or of the shared
// expert).  LPR = min(32, cols/32) lanes share a row; lane q of a row reads
// the row's 16-byte code chunks q, q+LPR, ... (32 codes each, two scale
// blocks) with 128-bit streaming loads, so RPW = 32/LPR rows run side by side.
// Codes become f16 pairs in registers (cvt e2m1x2); the activations of up to
// TC tokens sit in registers as f16 pairs (pre-scaled by a power of two);
// products accumulate in fp32 per 16-value block, are scaled by the block's
// E4M3 scale and summed in fp32.
#include "internal.h"

namespace moe {

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ldg_u16(const void* p) {
  unsigned short v;
  asm("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t word, uint32_t* o) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(word));
}

// acc[j] += sum over the chunk's 32 columns of w * x_j, for TC tokens.
template <int TC>
__device__ __forceinline__ void chunk_dot(uint4 cw, uint32_t sc2, const uint32_t (&xv)[TC][16], float (&acc)[TC]) {
  uint32_t w[16];
  e2m1x8_to_f16x2x4(cw.x, w + 0);
  e2m1x8_to_f16x2x4(cw.y, w + 4);
  e2m1x8_to_f16x2x4(cw.z, w + 8);
  e2m1x8_to_f16x2x4(cw.w, w + 12);
  const float2 s = f16x2_to_f32x2(e4m3x2_to_f16x2(sc2));
#pragma unroll
  for (int j = 0; j < TC; ++j) {
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int b = 0; b < 8; ++b) a0 = fma2_f16_f32(w[b], xv[j][b], a0);
#pragma unroll
    for (int b = 8; b < 16; ++b) a1 = fma2_f16_f32(w[b], xv[j][b], a1);
    acc[j] = fmaf(a0, s.x, acc[j]);
    acc[j] = fmaf(a1, s.y, acc[j]);
  }
}

struct DecodeArgs {
  const int32_t* num_groups;
  const int32_t* grp_off;
  const uint8_t* const* grp_blob;
  const int32_t* ent_tok;
  const int32_t* ent_pos;
  const __half* x16;   // [T, H]
  const float* xscale; // [T]
  float* h;            // [(maxTk + maxT) * Imax]
  float* o;            // [(maxTk + maxT) * H]
  const uint8_t* shared_blob;
  int T, H, I, I_s, Imax, maxTk;
  DevBlobLayout lay_r, lay_s;
  int rows_per_task;   // rows (or row pairs) per warp task
  int tasks_r, tasks_s;  // tasks per routed group / for the shared expert
  int32_t* err;
};

// Which group a task belongs to, its token count, weights and rows.
struct TaskInfo {
  const uint8_t* blob;
  int n, e0, shared, rows, r0, r1;
  const DevBlobLayout* lay;
};

__device__ __forceinline__ bool decode_task(const DecodeArgs& a, int task, int G, int rows_r, int rows_s, TaskInfo& ti) {
  if (task < G * a.tasks_r) {
    const int g = task / a.tasks_r, tile = task - g * a.tasks_r;
    ti.e0 = a.grp_off[g];
    ti.n = a.grp_off[g + 1] - ti.e0;
    ti.blob = a.grp_blob[g];
    ti.shared = 0;
    ti.rows = rows_r;
    ti.lay = &a.lay_r;
    ti.r0 = tile * a.rows_per_task;
  } else {
    const int tile = task - G * a.tasks_r;
    if (tile >= a.tasks_s) return false;
    ti.e0 = 0;
    ti.n = a.T;
    ti.blob = a.shared_blob;
    ti.shared = 1;
    ti.rows = rows_s;
    ti.lay = &a.lay_s;
    ti.r0 = tile * a.rows_per_task;
  }
  ti.r1 = min(ti.rows, ti.r0 + a.rows_per_task);
  return true;
}

// ------------------------------------------------------------------ gate/up
// h[row of entry][r] = SiLU(gs_g * <Wg[r], x>) * (gs_u * <Wu[r], x>)
template <int CPL, int TC>
__global__ void __launch_bounds__(256, 2) k_gateup(DecodeArgs a) {
  const int lane = threadIdx.x & 31;
  const int H = a.H;
  const int LPR = min(32, H / 32), RPW = 32 / LPR;
  const int q = lane % LPR, sub = lane / LPR;
  const int G = *a.num_groups;
  const int total = G * a.tasks_r + a.tasks_s;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const size_t code_row = H / 2, scale_row = H / 16;
  for (int task = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; task < total; task += nw) {
    TaskInfo ti;
    if (!decode_task(a, task, G, a.I, a.I_s, ti)) break;
    const uint8_t* gc = ti.blob ? ti.blob + ti.lay->code_off[0] : nullptr;
    const uint8_t* uc = ti.blob ? ti.blob + ti.lay->code_off[1] : nullptr;
    const uint8_t* gsc = ti.blob ? ti.blob + ti.lay->scale_off[0] : nullptr;
    const uint8_t* usc = ti.blob ? ti.blob + ti.lay->scale_off[1] : nullptr;
    float gs_g = 0.f, gs_u = 0.f;
    if (ti.blob) {
      const BlobHeader* hd = reinterpret_cast<const BlobHeader*>(ti.blob);
      gs_g = hd->gscale[0];
      gs_u = hd->gscale[1];
    }
    for (int j0 = 0; j0 < ti.n; j0 += TC) {
      uint32_t xv[CPL][TC][16];
      float inv_xs[TC];
      int hrow[TC];
#pragma unroll
      for (int j = 0; j < TC; ++j) {
        const bool ok = j0 + j < ti.n;
        const int tok = ok ? (ti.shared ? j0 + j : a.ent_tok[ti.e0 + j0 + j]) : 0;
        hrow[j] = ok ? (ti.shared ? a.maxTk + j0 + j : ti.e0 + j0 + j) : -1;
        inv_xs[j] = ok ? 1.0f / a.xscale[tok] : 0.f;
        const uint4* xr = reinterpret_cast<const uint4*>(a.x16 + size_t(tok) * H);
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
          const int c = q + LPR * i;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 t4 = ok ? xr[c * 4 + v] : make_uint4(0, 0, 0, 0);
            xv[i][j][4 * v + 0] = t4.x;
            xv[i][j][4 * v + 1] = t4.y;
            xv[i][j][4 * v + 2] = t4.z;
            xv[i][j][4 * v + 3] = t4.w;
          }
        }
      }
      for (int rs = ti.r0; rs < ti.r1; rs += RPW) {
        const int r = rs + sub;
        const bool rv = r < ti.r1 && ti.blob;
        float ag[TC], au[TC];
#pragma unroll
        for (int j = 0; j < TC; ++j) { ag[j] = 0.f; au[j] = 0.f; }
        if (rv) {
          uint4 cg[CPL], cu[CPL];
          uint32_t sg[CPL], su[CPL];
#pragma unroll
          for (int i = 0; i < CPL; ++i) {
            const int c = q + LPR * i;
            cg[i] = ldg_stream(gc + r * code_row + c * 16);
            cu[i] = ldg_stream(uc + r * code_row + c * 16);
            sg[i] = ldg_u16(gsc + r * scale_row + c * 2);
            su[i] = ldg_u16(usc + r * scale_row + c * 2);
          }
#pragma unroll
          for (int i = 0; i < CPL; ++i) {
            chunk_dot<TC>(cg[i], sg[i], xv[i], ag);
            chunk_dot<TC>(cu[i], su[i], xv[i], au);
          }
        }
#pragma unroll
        for (int j = 0; j < TC; ++j) {
          for (int o = LPR >> 1; o > 0; o >>= 1) {
            ag[j] += __shfl_xor_sync(0xffffffffu, ag[j], o);
            au[j] += __shfl_xor_sync(0xffffffffu, au[j], o);
          }
        }
        if (q == 0 && r < ti.r1) {
#pragma unroll
          for (int j = 0; j < TC; ++j) {
            if (hrow[j] >= 0) {
              const float g = ag[j] * inv_xs[j] * gs_g;
              const float u = au[j] * inv_xs[j] * gs_u;
              a.h[size_t(hrow[j]) * a.Imax + r] = ti.blob ? silu_f32(g) * u : 0.f;
            }
          }
        }
      }
    }
  }
}

// -------------------------------------------------------------------- down
// o[pos][r] = gs_d * <Wd[r], h_entry>; h enters as f16 with a per-entry
// power-of-two scale chosen from max|h_entry|.
template <int CPL, int TC>
__global__ void __launch_bounds__(256, 2) k_down(DecodeArgs a) {
  const int lane = threadIdx.x & 31;
  const int H = a.H;
  const int G = *a.num_groups;
  const int total = G * a.tasks_r + a.tasks_s;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  for (int task = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; task < total; task += nw) {
    TaskInfo ti;
    if (!decode_task(a, task, G, H, H, ti)) break;
    const int C = ti.shared ? a.I_s : a.I;  // contraction length
    const int LPR = min(32, C / 32), RPW = 32 / LPR;
    const int q = lane % LPR, sub = lane / LPR;
    const size_t code_row = C / 2, scale_row = C / 16;
    const uint8_t* dc = ti.blob ? ti.blob + ti.lay->code_off[2] : nullptr;
    const uint8_t* dsc = ti.blob ? ti.blob + ti.lay->scale_off[2] : nullptr;
    const float gs_d = ti.blob ? reinterpret_cast<const BlobHeader*>(ti.blob)->gscale[2] : 0.f;
    for (int j0 = 0; j0 < ti.n; j0 += TC) {
      uint32_t hv[CPL][TC][16];
      float inv_hs[TC];
      int orow[TC];
#pragma unroll
      for (int j = 0; j < TC; ++j) {
        const bool ok = j0 + j < ti.n;
        const int hr = ok ? (ti.shared ? a.maxTk + j0 + j : ti.e0 + j0 + j) : 0;
        orow[j] = ok ? (ti.shared ? a.maxTk + j0 + j : a.ent_pos[ti.e0 + j0 + j]) : -1;
        const float4* hp = reinterpret_cast<const float4*>(a.h + size_t(hr) * a.Imax);
        float m = 0.f;
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
          const int c = q + LPR * i;
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            float4 f = ok ? hp[c * 8 + v] : make_float4(0.f, 0.f, 0.f, 0.f);
            m = fmaxf(m, fmaxf(fmaxf(fabsf(f.x), fabsf(f.y)), fmaxf(fabsf(f.z), fabsf(f.w))));
          }
        }
        for (int o = LPR >> 1; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const float sc = pow2_scale_for(m);
        inv_hs[j] = 1.0f / sc;
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
          const int c = q + LPR * i;
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            float4 f = ok ? hp[c * 8 + v] : make_float4(0.f, 0.f, 0.f, 0.f);
            __half2 p0 = __floats2half2_rn(f.x * sc, f.y * sc);
            __half2 p1 = __floats2half2_rn(f.z * sc, f.w * sc);
            hv[i][j][2 * v + 0] = *reinterpret_cast<uint32_t*>(&p0);
            hv[i][j][2 * v + 1] = *reinterpret_cast<uint32_t*>(&p1);
          }
        }
      }
      for (int rs = ti.r0; rs < ti.r1; rs += RPW) {
        const int r = rs + sub;
        const bool rv = r < ti.r1 && ti.blob;
        float acc[TC];
#pragma unroll
        for (int j = 0; j < TC; ++j) acc[j] = 0.f;
        if (rv) {
          uint4 cw[CPL];
          uint32_t sw[CPL];
#pragma unroll
          for (int i = 0; i < CPL; ++i) {
            const int c = q + LPR * i;
            cw[i] = ldg_stream(dc + r * code_row + c * 16);
            sw[i] = ldg_u16(dsc + r * scale_row + c * 2);
          }
#pragma unroll
          for (int i = 0; i < CPL; ++i) chunk_dot<TC>(cw[i], sw[i], hv[i], acc);
        }
#pragma unroll
        for (int j = 0; j < TC; ++j)
          for (int o = LPR >> 1; o > 0; o >>= 1) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], o);
        if (q == 0 && r < ti.r1) {
#pragma unroll
          for (int j = 0; j < TC; ++j)
            if (orow[j] >= 0) a.o[size_t(orow[j]) * H + r] = ti.blob ? acc[j] * inv_hs[j] * gs_d : 0.f;
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
static int g_num_sms = 0;
static int num_sms() {
  if (!g_num_sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_num_sms <= 0) g_num_sms = 148;
  }
  return g_num_sms;
}

template <int CPL, int TC>
static void launch_gu(const DecodeArgs& a, int blocks, cudaStream_t s) {
  k_gateup<CPL, TC><<<blocks, 256, 0, s>>>(a);
}
template <int CPL, int TC>
static void launch_dn(const DecodeArgs& a, int blocks, cudaStream_t s) {
  k_down<CPL, TC><<<blocks, 256, 0, s>>>(a);
}

static int cpl_of(int cols) {
  const int chunks = cols / 32;
  return chunks <= 32 ? 1 : chunks / 32;
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

int launch_gateup_decode(const moe_layer_desc* d, int T, moe_ws* ws, cudaStream_t s) {
  DecodeArgs a = decode_args(d, T, ws);
  const int blocks = num_sms() * 2;
  // tasks of 8 rows (each a gate row and an up row)
  a.rows_per_task = 8;
  a.tasks_r = (a.I + a.rows_per_task - 1) / a.rows_per_task;
  a.tasks_s = a.I_s ? (a.I_s + a.rows_per_task - 1) / a.rows_per_task : 0;
  switch (cpl_of(a.H)) {
    case 1: launch_gu<1, 4>(a, blocks, s); break;
    case 2: launch_gu<2, 2>(a, blocks, s); break;
    case 4: launch_gu<4, 1>(a, blocks, s); break;
    default: return MOE_EINVAL;
  }
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

int launch_down_decode(const moe_layer_desc* d, int T, moe_ws* ws, cudaStream_t s) {
  DecodeArgs a = decode_args(d, T, ws);
  const int blocks = num_sms() * 2;
  // tasks of 16 output rows; contraction over I (routed) / I_s (shared)
  a.rows_per_task = 16;
  a.tasks_r = (a.H + a.rows_per_task - 1) / a.rows_per_task;
  a.tasks_s = a.I_s ? a.tasks_r : 0;
  const int cpl_d = cpl_of(a.I);
  if (a.I_s && cpl_of(a.I_s) != cpl_d) return MOE_EINVAL;
  switch (cpl_d) {
    case 1: launch_dn<1, 4>(a, blocks, s); break;
    case 2: launch_dn<2, 2>(a, blocks, s); break;
    case 4: launch_dn<4, 1>(a, blocks, s); break;
    default: return MOE_EINVAL;
  }
  MOE_LAUNCH_CHECK();
  return MOE_OK;
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
