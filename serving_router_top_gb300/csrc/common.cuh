// Internal definitions shared by the libmoe translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// ---------------------------------------------------------------- limits
constexpr int kMaxE = 1024;        // experts per layer (top-k keeps E/32 logits per lane)
constexpr int kMaxK = 32;          // experts per token
constexpr int kBarWords = 16;      // grid-barrier counter of the single-kernel decode (one 128-byte line)
constexpr int kStats = 5;          // lookup counters per layer: groups, hits, staged, missing, skipped
constexpr int kBlobHeader = 256;   // bytes before the first region of a blob
constexpr uint32_t kBlobMagic = 0x42454f4du;  // "MOEB"

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Slot blob: header, then codes of gate/up/down, then scales of gate/up/down.
// Matrix m in {0 gate [I x H], 1 up [I x H], 2 down [H x I]}; codes row-major
// [rows][cols/2] (low nibble = even column), scales row-major [rows][cols/16].
struct BlobLayout {
  size_t code_off[3], scale_off[3], bytes;
};

inline BlobLayout blob_layout(int H, int I) {
  BlobLayout L;
  size_t gu_codes = size_t(I) * H / 2, d_codes = size_t(H) * I / 2;
  size_t gu_sc = size_t(I) * H / 16, d_sc = size_t(H) * I / 16;
  size_t o = kBlobHeader;
  L.code_off[0] = o; o += align256(gu_codes);
  L.code_off[1] = o; o += align256(gu_codes);
  L.code_off[2] = o; o += align256(d_codes);
  L.scale_off[0] = o; o += align256(gu_sc);
  L.scale_off[1] = o; o += align256(gu_sc);
  L.scale_off[2] = o; o += align256(d_sc);
  o += 256;  // tail guard: bulk copies of a last partial 16-byte block never leave the blob
  L.bytes = o;
  return L;
}

struct BlobHeader {
  uint32_t magic, version;
  int32_t H, I;
  float gscale[3];
  uint32_t pad0;
};

// Device-side view of the same layout (offsets passed by value to kernels).
struct DevBlobLayout {
  uint32_t code_off[3], scale_off[3];
};
inline DevBlobLayout dev_layout(int H, int I) {
  BlobLayout L = blob_layout(H, I);
  DevBlobLayout d;
  for (int m = 0; m < 3; ++m) {
    d.code_off[m] = uint32_t(L.code_off[m]);
    d.scale_off[m] = uint32_t(L.scale_off[m]);
  }
  return d;
}

// ---------------------------------------------------------------- errors
// First error wins: a device error word starts at MOE_OK and takes the first
// non-zero code written.
__device__ __forceinline__ void set_error(int32_t* err, int code) {
  if (err) atomicCAS(err, MOE_OK, code);
}

// An L2 prefetch of the 128-byte line holding p (a hint: no data returns).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Adds one grouping's lookups to a layer's kStats counters.
__device__ __forceinline__ void add_stats(unsigned long long* st, int groups, int hit, int stg, int miss, int skip) {
  atomicAdd(st + 0, (unsigned long long)groups);
  atomicAdd(st + 1, (unsigned long long)hit);
  atomicAdd(st + 2, (unsigned long long)stg);
  atomicAdd(st + 3, (unsigned long long)miss);
  atomicAdd(st + 4, (unsigned long long)skip);
}

#define MOE_CUDA_TRY(expr)                   \
  do {                                       \
    cudaError_t e__ = (expr);                \
    if (e__ != cudaSuccess) return MOE_ECUDA; \
  } while (0)

#define MOE_LAUNCH_CHECK()                         \
  do {                                             \
    if (cudaGetLastError() != cudaSuccess) return MOE_ECUDA; \
  } while (0)

// ---------------------------------------------------------------- numerics
__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

// Two E2M1 codes (one byte; low nibble first) -> f16x2 (low half = even column).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t out;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(out) : "r"(byte));
  return out;
}

// Two E4M3 bytes (low byte first) -> f16x2; exact (E4M3 is a subset of f16).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t out;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(out) : "r"(two_bytes));
  return out;
}

__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t h2) {
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

// acc += a.lo*b.lo + a.hi*b.hi with f16 inputs and an fp32 accumulator
// (each product is exact in fp32; two roundings per call).
__device__ __forceinline__ float fma2_f16_f32(uint32_t a, uint32_t b, float acc) {
  asm("{\n\t.reg .f16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.f16 %0, al, bl, %0;\n\t"
      "fma.rn.f32.f16 %0, ah, bh, %0;\n\t}"
      : "+f"(acc)
      : "r"(a), "r"(b));
  return acc;
}

// SiLU and the logistic function with the fast divide (within 2 ulp; a divisor
// above 2^126 gives 0, which is also the limit there): the IEEE divide's
// branchy sequence would serialise an epilogue that evaluates many at once.
__device__ __forceinline__ float silu_f32(float z) { return __fdividef(z, 1.0f + __expf(-z)); }
__device__ __forceinline__ float sigmoid_f32(float z) { return __fdividef(1.0f, 1.0f + __expf(-z)); }

// Power-of-two scale that brings max|v| into [2^12, 2^13): values become f16
// without overflow, products with an E2M1 value (|.| <= 6) stay below 2^16.
__device__ __forceinline__ float pow2_scale_for(float amax) {
  if (!(amax > 0.f) || !isfinite(amax)) return 1.0f;
  int e;
  frexpf(amax, &e);            // amax = m * 2^e, m in [0.5, 1)
  return ldexpf(1.0f, 13 - e);  // amax * 2^(13-e) in [2^12, 2^13)
}

// y[t] cols 4c4..4c4+3 = sum_r w[t,r] * o[t*k + r] (rank order) + sigmoid(g_t) * o[shared t].
// The shared row counts as row k; the rows' loads (and their coefficients) are issued
// sixteen at a time before any is used, so up to 15 routed rows and the shared one take a
// single round trip.  The multiply-adds keep the rank order, the shared term last.
template <bool LDCG>
__device__ __forceinline__ float4 combine4(const float* o, const float* w, const float* gate_logit, bool has_shared,
                                           int t, int c4, int H, int k, int maxTk) {
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const int nrow = k + (has_shared ? 1 : 0);
  for (int r0 = 0; r0 < nrow; r0 += 16) {
    float4 v[16];
    float c[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int r = r0 + j;
      if (r < nrow) {
        const size_t row = r < k ? size_t(t * k + r) : size_t(maxTk + t);
        const float4* p = reinterpret_cast<const float4*>(o + row * H) + c4;
        v[j] = LDCG ? __ldcg(p) : *p;
        c[j] = r < k ? w[t * k + r] : gate_logit[t];
      }
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int r = r0 + j;
      if (r < nrow) {
        const float cf = r < k ? c[j] : sigmoid_f32(c[j]);
        acc.x = fmaf(cf, v[j].x, acc.x);
        acc.y = fmaf(cf, v[j].y, acc.y);
        acc.z = fmaf(cf, v[j].z, acc.z);
        acc.w = fmaf(cf, v[j].w, acc.w);
      }
    }
  }
  return acc;
}

// ---------------------------------------------------------------- launches
// Programmatic dependent launch: every hot-path kernel lets its successor be
// scheduled as soon as all of its own CTAs are running (pdl_trigger at entry)
// and waits for its predecessor's grid to complete -- with its memory visible
// -- before reading anything the predecessor may have written (pdl_wait).
// Launch latency of the chain is hidden; data order is unchanged.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace moe

// ---------------------------------------------------------------- opaque handles
struct moe_cache {
  int L, E, H, I, nslots, nstaging;
  size_t blob_bytes;
  const void* backing;        // device pointer usable by kernels (device memory or mapped host)
  int backing_on_device;
  int32_t* resid;             // [L*E]
  int32_t* stage;             // [L*E]
  float* heat;                // [L*E]
  int32_t* slot_owner;        // [nslots]
  int32_t* staging_owner;     // [nstaging]
  uint8_t* slots;             // nslots * blob_bytes
  uint8_t* staging;           // nstaging * blob_bytes
  unsigned long long* stats;  // [L][kStats]
  uint32_t* lru_tick;         // [nslots] global LRU: the clock value of each slot's last use (0: never)
  uint32_t* lru_clock;        // [1] global LRU: layer calls planned so far
  int32_t* plan_keys_scratch; // policy scratch (candidates), allocated at creation
  void* plan_scratch;
  size_t plan_scratch_bytes;
  cudaEvent_t ev_unmapped, ev_copied;
  cudaEvent_t ev_ring[5];     // streamed prefill: copied[2], used[2], start
  int next_free_slot, next_free_staging;
};

struct moe_ws {
  int maxT;
  moe_layer_shape s;
  // routing
  float* logits;        // [maxT, E]
  int32_t* topk_ids;    // [maxT, k]
  float* topk_w;        // [maxT, k]
  float* gate_logit;    // [maxT] shared-expert gate logits
  // groups
  int32_t* num_groups;  // [1]
  int32_t* grp_expert;  // [maxT*k]
  int32_t* grp_off;     // [maxT*k + 1]
  int32_t* grp_slot;    // [maxT*k]
  int32_t* grp_src;     // [maxT*k]
  const uint8_t** grp_blob;  // [maxT*k] resolved blob pointer (NULL when missing)
  int32_t* ent_tok;     // [maxT*k]
  int32_t* ent_pos;     // [maxT*k]
  // activations
  __half* x16;          // [maxT, H] x times a per-token power of two, f16
  float* xscale;        // [maxT] that power of two
  float* h;             // [maxT*k + maxT, max(I, I_shared)] routed entries then shared rows
  float* hmax;          // [maxT*k + maxT] max|h| per row
  int32_t* tile_off;    // [E + 2] prefill: N tiles before each group
  int32_t* tile_grp;    // [E + maxT*k/128 + 2] prefill: group of each N tile
  int32_t* grange;      // [2E + 2] streamed prefill: the group range of each unit
  __half* h16;          // [maxT*k + maxT, max(I, I_shared)] prefill: h as f16 times a per-row power of two
  float* yacc;          // [maxT, H] prefill: fp32 output accumulator
  __half* xg;           // [maxT*k + maxT, H] prefill: gate/up B rows, f16 x 2^p (in the o region, unused
                        // by prefill)
  float* xinv;          // [maxT*k + maxT] prefill: 2^-p of each xg row
  float* part;          // split-K partial tiles: [split_blocks][8 slices][32 lanes][8]
  int* cnt;             // [split_blocks] arrival counters, zero between calls
  size_t split_blocks;
  float* o;             // [maxT*k + maxT, H] routed outputs by position, then shared outputs
  int32_t* grp_scratch; // [(maxT/256 + 1) * E + E] grouping of long windows: per-tile counts, offsets
  int32_t* error;       // [1]
  unsigned long long* bar;  // [kBarWords] grid-barrier arrivals of the single-kernel decode (zero at creation)
  unsigned bar_extra;   // arrivals that barrier waits for beyond the grid (0; a fault-injection hook for tests)
  unsigned long long wait_ns;  // bound of each grid-barrier wait
  int decode_path;      // MOE_DECODE_FUSED or MOE_DECODE_CHAIN
  int fused_heat;       // groupings with a cache also add the window's counts to the layer's heat
  int tail_skip;        // groupings drop non-resident experts ranked at or past this by all choosers (0: off)
  // optional per-kernel timing of the most recent call
  int prof_on, prof_n;
  cudaEvent_t prof_ev[2 * 16];
  const char* prof_name[16];
};

namespace moe {
// Brackets one kernel launch with events when the workspace profiles.
struct ProfScope {
  moe_ws* ws;
  int idx;
  cudaStream_t s;
  // Inside stream capture the records become external event nodes of the graph,
  // so the times stay readable after each replay.
  static void record(cudaEvent_t e, cudaStream_t st) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing(st, &cs);
    if (cs == cudaStreamCaptureStatusActive)
      cudaEventRecordWithFlags(e, st, cudaEventRecordExternal);
    else
      cudaEventRecord(e, st);
  }
  ProfScope(moe_ws* w, const char* name, cudaStream_t st) : ws(w), idx(-1), s(st) {
    if (ws && ws->prof_on && ws->prof_n < 16) {
      idx = ws->prof_n++;
      ws->prof_name[idx] = name;
      record(ws->prof_ev[2 * idx], s);
    }
  }
  ~ProfScope() {
    if (idx >= 0) record(ws->prof_ev[2 * idx + 1], s);
  }
};
}  // namespace moe
