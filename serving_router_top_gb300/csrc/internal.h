// Kernel launchers shared between libmoe translation units (not part of the ABI).
#pragma once
#include "common.cuh"

namespace moe {

int launch_router(const uint16_t* x, const uint16_t* w_router, const float* bias, const uint16_t* w_gate,
                  float* logits, float* gate_logit, int T, int H, int E, cudaStream_t s, __half* x16 = nullptr,
                  float* xscale = nullptr);
int launch_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w, int32_t* err, cudaStream_t s);

constexpr int kNotFused = -2;
int launch_topk_group(const float* logits, int T, int k, int E, int layer, moe_cache* c, moe_ws* ws, cudaStream_t s);
// lookup = false: the groups' sources are left for the caller to bind (streamed prefill)
int launch_group(const int32_t* ids, int T, int k, int E, int layer, moe_cache* c, moe_ws* ws, cudaStream_t s,
                 bool lookup = true);

// Decode expert path (GEMVs over the slot blobs, mma.sync on the tensor cores).
int launch_gateup_decode(const moe_layer_desc* d, int T, moe_ws* ws, cudaStream_t s);
int launch_down_decode(const moe_layer_desc* d, int T, moe_ws* ws, cudaStream_t s);
int launch_combine(const moe_layer_desc* d, void* y, int y_is_fp32, int T, moe_ws* ws, cudaStream_t s);
// Decode GEMVs for windows of at most 8 tokens (every warp streams weight rows into registers).
constexpr int kGemvNotApplicable = -1;
int launch_gemv_decode(bool gateup, const moe_layer_desc* d, int T, moe_ws* ws, cudaStream_t s);

// The whole decode forward as one cooperative kernel (router, top-k, groups and
// lookup, gate/up, down, combine); kNotFused when the shapes call for the chain.
int launch_decode_fused(const moe_layer_desc* d, moe_cache* c, const uint16_t* x, void* y, int y_is_fp32, int T,
                        moe_ws* ws, cudaStream_t s);

// Activation rows -> R NVFP4 terms (codes [rows*R][K/2], scales [rows*R][K/16], global
// scales [rows*R]); rows bf16 (src_is_fp32 = 0) or fp32, ld elements apart.
int launch_split_nvfp4(const void* src, int src_is_fp32, int rows, int K, int ld, int R, uint8_t* codes,
                       uint8_t* scales, float* gscale, cudaStream_t s);

// Prefill path (tcgen05 GEMMs): router logits and gate logit, then the
// experts, which write y directly.  x rows must be 16-byte aligned.
bool prefill_supported(const moe_layer_shape& s);
int launch_prefill_router(const moe_layer_desc* d, const uint16_t* x, int T, moe_ws* ws, cudaStream_t s);
int launch_prefill_experts(const moe_layer_desc* d, const moe_cache* c, const uint16_t* x, void* y, int y_is_fp32, int T,
                           moe_ws* ws, cudaStream_t s);
int launch_prefill_streamed(const moe_layer_desc* d, moe_cache* c, const uint16_t* x, void* y, int y_is_fp32, int T,
                            int U, int buffers, moe_ws* ws, cudaStream_t s, cudaStream_t cs);
int launch_prefill_layers_streamed(const moe_layer_desc* d, int L, float* x_res, uint16_t* xn, uint16_t* y, int T,
                                   moe_cache* c, moe_ws* ws, int buffers, float eps, cudaStream_t s,
                                   cudaStream_t cs);

// Policy.
int launch_heat_update(moe_cache* c, const int32_t* ids, int T, int k, int layer, int32_t* err, cudaStream_t s);
int launch_plan_swaps(moe_cache* c, const moe_policy_cfg* p, moe_swap* plan, int32_t* n, cudaStream_t s);
// flat_cold: the plan's cold_expert is the evicted expert's layer * E + expert
// (-1: an empty slot), as global LRU plans write it.
int launch_apply_swaps(moe_cache* c, const moe_swap* plan, const int32_t* n, int max_swaps, cudaStream_t compute,
                       cudaStream_t copy, bool flat_cold = false);
// Global LRU: refresh the last call's hits and plan its admissions (k_lru.cu).
constexpr int kLruMaxK = 32;
int launch_lru_plan(moe_cache* c, const moe_ws* ws, int layer, int K, moe_swap* plan, int32_t* n, cudaStream_t s);
// Planner kernels (defined with the policy), also launched on caller tables.
__global__ void __launch_bounds__(1024) k_plan_layer(float* __restrict__ heat, const int32_t* __restrict__ resid, int E,
                                                     int P, float threshold, float decay,
                                                     unsigned long long* __restrict__ cand, int cand_stride,
                                                     int32_t* __restrict__ cand_count, int32_t* __restrict__ cold_of);
__global__ void __launch_bounds__(1024) k_plan_merge(const unsigned long long* __restrict__ cand, int cand_stride,
                                                     const int32_t* __restrict__ cand_count, int L, int E, int P,
                                                     const int32_t* __restrict__ resid,
                                                     const int32_t* __restrict__ cold_of, int max_swaps,
                                                     moe_swap* __restrict__ plan, int32_t* __restrict__ n_out);
int launch_blob_copy(moe_cache* c, const int32_t* src_index, const int32_t* dst_index, int n, int to_staging,
                     cudaStream_t s);

}  // namespace moe
