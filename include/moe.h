/*
 * moe.h -- C ABI of libmoe: the MoE layer forward over a slot-addressed expert
 * cache, and the adaptive cache policy beside it, for one NVIDIA GB300
 * (sm_103a).
 *
 * Everything here follows the problem statement of the Strata expert-paths
 * page (hanayo.cn, "显存里缓存的是什么？", "路由以后，专家怎样分工？",
 * "哪些专家能长期留在显存？") and the FreeToken reading notes
 * (zhongzhuzhou.org, sections 3.3 and 4): experts are identified by
 * (layer, expert); a residency table maps that identity to a cache slot or to
 * a "not resident" sentinel; tokens that chose the same expert form one group
 * with input and output positions; the expert computes gate/up, SiLU(gate)*up
 * and the down projection on 4-bit block-scaled weights; outputs are merged
 * with the routing weights plus a gated shared expert; heat counters with
 * decay drive same-layer hot-in/cold-out swaps, and a swapped slot is
 * published only after its copy has landed.
 *
 * Conventions for every call
 *   - Pointers named *_dev / tensors are DEVICE memory owned by the caller,
 *     unless the argument says "host".  bf16 tensors are passed as raw 16-bit
 *     patterns (uint16_t).  All arrays are dense row-major.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *     compute call is asynchronous on that stream; it allocates nothing and
 *     does not synchronise.  The caller keeps the arguments alive until the
 *     stream has passed the call.
 *   - The return value reports errors the host can see at call time:
 *     MOE_OK, MOE_EINVAL (bad shape, k > E, NULL pointer, size limits),
 *     MOE_ENOMEM, MOE_ECUDA (a CUDA call or kernel launch failed).
 *     Conditions only the device can see (an expert neither resident nor
 *     staged, an index out of range, a NaN logit, a bounded wait that
 *     expired) are recorded in the workspace's device error word; the
 *     kernels never trap.  moe_sync_status() synchronises the stream, returns
 *     the first recorded device error and clears it.
 *   - Handles (moe_cache, moe_ws) are owned by the library and hold device
 *     memory allocated at creation.  They are not thread-safe; one stream
 *     should drive a workspace at a time.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* == cudaStream_t */

enum {
  MOE_OK = 0,
  MOE_EINVAL = 1,
  MOE_ENOMEM = 2,
  MOE_ECUDA = 3,
  MOE_EMISSING = 4, /* device: a routed expert is neither resident nor staged */
  MOE_ERANGE = 5,   /* device: an index (slot, expert id) is out of range     */
  MOE_ENAN = 6,     /* device: a router logit is NaN                          */
  MOE_ETIMEOUT = 7  /* device: a bounded wait gave up                          */
};

/* Source of a group's weights, as resolved by the residency lookup. */
enum { MOE_SRC_MISSING = -1, MOE_SRC_RESIDENT = 0, MOE_SRC_STAGED = 1, MOE_SRC_SKIPPED = 2 };

/* Forward modes. */
enum { MOE_MODE_AUTO = 0, MOE_MODE_DECODE = 1, MOE_MODE_PREFILL = 2 };

/* Decode paths (moe_ws_set_decode_path). */
enum { MOE_DECODE_FUSED = 0, MOE_DECODE_CHAIN = 1 };

typedef struct moe_cache moe_cache; /* residency + staging tables, slot pools, heats, backing store */
typedef struct moe_ws moe_ws;       /* per-call scratch: logits, ids, groups, h, o, error word */

/* ------------------------------------------------------------------ shapes */

/* One MoE layer.  H hidden, I routed intermediate, E experts, k per token,
 * I_shared shared-expert intermediate (0 = no shared expert).
 * Limits: H, I and a nonzero I_shared powers of two in [64, 4096];
 * 1 <= k <= min(E, 32); 1 <= E <= 1024.  Anything else is MOE_EINVAL. */
typedef struct {
  int H, I, E, k, I_shared;
} moe_layer_shape;

/* Per-layer weights that live outside the expert cache. */
typedef struct {
  const uint16_t* w_router;      /* bf16 [E, H]; NULL -> logits are an input (see moe_route) */
  const float* bias;             /* fp32 [E] added to the logits, or NULL                    */
  const uint16_t* w_shared_gate; /* bf16 [H] shared-expert gate vector, or NULL               */
  const void* shared_blob;       /* device blob of the shared expert (moe_pack_expert), or NULL */
  int layer;                     /* layer index in the cache's (layer, expert) space          */
  moe_layer_shape s;
} moe_layer_desc;

/* ------------------------------------------------------------- weight blobs
 * Canonical matrix format (the NVFP4 row layout of the Qwen3.8-Flash-Next
 * DGX Spark deployment notes, "一个 160 维向量在 packed 文件中占 90 字节" and
 * "NVFP4 code 和 scale 如何反量化"): rows x cols values, each row cols/2 code
 * bytes (two E2M1 codes per byte, low nibble = even column) followed by
 * cols/16 FP8-E4M3 block scales (one per 16 columns); one FP32 global scale
 * per matrix.  value = E2M1(code) * E4M3(scale) * global.
 *
 * An expert blob is the library's slot layout of one expert's three matrices
 * gate [I x H], up [I x H], down [H x I]: a 256-byte header, then code and
 * scale regions per matrix, each 256-byte aligned.  moe_blob_bytes() gives
 * its size; all slots of a cache have that stride. */
size_t moe_blob_bytes(int H, int I);

/* Repack one expert from canonical packed rows (HOST pointers: gate and up
 * [I][9H/16] bytes, down [H][9I/16] bytes) into a HOST blob buffer of
 * moe_blob_bytes(H, I) bytes.  Synchronous, host only. */
int moe_pack_expert(const uint8_t* gate_rows, const uint8_t* up_rows, const uint8_t* down_rows, int H, int I,
                    float gscale_gate, float gscale_up, float gscale_down, void* blob_out_host);

/* -------------------------------------------------------------- the cache */

/* Create a cache for L layers x E experts of shape (H, I): `nslots` cache
 * slots and `nstaging` staging slots in device memory, the residency and
 * staging tables (all -1), fp32 heat counters (0) and statistics.
 * `backing` holds the blobs of all L*E experts, expert (l, e) at offset
 * (l*E + e) * moe_blob_bytes(H, I); it is device memory when
 * backing_on_device != 0, else page-locked host memory (cudaHostAlloc'd or
 * cudaHostRegister'ed) that the device reads directly.  The caller owns it
 * and keeps it alive and unchanged while the cache exists (it is the source
 * of truth; evicted experts need no copy back).  Synchronous. */
int moe_cache_create(moe_cache** out, int L, int E, int H, int I, int nslots, int nstaging, const void* backing,
                     int backing_on_device);
int moe_cache_destroy(moe_cache* c);

/* Admit one expert into a free slot (the Strata page's admit(): only while a
 * free slot exists; otherwise *slot_out = -1 and the expert stays
 * non-resident).  Copies its blob from the backing store.  Synchronous. */
int moe_cache_admit(moe_cache* c, int layer, int expert, int32_t* slot_out);

/* Bulk set-up: make exactly the experts with mask_host[l*E+e] != 0 resident
 * (admitted in (layer, expert) order), or staged when `staging` != 0.
 * Synchronous.  Fails with MOE_ENOMEM when the pool is too small. */
int moe_cache_fill(moe_cache* c, const uint8_t* mask_host, int staging);

/* Device pointers to the cache's tables (valid for the cache's lifetime):
 * resid / stage int32 [L*E] (slot or -1), heat fp32 [L*E], slot_owner int32
 * [nslots] (l*E+e or -1), slot and staging pool bases; the global LRU's
 * lru_tick uint32 [nslots] (the LRU clock at each slot's last use, 0: never)
 * and lru_clock uint32 [1] (layer calls planned so far). */
typedef struct {
  int32_t* resid;
  int32_t* stage;
  float* heat;
  int32_t* slot_owner;
  void* slots;
  void* staging;
  size_t blob_bytes;
  int L, E, nslots, nstaging;
  uint32_t* lru_tick;
  uint32_t* lru_clock;
} moe_cache_view;
int moe_cache_get_view(const moe_cache* c, moe_cache_view* out);

/* Per-layer counters accumulated on the device: out_host receives
 * int64 [L][5] = {lookups, resident hits, staged, missing, skipped by the
 * tail skip}.  Synchronous. */
int moe_get_stats(const moe_cache* c, int64_t* out_host);

/* ---------------------------------------------------------- the workspace */

/* Scratch for layer calls of up to maxT tokens of shape s (device memory,
 * sized at creation).  Holds logits, top-k ids/weights, the expert groups,
 * the intermediate h, per-position expert outputs and the error word. */
int moe_ws_create(moe_ws** out, int maxT, moe_layer_shape s);
int moe_ws_destroy(moe_ws* ws);

/* Device pointers to the groups written by the last moe_group /
 * moe_layer_forward on this workspace (capacities maxT*k):
 *   num_groups int32[1]; grp_expert int32[G] ascending; grp_off int32[G+1];
 *   grp_slot int32[G] (slot or staging index, -1 missing);
 *   grp_src int32[G] (MOE_SRC_*); ent_tok int32[T*k]; ent_pos int32[T*k]
 *   (t*k + r), entries of group g at [grp_off[g], grp_off[g+1]) by token. */
typedef struct {
  int32_t* num_groups;
  int32_t* grp_expert;
  int32_t* grp_off;
  int32_t* grp_slot;
  int32_t* grp_src;
  int32_t* ent_tok;
  int32_t* ent_pos;
  float* logits;    /* fp32 [maxT, E] */
  int32_t* topk_ids; /* int32 [maxT, k] */
  float* topk_w;    /* fp32 [maxT, k] */
  int32_t* error;   /* int32[1] device error word (first error wins) */
} moe_ws_view;
int moe_ws_get_view(const moe_ws* ws, moe_ws_view* out);

/* Optional per-kernel timing.  When enabled, every hot-path call on this
 * workspace records a CUDA event pair around each kernel it launches, on the
 * call's stream.  moe_ws_kernel_times() synchronises on the last event and
 * writes, for the kernels of the most recent call in launch order, their
 * elapsed milliseconds (ms_out[i]) and static names (names_out[i], may be
 * NULL); *n_out receives the count (at most `max`).  Off by default. */
int moe_ws_set_profiling(moe_ws* ws, int enable);

/* Optional tail skip (Strata page, "还有一条会改变输出的路径：跳过尾部专家"):
 * with min_rank > 0, the grouping of later calls on this workspace drops a
 * group whose expert is not resident (staged or missing) when every entry has
 * a zero-based rank (its position r in the token's list) of at least
 * min_rank.  A dropped group keeps its place in the group arrays with source
 * MOE_SRC_SKIPPED, slot -1 and no blob; its entries' expert outputs are zero,
 * so the layer output moves by minus those entries' weighted outputs (the
 * other weights are not renormalised), and a dropped missing expert records
 * no MOE_EMISSING.  min_rank = 0 (the default) turns it off; min_rank >= k
 * drops nothing.  Applies where the grouping looks experts up (moe_group,
 * moe_layer_forward), not to moe_layer_forward_streamed.  MOE_EINVAL when
 * min_rank < 0.  Host-side setting, no stream work. */
int moe_ws_set_tail_skip(moe_ws* ws, int min_rank);

/* Heat update inside the grouping (Strata page, "哪些专家能长期留在显存？":
 * heat counts how often the router picks an expert).  With enable != 0, the
 * grouping of later moe_layer_forward and moe_group calls on this workspace
 * with a cache also adds the window's selection counts to the cache's heat
 * row of the call's layer, with the arithmetic of cache_heat_update
 * (heat = fl32(heat + (float)count), each selected expert once per call); the
 * caller then leaves cache_heat_update out.  Off by default.  Host-side
 * setting, no stream work. */
int moe_ws_set_fused_heat(moe_ws* ws, int enable);
int moe_ws_kernel_times(moe_ws* ws, int max, float* ms_out, const char** names_out, int* n_out);

/* Decode path of later moe_layer_forward calls on this workspace (the same
 * layer in either case: Strata page, "路由以后，专家怎样分工？").
 * MOE_DECODE_FUSED (the default) runs a decode call as ONE cooperative kernel
 * -- router, top-k, groups and lookup (with the heat update and the tail skip
 * when set), gate/up, down, combine, separated by grid barriers -- whenever the
 * shapes fit it: T <= 16, T*k <= 256, E <= 1024, H a power of two in
 * [512, 2048], I a power of two in [256, 1024], I_shared 0 or I, each CTA's
 * router rows (E + 1 over the SM count, rounded up) times H / 512 at most 32,
 * its shared-memory layout within 227 KB, x, y and w_router 16-byte aligned,
 * the shared blob 32-byte aligned; other calls run the chain.  MOE_DECODE_CHAIN always runs the chain of kernels (router,
 * top-k + groups, gate/up, down, combine).  The single kernel needs every
 * SM of the device for its CTAs (a cooperative launch: MOE_ECUDA if the device
 * cannot hold them at once).  Results agree within the layer's tolerance, not
 * bit for bit (the fp32 sums run in another order); ids, groups and lookups
 * are decided on each path's own logits.  MOE_EINVAL for another value.
 * Host-side setting, no stream work. */
int moe_ws_set_decode_path(moe_ws* ws, int path);

/* Fault-injection hook for tests of the bounded waits: the grid barriers of
 * the single-kernel decode give up after wait_ns nanoseconds (default one
 * second) and, with phantom_arrivals > 0, wait for that many arrivals beyond
 * the grid, which never come -- so the wait expires, MOE_ETIMEOUT is recorded
 * in the device error word, the CTAs skip the rest of the call (its outputs
 * are undefined) and the context stays usable.  moe_sync_status() resets the
 * barrier when it returns MOE_ETIMEOUT.  phantom_arrivals 0 restores normal
 * operation; wait_ns 0, phantom_arrivals < 0 or > 1024 is MOE_EINVAL.
 * Host-side setting, no stream work. */
int moe_ws_set_wait_test(moe_ws* ws, unsigned long long wait_ns, int phantom_arrivals);

/* Synchronise `stream`, return the device error word (MOE_OK if none) and
 * reset it to MOE_OK (after MOE_ETIMEOUT also the single-kernel decode's grid
 * barrier). */
int moe_sync_status(moe_ws* ws, moe_stream_t stream);
const char* moe_strerror(int code);

/* ------------------------------------------------------- the hot path calls */

/* Router logits and top-k with renormalised weights (Strata page, "显存里缓存
 * 的是什么？": the router picks each token's experts and their merge weights).
 *   x: bf16 [T, H]; w_router: bf16 [E, H] or NULL; bias: fp32 [E] or NULL;
 *   logits_io: fp32 [T, E] -- output l = x.W_r^T + bias (fp32 accumulate)
 *   when w_router != NULL, else an INPUT (same-logits mode);
 *   topk_ids: int32 [T, k] -- the k largest logits, weight descending, ties
 *   to the lower expert id; topk_w: fp32 [T, k] -- exp(l - l_max) / sum over
 *   the k chosen (= softmax over E renormalised over the k).
 * A NaN logit records MOE_ENAN in err_dev (int32[1], may be NULL). */
int moe_route(const uint16_t* x, const uint16_t* w_router, const float* bias, float* logits_io, int T, int H, int E,
              int k, int32_t* topk_ids, float* topk_w, int32_t* err_dev, moe_stream_t stream);

/* Dedupe one layer's selections into expert groups and look each group up
 * (Strata page, "路由以后，专家怎样分工？": repeated experts of a layer and
 * window form one group recording input and output positions; "哪些专家能长期
 * 留在显存？": (layer, expert) -> slot or sentinel).  topk_ids int32 [T, k]
 * (each row distinct ids in [0, E)).  Writes the workspace's group arrays
 * (moe_ws_view): groups by ascending expert id, entries by ascending token,
 * position t*k + r; slot from the residency table, else the staging table,
 * else MOE_SRC_MISSING (also recorded as MOE_EMISSING); with the workspace's
 * tail skip on, MOE_SRC_SKIPPED for the groups it drops (moe_ws_set_tail_skip).
 * Updates the cache's lookup counters.  Out-of-range ids record MOE_ERANGE.
 * MOE_EINVAL when T exceeds the workspace's maxT, k or E differ from the
 * workspace's shape, or E from the cache's. */
int moe_group(const int32_t* topk_ids, int T, int k, int E, int layer, moe_cache* c, moe_ws* ws,
              moe_stream_t stream);

/* The whole layer: router -> top-k -> groups -> lookup -> SwiGLU experts on
 * the slot blobs -> routing-weighted combine + sigmoid-gated shared expert:
 *   y[t] = sigmoid(x_t . w_sg) * S(x_t) + sum_r w[t,r] * E_{ids[t,r]}(x_t)
 * (Strata page, "路由以后，专家怎样分工？"; FreeToken notes section 3.2: the
 * merge is exact, no expert dropped unless the workspace's tail skip is on).  x: bf16 [T, H]; y: bf16 [T, H], or
 * fp32 [T, H] when y_is_fp32.  T <= the workspace's maxT.  mode selects the
 * decode kernels (the single-kernel decode or the chain: CUDA-core router,
 * mma.sync expert tiles) or the prefill kernels (router and grouped expert
 * GEMMs on the tensor cores); AUTO takes prefill from 32 tokens on where the
 * shape and the pointers allow it, else decode (from 32 tokens the grouped
 * GEMMs' 128-row weight tiles, reused across a group's tokens, are faster
 * than decode's 16-row units).  MOE_MODE_PREFILL needs H >= 128 and
 * 16-byte aligned x, y, w_router and w_shared_gate, else MOE_EINVAL; its y
 * accumulates in fp32 with atomic adds, so the order of the (at most k + 1)
 * terms per element may vary between runs. */
int moe_layer_forward(const moe_layer_desc* d, const uint16_t* x, void* y, int y_is_fp32, int T, moe_cache* c,
                      moe_ws* ws, int mode, moe_stream_t stream);

/* The prefill forward with the layer's routed experts streamed through the
 * staging pool (Strata expert paths, "PCIe 搬运怎样与计算重叠？": the copy stream
 * fills a staging slot and records `copied`, the compute stream waits on it,
 * computes and records `used`, and the copy stream waits on `used` before it
 * overwrites the slot).  The residency and staging tables are not consulted:
 * experts e in [u*U, u*U + U) form unit u; copy_stream copies their blobs
 * (one cudaMemcpyAsync of n*blob_bytes per unit, n <= U, from the cache's
 * backing pool, device or pinned host) into staging slots (u % 2)*U ..; stream
 * runs the grouped GEMMs of that unit's groups once they have landed.  The
 * shared expert runs with unit 0.  buffers = 2 double-buffers the units
 * (unit u + 1 copies while unit u computes); buffers = 1 keeps one half, so
 * each copy waits for the previous unit's GEMMs (the FreeToken notes'
 * "second buffer off" ablation, section 5.3).  Same arguments, layout and
 * result as moe_layer_forward in prefill mode, plus: U >= 1 with buffers*U <=
 * the cache's staging slots, buffers 1 or 2, a backing pool, and copy_stream
 * a stream other than stream, else MOE_EINVAL.  Both streams may be used again
 * as soon as the call returns; the staging slots' contents and table entries
 * are left undefined for lookups (the staging table itself is not changed). */
int moe_layer_forward_streamed(const moe_layer_desc* d, const uint16_t* x, void* y, int y_is_fp32, int T,
                               moe_cache* c, moe_ws* ws, int U, int buffers, moe_stream_t stream,
                               moe_stream_t copy_stream);

/* Activation rows as sums of NVFP4 terms, the B operands of the block-scaled
 * FP4 prefill GEMMs.  The format is the weights' (PLE offload page, "NVFP4 code
 * 和 scale 如何反量化": value = E2M1 code x FP8-E4M3 scale per 16 values x FP32
 * global scale); the pages give its decoding, and this quantiser is its plain
 * reading, applied R times to the remaining residual: term r of row i is
 * q = Q(v - q_1 - ... - q_{r-1}), Q with
 *   G: the smallest power of two with max|row| / (6 G) <= 448;
 *   s: per 16 values, the smallest non-negative E4M3 value with 6 s G >= max|block|;
 *   code: the E2M1 value nearest to v / (s G) (correctly rounded quotient), ties to even.
 *   src     rows x K activations, row i at src + i * ld elements: bf16 (src_is_fp32 = 0)
 *           or fp32; 16-byte aligned, ld a multiple of 8;
 *   codes   uint8 [rows * R][K / 2] out: term r of row i at row i * R + r, low nibble =
 *           even column; 8-byte aligned;
 *   scales  uint8 [rows * R][K / 16] out: the E4M3 block scales (sign bit clear);
 *   gscale  fp32 [rows * R] out: the global scales.
 * K a power of two in [64, 4096], 1 <= R <= 8, else MOE_EINVAL.  The residual is
 * kept in fp32: exact for bf16 rows, within one rounding per term for fp32 rows.
 * Asynchronous on `stream`. */
int moe_nvfp4_split(const void* src, int src_is_fp32, int rows, int K, int ld, int R, uint8_t* codes,
                    uint8_t* scales, float* gscale, moe_stream_t stream);

/* Several MoE layers of a prefill chunk, each layer's experts streamed whole
 * through the staging pool one layer ahead (FreeToken notes, section 3.1: layer
 * l + 1's experts copy into the second buffer while layer l computes with the
 * first; section 5.3: with the second buffer off, each copy waits until the
 * previous layer is done).  The layers sit on an fp32 residual stream as in
 * moe_residual_rmsnorm: for l = 0 .. L-1, x_res += y (l > 0), xn = bf16(RMSNorm
 * (x_res)), y = MoE_l(xn) in prefill mode; finally x_res += y.
 *   d       moe_layer_desc [L] (host), the same H, E and k, each with its layer;
 *   x_res   fp32 [T, H] device, the residual stream, updated in place (16-byte aligned);
 *   xn, y   bf16 [T, H] device scratch (16-byte aligned); on return xn holds the
 *           normalised final stream, y the last layer's output.
 * Layer l uses staging slots h * E .. h * E + E - 1 with h = l % buffers: the copy
 * stream waits on `used` of the layer that last read half h, copies the layer's E
 * blobs from the cache's backing pool (device or pinned host) in one
 * cudaMemcpyAsync and records `copied`; the compute stream waits on `copied` before
 * the layer's expert GEMMs and records `used` after them.  The residency and
 * staging tables are not consulted or changed.  buffers 1 or 2, buffers * E <= the
 * cache's staging slots, a backing pool, eps > 0, copy_stream distinct from
 * stream, and every layer valid for moe_layer_forward in prefill mode, else
 * MOE_EINVAL.  Both streams may be reused as soon as the call returns. */
int moe_layers_forward_streamed(const moe_layer_desc* d, int L, float* x_res, uint16_t* xn, uint16_t* y, int T,
                                moe_cache* c, moe_ws* ws, int buffers, float eps, moe_stream_t stream,
                                moe_stream_t copy_stream);

/* Heat update (Strata page, "哪些专家能长期留在显存？": accumulate how often
 * each expert is routed to): heat[layer*E+e] = fl32(heat + (float)count_e)
 * with count_e the number of (token, rank) selections of e in topk_ids
 * int32 [T, k].  Out-of-range ids record MOE_ERANGE in err_dev (may be NULL). */
int cache_heat_update(moe_cache* c, const int32_t* topk_ids, int T, int k, int layer, int32_t* err_dev,
                      moe_stream_t stream);

typedef struct {
  int layer, hot_expert, cold_expert, slot;
  float diff;
} moe_swap;

typedef struct {
  float threshold; /* 1.5f  */
  int max_swaps;   /* 96    */
  float decay;     /* 0.7f  */
} moe_policy_cfg;

/* One planning round (same section: pair hot non-resident with cold resident
 * experts of the same layer when the heat difference reaches the threshold,
 * sort by difference, cap per round, then decay all heats):
 *   per layer, non-resident experts by heat desc (id asc) are paired i-th with
 *   resident experts by heat asc (id asc) while fl32(h_hot - h_cold) >=
 *   threshold; candidates of all layers ordered by (diff desc, layer asc,
 *   hot id asc); the first max_swaps written to plan_dev (moe_swap[max_swaps],
 *   device) and their number to n_dev (int32[1], device); then every heat
 *   becomes fl32(heat * decay).  A NaN difference (a NaN heat, or infinite
 *   heats on both sides) fails the test, so it ends its layer's pairing there.
 *   Requires L*E <= 32768 and max_swaps <= 4096. */
int cache_plan_swaps(moe_cache* c, const moe_policy_cfg* p, moe_swap* plan_dev, int32_t* n_dev, moe_stream_t stream);

/* Residual stream and RMS normalisation between the layers of a decode stack.
 * The pages give the model as MoE layers in sequence but have no counterpart
 * to this step: it is the wrapper of the 48-layer decode workload,
 * x_{l+1} = x_l + MoE_l(RMSNorm(x_l)), with unit RMSNorm weight.
 *   x_res   float [T, H] device, the residual stream, updated in place:
 *           x_res += y_prev when y_prev != NULL (bf16 [T, H], the previous
 *           layer's output);
 *   xn_out  bf16 [T, H] device: bf16(x_res / sqrt(mean(x_res^2) + eps)),
 *           the next layer's input.
 * fp32 arithmetic (sum of squares in fp32, correctly rounded sqrt and
 * division).  H a multiple of 4 and at most 4096, eps > 0, x_res 16-byte and
 * the bf16 arrays 8-byte aligned, else MOE_EINVAL. */
int moe_residual_rmsnorm(float* x_res, const uint16_t* y_prev, uint16_t* xn_out, int T, int H, float eps,
                         moe_stream_t stream);

/* cache_plan_swaps on caller-owned tables, allocating nothing.  The pages
 * have no counterpart to this call: it exists for callers that cannot
 * allocate device memory where they plan -- a serving loop whose memory is
 * handed out by its own allocator under a fixed budget (a cudaMalloc would
 * step outside the budget or fail when it is spent), or one that keeps the
 * heat and residency tables in its own buffers without a moe_cache handle.
 *   heat_dev  float [L, E] device, read and then decayed in place (as the
 *             handle's heat table is by cache_plan_swaps);
 *   resid_dev int32 [L, E] device, slot of each resident expert, negative
 *             when not resident (the layout of moe_cache_view.resid).
 * The plan, its order, n_dev and the decayed heats are exactly those of
 * cache_plan_swaps on the same tables.  The planner's scratch is a 260 KB
 * static device array inside the library, so the sizes it takes are capped:
 * L <= 1024, E <= 1024, L*E <= 32768 and L*ceil(E/2) <= 16384; larger sizes
 * (and max_swaps outside 0..4096, threshold <= 0, NULL pointers) return
 * MOE_EINVAL before anything is launched.  Nothing in the scratch needs to
 * start at zero.  The scratch's address is looked up on the first call on
 * each device (with that device current); the lookup may load the module,
 * which a stream capture does not allow, so make the first call on each
 * device before any capture.  The looked-up address is kept for the life of
 * the process: after a cudaDeviceReset (or any teardown of the device's
 * primary context) it is stale, so do not call this function again in that
 * process.  All calls on one device share the scratch: calls that overlap in
 * time (other streams, other threads) race and must be serialised by the
 * caller.  Heats may be NaN or infinite: a layer's pairing stops at the first
 * pair whose difference fails the threshold test, as in cache_plan_swaps. */
int cache_plan_swaps_noalloc(float* heat_dev, const int32_t* resid_dev, int L, int E, const moe_policy_cfg* p,
                             moe_swap* plan_dev, int32_t* n_dev, moe_stream_t stream);

/* Execute a plan (same section: new weights are visible only after the copy
 * completes; a slot is reused only after earlier reads finished):
 *   on `compute`: unmap each cold expert (resid = -1), record event
 *   "unmapped";  on `copy`: wait "unmapped", copy each hot blob from the
 *   backing store into the slot, record "copied";  on `compute`: wait
 *   "copied", publish (resid[hot] = slot).  Kernels queued on `compute`
 *   before this call finish reading the old slots before the copy starts;
 *   kernels queued after it see either the old mapping (never) or the new one.
 *   No host synchronisation; n_dev is read on the device. */
int moe_cache_apply_swaps(moe_cache* c, const moe_swap* plan_dev, const int32_t* n_dev, moe_stream_t compute,
                          moe_stream_t copy);

/* Global LRU over the slots (FreeToken reading notes, section 3.3: one LRU for
 * every layer's (layer, expert) -- a hit refreshes its recency, a fill admits
 * the newly chosen expert, the least recently used is evicted; section 4: one
 * pass finds K victim candidates and the misses take the first q <= K).  Call
 * after a layer call's grouping on ws (moe_group, moe_layer_forward) for layer
 * `layer`: advances the cache's LRU clock, marks the slots of the call's
 * resident groups as used now, then writes into plan_dev (device moe_swap[K])
 * and *n_dev (device int32) the admissions: the call's i-th miss (a group that
 * is staged or missing, in group order) into the i-th victim, the victims
 * being the slots this call did not use, empty slots first, then least
 * recently used first, ties to the lower slot.  In an entry, `layer` and
 * hot_expert name the admitted expert, cold_expert the evicted one as
 * layer * E + expert (-1: the slot was empty), slot the slot, diff is 0; the
 * slots taken count as used now.  1 <= K <= 32 and a cache of 1 to 2^24 - 1
 * slots, else MOE_EINVAL.  The clock
 * is 32-bit: past 2^32 - 2 calls the device records MOE_ERANGE.  Async on
 * `stream`; execute the plan with moe_cache_apply_lru. */
int cache_lru_plan(moe_cache* c, const moe_ws* ws, int layer, int K, moe_swap* plan_dev, int32_t* n_dev,
                   moe_stream_t stream);

/* Executes an LRU plan with the publish-after-copy order of
 * moe_cache_apply_swaps (evicted entries cleared on `compute`; blobs copied
 * from the backing store on `copy` after that; admitted entries published on
 * `compute` after the copies), the evicted expert given by its flat id.  An
 * entry whose evicted expert does not own its slot (or whose slot is not
 * empty when no expert is named) is skipped, as moe_cache_apply_swaps skips
 * an inconsistent entry. */
int moe_cache_apply_lru(moe_cache* c, const moe_swap* plan_dev, const int32_t* n_dev, moe_stream_t compute,
                        moe_stream_t copy);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
