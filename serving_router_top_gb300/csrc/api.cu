// Host side of the C ABI declared in include/moe.h: argument checks, handle
// lifecycle, and the launch sequence of each call.  No call on the hot path
// allocates or synchronises.
#include <stdlib.h>
#include <string.h>

#include <vector>

#include "internal.h"

using namespace moe;

namespace {

// AUTO mode runs the prefill (tcgen05 grouped GEMM) path from this many tokens on.
constexpr int kPrefillMinTokens = 32;  // measured crossover: 16 tokens still faster on the decode kernels

bool shape_ok(const moe_layer_shape& s) {
  // row widths: powers of two from 64 to 4096 (lanes per row and chunks per lane are powers of two)
  auto cols_ok = [](int c) { return c >= 64 && c <= 4096 && (c & (c - 1)) == 0; };
  if (!cols_ok(s.H) || !cols_ok(s.I)) return false;
  if (s.I_shared != 0 && !cols_ok(s.I_shared)) return false;
  if (s.E < 1 || s.E > kMaxE || s.k < 1 || s.k > kMaxK || s.k > s.E) return false;
  return true;
}

// Bump allocator over one cudaMalloc.
struct Carve {
  size_t off = 0;
  template <class T>
  size_t take(size_t count) {
    off = (off + 255) & ~size_t(255);
    size_t at = off;
    off += count * sizeof(T);
    return at;
  }
};

}  // namespace

extern "C" {

const char* moe_strerror(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_EINVAL: return "invalid argument";
    case MOE_ENOMEM: return "out of memory";
    case MOE_ECUDA: return "CUDA call or kernel launch failed";
    case MOE_EMISSING: return "a routed expert is neither resident nor staged";
    case MOE_ERANGE: return "index out of range";
    case MOE_ENAN: return "NaN router logit";
    case MOE_ETIMEOUT: return "bounded wait expired";
    default: return "unknown error";
  }
}

size_t moe_blob_bytes(int H, int I) {
  if (H <= 0 || I <= 0 || H % 32 || I % 32) return 0;
  return blob_layout(H, I).bytes;
}

int moe_pack_expert(const uint8_t* gate_rows, const uint8_t* up_rows, const uint8_t* down_rows, int H, int I,
                    float gscale_gate, float gscale_up, float gscale_down, void* blob_out_host) {
  if (!gate_rows || !up_rows || !down_rows || !blob_out_host || H <= 0 || I <= 0 || H % 32 || I % 32)
    return MOE_EINVAL;
  const BlobLayout L = blob_layout(H, I);
  uint8_t* out = static_cast<uint8_t*>(blob_out_host);
  memset(out, 0, L.bytes);
  BlobHeader hd;
  memset(&hd, 0, sizeof(hd));
  hd.magic = kBlobMagic;
  hd.version = 1;
  hd.H = H;
  hd.I = I;
  hd.gscale[0] = gscale_gate;
  hd.gscale[1] = gscale_up;
  hd.gscale[2] = gscale_down;
  memcpy(out, &hd, sizeof(hd));
  const uint8_t* src[3] = {gate_rows, up_rows, down_rows};
  const int rows[3] = {I, I, H}, cols[3] = {H, H, I};
  for (int m = 0; m < 3; ++m) {
    const size_t cb = size_t(cols[m]) / 2, sb = size_t(cols[m]) / 16, rb = cb + sb;
    for (int r = 0; r < rows[m]; ++r) {
      memcpy(out + L.code_off[m] + size_t(r) * cb, src[m] + size_t(r) * rb, cb);
      memcpy(out + L.scale_off[m] + size_t(r) * sb, src[m] + size_t(r) * rb + cb, sb);
    }
  }
  return MOE_OK;
}

// ------------------------------------------------------------------ cache
int moe_cache_create(moe_cache** out, int L, int E, int H, int I, int nslots, int nstaging, const void* backing,
                     int backing_on_device) {
  if (!out || L <= 0 || E <= 0 || E > kMaxE || L > 65535 || nslots < 0 || nstaging < 0 || H % 32 || I % 32 ||
      H <= 0 || I <= 0)
    return MOE_EINVAL;
  *out = nullptr;
  moe_cache* c = static_cast<moe_cache*>(calloc(1, sizeof(moe_cache)));
  if (!c) return MOE_ENOMEM;
  c->L = L;
  c->E = E;
  c->H = H;
  c->I = I;
  c->nslots = nslots;
  c->nstaging = nstaging;
  c->blob_bytes = blob_layout(H, I).bytes;
  c->backing_on_device = backing_on_device;
  if (backing) {
    if (backing_on_device) {
      c->backing = backing;
    } else {
      void* dp = nullptr;
      if (cudaHostGetDevicePointer(&dp, const_cast<void*>(backing), 0) != cudaSuccess) {
        cudaGetLastError();
        free(c);
        return MOE_EINVAL;
      }
      c->backing = dp;
    }
  }
  const size_t LE = size_t(L) * E;
  const int stride = (E + 1) / 2;
  c->plan_scratch_bytes = size_t(L) * stride * 8 + size_t(L) * 4 + LE * 4;
  bool ok = cudaMalloc(&c->resid, LE * 4) == cudaSuccess && cudaMalloc(&c->stage, LE * 4) == cudaSuccess &&
            cudaMalloc(&c->heat, LE * 4) == cudaSuccess &&
            cudaMalloc(&c->slot_owner, size_t(nslots > 0 ? nslots : 1) * 4) == cudaSuccess &&
            cudaMalloc(&c->staging_owner, size_t(nstaging > 0 ? nstaging : 1) * 4) == cudaSuccess &&
            cudaMalloc(&c->stats, size_t(L) * kStats * 8) == cudaSuccess &&
            cudaMalloc(&c->lru_tick, size_t(nslots > 0 ? nslots : 1) * 4 + 4) == cudaSuccess &&
            cudaMalloc(&c->plan_scratch, c->plan_scratch_bytes) == cudaSuccess;
  if (ok) c->lru_clock = c->lru_tick + (nslots > 0 ? nslots : 1);
  if (ok && nslots > 0) ok = cudaMalloc(&c->slots, size_t(nslots) * c->blob_bytes) == cudaSuccess;
  if (ok && nstaging > 0) ok = cudaMalloc(&c->staging, size_t(nstaging) * c->blob_bytes) == cudaSuccess;
  if (ok) ok = cudaEventCreateWithFlags(&c->ev_unmapped, cudaEventDisableTiming) == cudaSuccess &&
               cudaEventCreateWithFlags(&c->ev_copied, cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; ok && i < 5; ++i) ok = cudaEventCreateWithFlags(&c->ev_ring[i], cudaEventDisableTiming) == cudaSuccess;
  if (ok)
    ok = cudaMemset(c->resid, 0xff, LE * 4) == cudaSuccess && cudaMemset(c->stage, 0xff, LE * 4) == cudaSuccess &&
         cudaMemset(c->heat, 0, LE * 4) == cudaSuccess &&
         cudaMemset(c->slot_owner, 0xff, size_t(nslots > 0 ? nslots : 1) * 4) == cudaSuccess &&
         cudaMemset(c->staging_owner, 0xff, size_t(nstaging > 0 ? nstaging : 1) * 4) == cudaSuccess &&
         cudaMemset(c->stats, 0, size_t(L) * kStats * 8) == cudaSuccess &&
         cudaMemset(c->lru_tick, 0, size_t(nslots > 0 ? nslots : 1) * 4 + 4) == cudaSuccess &&
         cudaMemset(c->plan_scratch, 0, c->plan_scratch_bytes) == cudaSuccess && cudaDeviceSynchronize() == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    moe_cache_destroy(c);
    return MOE_ENOMEM;
  }
  *out = c;
  return MOE_OK;
}

int moe_cache_destroy(moe_cache* c) {
  if (!c) return MOE_OK;
  cudaFree(c->resid);
  cudaFree(c->stage);
  cudaFree(c->heat);
  cudaFree(c->slot_owner);
  cudaFree(c->staging_owner);
  cudaFree(c->stats);
  cudaFree(c->lru_tick);
  cudaFree(c->plan_scratch);
  cudaFree(c->slots);
  cudaFree(c->staging);
  if (c->ev_unmapped) cudaEventDestroy(c->ev_unmapped);
  if (c->ev_copied) cudaEventDestroy(c->ev_copied);
  for (int i = 0; i < 5; ++i)
    if (c->ev_ring[i]) cudaEventDestroy(c->ev_ring[i]);
  free(c);
  return MOE_OK;
}

static int copy_blob_to(moe_cache* c, int flat, uint8_t* dst) {
  if (!c->backing) return MOE_EINVAL;
  const uint8_t* src = static_cast<const uint8_t*>(c->backing) + size_t(flat) * c->blob_bytes;
  MOE_CUDA_TRY(cudaMemcpy(dst, src, c->blob_bytes, cudaMemcpyDefault));
  return MOE_OK;
}

int moe_cache_admit(moe_cache* c, int layer, int expert, int32_t* slot_out) {
  if (!c || !slot_out || layer < 0 || layer >= c->L || expert < 0 || expert >= c->E) return MOE_EINVAL;
  const int flat = layer * c->E + expert;
  int32_t cur = -1;
  MOE_CUDA_TRY(cudaMemcpy(&cur, c->resid + flat, 4, cudaMemcpyDeviceToHost));
  if (cur >= 0) { *slot_out = cur; return MOE_OK; }
  if (c->next_free_slot >= c->nslots) { *slot_out = -1; return MOE_OK; }
  const int slot = c->next_free_slot;
  int rc = copy_blob_to(c, flat, c->slots + size_t(slot) * c->blob_bytes);
  if (rc) return rc;
  MOE_CUDA_TRY(cudaMemcpy(c->resid + flat, &slot, 4, cudaMemcpyHostToDevice));
  MOE_CUDA_TRY(cudaMemcpy(c->slot_owner + slot, &flat, 4, cudaMemcpyHostToDevice));
  c->next_free_slot++;
  *slot_out = slot;
  return MOE_OK;
}

int moe_cache_fill(moe_cache* c, const uint8_t* mask_host, int staging) {
  if (!c || !mask_host || !c->backing) return MOE_EINVAL;
  const size_t LE = size_t(c->L) * c->E;
  int32_t* table = staging ? c->stage : c->resid;
  int32_t* owner = staging ? c->staging_owner : c->slot_owner;
  uint8_t* pool = staging ? c->staging : c->slots;
  int& next = staging ? c->next_free_staging : c->next_free_slot;
  const int cap = staging ? c->nstaging : c->nslots;
  std::vector<int32_t> tab(LE), own(size_t(cap > 0 ? cap : 1), -1);
  MOE_CUDA_TRY(cudaMemcpy(tab.data(), table, LE * 4, cudaMemcpyDeviceToHost));
  if (cap > 0) MOE_CUDA_TRY(cudaMemcpy(own.data(), owner, size_t(cap) * 4, cudaMemcpyDeviceToHost));
  for (size_t f = 0; f < LE; ++f) {
    if (!mask_host[f] || tab[f] >= 0) continue;
    if (next >= cap) return MOE_ENOMEM;
    const int slot = next++;
    const uint8_t* src = static_cast<const uint8_t*>(c->backing) + f * c->blob_bytes;
    MOE_CUDA_TRY(cudaMemcpyAsync(pool + size_t(slot) * c->blob_bytes, src, c->blob_bytes, cudaMemcpyDefault, 0));
    tab[f] = slot;
    own[slot] = int32_t(f);
  }
  MOE_CUDA_TRY(cudaMemcpy(table, tab.data(), LE * 4, cudaMemcpyHostToDevice));
  if (cap > 0) MOE_CUDA_TRY(cudaMemcpy(owner, own.data(), size_t(cap) * 4, cudaMemcpyHostToDevice));
  MOE_CUDA_TRY(cudaDeviceSynchronize());
  return MOE_OK;
}

int moe_cache_get_view(const moe_cache* c, moe_cache_view* v) {
  if (!c || !v) return MOE_EINVAL;
  v->resid = c->resid;
  v->stage = c->stage;
  v->heat = c->heat;
  v->slot_owner = c->slot_owner;
  v->slots = c->slots;
  v->staging = c->staging;
  v->blob_bytes = c->blob_bytes;
  v->L = c->L;
  v->E = c->E;
  v->nslots = c->nslots;
  v->nstaging = c->nstaging;
  v->lru_tick = c->lru_tick;
  v->lru_clock = c->lru_clock;
  return MOE_OK;
}

int moe_get_stats(const moe_cache* c, int64_t* out_host) {
  if (!c || !out_host) return MOE_EINVAL;
  MOE_CUDA_TRY(cudaMemcpy(out_host, c->stats, size_t(c->L) * kStats * 8, cudaMemcpyDeviceToHost));
  return MOE_OK;
}

// -------------------------------------------------------------- workspace
int moe_ws_create(moe_ws** out, int maxT, moe_layer_shape s) {
  if (!out || maxT <= 0 || !shape_ok(s)) return MOE_EINVAL;
  *out = nullptr;
  moe_ws* w = static_cast<moe_ws*>(calloc(1, sizeof(moe_ws)));
  if (!w) return MOE_ENOMEM;
  w->maxT = maxT;
  w->s = s;
  const size_t Tk = size_t(maxT) * s.k;
  const size_t Imax = size_t(s.I > s.I_shared ? s.I : s.I_shared);
  Carve cv;
  const size_t o_logits = cv.take<float>(size_t(maxT) * s.E);
  const size_t o_ids = cv.take<int32_t>(Tk);
  const size_t o_w = cv.take<float>(Tk);
  const size_t o_gl = cv.take<float>(maxT);
  const size_t o_ng = cv.take<int32_t>(1);
  const size_t o_ge = cv.take<int32_t>(Tk);
  const size_t o_go = cv.take<int32_t>(Tk + 1);
  const size_t o_gs = cv.take<int32_t>(Tk);
  const size_t o_gsrc = cv.take<int32_t>(Tk);
  const size_t o_gb = cv.take<const uint8_t*>(Tk);
  const size_t o_et = cv.take<int32_t>(Tk);
  const size_t o_ep = cv.take<int32_t>(Tk);
  const size_t o_x16 = cv.take<__half>(size_t(maxT) * s.H);
  const size_t o_xs = cv.take<float>(maxT);
  const size_t o_h = cv.take<float>((Tk + maxT) * Imax);
  const size_t o_hmax = cv.take<float>(Tk + maxT);
  const size_t o_xinv = cv.take<float>(Tk + maxT);
  // split-K scratch: K is sliced only for calls of at most 8 tokens, so at most
  // min(8k, E) groups of up to max(H, I)/16 row blocks, plus the shared expert's
  const int small_groups = (maxT < 8 ? maxT : 8) * s.k < s.E ? (maxT < 8 ? maxT : 8) * s.k : s.E;
  const int rb_max = (s.H > s.I ? s.H : s.I) / 16;
  const size_t split_blocks = size_t(small_groups + 1) * rb_max;
  const size_t o_part = cv.take<float>(split_blocks * 8 * 32 * 8);
  const size_t o_toff = cv.take<int32_t>(size_t(s.E) + 2);
  const size_t o_tgrp = cv.take<int32_t>(size_t(s.E) + Tk / 128 + 2);
  const size_t o_grange = cv.take<int32_t>(2 * size_t(s.E) + 2);
  const size_t o_h16 = cv.take<__half>((Tk + maxT) * Imax);
  const size_t o_yacc = cv.take<float>(size_t(maxT) * s.H);
  const size_t o_cnt = cv.take<int>(split_blocks);
  const size_t o_o = cv.take<float>((Tk + maxT) * s.H);
  const size_t o_gscr = cv.take<int32_t>((size_t(maxT) / 256 + 2) * s.E);
  const size_t o_err = cv.take<int32_t>(1);
  const size_t o_bar = cv.take<unsigned long long>(kBarWords);
  uint8_t* base = nullptr;
  if (cudaMalloc(&base, cv.off) != cudaSuccess) {
    cudaGetLastError();
    free(w);
    return MOE_ENOMEM;
  }
  w->logits = reinterpret_cast<float*>(base + o_logits);
  w->topk_ids = reinterpret_cast<int32_t*>(base + o_ids);
  w->topk_w = reinterpret_cast<float*>(base + o_w);
  w->gate_logit = reinterpret_cast<float*>(base + o_gl);
  w->num_groups = reinterpret_cast<int32_t*>(base + o_ng);
  w->grp_expert = reinterpret_cast<int32_t*>(base + o_ge);
  w->grp_off = reinterpret_cast<int32_t*>(base + o_go);
  w->grp_slot = reinterpret_cast<int32_t*>(base + o_gs);
  w->grp_src = reinterpret_cast<int32_t*>(base + o_gsrc);
  w->grp_blob = reinterpret_cast<const uint8_t**>(base + o_gb);
  w->ent_tok = reinterpret_cast<int32_t*>(base + o_et);
  w->ent_pos = reinterpret_cast<int32_t*>(base + o_ep);
  w->x16 = reinterpret_cast<__half*>(base + o_x16);
  w->xscale = reinterpret_cast<float*>(base + o_xs);
  w->h = reinterpret_cast<float*>(base + o_h);
  w->hmax = reinterpret_cast<float*>(base + o_hmax);
  w->part = reinterpret_cast<float*>(base + o_part);
  w->tile_off = reinterpret_cast<int32_t*>(base + o_toff);
  w->tile_grp = reinterpret_cast<int32_t*>(base + o_tgrp);
  w->grange = reinterpret_cast<int32_t*>(base + o_grange);
  w->h16 = reinterpret_cast<__half*>(base + o_h16);
  w->yacc = reinterpret_cast<float*>(base + o_yacc);
  w->xg = reinterpret_cast<__half*>(base + o_o);  // (Tk+maxT)*H 16-bit values fit in (Tk+maxT)*H floats
  w->xinv = reinterpret_cast<float*>(base + o_xinv);
  w->cnt = reinterpret_cast<int*>(base + o_cnt);
  w->split_blocks = split_blocks;
  w->o = reinterpret_cast<float*>(base + o_o);
  w->grp_scratch = reinterpret_cast<int32_t*>(base + o_gscr);
  w->error = reinterpret_cast<int32_t*>(base + o_err);
  w->bar = reinterpret_cast<unsigned long long*>(base + o_bar);
  w->bar_extra = 0;
  w->wait_ns = 1000000000ull;  // one second
  w->decode_path = MOE_DECODE_FUSED;
  if (cudaMemset(base, 0, cv.off) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    cudaFree(base);
    free(w);
    return MOE_ECUDA;
  }
  *out = w;
  return MOE_OK;
}

int moe_ws_destroy(moe_ws* w) {
  if (!w) return MOE_OK;
  for (int i = 0; i < 32; ++i)
    if (w->prof_ev[i]) cudaEventDestroy(w->prof_ev[i]);
  cudaFree(w->logits);  // first carve of the single allocation
  free(w);
  return MOE_OK;
}

int moe_ws_get_view(const moe_ws* w, moe_ws_view* v) {
  if (!w || !v) return MOE_EINVAL;
  v->num_groups = w->num_groups;
  v->grp_expert = w->grp_expert;
  v->grp_off = w->grp_off;
  v->grp_slot = w->grp_slot;
  v->grp_src = w->grp_src;
  v->ent_tok = w->ent_tok;
  v->ent_pos = w->ent_pos;
  v->logits = w->logits;
  v->topk_ids = w->topk_ids;
  v->topk_w = w->topk_w;
  v->error = w->error;
  return MOE_OK;
}

int moe_ws_set_fused_heat(moe_ws* w, int enable) {
  if (!w) return MOE_EINVAL;
  w->fused_heat = enable ? 1 : 0;
  return MOE_OK;
}

int moe_ws_set_decode_path(moe_ws* w, int path) {
  if (!w || (path != MOE_DECODE_FUSED && path != MOE_DECODE_CHAIN)) return MOE_EINVAL;
  w->decode_path = path;
  return MOE_OK;
}

int moe_ws_set_wait_test(moe_ws* w, unsigned long long wait_ns, int phantom_arrivals) {
  if (!w || wait_ns == 0 || phantom_arrivals < 0 || phantom_arrivals > 1024) return MOE_EINVAL;
  w->wait_ns = wait_ns;
  w->bar_extra = unsigned(phantom_arrivals);
  return MOE_OK;
}

int moe_ws_set_tail_skip(moe_ws* w, int min_rank) {
  if (!w || min_rank < 0) return MOE_EINVAL;
  w->tail_skip = min_rank;
  return MOE_OK;
}

int moe_ws_set_profiling(moe_ws* w, int enable) {
  if (!w) return MOE_EINVAL;
  if (enable && !w->prof_ev[0]) {
    for (int i = 0; i < 32; ++i) MOE_CUDA_TRY(cudaEventCreate(&w->prof_ev[i]));
  }
  w->prof_on = enable ? 1 : 0;
  w->prof_n = 0;
  return MOE_OK;
}

int moe_ws_kernel_times(moe_ws* w, int max, float* ms_out, const char** names_out, int* n_out) {
  if (!w || !ms_out || !n_out || max < 0) return MOE_EINVAL;
  const int n = w->prof_n < max ? w->prof_n : max;
  if (n > 0) MOE_CUDA_TRY(cudaEventSynchronize(w->prof_ev[2 * (w->prof_n - 1) + 1]));
  for (int i = 0; i < n; ++i) {
    float ms = 0.f;
    MOE_CUDA_TRY(cudaEventElapsedTime(&ms, w->prof_ev[2 * i], w->prof_ev[2 * i + 1]));
    ms_out[i] = ms;
    if (names_out) names_out[i] = w->prof_name[i];
  }
  *n_out = n;
  return MOE_OK;
}

int moe_sync_status(moe_ws* w, moe_stream_t stream) {
  if (!w) return MOE_EINVAL;
  MOE_CUDA_TRY(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
  int32_t e = 0;
  MOE_CUDA_TRY(cudaMemcpy(&e, w->error, 4, cudaMemcpyDeviceToHost));
  MOE_CUDA_TRY(cudaMemset(w->error, 0, 4));
  // a grid-barrier wait that gave up leaves the barrier's count behind: start it afresh
  if (e == MOE_ETIMEOUT) MOE_CUDA_TRY(cudaMemset(w->bar, 0, kBarWords * sizeof(unsigned long long)));
  return e;
}

// ------------------------------------------------------------ hot path
int moe_route(const uint16_t* x, const uint16_t* w_router, const float* bias, float* logits_io, int T, int H, int E,
              int k, int32_t* topk_ids, float* topk_w, int32_t* err_dev, moe_stream_t stream) {
  if (T < 0 || E < 1 || E > kMaxE || k < 1 || k > kMaxK || k > E || !logits_io || !topk_ids || !topk_w)
    return MOE_EINVAL;
  if (w_router && (!x || H <= 0 || H % 8)) return MOE_EINVAL;
  if (T == 0) return MOE_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int rc;
  if (w_router && (rc = launch_router(x, w_router, bias, nullptr, logits_io, nullptr, T, H, E, s))) return rc;
  return launch_topk(logits_io, T, E, k, topk_ids, topk_w, err_dev, s);
}

int moe_group(const int32_t* topk_ids, int T, int k, int E, int layer, moe_cache* c, moe_ws* ws, moe_stream_t stream) {
  if (!topk_ids || !c || !ws || T < 0 || T > ws->maxT || k != ws->s.k || E != c->E || E != ws->s.E || E > kMaxE ||
      layer < 0 || layer >= c->L)
    return MOE_EINVAL;
  if (T == 0) return MOE_OK;
  return launch_group(topk_ids, T, k, E, layer, c, ws, reinterpret_cast<cudaStream_t>(stream));
}

// Argument checks shared by the forward calls; MOE_OK when they pass.
static int forward_args_ok(const moe_layer_desc* d, const uint16_t* x, void* y, int T, const moe_cache* c,
                           const moe_ws* ws, bool prefill) {
  if (!d || !x || !y || !c || !ws || !d->w_router) return MOE_EINVAL;
  const moe_layer_shape& s = d->s;
  if (!shape_ok(s) || T < 0 || T > ws->maxT || s.H != ws->s.H || s.k != ws->s.k || s.E != ws->s.E ||
      s.I > ws->s.I || s.I_shared > ws->s.I_shared || s.E != c->E || s.H != c->H || s.I != c->I || d->layer < 0 ||
      d->layer >= c->L)
    return MOE_EINVAL;
  if (s.I_shared > 0 && (!d->shared_blob || !d->w_shared_gate)) return MOE_EINVAL;
  if (prefill && (!prefill_supported(s) || (reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(y) & 15) ||
                  (reinterpret_cast<uintptr_t>(d->w_router) & 15) ||
                  (s.I_shared > 0 && (reinterpret_cast<uintptr_t>(d->w_shared_gate) & 15))))
    return MOE_EINVAL;
  return MOE_OK;
}

int moe_layer_forward_streamed(const moe_layer_desc* d, const uint16_t* x, void* y, int y_is_fp32, int T,
                               moe_cache* c, moe_ws* ws, int U, int buffers, moe_stream_t stream,
                               moe_stream_t copy_stream) {
  int rc;
  if ((rc = forward_args_ok(d, x, y, T, c, ws, true))) return rc;
  if (U < 1 || (buffers != 1 && buffers != 2) || buffers * U > c->nstaging || !c->backing || !copy_stream ||
      copy_stream == stream)
    return MOE_EINVAL;
  if (T == 0) return MOE_OK;
  const moe_layer_shape& s = d->s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  ws->prof_n = 0;
  {
    ProfScope p(ws, "router", st);
    if ((rc = launch_prefill_router(d, x, T, ws, st))) return rc;
  }
  {
    ProfScope p(ws, "topk", st);
    if ((rc = launch_topk(ws->logits, T, s.E, s.k, ws->topk_ids, ws->topk_w, ws->error, st))) return rc;
  }
  {
    ProfScope p(ws, "group", st);
    if ((rc = launch_group(ws->topk_ids, T, s.k, s.E, d->layer, c, ws, st, false))) return rc;
  }
  return launch_prefill_streamed(d, c, x, y, y_is_fp32, T, U, buffers, ws, st,
                                 reinterpret_cast<cudaStream_t>(copy_stream));
}

int moe_layers_forward_streamed(const moe_layer_desc* d, int L, float* x_res, uint16_t* xn, uint16_t* y, int T,
                                moe_cache* c, moe_ws* ws, int buffers, float eps, moe_stream_t stream,
                                moe_stream_t copy_stream) {
  if (!d || L < 1 || !x_res || !xn || !y || (buffers != 1 && buffers != 2) || !(eps > 0.f) || !c || !c->backing ||
      !copy_stream || copy_stream == stream)
    return MOE_EINVAL;
  int rc;
  for (int l = 0; l < L; ++l) {
    if ((rc = forward_args_ok(&d[l], xn, y, T, c, ws, true))) return rc;
    if (d[l].s.H != d[0].s.H || d[l].s.E != d[0].s.E || d[l].s.k != d[0].s.k) return MOE_EINVAL;
  }
  if (size_t(buffers) * d[0].s.E > size_t(c->nstaging) || (reinterpret_cast<uintptr_t>(x_res) & 15) ||
      d[0].s.H % 4 || d[0].s.H > 4096)
    return MOE_EINVAL;
  if (T == 0) return MOE_OK;
  ws->prof_n = 0;
  return launch_prefill_layers_streamed(d, L, x_res, xn, y, T, c, ws, buffers, eps, reinterpret_cast<cudaStream_t>(stream),
                                        reinterpret_cast<cudaStream_t>(copy_stream));
}

int moe_layer_forward(const moe_layer_desc* d, const uint16_t* x, void* y, int y_is_fp32, int T, moe_cache* c,
                      moe_ws* ws, int mode, moe_stream_t stream) {
  if (!d || !x || !y || !c || !ws || !d->w_router) return MOE_EINVAL;
  const moe_layer_shape& s = d->s;
  if (!shape_ok(s) || T < 0 || T > ws->maxT || s.H != ws->s.H || s.k != ws->s.k || s.E != ws->s.E ||
      s.I > ws->s.I || s.I_shared > ws->s.I_shared || s.E != c->E || s.H != c->H || s.I != c->I || d->layer < 0 ||
      d->layer >= c->L)
    return MOE_EINVAL;
  if (s.I_shared > 0 && (!d->shared_blob || !d->w_shared_gate)) return MOE_EINVAL;
  if (mode != MOE_MODE_AUTO && mode != MOE_MODE_DECODE && mode != MOE_MODE_PREFILL) return MOE_EINVAL;
  if (T == 0) return MOE_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int rc;
  // decode kernels for small windows, tcgen05 grouped GEMMs from kPrefillMinTokens on
  const bool prefill_ok = prefill_supported(s) && !(reinterpret_cast<uintptr_t>(x) & 15) &&
                          !(reinterpret_cast<uintptr_t>(y) & 15) && !(reinterpret_cast<uintptr_t>(d->w_router) & 15) &&
                          !(s.I_shared > 0 && (reinterpret_cast<uintptr_t>(d->w_shared_gate) & 15));
  if (mode == MOE_MODE_PREFILL && !prefill_ok) return MOE_EINVAL;
  const bool prefill = mode == MOE_MODE_PREFILL || (mode == MOE_MODE_AUTO && T >= kPrefillMinTokens && prefill_ok);
  ws->prof_n = 0;
  if (!prefill && ws->decode_path == MOE_DECODE_FUSED) {  // one cooperative kernel where the shapes fit
    ProfScope p(ws, "decode_fused", st);
    rc = launch_decode_fused(d, c, x, y, y_is_fp32, T, ws, st);
    if (rc != kNotFused) return rc;
    ws->prof_n = 0;
  }
  {
    ProfScope p(ws, "router", st);
    if (prefill)
      rc = launch_prefill_router(d, x, T, ws, st);
    else
      rc = launch_router(x, d->w_router, d->bias, s.I_shared > 0 ? d->w_shared_gate : nullptr, ws->logits,
                         ws->gate_logit, T, s.H, s.E, st, ws->x16, ws->xscale);
    if (rc) return rc;
  }
  if (!prefill && T <= 32 && T * s.k <= 4096) {  // small windows: top-k and grouping in one launch
    ProfScope p(ws, "topk_group", st);
    if ((rc = launch_topk_group(ws->logits, T, s.k, s.E, d->layer, c, ws, st))) return rc;
  } else {
    {
      ProfScope p(ws, "topk", st);
      if ((rc = launch_topk(ws->logits, T, s.E, s.k, ws->topk_ids, ws->topk_w, ws->error, st))) return rc;
    }
    {
      ProfScope p(ws, "group", st);
      if ((rc = launch_group(ws->topk_ids, T, s.k, s.E, d->layer, c, ws, st))) return rc;
    }
  }
  if (prefill) return launch_prefill_experts(d, c, x, y, y_is_fp32, T, ws, st);
  {
    ProfScope p(ws, "gateup_decode", st);
    if ((rc = launch_gateup_decode(d, T, ws, st))) return rc;
  }
  {
    ProfScope p(ws, "down_decode", st);
    if ((rc = launch_down_decode(d, T, ws, st))) return rc;
  }
  ProfScope p(ws, "combine", st);
  return launch_combine(d, y, y_is_fp32, T, ws, st);
}

int cache_heat_update(moe_cache* c, const int32_t* topk_ids, int T, int k, int layer, int32_t* err_dev,
                      moe_stream_t stream) {
  if (!c || !topk_ids || T < 0 || k < 1 || layer < 0 || layer >= c->L) return MOE_EINVAL;
  return launch_heat_update(c, topk_ids, T, k, layer, err_dev, reinterpret_cast<cudaStream_t>(stream));
}

int cache_plan_swaps(moe_cache* c, const moe_policy_cfg* p, moe_swap* plan_dev, int32_t* n_dev, moe_stream_t stream) {
  if (!c || !p || !plan_dev || !n_dev || p->max_swaps < 0 || p->max_swaps > 4096 || !(p->threshold > 0.f) ||
      size_t(c->L) * c->E > 32768 || c->L > 1024)
    return MOE_EINVAL;
  return launch_plan_swaps(c, p, plan_dev, n_dev, reinterpret_cast<cudaStream_t>(stream));
}

int moe_cache_apply_swaps(moe_cache* c, const moe_swap* plan_dev, const int32_t* n_dev, moe_stream_t compute,
                          moe_stream_t copy) {
  if (!c || !plan_dev || !n_dev || !c->backing) return MOE_EINVAL;
  // each planned swap reuses a distinct slot, so at most min(nslots, 4096) swaps exist
  return launch_apply_swaps(c, plan_dev, n_dev, c->nslots < 4096 ? c->nslots : 4096,
                            reinterpret_cast<cudaStream_t>(compute), reinterpret_cast<cudaStream_t>(copy));
}

int cache_lru_plan(moe_cache* c, const moe_ws* ws, int layer, int K, moe_swap* plan_dev, int32_t* n_dev,
                   moe_stream_t stream) {
  if (!c || !ws || !plan_dev || !n_dev || layer < 0 || layer >= c->L || K < 1 || K > kLruMaxK || c->nslots < 1 ||
      c->nslots >= (1 << 24))
    return MOE_EINVAL;
  return launch_lru_plan(c, ws, layer, K, plan_dev, n_dev, reinterpret_cast<cudaStream_t>(stream));
}

int moe_cache_apply_lru(moe_cache* c, const moe_swap* plan_dev, const int32_t* n_dev, moe_stream_t compute,
                        moe_stream_t copy) {
  if (!c || !plan_dev || !n_dev || !c->backing) return MOE_EINVAL;
  return launch_apply_swaps(c, plan_dev, n_dev, kLruMaxK, reinterpret_cast<cudaStream_t>(compute),
                            reinterpret_cast<cudaStream_t>(copy), /*flat_cold=*/true);
}

}  // extern "C"
