// Prefill path: the router and the grouped expert GEMMs on the tcgen05 tensor cores.
//
// Strata expert paths, "PCIe 搬运怎样与计算重叠？" / FreeToken notes section 3.1:
// a long prompt is processed in chunks and its tokens are grouped per expert,
// so every expert runs once per chunk as a GEMM over its group.  Here:
//   router:   [W_r; w_gate] (E+1 x H) . X^T (H x T)      -> logits, gate logit
//   gate/up:  [Wg; Wu] (2I x H) . X_g^T (H x n)           -> h = SiLU(g) * u, max|h| per row
//   down:     Wd (H x I) . h_g^T (I x n)                  -> y += w * o        (fp32)
//
// Operands.  A = 128 weight rows per tile.  Expert weights are dequantised by
// the CTA from E2M1 codes x E4M3 block scale -- exact in bf16 and in f16:
// every product has at most 6 significant bits and magnitude 2^-10 .. 2688 --
// straight into shared memory in the 128-byte-swizzled K-major layout the
// tensor core reads (router rows are bf16 already and are copied as they
// are).  B = up to 256 token rows of the group, gathered with cp.async: the
// bf16 activations themselves for the router and gate/up (both operands bf16,
// so nothing is rounded), and for the down GEMM h as f16 times a per-row power
// of two (both operands f16; h keeps 11 significant bits -- bf16 h, with 8,
// would leave about 1.2% of rms(y) as error).  D = fp32 in tensor memory
// (tcgen05.mma kind::f16, issued by one thread), read back with tcgen05.ld.
// The global scale is applied in the epilogue, in fp32.
//
// Roles (one persistent CTA per SM, 9 warps):
//   warps 0-3  producers: cp.async of the raw code/scale row of each thread
//              and of the token rows, dequantisation into the A stage;
//   warps 4-7  epilogue: TMEM -> registers -> h / y / logits;
//   warp  8    TMEM owner (512 columns = two 256-column accumulators) and
//              MMA issuer (one lane).
// A 4-stage ring guarded by mbarriers (full: 128 producer arrivals, empty:
// tcgen05.commit) feeds the MMAs; the two accumulators (acc_full: commit,
// acc_empty: 128 epilogue arrivals) let the epilogue of one tile overlap the
// MMAs of the next.  Every wait is bounded (2 s) and reports MOE_ETIMEOUT
// instead of hanging; the MMA issuer drains its MMAs before TMEM is freed.
#include "internal.h"

namespace moe {
namespace prefill {

constexpr int kBK = 64;           // K per stage (one 128-byte swizzle atom of bf16)
constexpr int kNT = 256;          // tokens per tile (accumulator columns)
constexpr int kStages = 4;
constexpr int kPD = kStages - 1;  // chunks in flight ahead of the one being dequantised
constexpr int kProducers = 128;
constexpr int kEpi = 128;
constexpr int kThreads = kProducers + kEpi + 32;
constexpr int kABytes = 128 * kBK * 2;   // 16 KB
constexpr int kBBytes = kNT * kBK * 2;   // 32 KB
constexpr int kCodeBytes = 128 * 32;     // raw codes of one chunk: 32 bytes per row
constexpr int kScaleBytes = 128 * 4;     // raw scales of one chunk: 4 bytes per row
constexpr int kBarriers = 2 * kStages + 2 + 2 + 1;
constexpr size_t kSmemBytes = size_t(kStages) * (kABytes + kBBytes + kCodeBytes + kScaleBytes) + kBarriers * 8 + 8 +
                              2 * kNT * 8 + 1024;
constexpr uint64_t kWaitNs = 2000000000ull;  // a wait that lasts this long has failed

enum Mode { kGateUp = 0, kDown = 1, kRouter = 2 };

__device__ __forceinline__ uint32_t su32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
// 128-byte swizzled K-major atom: row r, 16-byte chunk c
__device__ __forceinline__ int sw128(int r, int c) { return (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4); }

__device__ __forceinline__ uint64_t kmajor_desc(const void* base) {
  const uint64_t a = su32(base);
  return ((a >> 4) & 0x3FFF) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) | (uint64_t(1) << 46) |
         (uint64_t(2) << 61);
}
__device__ __forceinline__ void bar_init(uint64_t* b, int n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n));
}
__device__ __forceinline__ void bar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Waits for the phase with parity `par` to complete; false after kWaitNs.
__device__ __forceinline__ bool bar_wait(uint64_t* b, uint32_t par) {
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(su32(b)), "r"(par)
        : "memory");
    if (ok) return true;
    if (i == 0) t0 = now_ns();
    else if ((i & 255) == 0 && now_ns() - t0 > kWaitNs) return false;
  }
}
__device__ __forceinline__ void commit_to(uint64_t* b) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(b))
               : "memory");
}
// cp.async without a compiler memory clobber: the sources are never written by
// this kernel, and the wait_group below carries the ordering of shared memory.
__device__ __forceinline__ void cp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(su32(dst)), "l"(src));
}
__device__ __forceinline__ void cp4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(su32(dst)), "l"(src));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_wait_pd() { asm volatile("cp.async.wait_group %0;" ::"n"(kPD) : "memory"); }
__device__ __forceinline__ void cp_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kEpi) : "memory"); }

struct Args {
  const int32_t* num_groups;
  const int32_t* grp_off;
  const uint8_t* const* grp_blob;
  const int32_t* ent_tok;
  const int32_t* ent_pos;
  const int32_t* tile_off;   // [G+1] N tiles before each group
  const uint16_t* bsrc;      // B rows: x [T, H] bf16 (router, gate/up) or h16 [rows, Imax] f16 (down)
  int bstride;               // elements per B row
  float* h;                  // gate/up output h (fp32) [maxTk + maxT, Imax]
  float* hmax;               // gate/up: max|h| per row [maxTk + maxT]
  const float* topk_w;       // [T*k]
  const float* gate_logit;   // [T]
  float* yacc;               // down output accumulator [T, H] fp32
  const uint8_t* shared_blob;
  const uint16_t* w_router;  // router: [E, H] bf16
  const uint16_t* w_gate;    // router: [H] bf16 shared-expert gate row, or null
  const float* bias;         // router: [E] or null
  float* logits;             // router: [T, E]
  float* gate_out;           // router: [T]
  int T, H, I, I_s, Imax, maxTk, k, E;
  DevBlobLayout lay_r, lay_s;
  int32_t* err;
};

struct Item {
  const uint8_t* blob;
  int shared, nt, mt, n, e0, C, KC;
};

// Work list of one GEMM: (routed N tile, M tile) pairs in group order (M tile
// fastest, so CTAs running at the same time share the token tile in L2), then
// the shared expert's tiles; for the router, (token tile, row tile) pairs.
struct Sched {
  int G, routed_tiles, mt_r, mt_s, n_items;
};

template <int MODE>
__device__ __forceinline__ Sched make_sched(const Args& a) {
  Sched s;
  const int ntok = (a.T + kNT - 1) / kNT;
  if (MODE == kRouter) {
    s.G = 0;
    s.routed_tiles = 0;
    s.mt_r = (a.E + (a.w_gate ? 1 : 0) + 127) / 128;
    s.mt_s = 0;
    s.n_items = ntok * s.mt_r;
    return s;
  }
  s.G = *a.num_groups;
  s.routed_tiles = a.tile_off[s.G];
  s.mt_r = MODE == kGateUp ? (2 * a.I) / 128 : a.H / 128;
  s.mt_s = a.shared_blob ? (MODE == kGateUp ? (2 * a.I_s) / 128 : a.H / 128) : 0;
  s.n_items = s.routed_tiles * s.mt_r + ntok * s.mt_s;
  return s;
}

template <int MODE>
__device__ __forceinline__ void item_of(const Args& a, const Sched& sc, int it, Item& x) {
  if (MODE == kRouter) {
    x.nt = it / sc.mt_r;
    x.mt = it - x.nt * sc.mt_r;
    x.shared = 0;
    x.e0 = 0;
    x.n = min(kNT, a.T - x.nt * kNT);
    x.blob = nullptr;
    x.C = a.H;
  } else if (it < sc.routed_tiles * sc.mt_r) {
    const int ti = it / sc.mt_r;
    x.mt = it - ti * sc.mt_r;
    int lo = 0, hi = sc.G - 1;  // last group with tile_off[g] <= ti
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.tile_off[mid] <= ti) lo = mid;
      else hi = mid - 1;
    }
    x.nt = ti - a.tile_off[lo];
    x.shared = 0;
    x.e0 = a.grp_off[lo];
    x.n = min(kNT, a.grp_off[lo + 1] - x.e0 - x.nt * kNT);
    x.blob = a.grp_blob[lo];
    x.C = MODE == kGateUp ? a.H : a.I;
  } else {
    const int r = it - sc.routed_tiles * sc.mt_r;
    x.nt = r / sc.mt_s;
    x.mt = r - x.nt * sc.mt_s;
    x.shared = 1;
    x.e0 = 0;
    x.n = min(kNT, a.T - x.nt * kNT);
    x.blob = a.shared_blob;
    x.C = MODE == kGateUp ? a.H : a.I_s;
  }
  x.KC = x.C / kBK;
}

// Weight row of A-tile row r.  gate/up tiles interleave: within each 32-row
// quarter, rows 0-15 are gate rows and rows 16-31 the up rows of the same 16
// intermediates, so each epilogue warp holds both halves of its h values.
template <int MODE>
__device__ __forceinline__ void a_row(int mt, int r, int& mat, int& wrow) {
  if (MODE == kGateUp) {
    const int q = r >> 5, l = r & 31;
    mat = l < 16 ? 0 : 1;
    wrow = mt * 64 + q * 16 + (l & 15);
  } else {
    mat = 2;
    wrow = mt * 128 + r;
  }
}

// B row (in bsrc) of token-tile column j.
template <int MODE>
__device__ __forceinline__ int b_row(const Args& a, const Item& x, int j) {
  const int ent = x.nt * kNT + j;
  if (MODE == kRouter) return ent;
  if (MODE == kGateUp) return x.shared ? ent : a.ent_tok[x.e0 + ent];
  return x.shared ? a.maxTk + ent : x.e0 + ent;
}

__device__ __forceinline__ uint32_t bf16x2_of(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// 32 code bytes + 4 E4M3 scales of one weight row chunk -> 64 values code x
// scale (exact) as bf16 (BF16) or f16 in the row's 8 swizzled 16-byte chunks.
template <bool BF16>
__device__ __forceinline__ void dequant_row(const uint8_t* codes, const uint8_t* scales, uint8_t* at, int row) {
  const uint4 c0 = *reinterpret_cast<const uint4*>(codes), c1 = *reinterpret_cast<const uint4*>(codes + 16);
  const uint32_t sc4 = *reinterpret_cast<const uint32_t*>(scales);
  const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
  for (int blk = 0; blk < 4; ++blk) {  // 16 values = 8 code bytes, one scale
    const uint32_t sb = (sc4 >> (8 * blk)) & 0xffu;
    const uint32_t sh = e4m3x2_to_f16x2(sb | (sb << 8));  // the scale in both halves, f16 (exact)
    // bf16: the scale x 2^112 (exact: at most 4 significant bits, below 2^121)
    const float sf = BF16 ? f16x2_to_f32x2(sh).x * 0x1p112f : 0.f;
    const uint32_t sp = BF16 ? bf16x2_of(sf, sf) : sh;
    uint32_t hv[8];
#pragma unroll
    for (int w2 = 0; w2 < 2; ++w2) {
      uint32_t o[4];
      asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
          "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
          "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
          : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
          : "r"(cw[2 * blk + w2]));
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        if (BF16) {
          // f16 bits of an E2M1 value moved into the bf16 field layout: read as
          // bf16 they are the value x 2^-112 (exponent bias 15 vs 127); zero
          // stays zero and the sign stays in place.  The 2^112 in the scale
          // operand cancels the factor, so the product is code x scale exactly.
          const uint32_t t = ((o[b] >> 3) & 0x0fff0fffu) | (o[b] & 0x80008000u);
          asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(hv[4 * w2 + b]) : "r"(t), "r"(sp));
        } else {
          asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(hv[4 * w2 + b]) : "r"(o[b]), "r"(sp));
        }
      }
    }
    *reinterpret_cast<uint4*>(at + sw128(row, 2 * blk)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
    *reinterpret_cast<uint4*>(at + sw128(row, 2 * blk + 1)) = make_uint4(hv[4], hv[5], hv[6], hv[7]);
  }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) k_gemm(Args a) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the 128-byte swizzle pattern is a function of the shared address: atoms start on 1 KB
  uint8_t* smem = smem_raw + ((1024u - (su32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem;                                        // [kStages][16 KB]
  uint8_t* sB = sA + kStages * kABytes;                      // [kStages][32 KB]
  uint8_t* sCode = sB + kStages * kBBytes;                   // [kStages][128][32]
  uint8_t* sScale = sCode + kStages * kCodeBytes;            // [kStages][128][4]
  uint64_t* full = reinterpret_cast<uint64_t*>(sScale + kStages * kScaleBytes);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;   // [2]
  uint64_t* acc_empty = acc_full + 2;     // [2]
  uint64_t* drain = acc_empty + 2;
  uint32_t* taddr_s = reinterpret_cast<uint32_t*>(drain + 1);
  int32_t* s_tok = reinterpret_cast<int32_t*>(drain + 2);  // [2][kNT] down: token of each column
  float* s_w = reinterpret_cast<float*>(s_tok + 2 * kNT);  // [2][kNT] down: its weight
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const Sched sc = make_sched<MODE>(a);

  if (warp == 8) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(taddr_s)),
                 "r"(2 * kNT));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      bar_init(&full[s], kProducers);
      bar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      bar_init(&acc_full[b], 1);
      bar_init(&acc_empty[b], kEpi);
    }
    bar_init(drain, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  const uint32_t taddr = *taddr_s;
  bool failed = false;

  if (warp == 8) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int q = 0, done = 0;
      for (int it = blockIdx.x; it < sc.n_items && !failed; it += gridDim.x, ++done) {
        Item x;
        item_of<MODE>(a, sc, it, x);
        const int npad = (x.n + 15) & ~15;
        const int buf = done & 1;
        // kind::f16: D f32, A and B both bf16 (router, gate/up) or both f16
        // (down), both K-major, N = npad, M = 128
        const uint32_t ab = MODE == kDown ? 0u : 1u;
        const uint32_t idesc = (1u << 4) | (ab << 7) | (ab << 10) | (uint32_t(npad >> 3) << 17) |
                               (uint32_t(128 >> 4) << 24);
        if (done >= 2 && !bar_wait(&acc_empty[buf], ((done >> 1) - 1) & 1)) {
          failed = true;
          break;
        }
        const uint32_t dt = taddr + uint32_t(buf * kNT);
        for (int kc = 0; kc < x.KC; ++kc, ++q) {
          const int s = q % kStages;
          if (!bar_wait(&full[s], (q / kStages) & 1)) {
            failed = true;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;");
          const uint64_t da = kmajor_desc(sA + s * kABytes), db = kmajor_desc(sB + s * kBBytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint32_t accum = (kc > 0 || k > 0) ? 1u : 0u;
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dt),
                "l"(da + uint64_t(k * 2)), "l"(db + uint64_t(k * 2)), "r"(idesc), "r"(accum));
          }
          commit_to(&empty[s]);
        }
        if (!failed) commit_to(&acc_full[buf]);
      }
      // every MMA issued has completed before the accumulators are freed
      commit_to(drain);
      if (!bar_wait(drain, 0)) failed = true;
      if (failed) set_error(a.err, MOE_ETIMEOUT);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ producers
    int iss_it = blockIdx.x, iss_kc = 0, iss_q = 0;
    Item ix;
    bool iss_ok = iss_it < sc.n_items;
    const uint16_t* bp[kNT / 16];  // this thread's token rows: j = tid/8 + 16m, chunk tid%8
    const uint8_t* code_p = nullptr;
    const uint8_t* scale_p = nullptr;
    const uint16_t* arow = nullptr;  // router: this thread's weight row
    auto load_item = [&]() {
      item_of<MODE>(a, sc, iss_it, ix);
#pragma unroll
      for (int m = 0; m < kNT / 16; ++m) {
        const int j = (tid >> 3) + 16 * m;
        bp[m] = j < ix.n ? a.bsrc + size_t(b_row<MODE>(a, ix, j)) * a.bstride + (tid & 7) * 8 : nullptr;
      }
      if (MODE == kRouter) {
        const int r = ix.mt * 128 + tid;
        arow = r < a.E ? a.w_router + size_t(r) * a.H : (r == a.E ? a.w_gate : nullptr);
      } else {
        int mat, wrow;
        a_row<MODE>(ix.mt, tid, mat, wrow);
        const DevBlobLayout& lay = ix.shared ? a.lay_s : a.lay_r;
        code_p = ix.blob ? ix.blob + lay.code_off[mat] + size_t(wrow) * (ix.C / 2) : nullptr;
        scale_p = ix.blob ? ix.blob + lay.scale_off[mat] + size_t(wrow) * (ix.C / 16) : nullptr;
      }
    };
    if (iss_ok) load_item();
    auto issue = [&]() {
      if (iss_ok) {
        const int s = iss_q % kStages;
        if (!failed && iss_q >= kStages && !bar_wait(&empty[s], ((iss_q / kStages) - 1) & 1)) failed = true;
        failed = __any_sync(0xffffffffu, failed);  // warp-uniform
        if (!failed) {
          if (MODE == kRouter) {
            if (arow) {
              uint8_t* at = sA + s * kABytes;
#pragma unroll
              for (int c = 0; c < 8; ++c) cp16(at + sw128(tid, c), arow + iss_kc * kBK + c * 8);
            }
          } else if (code_p) {
            uint8_t* cd = sCode + s * kCodeBytes + tid * 32;
            cp16(cd, code_p + iss_kc * 32);
            cp16(cd + 16, code_p + iss_kc * 32 + 16);
            cp4(sScale + s * kScaleBytes + tid * 4, scale_p + iss_kc * 4);
          }
          uint8_t* bt = sB + s * kBBytes;
#pragma unroll
          for (int m = 0; m < kNT / 16; ++m)
            if (bp[m]) cp16(bt + sw128((tid >> 3) + 16 * m, tid & 7), bp[m] + iss_kc * kBK);
        }
        ++iss_q;
        if (++iss_kc == ix.KC) {
          iss_kc = 0;
          iss_it += gridDim.x;
          iss_ok = iss_it < sc.n_items;
          if (iss_ok) load_item();
        }
      }
      cp_commit();
    };
    for (int p = 0; p < kPD; ++p) issue();

    int q = 0;
    for (int it = blockIdx.x; it < sc.n_items; it += gridDim.x) {
      Item x;
      item_of<MODE>(a, sc, it, x);
      for (int kc = 0; kc < x.KC; ++kc, ++q) {
        issue();       // chunk q + kPD
        cp_wait_pd();  // this thread's copies of chunk q have landed
        const int s = q % kStages;
        if (MODE != kRouter && x.blob && !failed)
          dequant_row<MODE == kGateUp>(sCode + s * kCodeBytes + tid * 32, sScale + s * kScaleBytes + tid * 4,
                                       sA + s * kABytes, tid);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        bar_arrive(&full[s]);
      }
    }
    cp_wait_all();
    if (failed) set_error(a.err, MOE_ETIMEOUT);
  } else {
    // ------------------------------------------------------------ epilogue
    const int et = tid - kProducers, qw = warp & 3;
    int done = 0;
    for (int it = blockIdx.x; it < sc.n_items; it += gridDim.x, ++done) {
      Item x;
      item_of<MODE>(a, sc, it, x);
      const int buf = done & 1;
      if (MODE == kDown) {
        for (int j = et; j < x.n; j += kEpi) {
          const int ent = x.nt * kNT + j;
          int tok;
          float w;
          if (x.shared) {
            tok = ent;
            w = sigmoid_f32(a.gate_logit[tok]);
          } else {
            const int pos = a.ent_pos[x.e0 + ent];
            tok = pos / a.k;
            w = a.topk_w[pos];
          }
          // B row = h x 2^p (the power of two the conversion to f16 chose)
          const int hrow = x.shared ? a.maxTk + ent : x.e0 + ent;
          s_tok[buf * kNT + j] = tok;
          s_w[buf * kNT + j] = w / pow2_scale_for(a.hmax[hrow]);
        }
        epi_sync();
      }
      if (!failed && !bar_wait(&acc_full[buf], (done >> 1) & 1)) failed = true;
      failed = __any_sync(0xffffffffu, failed);
      asm volatile("tcgen05.fence::after_thread_sync;");
      const float gs0 = x.blob ? reinterpret_cast<const BlobHeader*>(x.blob)->gscale[MODE == kGateUp ? 0 : 2] : 0.f;
      const float gs1 = x.blob ? reinterpret_cast<const BlobHeader*>(x.blob)->gscale[1] : 0.f;
      const int npad = (x.n + 15) & ~15;
      const uint32_t tb = taddr + uint32_t(buf * kNT) + (uint32_t(qw * 32) << 16);
      const int row = x.mt * 128 + qw * 32 + lane;  // router / down: output row of this lane
      const float rbias = (MODE == kRouter && a.bias && row < a.E) ? a.bias[row] : 0.f;
      for (int c0 = 0; c0 < npad && !failed; c0 += 16) {
        uint32_t v[16];
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
              "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
            : "r"(tb + uint32_t(c0)));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        if (MODE == kGateUp) {
          // lanes 0-15 hold gate rows, 16-31 the matching up rows: the low lanes
          // finish columns 0-7 of this slice, the high lanes columns 8-15
          const bool hi = lane >= 16;
          const int i = x.mt * 64 + qw * 16 + (lane & 15);
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const float mine_lo = __uint_as_float(v[jj]), mine_hi = __uint_as_float(v[jj + 8]);
            const float recv = __shfl_xor_sync(0xffffffffu, hi ? mine_lo : mine_hi, 16);
            const float g = hi ? recv : mine_lo, u = hi ? mine_hi : recv;
            const int j = c0 + jj + (hi ? 8 : 0);
            const int ent = x.nt * kNT + j;
            const int hrow = x.shared ? a.maxTk + ent : x.e0 + ent;
            float hv = 0.f;
            if (j < x.n) {
              hv = x.blob ? silu_f32(g * gs0) * (u * gs1) : 0.f;
              a.h[size_t(hrow) * a.Imax + i] = hv;
            }
            // max|h| of this column over the warp's 16 intermediates
            float m = fabsf(hv);
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            if ((lane & 15) == 0 && j < x.n) atomicMax(reinterpret_cast<unsigned int*>(a.hmax) + hrow, __float_as_uint(m));
          }
        } else if (MODE == kDown) {
          if (x.blob) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int j = c0 + jj;
              if (j < x.n)
                atomicAdd(a.yacc + size_t(s_tok[buf * kNT + j]) * a.H + row,
                          __uint_as_float(v[jj]) * gs0 * s_w[buf * kNT + j]);
            }
          }
        } else {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int j = c0 + jj;
            const int tok = x.nt * kNT + j;
            const float d = __uint_as_float(v[jj]);
            if (j < x.n) {
              if (row < a.E) a.logits[size_t(tok) * a.E + row] = __fadd_rn(d, rbias);
              else if (row == a.E && a.w_gate) a.gate_out[tok] = d;
            }
          }
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;");
      bar_arrive(&acc_empty[buf]);
    }
    if (failed) set_error(a.err, MOE_ETIMEOUT);
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  if (warp == 8) {
    asm volatile("tcgen05.fence::after_thread_sync;");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(2 * kNT));
  }
}

// N tiles per group, as an exclusive prefix: tile_off[g] = sum_{g'<g} ceil(n_g'/kNT).
__global__ void __launch_bounds__(1024) k_tiles(const int32_t* __restrict__ num_groups, const int32_t* __restrict__ grp_off,
                                                int32_t* __restrict__ tile_off) {
  pdl_trigger();
  pdl_wait();
  __shared__ int ws[32];
  const int G = *num_groups;
  int carry = 0;
  for (int base = 0; base < G; base += blockDim.x) {
    const int g = base + threadIdx.x;
    const int v = g < G ? (grp_off[g + 1] - grp_off[g] + kNT - 1) / kNT : 0;
    int x = v;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) ws[w] = x;
    __syncthreads();
    if (w == 0) {
      int s = lane < (blockDim.x >> 5) ? ws[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += y;
      }
      ws[lane] = s;
    }
    __syncthreads();
    const int before = (w ? ws[w - 1] : 0) + carry;
    if (g < G) tile_off[g] = before + x - v;
    carry += ws[(blockDim.x >> 5) - 1];
    __syncthreads();
  }
  if (threadIdx.x == 0) tile_off[G] = carry;
}

// h (fp32) -> f16 times a per-row power of two chosen from max|h_row|.
__global__ void __launch_bounds__(256) k_h16(const float* __restrict__ h, const float* __restrict__ hmax,
                                             __half* __restrict__ h16, const int32_t* __restrict__ grp_off,
                                             const int32_t* __restrict__ num_groups, int Imax, int maxTk, int T,
                                             int has_shared) {
  pdl_trigger();
  pdl_wait();
  const int routed = grp_off[*num_groups];
  const int rows = routed + (has_shared ? T : 0);
  const int per = Imax / 4;
  for (size_t idx = size_t(blockIdx.x) * blockDim.x + threadIdx.x; idx < size_t(rows) * per;
       idx += size_t(gridDim.x) * blockDim.x) {
    const int rr = int(idx / per), c4 = int(idx - size_t(rr) * per);
    const int row = rr < routed ? rr : maxTk + (rr - routed);
    const float sc = pow2_scale_for(hmax[row]);
    const float4 f = reinterpret_cast<const float4*>(h + size_t(row) * Imax)[c4];
    __half2 p0 = __floats2half2_rn(f.x * sc, f.y * sc), p1 = __floats2half2_rn(f.z * sc, f.w * sc);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&p0);
    u.y = *reinterpret_cast<uint32_t*>(&p1);
    reinterpret_cast<uint2*>(h16 + size_t(row) * Imax)[c4] = u;
  }
}

// y = bf16(yacc)
__global__ void __launch_bounds__(256) k_cast_bf16(const float* __restrict__ yacc, uint16_t* __restrict__ y, size_t n4) {
  pdl_trigger();
  pdl_wait();
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += size_t(gridDim.x) * blockDim.x) {
    const float4 f = reinterpret_cast<const float4*>(yacc)[i];
    __nv_bfloat162 p0 = __floats2bfloat162_rn(f.x, f.y), p1 = __floats2bfloat162_rn(f.z, f.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&p0);
    u.y = *reinterpret_cast<uint32_t*>(&p1);
    reinterpret_cast<uint2*>(y)[i] = u;
  }
}

}  // namespace prefill

static int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

template <int MODE>
static int launch_gemm(const prefill::Args& a, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(prefill::k_gemm<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(prefill::kSmemBytes)) != cudaSuccess)
      return MOE_ECUDA;
    attr = true;
  }
  if (launch_pdl(prefill::k_gemm<MODE>, dim3(sm_count()), dim3(prefill::kThreads), prefill::kSmemBytes, s, a) !=
      cudaSuccess)
    return MOE_ECUDA;
  return MOE_OK;
}

bool prefill_supported(const moe_layer_shape& s) {
  return s.H >= 128 && s.I >= 64 && (s.I_shared == 0 || s.I_shared >= 64);
}

static prefill::Args base_args(const moe_layer_desc* d, int T, moe_ws* ws) {
  prefill::Args a = {};
  const moe_layer_shape& sh = d->s;
  const bool has_shared = sh.I_shared > 0 && d->shared_blob;
  a.num_groups = ws->num_groups;
  a.grp_off = ws->grp_off;
  a.grp_blob = ws->grp_blob;
  a.ent_tok = ws->ent_tok;
  a.ent_pos = ws->ent_pos;
  a.tile_off = ws->tile_off;
  a.h = ws->h;
  a.hmax = ws->hmax;
  a.topk_w = ws->topk_w;
  a.gate_logit = ws->gate_logit;
  a.shared_blob = has_shared ? reinterpret_cast<const uint8_t*>(d->shared_blob) : nullptr;
  a.T = T;
  a.H = sh.H;
  a.I = sh.I;
  a.I_s = has_shared ? sh.I_shared : 0;
  a.Imax = ws->s.I > ws->s.I_shared ? ws->s.I : ws->s.I_shared;
  a.maxTk = ws->maxT * ws->s.k;
  a.k = sh.k;
  a.E = sh.E;
  a.lay_r = dev_layout(sh.H, sh.I);
  a.lay_s = dev_layout(sh.H, has_shared ? sh.I_shared : sh.I);
  a.err = ws->error;
  return a;
}

int launch_prefill_router(const moe_layer_desc* d, const uint16_t* x, int T, moe_ws* ws, cudaStream_t s) {
  prefill::Args a = base_args(d, T, ws);
  a.bsrc = x;
  a.bstride = d->s.H;
  a.w_router = d->w_router;
  a.w_gate = d->s.I_shared > 0 ? d->w_shared_gate : nullptr;
  a.bias = d->bias;
  a.logits = ws->logits;
  a.gate_out = ws->gate_logit;
  return launch_gemm<prefill::kRouter>(a, s);
}

// The expert part of a prefill call: tiles, gate/up GEMM (h and max|h| per
// row), h -> f16 times a per-row power of two, down GEMM accumulating w*o
// into an fp32 buffer, and the output cast.
int launch_prefill_experts(const moe_layer_desc* d, const uint16_t* x, void* y, int y_is_fp32, int T, moe_ws* ws,
                           cudaStream_t s) {
  using namespace prefill;
  const moe_layer_shape& sh = d->s;
  Args a = base_args(d, T, ws);
  float* yacc = y_is_fp32 ? static_cast<float*>(y) : ws->yacc;
  a.yacc = yacc;
  {
    ProfScope p(ws, "tiles_zero", s);
    if (launch_pdl(k_tiles, dim3(1), dim3(1024), 0, s, ws->num_groups, ws->grp_off, ws->tile_off) != cudaSuccess)
      return MOE_ECUDA;
    MOE_CUDA_TRY(cudaMemsetAsync(yacc, 0, size_t(T) * sh.H * 4, s));
  }
  int rc;
  {
    ProfScope p(ws, "gateup_gemm", s);
    a.bsrc = x;
    a.bstride = sh.H;
    if ((rc = launch_gemm<kGateUp>(a, s))) return rc;
  }
  {
    ProfScope p(ws, "h16", s);
    if (launch_pdl(k_h16, dim3(sm_count() * 8), dim3(256), 0, s, ws->h, ws->hmax, ws->h16, ws->grp_off,
                   ws->num_groups, a.Imax, a.maxTk, T, a.shared_blob ? 1 : 0) != cudaSuccess)
      return MOE_ECUDA;
  }
  {
    ProfScope p(ws, "down_gemm", s);
    a.bsrc = reinterpret_cast<const uint16_t*>(ws->h16);
    a.bstride = a.Imax;
    if ((rc = launch_gemm<kDown>(a, s))) return rc;
  }
  if (!y_is_fp32) {
    ProfScope p(ws, "cast", s);
    const size_t n4 = size_t(T) * sh.H / 4;
    if (launch_pdl(k_cast_bf16, dim3(sm_count() * 8), dim3(256), 0, s, ws->yacc, static_cast<uint16_t*>(y), n4) !=
        cudaSuccess)
      return MOE_ECUDA;
  }
  return MOE_OK;
}

}  // namespace moe
