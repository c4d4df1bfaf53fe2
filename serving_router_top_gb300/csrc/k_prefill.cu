// Prefill path: the router and the grouped expert GEMMs on the tcgen05 tensor cores.
//
// Strata expert paths, "PCIe 搬运怎样与计算重叠？" / FreeToken notes section 3.1:
// a long prompt is processed in chunks and its tokens are grouped per expert,
// so every expert runs once per chunk as a GEMM over its group.  Here:
//   router:   [W_r; w_gate] (E+1 x H) . X^T (H x T)      -> logits, gate logit
//   gate/up:  [Wg; Wu] (2I x H) . X_g^T (H x n)           -> h = SiLU(g) * u
//   down:     Wd (H x I) . h_g^T (I x n)                  -> y += w * o        (fp32)
//
// Operands.  A = 128 weight rows per tile.  Expert weights are dequantised by
// the CTA from E2M1 codes x E4M3 block scale -- exact in bf16 and in f16:
// every product has at most 6 significant bits and magnitude 2^-10 .. 2688 --
// straight into shared memory in the 128-byte-swizzled K-major layout the
// tensor core reads (router rows are bf16 already and are copied as they
// are).  B = up to 192 token rows, one TMA box of 64 columns x 192 rows per
// chunk from a row-major matrix in which every token tile is contiguous: for
// the router x itself (bf16 like its weights); for gate/up the token rows
// copied into group order as f16 times a power of two per token (exact for
// bf16 values in the f16 normal range; see k_x16_grouped); for the down GEMM
// h as f16 times a power of two per row (h keeps 11 significant bits -- bf16
// h, with 8, would leave about 1.2% of rms(y) as error).  The epilogue divides
// the powers of two out again.  D = fp32 in tensor memory (tcgen05.mma
// kind::f16, issued by one thread), read back with tcgen05.ld.
// The global scale is applied in the epilogue, in fp32.
//
// Roles (one persistent CTA per SM, 27 warps):
//   warps 0-7   producers: two threads per weight row dequantise two chunks per
//               step from the code ring into their A stages (router rows:
//               cp.async straight into the A stage);
//   warps 8-23  epilogue: TMEM -> registers -> h / y / logits, four warps per
//               TMEM lane quadrant, each taking 16 of every 64 columns;
//   warp  24    TMEM owner (512 columns: two accumulators of up to 192) and
//               MMA issuer (one lane);
//   warp  25    B loader: one TMA box per chunk;
//   warp  26    code loader: per four chunks, one TMA box (128 bytes of each
//               of the tile's weight rows) per weight matrix from a 3-D map
//               over the expert's arena, and the rows' scales with cp.async,
//               into a ring of two code groups.
// Rings of 4 weight (A) and 5 token (B) stages guarded by mbarriers (full:
// one arrival per producer warp; full_b: the loader's expected bytes; empty,
// empty_b: tcgen05.commit) feed the MMAs; the two accumulators (acc_full:
// commit; acc_empty: one arrival per epilogue warp) let the epilogue of one
// tile overlap the MMAs of the next.  Every wait is bounded (2 s) and reports
// MOE_ETIMEOUT instead of hanging; the MMA issuer drains its MMAs before TMEM
// is freed.
#include <cudaTypedefs.h>

#include <cstring>

#include "internal.h"

namespace moe {
namespace prefill {

constexpr int kBK = 64;           // K per stage (one 128-byte swizzle atom of bf16)
constexpr int kNT = 192;          // tokens per tile (accumulator columns)
constexpr int kAccCols = 256;     // TMEM columns between the two accumulators (512 allocated)
constexpr int kAStages = 4;  // dequantised weight tiles
constexpr int kBStages = 5;  // token tiles
constexpr int kBPrefetch = 4;  // token tiles prefetched into L2 beyond the ring
constexpr int kProducers = 256;  // groups of eight warps, two threads per weight row in each
constexpr int kPGroups = kProducers / 256;
constexpr int kGChunks = 4;      // chunks per code group: one 128-byte line of every weight row
constexpr int kGStages = 2;      // code groups in flight
constexpr int kGCodeBytes = 128 * 128;  // raw codes of a group: [128 rows][128 B], 16-byte pieces swizzled
constexpr int kGScaleBytes = 128 * 16;  // raw scales of a group: [128 rows][16 B]
constexpr int kEpi = 512;  // sixteen warps: four per TMEM lane quadrant, each taking 16 of every 64 columns
constexpr int kEpiPerQuad = kEpi / 128;
constexpr int kThreads = kProducers + kEpi + 96;
constexpr int kMmaWarp = (kProducers + kEpi) / 32;
constexpr int kLoadWarp = kMmaWarp + 1;
constexpr int kCodeWarp = kMmaWarp + 2;
constexpr int kABytes = 128 * kBK * 2;   // 16 KB
constexpr int kBBytes = kNT * kBK * 2;   // 24 KB
constexpr int kBarriers = 2 * kAStages + 2 * kBStages + 2 * kGStages + 2 + 2 + 1;
constexpr size_t kSmemBytes = size_t(kAStages) * kABytes + size_t(kBStages) * kBBytes +
                              size_t(kGStages) * (kGCodeBytes + kGScaleBytes) + kBarriers * 8 + 8 + 2 * kNT * 8 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
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
// One arrival that also expects `bytes` of asynchronous copies on the barrier.
__device__ __forceinline__ void expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
// Box of the 2-D tensor behind `tm` (64 columns x kNT rows from (col, row),
// 128-byte swizzle, rows past the tensor read as zeros) -> dst; completion
// counted on b.
__device__ __forceinline__ void tile_load(void* dst, const CUtensorMap* tm, int col, int row, uint64_t* b) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          su32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(col), "r"(row), "r"(su32(b))
      : "memory");
}
// Box of the 3-D tensor behind `tm` at (x, y, z) -> dst; completion counted on b.
__device__ __forceinline__ void tile_load3(void* dst, const CUtensorMap* tm, int x, int y, int z, uint64_t* b) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
          "r"(su32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(su32(b))
      : "memory");
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
__device__ __forceinline__ void cp8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(su32(dst)), "l"(src));
}
__device__ __forceinline__ void cp4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(su32(dst)), "l"(src));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kEpi) : "memory"); }

// Raw-code tensor maps of the expert GEMMs: [cache slots, staging slots, shared
// expert][weight matrix of the tile: gate, up (gate/up GEMM) or down].
struct CodeMaps {
  CUtensorMap m[3][2];
};

struct Args {
  CodeMaps cmaps;            // expert GEMMs: raw codes, one 3-D map per arena and matrix
  const int32_t* num_groups;
  const int32_t* grp_off;
  const uint8_t* const* grp_blob;
  const int32_t* ent_tok;
  const int32_t* ent_pos;
  const int32_t* tile_off;
  const int32_t* tile_grp;
  const int32_t* grange;     // [2] groups g0 .. g1-1 of this launch, or null for all
  int with_shared;           // this launch also runs the shared expert's tiles
  const int32_t* grp_src;    // MOE_SRC_RESIDENT (cache slot) or MOE_SRC_STAGED (staging slot)
  const int32_t* grp_slot;   // [G+1] N tiles before each group
  float* h;                  // gate/up output h (fp32) [maxTk + maxT, Imax]
  float* hmax;               // down: max|h| per row [maxTk + maxT]
  const float* xinv;         // gate/up: inverse power of two of each B row [maxTk + maxT]
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
  int g;  // routed: the group; -1 otherwise
};

// Work list of one GEMM: (routed N tile, M tile) pairs in group order (M tile
// fastest, so CTAs running at the same time share the token tile in L2), then
// the shared expert's tiles; for the router, (token tile, row tile) pairs.
struct Sched {
  int t0, routed_tiles, mt_r, mt_s, n_items;  // t0: the first N tile of the group range
};

template <int MODE>
__device__ __forceinline__ Sched make_sched(const Args& a) {
  Sched s;
  const int ntok = (a.T + kNT - 1) / kNT;
  if (MODE == kRouter) {
    s.t0 = 0;
    s.routed_tiles = 0;
    s.mt_r = (a.E + (a.w_gate ? 1 : 0) + 127) / 128;
    s.mt_s = 0;
    s.n_items = ntok * s.mt_r;
    return s;
  }
  // the groups [g0, g1) of this launch: all of them, or one unit of a streamed call
  const int g0 = a.grange ? a.grange[0] : 0, g1 = a.grange ? a.grange[1] : *a.num_groups;
  s.t0 = a.tile_off[g0];
  s.routed_tiles = a.tile_off[g1] - s.t0;
  s.mt_r = MODE == kGateUp ? (2 * a.I) / 128 : a.H / 128;
  s.mt_s = a.shared_blob && a.with_shared ? (MODE == kGateUp ? (2 * a.I_s) / 128 : a.H / 128) : 0;
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
    x.g = -1;
  } else if (it < sc.routed_tiles * sc.mt_r) {
    const int tl = it / sc.mt_r;
    x.mt = it - tl * sc.mt_r;
    const int ti = sc.t0 + tl;
    const int lo = a.tile_grp[ti];
    x.g = lo;
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
    x.g = -1;
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

// First B row of a token tile; the tile's rows follow it.  Router: x [T, H];
// gate/up: xg [maxT*k + maxT, H] and down: h16 [maxT*k + maxT, Imax], both
// routed entries in group order, then the shared expert's rows in token order.
template <int MODE>
__device__ __forceinline__ int b_row0(const Args& a, const Item& x) {
  const int ent = x.nt * kNT;
  if (MODE == kRouter) return ent;
  return x.shared ? a.maxTk + ent : x.e0 + ent;
}

// Half of one weight row chunk: 16 code bytes (32 columns, low nibble first;
// scale blocks 2*half and 2*half+1 of the row's four E4M3 scales sc4) ->
// code x scale as f16 (exact) in the row's swizzled 16-byte chunks 4*half ..
// 4*half+3.
__device__ __forceinline__ void dequant_half(uint4 codes, uint32_t sc4, int half, uint8_t* at, int row) {
  const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
  for (int bl = 0; bl < 2; ++bl) {
    const int blk = 2 * half + bl;
    const uint32_t sb = (sc4 >> (8 * blk)) & 0xffu;
    const uint32_t sp = e4m3x2_to_f16x2(sb | (sb << 8));  // the scale in both halves, f16 (exact)
    uint32_t hv[8];
#pragma unroll
    for (int w2 = 0; w2 < 2; ++w2) {
      uint32_t o[4];
      asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
          "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
          "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
          : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
          : "r"(cw[2 * bl + w2]));
#pragma unroll
      for (int b = 0; b < 4; ++b) asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(hv[4 * w2 + b]) : "r"(o[b]), "r"(sp));
    }
    *reinterpret_cast<uint4*>(at + sw128(row, 2 * blk)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
    *reinterpret_cast<uint4*>(at + sw128(row, 2 * blk + 1)) = make_uint4(hv[4], hv[5], hv[6], hv[7]);
  }
}

// Non-blocking look at a phase; true once the phase with parity `par` completed.
__device__ __forceinline__ bool bar_test(uint64_t* b, uint32_t par) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(su32(b)), "r"(par)
      : "memory");
  return ok != 0;
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) k_gemm(const __grid_constant__ Args a,
                                                       const __grid_constant__ CUtensorMap tm_r,
                                                       const __grid_constant__ CUtensorMap tm_s) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the 128-byte swizzle pattern is a function of the shared address: atoms start on 1 KB
  uint8_t* smem = smem_raw + ((1024u - (su32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem;                                        // [kAStages][16 KB]
  uint8_t* sB = sA + kAStages * kABytes;                     // [kBStages][32 KB]
  uint8_t* sG = sB + kBStages * kBBytes;                      // [kGStages][128][128]
  uint8_t* sGS = sG + kGStages * kGCodeBytes;                // [kGStages][128][16]
  uint64_t* full = reinterpret_cast<uint64_t*>(sGS + kGStages * kGScaleBytes);
  uint64_t* empty = full + kAStages;      // [kAStages]
  uint64_t* full_b = empty + kAStages;    // [kBStages]
  uint64_t* empty_b = full_b + kBStages;  // [kBStages]
  uint64_t* gfull = empty_b + kBStages;   // [kGStages]
  uint64_t* gempty = gfull + kGStages;    // [kGStages]
  uint64_t* acc_full = gempty + kGStages; // [2]
  uint64_t* acc_empty = acc_full + 2;     // [2]
  uint64_t* drain = acc_empty + 2;
  uint32_t* taddr_s = reinterpret_cast<uint32_t*>(drain + 1);
  int32_t* s_tok = reinterpret_cast<int32_t*>(drain + 2);  // [2][kNT] down: token of each column
  float* s_w = reinterpret_cast<float*>(s_tok + 2 * kNT);  // [2][kNT] down: its weight; gate/up: 2^-p
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const Sched sc = make_sched<MODE>(a);

  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(taddr_s)),
                 "r"(2 * kAccCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int s = 0; s < kAStages; ++s) {
      bar_init(&full[s], 8);  // one arrival per warp of the producer group writing it
      bar_init(&empty[s], 1);
    }
    for (int s = 0; s < kBStages; ++s) {
      bar_init(&full_b[s], 1);
      bar_init(&empty_b[s], 1);
    }
    for (int g = 0; g < kGStages; ++g) {
      bar_init(&gfull[g], 33);               // the code loader: expected bytes + each lane's scale copies
      bar_init(&gempty[g], kProducers / 32);  // one arrival per producer warp
    }
    for (int b = 0; b < 2; ++b) {
      bar_init(&acc_full[b], 1);
      bar_init(&acc_empty[b], kEpi / 32);  // one arrival per epilogue warp
    }
    bar_init(drain, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  const uint32_t taddr = *taddr_s;
  bool failed = false;

  if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int q = 0, done = 0;
      uint32_t ready = 0;  // bits: the next pair's A and B stages (1, 2: first chunk; 4, 8: second) seen full
      for (int it = blockIdx.x; it < sc.n_items && !failed; it += gridDim.x, ++done) {
        Item x;
        item_of<MODE>(a, sc, it, x);
        const int npad = (x.n + 15) & ~15;
        const int buf = done & 1;
        // kind::f16: D f32, A and B both bf16 (router) or both f16 (gate/up,
        // down), both K-major, N = npad, M = 128
        const uint32_t ab = MODE == kRouter ? 1u : 0u;
        const uint32_t idesc = (1u << 4) | (ab << 7) | (ab << 10) | (uint32_t(npad >> 3) << 17) |
                               (uint32_t(128 >> 4) << 24);
        if (done >= 2 && !bar_wait(&acc_empty[buf], ((done >> 1) - 1) & 1)) {
          failed = true;
          break;
        }
        const uint32_t dt = taddr + uint32_t(buf * kAccCols);
        // two chunks per step: one block takes a look at the next two chunks'
        // barriers, issues the eight MMAs of these two, commits their stages
        // free, and only then reads the looks' results, so the barrier
        // round trips pass while the MMAs are issued
        for (int kc = 0; kc < x.KC; kc += 2, q += 2) {
          const bool two = kc + 1 < x.KC;  // an odd last chunk goes alone (its partner slot repeats it)
          const int q1 = two ? q + 1 : q;
          const int s0 = q % kAStages, b0 = q % kBStages, s1 = q1 % kAStages, b1 = q1 % kBStages;
          if ((!(ready & 1) && !bar_wait(&full[s0], (q / kAStages) & 1)) ||
              (!(ready & 2) && !bar_wait(&full_b[b0], (q / kBStages) & 1)) ||
              (!(ready & 4) && !bar_wait(&full[s1], (q1 / kAStages) & 1)) ||
              (!(ready & 8) && !bar_wait(&full_b[b1], (q1 / kBStages) & 1))) {
            failed = true;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;");
          const uint64_t da0 = kmajor_desc(sA + s0 * kABytes), db0 = kmajor_desc(sB + b0 * kBBytes);
          const uint64_t da1 = kmajor_desc(sA + s1 * kABytes), db1 = kmajor_desc(sB + b1 * kBBytes);
          // the pair after this one, in the global chunk order
          const int n0 = q + (two ? 2 : 1), n1 = n0 + 1;
          const uint32_t acc0 = kc > 0 ? 1u : 0u;
          const uint32_t two_u = two ? 1u : 0u;
          uint32_t r0, r1, r2, r3;
          asm volatile(
              "{\n\t.reg .pred t0, t1, t2, t3, p0, p1, pt;\n\t"
              "mbarrier.test_wait.parity.shared::cta.b64 t0, [%6], %7;\n\t"
              "mbarrier.test_wait.parity.shared::cta.b64 t1, [%8], %9;\n\t"
              "mbarrier.test_wait.parity.shared::cta.b64 t2, [%10], %11;\n\t"
              "mbarrier.test_wait.parity.shared::cta.b64 t3, [%12], %13;\n\t"
              "setp.ne.u32 p0, %14, 0;\n\t"
              "setp.eq.u32 p1, %14, %14;\n\t"
              "setp.ne.u32 pt, %15, 0;\n\t"
              "tcgen05.mma.cta_group::1.kind::f16 [%4], %16, %17, %5, p0;\n\t"
              "tcgen05.mma.cta_group::1.kind::f16 [%4], %18, %19, %5, p1;\n\t"
              "tcgen05.mma.cta_group::1.kind::f16 [%4], %20, %21, %5, p1;\n\t"
              "tcgen05.mma.cta_group::1.kind::f16 [%4], %22, %23, %5, p1;\n\t"
              "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%24];\n\t"
              "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%25];\n\t"
              "@pt tcgen05.mma.cta_group::1.kind::f16 [%4], %26, %27, %5, p1;\n\t"
              "@pt tcgen05.mma.cta_group::1.kind::f16 [%4], %28, %29, %5, p1;\n\t"
              "@pt tcgen05.mma.cta_group::1.kind::f16 [%4], %30, %31, %5, p1;\n\t"
              "@pt tcgen05.mma.cta_group::1.kind::f16 [%4], %32, %33, %5, p1;\n\t"
              "@pt tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%34];\n\t"
              "@pt tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%35];\n\t"
              "selp.u32 %0, 1, 0, t0;\n\t"
              "selp.u32 %1, 2, 0, t1;\n\t"
              "selp.u32 %2, 4, 0, t2;\n\t"
              "selp.u32 %3, 8, 0, t3;\n\t}"
              : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
              : "r"(dt), "r"(idesc), "r"(su32(&full[n0 % kAStages])), "r"(uint32_t((n0 / kAStages) & 1)),
                "r"(su32(&full_b[n0 % kBStages])), "r"(uint32_t((n0 / kBStages) & 1)),
                "r"(su32(&full[n1 % kAStages])), "r"(uint32_t((n1 / kAStages) & 1)),
                "r"(su32(&full_b[n1 % kBStages])), "r"(uint32_t((n1 / kBStages) & 1)), "r"(acc0), "r"(two_u),
                "l"(da0), "l"(db0), "l"(da0 + 2), "l"(db0 + 2), "l"(da0 + 4), "l"(db0 + 4), "l"(da0 + 6), "l"(db0 + 6),
                "r"(su32(&empty[s0])), "r"(su32(&empty_b[b0])), "l"(da1), "l"(db1), "l"(da1 + 2), "l"(db1 + 2),
                "l"(da1 + 4), "l"(db1 + 4), "l"(da1 + 6), "l"(db1 + 6), "r"(su32(&empty[s1])), "r"(su32(&empty_b[b1]))
              : "memory");
          ready = r0 | r1 | r2 | r3;
          if (!two) --q;  // the loop adds two; a lone last chunk counts one
        }
        if (!failed) commit_to(&acc_full[buf]);
      }
      // every MMA issued has completed before the accumulators are freed
      commit_to(drain);
      if (!bar_wait(drain, 0)) failed = true;
      if (failed) set_error(a.err, MOE_ETIMEOUT);
    }
  } else if (warp < kProducers / 32) {
    // ------------------------------------------------------------ producers
    const int pg = tid >> 8;                                // producer group
    const int prow = (tid & 255) >> 1, half = tid & 1;      // this thread's weight row and half of it
    // the chunks of this CTA's items, in order: the next one to copy
    int iss_it = blockIdx.x, iss_kc = 0;
    Item ix;
    bool iss_ok = iss_it < sc.n_items;
    const uint16_t* arow = nullptr;  // router: this thread's weight row
    auto load_item = [&]() {
      item_of<MODE>(a, sc, iss_it, ix);
      if (MODE == kRouter) {
        const int r = ix.mt * 128 + prow;
        arow = r < a.E ? a.w_router + size_t(r) * a.H : (r == a.E ? a.w_gate : nullptr);
      }
    };
    if (iss_ok) load_item();

    if (MODE == kRouter) {
      // Router rows are bf16 already: the first producer group copies them
      // straight into the A stage, kAStages - 1 chunks ahead (into the stage
      // of chunk q - 1, whose MMAs have run while chunk q was landing).
      if (pg != 0) iss_ok = false;
      int iss_q = 0;
      auto issue = [&]() {
        if (iss_ok) {
          const int s = iss_q % kAStages;
          if (!failed && iss_q >= kAStages && !bar_wait(&empty[s], ((iss_q / kAStages) - 1) & 1)) failed = true;
          failed = __any_sync(0xffffffffu, failed);  // warp-uniform
          if (!failed && arow) {
            uint8_t* at = sA + s * kABytes;
#pragma unroll
            for (int c = 4 * half; c < 4 * half + 4; ++c) cp16(at + sw128(prow, c), arow + iss_kc * kBK + c * 8);
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
      for (int p = 0; p < kAStages - 1; ++p) issue();
      int q = 0;
      for (int it = blockIdx.x; it < sc.n_items && pg == 0; it += gridDim.x) {
        Item x;
        item_of<MODE>(a, sc, it, x);
        for (int kc = 0; kc < x.KC; ++kc, ++q) {
          cp_wait<kAStages - 2>();  // chunk q has landed (q+1 .. q+kAStages-2 may be in flight)
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) bar_arrive(&full[q % kAStages]);
          issue();
        }
      }
      cp_wait_all();
    } else {
      // Expert weights arrive in code groups of kGChunks chunks (one 128-byte
      // line of each of the tile's 128 weight rows, landed by the code loader
      // in rows of the box order: for gate/up the 64 gate rows, then the 64
      // up rows).  Producer group pg dequantises chunks 2pg and 2pg+1 of each
      // code group into their A stages (each free once the MMAs of chunk
      // c - kAStages completed): the two groups work on neighbouring chunks
      // at the same time, and a group's fixed costs per step are shared by
      // two chunks.
      // the ring row of this thread's tile row (its 128-byte swizzle: grow & 7)
      const int grow = MODE == kGateUp ? (((prow & 31) >= 16) ? 64 : 0) + (prow >> 5) * 16 + (prow & 15) : prow;
      int c = 0, g = 0;  // first chunk of the code group; code groups consumed
      for (int it = blockIdx.x; it < sc.n_items; it += gridDim.x) {
        Item x;
        item_of<MODE>(a, sc, it, x);
        for (int c_in = 0; c_in < x.KC; c_in += kGChunks, ++g) {
          const int nch = min(kGChunks, x.KC - c_in);
          const int gs = g % kGStages;
          if (!failed && !bar_wait(&gfull[gs], (g / kGStages) & 1)) failed = true;
          // this group's chunk pairs of the code group: chunks kk, kk + 1 for
          // kk = 2 pg, 2 pg + 2 kPGroups, ...
          for (int kk = 2 * pg; kk < nch; kk += 2 * kPGroups) {
            const int mine = min(2, nch - kk);  // chunks it dequantises: 1 or 2 (warp-uniform)
            const int c0 = c + kk;
            const bool two = mine == 2;
            const int s0 = c0 % kAStages, s1 = (c0 + 1) % kAStages;
            // A stages free: both looks issued before either result is needed
            if (!failed) {
              const bool w0 = c0 >= kAStages, w1 = two && c0 + 1 >= kAStages;
              const uint32_t p0 = ((c0 / kAStages) - 1) & 1, p1 = (((c0 + 1) / kAStages) - 1) & 1;
              const bool f0 = !w0 || bar_test(&empty[s0], p0);
              const bool f1 = !w1 || bar_test(&empty[s1], p1);
              if ((!f0 && !bar_wait(&empty[s0], p0)) || (!f1 && !bar_wait(&empty[s1], p1))) failed = true;
            }
            failed = __any_sync(0xffffffffu, failed);  // warp-uniform
            if (!failed && x.blob) {
              const uint8_t* gc = sG + gs * kGCodeBytes + grow * 128;
              const uint8_t* gsc = sGS + gs * kGScaleBytes + grow * 16;
              const int j0 = 2 * kk + half, j1 = 2 * (kk + 1) + half;  // this thread's 16-byte pieces
              const uint4 cw0 = *reinterpret_cast<const uint4*>(gc + ((j0 ^ (grow & 7)) << 4));
              const uint32_t sc0 = *reinterpret_cast<const uint32_t*>(gsc + kk * 4);
              uint4 cw1 = make_uint4(0u, 0u, 0u, 0u);
              uint32_t sc1 = 0u;
              if (two) {
                cw1 = *reinterpret_cast<const uint4*>(gc + ((j1 ^ (grow & 7)) << 4));
                sc1 = *reinterpret_cast<const uint32_t*>(gsc + (kk + 1) * 4);
              }
              dequant_half(cw0, sc0, half, sA + s0 * kABytes, prow);
              if (two) dequant_half(cw1, sc1, half, sA + s1 * kABytes, prow);
            }
            // every thread's shared-memory writes are made visible to the
            // tensor core (async proxy) before one lane of the synchronised
            // warp arrives for each chunk
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
              bar_arrive(&full[s0]);
              if (two) bar_arrive(&full[s1]);
            }
          }
          __syncwarp();
          if (lane == 0) bar_arrive(&gempty[gs]);  // the warp is done with the code group
          c += nch;
        }
      }
    }
    if (failed) set_error(a.err, MOE_ETIMEOUT);
  } else if (warp == kLoadWarp) {
    // ------------------------------------------------------------ B loader
    // Token tiles are contiguous rows: one box per chunk into the B ring
    // (columns past n hold other rows or zeros and are never read back), and
    // an L2 prefetch of the box kBPrefetch chunks further on, so that the load
    // into a freshly freed stage finds its rows in L2.
    int q = 0;
    int pf_it = blockIdx.x, pf_kc = 0;  // the chunk to prefetch next
    Item px;
    bool pf_ok = pf_it < sc.n_items;
    if (pf_ok) item_of<MODE>(a, sc, pf_it, px);
    auto prefetch_next = [&]() {
      if (!pf_ok) return;
      if (lane == 0) {
        const CUtensorMap* tm = px.shared ? &tm_s : &tm_r;
        asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                         reinterpret_cast<uint64_t>(tm)),
                     "r"(pf_kc * kBK), "r"(b_row0<MODE>(a, px))
                     : "memory");
      }
      if (++pf_kc == px.KC) {
        pf_kc = 0;
        pf_it += gridDim.x;
        pf_ok = pf_it < sc.n_items;
        if (pf_ok) item_of<MODE>(a, sc, pf_it, px);
      }
    };
    for (int p = 0; p < kBStages + kBPrefetch; ++p) prefetch_next();
    for (int it = blockIdx.x; it < sc.n_items && !failed; it += gridDim.x) {
      Item x;
      item_of<MODE>(a, sc, it, x);
      const CUtensorMap* tm = x.shared ? &tm_s : &tm_r;
      const int row0 = b_row0<MODE>(a, x);
      for (int kc = 0; kc < x.KC; ++kc, ++q) {
        const int s = q % kBStages;
        if (q >= kBStages && !bar_wait(&empty_b[s], ((q / kBStages) - 1) & 1)) failed = true;
        failed = __any_sync(0xffffffffu, failed);
        if (failed) break;
        if (lane == 0) {
          expect_tx(&full_b[s], kBBytes);
          tile_load(sB + s * kBBytes, tm, kc * kBK, row0, &full_b[s]);
        }
        __syncwarp();
        prefetch_next();
      }
    }
    // the copies of the last stages have landed before the CTA can leave
    for (int qq = q > kBStages ? q - kBStages : 0; qq < q; ++qq)
      if (!bar_wait(&full_b[qq % kBStages], (qq / kBStages) & 1)) failed = true;
    if (failed && lane == 0) set_error(a.err, MOE_ETIMEOUT);
  } else if (warp == kCodeWarp) {
    // ------------------------------------------------------------ code loader
    // Per code group: one TMA box (128 bytes x 64 or 128 rows) of raw codes per
    // weight matrix of the tile from the 3-D map of the expert's arena (cache
    // slots, staging slots or the shared expert), and the rows' scale bytes
    // with cp.async, four rows per lane.
    if (MODE != kRouter) {
      int g = 0;
      for (int it = blockIdx.x; it < sc.n_items && !failed; it += gridDim.x) {
        Item x;
        item_of<MODE>(a, sc, it, x);
        int arena = 2, slot = 0;  // shared expert
        if (!x.shared) {
          arena = a.grp_src[x.g] == MOE_SRC_STAGED ? 1 : 0;
          slot = max(a.grp_slot[x.g], 0);
        }
        const DevBlobLayout& lay = x.shared ? a.lay_s : a.lay_r;
        const uint8_t* srow[4];  // scale rows lane + 32u, in box order
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int r = lane + 32 * u;
          int mat, wrow;
          if (MODE == kGateUp) {
            mat = r >= 64 ? 1 : 0;
            wrow = x.mt * 64 + (r & 63);
          } else {
            mat = 2;
            wrow = x.mt * 128 + r;
          }
          srow[u] = x.blob ? x.blob + lay.scale_off[mat] + size_t(wrow) * (x.C / 16) : nullptr;
        }
        const int rowbytes = x.C / 2;
        for (int gi = 0; gi * 128 < rowbytes; ++gi, ++g) {
          const int gs = g % kGStages;
          if (g >= kGStages && !bar_wait(&gempty[gs], ((g / kGStages) - 1) & 1)) failed = true;
          failed = __any_sync(0xffffffffu, failed);
          if (failed) break;
          if (lane == 0) {
            if (x.blob) {
              expect_tx(&gfull[gs], kGCodeBytes);
              uint8_t* dst = sG + gs * kGCodeBytes;
              if (MODE == kGateUp) {
                tile_load3(dst, &a.cmaps.m[arena][0], gi * 128, x.mt * 64, slot, &gfull[gs]);
                tile_load3(dst + 64 * 128, &a.cmaps.m[arena][1], gi * 128, x.mt * 64, slot, &gfull[gs]);
              } else {
                tile_load3(dst, &a.cmaps.m[arena][0], gi * 128, x.mt * 128, slot, &gfull[gs]);
              }
            } else {
              // a missing or skipped expert: nothing to copy (its arena's map may
              // not exist), the stage completes on the arrivals alone
              bar_arrive(&gfull[gs]);
            }
          }
          const int gbytes = min(128, rowbytes - gi * 128);  // 32 per chunk
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (!srow[u]) continue;
            uint8_t* d = sGS + gs * kGScaleBytes + (lane + 32 * u) * 16;
            const uint8_t* sp = srow[u] + gi * 16;
            if (gbytes == 128) cp16(d, sp);
            else if (gbytes == 64) cp8(d, sp);
            else cp4(d, sp);
          }
          asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(su32(&gfull[gs])) : "memory");
        }
      }
      // every copy has landed before the CTA can leave
      cp_wait_all();
      for (int gg = g > kGStages ? g - kGStages : 0; gg < g; ++gg)
        if (!bar_wait(&gfull[gg % kGStages], (gg / kGStages) & 1)) failed = true;
      if (failed && lane == 0) set_error(a.err, MOE_ETIMEOUT);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int et = tid - kProducers, qw = warp & 3;
    // down: each thread's columns et and et + kEpi of an item -- the token, the
    // routing weight (or the shared gate logit) and max|h| of the row -- are
    // loaded one item ahead, so their dependent loads run under the previous
    // item's atomic adds
    constexpr int kCols = (kNT + kEpi - 1) / kEpi;
    int c_tok[kCols];
    float c_w[kCols], c_hm[kCols];
    auto fetch_cols = [&](const Item& xi) {
#pragma unroll
      for (int q = 0; q < kCols; ++q) {
        const int j = et + q * kEpi;
        c_tok[q] = 0;
        c_w[q] = 0.f;
        c_hm[q] = 0.f;
        if (j < xi.n) {
          const int ent = xi.nt * kNT + j;
          if (xi.shared) {
            c_tok[q] = ent;
            c_w[q] = a.gate_logit[ent];
            c_hm[q] = a.hmax[a.maxTk + ent];
          } else {
            const int pos = a.ent_pos[xi.e0 + ent];
            c_tok[q] = pos;  // the token is pos / k
            c_w[q] = a.topk_w[pos];
            c_hm[q] = a.hmax[xi.e0 + ent];
          }
        }
      }
    };
    if (MODE == kDown && blockIdx.x < sc.n_items) {
      Item x0;
      item_of<MODE>(a, sc, blockIdx.x, x0);
      fetch_cols(x0);
    }
    int done = 0;
    for (int it = blockIdx.x; it < sc.n_items; it += gridDim.x, ++done) {
      Item x;
      item_of<MODE>(a, sc, it, x);
      const int buf = done & 1;
      if (MODE == kDown) {
#pragma unroll
        for (int q = 0; q < kCols; ++q) {
          const int j = et + q * kEpi;
          if (j < x.n) {
            // B row = h x 2^p (the power of two the conversion to f16 chose)
            s_tok[buf * kNT + j] = x.shared ? c_tok[q] : c_tok[q] / a.k;
            s_w[buf * kNT + j] = (x.shared ? sigmoid_f32(c_w[q]) : c_w[q]) / pow2_scale_for(c_hm[q]);
          }
        }
        epi_sync();
        if (it + int(gridDim.x) < sc.n_items) {
          Item xn;
          item_of<MODE>(a, sc, it + gridDim.x, xn);
          fetch_cols(xn);
        }
      } else if (MODE == kGateUp) {
        // B row = x_t x 2^p: the inverse power of two of each column
        for (int j = et; j < x.n; j += kEpi) {
          const int ent = x.nt * kNT + j;
          s_w[buf * kNT + j] = a.xinv[x.shared ? a.maxTk + ent : x.e0 + ent];
        }
        epi_sync();
      }
      if (!failed && !bar_wait(&acc_full[buf], (done >> 1) & 1)) failed = true;
      failed = __any_sync(0xffffffffu, failed);
      asm volatile("tcgen05.fence::after_thread_sync;");
      const float gs0 = x.blob ? reinterpret_cast<const BlobHeader*>(x.blob)->gscale[MODE == kGateUp ? 0 : 2] : 0.f;
      const float gs1 = x.blob ? reinterpret_cast<const BlobHeader*>(x.blob)->gscale[1] : 0.f;
      const int npad = (x.n + 15) & ~15;
      const uint32_t tb = taddr + uint32_t(buf * kAccCols) + (uint32_t(qw * 32) << 16);
      const int row = x.mt * 128 + qw * 32 + lane;  // router / down: output row of this lane
      const float rbias = (MODE == kRouter && a.bias && row < a.E) ? a.bias[row] : 0.f;
      // gate/up: h row of column 0 of this tile and this lane's intermediate
      float* hcol = nullptr;
      if (MODE == kGateUp)
        hcol = a.h + size_t(x.shared ? a.maxTk + x.nt * kNT : x.e0 + x.nt * kNT) * a.Imax + x.mt * 64 + qw * 16 +
               (lane & 15);
      // of every 16 kEpiPerQuad accumulator columns this warp takes 16 (the other
      // warps of its lane quadrant the others); columns past npad are read and
      // ignored: the buffer's 256 columns are all allocated
      const int eh = (warp - kProducers / 32) >> 2;
      for (int c0 = 0; c0 < npad && !failed; c0 += 16 * kEpiPerQuad) {
        const int cb = c0 + 16 * eh;  // this warp's first column
        uint32_t v[16];
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
              "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
            : "r"(tb + uint32_t(cb)));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        if (MODE == kGateUp) {
          // lanes 0-15 hold gate rows, 16-31 the matching up rows: of the 16
          // columns the low lanes finish the first 8, the high lanes the last 8
          const bool hi = lane >= 16;
#pragma unroll
          for (int b = 0; b < 8; ++b) {
            const float mine_lo = __uint_as_float(v[b]), mine_hi = __uint_as_float(v[b + 8]);
            const float recv = __shfl_xor_sync(0xffffffffu, hi ? mine_lo : mine_hi, 16);
            const float g = hi ? recv : mine_lo, u = hi ? mine_hi : recv;
            const int j = cb + b + (hi ? 8 : 0);
            if (j < x.n) {
              const float xi = s_w[buf * kNT + j];
              hcol[size_t(j) * a.Imax] = x.blob ? silu_f32(g * (gs0 * xi)) * (u * (gs1 * xi)) : 0.f;
            }
          }
        } else if (MODE == kDown) {
          // y[token] += w x o_e (fp32 atomic adds in L2: a token's k + 1
          // terms come from different CTAs); a missing expert adds nothing
          if (x.blob) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int j = cb + jj;
              if (j < x.n)
                atomicAdd(a.yacc + size_t(s_tok[buf * kNT + j]) * a.H + row,
                          __uint_as_float(v[jj]) * gs0 * s_w[buf * kNT + j]);
            }
          }
        } else {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int j = cb + jj;
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
      __syncwarp();
      if (lane == 0) bar_arrive(&acc_empty[buf]);
    }
    if (failed) set_error(a.err, MOE_ETIMEOUT);
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.fence::after_thread_sync;");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(2 * kAccCols));
  }
}

// N tiles per group, as an exclusive prefix: tile_off[g] = sum_{g'<g} ceil(n_g'/kNT),
// and the group of every tile: tile_grp[t] = g for tile_off[g] <= t < tile_off[g+1].
__global__ void __launch_bounds__(1024) k_tiles(const int32_t* __restrict__ num_groups, const int32_t* __restrict__ grp_off,
                                                int32_t* __restrict__ tile_off, int32_t* __restrict__ tile_grp) {
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
    if (g < G) {
      tile_off[g] = before + x - v;
      for (int t = 0; t < v; ++t) tile_grp[before + x - v + t] = g;
    }
    carry += ws[(blockDim.x >> 5) - 1];
    __syncthreads();
  }
  if (threadIdx.x == 0) tile_off[G] = carry;
}

// h (fp32) -> f16 times a per-row power of two chosen from max|h_row| over the
// row's I (routed) or I_s (shared) columns; the max goes to hmax for the down
// GEMM's epilogue, which divides the power of two out again.  One warp per row.
__global__ void __launch_bounds__(256) k_h16(const float* __restrict__ h, float* __restrict__ hmax,
                                             __half* __restrict__ h16, const int32_t* __restrict__ grp_off,
                                             const int32_t* __restrict__ num_groups,
                                             const int32_t* __restrict__ grange, int Imax, int I, int I_s,
                                             int maxTk, int T, int has_shared) {
  pdl_trigger();
  pdl_wait();
  // the entries of groups [g0, g1) (all groups, or one unit), then the shared rows
  const int e0 = grange ? grp_off[grange[0]] : 0;
  const int routed = (grange ? grp_off[grange[1]] : grp_off[*num_groups]) - e0;
  const int rows = routed + (has_shared ? T : 0);
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  for (int rr = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); rr < rows; rr += nwarps) {
    const int row = rr < routed ? e0 + rr : maxTk + (rr - routed);
    const int n4 = (rr < routed ? I : I_s) / 4;
    const float4* src = reinterpret_cast<const float4*>(h + size_t(row) * Imax);
    float m = 0.f;
    for (int c4 = lane; c4 < n4; c4 += 32) {
      const float4 f = src[c4];
      m = fmaxf(m, fmaxf(fmaxf(fabsf(f.x), fabsf(f.y)), fmaxf(fabsf(f.z), fabsf(f.w))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) hmax[row] = m;
    const float sc = pow2_scale_for(m);
    for (int c4 = lane; c4 < n4; c4 += 32) {
      const float4 f = src[c4];
      __half2 p0 = __floats2half2_rn(f.x * sc, f.y * sc), p1 = __floats2half2_rn(f.z * sc, f.w * sc);
      uint2 u;
      u.x = *reinterpret_cast<uint32_t*>(&p0);
      u.y = *reinterpret_cast<uint32_t*>(&p1);
      reinterpret_cast<uint2*>(h16 + size_t(row) * Imax)[c4] = u;
    }
  }
}

// B rows of the gate/up GEMM: token rows as f16 times a power of two per token
// (max|x_t| brought into [2^12, 2^13)), in group order for the routed entries
// (row e = x[ent_tok[e]]) and in token order for the shared expert (row
// maxTk + t); xinv gets the inverse power of two of each row.  bf16 values have
// 8 significant bits, so the scaled value is exact in f16 unless it falls below
// the f16 normal range, where the error stays under 2^-25 max|x_t|.  One warp
// per row, the row held in registers: PER 16-byte pieces per lane (H <= 256 PER).
template <int PER>
__global__ void __launch_bounds__(256) k_x16_grouped(const uint16_t* __restrict__ x, __half* __restrict__ xg,
                                                     float* __restrict__ xinv, const int32_t* __restrict__ ent_tok,
                                                     const int32_t* __restrict__ grp_off,
                                                     const int32_t* __restrict__ num_groups, int H, int maxTk, int T,
                                                     int has_shared) {
  pdl_trigger();
  pdl_wait();
  const int routed = grp_off[*num_groups];
  const int rows = routed + (has_shared ? T : 0);
  const int lane = threadIdx.x & 31, n16 = H / 8;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  for (int rr = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); rr < rows; rr += nwarps) {
    const int tok = rr < routed ? ent_tok[rr] : rr - routed;
    const int orow = rr < routed ? rr : maxTk + (rr - routed);
    const uint4* src = reinterpret_cast<const uint4*>(x + size_t(tok) * H);
    uint4 v[PER];
    float m = 0.f;
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int c = u * 32 + lane;
      v[u] = c < n16 ? src[c] : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[q] << 16)), fabsf(__uint_as_float(w[q] & 0xffff0000u))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float sc = pow2_scale_for(m);
    if (lane == 0) xinv[orow] = 1.0f / sc;
    uint4* dst = reinterpret_cast<uint4*>(xg + size_t(orow) * H);
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int c = u * 32 + lane;
      if (c < n16) {
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const __half2 hh = __floats2half2_rn(__uint_as_float(w[q] << 16) * sc, __uint_as_float(w[q] & 0xffff0000u) * sc);
          o[q] = *reinterpret_cast<const uint32_t*>(&hh);
        }
        dst[c] = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
}

// One unit of a streamed prefill call: the groups of experts u*U .. u*U+U-1
// (groups are in ascending expert id, so they are a contiguous range) take
// their weights from staging slots base + (e - u*U); grange gets the range.
__global__ void __launch_bounds__(256) k_unit_bind(int u, int U, int base, const int32_t* __restrict__ num_groups,
                                                   const int32_t* __restrict__ grp_expert, int32_t* __restrict__ grp_src,
                                                   int32_t* __restrict__ grp_slot, const uint8_t** __restrict__ grp_blob,
                                                   const uint8_t* staging, size_t blob_bytes, int32_t* __restrict__ grange) {
  pdl_trigger();
  pdl_wait();
  const int G = *num_groups;
  const int lo_e = u * U, hi_e = lo_e + U;
  // first group with expert >= lo_e, and >= hi_e (binary searches)
  auto lower = [&](int v) {
    int lo = 0, hi = G;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (grp_expert[mid] < v) lo = mid + 1;
      else hi = mid;
    }
    return lo;
  };
  const int g0 = lower(lo_e), g1 = lower(hi_e);
  for (int g = g0 + int(threadIdx.x); g < g1; g += blockDim.x) {
    const int slot = base + (grp_expert[g] - lo_e);
    grp_src[g] = MOE_SRC_STAGED;
    grp_slot[g] = slot;
    grp_blob[g] = staging + size_t(slot) * blob_bytes;
  }
  if (threadIdx.x == 0) {
    grange[0] = g0;
    grange[1] = g1;
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

// Tensor map of a row-major [rows, cols] matrix of 16-bit values for the B
// loader: boxes of 64 columns x kNT rows, 128-byte swizzle.  Needs a 16-byte
// aligned base and cols % 8 == 0.
static int encode_rows(CUtensorMap* tm, const void* base, int cols, int rows) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }();
  if (!encode || (reinterpret_cast<uintptr_t>(base) & 15) || cols % 8 || rows <= 0) return MOE_ECUDA;
  const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(cols) * 2};
  const cuuint32_t box[2] = {cuuint32_t(prefill::kBK), cuuint32_t(prefill::kNT)};
  const cuuint32_t es[2] = {1, 1};
  if (encode(tm, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return MOE_ECUDA;
  return MOE_OK;
}

// B of routed tiles from [r_rows, cols] at r_base, of shared-expert tiles from
// [s_rows, cols] at s_base.
// Map of the raw codes of one weight matrix in n blobs spaced `stride` bytes
// apart (a cache arena, or one blob): [n][rows][rowbytes] bytes, boxes of
// 128 bytes (four chunks of a row) x boxrows rows, 128-byte swizzle.
static int encode_codes(CUtensorMap* tm, const uint8_t* base, int rowbytes, int rows, int n, size_t stride,
                        int boxrows) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return MOE_ECUDA;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  if ((reinterpret_cast<uintptr_t>(base) & 15) || rowbytes % 16 || stride % 16 || n <= 0 || rows <= 0) return MOE_ECUDA;
  const cuuint64_t dims[3] = {cuuint64_t(rowbytes), cuuint64_t(rows), cuuint64_t(n)};
  const cuuint64_t strides[2] = {cuuint64_t(rowbytes), cuuint64_t(stride)};
  const cuuint32_t box[3] = {128, cuuint32_t(boxrows), 1};
  const cuuint32_t es[3] = {1, 1, 1};
  if (encode(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return MOE_ECUDA;
  return MOE_OK;
}

// The raw-code maps of a GEMM over the cache arenas and the shared expert.
static int code_maps(prefill::CodeMaps* cm, bool gateup, const moe_layer_desc* d, const moe_cache* c) {
  using namespace prefill;
  std::memset(cm, 0, sizeof(*cm));
  const moe_layer_shape& sh = d->s;
  const int nmat = gateup ? 2 : 1;
  for (int i = 0; i < nmat; ++i) {
    const int mat = gateup ? i : 2;
    const DevBlobLayout lr = dev_layout(sh.H, sh.I);
    const int rowbytes = (gateup ? sh.H : sh.I) / 2, rows = gateup ? sh.I : sh.H, boxrows = gateup ? 64 : 128;
    int rc;
    if (c->nslots > 0 &&
        (rc = encode_codes(&cm->m[0][i], c->slots + lr.code_off[mat], rowbytes, rows, c->nslots, c->blob_bytes, boxrows)))
      return rc;
    if (c->nstaging > 0 && (rc = encode_codes(&cm->m[1][i], c->staging + lr.code_off[mat], rowbytes, rows,
                                              c->nstaging, c->blob_bytes, boxrows)))
      return rc;
    if (sh.I_shared > 0 && d->shared_blob) {
      const DevBlobLayout ls = dev_layout(sh.H, sh.I_shared);
      const int srb = (gateup ? sh.H : sh.I_shared) / 2, srows = gateup ? sh.I_shared : sh.H;
      if ((rc = encode_codes(&cm->m[2][i], static_cast<const uint8_t*>(d->shared_blob) + ls.code_off[mat], srb, srows,
                             1, (size_t(srb) * srows + 15) & ~size_t(15), boxrows)))
        return rc;
    }
  }
  return MOE_OK;
}

template <int MODE>
static int launch_gemm(const prefill::Args& a, const void* r_base, int r_rows, const void* s_base, int s_rows, int cols,
                       cudaStream_t s) {
  alignas(64) CUtensorMap tm_r, tm_s;
  if (int rc = encode_rows(&tm_r, r_base, cols, r_rows)) return rc;
  if (int rc = encode_rows(&tm_s, s_base, cols, s_rows)) return rc;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(prefill::k_gemm<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(prefill::kSmemBytes)) != cudaSuccess)
      return MOE_ECUDA;
    attr = true;
  }
  if (launch_pdl(prefill::k_gemm<MODE>, dim3(sm_count()), dim3(prefill::kThreads), prefill::kSmemBytes, s, a, tm_r, tm_s) !=
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
  a.tile_grp = ws->tile_grp;
  a.grp_src = ws->grp_src;
  a.grp_slot = ws->grp_slot;
  a.h = ws->h;
  a.hmax = ws->hmax;
  a.xinv = ws->xinv;
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
  a.w_router = d->w_router;
  a.w_gate = d->s.I_shared > 0 ? d->w_shared_gate : nullptr;
  a.bias = d->bias;
  a.logits = ws->logits;
  a.gate_out = ws->gate_logit;
  return launch_gemm<prefill::kRouter>(a, x, T, x, T, d->s.H, s);
}

// The expert part of a prefill call: tiles, gate/up GEMM (h), max|h| per row
// and h -> f16 times a per-row power of two, down GEMM accumulating w*o
// into an fp32 buffer, and the output cast.
// The start of a prefill call's expert part: N tiles per group, the zeroed
// fp32 accumulator, the gate/up B rows in group order.
static int prefill_begin(prefill::Args& a, const moe_layer_desc* d, const uint16_t* x, void* y, int y_is_fp32, int T,
                         moe_ws* ws, cudaStream_t s) {
  using namespace prefill;
  const moe_layer_shape& sh = d->s;
  float* yacc = y_is_fp32 ? static_cast<float*>(y) : ws->yacc;
  a.yacc = yacc;
  {
    ProfScope p(ws, "tiles_zero", s);
    if (launch_pdl(k_tiles, dim3(1), dim3(1024), 0, s, ws->num_groups, ws->grp_off, ws->tile_off, ws->tile_grp) !=
        cudaSuccess)
      return MOE_ECUDA;
    MOE_CUDA_TRY(cudaMemsetAsync(yacc, 0, size_t(T) * sh.H * 4, s));
  }
  {
    ProfScope p(ws, "x16_grouped", s);
    auto kern = sh.H <= 256 ? k_x16_grouped<1> : sh.H <= 512 ? k_x16_grouped<2> : sh.H <= 1024 ? k_x16_grouped<4>
              : sh.H <= 2048 ? k_x16_grouped<8> : k_x16_grouped<16>;
    if (sh.H > 4096) return MOE_EINVAL;
    if (launch_pdl(kern, dim3(sm_count() * 8), dim3(256), 0, s, x, ws->xg, ws->xinv, ws->ent_tok, ws->grp_off,
                   ws->num_groups, sh.H, a.maxTk, T, a.shared_blob ? 1 : 0) != cudaSuccess)
      return MOE_ECUDA;
  }
  return MOE_OK;
}

// gate/up GEMM, h -> f16, down GEMM over the groups in grange (null: all of
// them), with the shared expert's tiles when with_shared.
static int prefill_groups(prefill::Args& a, const moe_layer_desc* d, const moe_cache* c, int T, moe_ws* ws,
                          const int32_t* grange, int with_shared, bool prof, cudaStream_t s) {
  using namespace prefill;
  const moe_layer_shape& sh = d->s;
  a.grange = grange;
  a.with_shared = with_shared;
  int rc;
  {
    ProfScope p(prof ? ws : nullptr, "gateup_gemm", s);
    if ((rc = code_maps(&a.cmaps, true, d, c))) return rc;
    if ((rc = launch_gemm<kGateUp>(a, ws->xg, a.maxTk + ws->maxT, ws->xg, a.maxTk + ws->maxT, sh.H, s))) return rc;
  }
  {
    ProfScope p(prof ? ws : nullptr, "h16", s);
    if (launch_pdl(k_h16, dim3(sm_count() * 8), dim3(256), 0, s, ws->h, ws->hmax, ws->h16, ws->grp_off,
                   ws->num_groups, grange, a.Imax, a.I, a.I_s, a.maxTk, T, a.shared_blob && with_shared ? 1 : 0) !=
        cudaSuccess)
      return MOE_ECUDA;
  }
  {
    ProfScope p(prof ? ws : nullptr, "down_gemm", s);
    if ((rc = code_maps(&a.cmaps, false, d, c))) return rc;
    if ((rc = launch_gemm<kDown>(a, ws->h16, a.maxTk + ws->maxT, ws->h16, a.maxTk + ws->maxT, a.Imax, s))) return rc;
  }
  return MOE_OK;
}

// y = bf16 of the accumulator (fp32 outputs were accumulated in place).
static int prefill_end(const moe_layer_desc* d, void* y, int y_is_fp32, int T, moe_ws* ws, cudaStream_t s) {
  using namespace prefill;
  if (!y_is_fp32) {
    ProfScope p(ws, "cast", s);
    const size_t n4 = size_t(T) * d->s.H / 4;
    if (launch_pdl(k_cast_bf16, dim3(sm_count() * 8), dim3(256), 0, s, ws->yacc, static_cast<uint16_t*>(y), n4) !=
        cudaSuccess)
      return MOE_ECUDA;
  }
  return MOE_OK;
}

// The expert part of a prefill call: tiles, gate/up GEMM (h), max|h| per row
// and h -> f16 times a per-row power of two, down GEMM accumulating w*o
// into an fp32 buffer, and the output cast.
int launch_prefill_experts(const moe_layer_desc* d, const moe_cache* c, const uint16_t* x, void* y, int y_is_fp32, int T,
                           moe_ws* ws, cudaStream_t s) {
  prefill::Args a = base_args(d, T, ws);
  int rc;
  if ((rc = prefill_begin(a, d, x, y, y_is_fp32, T, ws, s))) return rc;
  if ((rc = prefill_groups(a, d, c, T, ws, nullptr, 1, true, s))) return rc;
  return prefill_end(d, y, y_is_fp32, T, ws, s);
}

// The expert part of a streamed prefill call (Strata expert paths: the copy
// stream fills a staging slot and records `copied`, the compute stream waits
// on it, runs the unit and records `used`, and the copy stream waits on `used`
// before it overwrites the slot).  Units of U consecutive expert ids go from
// the cache's backing pool (one copy of n*blob_bytes per unit) into half u%2 of
// the staging pool; the unit's groups are bound to those slots and only they
// run.  The shared expert runs with the first unit.
int launch_prefill_streamed(const moe_layer_desc* d, moe_cache* c, const uint16_t* x, void* y, int y_is_fp32, int T,
                            int U, int buffers, moe_ws* ws, cudaStream_t s, cudaStream_t cs) {
  using namespace prefill;
  const moe_layer_shape& sh = d->s;
  prefill::Args a = base_args(d, T, ws);
  int rc;
  // the copy stream starts after everything already queued on the compute
  // stream (an earlier call may still read the staging pool)
  MOE_CUDA_TRY(cudaEventRecord(c->ev_ring[4], s));
  MOE_CUDA_TRY(cudaStreamWaitEvent(cs, c->ev_ring[4], 0));
  if ((rc = prefill_begin(a, d, x, y, y_is_fp32, T, ws, s))) return rc;
  const int nunits = (sh.E + U - 1) / U;
  const uint8_t* pool = static_cast<const uint8_t*>(c->backing) + size_t(d->layer) * sh.E * c->blob_bytes;
  for (int u = 0; u < nunits; ++u) {
    // two buffers: unit u + 1 copies into the other half while unit u computes;
    // one buffer: each copy waits for the previous unit's GEMMs
    const int half = buffers == 2 ? (u & 1) : 0, n = sh.E - u * U < U ? sh.E - u * U : U;
    cudaEvent_t copied = c->ev_ring[half], used = c->ev_ring[2 + half];
    if (u >= buffers) MOE_CUDA_TRY(cudaStreamWaitEvent(cs, used, 0));
    MOE_CUDA_TRY(cudaMemcpyAsync(c->staging + size_t(half) * U * c->blob_bytes, pool + size_t(u) * U * c->blob_bytes,
                                 size_t(n) * c->blob_bytes, cudaMemcpyDefault, cs));
    MOE_CUDA_TRY(cudaEventRecord(copied, cs));
    MOE_CUDA_TRY(cudaStreamWaitEvent(s, copied, 0));
    int32_t* grange = ws->grange + 2 * u;
    if (launch_pdl(k_unit_bind, dim3(1), dim3(256), 0, s, u, U, half * U, ws->num_groups, ws->grp_expert, ws->grp_src,
                   ws->grp_slot, ws->grp_blob, static_cast<const uint8_t*>(c->staging), c->blob_bytes, grange) !=
        cudaSuccess)
      return MOE_ECUDA;
    if ((rc = prefill_groups(a, d, c, T, ws, grange, u == 0 ? 1 : 0, false, s))) return rc;
    MOE_CUDA_TRY(cudaEventRecord(used, s));
  }
  // the copy stream's last work is behind the compute stream's last wait
  return prefill_end(d, y, y_is_fp32, T, ws, s);
}

// Several layers of a prefill chunk with each layer's experts streamed whole into
// one half of the staging pool (FreeToken notes, section 3.1: while layer l computes
// with the experts of one buffer, layer l + 1's are copied into the other; section
// 5.3: with the second buffer off, each copy waits for the previous layer).  Per
// layer l, half h = l % buffers: the copy stream waits until the layer that last
// used half h is done (`used`), copies layer l's E blobs from the backing pool in
// one cudaMemcpyAsync and records `copied`; the compute stream adds the previous
// layer's output to the residual stream and normalises it, waits on `copied`,
// runs the layer's prefill with every group bound to staging slot h * E + expert,
// and records `used`.  A final residual add closes the stack.
int launch_prefill_layers_streamed(const moe_layer_desc* d, int L, float* x_res, uint16_t* xn, uint16_t* y, int T,
                                   moe_cache* c, moe_ws* ws, int buffers, float eps, cudaStream_t s,
                                   cudaStream_t cs) {
  using namespace prefill;
  const moe_layer_shape& sh = d[0].s;
  const size_t layer_bytes = size_t(sh.E) * c->blob_bytes;
  int rc;
  MOE_CUDA_TRY(cudaEventRecord(c->ev_ring[4], s));
  MOE_CUDA_TRY(cudaStreamWaitEvent(cs, c->ev_ring[4], 0));
  for (int l = 0; l < L; ++l) {
    const int half = l % buffers;
    cudaEvent_t copied = c->ev_ring[half], used = c->ev_ring[2 + half];
    if (l >= buffers) MOE_CUDA_TRY(cudaStreamWaitEvent(cs, used, 0));
    const uint8_t* pool = static_cast<const uint8_t*>(c->backing) + size_t(d[l].layer) * layer_bytes;
    MOE_CUDA_TRY(cudaMemcpyAsync(c->staging + size_t(half) * layer_bytes, pool, layer_bytes, cudaMemcpyDefault, cs));
    MOE_CUDA_TRY(cudaEventRecord(copied, cs));
    if ((rc = moe_residual_rmsnorm(x_res, l > 0 ? y : nullptr, xn, T, sh.H, eps, reinterpret_cast<moe_stream_t>(s))))
      return rc;
    if ((rc = launch_prefill_router(&d[l], xn, T, ws, s))) return rc;
    if ((rc = launch_topk(ws->logits, T, sh.E, sh.k, ws->topk_ids, ws->topk_w, ws->error, s))) return rc;
    if ((rc = launch_group(ws->topk_ids, T, sh.k, sh.E, d[l].layer, c, ws, s, false))) return rc;
    prefill::Args a = base_args(&d[l], T, ws);
    if ((rc = prefill_begin(a, &d[l], xn, y, 0, T, ws, s))) return rc;
    MOE_CUDA_TRY(cudaStreamWaitEvent(s, copied, 0));
    if (launch_pdl(k_unit_bind, dim3(1), dim3(256), 0, s, 0, sh.E, half * sh.E, ws->num_groups, ws->grp_expert,
                   ws->grp_src, ws->grp_slot, ws->grp_blob, static_cast<const uint8_t*>(c->staging), c->blob_bytes,
                   ws->grange) != cudaSuccess)
      return MOE_ECUDA;
    if ((rc = prefill_groups(a, &d[l], c, T, ws, ws->grange, 1, false, s))) return rc;
    MOE_CUDA_TRY(cudaEventRecord(used, s));
    if ((rc = prefill_end(&d[l], y, 0, T, ws, s))) return rc;
  }
  return moe_residual_rmsnorm(x_res, y, xn, T, sh.H, eps, reinterpret_cast<moe_stream_t>(s));
}

}  // namespace moe
