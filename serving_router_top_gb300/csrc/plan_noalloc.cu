// Swap planning that allocates nothing: cache_plan_swaps_noalloc.
//
// Same computation and kernels as cache_plan_swaps, but on caller-owned heat
// and residency tables and with the planner's scratch in a file-scope device
// array instead of memory allocated at cache creation.  It serves callers
// that cannot allocate device memory at the point where they plan: a serving
// loop that runs under a fixed memory budget handed out by its own
// allocator (a cudaMalloc there would take memory outside the budget or fail
// once the budget is spent), or one that keeps the policy tables in its own
// buffers and has no moe_cache handle to plan through.
//
// The scratch's address is looked up once per device (cudaGetSymbolAddress,
// on the first call made while that device is current).  The lookup may load
// the module, which is not allowed while a stream is being captured, so the
// first call on each device should come before any capture.  The address is
// kept for the life of the process; a device reset (cudaDeviceReset, or any
// teardown of the primary context) leaves it stale, so the library must not be
// called again in that process after one.
#include <mutex>

#include "internal.h"

namespace moe {
namespace {

constexpr int kNaMaxL = 1024;     // layers
constexpr int kNaMaxLE = 32768;   // layers x experts
constexpr int kNaMaxKeys = 16384; // candidate keys: layers x ceil(experts / 2)

// [keys: kNaMaxKeys x u64][candidates per layer: kNaMaxL x i32][cold partner: kNaMaxLE x i32]
// (260 KB).  Nothing in it needs to start at zero: every element the merge
// reads was written earlier in the same call.
constexpr size_t kNaKeyBytes = size_t(kNaMaxKeys) * 8;
constexpr size_t kNaCountBytes = size_t(kNaMaxL) * 4;
constexpr size_t kNaScratchBytes = kNaKeyBytes + kNaCountBytes + size_t(kNaMaxLE) * 4;
__device__ __align__(256) unsigned char g_plan_scratch[kNaScratchBytes];

constexpr int kNaMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kNaMaxDevices];

// Device address of g_plan_scratch on the current device.
int scratch_of_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNaMaxDevices) return MOE_ECUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_plan_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return MOE_ECUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

int pow2_at_least(int n) {
  int p = 1;
  while (p < n) p <<= 1;
  return p;
}

}  // namespace
}  // namespace moe

extern "C" int cache_plan_swaps_noalloc(float* heat_dev, const int32_t* resid_dev, int L, int E,
                                        const moe_policy_cfg* p, moe_swap* plan_dev, int32_t* n_dev,
                                        moe_stream_t stream) {
  using namespace moe;
  if (!heat_dev || !resid_dev || !p || !plan_dev || !n_dev || p->max_swaps < 0 || p->max_swaps > 4096 ||
      !(p->threshold > 0.f))
    return MOE_EINVAL;
  const int stride = (E + 1) / 2;
  // the static scratch's capacity
  if (L < 1 || E < 1 || L > kNaMaxL || E > kMaxE || size_t(L) * E > size_t(kNaMaxLE) ||
      size_t(L) * stride > size_t(kNaMaxKeys))
    return MOE_EINVAL;
  void* scratch = nullptr;
  int rc = scratch_of_current_device(&scratch);
  if (rc) return rc;
  auto* cand = static_cast<unsigned long long*>(scratch);
  int32_t* cnt = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(scratch) + kNaKeyBytes);
  int32_t* cold_of = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(scratch) + kNaKeyBytes + kNaCountBytes);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  const int P = pow2_at_least(E);
  const size_t smem1 = size_t(2) * P * 8;
  if (smem1 > 48 * 1024 &&
      cudaFuncSetAttribute(k_plan_layer, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem1)) != cudaSuccess)
    return MOE_ECUDA;
  k_plan_layer<<<L, 1024, smem1, s>>>(heat_dev, resid_dev, E, P, p->threshold, p->decay, cand, stride, cnt, cold_of);
  MOE_LAUNCH_CHECK();
  const int PM = pow2_at_least(L * stride > 1 ? L * stride : 2);
  const size_t smem2 = size_t(PM) * 8;
  if (smem2 > 48 * 1024 &&
      cudaFuncSetAttribute(k_plan_merge, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem2)) != cudaSuccess)
    return MOE_ECUDA;
  k_plan_merge<<<1, 1024, smem2, s>>>(cand, stride, cnt, L, E, PM, resid_dev, cold_of, p->max_swaps, plan_dev, n_dev);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}
