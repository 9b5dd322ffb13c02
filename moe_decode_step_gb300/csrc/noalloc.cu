// Router + top-k without any allocation.
//
// Some callers cannot call cudaMalloc: code that runs inside a CUDA-graph
// capture it does not control, allocator-less runtimes that hand over a fixed
// pool of device memory, or callers that must not synchronise the device
// (cudaMalloc and cudaFree can).  moe_router_topk needs a layer handle whose
// workspace was allocated at create time; this entry point instead keeps its
// scratch (router logits, the completion ticket and the routing tables the
// top-k kernel writes) in one file-scope device array, sized for the largest
// supported problem, which every GPU that loads the library holds until the
// process exits.
//
// The host never dereferences that array: `g_noalloc_scratch` in host code is
// only a stand-in symbol, so the current device's real address is fetched
// with cudaGetSymbolAddress on every call and passed to the kernels.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "moe_decode.h"
#include "common.cuh"
#include "stream.cuh"
#include "topk.cuh"

using namespace moe;

namespace moe_internal {
int cuda_fail(cudaError_t e);
}

namespace {

constexpr int kMaxRows = 64;          // B
constexpr int kMaxExperts = 1024;     // E
constexpr int kMaxTopK = 32;          // k
constexpr int kMaxD = 7680;           // d, as for a layer
constexpr size_t kLogitsBytes = (size_t)kMaxRows * kMaxExperts * 4;
constexpr size_t kPairs = (size_t)kMaxRows * kMaxTopK;

// Layout of the scratch array (byte offsets, each 256-aligned).  The ticket
// and the status word sit side by side so one 8-byte clear resets both.
constexpr size_t kOffLogits = 0;
constexpr size_t kOffDone = kOffLogits + kLogitsBytes;
constexpr size_t kOffStatus = kOffDone + 4;
constexpr size_t kOffNActive = kOffDone + 256;
constexpr size_t kOffActiveExpert = kOffNActive + 256;
constexpr size_t kOffActiveOff = kOffActiveExpert + kMaxExperts * 4;
constexpr size_t kOffPairList = kOffActiveOff + (kMaxExperts + 64) * 4;
constexpr size_t kOffHAmax = kOffPairList + kPairs * 4;
constexpr size_t kScratchBytes = kOffHAmax + kPairs * 4;   // 284,416 bytes

__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

inline bool aligned16_noalloc(const void* p) { return ((uintptr_t)p & 15u) == 0; }

#define NOALLOC_ROUTER_KERNEL stream_gemv_kernel<kWfBf16, false, false, false, 1, 2, 4>

// The router kernel's shared-memory budget: its stage ring for any d up to
// kMaxD fits, so the kernel's attribute is set once per device to this.
constexpr int kRouterSmemBudget = 110 * 1024;

struct Shape {
  int threads = 0, grid = 0, NS = 0, stage_bytes = 0, smem = 0, red_pp = 0;
};

constexpr int kMaxDevices = 64;
constexpr int kShapes = kMaxD / 256;   // one per d = 256, 512, ..., kMaxD
std::mutex g_setup_mutex;
bool g_attr_set[kMaxDevices] = {};
Shape g_shape[kMaxDevices][kShapes];

// The router kernel's launch shape for (device, d), computed once.  The
// kernel's dynamic shared-memory limit is raised once per device to the
// largest any d needs, so calls with different d never lower it for another
// caller.  Host-side work only: no stream, no allocation.
int launch_shape(int dev, int d, Shape* out) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(NOALLOC_ROUTER_KERNEL,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kRouterSmemBudget);
    if (e != cudaSuccess) return moe_internal::cuda_fail(e);
    g_attr_set[dev] = true;
  }
  Shape& s = g_shape[dev][d / 256 - 1];
  if (s.threads == 0) {
    using Sh = StreamShape<false, 8, 4>;
    const int KW = (d + Sh::WARP_K - 1) / Sh::WARP_K;
    const int stage = (int)((stream_rows_bytes(d, 1) + 127) / 128 * 128);
    const int red_pp = stream_red_pp(KW, false, 1, 4);
    const int red = 2 * red_pp * 4 + 64;
    const int NS = std::min(8, (kRouterSmemBudget - red) / (stage + 16));
    if (NS < 2) return MOE_ERR_UNSUPPORTED;
    const int smem = NS * stage + NS * 16 + red;
    int occ = 0, n_sm = 0;
    cudaError_t e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, NOALLOC_ROUTER_KERNEL, 32 * (KW + 1),
                                                        smem);
    if (e != cudaSuccess) return moe_internal::cuda_fail(e);
    if (occ < 1) return MOE_ERR_UNSUPPORTED;
    s.threads = 32 * (KW + 1);
    s.grid = occ * n_sm;
    s.NS = NS;
    s.stage_bytes = stage;
    s.smem = smem;
    s.red_pp = red_pp;
  }
  *out = s;
  return MOE_OK;
}

// This device's address of the scratch array.  Looked up on every call (a
// host-side query): a cached address could outlive its context.
int scratch_address(unsigned char** p) {
  void* v = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&v, g_noalloc_scratch);
  if (e != cudaSuccess) return moe_internal::cuda_fail(e);
  if (!v) return MOE_ERR_CUDA;
  *p = static_cast<unsigned char*>(v);
  return MOE_OK;
}

}  // namespace

extern "C" int moe_router_topk_noalloc(void* stream, const void* router_w, const float* router_bias,
                                       const void* x, int B, int d, int n_experts, int top_k,
                                       float routed_scale, int32_t* idx, float* w) {
  if (!router_w || !router_bias || !x || !idx || !w) return MOE_ERR_INVALID_ARG;
  if (d <= 0 || d % 256 != 0 || top_k < 1 || n_experts < top_k || !(routed_scale > 0.f))
    return MOE_ERR_INVALID_ARG;
  // sizes beyond the scratch array or the tested launch shapes
  if (B < 1 || B > kMaxRows || n_experts > kMaxExperts || top_k > kMaxTopK || d > kMaxD)
    return MOE_ERR_UNSUPPORTED;
  if (!aligned16_noalloc(router_w) || !aligned16_noalloc(x)) return MOE_ERR_UNSUPPORTED;
  // an error left pending by earlier work is reported as it is, not blamed on
  // this call's launches
  cudaError_t e = cudaPeekAtLastError();
  if (e != cudaSuccess) return moe_internal::cuda_fail(e);
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return moe_internal::cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  Shape s;
  unsigned char* scratch = nullptr;
  int rc = launch_shape(dev, d, &s);
  if (rc || (rc = scratch_address(&scratch))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the ticket and the status word start at zero; everything else is
  // overwritten before use
  if ((e = cudaMemsetAsync(scratch + kOffDone, 0, 8, st)) != cudaSuccess)
    return moe_internal::cuda_fail(e);

  StreamArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q = static_cast<const uint8_t*>(router_w);
  a.K = d;
  a.N = n_experts;
  a.k = top_k;
  a.B = B;
  a.x = static_cast<const uint16_t*>(x);
  a.out = reinterpret_cast<float*>(scratch + kOffLogits);
  a.status = reinterpret_cast<int*>(scratch + kOffStatus);
  a.NS = s.NS;
  a.stage_bytes = s.stage_bytes;
  a.red_pp = s.red_pp;
  a.kc = 1;
  const int grid = std::min(s.grid, (n_experts + 1) / 2);
  NOALLOC_ROUTER_KERNEL<<<grid, s.threads, s.smem, st>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return moe_internal::cuda_fail(e);

  TopkArgs t{};
  t.logits = reinterpret_cast<const float*>(scratch + kOffLogits);
  t.bias = router_bias;
  t.B = B;
  t.d = d;
  t.E = n_experts;
  t.k = top_k;
  t.routed_scale = routed_scale;
  t.topk_idx = idx;
  t.topk_w = w;
  t.done = reinterpret_cast<unsigned*>(scratch + kOffDone);
  t.n_active = reinterpret_cast<int*>(scratch + kOffNActive);
  t.active_expert = reinterpret_cast<int*>(scratch + kOffActiveExpert);
  t.active_off = reinterpret_cast<int*>(scratch + kOffActiveOff);
  t.pair_list = reinterpret_cast<int*>(scratch + kOffPairList);
  t.h_amax = reinterpret_cast<unsigned*>(scratch + kOffHAmax);
  topk_kernel<<<B, kTopkThreads, 0, st>>>(t);
  if ((e = cudaGetLastError()) != cudaSuccess) return moe_internal::cuda_fail(e);
  return MOE_OK;
}

extern "C" int moe_router_topk_noalloc_status(int* device_status) {
  if (!device_status) return MOE_ERR_INVALID_ARG;
  unsigned char* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc) return rc;
  cudaError_t e = cudaDeviceSynchronize();
  int v = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&v, scratch + kOffStatus, sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(scratch + kOffStatus, 0, sizeof(int));
  if (e != cudaSuccess) return moe_internal::cuda_fail(e);
  *device_status = v;
  return MOE_OK;
}
