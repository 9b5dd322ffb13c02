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
// only a stand-in symbol, so each device's real address is fetched once with
// cudaGetSymbolAddress (with that device current) and passed to the kernels.
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

namespace {

constexpr int kMaxRows = 64;          // B
constexpr int kMaxExperts = 1024;     // E
constexpr int kMaxTopK = 32;          // k
constexpr size_t kLogitsBytes = (size_t)kMaxRows * kMaxExperts * 4;
constexpr size_t kPairs = (size_t)kMaxRows * kMaxTopK;

// Layout of the scratch array (byte offsets, each 256-aligned).
constexpr size_t kOffLogits = 0;
constexpr size_t kOffDone = kOffLogits + kLogitsBytes;
constexpr size_t kOffNActive = kOffDone + 256;
constexpr size_t kOffActiveExpert = kOffNActive + 256;
constexpr size_t kOffActiveOff = kOffActiveExpert + kMaxExperts * 4;
constexpr size_t kOffPairList = kOffActiveOff + (kMaxExperts + 64) * 4;
constexpr size_t kOffHAmax = kOffPairList + kPairs * 4;
constexpr size_t kOffStatus = kOffHAmax + kPairs * 4;
constexpr size_t kScratchBytes = kOffStatus + 256;   // 284,672 bytes

__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

inline bool aligned16_noalloc(const void* p) { return ((uintptr_t)p & 15u) == 0; }

#define NOALLOC_ROUTER_KERNEL stream_gemv_kernel<kWfBf16, false, false, false, 1, 2, 4>

struct DeviceSetup {
  unsigned char* scratch = nullptr;   // device address of g_noalloc_scratch
  int threads = 0, grid = 0, NS = 0, stage_bytes = 0, smem = 0, red_pp = 0;
  int d = 0;                          // hidden size the launch shape was sized for
};

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
DeviceSetup g_setup[kMaxDevices];

// Once per (device, d): the scratch address and the router kernel's launch
// shape.  Must run before any stream capture on that device.
int device_setup(int dev, int d, DeviceSetup* out) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  DeviceSetup& s = g_setup[dev];
  if (!s.scratch) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    s.scratch = static_cast<unsigned char*>(p);
  }
  if (s.d != d) {
    using Sh = StreamShape<false, 8, 4>;
    const int KW = (d + Sh::WARP_K - 1) / Sh::WARP_K;
    const int stage = (int)((stream_rows_bytes(d, 1) + 127) / 128 * 128);
    const int red_pp = stream_red_pp(KW, false, 1, 4);
    const int red = 2 * red_pp * 4 + 64;
    const int budget = 110 * 1024;
    const int NS = std::min(8, (budget - red) / (stage + 16));
    if (NS < 2) return MOE_ERR_UNSUPPORTED;
    const int smem = NS * stage + NS * 16 + red;
    if (cudaFuncSetAttribute(NOALLOC_ROUTER_KERNEL, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
      return MOE_ERR_CUDA;
    int occ = 0, n_sm = 0;
    if (cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, NOALLOC_ROUTER_KERNEL, 32 * (KW + 1),
                                                      smem) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (occ < 1) return MOE_ERR_UNSUPPORTED;
    s.threads = 32 * (KW + 1);
    s.grid = occ * n_sm;
    s.NS = NS;
    s.stage_bytes = stage;
    s.smem = smem;
    s.red_pp = red_pp;
    s.d = d;
  }
  *out = s;
  return MOE_OK;
}

}  // namespace

extern "C" int moe_router_topk_noalloc(void* stream, const void* router_w, const float* router_bias,
                                       const void* x, int B, int d, int n_experts, int top_k,
                                       float routed_scale, int32_t* idx, float* w) {
  if (!router_w || !router_bias || !x || !idx || !w) return MOE_ERR_INVALID_ARG;
  if (d <= 0 || d % 256 != 0 || d > 8192 || top_k < 1 || n_experts < top_k ||
      !(routed_scale > 0.f))
    return MOE_ERR_INVALID_ARG;
  // sizes beyond the scratch array
  if (B < 1 || B > kMaxRows || n_experts > kMaxExperts || top_k > kMaxTopK)
    return MOE_ERR_UNSUPPORTED;
  if (!aligned16_noalloc(router_w) || !aligned16_noalloc(x)) return MOE_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  DeviceSetup s;
  int rc = device_setup(dev, d, &s);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the ticket must start at zero; everything else is overwritten before use
  if (cudaMemsetAsync(s.scratch + kOffDone, 0, 4, st) != cudaSuccess) return MOE_ERR_CUDA;

  StreamArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q = static_cast<const uint8_t*>(router_w);
  a.K = d;
  a.N = n_experts;
  a.k = top_k;
  a.B = B;
  a.x = static_cast<const uint16_t*>(x);
  a.out = reinterpret_cast<float*>(s.scratch + kOffLogits);
  a.status = reinterpret_cast<int*>(s.scratch + kOffStatus);
  a.NS = s.NS;
  a.stage_bytes = s.stage_bytes;
  a.red_pp = s.red_pp;
  a.kc = 1;
  const int grid = std::min(s.grid, (n_experts + 1) / 2);
  NOALLOC_ROUTER_KERNEL<<<grid, s.threads, s.smem, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;

  TopkArgs t{};
  t.logits = reinterpret_cast<const float*>(s.scratch + kOffLogits);
  t.bias = router_bias;
  t.B = B;
  t.d = d;
  t.E = n_experts;
  t.k = top_k;
  t.routed_scale = routed_scale;
  t.topk_idx = idx;
  t.topk_w = w;
  t.done = reinterpret_cast<unsigned*>(s.scratch + kOffDone);
  t.n_active = reinterpret_cast<int*>(s.scratch + kOffNActive);
  t.active_expert = reinterpret_cast<int*>(s.scratch + kOffActiveExpert);
  t.active_off = reinterpret_cast<int*>(s.scratch + kOffActiveOff);
  t.pair_list = reinterpret_cast<int*>(s.scratch + kOffPairList);
  t.h_amax = reinterpret_cast<unsigned*>(s.scratch + kOffHAmax);
  topk_kernel<<<B, kTopkThreads, 0, st>>>(t);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}
