// C ABI of the MoE decode layer (see include/moe_decode.h for the contract).
//
// One forward = five kernels on the caller's stream, chained with programmatic
// dependent launch:
//   router GEMV (streamed bf16) -> top-k + routing tables
//   -> FC1: shared gate/up (bf16) then routed gate/up (MXFP4), SwiGLU
//   -> FC2: shared down (bf16) then routed down (MXFP4)
//   -> tail (combine + residual + RMSNorm)
// The shared expert streams first inside FC1/FC2: its weights do not depend on
// the routing, so FC1 starts them while top-k is still finishing (on the one
// SM FC1 leaves it at one row).  At one row on the mma.sync path FC1 and FC2
// are one persistent launch (stream_expert_kernel, four launches in all):
// FC2's weights stream into the stage ring while FC1's last items are
// consumed, and grid-wide counters replace the kernel boundary.
// Optional second stream (chained layers only): L2 prefetch of the next
// layer's router and shared-expert weights.
// No allocation, no host synchronisation: capturable into a CUDA graph.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <new>

#include "moe_decode.h"
#include "common.cuh"
#include "mxfp4.cuh"
#include "stream.cuh"
#include "tail.cuh"
#include "tc.cuh"
#include "topk.cuh"

using namespace moe;

namespace moe_internal {

std::atomic<int> g_last_cuda_error{0};

// Records a failed CUDA call for moe_last_cuda_error (shared by every entry
// point of the library).
int cuda_fail(cudaError_t e) {
  g_last_cuda_error.store((int)e);
  return MOE_ERR_CUDA;
}

}  // namespace moe_internal

namespace {

using moe_internal::cuda_fail;
using moe_internal::g_last_cuda_error;

#define MOE_CUDA(call)                             \
  do {                                             \
    cudaError_t e_ = (call);                       \
    if (e_ != cudaSuccess) return cuda_fail(e_);   \
  } while (0)

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

enum { kTimeRouterStart, kTimeRouterEnd, kTimeFc1End, kTimeFc2End, kTimeTailEnd, kNumTimeEvents };

struct Workspace {
  float* logits;
  unsigned* done;
  int32_t* topk_idx;
  float* topk_w;
  int* n_active;
  int* active_expert;
  int* active_off;
  int* pair_list;
  unsigned* h_amax;
  float* h;
  float* y_pair;
  float* hs;
  float* y_s;
  int* status;
  unsigned long long* trace;
  uint16_t* x_stage;
  uint16_t* res_stage;
  uint16_t* out_stage;
  // tensor-core expert path: activation planes of x and h, stream-K partials
  uint8_t* x_act;    // x planes [B][4d]
  uint8_t* x_code;   // their plane-0 code per row [B]
  uint8_t* h_act;    // h planes [P][4f]
  uint8_t* h_sfb;    // h plane scales per run, in the tensor-memory copy's atom order [P][4f]
  float* partial;
  unsigned* flags;
  // tensor-core dense pass: h_s as (hi, lo) bf16 columns for the shared down
  // projection, stream-K partials
  uint8_t* hs_hl;    // [f_shared / 8][2 B padded][16 bytes]
  float* dpartial;
  unsigned* dflags;
  // the tensor-core router's own stream-K slots (FC1's dense pass may run
  // while the router's last CTAs finish)
  float* rpartial;
  unsigned* rflags;
  // the one-row expert kernel's grid-wide counters: CTAs whose shared-expert
  // rows h_s [0] and routed rows h [1] are written (zeroed by top-k)
  unsigned* done_counts;
};

// Launch shape of one streaming-GEMV step.
struct StreamPlan {
  int threads = 0, grid = 0, NS = 0, stage_bytes = 0, smem = 0, red_pp = 0;
  int kc = 1;      // K chunks per item of the MXFP4 segment (CUDA-core path)
  int tc_kc = 0;   // K elements per stage of the tensor-core routed pass
  int dense_kc = 0;   // K elements per stage of the tensor-core dense pass
  int dense_ctas = 0;   // CTAs of the dense pass (0: the whole grid)
  int kc2 = 1;     // the fused one-row expert kernel: K chunks per item of routed FC2
};

enum { kStepRouter, kStepFc1, kStepFc2, kStepTc1, kStepTc2, kStepTcRouter, kStepExpert,
       kNumSteps };

// Expert paths: mma.sync on the tiled layouts (the GEMV regime: weights
// converted to f16 in registers), or tcgen05 on the UMMA layouts (block-scaled
// MMAs).  By default a layer keeps both and takes the tensor-core path from
// kTcMinBatch rows on: at B = 1 every routed expert has one activation row and
// the register path streams faster; from two rows per forward the MMA path
// does (measured at full size, B = 8 and 64).
enum { kPathAuto = 0, kPathMmaSync = 1, kPathTc = 2 };
constexpr int kTcMinBatch = 2;

// Expert weights in one path's layouts (FC1 gate/up pairs, FC2 rows): the
// caller's when given in those layouts, else a copy relaid at create time.
struct ExpertWeights {
  const uint8_t *gu_q = nullptr, *gu_s = nullptr, *d_q = nullptr, *d_s = nullptr;
  int layout_gu = 0, layout_d = 0;
  void* owned = nullptr;
  bool ok = false;
};

}  // namespace

struct moe_layer {
  moe_dims_t dims;
  moe_weights_t w;
  int device = 0;
  int n_sm = 0;
  int smem_optin = 0;   // largest dynamic shared memory a block may opt into
  void* ws_base = nullptr;
  Workspace ws{};
  cudaEvent_t ev_time[kNumTimeEvents] = {};
  bool timing = false, timed_once = false, tracing = false;
  moe_layer* next = nullptr;
  StreamPlan plan[kNumSteps][3];   // by batch class (B = 1, B <= 8, B > 8)
  size_t q_gu_stride = 0, s_gu_stride = 0, q_d_stride = 0, s_d_stride = 0;
  ExpertWeights wm;   // mma.sync path (tiled layouts), when kept
  ExpertWeights wt;   // tcgen05 path (UMMA layouts), when kept
  int tc_min_batch = kTcMinBatch;
  // failure-detection test hook (moe_debug_set_fault)
  // tcgen05 path: the shared expert's bf16 weights in the dense pass's tiles
  uint8_t* sh_gu_umma = nullptr;
  uint8_t* sh_d_umma = nullptr;
  uint8_t* router_umma = nullptr;   // router weights in 128-row tiles (last one zero-padded)
  void* sh_owned = nullptr;
  void* encode_tiled = nullptr;   // the driver's tensor-map encoder
  // failure-detection test hook (moe_debug_set_fault)
  int debug_fault = 0;
  int act_fmt = 0;   // routed experts' activations: 0 exact, 1 MXFP8 (moe_set_act_format)
  // moe_decode_forward_host: the host-buffer forward captured as one CUDA graph
  // (copies and kernels), reused while these arguments stay the same
  struct HostGraph {
    cudaGraphExec_t exec = nullptr;
    cudaStream_t stream = nullptr;
    const void* x = nullptr;
    void *res = nullptr, *out = nullptr;
    int B = 0, fault = 0;
    unsigned long long fault_ns = 0;
    bool timing = false, tracing = false;
    moe_layer* next = nullptr;
  } hg;
  unsigned long long debug_wait_ns = 0;
};

namespace {

template <typename T>
T* carve(char*& p, size_t count) {
  T* r = reinterpret_cast<T*>(p);
  p += (count * sizeof(T) + 255) & ~size_t(255);
  return r;
}

size_t workspace_bytes(const moe_dims_t& d, Workspace* ws, char* base) {
  char* p = base;
  const size_t B = d.max_batch, E = d.n_experts, k = d.top_k, P = B * k;
  Workspace w;
  w.logits = carve<float>(p, B * E);
  w.done = carve<unsigned>(p, 1);
  w.topk_idx = carve<int32_t>(p, P);
  w.topk_w = carve<float>(p, P);
  w.n_active = carve<int>(p, 1);
  w.active_expert = carve<int>(p, E);
  w.active_off = carve<int>(p, E + 1);
  w.pair_list = carve<int>(p, P);
  w.h_amax = carve<unsigned>(p, P);
  w.h = carve<float>(p, P * d.f);
  w.y_pair = carve<float>(p, P * d.d);
  w.hs = carve<float>(p, B * d.f_shared);
  w.y_s = carve<float>(p, B * d.d);
  w.status = carve<int>(p, 1);
  w.trace = carve<unsigned long long>(p, kTraceSlots);
  w.x_stage = carve<uint16_t>(p, B * d.d);
  w.res_stage = carve<uint16_t>(p, B * d.d);
  w.out_stage = carve<uint16_t>(p, B * d.d);
  w.x_act = carve<uint8_t>(p, B * planes_row_bytes(d.d));
  w.x_code = carve<uint8_t>(p, B);
  w.h_act = carve<uint8_t>(p, P * planes_row_bytes(d.f));
  w.h_sfb = carve<uint8_t>(p, P * 4 * (size_t)d.f);   // at most P runs
  w.partial = carve<float>(p, (size_t)kTcMaxCtas * kTcRmax * 128);
  w.flags = carve<unsigned>(p, kTcMaxCtas);
  w.hs_hl = carve<uint8_t>(p, (size_t)d.f_shared * dense_np(2 * (int)B) * 2);
  w.dpartial = carve<float>(p, (size_t)kTcMaxCtas * kTcDenseMaxN * 128);
  w.dflags = carve<unsigned>(p, kTcMaxCtas);
  w.rpartial = carve<float>(p, (size_t)kTcMaxCtas * kTcDenseMaxN * 128);
  w.rflags = carve<unsigned>(p, kTcMaxCtas);
  w.done_counts = carve<unsigned>(p, 2);
  if (ws) *ws = w;
  return (size_t)(p - base);
}

int validate_dims(const moe_dims_t& d) {
  if (d.d <= 0 || d.d % 256 != 0 || d.d > 7680) return MOE_ERR_INVALID_ARG;
  if (d.f <= 0 || d.f % 256 != 0 || d.f > 3072) return MOE_ERR_INVALID_ARG;
  if (d.f_shared <= 0 || d.f_shared % 256 != 0 || d.f_shared > 4096) return MOE_ERR_INVALID_ARG;
  if (d.top_k < 1 || d.top_k > 32) return MOE_ERR_INVALID_ARG;
  if (d.n_experts < d.top_k || d.n_experts > 1024) return MOE_ERR_INVALID_ARG;
  if (d.max_batch < 1 || d.max_batch > 64) return MOE_ERR_INVALID_ARG;
  if (!(d.routed_scale > 0.f) || !(d.rms_eps >= 0.f)) return MOE_ERR_INVALID_ARG;
  if (d.mxfp4_layout != 0 && d.mxfp4_layout != 1 && d.mxfp4_layout != 3) return MOE_ERR_UNSUPPORTED;
  if (d.expert_path < 0 || d.expert_path > 2) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// Kernel instantiations.  FC1 and FC2 each stream the shared expert (dense
// bf16, segment A) and the routed experts (MXFP4 on the tensor cores, segment
// B) in one launch; the variant is picked by batch class (B = 1, B <= 8,
// B > 8), which sets how many activation rows one pass of the shared expert
// carries (the routed segment takes up to 8 per pass at any batch).
// Routed FC1: items of one tile (8 gate/up row pairs), at most 16 K blocks
// per warp (d <= 7680 with 15 consumer warps).  Routed FC2: items of two
// tiles (32 rows), 4 K blocks per warp (f <= 1920) or at most 12 (f <= 4096).
using RouterCfg = StreamCfg<kWfBf16, false, false, false, 1, 1, 4>;
template <int R>
using Sh1Cfg = StreamCfg<kWfBf16, true, false, false, 1, 4, R, false, 1, 1, 8, 2>;
using Fc1Cfg = StreamCfg<kWfMx, true, false, true, 8, 8, 8, true, 1, 16>;
template <int R>
using Sh2Cfg = StreamCfg<kWfBf16, false, true, false, 8, 16, R, false, 1, 1, 4, 1>;
template <int NBM, int TM, int RM>
using Fc2Cfg = StreamCfg<kWfMx, false, true, true, 16 * TM, 16 * TM, RM, true, TM, NBM>;
#define MOE_ROUTER_KERNEL stream_gemv_kernel<kWfBf16, false, false, false, 1, 1, 4>
// One activation row (batch class 0): the routed step takes one row per
// expert with its x operand in shared memory.
#ifndef MOE_FC1_TM_B1
#define MOE_FC1_TM_B1 1
#endif
using Fc1OneRowCfg = StreamCfg<kWfMx, true, false, true, 8 * MOE_FC1_TM_B1, 8 * MOE_FC1_TM_B1, 1,
                               true, MOE_FC1_TM_B1, 16, 8, 4, true>;
#define MOE_FC1_KERNEL(RS) stream_dual_kernel<Sh1Cfg<RS>, Fc1Cfg, false>
#define MOE_FC1_KERNEL_ONE_ROW stream_dual_kernel<Sh1Cfg<1>, Fc1OneRowCfg, false>
// FC2 at batch class 0 (B = 1: one activation row per routed expert) takes
// items of MOE_FC2_TM_B1 tiles with one-column partials.
#ifndef MOE_FC2_TM_B1
#define MOE_FC2_TM_B1 4
#endif
#define MOE_FC2_TM(RS) ((RS) == 1 ? MOE_FC2_TM_B1 : 2)
#define MOE_FC2_RM(RS) ((RS) == 1 ? 1 : 8)
#define MOE_FC2_KERNEL(RS, NBM) \
  stream_dual_kernel<Sh2Cfg<RS>, Fc2Cfg<NBM, MOE_FC2_TM(RS), MOE_FC2_RM(RS)>, true>
// One row, both expert steps in one launch (FC1's and FC2's configurations).
#define MOE_EXPERT_KERNEL(NBM) \
  stream_expert_kernel<Sh1Cfg<1>, Fc1OneRowCfg, Sh2Cfg<1>, Fc2Cfg<NBM, MOE_FC2_TM(1), 1>>
// The same with MXFP8 activations (moe_set_act_format): x and h rounded to
// E4M3 with one E8M0 scale per 32 elements, then the same f16 MMAs.
using Fc1OneRowCfgF8 = StreamCfg<kWfMx, true, false, true, 8 * MOE_FC1_TM_B1, 8 * MOE_FC1_TM_B1, 1,
                                 true, MOE_FC1_TM_B1, 16, 8, 4, true, true>;
template <int NBM, int TM>
using Fc2CfgF8 = StreamCfg<kWfMx, false, true, true, 16 * TM, 16 * TM, 1, true, TM, NBM, 8, 4,
                           false, true>;
#define MOE_EXPERT_KERNEL_F8(NBM) \
  stream_expert_kernel<Sh1Cfg<1>, Fc1OneRowCfgF8, Sh2Cfg<1>, Fc2CfgF8<NBM, MOE_FC2_TM(1)>>
// Tensor-core path: FC1 streams the shared gate/up first (while top-k runs),
// FC2 the shared down first (its weights requested before FC1 is waited for).
#define MOE_TC1_KERNEL tc_kernel<true>
#define MOE_TC2_KERNEL tc_kernel<false>

int batch_class(int B) { return B == 1 ? 0 : (B <= 8 ? 1 : 2); }

// Shared-memory budget per CTA: how many CTAs of a step share an SM, chosen
// from each instantiation's register footprint.
constexpr int kBudget1 = 220 * 1024;   // one CTA per SM
constexpr int kBudget2 = 110 * 1024;   // two

// Consumer warps one segment needs for row length K.
template <class C>
int seg_warps(int K) {
  if constexpr (C::MMA) return kMmaWarps;
  else {
    using Sh = StreamShape<C::ACTH, C::CW, C::NQ>;
    return (K + Sh::WARP_K - 1) / Sh::WARP_K;
  }
}

// Largest stage of an MXFP4 segment (bytes).
#ifndef MOE_MX_STAGE_MAX
#define MOE_MX_STAGE_MAX (56 * 1024)
#endif

// K chunks per item of a tensor-core segment: the fewest that keep a stage
// within MOE_MX_STAGE_MAX while every warp's blocks stay inside one chunk.
template <class C>
int seg_kc(int K, int KW) {
  if constexpr (C::MMA) {
    const int nblk = K / 32, NB = mx_warp_blocks(K, KW);
    for (int kc = 1; kc <= 16; ++kc) {
      if (nblk % kc != 0) continue;
      const int CB = nblk / kc;
      if (kc > 1 && CB % NB != 0) continue;
      if (mx_stage_bytes(K, C::TM, kc) <= MOE_MX_STAGE_MAX) return kc;
    }
    return 1;
  } else {
    return 1;
  }
}

template <class C>
size_t seg_stage_bytes(int K, int kc) {
  if constexpr (C::MMA) return mx_stage_bytes(K, C::TM, kc);
  else return (size_t)(C::GLU ? 2 : 1) * stream_rows_bytes(K, C::SP);
}

// A tensor-core segment fits the launch: its K blocks per warp within NBMAX,
// one epilogue thread per item output, whole tiles of rows.
template <class C>
bool seg_fits(int K, int N, int KW) {
  if constexpr (C::MMA) {
    return mx_warp_blocks(K, KW) <= C::NBMAX && C::RW * C::RMAX <= 32 * KW &&
           N % (C::GLU ? 8 : 16) == 0 && K % 128 == 0;
  } else {
    return true;
  }
}

// Launch shape for a kernel whose segments have row lengths KA, KB and output
// rows NA, NB (segment B is the routed one).
template <class A, class B, typename Kern>
int plan_kernel(Kern kern, int KA, int NA, int KB, int NB, int n_sm, int budget, StreamPlan* p) {
  const int KW = std::max(seg_warps<A>(KA), seg_warps<B>(KB));
  if (KW > kMmaWarps) return MOE_ERR_UNSUPPORTED;   // more consumer warps than a CTA holds
  if (!seg_fits<A>(KA, NA, KW) || !seg_fits<B>(KB, NB, KW)) return MOE_ERR_UNSUPPORTED;
  StreamPlan r;
  r.threads = 32 * (KW + 1);
  r.kc = seg_kc<B>(KB, KW);
  const size_t sa = seg_stage_bytes<A>(KA, 1), sb = seg_stage_bytes<B>(KB, r.kc);
  r.stage_bytes = (int)((std::max(sa, sb) + 127) / 128 * 128);
  r.red_pp = std::max(stream_red_pp(KW, A::MMA, A::TM, A::RMAX),
                      stream_red_pp(KW, B::MMA, B::TM, B::RMAX));
  // an XS routed segment keeps its x operand after the partial buffers
  const int red_bytes = 2 * r.red_pp * 4 + 64 + (B::XS ? xs_extra_bytes(KB) : 0) +
                        (B::ROUTED && B::RMAX == 1 ? kOneRowTablesBytes : 0);
  r.NS = std::min(16, (budget - red_bytes) / (r.stage_bytes + 16));
  if (r.NS < 2 || r.NS < 2 * r.kc) return MOE_ERR_UNSUPPORTED;
  r.smem = r.NS * r.stage_bytes + r.NS * 16 + red_bytes;
  MOE_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, r.smem));
  int occ = 0;
  MOE_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, r.threads, r.smem));
  if (occ < 1) return MOE_ERR_UNSUPPORTED;
  r.grid = occ * n_sm;
  *p = r;
  return MOE_OK;
}

// FC2 comes in two instantiations by K blocks per warp (4 or 12).
bool fc2_small(const moe_dims_t& d) { return mx_warp_blocks(d.f, kMmaWarps) <= 4; }

template <int RS>
int plan_fc2(moe_layer* L, const moe_dims_t& d, int n, StreamPlan* p) {
  if (fc2_small(d))
    return plan_kernel<Sh2Cfg<RS>, Fc2Cfg<4, MOE_FC2_TM(RS), MOE_FC2_RM(RS)>>(
        MOE_FC2_KERNEL(RS, 4), d.f_shared, d.d, d.f, d.d, n, kBudget1, p);
  return plan_kernel<Sh2Cfg<RS>, Fc2Cfg<12, MOE_FC2_TM(RS), MOE_FC2_RM(RS)>>(
      MOE_FC2_KERNEL(RS, 12), d.f_shared, d.d, d.f, d.d, n, kBudget1, p);
}

// Launch shape of the fused one-row expert kernel: the four segments (shared
// gate/up, routed gate/up, shared down, routed down) share one stage ring of
// the largest segment stage; the routed segments keep their own K chunking.
// One CTA per SM, one SM left for top-k: the grid-wide barrier between the
// steps needs every CTA resident.
template <class A1, class B1, class A2, class B2, typename Kern>
int plan_expert(Kern kern, const moe_dims_t& d, int n_sm, int budget, StreamPlan* p) {
  const int KW = std::max(std::max(seg_warps<A1>(d.d), seg_warps<B1>(d.d)),
                          std::max(seg_warps<A2>(d.f_shared), seg_warps<B2>(d.f)));
  if (KW > kMmaWarps || n_sm < 2) return MOE_ERR_UNSUPPORTED;
  if (!seg_fits<A1>(d.d, d.f_shared, KW) || !seg_fits<B1>(d.d, d.f, KW) ||
      !seg_fits<A2>(d.f_shared, d.d, KW) || !seg_fits<B2>(d.f, d.d, KW))
    return MOE_ERR_UNSUPPORTED;
  StreamPlan r;
  r.threads = 32 * (KW + 1);
  r.kc = seg_kc<B1>(d.d, KW);
  r.kc2 = seg_kc<B2>(d.f, KW);
  cudaFuncAttributes fa;
  MOE_CUDA(cudaFuncGetAttributes(&fa, kern));
  budget -= (int)fa.sharedSizeBytes;   // static shared memory of the kernel, if any
  const size_t st = std::max(std::max(seg_stage_bytes<A1>(d.d, 1), seg_stage_bytes<B1>(d.d, r.kc)),
                             std::max(seg_stage_bytes<A2>(d.f_shared, 1),
                                      seg_stage_bytes<B2>(d.f, r.kc2)));
  r.stage_bytes = (int)((st + 127) / 128 * 128);
  r.red_pp = std::max(std::max(stream_red_pp(KW, A1::MMA, A1::TM, A1::RMAX),
                               stream_red_pp(KW, B1::MMA, B1::TM, B1::RMAX)),
                      std::max(stream_red_pp(KW, A2::MMA, A2::TM, A2::RMAX),
                               stream_red_pp(KW, B2::MMA, B2::TM, B2::RMAX)));
  const int red_bytes = 2 * r.red_pp * 4 + 64 + xs_extra_bytes(d.d) + kOneRowTablesBytes;
  r.NS = std::min(16, (budget - red_bytes) / (r.stage_bytes + 16));
  if (r.NS < 2 || r.NS < 2 * r.kc || r.NS < 2 * r.kc2) return MOE_ERR_UNSUPPORTED;
  r.smem = r.NS * r.stage_bytes + r.NS * 16 + red_bytes;
  MOE_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, r.smem));
  int occ = 0;
  MOE_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, r.threads, r.smem));
  if (occ != 1) return MOE_ERR_UNSUPPORTED;
  r.grid = n_sm - 1;
  *p = r;
  return MOE_OK;
}

// Launch shape of a tensor-core kernel: six warps, a stage ring sized for the
// larger pass (routed: rmax pairs; dense: np_max columns), and tensor memory
// for two accumulators, a scale slot per stage and the activation scales.
template <typename Kern>
int plan_tc(Kern kern, int K, int K_dense, int rmax, int np_max, bool rowscale, int E, int n_sm,
            int budget, StreamPlan* p) {
  if (K % 256 != 0 || K_dense % 128 != 0 || n_sm > kTcMaxCtas) return MOE_ERR_UNSUPPORTED;
  if (np_max > kTcDenseMaxN) return MOE_ERR_UNSUPPORTED;
  StreamPlan r;
  r.threads = kTcThreads;
  r.kc = 1;
  r.tc_kc = K % 512 == 0 ? 512 : 256;
  r.dense_kc = np_max <= 64 ? 128 : 64;
  const size_t st = std::max(tc_stage_bytes(r.tc_kc, rmax), dense_stage_bytes(r.dense_kc, np_max));
  r.stage_bytes = (int)((st + 127) / 128 * 128);
  const int extra = (int)tc_smem_bytes(E, K, rowscale);
  r.NS = std::min(16, (budget - extra) / (r.stage_bytes + 16));
  auto cols = [&](int ns) { return tc_tmem_cols(K, r.tc_kc, ns, rowscale); };
  while (r.NS > 2 && cols(r.NS) > kTcCols) --r.NS;
  if (r.NS < 2 || cols(r.NS) > kTcCols) return MOE_ERR_UNSUPPORTED;
  // at least 116 KB: a second CTA on the SM would wait in tcgen05.alloc
  r.smem = std::max((int)tc_kernel_smem(r.NS, r.stage_bytes, E, K, rowscale), 116 * 1024);
  if (r.smem > budget) return MOE_ERR_UNSUPPORTED;
  // one instantiation serves every batch class: allow the largest plan's size
  MOE_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, budget));
  int occ = 0;
  MOE_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, r.threads, r.smem));
  if (occ != 1) return MOE_ERR_UNSUPPORTED;
  r.grid = n_sm;
  *p = r;
  return MOE_OK;
}

// Largest batch of each batch class (B = 1, B <= 8, B <= 64).
constexpr int kClassMaxB[3] = {1, 8, 64};

// Launch shape of the tensor-core router: a stage ring of dense stages.
int plan_tc_router(int K, int np_max, int E, int n_sm, int budget, StreamPlan* p) {
  if (K % 128 != 0 || n_sm > kTcMaxCtas || np_max > 64) return MOE_ERR_UNSUPPORTED;
  StreamPlan r;
  r.threads = kTcThreads;
  r.dense_kc = 128;
  r.stage_bytes = (int)((dense_stage_bytes(r.dense_kc, np_max) + 127) / 128 * 128);
  const int extra = (int)tc_smem_bytes(E, K, true);
  r.NS = std::min(16, (budget - extra) / (r.stage_bytes + 16));
  if (r.NS < 2) return MOE_ERR_UNSUPPORTED;
  r.smem = std::max((int)tc_kernel_smem(r.NS, r.stage_bytes, E, K, true), 116 * 1024);
  if (r.smem > budget) return MOE_ERR_UNSUPPORTED;
  MOE_CUDA(cudaFuncSetAttribute(tc_router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                budget));
  int occ = 0;
  MOE_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, tc_router_kernel, r.threads,
                                                         r.smem));
  if (occ != 1) return MOE_ERR_UNSUPPORTED;
  r.grid = n_sm;
  // the logits on at most four CTAs per 128-row tile (each tile's finisher
  // adds the others' partial sums, one round trip to L2 per CTA); the other
  // CTAs quantize the x planes
  r.dense_ctas = std::min(n_sm, (E + 127) / 128 * 4);
  *p = r;
  return MOE_OK;
}

int plan_mma(moe_layer* L);

int plan_all(moe_layer* L) {
  const moe_dims_t& d = L->dims;
  const int n = L->n_sm;
  int rc;
#define MOE_PLAN(expr) \
  if ((rc = (expr))) return rc;
  MOE_PLAN((plan_kernel<RouterCfg, RouterCfg>(MOE_ROUTER_KERNEL, d.d, d.n_experts, d.d,
                                              d.n_experts, n, kBudget2,
                                              &L->plan[kStepRouter][0])));
  if (L->wt.ok) {
    const int E = d.n_experts;
    // one CTA per SM: all the shared memory a block may opt into
    const int bud = std::max(kBudget1, L->smem_optin);
    for (int c = 0; c < 3; ++c) {
      const int rmax = c == 0 ? 1 : kTcRmax;
      MOE_PLAN((plan_tc(MOE_TC1_KERNEL, d.d, d.d, rmax, dense_np(kClassMaxB[c]), true, E, n, bud,
                        &L->plan[kStepTc1][c])));
      MOE_PLAN((plan_tc(MOE_TC2_KERNEL, d.f, d.f_shared, rmax, dense_np(2 * kClassMaxB[c]), false,
                        E, n, bud, &L->plan[kStepTc2][c])));
      MOE_PLAN((plan_tc_router(d.d, dense_np(kClassMaxB[c]), E, n, bud,
                               &L->plan[kStepTcRouter][c])));
    }
  }
  if (L->wm.ok && (rc = plan_mma(L))) return rc;
#undef MOE_PLAN
  return MOE_OK;
}

// Launch shapes of the mma.sync path's kernels (they depend on the dims and
// the device alone).
int plan_mma(moe_layer* L) {
  const moe_dims_t& d = L->dims;
  const int n = L->n_sm;
  int rc;
#define MOE_PLAN(expr) \
  if ((rc = (expr))) return rc;
  MOE_PLAN((plan_kernel<Sh1Cfg<1>, Fc1OneRowCfg>(MOE_FC1_KERNEL_ONE_ROW, d.d, d.f_shared, d.d,
                                                 d.f, n, kBudget1, &L->plan[kStepFc1][0])));
  MOE_PLAN((plan_kernel<Sh1Cfg<2>, Fc1Cfg>(MOE_FC1_KERNEL(2), d.d, d.f_shared, d.d, d.f, n,
                                           kBudget1, &L->plan[kStepFc1][1])));
  MOE_PLAN((plan_kernel<Sh1Cfg<4>, Fc1Cfg>(MOE_FC1_KERNEL(4), d.d, d.f_shared, d.d, d.f, n,
                                           kBudget1, &L->plan[kStepFc1][2])));
  MOE_PLAN((plan_fc2<1>(L, d, n, &L->plan[kStepFc2][0])));
  MOE_PLAN((plan_fc2<2>(L, d, n, &L->plan[kStepFc2][1])));
  MOE_PLAN((plan_fc2<4>(L, d, n, &L->plan[kStepFc2][2])));
  // the fused one-row kernel: [0] exact activations, [1] MXFP8 activations
  const int bud1 = std::max(kBudget1, L->smem_optin);
  if (fc2_small(d)) {
    MOE_PLAN((plan_expert<Sh1Cfg<1>, Fc1OneRowCfg, Sh2Cfg<1>, Fc2Cfg<4, MOE_FC2_TM(1), 1>>(
        MOE_EXPERT_KERNEL(4), d, n, bud1, &L->plan[kStepExpert][0])));
    MOE_PLAN((plan_expert<Sh1Cfg<1>, Fc1OneRowCfgF8, Sh2Cfg<1>, Fc2CfgF8<4, MOE_FC2_TM(1)>>(
        MOE_EXPERT_KERNEL_F8(4), d, n, bud1, &L->plan[kStepExpert][1])));
  } else {
    MOE_PLAN((plan_expert<Sh1Cfg<1>, Fc1OneRowCfg, Sh2Cfg<1>, Fc2Cfg<12, MOE_FC2_TM(1), 1>>(
        MOE_EXPERT_KERNEL(12), d, n, bud1, &L->plan[kStepExpert][0])));
    MOE_PLAN((plan_expert<Sh1Cfg<1>, Fc1OneRowCfgF8, Sh2Cfg<1>, Fc2CfgF8<12, MOE_FC2_TM(1)>>(
        MOE_EXPERT_KERNEL_F8(12), d, n, bud1, &L->plan[kStepExpert][1])));
  }
#undef MOE_PLAN
  return MOE_OK;
}

// Launch with programmatic stream serialization when `pdl` (the kernel may
// start while its predecessor in the stream finishes; it waits with
// griddepcontrol.wait before touching the predecessor's results).
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                      cudaStream_t st, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Timing events: inside a stream capture they must be external record nodes so
// that every graph replay records them.
cudaError_t record_time(moe_layer* L, int which, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(st, &cs);
  if (e != cudaSuccess) return e;
  if (cs == cudaStreamCaptureStatusActive)
    return cudaEventRecordWithFlags(L->ev_time[which], st, cudaEventRecordExternal);
  return cudaEventRecord(L->ev_time[which], st);
}

StreamArgs base_args(moe_layer* L) {
  StreamArgs a;
  std::memset(&a, 0, sizeof(a));
  a.k = L->dims.top_k;
  a.n_active = L->ws.n_active;
  a.active_expert = L->ws.active_expert;
  a.active_off = L->ws.active_off;
  a.pair_list = L->ws.pair_list;
  a.status = L->ws.status;
  a.trace = L->tracing ? L->ws.trace : nullptr;
  return a;
}

template <typename K>
int launch_step(moe_layer* L, K kern, const StreamPlan& p, StreamArgs a, int n_items_cap,
                cudaStream_t st, bool pdl) {
  a.NS = p.NS;
  a.stage_bytes = p.stage_bytes;
  a.red_pp = p.red_pp;
  a.kc = p.kc;
  const int grid = n_items_cap > 0 ? std::min(p.grid, n_items_cap) : p.grid;
  MOE_CUDA(launch_ex(kern, dim3(grid), dim3(p.threads), (size_t)p.smem, st, pdl, a));
  return MOE_OK;
}

// The tensor-core path for a forward of B rows?
bool use_tc(const moe_layer* L, int B) { return L->wt.ok && (!L->wm.ok || B >= L->tc_min_batch); }


int launch_router_tc(moe_layer* L, cudaStream_t st, const void* x, int B);

// Rows from which the tensor-core path computes the router logits on the
// tensor cores too (one dense pass whatever the batch) rather than with the
// CUDA-core GEMV (passes of 4 rows): measured at B = 16, 17 against 27 us for
// the router; at B = 64 the dense pass is faster.
#ifndef MOE_TC_ROUTER_MIN_B
#define MOE_TC_ROUTER_MIN_B 25
#endif

int launch_router(moe_layer* L, cudaStream_t st, const void* x, int B, int32_t* idx, float* w) {
  const moe_dims_t& d = L->dims;
  StreamArgs a = base_args(L);
  a.q = static_cast<const uint8_t*>(L->w.router_w);
  a.K = d.d;
  a.N = d.n_experts;
  a.B = B;
  a.x = static_cast<const uint16_t*>(x);
  a.out = L->ws.logits;
  a.trace_id = 0;
  int rc;
  if (use_tc(L, B) && batch_class(B) == 2 && B >= MOE_TC_ROUTER_MIN_B) {
    // from MOE_TC_ROUTER_MIN_B rows the CUDA-core router is compute-bound
    // (passes of 4 rows): logits on the tensor cores, plus the activation
    // planes the tensor-core FC1 streams
    if ((rc = launch_router_tc(L, st, x, B))) return rc;
  } else {
    if (use_tc(L, B)) {   // the activation planes the tensor-core FC1 streams
      a.xq = L->ws.x_act;
      a.xq_code = L->ws.x_code;
      a.xq_f8 = L->act_fmt == 1;
    }
    // programmatic launch: behind the previous layer's tail the router
    // streams its weights while that tail runs (it waits before reading x)
    rc = launch_step(L, MOE_ROUTER_KERNEL, L->plan[kStepRouter][0], a, d.n_experts, st, true);
    if (rc) return rc;
  }
  TopkArgs t{};
  t.logits = L->ws.logits;
  t.bias = L->w.router_bias;
  t.B = B;
  t.d = d.d;
  t.E = d.n_experts;
  t.k = d.top_k;
  t.routed_scale = d.routed_scale;
  t.topk_idx = idx;
  t.topk_w = w;
  t.done = L->ws.done;
  t.n_active = L->ws.n_active;
  t.active_expert = L->ws.active_expert;
  t.active_off = L->ws.active_off;
  t.pair_list = L->ws.pair_list;
  t.h_amax = L->ws.h_amax;
  t.trace = L->tracing ? L->ws.trace : nullptr;
  // one row on the mma.sync path: FC2 streams its routed weights under this flag
  t.reset_counts = (!use_tc(L, B) && idx == L->ws.topk_idx) ? L->ws.done_counts : nullptr;
  MOE_CUDA(launch_ex(topk_kernel, dim3(B), dim3(kTopkThreads), 0, st, true, t));
  return MOE_OK;
}

template <typename K>
int launch_dual(K kern, const StreamPlan& p, StreamArgs a0, StreamArgs a1, cudaStream_t st,
                int grid) {
  a0.NS = a1.NS = p.NS;
  a0.stage_bytes = a1.stage_bytes = p.stage_bytes;
  a0.red_pp = a1.red_pp = p.red_pp;
  a0.kc = a1.kc = p.kc;
  MOE_CUDA(launch_ex(kern, dim3(grid), dim3(p.threads), (size_t)p.smem, st, true, a0, a1));
  return MOE_OK;
}

// CTAs of FC1 on the mma.sync path.  At B = 1 one SM holds the top-k CTA
// when FC1 launches; a CTA waiting for it would start (and finish) last, so
// FC1 leaves that SM out.
int fc1_grid(const moe_layer* L, int B) {
  const int g = L->plan[kStepFc1][batch_class(B)].grid;
  return B == 1 ? std::max(1, g - 1) : g;
}

// FC1: shared gate/up (bf16) then routed gate/up (MXFP4), SwiGLU epilogues.
int launch_fc1(moe_layer* L, cudaStream_t st, const void* x, int B) {
  const moe_dims_t& d = L->dims;
  StreamArgs sa = base_args(L);
  sa.q = static_cast<const uint8_t*>(L->w.shared_gu);
  sa.K = d.d;
  sa.N = d.f_shared;
  sa.B = B;
  sa.x = static_cast<const uint16_t*>(x);
  sa.out = L->ws.hs;
  StreamArgs ra = base_args(L);
  ra.q = L->wm.gu_q;
  ra.s = L->wm.gu_s;
  ra.q_stride = L->q_gu_stride;
  ra.s_stride = L->s_gu_stride;
  ra.K = d.d;
  ra.N = d.f;
  ra.x = static_cast<const uint16_t*>(x);
  ra.out = L->ws.h;
  ra.out_amax = L->ws.h_amax;
  sa.trace_id = ra.trace_id = 2;
  const int grid = fc1_grid(L, B);
  const StreamPlan& p = L->plan[kStepFc1][batch_class(B)];
  switch (batch_class(B)) {
    case 0: return launch_dual(MOE_FC1_KERNEL_ONE_ROW, p, sa, ra, st, grid);
    case 1: return launch_dual(MOE_FC1_KERNEL(2), p, sa, ra, st, grid);
    default: return launch_dual(MOE_FC1_KERNEL(4), p, sa, ra, st, grid);
  }
}

// Tensor-core path: the routed step's arguments common to FC1 and FC2.
TcArgs tc_base_args(moe_layer* L, const StreamPlan& p) {
  TcArgs b;
  std::memset(&b, 0, sizeof(b));
  b.n_active = L->ws.n_active;
  b.active_expert = L->ws.active_expert;
  b.active_off = L->ws.active_off;
  b.pair_list = L->ws.pair_list;
  b.partial = L->ws.partial;
  b.flags = L->ws.flags;
  b.status = L->ws.status;
  b.NS = p.NS;
  b.stage_bytes = p.stage_bytes;
  b.KC = p.tc_kc;
  b.trace = L->tracing ? L->ws.trace : nullptr;
  return b;
}

// The dense pass's arguments common to FC1 and FC2.
TcDense dense_base_args(moe_layer* L, const StreamPlan& p, int B) {
  TcDense dn;
  std::memset(&dn, 0, sizeof(dn));
  dn.KC = p.dense_kc;
  dn.B = B;
  dn.partial = L->ws.dpartial;
  dn.flags = L->ws.dflags;
  return dn;
}

template <typename K>
int launch_tc(K kern, const StreamPlan& p, const TcArgs& b, const TcDense& dn,
              const CUtensorMap& xmap, cudaStream_t st, int grid) {
  MOE_CUDA(launch_ex(kern, dim3(grid), dim3(p.threads), (size_t)p.smem, st, true, b, dn, xmap));
  return MOE_OK;
}

// Tensor map of x [B][d] (bf16, row-major) with a box of 8 K elements x NP
// rows; rows past B read as zeros.
int encode_x_map(moe_layer* L, const void* x, int B, int NP, CUtensorMap* map) {
  using Encode = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  if (!L->encode_tiled) return MOE_ERR_UNSUPPORTED;
  const cuuint64_t dims[2] = {(cuuint64_t)L->dims.d, (cuuint64_t)B};
  const cuuint64_t strides[1] = {(cuuint64_t)L->dims.d * 2};
  const cuuint32_t box[2] = {8, (cuuint32_t)NP};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = reinterpret_cast<Encode>(L->encode_tiled)(
      map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_UNSUPPORTED;
}

// The router on the tensor-core path: logits [B][E] as a dense pass on x, and
// the x planes of the routed FC1.  The first kernel of a forward: no
// programmatic launch (everything before it in the stream has finished).
int launch_router_tc(moe_layer* L, cudaStream_t st, const void* x, int B) {
  const moe_dims_t& d = L->dims;
  const StreamPlan& p = L->plan[kStepTcRouter][batch_class(B)];
  TcDense dn = dense_base_args(L, p, B);
  dn.w = L->router_umma;
  dn.K = d.d;
  dn.tiles = (d.n_experts + 127) / 128;
  dn.N = d.n_experts;
  dn.NP = dense_np(B);
  dn.out = L->ws.logits;
  dn.partial = L->ws.rpartial;
  dn.flags = L->ws.rflags;
  dn.ctas = p.dense_ctas;
  TcXPlanes xp;
  xp.x = static_cast<const uint16_t*>(x);
  xp.B = B;
  xp.K = d.d;
  xp.xq = L->ws.x_act;
  xp.xq_code = L->ws.x_code;
  xp.f8 = L->act_fmt == 1;
  CUtensorMap xmap;
  int rc = encode_x_map(L, x, B, dn.NP, &xmap);
  if (rc) return rc;
  MOE_CUDA(launch_ex(tc_router_kernel, dim3(p.grid), dim3(p.threads), (size_t)p.smem, st, false,
                     dn, xmap, xp, p.NS, p.stage_bytes, L->ws.status,
                     L->tracing ? L->ws.trace : (unsigned long long*)nullptr));
  return MOE_OK;
}

// FC1 on the tensor-core path: the shared gate/up as a dense pass on x, then
// routed gate/up (x planes x UMMA-layout weights), SwiGLU, h and its planes.
int launch_fc1_tc(moe_layer* L, cudaStream_t st, const void* x, int B) {
  const moe_dims_t& d = L->dims;
  const StreamPlan& p = L->plan[kStepTc1][batch_class(B)];
  TcArgs b = tc_base_args(L, p);
  b.q = L->wt.gu_q;
  b.s = L->wt.gu_s;
  b.q_stride = L->q_gu_stride;
  b.s_stride = L->s_gu_stride;
  b.K = d.d;
  b.tiles = d.f / 64;
  b.N = d.f;
  b.act_div = d.top_k;
  b.rowscale = 1;
  b.act = L->ws.x_act;
  b.act_code = L->ws.x_code;
  b.out = L->ws.h;
  b.out_amax = L->ws.h_amax;
  b.out_act = L->ws.h_act;
  b.out_sfb = L->ws.h_sfb;
  b.out_f8 = L->act_fmt == 1;
  b.trace_id = 2;
  TcDense dn = dense_base_args(L, p, B);
  dn.w = L->sh_gu_umma;
  dn.K = d.d;
  dn.tiles = d.f_shared / 64;
  dn.N = d.f_shared;
  dn.NP = dense_np(B);
  dn.out = L->ws.hs;
  dn.out_hl = L->ws.hs_hl;
  dn.out_np = dense_np(2 * B);
  CUtensorMap xmap;
  int rc = encode_x_map(L, x, B, dn.NP, &xmap);
  if (rc) return rc;
  // at B = 1 one SM holds the top-k CTA when FC1 launches (see launch_fc1)
  const int grid = B == 1 ? std::max(1, p.grid - 1) : p.grid;
  return launch_tc(MOE_TC1_KERNEL, p, b, dn, xmap, st, grid);
}

// FC2 on the tensor-core path: the shared down as a dense pass on h_s's
// (hi, lo) columns, then routed down (h planes x UMMA-layout weights).
int launch_fc2_tc(moe_layer* L, cudaStream_t st, int B) {
  const moe_dims_t& d = L->dims;
  const StreamPlan& p = L->plan[kStepTc2][batch_class(B)];
  TcArgs b = tc_base_args(L, p);
  b.q = L->wt.d_q;
  b.s = L->wt.d_s;
  b.q_stride = L->q_d_stride;
  b.s_stride = L->s_d_stride;
  b.K = d.f;
  b.tiles = d.d / 128;
  b.N = d.d;
  b.act_div = 1;
  b.rowscale = 0;
  b.act = L->ws.h_act;
  b.act_sfb = L->ws.h_sfb;
  b.out = L->ws.y_pair;
  b.trace_id = 3;
  TcDense dn = dense_base_args(L, p, B);
  dn.w = L->sh_d_umma;
  dn.act = L->ws.hs_hl;
  dn.K = d.f_shared;
  dn.tiles = d.d / 128;
  dn.N = d.d;
  dn.NP = dense_np(2 * B);
  dn.hilo = 1;
  dn.out = L->ws.y_s;
  CUtensorMap unused;
  std::memset(&unused, 0, sizeof(unused));
  return launch_tc(MOE_TC2_KERNEL, p, b, dn, unused, st, p.grid);
}

// FC2: shared down (bf16, h_s) then routed down (MXFP4, h).
int launch_fc2(moe_layer* L, cudaStream_t st, int B) {
  const moe_dims_t& d = L->dims;
  StreamArgs sa = base_args(L);
  sa.q = static_cast<const uint8_t*>(L->w.shared_d);
  sa.K = d.f_shared;
  sa.N = d.d;
  sa.B = B;
  sa.h = L->ws.hs;
  sa.out = L->ws.y_s;
  StreamArgs ra = base_args(L);
  ra.q = L->wm.d_q;
  ra.s = L->wm.d_s;
  ra.q_stride = L->q_d_stride;
  ra.s_stride = L->s_d_stride;
  ra.K = d.f;
  ra.N = d.d;
  ra.h = L->ws.h;
  ra.h_amax = L->ws.h_amax;
  ra.out = L->ws.y_pair;
  sa.trace_id = ra.trace_id = 3;
  const StreamPlan& p = L->plan[kStepFc2][batch_class(B)];
  if (fc2_small(d)) {
    switch (batch_class(B)) {
      case 0: return launch_dual(MOE_FC2_KERNEL(1, 4), p, sa, ra, st, p.grid);
      case 1: return launch_dual(MOE_FC2_KERNEL(2, 4), p, sa, ra, st, p.grid);
      default: return launch_dual(MOE_FC2_KERNEL(4, 4), p, sa, ra, st, p.grid);
    }
  }
  switch (batch_class(B)) {
    case 0: return launch_dual(MOE_FC2_KERNEL(1, 12), p, sa, ra, st, p.grid);
    case 1: return launch_dual(MOE_FC2_KERNEL(2, 12), p, sa, ra, st, p.grid);
    default: return launch_dual(MOE_FC2_KERNEL(4, 12), p, sa, ra, st, p.grid);
  }
}

// One row on the mma.sync path: FC1 and FC2 in one launch (see
// stream_expert_kernel), the segments' arguments as launch_fc1 and launch_fc2
// build them.
int launch_expert(moe_layer* L, cudaStream_t st, const void* x) {
  const moe_dims_t& d = L->dims;
  const bool f8 = L->act_fmt == 1;
  const StreamPlan& p = L->plan[kStepExpert][f8 ? 1 : 0];
  StreamArgs4 g;
  std::memset(&g, 0, sizeof(g));
  StreamArgs& s1 = g.a[0];
  s1 = base_args(L);
  s1.q = static_cast<const uint8_t*>(L->w.shared_gu);
  s1.K = d.d;
  s1.N = d.f_shared;
  s1.B = 1;
  s1.x = static_cast<const uint16_t*>(x);
  s1.out = L->ws.hs;
  StreamArgs& r1 = g.a[1];
  r1 = base_args(L);
  r1.q = L->wm.gu_q;
  r1.s = L->wm.gu_s;
  r1.q_stride = L->q_gu_stride;
  r1.s_stride = L->s_gu_stride;
  r1.K = d.d;
  r1.N = d.f;
  r1.x = static_cast<const uint16_t*>(x);
  r1.out = L->ws.h;
  r1.out_amax = L->ws.h_amax;
  r1.done_count = L->ws.done_counts;
  r1.wait_ns = L->debug_fault == 1 ? L->debug_wait_ns : 0;
  StreamArgs& s2 = g.a[2];
  s2 = base_args(L);
  s2.q = static_cast<const uint8_t*>(L->w.shared_d);
  s2.K = d.f_shared;
  s2.N = d.d;
  s2.B = 1;
  s2.h = L->ws.hs;
  s2.out = L->ws.y_s;
  StreamArgs& r2 = g.a[3];
  r2 = base_args(L);
  r2.q = L->wm.d_q;
  r2.s = L->wm.d_s;
  r2.q_stride = L->q_d_stride;
  r2.s_stride = L->s_d_stride;
  r2.K = d.f;
  r2.N = d.d;
  r2.h = L->ws.h;
  r2.h_amax = L->ws.h_amax;
  r2.out = L->ws.y_pair;
  for (int i = 0; i < 4; ++i) {
    g.a[i].NS = p.NS;
    g.a[i].stage_bytes = p.stage_bytes;
    g.a[i].red_pp = p.red_pp;
    g.a[i].kc = 1;
    g.a[i].trace_id = i < 2 ? 2 : 3;
  }
  r1.kc = p.kc;
  r2.kc = p.kc2;
  g.skip_count = L->debug_fault == 1;
  const dim3 grid(p.grid), block(p.threads);
  if (f8) {
    if (fc2_small(d))
      MOE_CUDA(launch_ex(MOE_EXPERT_KERNEL_F8(4), grid, block, (size_t)p.smem, st, true, g));
    else
      MOE_CUDA(launch_ex(MOE_EXPERT_KERNEL_F8(12), grid, block, (size_t)p.smem, st, true, g));
  } else if (fc2_small(d)) {
    MOE_CUDA(launch_ex(MOE_EXPERT_KERNEL(4), grid, block, (size_t)p.smem, st, true, g));
  } else {
    MOE_CUDA(launch_ex(MOE_EXPERT_KERNEL(12), grid, block, (size_t)p.smem, st, true, g));
  }
  return MOE_OK;
}

int launch_tail(moe_layer* L, cudaStream_t st, int B, void* residual, void* out, float* y_r_dbg,
                float* z_dbg, float* out_dbg, bool pdl) {
  TailArgs a{};
  a.y_pair = L->ws.y_pair;
  a.topk_w = L->ws.topk_w;
  a.y_s = L->ws.y_s;
  a.gamma = static_cast<const uint16_t*>(L->w.rms_gamma);
  a.residual = static_cast<uint16_t*>(residual);
  a.out = static_cast<uint16_t*>(out);
  a.y_r_dbg = y_r_dbg;
  a.z_dbg = z_dbg;
  a.out_dbg = out_dbg;
  a.B = B;
  a.d = L->dims.d;
  a.k = L->dims.top_k;
  a.eps = L->dims.rms_eps;
  a.trace = L->tracing ? L->ws.trace : nullptr;
  a.h_amax = L->ws.h_amax;
  if (L->next) {
    // the next layer's router weights into L2 from the tail's CTAs, which
    // start while this layer's expert kernels finish: HBM is then idle but
    // for the last expert items, and the next router streams those weights
    // first.  Prefetching more (the next shared expert) or earlier (while
    // this layer's experts stream) only competes with them for HBM.
    a.pref = static_cast<const char*>(L->next->w.router_w);
    a.pref_bytes = (size_t)L->next->dims.n_experts * L->next->dims.d * 2;
  }
  MOE_CUDA(launch_ex(tail_kernel, dim3(kTailCluster, B), dim3(L->dims.d / 32), 0, st, pdl, a));
  return MOE_OK;
}

int check_forward_args(moe_layer* L, const void* x, int B) {
  if (!L) return MOE_ERR_INVALID_ARG;
  if (B < 1 || B > L->dims.max_batch) return MOE_ERR_UNSUPPORTED;
  if (!x) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int forward_impl(moe_layer* L, cudaStream_t st, const void* x, int B, void* residual, void* out,
                 float* y_r_dbg, float* y_s_dbg, float* h_dbg, float* z_dbg, float* out_dbg) {
  int rc = check_forward_args(L, x, B);
  if (rc) return rc;
  if (!residual || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(residual) || !aligned16(out)) return MOE_ERR_UNSUPPORTED;
  const bool tm = L->timing;
  const bool tc = use_tc(L, B);
  // MXFP8 activations: the tensor-core path (its activation planes hold the
  // rounded values) or the one-row mma.sync kernel, not the mma.sync batches
  if (L->act_fmt == 1 && !tc && B != 1) return MOE_ERR_UNSUPPORTED;
  if (L->tracing) {
    MOE_CUDA(cudaMemsetAsync(L->ws.trace, 0xFF, 8 * sizeof(unsigned long long), st));
    MOE_CUDA(cudaMemsetAsync(L->ws.trace + 8, 0, 8 * sizeof(unsigned long long), st));
  }
  if (tm) MOE_CUDA(record_time(L, kTimeRouterStart, st));
  if ((rc = launch_router(L, st, x, B, L->ws.topk_idx, L->ws.topk_w))) return rc;
  if (tm) MOE_CUDA(record_time(L, kTimeRouterEnd, st));
  if (!tc && B == 1) {   // one launch for both expert steps
    if ((rc = launch_expert(L, st, x))) return rc;
    if (tm) MOE_CUDA(record_time(L, kTimeFc1End, st));
    if (tm) MOE_CUDA(record_time(L, kTimeFc2End, st));
  } else {
    if ((rc = tc ? launch_fc1_tc(L, st, x, B) : launch_fc1(L, st, x, B))) return rc;
    if (tm) MOE_CUDA(record_time(L, kTimeFc1End, st));
    if ((rc = tc ? launch_fc2_tc(L, st, B) : launch_fc2(L, st, B))) return rc;
    if (tm) MOE_CUDA(record_time(L, kTimeFc2End, st));
  }
  if ((rc = launch_tail(L, st, B, residual, out, y_r_dbg, z_dbg, out_dbg, true))) return rc;
  if (tm) {
    MOE_CUDA(record_time(L, kTimeTailEnd, st));
    L->timed_once = true;
  }
  const size_t P = (size_t)B * L->dims.top_k;
  if (y_s_dbg)
    MOE_CUDA(cudaMemcpyAsync(y_s_dbg, L->ws.y_s, (size_t)B * L->dims.d * 4,
                             cudaMemcpyDeviceToDevice, st));
  if (h_dbg)
    MOE_CUDA(cudaMemcpyAsync(h_dbg, L->ws.h, P * L->dims.f * 4, cudaMemcpyDeviceToDevice, st));
  return MOE_OK;
}

// n_mat matrices rows x k from layout `from` to layout `to` (default stream).
int relayout_device(const uint8_t* q_in, const uint8_t* s_in, int64_t n_mat, int64_t rows,
                    int64_t k, int from, int to, uint8_t* q_out, uint8_t* s_out) {
  if (!mx_layout_ok(rows, k, from) || !mx_layout_ok(rows, k, to)) return MOE_ERR_UNSUPPORTED;
  const int64_t qb = rows * (k / 2), sb = rows * (k / 32);
  const int64_t total = rows * (k / 32);
  if (total == 0) return MOE_OK;
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, 152 * 32);
  for (int64_t m = 0; m < n_mat; ++m) {
    mxfp4_relayout_kernel<<<(unsigned)blocks, 256>>>(q_in + m * qb, s_in + m * sb, rows, k, from,
                                                     q_out + m * qb, s_out + m * sb, to);
    MOE_CUDA(cudaGetLastError());
  }
  return MOE_OK;
}

// One path's expert weights: borrowed when the caller's layout (dims
// mxfp4_layout) is the path's (`want`: 1 tiled, 3 UMMA), else relaid into a
// copy the handle owns.
int setup_weights(moe_layer* L, const moe_weights_t& w, int want, ExpertWeights& ew) {
  const moe_dims_t& d = L->dims;
  ew.layout_gu = want == 3 ? kMxUmmaPairs : kMxTiledPairs;
  ew.layout_d = want == 3 ? kMxUmma : kMxTiled;
  if (d.mxfp4_layout == want) {
    ew.gu_q = w.w_gu_q;
    ew.gu_s = w.w_gu_s;
    ew.d_q = w.w_d_q;
    ew.d_s = w.w_d_s;
    ew.ok = true;
    return MOE_OK;
  }
  const size_t E = d.n_experts, f = d.f, dd = d.d;
  const size_t total = E * (L->q_gu_stride + L->s_gu_stride + L->q_d_stride + L->s_d_stride);
  if (cudaMalloc(&ew.owned, total) != cudaSuccess) {
    cudaGetLastError();
    ew.owned = nullptr;
    return MOE_ERR_ALLOC;
  }
  uint8_t* gq = static_cast<uint8_t*>(ew.owned);
  uint8_t* gs = gq + E * L->q_gu_stride;
  uint8_t* dq = gs + E * L->s_gu_stride;
  uint8_t* ds = dq + E * L->q_d_stride;
  const int from_gu = d.mxfp4_layout == 0 ? kMxCanonical
                      : d.mxfp4_layout == 1 ? kMxTiledPairs : kMxUmmaPairs;
  const int from_d = d.mxfp4_layout == 0 ? kMxCanonical : d.mxfp4_layout == 1 ? kMxTiled : kMxUmma;
  int rc;
  if ((rc = relayout_device(w.w_gu_q, w.w_gu_s, (int64_t)E, 2 * (int64_t)f, (int64_t)dd, from_gu,
                            ew.layout_gu, gq, gs)) ||
      (rc = relayout_device(w.w_d_q, w.w_d_s, (int64_t)E, (int64_t)dd, (int64_t)f, from_d,
                            ew.layout_d, dq, ds)))
    return rc;
  MOE_CUDA(cudaStreamSynchronize(nullptr));
  ew.gu_q = gq;
  ew.gu_s = gs;
  ew.d_q = dq;
  ew.d_s = ds;
  ew.ok = true;
  return MOE_OK;
}

// The tensor-core path's shared-expert weights: bf16 copies in the dense
// pass's 128-row tiles (gate/up pairs for FC1, rows for FC2), and the
// driver's tensor-map encoder for x.
int setup_dense(moe_layer* L) {
  const moe_dims_t& d = L->dims;
  const size_t gu = (size_t)2 * d.f_shared * d.d * 2, dn = (size_t)d.d * d.f_shared * 2;
  const size_t rt = (size_t)(d.n_experts + 127) / 128 * 128 * d.d * 2;
  if (cudaMalloc(&L->sh_owned, gu + dn + rt) != cudaSuccess) {
    cudaGetLastError();
    L->sh_owned = nullptr;
    return MOE_ERR_ALLOC;
  }
  L->sh_gu_umma = static_cast<uint8_t*>(L->sh_owned);
  L->sh_d_umma = L->sh_gu_umma + gu;
  L->router_umma = L->sh_d_umma + dn;
  MOE_CUDA(cudaMemset(L->router_umma, 0, rt));
  dense_relayout_kernel<<<L->n_sm * 8, 256>>>(static_cast<const uint16_t*>(L->w.router_w),
                                               (int64_t)d.n_experts, d.d, 0, L->router_umma);
  MOE_CUDA(cudaGetLastError());
  dense_relayout_kernel<<<L->n_sm * 8, 256>>>(static_cast<const uint16_t*>(L->w.shared_gu),
                                               2LL * d.f_shared, d.d, 1, L->sh_gu_umma);
  MOE_CUDA(cudaGetLastError());
  dense_relayout_kernel<<<L->n_sm * 8, 256>>>(static_cast<const uint16_t*>(L->w.shared_d),
                                               (int64_t)d.d, d.f_shared, 0, L->sh_d_umma);
  MOE_CUDA(cudaGetLastError());
  MOE_CUDA(cudaStreamSynchronize(nullptr));
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  void* fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn) {
    cudaGetLastError();
    return MOE_ERR_UNSUPPORTED;
  }
  L->encode_tiled = fn;
  return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_status_string(int s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported (use another implementation)";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_ALLOC: return "allocation failed";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

int moe_last_cuda_error(void) { return g_last_cuda_error.load(); }

int moe_layer_create(const moe_dims_t* dims, const moe_weights_t* weights, moe_layer_t* out) {
  if (!dims || !weights || !out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  int rc = validate_dims(*dims);
  if (rc) return rc;
  const moe_weights_t& w = *weights;
  const void* ptrs[] = {w.router_w, w.router_bias, w.w_gu_q, w.w_gu_s, w.w_d_q,
                        w.w_d_s,    w.shared_gu,   w.shared_d, w.rms_gamma};
  for (const void* p : ptrs) {
    if (!p) return MOE_ERR_INVALID_ARG;
    if (!aligned16(p)) return MOE_ERR_UNSUPPORTED;
  }
  int dev = 0;
  MOE_CUDA(cudaGetDevice(&dev));
  cudaDeviceProp prop;
  MOE_CUDA(cudaGetDeviceProperties(&prop, dev));
  if (prop.major != 10 || prop.minor != 3) return MOE_ERR_UNSUPPORTED;

  moe_layer* L = new (std::nothrow) moe_layer();
  if (!L) return MOE_ERR_ALLOC;
  L->dims = *dims;
  L->w = w;
  L->device = dev;
  L->n_sm = prop.multiProcessorCount;
  L->smem_optin = (int)prop.sharedMemPerBlockOptin;
  const size_t f = dims->f, dd = dims->d;
  L->q_gu_stride = 2 * f * dd / 2;
  L->s_gu_stride = 2 * f * dd / 32;
  L->q_d_stride = dd * f / 2;
  L->s_d_stride = dd * f / 32;
  const size_t bytes = workspace_bytes(*dims, nullptr, nullptr);
  if (cudaMalloc(&L->ws_base, bytes) != cudaSuccess) {
    cudaGetLastError();
    delete L;
    return MOE_ERR_ALLOC;
  }
  workspace_bytes(*dims, &L->ws, static_cast<char*>(L->ws_base));
  auto fail = [&](cudaError_t e) {
    moe_layer_destroy(L);
    return cuda_fail(e);
  };
  cudaError_t e;
  if ((e = cudaMemset(L->ws_base, 0, bytes)) != cudaSuccess) return fail(e);
  for (int i = 0; i < kNumTimeEvents; ++i)
    if ((e = cudaEventCreate(&L->ev_time[i])) != cudaSuccess) return fail(e);
  // the expert paths kept (both by default, see kTcMinBatch) fix the layouts
  // the kernels read; a layer that only ever sees one row keeps one
  int path = (dims->expert_path == kPathAuto && dims->max_batch == 1) ? kPathMmaSync
                                                                      : dims->expert_path;
  if (path != kPathTc) {
    // a shape whose stage rings the mma.sync kernels cannot fit leaves an
    // automatic layer to the tensor-core path alone
    rc = plan_mma(L);
    if (rc == MOE_ERR_UNSUPPORTED && dims->expert_path == kPathAuto) {
      path = kPathTc;
    } else if (rc) {
      moe_layer_destroy(L);
      return rc;
    }
  }
  if (path != kPathTc && (rc = setup_weights(L, w, 1, L->wm))) {
    moe_layer_destroy(L);
    return rc;
  }
  if (path != kPathMmaSync &&
      ((rc = setup_weights(L, w, 3, L->wt)) || (rc = setup_dense(L)))) {
    moe_layer_destroy(L);
    return rc;
  }
  L->tc_min_batch = path == kPathTc ? 1 : kTcMinBatch;
  if ((rc = plan_all(L))) {
    moe_layer_destroy(L);
    return rc;
  }
  *out = L;
  return MOE_OK;
}

int moe_layer_destroy(moe_layer_t L) {
  if (!L) return MOE_OK;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(L->device);
  cudaDeviceSynchronize();
  if (L->hg.exec) cudaGraphExecDestroy(L->hg.exec);
  for (int i = 0; i < kNumTimeEvents; ++i)
    if (L->ev_time[i]) cudaEventDestroy(L->ev_time[i]);
  if (L->ws_base) cudaFree(L->ws_base);
  if (L->wm.owned) cudaFree(L->wm.owned);
  if (L->wt.owned) cudaFree(L->wt.owned);
  if (L->sh_owned) cudaFree(L->sh_owned);
  cudaSetDevice(prev);
  delete L;
  return MOE_OK;
}

int moe_router_topk(moe_layer_t L, void* stream, const void* x, int B, int32_t* idx, float* w) {
  int rc = check_forward_args(L, x, B);
  if (rc) return rc;
  if (!idx || !w) return MOE_ERR_INVALID_ARG;
  return launch_router(L, static_cast<cudaStream_t>(stream), x, B, idx, w);
}

int moe_decode_forward(moe_layer_t L, void* stream, const void* x, int B, void* residual,
                       void* out) {
  return forward_impl(L, static_cast<cudaStream_t>(stream), x, B, residual, out, nullptr, nullptr,
                      nullptr, nullptr, nullptr);
}

int moe_decode_forward_debug(moe_layer_t L, void* stream, const void* x, int B, void* residual,
                             void* out, float* y_routed, float* y_shared, float* h, float* z,
                             float* out_f32) {
  return forward_impl(L, static_cast<cudaStream_t>(stream), x, B, residual, out, y_routed,
                      y_shared, h, z, out_f32);
}

namespace {

// The host-buffer forward's work on `st`: the two input copies into the
// workspace staging buffers, the forward, the two output copies.
int enqueue_forward_host(moe_layer* L, cudaStream_t st, const void* x_host, int B,
                         void* residual_host, void* out_host) {
  const size_t bytes = (size_t)B * L->dims.d * 2;
  MOE_CUDA(cudaMemcpyAsync(L->ws.x_stage, x_host, bytes, cudaMemcpyHostToDevice, st));
  MOE_CUDA(cudaMemcpyAsync(L->ws.res_stage, residual_host, bytes, cudaMemcpyHostToDevice, st));
  int rc = forward_impl(L, st, L->ws.x_stage, B, L->ws.res_stage, L->ws.out_stage, nullptr,
                        nullptr, nullptr, nullptr, nullptr);
  if (rc) return rc;
  MOE_CUDA(cudaMemcpyAsync(residual_host, L->ws.res_stage, bytes, cudaMemcpyDeviceToHost, st));
  MOE_CUDA(cudaMemcpyAsync(out_host, L->ws.out_stage, bytes, cudaMemcpyDeviceToHost, st));
  return MOE_OK;
}

bool pinned(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

}  // namespace

int moe_decode_forward_host(moe_layer_t L, void* stream, const void* x_host, int B,
                            void* residual_host, void* out_host) {
  if (!L || !x_host || !residual_host || !out_host) return MOE_ERR_INVALID_ARG;
  if (B < 1 || B > L->dims.max_batch) return MOE_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Pinned buffers on a stream of the caller's: one CUDA graph of the copies
  // and the kernels, captured on first use and replayed while the arguments
  // (and the layer's timing, trace, prefetch and test-hook settings) stay the
  // same, so a call costs one graph launch and the sync instead of nine
  // enqueues.  Otherwise (the legacy default stream, pageable memory) the
  // same work is enqueued call by call.
  if (st == nullptr || !pinned(x_host) || !pinned(residual_host) || !pinned(out_host)) {
    int rc = enqueue_forward_host(L, st, x_host, B, residual_host, out_host);
    if (rc) return rc;
    MOE_CUDA(cudaStreamSynchronize(st));
    return MOE_OK;
  }
  moe_layer::HostGraph& g = L->hg;
  const bool same = g.exec && g.stream == st && g.x == x_host && g.res == residual_host &&
                    g.out == out_host && g.B == B && g.timing == L->timing &&
                    g.tracing == L->tracing && g.next == L->next && g.fault == L->debug_fault &&
                    g.fault_ns == L->debug_wait_ns;
  if (!same) {
    if (g.exec) {
      MOE_CUDA(cudaGraphExecDestroy(g.exec));
      g.exec = nullptr;
    }
    MOE_CUDA(cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal));
    const int rc = enqueue_forward_host(L, st, x_host, B, residual_host, out_host);
    cudaGraph_t graph = nullptr;
    const cudaError_t ec = cudaStreamEndCapture(st, &graph);
    if (rc) {
      if (graph) cudaGraphDestroy(graph);
      return rc;
    }
    MOE_CUDA(ec);
    const cudaError_t ei = cudaGraphInstantiate(&g.exec, graph, 0);
    cudaGraphDestroy(graph);
    MOE_CUDA(ei);
    g.stream = st;
    g.x = x_host;
    g.res = residual_host;
    g.out = out_host;
    g.B = B;
    g.timing = L->timing;
    g.tracing = L->tracing;
    g.next = L->next;
    g.fault = L->debug_fault;
    g.fault_ns = L->debug_wait_ns;
  }
  MOE_CUDA(cudaGraphLaunch(g.exec, st));
  MOE_CUDA(cudaStreamSynchronize(st));
  return MOE_OK;
}

int moe_debug_dequant(moe_layer_t L, void* stream, int expert, int which, float* out) {
  if (!L || !out || expert < 0 || expert >= L->dims.n_experts || (which != 0 && which != 1))
    return MOE_ERR_INVALID_ARG;
  const int64_t rows = which == 0 ? 2LL * L->dims.f : L->dims.d;
  const int64_t k = which == 0 ? L->dims.d : L->dims.f;
  const ExpertWeights& ew = L->wt.ok ? L->wt : L->wm;
  const uint8_t* q = (which == 0 ? ew.gu_q : ew.d_q) +
                     (size_t)expert * (which == 0 ? L->q_gu_stride : L->q_d_stride);
  const uint8_t* s = (which == 0 ? ew.gu_s : ew.d_s) +
                     (size_t)expert * (which == 0 ? L->s_gu_stride : L->s_d_stride);
  const int layout = which == 0 ? ew.layout_gu : ew.layout_d;
  const int64_t blocks = std::min<int64_t>((rows * (k / 32) + 255) / 256, 4096);
  mxfp4_dequant_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      q, s, rows, k, layout, out);
  MOE_CUDA(cudaGetLastError());
  return MOE_OK;
}

int moe_set_act_format(moe_layer_t L, int fmt) {
  if (!L || fmt < 0 || fmt > 1) return MOE_ERR_INVALID_ARG;
  L->act_fmt = fmt;
  return MOE_OK;
}

int moe_set_prefetch_next(moe_layer_t L, moe_layer_t next) {
  if (!L) return MOE_ERR_INVALID_ARG;
  if (next && next->device != L->device) return MOE_ERR_INVALID_ARG;
  L->next = next;
  return MOE_OK;
}

int moe_layer_status(moe_layer_t L, int* device_status) {
  if (!L || !device_status) return MOE_ERR_INVALID_ARG;
  MOE_CUDA(cudaDeviceSynchronize());
  int v = 0;
  MOE_CUDA(cudaMemcpy(&v, L->ws.status, sizeof(int), cudaMemcpyDeviceToHost));
  MOE_CUDA(cudaMemset(L->ws.status, 0, sizeof(int)));
  *device_status = v;
  return MOE_OK;
}

int moe_debug_set_fault(moe_layer_t L, int fault, unsigned long long wait_ns) {
  if (!L || fault < 0 || fault > 1) return MOE_ERR_INVALID_ARG;
  L->debug_fault = fault;
  L->debug_wait_ns = fault ? wait_ns : 0;
  return MOE_OK;
}

int moe_set_timing(moe_layer_t L, int enable) {
  if (!L) return MOE_ERR_INVALID_ARG;
  L->timing = enable != 0;
  L->timed_once = false;
  return MOE_OK;
}

int moe_get_timing(moe_layer_t L, float* us, int n) {
  if (!L || !us || n < 0) return MOE_ERR_INVALID_ARG;
  if (!L->timed_once) return MOE_ERR_INVALID_ARG;
  MOE_CUDA(cudaEventSynchronize(L->ev_time[kTimeTailEnd]));
  float t[6];
  MOE_CUDA(cudaEventElapsedTime(&t[0], L->ev_time[kTimeRouterStart], L->ev_time[kTimeRouterEnd]));
  MOE_CUDA(cudaEventElapsedTime(&t[1], L->ev_time[kTimeRouterEnd], L->ev_time[kTimeFc1End]));
  MOE_CUDA(cudaEventElapsedTime(&t[2], L->ev_time[kTimeFc1End], L->ev_time[kTimeFc2End]));
  t[3] = 0.f;   // the shared expert streams inside FC1 and FC2
  MOE_CUDA(cudaEventElapsedTime(&t[4], L->ev_time[kTimeFc2End], L->ev_time[kTimeTailEnd]));
  MOE_CUDA(cudaEventElapsedTime(&t[5], L->ev_time[kTimeRouterStart], L->ev_time[kTimeTailEnd]));
  for (int i = 0; i < n && i < 6; ++i) us[i] = t[i] * 1000.f;
  return MOE_OK;
}

int moe_set_trace(moe_layer_t L, int enable) {
  if (!L) return MOE_ERR_INVALID_ARG;
  L->tracing = enable != 0;
  return MOE_OK;
}

int moe_get_trace(moe_layer_t L, unsigned long long* ns, int n) {
  if (!L || !ns || n < 0) return MOE_ERR_INVALID_ARG;
  unsigned long long t[kTraceSlots];
  MOE_CUDA(cudaDeviceSynchronize());
  MOE_CUDA(cudaMemcpy(t, L->ws.trace, sizeof(t), cudaMemcpyDeviceToHost));
  for (int i = 0; i < n && i < 10; ++i) ns[i] = (i % 2 == 0) ? t[i / 2] : t[8 + i / 2];
  return MOE_OK;
}

int moe_launches_per_forward(moe_layer_t L, int B) {
  if (!L || B < 1 || B > L->dims.max_batch) return -1;
  // router, top-k, FC1 (shared + routed), FC2 (shared + routed), tail; one
  // row on the mma.sync path takes FC1 and FC2 in one launch
  return (B == 1 && !use_tc(L, B)) ? 4 : 5;
}

size_t mxfp4_packed_bytes(int64_t rows, int64_t k, int layout, size_t* scale_bytes) {
  if (!mx_layout_ok(rows, k, layout)) return 0;
  if (scale_bytes) *scale_bytes = (size_t)(rows * (k / 32));
  return (size_t)(rows * (k / 2));
}

int mxfp4_pack(const float* w, int64_t rows, int64_t k, uint8_t* q, uint8_t* s, int layout) {
  if (!w || !q || !s || rows < 0 || k <= 0 || k % 32 != 0) return MOE_ERR_INVALID_ARG;
  if (!mx_layout_ok(rows, k, layout)) return MOE_ERR_UNSUPPORTED;
  const int64_t nb = k / 32;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < nb; ++b) {
      uint8_t qb[16];
      const uint8_t sb = mx_pack_block(w + r * k + b * 32, qb);
      mx_store_block(q, s, r, b, rows, k, layout, qb, sb);
    }
  return MOE_OK;
}

int mxfp4_pack_device(void* stream, const float* w, int64_t rows, int64_t k, uint8_t* q,
                      uint8_t* s, int layout) {
  if (!w || !q || !s || rows < 0 || k <= 0 || k % 32 != 0) return MOE_ERR_INVALID_ARG;
  if (!mx_layout_ok(rows, k, layout)) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(w) || !aligned16(q)) return MOE_ERR_UNSUPPORTED;
  const int64_t total = rows * (k / 32);
  if (total == 0) return MOE_OK;
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, 152 * 32);
  mxfp4_pack_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(w, rows, k, q,
                                                                                     s, layout);
  MOE_CUDA(cudaGetLastError());
  return MOE_OK;
}

int mxfp4_repack(const uint8_t* q_in, const uint8_t* s_in, int64_t rows, int64_t k, int from,
                 int to, uint8_t* q_out, uint8_t* s_out) {
  if (!q_in || !s_in || !q_out || !s_out || rows < 0 || k <= 0) return MOE_ERR_INVALID_ARG;
  if (!mx_layout_ok(rows, k, from) || !mx_layout_ok(rows, k, to)) return MOE_ERR_UNSUPPORTED;
  const int64_t nb = k / 32;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < nb; ++b) {
      uint8_t qb[16];
      const uint8_t sb = mx_load_block(q_in, s_in, r, b, rows, k, from, qb);
      mx_store_block(q_out, s_out, r, b, rows, k, to, qb, sb);
    }
  return MOE_OK;
}

int mxfp4_retile_device(void* stream, const uint8_t* q_in, const uint8_t* s_in, int64_t n_mat,
                        int64_t rows, int64_t k, int layout, uint8_t* q_out, uint8_t* s_out) {
  if (!q_in || !s_in || !q_out || !s_out || n_mat < 0 || rows < 0 || k <= 0)
    return MOE_ERR_INVALID_ARG;
  if (layout == kMxCanonical || !mx_layout_ok(rows, k, layout)) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(q_in) || !aligned16(q_out)) return MOE_ERR_UNSUPPORTED;
  const int64_t qb = rows * (k / 2), sb = rows * (k / 32);
  const int64_t total = rows * (k / 32);
  if (total == 0) return MOE_OK;
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, 152 * 32);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  for (int64_t m = 0; m < n_mat; ++m) {
    mxfp4_retile_kernel<<<(unsigned)blocks, 256, 0, st>>>(q_in + m * qb, s_in + m * sb, rows, k,
                                                         q_out + m * qb, s_out + m * sb, layout);
    MOE_CUDA(cudaGetLastError());
  }
  return MOE_OK;
}

}  // extern "C"
