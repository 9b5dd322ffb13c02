// The front of the layer for one row (B = 1) in a single launch: router GEMV,
// top-k, shared-expert gate/up and routed gate/up ("Kimi K3 on GB300: 13
// kernels a layer...", section "What the fused path changes": the MoE front
// fused into one kernel that starts early, and one persistent routed-expert
// kernel; section "Why batch 1 on a rack is not only a bandwidth problem":
// short, dependent steps leave HBM idle).
//
// Three steps share one stage ring (stream.cuh):
//   R  router rows (bf16) -> logits [E] in global memory
//   A  shared gate/up (bf16) -> h_s, SwiGLU
//   B  routed gate/up (MXFP4, mma.sync) -> h, SwiGLU
// After R every CTA's consumers make their logits visible and count the CTA in
// (one atomic per CTA), stage the routed step's x operand, consume the first
// of their A items (the other CTAs finish their router rows meanwhile), then
//   - wait, bounded, until all CTAs have counted in,
//   - select the row's experts themselves from all E logits, with the same
//     keys, order and weights as topk_kernel, into routing tables in shared
//     memory (k experts, one pair each, ordered by expert id),
// and consume the rest of A; CTA 0 also writes the tables to global memory
// for FC2 and the tail and raises the route flag.  The producer streams R and
// A without waiting for anything and learns the routing from a shared-memory
// barrier before B, so the selection runs while A's stages stream in, and
// the routed step reads no table from global memory.  Until B the producer
// keeps only a few stages in flight (the host sets R's and A's lag): every
// step of the chain above is a dependent round trip to L2, and a memory
// queue of whole stage rings from every SM would make each one wait
// microseconds behind the stream.  The counter and the flag are zeroed again
// by the tail kernel of the same forward.
#pragma once

#include "common.cuh"
#include "stream.cuh"
#include "topk.cuh"

namespace moe {

struct FrontArgs {
  const float* bias;      // [E], a static weight
  int E, k;
  float routed_scale;
  unsigned* count;        // CTAs past the router step (zero at rest)
  unsigned* route_flag;   // raised by CTA 0 once the global tables are written (zero at rest)
  int32_t* topk_idx;      // [k], descending by biased score
  float* topk_w;          // [k]
  int* n_active;          // global routing tables (as topk_kernel writes them)
  int* active_expert;
  int* active_off;
  int* pair_list;
  // failure-detection test hook: CTA skip_arrive_cta (-1: none) does not
  // count itself in, so every CTA's wait for the count expires after wait_ns
  unsigned long long wait_ns;
  int skip_arrive_cta;
};

// Routing tables of one row in shared memory, and the barrier the producer
// waits on for them.
struct FrontRoute {
  uint64_t bar;
  int n_active;
  int expert[32];
  int off[33];
  int pair[32];
  int xshift;   // the routed step's x operand is x * 2^-xshift in f16
};
constexpr int kFrontRouteBytes = (int)((sizeof(FrontRoute) + 127) / 128 * 128);
// After the routing tables: the routed step's x operand, f16, 16 bytes per
// 8 elements (2 K bytes for a row of K).
__host__ __device__ inline int front_extra_bytes(int K) { return kFrontRouteBytes + 2 * K; }

// 32-expert chunks per consumer warp in the selection (E <= 32 * 4 * KW).
constexpr int kFrontMaxChunks = 4;
// Shared memory the selection borrows from the cross-slab partial buffers
// (idle between steps): 2 x 16 sorted lists of 32 keys, then E <= 1024 scores.
constexpr int kFrontScratchBytes = 2 * 16 * 32 * 8 + 1024 * 4;

__device__ __forceinline__ FrontRoute* front_route(float* red, int red_pp) {
  return reinterpret_cast<FrontRoute*>(reinterpret_cast<uint8_t*>(red + 2 * (size_t)red_pp) + 64);
}

// Wait until *c >= target (acquire), at most limit_ns.
__device__ __forceinline__ void wait_count(const unsigned* c, unsigned target, int* status,
                                           unsigned long long limit_ns) {
  if (ld_acquire_u32(c) >= target) return;
  const unsigned long long t0 = global_ns();
  while (ld_acquire_u32(c) < target) {
    if (global_ns() - t0 > limit_ns) {
      if (status) atomicExch(status, kStatusTimeout);
      return;
    }
  }
}

#ifndef MOE_FRONT_COMPACT
#define MOE_FRONT_COMPACT 0
#endif

// The bitonic sort of 32 keys as two loops (a few hundred bytes of code
// instead of the unrolled network's several KB).
__device__ __forceinline__ uint64_t warp_sort_desc_loop(uint64_t key, int lane) {
#pragma unroll 1
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll 1
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint64_t ok = __shfl_xor_sync(0xffffffffu, key, stride);
      const bool desc = (lane & size) == 0 || size == 32;
      const bool lower = (lane & stride) == 0;
      const bool take = (lower == desc) ? (ok > key) : (ok < key);
      if (take) key = ok;
    }
  }
  return key;
}

// Selection of one row by the KW consumer warps.  Warp w sorts the 32-expert
// chunks w, w + KW, ... and merges them into one sorted list of its 32 best
// keys; the KW lists then meet in a tournament through shared memory, a round
// per consumer barrier.  Warp 0 turns the winning k keys into the tables.
// publish = false: tables in shared memory only (CTA 0 writes no global
// tables and raises no flag).
__device__ __forceinline__ void front_topk(const FrontArgs& f, const float* logits, float* scratch,
                                           FrontRoute* rt, const float (&bias)[kFrontMaxChunks],
                                           int kw, int KW, int lane, int cthreads, bool publish) {
  uint64_t* lists = reinterpret_cast<uint64_t*>(scratch);   // [2][16][32]
  float* s_sc = scratch + 2 * 16 * 32 * 2;                   // [E]
  const int nch = (f.E + 31) >> 5;
  float l[kFrontMaxChunks];
#pragma unroll
  for (int i = 0; i < kFrontMaxChunks; ++i) {   // every logit load before the first use
    const int t = (kw + i * KW) * 32 + lane;
    l[i] = t < f.E ? __ldcg(logits + t) : 0.f;
  }
  uint64_t best = 0ull;
#if MOE_FRONT_COMPACT
#pragma unroll 1
#else
#pragma unroll
#endif
  for (int i = 0; i < kFrontMaxChunks; ++i) {
    const int ch = kw + i * KW;
    if (ch < nch) {   // warp-uniform
      const int t = ch * 32 + lane;
      uint64_t key = 0ull;
      if (t < f.E) {
        const float li = i == 0 ? l[0] : i == 1 ? l[1] : i == 2 ? l[2] : l[3];
        const float bi = i == 0 ? bias[0] : i == 1 ? bias[1] : i == 2 ? bias[2] : bias[3];
        const float s = topk_score(li);
        s_sc[t] = s;
        key = topk_key(s, bi, t);
      }
#if MOE_FRONT_COMPACT
      key = warp_sort_desc_loop(key, lane);
#else
      key = warp_bitonic_sort_desc(key, lane);
#endif
      if (i == 0) {
        best = key;
      } else {
        // the elementwise maximum of one sorted list and the other reversed
        // is a bitonic sequence holding the 32 largest keys of both
        const uint64_t y = __shfl_sync(0xffffffffu, key, 31 - lane);
        best = warp_bitonic_merge_desc(best > y ? best : y, lane);
      }
    }
  }
  if (kw < 16) lists[kw * 32 + lane] = best;
  consumer_sync(cthreads);
  int n = min(KW, 16), src = 0;
  while (n > 1) {
    const int half = n >> 1;
    const uint64_t* s = lists + src * 512;
    uint64_t* d = lists + (src ^ 1) * 512;
    if (kw < half) {
      const uint64_t x = s[(2 * kw) * 32 + lane];
      const uint64_t y = s[(2 * kw + 1) * 32 + 31 - lane];
      d[kw * 32 + lane] = warp_bitonic_merge_desc(x > y ? x : y, lane);
    } else if (kw == half && (n & 1)) {
      d[kw * 32 + lane] = s[(n - 1) * 32 + lane];
    }
    n = half + (n & 1);
    src ^= 1;
    consumer_sync(cthreads);
  }
  if (kw != 0) return;
  const int k = f.k;
  const int e = min(max(topk_key_expert(lists[src * 512 + lane]), 0), f.E - 1);
  const float s = lane < k ? s_sc[e] : 0.f;
  float ssum = 0.f;
  for (int i = 0; i < k; ++i) ssum += __shfl_sync(0xffffffffu, s, i);   // in rank order
  const float w = f.routed_scale * s / ssum;
  int slot = 0;   // rank of e among the selected ids: the tables go by expert id
  for (int i = 0; i < k; ++i) slot += __shfl_sync(0xffffffffu, e, i) < e ? 1 : 0;
  if (lane < k) {
    rt->expert[slot] = e;
    rt->pair[slot] = lane;
    rt->off[lane] = lane;
  }
  if (lane == 0) {
    rt->n_active = k;
    rt->off[k] = k;
  }
  if (publish && blockIdx.x == 0) {
    if (lane < k) {
      f.topk_idx[lane] = e;
      f.topk_w[lane] = w;
      f.active_expert[slot] = e;
      f.pair_list[slot] = lane;
      f.active_off[lane] = lane;
    }
    if (lane == 0) {
      *f.n_active = k;
      f.active_off[k] = k;
    }
    __threadfence();
    __syncwarp();
    if (lane == 0) st_release_u32(f.route_flag, 1u);
  }
}

// The routed step's x operand in shared memory (XS steps of stream.cuh): the
// row's max |x| picks the power-of-two scale that keeps f16 in range, then
// entry i holds elements 8i..8i+7 as f16 pairs (entry 4 b + t: block b, lane
// quad t).  scratch: KW words.
__device__ __forceinline__ void front_x_operand(const uint16_t* x, int K, uint4* xs, int* xshift,
                                                unsigned* scratch, int kw, int KW, int lane,
                                                int ct, int cthreads) {
  const uint4* xr = reinterpret_cast<const uint4*>(x);
  uint32_t mx = 0;
  for (int i = ct; i < K / 8; i += cthreads) {
    const uint4 v = xr[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) mx = max(mx, max(w[j] & 0x7FFFu, (w[j] >> 16) & 0x7FFFu));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) scratch[kw] = mx;
  consumer_sync(cthreads);
  uint32_t amax = 0;
  for (int w = 0; w < KW; ++w) amax = max(amax, scratch[w]);
  const int shift = f16_shift_for_amax(bf16_bits_to_f32(amax));
  const float sc = pow2f(-shift);
  if (ct == 0) *xshift = shift;
  for (int i = ct; i < K / 8; i += cthreads) {
    const uint4 v = xr[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint4 o;
    o.x = pack_f16x2(__uint_as_float(w[0] << 16) * sc, __uint_as_float(w[0] & 0xFFFF0000u) * sc);
    o.y = pack_f16x2(__uint_as_float(w[1] << 16) * sc, __uint_as_float(w[1] & 0xFFFF0000u) * sc);
    o.z = pack_f16x2(__uint_as_float(w[2] << 16) * sc, __uint_as_float(w[2] & 0xFFFF0000u) * sc);
    o.w = pack_f16x2(__uint_as_float(w[3] << 16) * sc, __uint_as_float(w[3] & 0xFFFF0000u) * sc);
    xs[i] = o;
  }
}

// Warp 0 lane 0 produces; warps 1..KW consume (KW = blockDim.x / 32 - 1).
// Dynamic shared memory: the streaming kernels' carve-up (stream_smem_init)
// followed by front_extra_bytes(K) for the routing tables and the routed
// step's x operand; the cross-slab partial buffers must hold
// kFrontScratchBytes.
template <class RC, class AC, class BC>
__global__ void __launch_bounds__(32 * (kMmaWarps + 1), 1)
    stream_front_kernel(const StreamArgs ar, const StreamArgs a0, const StreamArgs a1,
                        const FrontArgs f) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KW = (int)(blockDim.x >> 5) - 1;
  trace_begin(a0.trace, a0.trace_id);
  float* red = reinterpret_cast<float*>(smem + (size_t)a0.NS * a0.stage_bytes + (size_t)a0.NS * 16);
  FrontRoute* rt = front_route(red, a0.red_pp);
  if (threadIdx.x == 0) mbar_init(&rt->bar, 1);   // fenced and synced by stream_smem_init
  const StreamSmem m = stream_smem_init(smem, a0.NS, a0.stage_bytes, a0.red_pp, KW);
  pdl_launch_dependents();
  // the routed step reads its tables from this CTA's shared memory
  uint4* xs = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(rt) + kFrontRouteBytes);
  StreamArgs b = a1;
  b.n_active = &rt->n_active;
  b.active_expert = rt->expert;
  b.active_off = rt->off;
  b.pair_list = rt->pair;
  b.xs = xs;
  b.xs_shift = &rt->xshift;
  SegPrior pr;
  cfg_add_prior<RC>(ar, pr);
  cfg_add_prior<AC>(a0, pr);
  uint32_t stage = 0;
  if (warp == 0) {
    if (lane == 0) {
      // router and shared weights are static: no wait before streaming them
      cfg_produce<RC>(ar, SegPrior(), m.stages, m.full, m.empty, stage);
      cfg_produce<AC>(a0, SegPrior(), m.stages, m.full, m.empty, stage);
      mbar_wait(&rt->bar, 0, a0.status);
      cfg_produce<BC>(b, pr, m.stages, m.full, m.empty, stage);
      stream_drain(a0, m.empty, stage);
    }
    __syncwarp();
  } else {
    const int kw = warp - 1, ct = (int)threadIdx.x - 32, cthreads = 32 * KW;
    float bias[kFrontMaxChunks];
#pragma unroll
    for (int i = 0; i < kFrontMaxChunks; ++i) {
      const int t = (kw + i * KW) * 32 + lane;
      bias[i] = t < f.E ? __ldg(f.bias + t) : 0.f;
    }
    pdl_wait_prerequisites();   // x may be the previous kernel's output
    int pp = 0, rp = 0;
    cfg_consume<RC>(ar, SegPrior(), m.stages, m.full, m.empty, m.red, stage, pp, rp, kw, KW, lane);
    // count this CTA in once its logits are visible GPU-wide (the barrier
    // orders every consumer's stores before the arriving thread's fence)
    consumer_sync(cthreads);
    if (ct == 0 && (int)blockIdx.x != f.skip_arrive_cta) {
      __threadfence();
      atomicAdd(f.count, 1u);
    }
    // while the other CTAs finish their router rows: the routed step's x
    // operand and the first of this CTA's shared gate/up items
    front_x_operand(b.x, b.K, xs, &rt->xshift, reinterpret_cast<unsigned*>(m.red), kw, KW, lane,
                    ct, cthreads);
    consumer_sync(cthreads);
    cfg_consume<AC>(a0, SegPrior(), m.stages, m.full, m.empty, m.red, stage, pp, rp, kw, KW, lane,
                    0, 1);
    if (ct == 0) wait_count(f.count, gridDim.x, a0.status, f.wait_ns);
    consumer_sync(cthreads);
    front_topk(f, ar.out, m.red, rt, bias, kw, KW, lane, cthreads, true);
    consumer_sync(cthreads);
    if (ct == 0) mbar_arrive(&rt->bar);
    cfg_consume<AC>(a0, SegPrior(), m.stages, m.full, m.empty, m.red, stage, pp, rp, kw, KW, lane,
                    1, 1);
    cfg_consume<BC>(b, pr, m.stages, m.full, m.empty, m.red, stage, pp, rp, kw, KW, lane);
  }
  trace_end(a0.trace, a0.trace_id);
}

}  // namespace moe
