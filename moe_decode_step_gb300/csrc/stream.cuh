// Persistent streaming GEMV: one producer thread feeds a ring of shared-memory
// stages with bulk copies (cp.async.bulk + mbarrier); consumer warps compute
// from shared memory.
//
// It serves every weight-streaming step of the layer:
//   routed FC1   MXFP4 gate/up rows x x (bf16 -> f16), SwiGLU epilogue
//   routed FC2   MXFP4 down rows x h (fp32 -> f16)
//   router GEMV  bf16 rows x x (bf16)
//   shared FC1   bf16 gate/up rows x x, SwiGLU epilogue
//   shared FC2   bf16 down rows x h_s (fp32)
// ("Kimi K3 on GB300: 13 kernels a layer...", section "What the fused path
// changes": one persistent routed-expert kernel doing FC1 and FC2; section
// "Why batch 1 on a rack is not only a bandwidth problem": decode GEMVs are
// bound by HBM.)
//
// Work: an item is RW consecutive output rows (row pairs for gate/up) of one
// matrix; for routed steps the matrix is an active expert and the activation
// rows are that expert's (row, slot) pairs, taken R <= RMAX at a time.  CTA c
// owns a contiguous range of items, so the producer knows its whole sequence
// and runs ahead across item boundaries; the only coupling is the stage ring.
// Consumer warps split K (warp w owns a K slab), then combine their partial
// sums through shared memory in a fixed order (deterministic).
//
// Two consumer formulations:
//  * bf16 weights (router, shared expert): every lane owns a run of K
//    elements and keeps one fp32 partial per row; a butterfly reduce-scatter
//    then folds the lanes.
//  * MXFP4 weights (routed experts): the tensor cores (mma.sync m16n8k16,
//    f16 x f16 -> fp32) take the products, 16 weight rows by up to 8
//    activation rows per instruction.  Dequantising a nibble pair is one
//    cvt.rn.f16x2.e2m1x2; the per-row, per-block E8M0 scale is applied to the
//    fp32 result of the block's two MMAs.  Doing the products on the CUDA
//    cores instead costs about two issue slots per weight, which at 0.53
//    bytes per weight is more than an SM can issue at HBM speed.
#pragma once

#include "common.cuh"
#include "planes.cuh"

namespace moe {

enum { kWfMx = 0, kWfBf16 = 1 };

// Consumer warps of the MXFP4 (tensor-core) steps.
constexpr int kMmaWarps = 15;

struct StreamArgs {
  const uint8_t* q;          // MXFP4 nibbles (or bf16 weights) of matrix 0
  const uint8_t* s;          // MXFP4 scale bytes of matrix 0 (unused for bf16)
  size_t q_stride, s_stride; // bytes between experts (routed)
  int K;                     // row length in elements
  int N;                     // output rows (gate/up: row pairs, up row = N + i)
  int k;                     // top-k: pair p belongs to activation row p / k (routed)
  int B;                     // dense steps: activation rows
  const uint16_t* x;         // bf16 activations [rows][K]
  const float* h;            // fp32 activations [rows][K]
  const unsigned* h_amax;    // max |h| bits per row (MXFP4 h-activation steps)
  float* out;                // [rows][N]
  unsigned* out_amax;        // max |out| bits per row (routed FC1), or null
  const int* n_active;       // routing tables (routed steps)
  const int* active_expert;
  const int* active_off;
  const int* pair_list;
  int* status;               // device status word (bounded-wait timeouts)
  int NS;                    // stage buffers in the ring
  int stage_bytes;           // bytes per stage buffer (multiple of 128)
  int red_pp;                // floats per cross-slab partial buffer (two of them)
  int kc;                    // MXFP4 steps: K chunks (stages) per tile group
  unsigned long long* trace; // optional kernel trace (see trace_begin), or null
  int trace_id;
  uint8_t* xq;               // router only: activation planes of x [B][4K] (planes.cuh), or null
  uint8_t* xq_code;          // and their plane-0 codes, one per row [B]
  int xq_f8;                 // 1: the planes hold x's MXFP8 rounding (mxfp8_round8)
  // routed gate/up steps of one activation row whose operand sits in shared
  // memory (StreamCfg XS): per K block b and lane quad t, the f16 pairs of
  // elements 8t..8t+7 at xs[4 b + t], scaled by 2^-(*xs_shift)
  const uint4* xs;
  const int* xs_shift;
  // the one-row expert kernel (stream_expert_kernel): its two grid-wide
  // counters, and the limit of its wait before FC2's routed segment (0: the
  // default limit)
  unsigned* done_count;
  unsigned long long wait_ns;
};

// Lane layout of the bf16 steps: a lane owns NQ chunks of CW consecutive K
// elements, chunk q at slab + q*32*CW + lane*CW, so a warp covers WARP_K =
// 32*CW*NQ elements (narrow chunks spread a short K over more warps).
template <bool ACTH, int CW, int NQ>
struct StreamShape {
  static_assert(CW == 4 || CW == 8, "chunks of 4 or 8 elements");
  static constexpr int EPL = CW * NQ;                        // K elements per lane
  static constexpr int AW = ACTH ? EPL : EPL / 2;            // u32 registers per row
  static constexpr int WARP_K = 32 * EPL;                    // K elements per consumer warp
};

// Bytes of one bf16 stage holding `rows` rows (per half for gate/up).
__host__ __device__ inline size_t stream_rows_bytes(int K, int rows) {
  return (size_t)rows * K * 2;
}

// MXFP4 steps read the tiled layouts (16 mma rows per tile, see mxfp4.cuh).
// An item is TM consecutive tiles; its K blocks are split into kc chunks of
// CB = K/32/kc blocks, one stage each.  A stage holds, per tile, the chunk's
// nibbles (CB * 256 bytes: 512 bytes per block pair, 16 per lane), then per
// tile the chunk's scales (CB * 16 bytes: 64 per group of 4 blocks).
__host__ __device__ inline size_t mx_stage_bytes(int K, int TM, int kc) {
  return (size_t)TM * (K / 32 / kc) * 272;
}

// K blocks per consumer warp of an MXFP4 step: whole groups of 4.
__host__ __device__ inline int mx_warp_blocks(int K, int KW) {
  const int nblk = K / 32;
  return ((nblk + KW - 1) / KW + 3) / 4 * 4;
}

// Cross-slab partials: a bf16 step keeps up to 64 values per warp, a
// tensor-core step one per (mma row, column) of an item.  Floats per buffer
// (one of two) for KW consumer warps:
__host__ __device__ inline int stream_red_pp(int KW, bool mma, int TM, int RMAX) {
  return (mma ? TM * 16 * RMAX : 64) * KW;
}

// ---- activation slices of the bf16 steps (registers) ----------------------

// bf16 x-activation for bf16 weights, kept as raw bf16 pairs.
template <int CW, int NQ>
__device__ __forceinline__ void act_load_bf_x(const uint16_t* row, int slab, int lane, int K,
                                              uint32_t (&a)[CW * NQ / 2]) {
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    const int e = slab + q * 32 * CW + lane * CW;
    if constexpr (CW == 8) {
      const uint4 v = e < K ? *reinterpret_cast<const uint4*>(row + e) : make_uint4(0, 0, 0, 0);
      a[q * 4 + 0] = v.x;
      a[q * 4 + 1] = v.y;
      a[q * 4 + 2] = v.z;
      a[q * 4 + 3] = v.w;
    } else {
      const uint2 v = e < K ? *reinterpret_cast<const uint2*>(row + e) : make_uint2(0, 0);
      a[q * 2 + 0] = v.x;
      a[q * 2 + 1] = v.y;
    }
  }
}

// fp32 h-activation for bf16 weights, kept as fp32 bit patterns.
template <int CW, int NQ>
__device__ __forceinline__ void act_load_bf_h(const float* row, int slab, int lane, int K,
                                              uint32_t (&a)[CW * NQ]) {
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    const int e = slab + q * 32 * CW + lane * CW;
#pragma unroll
    for (int c = 0; c < CW / 4; ++c) {
      const float4 v = e < K ? __ldcg(reinterpret_cast<const float4*>(row + e) + c)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
      a[q * CW + c * 4 + 0] = __float_as_uint(v.x);
      a[q * CW + c * 4 + 1] = __float_as_uint(v.y);
      a[q * CW + c * 4 + 2] = __float_as_uint(v.z);
      a[q * CW + c * 4 + 3] = __float_as_uint(v.w);
    }
  }
}

// ---- one chunk of a bf16 weight row (in shared memory) against R activation
// slices; the caller has checked that the chunk lies inside K ----

// bf16 weights, x activation (bf16 pairs): acc[r] += w . x_r over CW elements.
template <int R, int CW, int NQ>
__device__ __forceinline__ void chunk_dot_bf_x(const uint8_t* wp, int q,
                                               const uint32_t (&a)[R][CW * NQ / 2],
                                               float (&acc)[R]) {
  uint32_t w[CW / 2];
  if constexpr (CW == 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(wp);
    w[0] = v.x;
    w[1] = v.y;
    w[2] = v.z;
    w[3] = v.w;
  } else {
    const uint2 v = *reinterpret_cast<const uint2*>(wp);
    w[0] = v.x;
    w[1] = v.y;
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
#pragma unroll
    for (int j = 0; j < CW / 2; ++j) acc[r] = fma2_bf16(w[j], a[r][q * (CW / 2) + j], acc[r]);
  }
}

// bf16 weights, fp32 activation: the bf16 weights widen exactly to fp32.
template <int R, int CW, int NQ>
__device__ __forceinline__ void chunk_dot_bf_h(const uint8_t* wp, int q,
                                               const uint32_t (&a)[R][CW * NQ], float (&acc)[R]) {
  uint32_t w[CW / 2];
  if constexpr (CW == 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(wp);
    w[0] = v.x;
    w[1] = v.y;
    w[2] = v.z;
    w[3] = v.w;
  } else {
    const uint2 v = *reinterpret_cast<const uint2*>(wp);
    w[0] = v.x;
    w[1] = v.y;
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    float s0 = acc[r], s1 = 0.f;
#pragma unroll
    for (int j = 0; j < CW / 2; ++j) {
      s0 = fmaf(__uint_as_float(w[j] << 16), __uint_as_float(a[r][q * CW + 2 * j]), s0);
      s1 = fmaf(__uint_as_float(w[j] & 0xFFFF0000u), __uint_as_float(a[r][q * CW + 2 * j + 1]), s1);
    }
    acc[r] = s0 + s1;
  }
}

// Reduce-scatter of V (power of two, <= 64) partials: returns the full warp sum
// of value index (lane >> (5 - m)) + 32*half for V = 64 (two halves), see
// warp_reduce_scatter.  For V = 64, `second` gets the second half's value.
template <int V>
__device__ __forceinline__ float stream_reduce(float (&v)[V], int lane, float& second) {
  if constexpr (V <= 32) {
    second = 0.f;
    return warp_reduce_scatter<V>(v, lane);
  } else {
    float lo[32], hi[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) { lo[i] = v[i]; hi[i] = v[32 + i]; }
    second = warp_reduce_scatter<32>(hi, lane);
    return warp_reduce_scatter<32>(lo, lane);
  }
}

// ---- work decoding, identical in the producer and the consumers ----------

struct StreamItem {
  int e;     // matrix (expert) index
  int p0;    // first pair in pair_list (routed)
  int pr;    // activation rows of this item
  int row0;  // first output row
};

template <bool ROUTED, int RW>
__device__ __forceinline__ int stream_n_items(const StreamArgs& a, int& tiles) {
  tiles = (a.N + RW - 1) / RW;
  return ROUTED ? ld_tab(a.n_active) * tiles : tiles;
}

template <bool ROUTED, int RW>
__device__ __forceinline__ StreamItem stream_item(const StreamArgs& a, int it, int tiles) {
  StreamItem m;
  if (ROUTED) {
    const int slot = it / tiles;
    m.e = ld_tab(a.active_expert + slot);
    m.p0 = ld_tab(a.active_off + slot);
    m.pr = ld_tab(a.active_off + slot + 1) - m.p0;
    m.row0 = (it % tiles) * RW;
  } else {
    m.e = 0;
    m.p0 = 0;
    m.pr = a.B;
    m.row0 = it * RW;
  }
  return m;
}

// Activation rows of the next pass: the bf16 steps take 4, 2 or 1 (a
// template parameter of their consumer); the tensor-core steps any count up
// to RMAX (mma columns).
template <int RMAX, bool MMA>
__device__ __forceinline__ int stream_pass_rows(int left) {
  if (MMA) return min(left, RMAX);
  return (RMAX >= 4 && left >= 4) ? 4 : ((RMAX >= 2 && left >= 2) ? 2 : 1);
}

// CTA c owns the contiguous item range [lo, hi).  Items are ordered expert by
// expert, so a range is a few runs of tiles that share one activation set:
// the consumers load activations once per (run, pass), not once per item.
__device__ __forceinline__ void stream_range(int n_items, int& lo, int& hi) {
  lo = (int)(((long long)blockIdx.x * n_items) / gridDim.x);
  hi = (int)(((long long)(blockIdx.x + 1) * n_items) / gridDim.x);
}

// Steps that run earlier in the same launch, split the standard way (at most
// two; n = 0: none), as item counts and weight bytes per item.
struct SegPrior {
  int n0 = 0;
  long long s0 = 0;
  int n1 = 0;
  long long s1 = 0;
};

__device__ __forceinline__ long long prior_bytes(const SegPrior& p, int c, int G) {
  return (long long)(((long long)c * p.n0) / G) * p.s0 + (long long)(((long long)c * p.n1) / G) * p.s1;
}

// First item of CTA c (of G) in a step of n items of ib bytes that follows
// `p`: chosen so that every CTA streams about the same bytes over all the
// steps of the launch, i.e. round((c T / G - P(c)) / ib) clamped to [0, n],
// T being the launch's total bytes and P(c) what CTAs 0..c-1 stream in the
// earlier steps.  (The earlier steps' per-CTA shares differ by up to one of
// their items; this step evens that out to half of one of its own.)
__device__ __forceinline__ int balanced_start(const SegPrior& p, int c, int G, int n, long long ib) {
  if (c >= G) return n;
  const long long total = (long long)p.n0 * p.s0 + (long long)p.n1 * p.s1 + (long long)n * ib;
  const long long num = (long long)c * total - (long long)G * prior_bytes(p, c, G);
  if (num <= 0 || ib <= 0) return 0;
  const long long den = (long long)G * ib;
  return (int)min((long long)n, (num + den / 2) / den);
}

// [lo, hi) for this CTA: the standard split without a prior, else balanced.
// Balanced starts need not increase with c when an earlier step's items are
// much larger than this step's share per CTA; an empty range (hi = lo) then
// leaves the items in between to the neighbours, which compute them both
// (identical values), so every item is still covered.
__device__ __forceinline__ void seg_range(const SegPrior& p, int n, long long ib, int& lo, int& hi) {
  if (p.n0 == 0 && p.n1 == 0) {
    stream_range(n, lo, hi);
    return;
  }
  const int c = blockIdx.x, G = gridDim.x;
  lo = balanced_start(p, c, G, n, ib);
  hi = max(lo, balanced_start(p, c + 1, G, n, ib));
}

// End of the run that starts at item `it` (same expert for routed steps; a
// dense step is one run).
template <bool ROUTED>
__device__ __forceinline__ int stream_run_end(int it, int hi, int tiles) {
  return ROUTED ? min(hi, (it / tiles + 1) * tiles) : hi;
}

template <bool ROUTED, int RW>
__device__ __forceinline__ int stream_row0(int it, int tiles) {
  return ROUTED ? (it % tiles) * RW : it * RW;
}

// Producer: lane 0 of warp 0 issues the bulk copies for items [lo, hi) of one
// step, continuing the CTA's running stage counter.  A bf16 stage holds SP
// rows (gate/up: SP gate rows then the SP matching up rows); an MXFP4 stage
// holds one K chunk of an item's TM tiles.
template <int WF, bool GLU, bool ROUTED, int SP, int RW, int RMAX, bool MMA, int TM>
__device__ __forceinline__ void stream_produce_range(const StreamArgs& a, int lo, int hi, int tiles,
                                                     uint8_t* stages, uint64_t* full,
                                                     uint64_t* empty, uint32_t& stage) {
  constexpr int G = GLU ? 2 : 1;
  const int SPI = MMA ? a.kc : RW / SP;
  const uint64_t pol = policy_evict_first();
  for (int it0 = lo; it0 < hi;) {
    const int run_end = stream_run_end<ROUTED>(it0, hi, tiles);
    const StreamItem m = stream_item<ROUTED, RW>(a, it0, tiles);
    const uint8_t* qe = a.q + (size_t)m.e * a.q_stride;
    for (int done = 0; done < m.pr; done += stream_pass_rows<RMAX, MMA>(m.pr - done)) {
      for (int it = it0; it < run_end; ++it) {
        const int row0 = stream_row0<ROUTED, RW>(it, tiles);
        for (int st = 0; st < SPI; ++st, ++stage) {
          const int buf = (int)(stage % (uint32_t)a.NS);
          const uint32_t use = stage / (uint32_t)a.NS;
          if (use > 0) mbar_wait(&empty[buf], (use - 1) & 1u, a.status);
          uint8_t* dst = stages + (size_t)buf * a.stage_bytes;
          if constexpr (MMA) {
            // tiles T0.. of the item, K chunk st: per tile its nibbles and scales
            const uint8_t* se = a.s + (size_t)m.e * a.s_stride;
            const int rows_per_tile = GLU ? 8 : 16;
            const int T0 = row0 / rows_per_tile;
            const int nvt = max(0, min(TM, a.N / rows_per_tile - T0));
            const uint32_t CB = (uint32_t)(a.K / 32 / a.kc);
            const size_t tq = (size_t)a.K * 8, ts = (size_t)a.K / 2;
            mbar_arrive_expect_tx(&full[buf], (uint32_t)nvt * CB * 272u);
            if (a.kc == 1) {   // the item's tiles are contiguous: one copy each part
              if (nvt > 0) {
                bulk_g2s(dst, qe + (size_t)T0 * tq, (uint32_t)nvt * CB * 256u, &full[buf], pol);
                bulk_g2s(dst + (size_t)TM * CB * 256, se + (size_t)T0 * ts,
                         (uint32_t)nvt * CB * 16u, &full[buf], pol);
              }
            } else {
              for (int t = 0; t < nvt; ++t) {
                bulk_g2s(dst + (size_t)t * CB * 256, qe + (size_t)(T0 + t) * tq + (size_t)st * CB * 256,
                         CB * 256u, &full[buf], pol);
                bulk_g2s(dst + (size_t)TM * CB * 256 + (size_t)t * CB * 16,
                         se + (size_t)(T0 + t) * ts + (size_t)st * CB * 16, CB * 16u, &full[buf],
                         pol);
              }
            }
          } else {
            const int r0 = row0 + st * SP;
            const int nv = max(0, min(SP, a.N - r0));
            const size_t half_bytes = (size_t)SP * a.K * 2;
            const uint32_t wb = (uint32_t)nv * a.K * 2;
            mbar_arrive_expect_tx(&full[buf], G * wb);
            if (nv > 0) {
              bulk_g2s(dst, qe + (size_t)r0 * a.K * 2, wb, &full[buf], pol);
              if (GLU)
                bulk_g2s(dst + half_bytes, qe + (size_t)(a.N + r0) * a.K * 2, wb, &full[buf], pol);
            }
          }
        }
      }
    }
    it0 = run_end;
  }
}

// Drain: wait until the last use of every buffer has been consumed, so no copy
// is still landing in this CTA's shared memory when it exits.
__device__ __forceinline__ void stream_drain(const StreamArgs& a, uint64_t* empty, uint32_t stage) {
  for (int b = 0; b < a.NS && (uint32_t)b < stage; ++b) {
    const uint32_t uses = (stage - (uint32_t)b + (uint32_t)a.NS - 1) / (uint32_t)a.NS;
    mbar_wait(&empty[b], (uses - 1) & 1u, a.status);
  }
}

// Activation row of pair/row id `pid`: x rows are indexed by batch row
// (pid / k for routed pairs), h rows by pair.
template <bool ROUTED>
__device__ __forceinline__ int stream_x_row(const StreamArgs& a, int pid) {
  return ROUTED ? pid / a.k : pid;
}

// Epilogue thread index of consumer thread ct when only the first `busy` of
// the KW consumer warps own K elements: the idle warps take the first
// outputs, so the per-item finalisation (partial sums, SwiGLU, stores) stays
// off the critical path of the warps that do the products.
__device__ __forceinline__ int stream_epi_index(int ct, int busy, int KW) {
  const int cthreads = 32 * KW, ct0 = busy < KW ? 32 * busy : 0;
  const int e = ct - ct0;
  return e < 0 ? e + cthreads : e;
}

// Sum of the n <= kMmaWarps partials at p, in order 0..n-1: the bound is a
// compile-time constant so every load issues before the dependent adds.
__device__ __forceinline__ float slab_sum(const float* p, int n) {
  float v[kMmaWarps];
#pragma unroll
  for (int w = 0; w < kMmaWarps; ++w) v[w] = w < n ? p[w] : 0.f;
  float s = 0.f;
#pragma unroll
  for (int w = 0; w < kMmaWarps; ++w) s += v[w];
  return s;
}

// Consumers of a bf16 step: one pass of R activation rows over the run
// [it0, run_end) of items that share them.  Activation slices and pair ids are
// loaded once; every item then streams its SPI stages, reduces and finalises.
template <bool GLU, bool ACTH, bool ROUTED, int SP, int RW, int R, int CW, int NQ>
__device__ __forceinline__ void stream_consume_run(const StreamArgs& a, const StreamItem& m,
                                                   int done, int it0, int run_end, int tiles,
                                                   uint8_t* stages, uint64_t* full,
                                                   uint64_t* empty, float* red, uint32_t& stage,
                                                   int& pp, int kw, int KW, int lane) {
  using Sh = StreamShape<ACTH, CW, NQ>;
  constexpr int G = GLU ? 2 : 1;
  constexpr int SPI = RW / SP;
  constexpr int V = RW * G * R;
  constexpr int VM = V < 32 ? V : 32;
  constexpr int M = VM == 1 ? 0 : VM == 2 ? 1 : VM == 4 ? 2 : VM == 8 ? 3 : VM == 16 ? 4 : 5;
  const size_t half_bytes = (size_t)SP * a.K * 2;
  const int slab = kw * Sh::WARP_K;
  const int cthreads = KW * 32;
  const int ct = (int)threadIdx.x - 32;

  int pid[R];
  uint32_t act[R][Sh::AW];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    pid[r] = ROUTED ? ld_tab(a.pair_list + m.p0 + done + r) : done + r;
    if constexpr (!ACTH)
      act_load_bf_x<CW, NQ>(a.x + (size_t)stream_x_row<ROUTED>(a, pid[r]) * a.K, slab, lane, a.K,
                            act[r]);
    else
      act_load_bf_h<CW, NQ>(a.h + (size_t)pid[r] * a.K, slab, lane, a.K, act[r]);
  }

  for (int it = it0; it < run_end; ++it) {
    const int row0 = stream_row0<ROUTED, RW>(it, tiles);
    float v[V];
#pragma unroll
    for (int st = 0; st < SPI; ++st) {
      const int buf = (int)(stage % (uint32_t)a.NS);
      mbar_wait(&full[buf], (stage / (uint32_t)a.NS) & 1u, a.status);
      const uint8_t* sb = stages + (size_t)buf * a.stage_bytes;
#pragma unroll
      for (int rr = 0; rr < SP; ++rr)
#pragma unroll
        for (int r = 0; r < R * G; ++r) v[(st * SP + rr) * R * G + r] = 0.f;
      // one warp-uniform test per chunk (K is a multiple of 32 * CW), then
      // all SP rows of the stage back to back
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        const int e = slab + q * 32 * CW + lane * CW;
        if (e < a.K) {
#pragma unroll
          for (int rr = 0; rr < SP; ++rr) {
            const int j = st * SP + rr;
#pragma unroll
            for (int gu = 0; gu < G; ++gu) {
              const uint8_t* wp = sb + gu * half_bytes + ((size_t)rr * a.K + e) * 2;
              float o[R];
#pragma unroll
              for (int r = 0; r < R; ++r) o[r] = v[(j * R + r) * G + gu];
              if constexpr (ACTH) chunk_dot_bf_h<R, CW, NQ>(wp, q, act, o);
              else chunk_dot_bf_x<R, CW, NQ>(wp, q, act, o);
#pragma unroll
              for (int r = 0; r < R; ++r) v[(j * R + r) * G + gu] = o[r];
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[buf]);
      ++stage;
    }

    // combine: lanes -> one value per lane group, then K slabs through shared memory
    float second;
    const float first = stream_reduce<V>(v, lane, second);
    float* rb = red + (size_t)pp * a.red_pp;
    if ((lane & ((1 << (5 - M)) - 1)) == 0) {
      const int vi = lane >> (5 - M);
      rb[vi * KW + kw] = first;
      if (V > 32) rb[(32 + vi) * KW + kw] = second;
    }
    consumer_sync(cthreads);
    const int busy = min(KW, (a.K + Sh::WARP_K - 1) / Sh::WARP_K);
    for (int t = stream_epi_index(ct, busy, KW); t < RW * R; t += cthreads) {
      const int j = t / R, r = t % R;
      const int row = row0 + j;
      if (row >= a.N) continue;
      int p = pid[0];
#pragma unroll
      for (int q = 1; q < R; ++q)
        if (q == r) p = pid[q];
      float* dst = a.out + (size_t)p * a.N + row;
      if constexpr (GLU) {
        const float* pg = rb + ((j * R + r) * 2) * KW;
        float g = 0.f, u = 0.f;
        g = slab_sum(pg, KW);
        u = slab_sum(pg + KW, KW);
        const float hv = g / (1.0f + expf(-g)) * u;
        *dst = hv;
        if (a.out_amax) atomicMax(a.out_amax + p, __float_as_uint(fabsf(hv)));
      } else {
        const float* pv = rb + (j * R + r) * KW;
        float acc = 0.f;
        acc = slab_sum(pv, KW);
        *dst = acc;
      }
    }
    pp ^= 1;
  }
}

// One K block of a lane's two mma rows against its activation column: wa, wb
// are nibble bytes [4t, 4t+4) of mma rows g and g+8 (elements 8t..8t+7 of the
// block), bytes 0 and 1 going to the first MMA and 2, 3 to the second, one
// f16 pair each; x holds the same eight elements of column g.  Both operands
// see one k permutation, which leaves the dot products unchanged.  The two
// MMAs sum the block from zero; the rows' block scales fa, fb then multiply
// the result into the fp32 accumulators (c1, c3: column 2t+1, skipped when
// ONE, i.e. a single activation row).
template <bool ONE>
__device__ __forceinline__ void mx_block_mma(uint32_t wa, uint32_t wb, float fa, float fb,
                                             const uint32_t (&x)[4], float& c0, float& c1,
                                             float& c2, float& c3) {
  uint32_t ha[4], hb[4];
  e2m1x8_to_f16x2(wa, ha);
  e2m1x8_to_f16x2(wb, hb);
  float d[4];
  mma_f16_16816_zero(d, ha[0], hb[0], ha[1], hb[1], x[0], x[1]);
  mma_f16_16816(d, ha[2], hb[2], ha[3], hb[3], x[2], x[3]);
  c0 = fmaf(fa, d[0], c0);
  c2 = fmaf(fb, d[2], c2);
  if (!ONE) {
    c1 = fmaf(fa, d[1], c1);
    c3 = fmaf(fb, d[3], c3);
  }
}

// E8M0 scale bytes at bit offset 8j of a word -> fp32 2^(code - 127) through
// the exponent field; code 0 (2^-127) becomes 0, which only drops products
// below 6 * 2^-127 * |activation|.
__device__ __forceinline__ float e8m0_byte0(uint32_t w) { return __uint_as_float((w << 23) & 0x7F800000u); }
__device__ __forceinline__ float e8m0_byte1(uint32_t w) { return __uint_as_float((w << 15) & 0x7F800000u); }
__device__ __forceinline__ float e8m0_byte2(uint32_t w) { return __uint_as_float((w << 7) & 0x7F800000u); }
__device__ __forceinline__ float e8m0_byte3(uint32_t w) { return __uint_as_float((w >> 1) & 0x7F800000u); }

// NQ groups of 4 K blocks of one tile (GUARD: only the first nb blocks):
// per group 8 scale bytes and two 16-byte nibble loads per lane.
template <bool ONE, int NQ, bool GUARD>
__device__ __forceinline__ void mx_group_run(const uint8_t* nib, const uint8_t* scl,
                                             const uint32_t (&X)[4 * NQ][4], int nb, float& c0,
                                             float& c1, float& c2, float& c3) {
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    if (GUARD && 4 * q >= nb) break;
    const uint2 sv = *reinterpret_cast<const uint2*>(scl + q * 64);
    const uint4 w0 = *reinterpret_cast<const uint4*>(nib + (2 * q) * 512);
    const uint4 w1 = *reinterpret_cast<const uint4*>(nib + (2 * q + 1) * 512);
    mx_block_mma<ONE>(w0.x, w0.y, e8m0_byte0(sv.x), e8m0_byte1(sv.x), X[4 * q], c0, c1, c2, c3);
    mx_block_mma<ONE>(w0.z, w0.w, e8m0_byte2(sv.x), e8m0_byte3(sv.x), X[4 * q + 1], c0, c1, c2, c3);
    mx_block_mma<ONE>(w1.x, w1.y, e8m0_byte0(sv.y), e8m0_byte1(sv.y), X[4 * q + 2], c0, c1, c2, c3);
    mx_block_mma<ONE>(w1.z, w1.w, e8m0_byte2(sv.y), e8m0_byte3(sv.y), X[4 * q + 3], c0, c1, c2, c3);
  }
}

// The same with the activation operand read from shared memory, one 16-byte
// load per block (xs points at this lane's entry of the warp's first block;
// blocks are 4 entries apart).
template <bool ONE, int NQ, bool GUARD>
__device__ __forceinline__ void mx_group_run_xs(const uint8_t* nib, const uint8_t* scl,
                                                const uint4* xs, int nb, float& c0, float& c1,
                                                float& c2, float& c3) {
  // not unrolled: four blocks (eight MMAs) per iteration already overlap, and
  // the shorter loop body leaves the kernel's code and registers smaller
#pragma unroll 1
  for (int q = 0; q < NQ; ++q) {
    if (GUARD && 4 * q >= nb) break;
    const uint2 sv = *reinterpret_cast<const uint2*>(scl + q * 64);
    const uint4 w0 = *reinterpret_cast<const uint4*>(nib + (2 * q) * 512);
    const uint4 w1 = *reinterpret_cast<const uint4*>(nib + (2 * q + 1) * 512);
    uint32_t x[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 v = xs[(4 * q + j) * 4];
      x[j][0] = v.x;
      x[j][1] = v.y;
      x[j][2] = v.z;
      x[j][3] = v.w;
    }
    mx_block_mma<ONE>(w0.x, w0.y, e8m0_byte0(sv.x), e8m0_byte1(sv.x), x[0], c0, c1, c2, c3);
    mx_block_mma<ONE>(w0.z, w0.w, e8m0_byte2(sv.x), e8m0_byte3(sv.x), x[1], c0, c1, c2, c3);
    mx_block_mma<ONE>(w1.x, w1.y, e8m0_byte0(sv.y), e8m0_byte1(sv.y), x[2], c0, c1, c2, c3);
    mx_block_mma<ONE>(w1.z, w1.w, e8m0_byte2(sv.y), e8m0_byte3(sv.y), x[3], c0, c1, c2, c3);
  }
}

// Consumers of an MXFP4 step (tensor cores): one pass of R <= RMAX activation
// rows, the mma columns, over the run [it0, run_end) of items of one expert.
//
// An item is TM tiles of 16 mma rows (tiled layouts, see mxfp4.cuh): plain
// steps put 16 consecutive output rows in a tile, gate/up steps 8 row pairs
// with gate row g in mma row g and its up row in mma row g + 8, so one lane
// ends with both halves of a pair.  Warp kw owns the NB K blocks from
// b0 = kw * NB (NB a multiple of 4, all in one K chunk) and reads, per pair of
// blocks, 16 bytes (lane-ordered, conflict-free) and per group of four, 8
// scale bytes.
// X holds the pass's activation operand; xkey/xshift remember which single x
// row it holds (-1: none), so a run of another expert on the same row (every
// run at B = 1) keeps it instead of reloading and re-reducing it.
template <bool GLU, bool ACTH, int TM, int NBMAX, int RMAX, bool ONE, bool XS, bool F8 = false>
__device__ __forceinline__ void stream_consume_run_mma(
    const StreamArgs& a, const StreamItem& m, int done, int R, int it0, int run_end, int tiles,
    uint8_t* stages, uint64_t* full, uint64_t* empty, float* red, uint32_t& stage, int& pp,
    int& rp, int kw, int KW, int lane, uint32_t (&X)[XS ? 1 : NBMAX][4], int& xkey, int& xshift) {
  constexpr int TR = GLU ? TM * 8 : TM * 16;   // output rows (pairs) per item
  const int g = lane >> 2, t = lane & 3;
  const int nblk = a.K >> 5;
  const int NB = mx_warp_blocks(a.K, KW);
  const int b0 = kw * NB;
  const int nb = max(0, min(NB, nblk - b0));
  const int CB = nblk / a.kc;
  const int chunk = nb > 0 ? b0 / CB : 0;
  const int lb0 = b0 - chunk * CB;
  const int cthreads = KW * 32;
  const int ct = (int)threadIdx.x - 32;

  // the column this lane feeds, and this thread's output column in the epilogue
  const int ci = min(g, R - 1);
  // outputs go first to the consumer warps that own no K blocks
  const int et = stream_epi_index(ct, min(KW, (nblk + NB - 1) / NB), KW);
  const int ei = et % R;
  const int cpid = ld_tab(a.pair_list + m.p0 + done + ci);
  const int epid = ld_tab(a.pair_list + m.p0 + done + ei);

  int eshift;
  // one x row for the whole pass (R = 1): the same key in every lane and warp
  const int key = (!ACTH && R == 1) ? cpid / a.k : -1;
  if constexpr (XS) {
    eshift = *a.xs_shift;   // the operand is in shared memory already
  } else if (!ACTH && key >= 0 && key == xkey) {
    eshift = xshift;
  } else if constexpr (!ACTH) {
    // x rows (bf16): the f16 scaling shift needs max |x| over the whole row,
    // which the KW warps hold together: reduce through shared memory.
    unsigned* s_amax = reinterpret_cast<unsigned*>(red + 2 * (size_t)a.red_pp);
    unsigned* slots = s_amax + (rp & 1) * 8;
    const uint16_t* xr = a.x + (size_t)(cpid / a.k) * a.K + 8 * t;
    uint32_t mx = 0;
#pragma unroll
    for (int b = 0; b < NBMAX; ++b) {
      uint4 v = make_uint4(0, 0, 0, 0);
      if (b < nb) v = *reinterpret_cast<const uint4*>(xr + (size_t)(b0 + b) * 32);
      X[b][0] = v.x;
      X[b][1] = v.y;
      X[b][2] = v.z;
      X[b][3] = v.w;
#pragma unroll
      for (int j = 0; j < 4; ++j) mx = max(mx, max(X[b][j] & 0x7FFFu, (X[b][j] >> 16) & 0x7FFFu));
    }
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    if (t == 0) atomicMax(slots + ci, mx);
    consumer_sync(cthreads);
    const int cshift = f16_shift_for_amax(bf16_bits_to_f32(slots[ci]));
    eshift = f16_shift_for_amax(bf16_bits_to_f32(slots[ei]));
    const float sc = pow2f(-cshift);
#pragma unroll
    for (int b = 0; b < NBMAX; ++b)
#pragma unroll
      for (int j = 0; j < 4; ++j)
        X[b][j] = pack_f16x2(__uint_as_float(X[b][j] << 16) * sc,
                             __uint_as_float(X[b][j] & 0xFFFF0000u) * sc);
    // the other parity's slots are free: every consumer is past this barrier
    if (kw == 0 && lane < 8) s_amax[((rp & 1) ^ 1) * 8 + lane] = 0u;
    rp ^= 1;
    xkey = key;
    xshift = eshift;
  } else {
    // h rows (fp32): the shift comes from FC1's per-pair max |h|
    const int cshift = f16_shift_for_amax(
        __int_as_float(ld_relaxed_gpu(reinterpret_cast<const int*>(a.h_amax) + cpid)));
    eshift = f16_shift_for_amax(
        __int_as_float(ld_relaxed_gpu(reinterpret_cast<const int*>(a.h_amax) + epid)));
    const float sc = pow2f(-cshift);
    const float* hr = a.h + (size_t)cpid * a.K + 8 * t;
#pragma unroll
    for (int b = 0; b < NBMAX; ++b) {
      float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
      if (b < nb) {
        v0 = __ldcg(reinterpret_cast<const float4*>(hr + (size_t)(b0 + b) * 32));
        v1 = __ldcg(reinterpret_cast<const float4*>(hr + (size_t)(b0 + b) * 32 + 4));
      }
      // MXFP8: the block's 32 values sit in this lane quad (all lanes take part)
      if constexpr (F8) mxfp8_round8(v0, v1);
      X[b][0] = pack_f16x2(v0.x * sc, v0.y * sc);
      X[b][1] = pack_f16x2(v0.z * sc, v0.w * sc);
      X[b][2] = pack_f16x2(v1.x * sc, v1.y * sc);
      X[b][3] = pack_f16x2(v1.z * sc, v1.w * sc);
    }
  }
  const float back = pow2f(eshift);
  const size_t nib_tile = (size_t)CB * 256, scl_base = (size_t)TM * CB * 256;
  // ring position of this warp's chunk and of the item's first stage, advanced
  // by kc per item without divisions (kc <= NS)
  const uint32_t NS = (uint32_t)a.NS, KC = (uint32_t)a.kc;
  uint32_t cbuf = (stage + (uint32_t)chunk) % NS, cph = ((stage + (uint32_t)chunk) / NS) & 1u;
  uint32_t ibuf = stage % NS;
  const int ej = et / R;   // this thread's output row (pair) within an item, column ei
  int row0 = stream_row0<true, TR>(it0, tiles);

  for (int it = it0; it < run_end; ++it, row0 += TR) {
    if (nb > 0) mbar_wait(&full[cbuf], cph, a.status);
    const uint8_t* sp = stages + (size_t)cbuf * a.stage_bytes;
    float acc[TM][4];
#pragma unroll
    for (int mb = 0; mb < TM; ++mb) {
      const uint8_t* nib = sp + mb * nib_tile + (size_t)(lb0 >> 1) * 512 + lane * 16;
      const uint8_t* scl = sp + scl_base + (size_t)mb * CB * 16 + (size_t)(lb0 >> 2) * 64 + g * 8;
      float c0 = 0.f, c1 = 0.f, c2 = 0.f, c3 = 0.f;
      if constexpr (XS) {
        const uint4* xs = a.xs + (size_t)b0 * 4 + t;
        if (nb == NBMAX) mx_group_run_xs<ONE, NBMAX / 4, false>(nib, scl, xs, nb, c0, c1, c2, c3);
        else mx_group_run_xs<ONE, NBMAX / 4, true>(nib, scl, xs, nb, c0, c1, c2, c3);
      } else if (nb == NBMAX) {   // the common case: one straight run the compiler can schedule
        mx_group_run<ONE, NBMAX / 4, false>(nib, scl, X, nb, c0, c1, c2, c3);
      } else {
        mx_group_run<ONE, NBMAX / 4, true>(nib, scl, X, nb, c0, c1, c2, c3);
      }
      acc[mb][0] = c0;
      acc[mb][1] = c1;
      acc[mb][2] = c2;
      acc[mb][3] = c3;
    }
    __syncwarp();
    if (lane == 0) {
      uint32_t b = ibuf;
      for (uint32_t s = 0; s < KC; ++s) {
        mbar_arrive(&empty[b]);
        if (++b == NS) b = 0;
      }
    }
    stage += KC;
    ibuf += KC;
    if (ibuf >= NS) ibuf -= NS;
    cbuf += KC;
    if (cbuf >= NS) {
      cbuf -= NS;
      cph ^= 1u;
    }

    // cross-slab combine: partial of (mma row, column) from warp kw at
    // ((mb*16 + row)*RMAX + column)*KW + kw
    float* rbuf = red + (size_t)pp * a.red_pp;
#pragma unroll
    for (int mb = 0; mb < TM; ++mb)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int col = 2 * t + (i & 1), row = g + 8 * (i >> 1);
        if (col < R) rbuf[((mb * 16 + row) * RMAX + col) * KW + kw] = acc[mb][i];
      }
    consumer_sync(cthreads);
    if (et < TR * R) {
      const int j = ej;
      const int row = row0 + j;
      if (row < a.N) {
        float* dst = a.out + (size_t)epid * a.N + row;
        if constexpr (GLU) {
          const float* pg = rbuf + (((j >> 3) * 16 + (j & 7)) * RMAX + ei) * KW;
          const float* pu = pg + 8 * RMAX * KW;
          float gs = 0.f, us = 0.f;
          gs = slab_sum(pg, KW);
          us = slab_sum(pu, KW);
          gs *= back;
          us *= back;
          const float hv = gs / (1.0f + expf(-gs)) * us;
          *dst = hv;
          if (a.out_amax) atomicMax(a.out_amax + epid, __float_as_uint(fabsf(hv)));
        } else {
          const float* pv = rbuf + (((j >> 4) * 16 + (j & 15)) * RMAX + ei) * KW;
          float sum = 0.f;
          sum = slab_sum(pv, KW);
          *dst = sum * back;
        }
      }
    }
    pp ^= 1;
  }
}

// Consumers: items [lo, hi) of one step, run by run, pass by pass.
template <int WF, bool GLU, bool ACTH, bool ROUTED, int SP, int RW, int RMAX, bool MMA, int TM,
          int NBMAX, int CW, int NQ, bool XS = false, bool F8 = false>
__device__ __forceinline__ void stream_consume_range(const StreamArgs& a, int lo, int hi, int tiles,
                                                     uint8_t* stages, uint64_t* full,
                                                     uint64_t* empty, float* red, uint32_t& stage,
                                                     int& pp, int& rp, int kw, int KW, int lane) {
  uint32_t X[MMA && !XS ? NBMAX : 1][4];
  int xkey = -1, xshift = 0;
  for (int it0 = lo; it0 < hi;) {
    const int run_end = stream_run_end<ROUTED>(it0, hi, tiles);
    const StreamItem m = stream_item<ROUTED, RW>(a, it0, tiles);
    for (int done = 0; done < m.pr;) {
      const int R = stream_pass_rows<RMAX, MMA>(m.pr - done);
      if constexpr (MMA) {
        if (RMAX == 1 || R == 1)
          stream_consume_run_mma<GLU, ACTH, TM, NBMAX, RMAX, true, XS, F8>(
              a, m, done, R, it0, run_end, tiles, stages, full, empty, red, stage, pp, rp, kw, KW,
              lane, X, xkey, xshift);
        else if constexpr (RMAX > 1)
          stream_consume_run_mma<GLU, ACTH, TM, NBMAX, RMAX, false, XS>(
              a, m, done, R, it0, run_end, tiles, stages, full, empty, red, stage, pp, rp, kw, KW,
              lane, X, xkey, xshift);
      } else {
        if (R == 1) {
          stream_consume_run<GLU, ACTH, ROUTED, SP, RW, 1, CW, NQ>(a, m, done, it0, run_end, tiles,
                                                           stages, full, empty, red, stage, pp,
                                                           kw, KW, lane);
        } else if constexpr (RMAX >= 2) {
          if (R == 2) {
            stream_consume_run<GLU, ACTH, ROUTED, SP, RW, 2, CW, NQ>(a, m, done, it0, run_end, tiles,
                                                             stages, full, empty, red, stage, pp,
                                                             kw, KW, lane);
          } else if constexpr (RMAX >= 4) {
            stream_consume_run<GLU, ACTH, ROUTED, SP, RW, 4, CW, NQ>(a, m, done, it0, run_end, tiles,
                                                             stages, full, empty, red, stage, pp,
                                                             kw, KW, lane);
          }
        }
      }
      done += R;
    }
    it0 = run_end;
  }
}

// Compile-time description of one streaming step.  MMA steps (MXFP4, routed)
// use tiles of TM x 16 mma rows (RW = 16 TM rows, or 8 TM pairs for gate/up)
// and at most NBMAX K blocks per consumer warp.
template <int WF_, bool GLU_, bool ACTH_, bool ROUTED_, int SP_, int RW_, int RMAX_,
          bool MMA_ = false, int TM_ = 1, int NBMAX_ = 1, int CW_ = 8, int NQ_ = 4,
          bool XS_ = false, bool F8_ = false>
struct StreamCfg {
  static constexpr int WF = WF_;
  static constexpr bool GLU = GLU_, ACTH = ACTH_, ROUTED = ROUTED_, MMA = MMA_;
  static constexpr bool XS = XS_;   // MMA steps of one x row: the operand in shared memory
  static constexpr int SP = SP_, RW = RW_, RMAX = RMAX_, TM = TM_, NBMAX = NBMAX_;
  static constexpr int CW = CW_, NQ = NQ_;   // bf16 steps: lane chunking (see StreamShape)
  static_assert(RW % SP == 0, "an item is a whole number of stages");
  static_assert(!MMA || (WF == kWfMx && ROUTED && RW == (GLU ? 8 : 16) * TM && RMAX <= 8),
                "tensor-core steps: routed MXFP4, one tile per item, at most 8 columns");
  static_assert(MMA || WF == kWfBf16, "MXFP4 steps run on the tensor cores");
  static_assert(!XS || (MMA && !ACTH && RMAX == 1), "a shared-memory operand holds one x row");
  // MXFP4 steps of one activation row with MXFP8 activations: x or h rounded
  // to E4M3 with one E8M0 scale per 32 elements (mxfp8_round8), then carried
  // into the same f16 MMAs exactly
  static constexpr bool F8 = F8_;
  static_assert(!F8 || (MMA && RMAX == 1), "MXFP8 activations: one-row MXFP4 steps");
};

// Weight bytes one item of a step streams: MXFP4 tiles of 16 rows (K/2
// nibble bytes + K/32 scale bytes per row), or RW bf16 rows (gate/up: pairs).
template <class C>
__device__ __forceinline__ long long cfg_item_bytes(const StreamArgs& a) {
  if constexpr (C::MMA) return (long long)C::TM * 17 * (a.K / 2);
  else return (long long)C::RW * (C::GLU ? 2 : 1) * a.K * 2;
}

// A dense step as the prior of a later step in the same launch.
template <class C>
__device__ __forceinline__ void cfg_add_prior(const StreamArgs& a, SegPrior& p) {
  int tiles;
  const int n = stream_n_items<C::ROUTED, C::RW>(a, tiles);
  if (p.n0 == 0) {
    p.n0 = n;
    p.s0 = cfg_item_bytes<C>(a);
  } else {
    p.n1 = n;
    p.s1 = cfg_item_bytes<C>(a);
  }
}

template <class C>
__device__ __forceinline__ void cfg_produce(const StreamArgs& a, const SegPrior& prior,
                                            uint8_t* stages, uint64_t* full, uint64_t* empty,
                                            uint32_t& stage) {
  int tiles, lo, hi;
  const int n = stream_n_items<C::ROUTED, C::RW>(a, tiles);
  seg_range(prior, n, cfg_item_bytes<C>(a), lo, hi);
  stream_produce_range<C::WF, C::GLU, C::ROUTED, C::SP, C::RW, C::RMAX, C::MMA, C::TM>(
      a, lo, hi, tiles, stages, full, empty, stage);
}

// Consumers of this CTA's items of step C; `part` (0 or 1) with `first`
// items in part 0 consumes only part 0 ([lo, lo + first)) or part 1 (the
// rest), so other work can run between the two (part < 0: all of them).
template <class C>
__device__ __forceinline__ void cfg_consume(const StreamArgs& a, const SegPrior& prior,
                                            uint8_t* stages, uint64_t* full, uint64_t* empty,
                                            float* red, uint32_t& stage, int& pp, int& rp, int kw,
                                            int KW, int lane, int part = -1, int first = 0) {
  int tiles, lo, hi;
  const int n = stream_n_items<C::ROUTED, C::RW>(a, tiles);
  seg_range(prior, n, cfg_item_bytes<C>(a), lo, hi);
  if (part == 0) hi = min(hi, lo + first);
  else if (part == 1) lo = min(hi, lo + first);
  stream_consume_range<C::WF, C::GLU, C::ACTH, C::ROUTED, C::SP, C::RW, C::RMAX, C::MMA, C::TM,
                       C::NBMAX, C::CW, C::NQ, C::XS, C::F8>(a, lo, hi, tiles, stages, full, empty,
                                                       red, stage, pp, rp, kw, KW, lane);
}

// Shared-memory carve-up common to both kernels.
struct StreamSmem {
  uint8_t* stages;
  uint64_t* full;
  uint64_t* empty;
  float* red;
};

__device__ __forceinline__ StreamSmem stream_smem_init(uint8_t* smem, int NS, int stage_bytes,
                                                       int red_pp, int KW) {
  StreamSmem m;
  m.stages = smem;
  m.full = reinterpret_cast<uint64_t*>(smem + (size_t)NS * stage_bytes);
  m.empty = m.full + NS;
  m.red = reinterpret_cast<float*>(m.empty + NS);
  if (threadIdx.x == 0) {
    for (int b = 0; b < NS; ++b) {
      mbar_init(&m.full[b], 1);
      mbar_init(&m.empty[b], (uint32_t)KW);
    }
    fence_barrier_init();
  }
  if (threadIdx.x < 16) reinterpret_cast<unsigned*>(m.red + (size_t)2 * red_pp)[threadIdx.x] = 0u;
  __syncthreads();
  return m;
}

// Single step.  Warp 0 produces, warps 1..KW consume (KW = blockDim.x/32 - 1).
// Dynamic shared memory: NS stages, NS full + NS empty mbarriers, two buffers
// of red_pp floats of cross-slab partials, 16 words of per-run activation
// maxima.
template <int WF, bool GLU, bool ACTH, bool ROUTED, int SP, int RW, int RMAX>
__global__ void __launch_bounds__(288, 1) stream_gemv_kernel(const StreamArgs a) {
  using C = StreamCfg<WF, GLU, ACTH, ROUTED, SP, RW, RMAX>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KW = (int)(blockDim.x >> 5) - 1;
  trace_begin(a.trace, a.trace_id);
  const StreamSmem m = stream_smem_init(smem, a.NS, a.stage_bytes, a.red_pp, KW);
  // The weights stream at once (they depend on nothing), but no thread lets
  // the next kernel launch before it has waited for this one's predecessor:
  // a kernel launched behind this one may read what that predecessor wrote
  // (the layer's input x) without waiting itself.
  uint32_t stage = 0;
  if (warp == 0) {
    if (lane == 0) {
      if (ROUTED) pdl_wait_prerequisites();
      cfg_produce<C>(a, SegPrior(), m.stages, m.full, m.empty, stage);
      pdl_wait_prerequisites();
      pdl_launch_dependents();
      stream_drain(a, m.empty, stage);
    } else {
      pdl_wait_prerequisites();
      pdl_launch_dependents();
    }
    __syncwarp();
  } else {
    pdl_wait_prerequisites();
    pdl_launch_dependents();
    if (a.xq) {
      // the activation planes of x for the tensor-core experts, one plane-0
      // code per row: a share of the B * K/32 blocks per CTA, one block per
      // warp, while the first stages land; each row this CTA touches first
      // gets its max |x| from all consumer warps (with xq_f8, of x's MXFP8
      // rounding, which the planes then hold)
      const int nb = a.K / 32, total = a.B * nb;
      const int lo = (int)((long long)total * blockIdx.x / gridDim.x);
      const int hi = (int)((long long)total * (blockIdx.x + 1) / gridDim.x);
      unsigned* slots = reinterpret_cast<unsigned*>(m.red);
      for (int row = lo / nb; lo < hi && row <= (hi - 1) / nb; ++row) {
        const uint16_t* xrow = a.x + (size_t)row * a.K;
        const uint32_t mx = row_amax_bits(xrow, a.K, (warp - 1) * 32 + lane, KW * 32, a.xq_f8);
        if (lane == 0) slots[warp - 1] = mx;
        consumer_sync(KW * 32);
        uint32_t amax = 0;
        for (int w = 0; w < KW; ++w) amax = max(amax, slots[w]);
        consumer_sync(KW * 32);
        const int c0 = planes_code0(__uint_as_float(amax));
        if (warp == 1 && lane == 0) a.xq_code[row] = (uint8_t)c0;
        const int b0 = max(lo, row * nb) - row * nb, b1 = min(hi, (row + 1) * nb) - row * nb;
        for (int blk = b0 + warp - 1; blk < b1; blk += KW) {
          float v = bf16_bits_to_f32(xrow[blk * 32 + lane]);
          if (a.xq_f8) v = mxfp8_round1(v);
          planes_block_c(v, lane, a.xq + (size_t)row * planes_row_bytes(a.K) + blk * 128, c0);
        }
      }
    }
    int pp = 0, rp = 0;
    cfg_consume<C>(a, SegPrior(), m.stages, m.full, m.empty, m.red, stage, pp, rp, warp - 1, KW,
                   lane);
  }
  trace_end(a.trace, a.trace_id);
}

// The x operand of an XS step (one activation row) in shared memory, by the
// KW consumer warps: the row's max |x| picks the power-of-two scale that keeps
// f16 in range, then entry i holds elements 8i..8i+7 as f16 pairs (entry
// 4 b + t: block b, lane quad t).  scratch: KW words.
template <bool F8 = false>
__device__ __forceinline__ void stage_x_operand(const uint16_t* x, int K, uint4* xs, int* xshift,
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
  // (K / 8 is a multiple of 32, so every warp runs whole iterations, and the
  // four chunks of a 32-element block sit in one lane quad)
  for (int i = ct; i < K / 8; i += cthreads) {
    const uint4 v = xr[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float4 f0 = make_float4(__uint_as_float(w[0] << 16), __uint_as_float(w[0] & 0xFFFF0000u),
                            __uint_as_float(w[1] << 16), __uint_as_float(w[1] & 0xFFFF0000u));
    float4 f1 = make_float4(__uint_as_float(w[2] << 16), __uint_as_float(w[2] & 0xFFFF0000u),
                            __uint_as_float(w[3] << 16), __uint_as_float(w[3] & 0xFFFF0000u));
    if constexpr (F8) mxfp8_round8(f0, f1);   // MXFP8 activations: the rounded values
    uint4 o;
    o.x = pack_f16x2(f0.x * sc, f0.y * sc);
    o.y = pack_f16x2(f0.z * sc, f0.w * sc);
    o.z = pack_f16x2(f1.x * sc, f1.y * sc);
    o.w = pack_f16x2(f1.z * sc, f1.w * sc);
    xs[i] = o;
  }
  consumer_sync(cthreads);   // the scratch words are free again, the operand complete
}

// Shared memory an XS step adds after the streaming carve-up: the shift word
// (16 bytes) and the operand (2 K bytes for a row of K).
__host__ __device__ inline int xs_extra_bytes(int K) { return 16 + 2 * K; }

// Routing tables of one activation row (top-k <= 32 experts, one pair each)
// in shared memory, for a routed step with RMAX = 1.  The producer brings
// them in with one round of bulk copies as soon as it knows the routing is
// final (every entry a one-row layer can use, valid or not, so the copies do
// not depend on n_active); producer and consumers then read no table from
// global memory, instead of a chain of dependent reads at each run.
struct OneRowTables {
  uint64_t bar;      // completes when the copies have landed
  uint64_t pad;
  int n_active[4];
  int expert[32];
  int off[36];
  int pair[32];
};
constexpr int kOneRowTablesBytes = (int)((sizeof(OneRowTables) + 127) / 128 * 128);
constexpr uint32_t kOneRowCopyBytes = 16 + 128 + 144 + 128;

// Producer: the copies of a's tables into t (addresses and sizes are 16-byte
// multiples; each source array's allocation extends to 256-byte multiples).
__device__ __forceinline__ void copy_one_row_tables(const StreamArgs& a, OneRowTables* t,
                                                    uint64_t policy) {
  // the tables were written through the generic proxy: order them before the
  // bulk copies' reads
  asm volatile("fence.proxy.async.global;" ::: "memory");
  mbar_arrive_expect_tx(&t->bar, kOneRowCopyBytes);
  bulk_g2s(t->n_active, a.n_active, 16, &t->bar, policy);
  bulk_g2s(t->expert, a.active_expert, 128, &t->bar, policy);
  bulk_g2s(t->off, a.active_off, 144, &t->bar, policy);
  bulk_g2s(t->pair, a.pair_list, 128, &t->bar, policy);
}

// a with its table pointers on t.
__device__ __forceinline__ StreamArgs with_one_row_tables(const StreamArgs& a, OneRowTables* t) {
  StreamArgs r = a;
  r.n_active = t->n_active;
  r.active_expert = t->expert;
  r.active_off = t->off;
  r.pair_list = t->pair;
  return r;
}

// Two steps in one launch sharing the stage ring: segment A (a dense step on
// static weights, e.g. the shared expert) then segment B (a routed step).  The
// producer streams A's weights before waiting for the predecessor kernel;
// A's consumers wait first only when A_WAITS (A's activations come from the
// predecessor).  The stage buffers are sized for the larger segment.
template <class A, class B, bool A_WAITS>
__global__ void __launch_bounds__(32 * (kMmaWarps + 1), 1)
    stream_dual_kernel(const StreamArgs a0, const StreamArgs a1_) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KW = (int)(blockDim.x >> 5) - 1;
  trace_begin(a0.trace, a0.trace_id);
  const StreamSmem m = stream_smem_init(smem, a0.NS, a0.stage_bytes, a0.red_pp, KW);
  pdl_launch_dependents();
  // an XS routed step: its x operand after the carve-up (the shift word, then
  // the operand)
  StreamArgs a1 = a1_;
  uint8_t* xe = reinterpret_cast<uint8_t*>(m.red + 2 * (size_t)a0.red_pp) + 64;
  if constexpr (B::XS) {
    a1.xs_shift = reinterpret_cast<int*>(xe);
    a1.xs = reinterpret_cast<uint4*>(xe + 16);
    xe += xs_extra_bytes(a1.K);
  }
  // one-row routed steps: the routing tables in shared memory
  constexpr bool kOneRow = B::ROUTED && B::RMAX == 1;
  OneRowTables* ort = reinterpret_cast<OneRowTables*>(xe);
  if constexpr (kOneRow) {
    if (threadIdx.x == 0) {
      mbar_init(&ort->bar, 1);
      fence_barrier_init();
    }
    __syncthreads();
  }
  uint32_t stage = 0;
  if (warp == 0) {
    if (lane == 0) {
      if (A::ROUTED) pdl_wait_prerequisites();
      cfg_produce<A>(a0, SegPrior(), m.stages, m.full, m.empty, stage);
      pdl_wait_prerequisites();
      SegPrior pr;
      if (!A::ROUTED) cfg_add_prior<A>(a0, pr);
      if constexpr (kOneRow) {
        copy_one_row_tables(a1, ort, policy_evict_last());
        mbar_wait(&ort->bar, 0, a1.status);
        cfg_produce<B>(with_one_row_tables(a1, ort), pr, m.stages, m.full, m.empty, stage);
      } else {
        cfg_produce<B>(a1, pr, m.stages, m.full, m.empty, stage);
      }
      stream_drain(a0, m.empty, stage);
    }
    __syncwarp();
  } else {
    if (A_WAITS || A::ROUTED) pdl_wait_prerequisites();
    if constexpr (B::XS) {
      // x is the layer's input (read by A as well): staged before A
      stage_x_operand(a1.x, a1.K, const_cast<uint4*>(a1.xs), const_cast<int*>(a1.xs_shift),
                      reinterpret_cast<unsigned*>(m.red), warp - 1, KW, lane,
                      (int)threadIdx.x - 32, 32 * KW);
    }
    int pp = 0, rp = 0;
    cfg_consume<A>(a0, SegPrior(), m.stages, m.full, m.empty, m.red, stage, pp, rp, warp - 1, KW,
                   lane);
    if (!(A_WAITS || A::ROUTED)) pdl_wait_prerequisites();
    SegPrior pr;
    if (!A::ROUTED) cfg_add_prior<A>(a0, pr);
    if constexpr (kOneRow) {
      mbar_wait(&ort->bar, 0, a1.status);
      cfg_consume<B>(with_one_row_tables(a1, ort), pr, m.stages, m.full, m.empty, m.red, stage, pp,
                     rp, warp - 1, KW, lane);
    } else {
      cfg_consume<B>(a1, pr, m.stages, m.full, m.empty, m.red, stage, pp, rp, warp - 1, KW, lane);
    }
  }
  trace_end(a0.trace, a0.trace_id);
}


// One row (B = 1): both expert steps of the layer in one persistent launch,
// segments A1 (shared gate/up, bf16), B1 (routed gate/up, MXFP4), A2 (shared
// down) and B2 (routed down).  The producer streams the four segments' weights
// back to back through one stage ring: the down weights do not depend on FC1's
// results, so they fill the ring while the last FC1 items are consumed and
// HBM stays busy across the FC1 -> FC2 boundary.  Each consumed segment of
// FC2 reads every CTA's FC1 outputs, so the consumers meet at two grid-wide
// barriers: each CTA adds 1 to counter 0 once its h_s rows (A1) are written
// and to counter 1 once its h rows and max |h| (B1) are; A2 waits (bounded)
// for counter 0 to reach the grid size, which it long has when a CTA gets
// there, so A2 runs while other CTAs still finish B1; B2 waits for counter 1.
// Every CTA of the grid must be resident at once: one CTA per SM and at most
// as many CTAs as SMs are free (the bounded waits turn anything else into a
// timeout status instead of a hang).
// a[0..3]: the segments' arguments (a[1], a[3] share the routing tables, which
// arrive in shared memory once top-k, the programmatic predecessor, is done);
// a[1].done_count: the two counters (zeroed by top-k); a[1].wait_ns: the
// limit of B2's wait (0: the default); skip_count: a failure-detection test
// hook (CTA 0 does not count its B1 outputs, so every CTA's wait expires).
struct StreamArgs4 {
  StreamArgs a[4];
  int skip_count;
};

template <class A1, class B1, class A2, class B2>
__global__ void __launch_bounds__(32 * (kMmaWarps + 1), 1)
    stream_expert_kernel(const StreamArgs4 args) {
  static_assert(B1::ROUTED && B1::RMAX == 1 && B2::ROUTED && B2::RMAX == 1 && B1::XS,
                "one activation row: routed steps with one column, FC1's x in shared memory");
  static_assert(!A1::ROUTED && !A2::ROUTED, "the shared expert is dense");
  static_assert(B1::F8 == B2::F8, "one activation format for both routed steps");
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KW = (int)(blockDim.x >> 5) - 1;
  const StreamArgs& a0 = args.a[0];
  trace_begin(a0.trace, 2);
  const StreamSmem m = stream_smem_init(smem, a0.NS, a0.stage_bytes, a0.red_pp, KW);
  pdl_launch_dependents();
  // after the carve-up: FC1's x operand (the shift word, then the operand),
  // then the routing tables
  StreamArgs b1 = args.a[1];
  uint8_t* xe = reinterpret_cast<uint8_t*>(m.red + 2 * (size_t)a0.red_pp) + 64;
  b1.xs_shift = reinterpret_cast<int*>(xe);
  b1.xs = reinterpret_cast<uint4*>(xe + 16);
  xe += xs_extra_bytes(b1.K);
  OneRowTables* ort = reinterpret_cast<OneRowTables*>(xe);
  if (threadIdx.x == 0) {
    mbar_init(&ort->bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  uint32_t stage = 0;
  if (warp == 0) {
    if (lane == 0) {
      cfg_produce<A1>(a0, SegPrior(), m.stages, m.full, m.empty, stage);
      pdl_wait_prerequisites();   // top-k's routing tables
      copy_one_row_tables(b1, ort, policy_evict_last());
      mbar_wait(&ort->bar, 0, b1.status);
      SegPrior p1;
      cfg_add_prior<A1>(a0, p1);
      cfg_produce<B1>(with_one_row_tables(b1, ort), p1, m.stages, m.full, m.empty, stage);
      cfg_produce<A2>(args.a[2], SegPrior(), m.stages, m.full, m.empty, stage);
      SegPrior p2;
      cfg_add_prior<A2>(args.a[2], p2);
      cfg_produce<B2>(with_one_row_tables(args.a[3], ort), p2, m.stages, m.full, m.empty, stage);
      stream_drain(a0, m.empty, stage);
    }
    __syncwarp();
  } else {
    const int ct = (int)threadIdx.x - 32, cthreads = 32 * KW, kw = warp - 1;
    // x is the layer's input (read by A1 as well): staged before A1
    stage_x_operand<B1::F8>(b1.x, b1.K, const_cast<uint4*>(b1.xs), const_cast<int*>(b1.xs_shift),
                            reinterpret_cast<unsigned*>(m.red), kw, KW, lane, ct, cthreads);
    int pp = 0, rp = 0;
    unsigned* const count = b1.done_count;
    cfg_consume<A1>(a0, SegPrior(), m.stages, m.full, m.empty, m.red, stage, pp, rp, kw, KW, lane);
    // this CTA's h_s rows are written (the barrier orders every consumer's
    // stores before the counting thread's fence)
    consumer_sync(cthreads);
    if (ct == 0) {
      __threadfence();
      atomicAdd(count, 1u);
    }
    pdl_wait_prerequisites();
    SegPrior p1;
    cfg_add_prior<A1>(a0, p1);
    mbar_wait(&ort->bar, 0, b1.status);
    cfg_consume<B1>(with_one_row_tables(b1, ort), p1, m.stages, m.full, m.empty, m.red, stage, pp,
                    rp, kw, KW, lane);
    // every CTA's h_s (for A2); this CTA's h rows and max |h| are written
    if (ct == 0) {
      wait_count_at_least(count, gridDim.x, b1.status, kWaitLimitNs);
      __threadfence();
    }
    consumer_sync(cthreads);
    if (ct == 0) {
      if (b1.trace) atomicMax(b1.trace + 8 + 2, global_ns());
      if (b1.trace) atomicMin(b1.trace + 3, global_ns());
      __threadfence();
      if (!(args.skip_count && blockIdx.x == 0)) atomicAdd(count + 1, 1u);
    }
    cfg_consume<A2>(args.a[2], SegPrior(), m.stages, m.full, m.empty, m.red, stage, pp, rp, kw, KW,
                    lane);
    // every CTA's h rows and max |h| (for B2)
    if (ct == 0) {
      wait_count_at_least(count + 1, gridDim.x, b1.status, b1.wait_ns ? b1.wait_ns : kWaitLimitNs);
      __threadfence();
    }
    consumer_sync(cthreads);
    SegPrior p2;
    cfg_add_prior<A2>(args.a[2], p2);
    cfg_consume<B2>(with_one_row_tables(args.a[3], ort), p2, m.stages, m.full, m.empty, m.red,
                    stage, pp, rp, kw, KW, lane);
  }
  trace_end(a0.trace, 3);
}

}  // namespace moe
