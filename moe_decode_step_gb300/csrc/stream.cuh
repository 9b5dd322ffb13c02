// Persistent streaming GEMV: one producer thread feeds a ring of shared-memory
// stages with bulk copies (cp.async.bulk + mbarrier), consumer warps compute
// from shared memory with their activation slice in registers.
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
// rows are that expert's (row, slot) pairs, taken R <= RMAX at a time.  Items
// are dealt to CTAs round-robin, so the producer knows its whole sequence and
// runs ahead across item boundaries; the only coupling is the stage ring.
// Consumer warps split K (warp w owns a K slab); partial sums stay in
// registers for the whole item, then a butterfly reduce-scatter and one
// shared-memory combine across the K slabs, in a fixed order (deterministic).
#pragma once

#include "common.cuh"

namespace moe {

enum { kWfMx = 0, kWfBf16 = 1 };

struct StreamArgs {
  const uint8_t* q;          // MXFP4 nibbles (or bf16 weights) of matrix 0
  const uint8_t* s;          // MXFP4 scale bytes of matrix 0 (unused for bf16)
  size_t q_stride, s_stride; // bytes between experts (routed)
  int K;                     // row length in elements
  int N;                     // output rows (gate/up: row pairs, up row = N + i)
  int k;                     // top-k: pair p belongs to activation row p / k (routed)
  int B;                     // dense steps: activation rows
  const uint16_t* x;         // bf16 activations [rows][K]
  const int* x_shift;        // f16 scaling shift per x row (MXFP4 x-activation steps)
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
  unsigned long long* trace; // optional kernel trace (see trace_begin), or null
  int trace_id;
};

// Elements per lane and activation registers per row, by format.
template <int WF, bool ACTH>
struct StreamShape {
  static constexpr int EPL = ACTH ? 16 : 32;                 // K elements per lane
  static constexpr int AW = (WF == kWfBf16 && ACTH) ? 16 : EPL / 2;  // u32 registers per row
  static constexpr int WARP_K = 32 * EPL;                    // K elements per consumer warp
};

// Bytes of one stage holding `rows` rows (per half for gate/up).
__host__ __device__ inline size_t stream_rows_bytes(int wf, int K, int rows) {
  return wf == kWfMx ? (size_t)rows * (K / 2 + K / 32) : (size_t)rows * K * 2;
}

// ---- activation slices (registers) --------------------------------------

// MXFP4 x-activation: 32 elements [blk*32, +32) of a bf16 row as f16x2,
// scaled by 2^-shift.
__device__ __forceinline__ void act_load_mx_x(const uint16_t* row, int blk, bool ok, int shift,
                                              uint32_t (&a)[16]) {
  if (!ok) {
#pragma unroll
    for (int t = 0; t < 16; ++t) a[t] = 0;
    return;
  }
  const float sc = pow2f(-shift);
  const uint4* p = reinterpret_cast<const uint4*>(row + blk * 32);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 v = p[c];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int t = 0; t < 4; ++t)
      a[c * 4 + t] = pack_f16x2(__uint_as_float(w[t] << 16) * sc,
                                __uint_as_float(w[t] & 0xFFFF0000u) * sc);
  }
}

// Raw bf16 pairs of the 32-element slice [blk*32, +32) of an x row.
__device__ __forceinline__ void act_load_raw_x(const uint16_t* row, int blk, bool ok,
                                               uint32_t (&a)[16]) {
  const uint4* p = reinterpret_cast<const uint4*>(row + blk * 32);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 v = ok ? p[c] : make_uint4(0, 0, 0, 0);
    a[c * 4 + 0] = v.x;
    a[c * 4 + 1] = v.y;
    a[c * 4 + 2] = v.z;
    a[c * 4 + 3] = v.w;
  }
}

// bf16 pairs -> f16x2 scaled by 2^-shift, in place.
__device__ __forceinline__ void act_convert_mx_x(int shift, uint32_t (&a)[16]) {
  const float sc = pow2f(-shift);
#pragma unroll
  for (int t = 0; t < 16; ++t)
    a[t] = pack_f16x2(__uint_as_float(a[t] << 16) * sc, __uint_as_float(a[t] & 0xFFFF0000u) * sc);
}

// MXFP4 h-activation: 16 elements [hb*16, +16) of an fp32 row as f16x2.
__device__ __forceinline__ void act_load_mx_h(const float* row, int hb, bool ok, int shift,
                                              uint32_t (&a)[8]) {
  if (!ok) {
#pragma unroll
    for (int t = 0; t < 8; ++t) a[t] = 0;
    return;
  }
  const float sc = pow2f(-shift);
  const float4* p = reinterpret_cast<const float4*>(row + hb * 16);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const float4 v = __ldcg(p + c);
    a[c * 2 + 0] = pack_f16x2(v.x * sc, v.y * sc);
    a[c * 2 + 1] = pack_f16x2(v.z * sc, v.w * sc);
  }
}

// bf16 x-activation for bf16 weights: elements slab + q*256 + lane*8 + [0,8),
// q < 4, kept as raw bf16 pairs.
__device__ __forceinline__ void act_load_bf_x(const uint16_t* row, int slab, int lane, int K,
                                              uint32_t (&a)[16]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int e = slab + q * 256 + lane * 8;
    const uint4 v = e < K ? *reinterpret_cast<const uint4*>(row + e) : make_uint4(0, 0, 0, 0);
    a[q * 4 + 0] = v.x;
    a[q * 4 + 1] = v.y;
    a[q * 4 + 2] = v.z;
    a[q * 4 + 3] = v.w;
  }
}

// fp32 h-activation for bf16 weights: elements slab + q*256 + lane*8 + [0,8),
// q < 2, kept as fp32 bit patterns.
__device__ __forceinline__ void act_load_bf_h(const float* row, int slab, int lane, int K,
                                              uint32_t (&a)[16]) {
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int e = slab + q * 256 + lane * 8;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const float4 v = e < K ? __ldcg(reinterpret_cast<const float4*>(row + e) + c)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
      a[q * 8 + c * 4 + 0] = __float_as_uint(v.x);
      a[q * 8 + c * 4 + 1] = __float_as_uint(v.y);
      a[q * 8 + c * 4 + 2] = __float_as_uint(v.z);
      a[q * 8 + c * 4 + 3] = __float_as_uint(v.w);
    }
  }
}

// ---- one weight row (in shared memory) against R activation slices -------

// MXFP4, 32-element block per lane: nibbles at q + blk*16, scale byte at s + blk.
template <int R>
__device__ __forceinline__ void row_dot_mx_x(const uint8_t* q, const uint8_t* s, int blk, bool ok,
                                             const uint32_t (&a)[R][16], float (&out)[R]) {
#pragma unroll
  for (int r = 0; r < R; ++r) out[r] = 0.f;
  if (!ok) return;
  const uint4 wq = *reinterpret_cast<const uint4*>(q + blk * 16);
  const float sc = e8m0_to_f32(s[blk]);
  const uint32_t words[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t hq[4];
    e2m1x8_to_f16x2(words[w], hq);
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const uint32_t xv = a[r][w * 4 + t];
        out[r] = fma2_f16s(hq[t], (unsigned short)(xv & 0xFFFFu), (unsigned short)(xv >> 16),
                           out[r]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) out[r] *= sc;
}

// MXFP4, 16-element half block per lane: nibbles at q + hb*8, scale at s + hb/2.
template <int R>
__device__ __forceinline__ void row_dot_mx_h(const uint8_t* q, const uint8_t* s, int hb, bool ok,
                                             const uint32_t (&a)[R][8], float (&out)[R]) {
#pragma unroll
  for (int r = 0; r < R; ++r) out[r] = 0.f;
  if (!ok) return;
  const uint2 wq = *reinterpret_cast<const uint2*>(q + hb * 8);
  const float sc = e8m0_to_f32(s[hb >> 1]);
  const uint32_t words[2] = {wq.x, wq.y};
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    uint32_t hq[4];
    e2m1x8_to_f16x2(words[w], hq);
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const uint32_t xv = a[r][w * 4 + t];
        out[r] = fma2_f16s(hq[t], (unsigned short)(xv & 0xFFFFu), (unsigned short)(xv >> 16),
                           out[r]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) out[r] *= sc;
}

// bf16 row (as bytes), x activation: 4 chunks of 8 at slab + q*256 + lane*8.
template <int R>
__device__ __forceinline__ void row_dot_bf_x(const uint8_t* wrow, int slab, int lane, int K,
                                             const uint32_t (&a)[R][16], float (&out)[R]) {
#pragma unroll
  for (int r = 0; r < R; ++r) out[r] = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int e = slab + q * 256 + lane * 8;
    if (e < K) {
      const uint4 v = *reinterpret_cast<const uint4*>(wrow + (size_t)e * 2);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float acc = out[r];
        acc = fma2_bf16(v.x, a[r][q * 4 + 0], acc);
        acc = fma2_bf16(v.y, a[r][q * 4 + 1], acc);
        acc = fma2_bf16(v.z, a[r][q * 4 + 2], acc);
        acc = fma2_bf16(v.w, a[r][q * 4 + 3], acc);
        out[r] = acc;
      }
    }
  }
}

// bf16 row, fp32 activation: 2 chunks of 8 at slab + q*256 + lane*8; the bf16
// weights widen exactly to fp32.
template <int R>
__device__ __forceinline__ void row_dot_bf_h(const uint8_t* wrow, int slab, int lane, int K,
                                             const uint32_t (&a)[R][16], float (&out)[R]) {
#pragma unroll
  for (int r = 0; r < R; ++r) out[r] = 0.f;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int e = slab + q * 256 + lane * 8;
    if (e < K) {
      const uint4 v = *reinterpret_cast<const uint4*>(wrow + (size_t)e * 2);
      const uint32_t ww[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float s0 = out[r], s1 = 0.f;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          s0 = fmaf(__uint_as_float(ww[t] << 16), __uint_as_float(a[r][q * 8 + 2 * t]), s0);
          s1 = fmaf(__uint_as_float(ww[t] & 0xFFFF0000u), __uint_as_float(a[r][q * 8 + 2 * t + 1]),
                    s1);
        }
        out[r] = s0 + s1;
      }
    }
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
  return ROUTED ? __ldcg(a.n_active) * tiles : tiles;
}

template <bool ROUTED, int RW>
__device__ __forceinline__ StreamItem stream_item(const StreamArgs& a, int it, int tiles) {
  StreamItem m;
  if (ROUTED) {
    const int slot = it / tiles;
    m.e = __ldcg(a.active_expert + slot);
    m.p0 = __ldcg(a.active_off + slot);
    m.pr = __ldcg(a.active_off + slot + 1) - m.p0;
    m.row0 = (it % tiles) * RW;
  } else {
    m.e = 0;
    m.p0 = 0;
    m.pr = a.B;
    m.row0 = it * RW;
  }
  return m;
}

template <int RMAX>
__device__ __forceinline__ int stream_pass_rows(int left) {
  return (RMAX >= 4 && left >= 4) ? 4 : ((RMAX >= 2 && left >= 2) ? 2 : 1);
}

// CTA c owns the contiguous item range [lo, hi).  Items are ordered expert by
// expert, so a range is a few runs of tiles that share one activation set:
// the consumers load activations once per (run, pass), not once per item.
__device__ __forceinline__ void stream_range(int n_items, int& lo, int& hi) {
  lo = (int)(((long long)blockIdx.x * n_items) / gridDim.x);
  hi = (int)(((long long)(blockIdx.x + 1) * n_items) / gridDim.x);
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
// step, continuing the CTA's running stage counter.
template <int WF, bool GLU, bool ROUTED, int SP, int RW, int RMAX>
__device__ __forceinline__ void stream_produce_range(const StreamArgs& a, int lo, int hi, int tiles,
                                                     uint8_t* stages, uint64_t* full,
                                                     uint64_t* empty, uint32_t& stage) {
  constexpr int G = GLU ? 2 : 1;
  constexpr int SPI = RW / SP;
  const uint64_t pol = policy_evict_first();
  const size_t half_bytes = WF == kWfMx ? (size_t)SP * (a.K / 2) : (size_t)SP * a.K * 2;
  const size_t s_off = (size_t)G * half_bytes;
  for (int it0 = lo; it0 < hi;) {
    const int run_end = stream_run_end<ROUTED>(it0, hi, tiles);
    const StreamItem m = stream_item<ROUTED, RW>(a, it0, tiles);
    const uint8_t* qe = a.q + (size_t)m.e * a.q_stride;
    for (int done = 0; done < m.pr; done += stream_pass_rows<RMAX>(m.pr - done)) {
      for (int it = it0; it < run_end; ++it) {
        const int row0 = stream_row0<ROUTED, RW>(it, tiles);
        for (int st = 0; st < SPI; ++st, ++stage) {
          const int buf = (int)(stage % (uint32_t)a.NS);
          const uint32_t use = stage / (uint32_t)a.NS;
          if (use > 0) mbar_wait(&empty[buf], (use - 1) & 1u, a.status);
          const int r0 = row0 + st * SP;
          const int nv = max(0, min(SP, a.N - r0));
          uint8_t* dst = stages + (size_t)buf * a.stage_bytes;
          if (WF == kWfMx) {
            const uint8_t* se = a.s + (size_t)m.e * a.s_stride;
            const uint32_t qb = (uint32_t)nv * (a.K / 2), sb = (uint32_t)nv * (a.K / 32);
            mbar_arrive_expect_tx(&full[buf], G * (qb + sb));
            if (nv > 0) {
              bulk_g2s(dst, qe + (size_t)r0 * (a.K / 2), qb, &full[buf], pol);
              bulk_g2s(dst + s_off, se + (size_t)r0 * (a.K / 32), sb, &full[buf], pol);
              if (GLU) {
                bulk_g2s(dst + half_bytes, qe + (size_t)(a.N + r0) * (a.K / 2), qb, &full[buf],
                         pol);
                bulk_g2s(dst + s_off + (size_t)SP * (a.K / 32),
                         se + (size_t)(a.N + r0) * (a.K / 32), sb, &full[buf], pol);
              }
            }
          } else {
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

template <int WF, bool ACTH, bool ROUTED>
__device__ __forceinline__ int stream_shift(const StreamArgs& a, int pid) {
  if (WF != kWfMx) return 0;
  if (ACTH) return f16_shift_for_amax(__uint_as_float(__ldcg(a.h_amax + pid)));
  return __ldcg(a.x_shift + stream_x_row<ROUTED>(a, pid));
}

// Consumers: one pass of R activation rows over the run [it0, run_end) of
// items that share them.  Activation slices, pair ids and scale shifts are
// loaded once; every item then streams its SPI stages, reduces and finalises.
template <int WF, bool GLU, bool ACTH, bool ROUTED, int SP, int RW, int R>
__device__ __forceinline__ void stream_consume_run(const StreamArgs& a, const StreamItem& m,
                                                   int done, int it0, int run_end, int tiles,
                                                   uint8_t* stages, uint64_t* full,
                                                   uint64_t* empty, float* red, uint32_t& stage,
                                                   int& pp, int& rp, int kw, int KW, int lane) {
  using Sh = StreamShape<WF, ACTH>;
  constexpr int G = GLU ? 2 : 1;
  constexpr int SPI = RW / SP;
  constexpr int V = RW * G * R;
  constexpr int VM = V < 32 ? V : 32;
  constexpr int M = VM == 1 ? 0 : VM == 2 ? 1 : VM == 4 ? 2 : VM == 8 ? 3 : VM == 16 ? 4 : 5;
  const size_t half_bytes = WF == kWfMx ? (size_t)SP * (a.K / 2) : (size_t)SP * a.K * 2;
  const size_t s_off = (size_t)G * half_bytes;
  const int blk = kw * 32 + lane;
  const bool ok = blk * Sh::EPL < a.K;
  const int slab = kw * Sh::WARP_K;
  const int cthreads = KW * 32;
  const int ct = (int)threadIdx.x - 32;

  int pid[R], shift[R];
  uint32_t act[R][Sh::AW];
  if constexpr (WF == kWfMx && !ACTH) {
    // x rows: the f16 scaling shift needs the whole row's max |x|; the KW
    // consumer warps together hold the whole row, so reduce across them.
    unsigned* s_amax = reinterpret_cast<unsigned*>(red + (size_t)2 * 64 * KW);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      pid[r] = ROUTED ? __ldcg(a.pair_list + m.p0 + done + r) : done + r;
      act_load_raw_x(a.x + (size_t)stream_x_row<ROUTED>(a, pid[r]) * a.K, blk, ok, act[r]);
      uint32_t mx = 0;
#pragma unroll
      for (int q = 0; q < 16; ++q)
        mx = max(mx, max(act[r][q] & 0x7FFFu, (act[r][q] >> 16) & 0x7FFFu));
      mx = __reduce_max_sync(0xffffffffu, mx);
      if (lane == 0) atomicMax(&s_amax[(rp & 1) * 4 + r], mx);
    }
    consumer_sync(KW * 32);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      shift[r] = f16_shift_for_amax(bf16_bits_to_f32(s_amax[(rp & 1) * 4 + r]));
      act_convert_mx_x(shift[r], act[r]);
    }
    // the other parity's slots are free: every consumer is past this barrier
    if (kw == 0 && lane < 4) s_amax[((rp & 1) ^ 1) * 4 + lane] = 0u;
    rp ^= 1;
  } else {
#pragma unroll
  for (int r = 0; r < R; ++r) {
    pid[r] = ROUTED ? __ldcg(a.pair_list + m.p0 + done + r) : done + r;
    shift[r] = stream_shift<WF, ACTH, ROUTED>(a, pid[r]);
    if constexpr (WF == kWfMx && ACTH) {
      act_load_mx_h(a.h + (size_t)pid[r] * a.K, blk, ok, shift[r], act[r]);
    } else if constexpr (!ACTH) {
      act_load_bf_x(a.x + (size_t)stream_x_row<ROUTED>(a, pid[r]) * a.K, slab, lane, a.K, act[r]);
    } else {
      act_load_bf_h(a.h + (size_t)pid[r] * a.K, slab, lane, a.K, act[r]);
    }
  }
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
      for (int rr = 0; rr < SP; ++rr) {
        const int j = st * SP + rr;
#pragma unroll
        for (int gu = 0; gu < G; ++gu) {
          float o[R];
          if constexpr (WF == kWfMx) {
            const uint8_t* qrow = sb + gu * half_bytes + (size_t)rr * (a.K / 2);
            const uint8_t* srow = sb + s_off + (size_t)(gu * SP + rr) * (a.K / 32);
            if constexpr (ACTH) row_dot_mx_h<R>(qrow, srow, blk, ok, act, o);
            else row_dot_mx_x<R>(qrow, srow, blk, ok, act, o);
          } else {
            const uint8_t* wrow = sb + gu * half_bytes + (size_t)rr * a.K * 2;
            if constexpr (ACTH) row_dot_bf_h<R>(wrow, slab, lane, a.K, act, o);
            else row_dot_bf_x<R>(wrow, slab, lane, a.K, act, o);
          }
#pragma unroll
          for (int r = 0; r < R; ++r) v[(j * R + r) * G + gu] = o[r];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[buf]);
      ++stage;
    }

    // combine: lanes -> one value per lane group, then K slabs through shared memory
    float second;
    const float first = stream_reduce<V>(v, lane, second);
    float* rb = red + (size_t)pp * 64 * KW;
    if ((lane & ((1 << (5 - M)) - 1)) == 0) {
      const int vi = lane >> (5 - M);
      rb[vi * KW + kw] = first;
      if (V > 32) rb[(32 + vi) * KW + kw] = second;
    }
    consumer_sync(cthreads);
    for (int t = ct; t < RW * R; t += cthreads) {
      const int j = t / R, r = t % R;
      const int row = row0 + j;
      if (row >= a.N) continue;
      int p = pid[0], sh = shift[0];
#pragma unroll
      for (int q = 1; q < R; ++q)
        if (q == r) { p = pid[q]; sh = shift[q]; }
      const float back = pow2f(sh);
      float* dst = a.out + (size_t)p * a.N + row;
      if constexpr (GLU) {
        const float* pg = rb + ((j * R + r) * 2) * KW;
        float g = 0.f, u = 0.f;
        for (int w = 0; w < KW; ++w) { g += pg[w]; u += pg[KW + w]; }
        g *= back;
        u *= back;
        const float hv = g / (1.0f + expf(-g)) * u;
        *dst = hv;
        if (a.out_amax) atomicMax(a.out_amax + p, __float_as_uint(fabsf(hv)));
      } else {
        const float* pv = rb + (j * R + r) * KW;
        float acc = 0.f;
        for (int w = 0; w < KW; ++w) acc += pv[w];
        *dst = acc * back;
      }
    }
    pp ^= 1;
  }
}

// Consumers: items [lo, hi) of one step, run by run, pass by pass.
template <int WF, bool GLU, bool ACTH, bool ROUTED, int SP, int RW, int RMAX>
__device__ __forceinline__ void stream_consume_range(const StreamArgs& a, int lo, int hi, int tiles,
                                                     uint8_t* stages, uint64_t* full,
                                                     uint64_t* empty, float* red, uint32_t& stage,
                                                     int& pp, int& rp, int kw, int KW, int lane) {
  for (int it0 = lo; it0 < hi;) {
    const int run_end = stream_run_end<ROUTED>(it0, hi, tiles);
    const StreamItem m = stream_item<ROUTED, RW>(a, it0, tiles);
    for (int done = 0; done < m.pr;) {
      const int R = stream_pass_rows<RMAX>(m.pr - done);
      if (R == 1) {
        stream_consume_run<WF, GLU, ACTH, ROUTED, SP, RW, 1>(a, m, done, it0, run_end, tiles,
                                                              stages, full, empty, red, stage, pp,
                                                              rp, kw, KW, lane);
      } else if constexpr (RMAX >= 2) {
        if (R == 2) {
          stream_consume_run<WF, GLU, ACTH, ROUTED, SP, RW, 2>(a, m, done, it0, run_end, tiles,
                                                                stages, full, empty, red, stage,
                                                                pp, rp, kw, KW, lane);
        } else if constexpr (RMAX >= 4) {
          stream_consume_run<WF, GLU, ACTH, ROUTED, SP, RW, 4>(a, m, done, it0, run_end, tiles,
                                                                stages, full, empty, red, stage,
                                                                pp, rp, kw, KW, lane);
        }
      }
      done += R;
    }
    it0 = run_end;
  }
}

// Compile-time description of one streaming step.
template <int WF_, bool GLU_, bool ACTH_, bool ROUTED_, int SP_, int RW_, int RMAX_>
struct StreamCfg {
  static constexpr int WF = WF_;
  static constexpr bool GLU = GLU_, ACTH = ACTH_, ROUTED = ROUTED_;
  static constexpr int SP = SP_, RW = RW_, RMAX = RMAX_;
  static_assert(RW % SP == 0, "an item is a whole number of stages");
};

template <class C>
__device__ __forceinline__ void cfg_produce(const StreamArgs& a, uint8_t* stages, uint64_t* full,
                                            uint64_t* empty, uint32_t& stage) {
  int tiles, lo, hi;
  const int n = stream_n_items<C::ROUTED, C::RW>(a, tiles);
  stream_range(n, lo, hi);
  stream_produce_range<C::WF, C::GLU, C::ROUTED, C::SP, C::RW, C::RMAX>(a, lo, hi, tiles, stages,
                                                                       full, empty, stage);
}

template <class C>
__device__ __forceinline__ void cfg_consume(const StreamArgs& a, uint8_t* stages, uint64_t* full,
                                            uint64_t* empty, float* red, uint32_t& stage, int& pp,
                                            int& rp, int kw, int KW, int lane) {
  int tiles, lo, hi;
  const int n = stream_n_items<C::ROUTED, C::RW>(a, tiles);
  stream_range(n, lo, hi);
  stream_consume_range<C::WF, C::GLU, C::ACTH, C::ROUTED, C::SP, C::RW, C::RMAX>(
      a, lo, hi, tiles, stages, full, empty, red, stage, pp, rp, kw, KW, lane);
}

// Shared-memory carve-up common to both kernels.
struct StreamSmem {
  uint8_t* stages;
  uint64_t* full;
  uint64_t* empty;
  float* red;
};

__device__ __forceinline__ StreamSmem stream_smem_init(uint8_t* smem, int NS, int stage_bytes,
                                                       int KW) {
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
  if (threadIdx.x < 8) reinterpret_cast<unsigned*>(m.red + (size_t)2 * 64 * KW)[threadIdx.x] = 0u;
  __syncthreads();
  return m;
}

// Single step.  Warp 0 produces, warps 1..KW consume (KW = blockDim.x/32 - 1).
// Dynamic shared memory: NS stages, NS full + NS empty mbarriers, 2 x 64 x KW
// floats of cross-slab partials, 8 words of per-run activation maxima.
template <int WF, bool GLU, bool ACTH, bool ROUTED, int SP, int RW, int RMAX>
__global__ void __launch_bounds__(288, 1) stream_gemv_kernel(const StreamArgs a) {
  using C = StreamCfg<WF, GLU, ACTH, ROUTED, SP, RW, RMAX>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KW = (int)(blockDim.x >> 5) - 1;
  trace_begin(a.trace, a.trace_id);
  const StreamSmem m = stream_smem_init(smem, a.NS, a.stage_bytes, KW);
  pdl_launch_dependents();
  uint32_t stage = 0;
  if (warp == 0) {
    if (lane == 0) {
      if (ROUTED) pdl_wait_prerequisites();
      cfg_produce<C>(a, m.stages, m.full, m.empty, stage);
      stream_drain(a, m.empty, stage);
    }
    __syncwarp();
  } else {
    pdl_wait_prerequisites();
    int pp = 0, rp = 0;
    cfg_consume<C>(a, m.stages, m.full, m.empty, m.red, stage, pp, rp, warp - 1, KW, lane);
  }
  trace_end(a.trace, a.trace_id);
}

// Two steps in one launch sharing the stage ring: segment A (a dense step on
// static weights, e.g. the shared expert) then segment B (a routed step).  The
// producer streams A's weights before waiting for the predecessor kernel;
// A's consumers wait first only when A_WAITS (A's activations come from the
// predecessor).  The stage buffers are sized for the larger segment.
template <class A, class B, bool A_WAITS>
__global__ void __launch_bounds__(288, 1) stream_dual_kernel(const StreamArgs a0,
                                                             const StreamArgs a1) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KW = (int)(blockDim.x >> 5) - 1;
  trace_begin(a0.trace, a0.trace_id);
  const StreamSmem m = stream_smem_init(smem, a0.NS, a0.stage_bytes, KW);
  pdl_launch_dependents();
  uint32_t stage = 0;
  if (warp == 0) {
    if (lane == 0) {
      if (A::ROUTED) pdl_wait_prerequisites();
      cfg_produce<A>(a0, m.stages, m.full, m.empty, stage);
      pdl_wait_prerequisites();
      cfg_produce<B>(a1, m.stages, m.full, m.empty, stage);
      stream_drain(a0, m.empty, stage);
    }
    __syncwarp();
  } else {
    if (A_WAITS || A::ROUTED) pdl_wait_prerequisites();
    int pp = 0, rp = 0;
    cfg_consume<A>(a0, m.stages, m.full, m.empty, m.red, stage, pp, rp, warp - 1, KW, lane);
    pdl_wait_prerequisites();
    cfg_consume<B>(a1, m.stages, m.full, m.empty, m.red, stage, pp, rp, warp - 1, KW, lane);
  }
  trace_end(a0.trace, a0.trace_id);
}

}  // namespace moe
