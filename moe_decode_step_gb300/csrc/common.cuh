// Device helpers shared by the MoE decode kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

constexpr int kWarp = 32;

// ---------------------------------------------------------------------------
// Loads.  Weights are streamed once per forward: no L1 allocation.  Routing
// tables and activations written by an earlier kernel are read with plain
// coherent loads (ld.global.cg / default), never the non-coherent path.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream_u128(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint2 ld_stream_u64(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ld_stream_u8(const uint8_t* p) {
  uint16_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// Routing-table entries live either in global memory (written by top-k, an
// earlier kernel the reader has waited for) or in the CTA's shared memory (a
// copy whose arrival the reader has waited for): either way final before the
// read, so a plain generic load.
__device__ __forceinline__ int ld_tab(const int* p) { return *p; }

// A word other CTAs of the same launch wrote before a release the reader has
// acquired: a relaxed load at GPU scope (bypasses a possibly stale L1 line).
__device__ __forceinline__ int ld_relaxed_gpu(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// Flag and counter accesses between CTAs of one or two kernels in flight.
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---------------------------------------------------------------------------
// MXFP4 decode.  cvt.rn.f16x2.e2m1x2 turns one byte (two E2M1 codes) into an
// f16x2; every E2M1 value is exact in f16.  E8M0 byte -> 2^(s-127) as fp32
// (byte 0 is the subnormal 2^-127).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
}

// D += A * B on the tensor cores: one m16n8k16 tile, f16 operands, fp32
// accumulators, in the register fragments of PTX mma.sync .row.col: with
// g = lane/4, t = lane%4, a0/a2 hold row g at k = 2t, 2t+1 / 2t+8, 2t+9 and
// a1/a3 the same k of row g+8; b0/b1 hold column g at k = 2t, 2t+1 /
// 2t+8, 2t+9; d0, d1 are (row g, columns 2t, 2t+1), d2, d3 the same for
// row g+8.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The same with zero accumulators: D = A * B.
__device__ __forceinline__ void mma_f16_16816_zero(float (&d)[4], uint32_t a0, uint32_t a1,
                                                   uint32_t a2, uint32_t a3, uint32_t b0,
                                                   uint32_t b1) {
  const float z = 0.f;
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(z));
}

__device__ __forceinline__ float e8m0_to_f32(uint32_t s) {
  return s ? __uint_as_float(s << 23) : __uint_as_float(0x00400000u);
}

__device__ __forceinline__ float f16_lo(uint32_t h2) {
  float f;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.f32.f16 %0, l;\n\t}" : "=f"(f) : "r"(h2));
  return f;
}
__device__ __forceinline__ float f16_hi(uint32_t h2) {
  float f;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.f32.f16 %0, h;\n\t}" : "=f"(f) : "r"(h2));
  return f;
}

// c + a.lo*b.lo + a.hi*b.hi with f16 inputs, exact products, fp32 accumulate.
__device__ __forceinline__ float fma2_f16(uint32_t a, uint32_t b, float c) {
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.f16 %0, al, bl, %0;\n\tfma.rn.f32.f16 %0, ah, bh, %0;\n\t}"
      : "+f"(c)
      : "r"(a), "r"(b));
  return c;
}

// Same with the activation already split into its two f16 halves (lets the
// compiler keep them in 16-bit registers across rows).
__device__ __forceinline__ float fma2_f16s(uint32_t a, unsigned short bl, unsigned short bh,
                                           float c) {
  asm("{\n\t.reg .b16 al, ah;\n\tmov.b32 {al, ah}, %1;\n\t"
      "fma.rn.f32.f16 %0, al, %2, %0;\n\tfma.rn.f32.f16 %0, ah, %3, %0;\n\t}"
      : "+f"(c)
      : "r"(a), "h"(bl), "h"(bh));
  return c;
}

// Same with bf16 inputs.
__device__ __forceinline__ float fma2_bf16(uint32_t a, uint32_t b, float c) {
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, al, bl, %0;\n\tfma.rn.f32.bf16 %0, ah, bh, %0;\n\t}"
      : "+f"(c)
      : "r"(a), "r"(b));
  return c;
}

// Nearest E2M1 magnitude code for a >= 0 (E2M1 magnitudes 0, .5, 1, 1.5, 2,
// 3, 4, 6 are codes 0..7); the midpoints 0.25, 1.25, 2.5, 5 round down (to the
// even codes 0, 2, 4, 6) and 0.75, 1.75, 3.5 round up (to the even codes 2, 4,
// 6).  Values above 5 become 6 (code 7), which also saturates everything larger.
__host__ __device__ inline uint32_t e2m1_magnitude_code(float a) {
  return (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) +
         (uint32_t)(a >= 1.75f) + (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) +
         (uint32_t)(a > 5.0f);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// fp32 -> bf16 bits, round to nearest even (inputs here are finite).
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
  return r;
}

// Two fp32 -> f16x2 (lo = a, hi = b), round to nearest even.
__device__ __forceinline__ uint32_t pack_f16x2(float a, float b) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}

// 2^e for integer e in [-126, 127].
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

// ---- MXFP8 activations (OCP MX v1.0: E4M3 elements, one E8M0 scale per 32)

// Scale exponent of a block of activations with maximum magnitude amax:
// floor(log2 amax) - 8 (8: the exponent of 256, E4M3's largest power of two),
// -127 for amax 0 or subnormal (where the clamp to [-127, 127] lands anyway).
__device__ __forceinline__ int e4m3_block_exp(float amax) {
  const int be = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
  return be == 0 ? -127 : max(-127, be - 127 - 8);
}

// 2^e for e in [-127, 127], exactly (2^-127 is a subnormal float).
__device__ __forceinline__ float pow2_e8m0(int e) {
  return e == -127 ? __uint_as_float(0x00400000u) : __uint_as_float((uint32_t)(e + 127) << 23);
}

// Two floats (already divided by their block scale) to their nearest E4M3
// values: cvt.rn.satfinite.e4m3x2.f32 (nearest, ties to even, magnitudes past
// 448 saturating: the OCP MX conversion with clamping), then back through
// cvt.rn.f16x2.e4m3x2 (exact).
__device__ __forceinline__ void e4m3x2_round(float& a, float& b) {
  float ra, rb;
  asm("{\n\t.reg .b16 c, lo, hi;\n\t.reg .b32 h;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 c, %3, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 h, c;\n\t"
      "mov.b32 {lo, hi}, h;\n\t"
      "cvt.f32.f16 %0, lo;\n\tcvt.f32.f16 %1, hi;\n\t}"
      : "=f"(ra), "=f"(rb)
      : "f"(a), "f"(b));
  a = ra;
  b = rb;
}

// MXFP8 rounding of one 32-element block held by a lane quad (lanes 4g..4g+3,
// 8 elements each; every lane of the warp takes part): scale 2^e with
// e = floor(log2 max |v|) - 8 over the block (e4m3_block_exp), each element
// replaced by its nearest E4M3 value times 2^e.  Exact in fp32.
__device__ __forceinline__ void mxfp8_round8(float4& v0, float4& v1) {
  float mx = fmaxf(fmaxf(fmaxf(fabsf(v0.x), fabsf(v0.y)), fmaxf(fabsf(v0.z), fabsf(v0.w))),
                   fmaxf(fmaxf(fabsf(v1.x), fabsf(v1.y)), fmaxf(fabsf(v1.z), fabsf(v1.w))));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  const int e = e4m3_block_exp(mx);
  const float inv = pow2_e8m0(-e), sc = pow2_e8m0(e);
  float f[8] = {v0.x * inv, v0.y * inv, v0.z * inv, v0.w * inv,
                v1.x * inv, v1.y * inv, v1.z * inv, v1.w * inv};
#pragma unroll
  for (int j = 0; j < 8; j += 2) e4m3x2_round(f[j], f[j + 1]);
  v0 = make_float4(f[0] * sc, f[1] * sc, f[2] * sc, f[3] * sc);
  v1 = make_float4(f[4] * sc, f[5] * sc, f[6] * sc, f[7] * sc);
}

// Exponent shift that keeps |v| <= amax below 2^15 after scaling by 2^-shift,
// so f16 (max 65504) never overflows: 0 for amax < 2^15.
__device__ __forceinline__ int f16_shift_for_amax(float amax) {
  const int e = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127;  // floor(log2) for normals
  return e >= 15 ? e - 14 : 0;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// MXFP8 rounding of one 32-element block held one element per lane (the whole
// warp takes part): the scale and the rounding of mxfp8_round8.
__device__ __forceinline__ float mxfp8_round1(float v) {
  const int e = e4m3_block_exp(warp_max(fabsf(v)));
  float q = v * pow2_e8m0(-e), unused = 0.0f;
  e4m3x2_round(q, unused);
  return q * pow2_e8m0(e);
}

// Butterfly reduce-scatter of V = 2^m per-lane partials over the warp.  On
// return, lane l holds the full warp sum of value index
//   vidx(l) = l >> (5 - m)            (the top m bits of the lane id)
// and every lane in a group of 2^(5-m) consecutive lanes holds the same value.
// Costs V - 1 + (5 - m) shuffles instead of 5 V.
template <int V>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[V], int lane) {
  static_assert(V >= 1 && V <= 32 && (V & (V - 1)) == 0, "V must be a power of two <= 32");
  int width = V;
  int bit = 16;
#pragma unroll
  for (int step = 0; (1 << step) < V; ++step) {
    const int half = width >> 1;
    const bool upper = (lane & bit) != 0;
#pragma unroll
    for (int i = 0; i < V / 2; ++i) {
      if (i < half) {
        const float send = upper ? v[i] : v[i + half];
        const float keep = upper ? v[i + half] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
      }
    }
    width = half;
    bit >>= 1;
  }
  float r = v[0];
#pragma unroll
  for (int b = 1; b <= 16; b <<= 1) {
    if (b <= bit) r += __shfl_xor_sync(0xffffffffu, r, b);
  }
  return r;
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Bulk-copy (TMA, non-tensor) + mbarrier helpers for the streaming kernels.
// Every wait is bounded: after ~2 s of polling it records MOE timeout (5) in
// the status word and returns, so a logic error can never hang the GPU.
// ---------------------------------------------------------------------------
namespace moe {

constexpr int kStatusTimeout = 5;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete; bounded (see above).
__device__ __forceinline__ void mbar_wait(uint64_t* bar, uint32_t parity, int* status) {
  if (mbar_try_wait(bar, parity)) return;
  const unsigned long long t0 = global_ns();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return;
    if (global_ns() - t0 > kWaitLimitNs) {
      if (status) atomicExch(status, kStatusTimeout);
      return;
    }
  }
}

// One thread waits (acquire) until the counter *c reaches target; bounded
// by limit_ns, after which it raises the timeout status and returns.
__device__ __forceinline__ void wait_count_at_least(const unsigned* c, unsigned target,
                                                    int* status, unsigned long long limit_ns) {
  if (ld_acquire_u32(c) >= target) return;
  const unsigned long long t0 = global_ns();
  while (ld_acquire_u32(c) < target) {
    if (global_ns() - t0 > limit_ns) {
      if (status) atomicExch(status, kStatusTimeout);
      return;
    }
  }
}

// Bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Named barrier over the consumer warps only (id 1; the producer never joins).
__device__ __forceinline__ void consumer_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue, and wait for the previous kernel's memory before reading it.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_prerequisites() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Optional kernel trace: slot id holds the earliest CTA start and slot 8 + id
// the latest CTA end (globaltimer ns) of kernel `id` in one forward.
constexpr int kTraceSlots = 16;
__device__ __forceinline__ void trace_begin(unsigned long long* trace, int id) {
  if (trace && threadIdx.x == 0) atomicMin(trace + id, global_ns());
}
__device__ __forceinline__ void trace_end(unsigned long long* trace, int id) {
  if (trace) {
    __syncthreads();
    if (threadIdx.x == 0) atomicMax(trace + 8 + id, global_ns());
  }
}

}  // namespace moe
