// The expert matmuls on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// One kernel per projection, two passes through one stage ring:
//  * routed pass (routed FC1 gate/up with the SwiGLU epilogue, or routed FC2
//    down): a block-scaled MXFP4 x MXFP4 MMA (kind::mxf4).  The weight tile
//    (128 rows, UMMA layout, see mxfp4.cuh) is operand A, the activation
//    planes of up to 8 (expert, row) pairs (8 planes each, see planes.cuh)
//    are operand B, and the E8M0 scales ride along in tensor memory;
//  * dense pass (the shared expert): bf16 weights x bf16 activations
//    (kind::f16), every batch row a column of one MMA, so the shared weights
//    stream once whatever the batch.  FC1 takes x straight from the caller's
//    buffer through a tensor map (cp.async.bulk.tensor), so it needs nothing
//    from the router and runs first, while top-k finishes; its epilogue
//    writes h_s both as fp32 and as (hi, lo) bf16 pairs, the operand of FC2's
//    dense pass (h_s = hi + lo to 2^-16 relative, far inside fp32 sums of
//    bf16 products).  FC2 runs its dense pass first too: its weight copies go
//    out before FC1 is waited for, and the (hi, lo) columns after.
//    From 25 rows the router is a dense pass of its own (tc_router_kernel).
// fp32 accumulators live in tensor memory until the epilogue reads them back;
// nothing is converted on the CUDA cores on the way in.
//
// Work split (both passes): units are (run, tile, K chunk), a run being one
// pass of <= 8 pairs of one active expert (the dense pass: one run).  CTA i
// takes units [i U / G, (i+1) U / G) (U units, G CTAs), so every CTA streams
// the same number of weight bytes.  A tile cut by a range boundary is
// finished by the CTA that holds its first chunk: the later CTAs leave their
// partial sums in a per-CTA slot and raise a flag at the start of their
// range; the finisher adds them in K order at the end of its own (so results
// do not depend on timing).
//
// Roles (7 warps): warp 0 lane 0 streams stages; warp 1 allocates tensor
// memory and its lane 0 issues the tensor-memory scale copies and MMAs and
// commits them to the stage's "empty" barrier and, per tile, to an
// accumulator barrier; warps 2..5 (tensor-memory lane quarters 2, 3, 0, 1)
// run the epilogues; warp 6 builds the routed run table.  Accumulators are double-buffered and scale
// slots ringed with the stages, so the MMA thread never waits for an epilogue
// in steady state.  Every wait is bounded (status 5 on timeout).
//
// Routed activation scales: FC1's x planes carry one code per row
// (planes.cuh), so the MMAs take scale 1 from two constant tensor-memory
// columns and the epilogue multiplies each plane's column by its scale.
// FC2's h planes carry per-block codes (each FC1 epilogue only sees 64
// values of an h row); FC1 writes them per run in the tensor-memory copy's
// atom order, and FC2 loads a run's whole set into tensor memory once, at the
// run's first unit (double buffered by run).  A block-scaled MMA costs about
// the same whatever N is (measured: about 158 SM cycles for M = 128, K = 64,
// any N up to 128, swizzled or not), and so does each scale copy: per stage
// the MMA thread issues only the weight-scale copies and the MMAs.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "common.cuh"
#include "planes.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// tcgen05 / UMMA wrappers
// ---------------------------------------------------------------------------
constexpr int kTcCols = 512;        // tensor-memory columns a CTA allocates (one CTA per SM)
constexpr int kTcRmax = 8;          // pairs per pass: N = 8 planes x 8 pairs = 64 columns
constexpr int kTcMaxCtas = 256;     // partial slots / flags in the workspace
constexpr int kTcDStride = 128;     // two accumulators of up to 128 columns
constexpr int kTcSfaCol = 256;      // D buffers take columns [0, 256)
constexpr int kTcXchg = 2 * 64 * 16;   // floats of the SwiGLU exchange (two buffers)

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Whole warp: allocate kTcCols columns, address written to *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst)),
               "n"(kTcCols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "n"(kTcCols)
               : "memory");
}
// 32 lanes x 32 bits, 2 consecutive columns per thread.
__device__ __forceinline__ void tmem_st2(uint32_t taddr, uint32_t a, uint32_t b) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1, %2};" ::"r"(taddr), "r"(a), "r"(b)
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// 32 lanes x 32 bits, 16 consecutive columns per thread (no wait).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// Shared-memory matrix descriptor: no swizzle, K-major core matrices of 8
// rows x 16 bytes; lbo = byte distance between core matrices along K, sbo =
// between groups of 8 rows.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (uint64_t)((lbo >> 4) & 0x3FFFu) << 16 |
         (uint64_t)((sbo >> 4) & 0x3FFFu) << 32 | (uint64_t)1 << 46;
}
// Instruction descriptor, kind::mxf4: E2M1 x E2M1, E8M0 scales, both K-major,
// M = 128, N columns; a_sf / b_sf select the scale byte pair of the step.
__device__ __forceinline__ uint32_t umma_idesc_mxf4(uint32_t a_sf, uint32_t b_sf, uint32_t N) {
  return (b_sf << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | (1u << 23) | (8u << 24) |
         (a_sf << 29);
}
__device__ __forceinline__ void umma_mxf4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}
// Copy 32 rows x 16 bytes of scales from shared memory into 4 columns of all
// four lane quarters.
__device__ __forceinline__ void umma_sf_copy(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc)
               : "memory");
}
// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}
// The four epilogue warps only (named barrier 2).
__device__ __forceinline__ void tc_epi_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Arguments, shared memory, schedule
// ---------------------------------------------------------------------------
struct TcArgs {
  const uint8_t* q;          // UMMA-layout nibbles (layout 4 for gate/up, 3 for down)
  const uint8_t* s;          // UMMA-layout scales
  size_t q_stride, s_stride; // bytes between experts
  int K;                     // row length
  int KC;                    // K elements per stage (256 or 512)
  int tiles;                 // 128-row weight tiles per expert
  int N;                     // outputs per pair (gate/up: f, down: d)
  int act_div;               // activation row of pair p: p / act_div
  int rowscale;              // 1: one plane-0 code per activation row; 0: per-block scales
  const uint8_t* act;        // activation planes [rows][4K]
  const uint8_t* act_code;   // rowscale: plane-0 code per activation row
  const uint8_t* act_sfb;    // !rowscale: the activation scales of each run, K/128 atoms
  const int* n_active;
  const int* active_expert;
  const int* active_off;
  const int* pair_list;
  float* out;                // [pairs][N]
  unsigned* out_amax;        // gate/up: max |h| bits per pair, or null
  uint8_t* out_act;          // gate/up: h planes [pairs][4N], or null
  uint8_t* out_sfb;          // gate/up: h plane scales per run (N/128 atoms), with out_act
  int out_f8;                // gate/up: 1 = the h planes hold h's MXFP8 rounding
  float* partial;            // [kTcMaxCtas][kTcRmax][128]
  unsigned* flags;           // [kTcMaxCtas], zero between forwards
  int* status;
  int NS, stage_bytes;       // the stage ring (shared by both passes)
  unsigned long long* trace; // optional kernel trace, or null
  int trace_id;
};

// A run's activation scales for the block-scaled MMA come as atoms of 4 K
// blocks (512 bytes, the 32x128b tensor-memory copy's order): the scale of
// row n = 8 r + p (pair r of the run, plane p) for block 4A + kb at byte
// 512 A + 16 (n % 32) + 4 (n / 32) + kb.  A run's K/128 atoms are contiguous,
// run rho's at rho * 4 K.
__host__ __device__ inline size_t tc_sfb_offset(int A, int n, int kb) {
  return (size_t)A * 512 + 16 * (n % 32) + 4 * (n / 32) + kb;
}

// Bytes of shared memory after the stage ring's barriers: barriers, the
// SwiGLU exchange (two buffers of 64 rows x 16 columns), two runs'
// activation-scale atoms (per-block steps, 4 K bytes each) and the run table.
__host__ __device__ inline size_t tc_sfb_smem(int K, bool rowscale) {
  return rowscale ? 0 : 2 * 4 * (size_t)K;
}
__host__ __device__ inline size_t tc_smem_bytes(int E, int K, bool rowscale) {
  return 128 + kTcXchg * 4 + tc_sfb_smem(K, rowscale) +
         ((size_t)(E + 1) * 4 + 127) / 128 * 128;
}
// One stage: weight nibbles (64 KC), weight scales (4 KC), then the planes of
// the pairs (4 KC each, room for at least two: the MMA reads N >= 16 rows).
constexpr int kTcPlaneOff = 68;   // planes start at 68 KC
__host__ __device__ inline size_t tc_stage_bytes(int KC, int rmax) {
  return (size_t)KC * kTcPlaneOff + (size_t)(rmax < 2 ? 2 : rmax) * 4 * KC;
}
// Tensor-memory columns: two accumulators (kTcDStride each), a weight-scale
// slot per stage, and either two constant activation-scale columns or two
// runs' scale sets (4 columns per 4 K blocks).
__host__ __device__ inline int tc_tmem_cols(int K, int KC, int NS, bool rowscale) {
  return kTcSfaCol + NS * (KC / 32) + (rowscale ? 2 : 2 * (K / 32));
}

struct TcSmem {
  uint64_t* acc_full;   // [2] accumulator written (commit)
  uint64_t* acc_empty;  // [2] accumulator read (4 epilogue warps)
  uint64_t* sched;      // run table ready (1)
  uint64_t* sfb_full;   // [2] a run's activation-scale atoms landed (bulk copy)
  uint64_t* sfb_empty;  // [2] and copied into tensor memory (commit)
  uint32_t* tbase;      // tensor-memory base address
  int* n_runs;
  float* xchg;          // [2][1024] up-half sums for the SwiGLU epilogues
  uint8_t* sfb;         // [2][4 K] activation-scale atoms of two runs (per-block steps)
  int* run_off;         // [n_active + 1] first run of each active slot
};

__device__ __forceinline__ TcSmem tc_smem(uint8_t* p, int K, bool rowscale) {
  TcSmem t;
  uint64_t* b = reinterpret_cast<uint64_t*>(p);
  t.acc_full = b;
  t.acc_empty = b + 2;
  t.sched = b + 4;
  t.sfb_full = b + 5;
  t.sfb_empty = b + 7;
  t.tbase = reinterpret_cast<uint32_t*>(b + 9);
  t.n_runs = reinterpret_cast<int*>(b + 9) + 1;
  t.xchg = reinterpret_cast<float*>(p + 128);
  t.sfb = p + 128 + kTcXchg * 4;
  t.run_off = reinterpret_cast<int*>(t.sfb + tc_sfb_smem(K, rowscale));
  return t;
}

struct TcRun {
  int e, p0, R;
};

// Run rho -> (expert, first pair, pairs): the active slot whose runs contain rho.
__device__ __forceinline__ TcRun tc_run(const TcArgs& b, const int* run_off, int nact, int rho) {
  int lo = 0, hi = nact;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (run_off[mid] <= rho) lo = mid;
    else hi = mid;
  }
  TcRun r;
  const int o1 = __ldcg(b.active_off + lo + 1);
  r.p0 = __ldcg(b.active_off + lo) + (rho - run_off[lo]) * kTcRmax;
  r.R = min(kTcRmax, o1 - r.p0);
  r.e = __ldcg(b.active_expert + lo);
  return r;
}

// Units [u0, u1) of CTA i out of G.
__device__ __forceinline__ void tc_range(int U, int i, int G, int& u0, int& u1) {
  u0 = (int)((long long)U * i / G);
  u1 = (int)((long long)U * (i + 1) / G);
}

// One warp: first run of every active slot (passes of <= kTcRmax pairs).
// Each lane first loads the pair counts of 8 slots (independent loads, one
// round trip to L2 per 256 slots), then the warp scans them.
__device__ __forceinline__ void tc_schedule(const TcArgs& b, const TcSmem& t, int lane) {
  const int nact = __ldcg(b.n_active);
  int base = 0;
  if (lane == 0) t.run_off[0] = 0;
  for (int s0 = 0; s0 < nact; s0 += 32 * 8) {
    int passes[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int s = s0 + 32 * i + lane;
      int pr = 0;
      if (s < nact) pr = __ldcg(b.active_off + s + 1) - __ldcg(b.active_off + s);
      passes[i] = (pr + kTcRmax - 1) / kTcRmax;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int incl = passes[i];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const int s = s0 + 32 * i + lane;
      if (s < nact) t.run_off[s + 1] = base + incl;
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncwarp();
  if (lane == 0) {
    *t.n_runs = base;
    mbar_arrive(t.sched);
  }
}

// ---------------------------------------------------------------------------
// Producer (warp 0, lane 0)
// ---------------------------------------------------------------------------
// Per unit both loops below do only a handful of adds: the ring position, the
// chunk index and the source pointers / descriptors advance incrementally, and
// everything that depends on the run is computed once per run.  (A single
// thread issues all the copies or all the MMAs of its CTA; with a division or
// a 64-bit descriptor rebuild per operand, its instruction latency alone
// would fall behind the HBM stream.)
__device__ __forceinline__ void tc_produce(const TcArgs& b, const TcSmem& t, uint8_t* stages,
                                           uint64_t* full, uint64_t* empty, uint32_t& stage) {
  mbar_wait(t.sched, 0, b.status);
  const int nact = __ldcg(b.n_active);
  const int nch = b.K / b.KC, upr = b.tiles * nch;
  int u0, u1;
  tc_range(*t.n_runs * upr, blockIdx.x, gridDim.x, u0, u1);
  if (u0 >= u1) return;
  const uint64_t pol_w = policy_evict_first(), pol_a = policy_evict_last();
  const uint32_t abytes = 64u * b.KC, sbytes = 4u * b.KC, pbytes = 4u * b.KC;
  const uint32_t poff = (uint32_t)kTcPlaneOff * b.KC;
  const uint32_t NS = (uint32_t)b.NS;
  uint32_t buf = stage % NS, use = stage / NS;
  int rho = u0 / upr, idx = u0 - rho * upr, c = idx % nch;
  for (int u = u0, lr = 0; u < u1; ++rho, ++lr, idx = 0, c = 0) {
    const TcRun run = tc_run(b, t.run_off, nact, rho);
    const int n = min(u1 - u, upr - idx);
    const uint8_t* qs = b.q + (size_t)run.e * b.q_stride + (size_t)idx * abytes;
    const uint8_t* ss = b.s + (size_t)run.e * b.s_stride + (size_t)idx * sbytes;
    if (!b.rowscale) {
      // the run's activation-scale atoms, once per run (buffer lr & 1)
      const uint32_t bytes = 4u * b.K, sb = (uint32_t)lr & 1u;
      if (lr >= 2) mbar_wait(&t.sfb_empty[sb], (uint32_t)((lr >> 1) - 1) & 1u, b.status);
      mbar_arrive_expect_tx(&t.sfb_full[sb], bytes);
      bulk_g2s(t.sfb + sb * bytes, b.act_sfb + (size_t)rho * bytes, bytes, &t.sfb_full[sb], pol_a);
    }
    const uint8_t* as[kTcRmax];
#pragma unroll
    for (int r = 0; r < kTcRmax; ++r)
      as[r] = b.act + (r < run.R ? (size_t)(__ldcg(b.pair_list + run.p0 + r) / b.act_div) *
                                       planes_row_bytes(b.K)
                                 : 0);
    const uint32_t tx = poff + (uint32_t)run.R * pbytes;
    for (int i = 0; i < n; ++i) {
      if (use > 0) mbar_wait(&empty[buf], (use - 1) & 1u, b.status);
      uint8_t* dst = stages + (size_t)buf * b.stage_bytes;
      mbar_arrive_expect_tx(&full[buf], tx);
      bulk_g2s(dst, qs, abytes, &full[buf], pol_w);
      bulk_g2s(dst + abytes, ss, sbytes, &full[buf], pol_w);
      const size_t aoff = (size_t)c * pbytes;
#pragma unroll
      for (int r = 0; r < kTcRmax; ++r)
        if (r < run.R) bulk_g2s(dst + poff + r * pbytes, as[r] + aoff, pbytes, &full[buf], pol_a);
      qs += abytes;
      ss += sbytes;
      if (++c == nch) c = 0;
      if (++buf == NS) {
        buf = 0;
        ++use;
      }
      ++stage;
    }
    u += n;
  }
}

// ---------------------------------------------------------------------------
// MMA issuer (warp 1, lane 0)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tc_mma(const TcArgs& b, const TcSmem& t, uint32_t T,
                                       uint8_t* stages, uint64_t* full, uint64_t* empty,
                                       uint32_t& stage, int& jobs) {
  mbar_wait(t.sched, 0, b.status);
  tc_fence_after();
  const int nact = __ldcg(b.n_active);
  const int nch = b.K / b.KC, upr = b.tiles * nch;
  int u0, u1;
  tc_range(*t.n_runs * upr, blockIdx.x, gridDim.x, u0, u1);
  if (u0 >= u1) return;
  const uint32_t KC = (uint32_t)b.KC, NS = (uint32_t)b.NS;
  const uint32_t nsteps = KC / 64, natoms = KC / 128;
  const bool rows = b.rowscale != 0;
  // descriptors of stage 0; stage s, K step j add (s * stage_bytes + step offset) / 16
  const uint32_t sa0 = smem_addr(stages);
  const uint32_t st16 = (uint32_t)b.stage_bytes >> 4;
  const uint64_t dA0 = umma_desc(sa0, 2048, 128);                     // weights: K blocks 2 KB apart
  const uint64_t dB0 = umma_desc(sa0 + kTcPlaneOff * KC, 128, 4 * KC); // planes: pairs 4 KC apart
  const uint64_t dS0 = umma_desc(sa0 + 64 * KC, 0, 128);               // weight scales: 32 rows x 16 B
  const uint64_t dT0 = umma_desc(smem_addr(t.sfb), 0, 128);            // a run's activation scales
  const uint32_t sfa0 = T + kTcSfaCol;
  const uint32_t sfb0 = T + kTcSfaCol + NS * (KC / 32);
  const uint32_t katoms = (uint32_t)b.K / 128;   // activation-scale atoms of a run
  uint32_t buf = stage % NS, ph = (stage / NS) & 1u;
  int rho = u0 / upr, idx = u0 - rho * upr, c = idx % nch;
  uint32_t jb = 0, acc = 0;
  bool newjob = true;
  for (int u = u0, lr = 0; u < u1; ++rho, ++lr, idx = 0, c = 0, newjob = true) {
    const int R = tc_run(b, t.run_off, nact, rho).R;
    uint32_t sfb_run = sfb0;
    if (!rows) {
      // the run's activation scales into tensor memory (buffer lr & 1; the
      // MMAs of run lr - 2, which read it, were issued before these copies)
      const uint32_t sb = (uint32_t)lr & 1u;
      mbar_wait(&t.sfb_full[sb], (uint32_t)(lr >> 1) & 1u, b.status);
      tc_fence_after();
      sfb_run = sfb0 + sb * 4 * katoms;
      const uint64_t d = dT0 + (uint64_t)((sb * 4 * (uint32_t)b.K) >> 4);
      for (uint32_t a = 0; a < katoms; ++a) umma_sf_copy(sfb_run + 4 * a, d + 32 * a);
      umma_commit(&t.sfb_empty[sb]);
    }
    const uint32_t npad = (uint32_t)max(16, (8 * R + 15) & ~15);
    // per K step: the weight scale pair 2 (j & 1); the activation scales the
    // same pair of the per-block atoms, or the constant columns (byte 0)
    const uint32_t id0 = umma_idesc_mxf4(0, 0, npad);
    const uint32_t id1 = umma_idesc_mxf4(2, rows ? 0 : 2, npad);
    const int n = min(u1 - u, upr - idx);
    for (int i = 0; i < n; ++i) {
      if (newjob) {   // a new tile job: a free accumulator, zero-initialised by its first MMA
        jb = (uint32_t)jobs & 1u;
        if (jobs >= 2) {
          mbar_wait(&t.acc_empty[jb], (uint32_t)((jobs >> 1) - 1) & 1u, b.status);
          tc_fence_after();
        }
        acc = 0;
      }
      mbar_wait(&full[buf], ph, b.status);
      tc_fence_after();
      const uint64_t off = (uint64_t)(buf * st16);
      const uint32_t sfa = sfa0 + buf * (KC / 32);
      for (uint32_t a = 0; a < natoms; ++a) umma_sf_copy(sfa + 4 * a, dS0 + off + 32 * a);
      const uint32_t sfb = rows ? sfb_run : sfb_run + 4 * (uint32_t)c * natoms;
      const uint32_t sfb_step = rows ? 0u : 4u;
      const uint32_t dcol = T + kTcDStride * jb;
#pragma unroll 8
      for (uint32_t j = 0; j < nsteps; ++j)
        umma_mxf4(dcol, dA0 + off + 256 * j, dB0 + off + 16 * j, (j & 1) ? id1 : id0,
                  sfa + 4 * (j >> 1), sfb + sfb_step * (j >> 1), acc | j);
      acc = 1;
      // the stage is free once these MMAs have read it
      umma_commit(&empty[buf]);
      newjob = c == nch - 1;
      if (newjob || u + i == u1 - 1) {
        umma_commit(&t.acc_full[jb]);
        ++jobs;
      }
      if (++c == nch) c = 0;
      if (++buf == NS) {
        buf = 0;
        ph ^= 1u;
      }
      ++stage;
    }
    u += n;
  }
}

// ---------------------------------------------------------------------------
// Epilogue (warps 2..5)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tc_wait_flag(const unsigned* f, int* status) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
  if (v) return;
  const unsigned long long t0 = global_ns();
  for (;;) {
    __nanosleep(64);
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    if (v) return;
    if (global_ns() - t0 > kWaitLimitNs) {
      if (status) atomicExch(status, kStatusTimeout);
      return;
    }
  }
}

template <bool GLU>
__device__ __forceinline__ void tc_epilogue(const TcArgs& b, const TcSmem& t, uint32_t T, int q,
                                            int lane, int& jobs, int& fin) {
  mbar_wait(t.sched, 0, b.status);
  const int nact = __ldcg(b.n_active);
  const int nch = b.K / b.KC, upr = b.tiles * nch;
  const int U = *t.n_runs * upr;
  int u0, u1;
  tc_range(U, blockIdx.x, gridDim.x, u0, u1);
  if (u0 >= u1) return;
  const uint32_t qaddr = (uint32_t)(32 * q) << 16;
  const int m = 32 * q + lane;   // MMA row of this thread
  int cur = -1;
  TcRun run{0, 0, 0};
  int pid[kTcRmax];
  float ps[kTcRmax][kPlanes];    // rowscale: the planes' scales of each pair's row
  for (int u = u0; u < u1;) {
    const int rho = u / upr, rem = u - rho * upr, tile = rem / nch, cs = rem - tile * nch;
    const int tile_end = rho * upr + (tile + 1) * nch;
    const int ue = min(u1, tile_end);
    const int ce = cs + (ue - u);
    if (rho != cur) {
      cur = rho;
      run = tc_run(b, t.run_off, nact, rho);
#pragma unroll
      for (int r = 0; r < kTcRmax; ++r) {
        pid[r] = r < run.R ? __ldcg(b.pair_list + run.p0 + r) : 0;
        const uint32_t c0 =
            (b.rowscale && r < run.R) ? (uint32_t)__ldcg(b.act_code + pid[r] / b.act_div) : 127u;
#pragma unroll
        for (int p = 0; p < kPlanes; ++p)
          ps[r][p] = b.rowscale ? __uint_as_float(planes_code(c0, p) << 23) : 1.0f;
      }
    }
    const int R = run.R;
    const int jb = jobs & 1;
    mbar_wait(&t.acc_full[jb], (uint32_t)(jobs >> 1) & 1u, b.status);
    tc_fence_after();
    float v[64];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (16 * i < 8 * R) tmem_ld16(T + qaddr + kTcDStride * (uint32_t)jb + 16 * i, v + 16 * i);
    tmem_wait_ld();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&t.acc_empty[jb]);
    ++jobs;
    float y[kTcRmax];
#pragma unroll
    for (int r = 0; r < kTcRmax; ++r) {
      float s = 0.f;
      if (r < R) {
#pragma unroll
        for (int p = 0; p < kPlanes; ++p) s = fmaf(ps[r][p], v[8 * r + p], s);
      }
      y[r] = s;
    }
    if (cs > 0) {
      // the tile's first chunks belong to an earlier CTA: leave the sums to it
      float* slot = b.partial + (size_t)blockIdx.x * (kTcRmax * 128);
#pragma unroll
      for (int r = 0; r < kTcRmax; ++r)
        if (r < R) slot[r * 128 + m] = y[r];
      tc_epi_sync();
      if (m == 0) {
        __threadfence();
        atomicExch(b.flags + blockIdx.x, 1u);
      }
      u = ue;
      continue;
    }
    if (ce < nch) {
      // later chunks of this tile were streamed by the next CTAs
      for (int j = blockIdx.x + 1; j < (int)gridDim.x; ++j) {
        int j0, j1;
        tc_range(U, j, gridDim.x, j0, j1);
        if (j0 >= tile_end) break;
        if (j1 <= j0) continue;
        if (lane == 0) tc_wait_flag(b.flags + j, b.status);
        __syncwarp();
        const float* slot = b.partial + (size_t)j * (kTcRmax * 128);
#pragma unroll
        for (int r = 0; r < kTcRmax; ++r)
          if (r < R) y[r] += __ldcg(slot + r * 128 + m);
      }
      tc_epi_sync();
      if (m == 0) {
        for (int j = blockIdx.x + 1; j < (int)gridDim.x; ++j) {
          int j0, j1;
          tc_range(U, j, gridDim.x, j0, j1);
          if (j0 >= tile_end) break;
          b.flags[j] = 0u;
        }
      }
    }
    if constexpr (GLU) {
      // rows 0..63 of the tile are gate rows, 64..127 the matching up rows
      float* xg = t.xchg + (fin & 1) * (kTcRmax * 64);
      if (q >= 2) {
#pragma unroll
        for (int r = 0; r < kTcRmax; ++r)
          if (r < R) xg[r * 64 + m - 64] = y[r];
      }
      tc_epi_sync();
      if (q < 2) {
        const int jcol = tile * 64 + m, blk = jcol / 32;
#pragma unroll
        for (int r = 0; r < kTcRmax; ++r) {
          if (r < R) {
            const float g = y[r], uu = xg[r * 64 + m];
            const float hv = g / (1.0f + expf(-g)) * uu;
            b.out[(size_t)pid[r] * b.N + jcol] = hv;
            const float hm = warp_max(fabsf(hv));
            if (lane == 0 && b.out_amax) atomicMax(b.out_amax + pid[r], __float_as_uint(hm));
            if (b.out_act) {
              // the down projection's B operand: h planes and their block scales
              // (out_f8: of h's MXFP8 rounding; out and out_amax keep h itself)
              const int c0 = planes_block(b.out_f8 ? mxfp8_round1(hv) : hv, lane,
                                          b.out_act + (size_t)pid[r] * planes_row_bytes(b.N) + blk * 128);
              if (lane < kPlanes) {
                const int n = 8 * r + lane;
                b.out_sfb[(size_t)rho * 4 * b.N + tc_sfb_offset(blk / 4, n, blk % 4)] =
                    (uint8_t)planes_code((uint32_t)c0, lane);
              }
            }
          }
        }
      }
      ++fin;
    } else {
      const int row = tile * 128 + m;
#pragma unroll
      for (int r = 0; r < kTcRmax; ++r)
        if (r < R) b.out[(size_t)pid[r] * b.N + row] = y[r];
    }
    u = ue;
  }
}

// ---------------------------------------------------------------------------
// Dense pass: the shared expert, bf16 x bf16 -> fp32 (kind::f16)
// ---------------------------------------------------------------------------
// Operand layouts (no swizzle, K-major core matrices of 8 rows x 16 bytes):
//  * weights: 128-row tiles, tile T at T * 256 K bytes, element (m, k) of a
//    tile at (k / 8) * 2048 + m * 16 + (k % 8) * 2.  Gate/up tiles hold 64
//    gate rows (MMA rows 0..63) and the matching 64 up rows (64..127), so one
//    lane quarter pair ends with both halves of a feature.
//  * activations: NP rows (a multiple of 16), element (n, k) at
//    (k / 8) * NP * 16 + n * 16 + (k % 8) * 2, so a stage's K groups are one
//    contiguous run (and one 8-element K group of a row-major [rows][K]
//    matrix is one tensor-map box of 8 x NP).
constexpr int kTcDenseMaxN = 128;   // MMA columns: 2 x 64 batch rows (hi, lo)

__host__ __device__ inline size_t dense_w_offset(int K, int T, int m, int k) {
  return (size_t)T * 256 * K + (size_t)(k / 8) * 2048 + (size_t)m * 16 + (size_t)(k % 8) * 2;
}
__host__ __device__ inline size_t dense_act_offset(int NP, int n, int k) {
  return ((size_t)(k / 8) * NP + n) * 16 + (size_t)(k % 8) * 2;
}
__host__ __device__ inline int dense_np(int rows) { return (rows + 15) / 16 * 16; }
__host__ __device__ inline size_t dense_stage_bytes(int KC, int NP) {
  return (size_t)256 * KC + (size_t)NP * KC * 2;
}

struct TcDense {
  const uint8_t* w;      // weight tiles (layout above)
  const uint8_t* act;    // activation operand (layout above), or null: x through the tensor map
  int K;                 // row length
  int KC;                // K elements per stage (64 or 128)
  int tiles;             // 128-row tiles
  int N;                 // output features (gate/up: features, 64 per tile; down: rows)
  int B;                 // batch rows
  int NP;                // MMA columns: pad16(B), or pad16(2 B) with hilo
  int hilo;              // row b is columns 2b, 2b + 1 (a (hi, lo) bf16 pair), else column b
  float* out;            // [B][N] fp32
  uint8_t* out_hl;       // gate/up: h_s as (hi, lo) bf16 columns 2b, 2b+1 (out_np columns)
  int out_np;
  float* partial;        // [kTcMaxCtas][kTcDenseMaxN][128]
  unsigned* flags;       // [kTcMaxCtas], zero between forwards
  int ctas;              // CTAs 0..ctas-1 share the pass (0: all of the grid)
};

__device__ __forceinline__ int dense_ctas(const TcDense& d) {
  return d.ctas > 0 ? min(d.ctas, (int)gridDim.x) : (int)gridDim.x;
}

// 2-D tensor-map load: box (8 K elements, NP rows) at (k0, 0) -> NP x 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Instruction descriptor, kind::f16: bf16 x bf16 -> fp32, both K-major,
// M = 128, N columns.
__device__ __forceinline__ uint32_t umma_idesc_bf16(uint32_t N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((128u >> 4) << 24);
}
__device__ __forceinline__ void umma_f16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Producer: per unit the tile's K chunk (one bulk copy) and the activation
// chunk (one bulk copy, or one tensor-map box per 8-element K group).  With
// `wait_between` (the activations come from the predecessor kernel, and the
// ring is empty: stage 0) the weights of the first NS units are requested
// first, the predecessor is waited for, and then their activation chunks.
__device__ __forceinline__ void dense_produce(const TcDense& d, const CUtensorMap* xmap,
                                              uint8_t* stages, uint64_t* full, uint64_t* empty,
                                              int NS_, int stage_bytes, uint32_t& stage,
                                              int* status, bool wait_between) {
  const int nch = d.K / d.KC, U = d.tiles * nch;
  const int G = dense_ctas(d);
  int u0 = 0, u1 = 0;
  if ((int)blockIdx.x < G) tc_range(U, blockIdx.x, G, u0, u1);
  if (u0 >= u1) {
    if (wait_between) pdl_wait_prerequisites();
    return;
  }
  const uint64_t pol_w = policy_evict_first(), pol_a = policy_evict_last();
  const uint32_t abytes = 256u * d.KC, bbytes = (uint32_t)d.NP * d.KC * 2u;
  const uint32_t gbytes = (uint32_t)d.NP * 16u;
  const uint32_t NS = (uint32_t)NS_;
  // chunk c of tile T at T * 256 K + c * abytes: the units of a range are contiguous
  const uint8_t* ws = d.w + (size_t)u0 * abytes;
  int npre = 0;
  if (wait_between) {
    npre = min(u1 - u0, NS_);
    for (int i = 0; i < npre; ++i) {
      uint8_t* dst = stages + (size_t)i * stage_bytes;
      mbar_arrive_expect_tx(&full[i], abytes + bbytes);
      bulk_g2s(dst, ws + (size_t)i * abytes, abytes, &full[i], pol_w);
    }
    pdl_wait_prerequisites();
    for (int i = 0; i < npre; ++i) {
      const int c = (u0 + i) % nch;
      bulk_g2s(stages + (size_t)i * stage_bytes + abytes, d.act + (size_t)c * bbytes, bbytes,
               &full[i], pol_a);
    }
    ws += (size_t)npre * abytes;
    stage += (uint32_t)npre;
  }
  uint32_t buf = stage % NS, use = stage / NS;
  int c = (u0 + npre) % nch;
  for (int u = u0 + npre; u < u1; ++u) {
    if (use > 0) mbar_wait(&empty[buf], (use - 1) & 1u, status);
    uint8_t* dst = stages + (size_t)buf * stage_bytes;
    mbar_arrive_expect_tx(&full[buf], abytes + bbytes);
    bulk_g2s(dst, ws, abytes, &full[buf], pol_w);
    if (d.act) {
      bulk_g2s(dst + abytes, d.act + (size_t)c * bbytes, bbytes, &full[buf], pol_a);
    } else {
      for (int g = 0; g < d.KC / 8; ++g)
        tma_load_2d(dst + abytes + g * gbytes, xmap, c * d.KC + 8 * g, 0, &full[buf], pol_a);
    }
    ws += abytes;
    if (++c == nch) c = 0;
    if (++buf == NS) {
      buf = 0;
      ++use;
    }
    ++stage;
  }
}

// MMA issuer: KC / 16 MMAs per unit into the job's accumulator.
__device__ __forceinline__ void dense_mma(const TcDense& d, const TcSmem& t, uint32_t T,
                                          uint8_t* stages, uint64_t* full, uint64_t* empty,
                                          int NS_, int stage_bytes, uint32_t& stage, int& jobs,
                                          int* status) {
  const int nch = d.K / d.KC, U = d.tiles * nch;
  const int G = dense_ctas(d);
  int u0 = 0, u1 = 0;
  if ((int)blockIdx.x < G) tc_range(U, blockIdx.x, G, u0, u1);
  if (u0 >= u1) return;
  const uint32_t NS = (uint32_t)NS_, KC = (uint32_t)d.KC, NP = (uint32_t)d.NP;
  const uint32_t sa0 = smem_addr(stages);
  const uint32_t st16 = (uint32_t)stage_bytes >> 4;
  const uint64_t dA0 = umma_desc(sa0, 2048, 128);              // weights: K groups 2 KB apart
  const uint64_t dB0 = umma_desc(sa0 + 256 * KC, NP * 16, 128); // activations: K groups NP*16 apart
  const uint32_t id = umma_idesc_bf16(NP);
  const uint32_t a_step = 4096u >> 4, b_step = (32u * NP) >> 4;   // per 16 K elements
  uint32_t buf = stage % NS, ph = (stage / NS) & 1u;
  int c = u0 % nch;
  uint32_t jb = 0;
  bool newjob = true;
  for (int u = u0; u < u1; ++u) {
    if (newjob) {   // a new tile job: a free accumulator, zero-initialised by its first MMA
      jb = (uint32_t)jobs & 1u;
      if (jobs >= 2) {
        mbar_wait(&t.acc_empty[jb], (uint32_t)((jobs >> 1) - 1) & 1u, status);
        tc_fence_after();
      }
    }
    mbar_wait(&full[buf], ph, status);
    tc_fence_after();
    const uint64_t off = (uint64_t)(buf * st16);
    const uint32_t dcol = T + kTcDStride * jb;
    const uint32_t acc0 = newjob ? 0u : 1u;
#pragma unroll 8
    for (uint32_t j = 0; j < KC / 16; ++j)
      umma_f16(dcol, dA0 + off + a_step * j, dB0 + off + b_step * j, id, acc0 | j);
    umma_commit(&empty[buf]);
    newjob = c == nch - 1;
    if (newjob || u == u1 - 1) {
      umma_commit(&t.acc_full[jb]);
      ++jobs;
    }
    if (++c == nch) c = 0;
    if (++buf == NS) {
      buf = 0;
      ph ^= 1u;
    }
    ++stage;
  }
}

// Epilogue: per tile job the NP accumulator columns of this thread's row, the
// stream-K fix-up, then gate/up: SwiGLU through the exchange (16 columns at a
// time) to h_s (fp32, and (hi, lo) bf16 for the down projection); plain:
// out[b] = column b, or column 2b + column 2b + 1 with hilo (rows past N,
// the padding of the last tile, are skipped).
template <bool GLU>
__device__ __forceinline__ void dense_epilogue(const TcDense& d, const TcSmem& t, uint32_t T,
                                               int q, int lane, int& jobs, int& fin, int* status) {
  const int nch = d.K / d.KC, U = d.tiles * nch;
  const int G = dense_ctas(d);
  int u0 = 0, u1 = 0;
  if ((int)blockIdx.x < G) tc_range(U, blockIdx.x, G, u0, u1);
  if (u0 >= u1) return;
  const uint32_t qaddr = (uint32_t)(32 * q) << 16;
  const int m = 32 * q + lane;   // MMA row of this thread
  const int NP = d.NP;
  constexpr int NCH = kTcDenseMaxN / 16;
  for (int u = u0; u < u1;) {
    const int tile = u / nch, cs = u - tile * nch;
    const int tile_end = (tile + 1) * nch;
    const int ue = min(u1, tile_end);
    const int ce = cs + (ue - u);
    const int jb = jobs & 1;
    mbar_wait(&t.acc_full[jb], (uint32_t)(jobs >> 1) & 1u, status);
    tc_fence_after();
    float v[kTcDenseMaxN];
#pragma unroll
    for (int i = 0; i < NCH; ++i)
      if (16 * i < NP) tmem_ld16(T + qaddr + kTcDStride * (uint32_t)jb + 16 * i, v + 16 * i);
    tmem_wait_ld();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&t.acc_empty[jb]);
    ++jobs;
    if (cs > 0) {
      // the tile's first chunks belong to an earlier CTA: leave the sums to it
      float* slot = d.partial + (size_t)blockIdx.x * (kTcDenseMaxN * 128);
#pragma unroll
      for (int n = 0; n < kTcDenseMaxN; ++n)
        if (n < NP) slot[n * 128 + m] = v[n];
      tc_epi_sync();
      if (m == 0) {
        __threadfence();
        atomicExch(d.flags + blockIdx.x, 1u);
      }
      u = ue;
      continue;
    }
    if (ce < nch) {
      // later chunks of this tile were streamed by the next CTAs: wait for
      // their flags in parallel (lane l polls CTA blockIdx.x + 1 + l), then
      // add their sums in K order
      for (int j0 = blockIdx.x + 1; j0 < G; j0 += 32) {
        const int j = j0 + lane;
        int a0 = tile_end, a1 = tile_end;
        if (j < G) tc_range(U, j, G, a0, a1);
        if (a0 < tile_end && a1 > a0) tc_wait_flag(d.flags + j, status);
        if (!__any_sync(0xffffffffu, a0 < tile_end)) break;
      }
      __syncwarp();
      for (int j = blockIdx.x + 1; j < G; ++j) {
        int j0, j1;
        tc_range(U, j, G, j0, j1);
        if (j0 >= tile_end) break;
        if (j1 <= j0) continue;
        const float* slot = d.partial + (size_t)j * (kTcDenseMaxN * 128);
#pragma unroll
        for (int n = 0; n < kTcDenseMaxN; ++n)
          if (n < NP) v[n] += __ldcg(slot + n * 128 + m);
      }
      tc_epi_sync();
      if (m == 0) {
        for (int j = blockIdx.x + 1; j < G; ++j) {
          int j0, j1;
          tc_range(U, j, G, j0, j1);
          if (j0 >= tile_end) break;
          d.flags[j] = 0u;
        }
      }
    }
    if constexpr (GLU) {
      // rows 0..63 of the tile are gate rows, 64..127 the matching up rows;
      // column b is batch row b
      const int feat = tile * 64 + (m & 63);
#pragma unroll
      for (int ci = 0; ci < NCH; ++ci) {
        if (16 * ci >= NP) break;
        float* xg = t.xchg + (fin & 1) * 1024;
        if (q >= 2) {
#pragma unroll
          for (int i = 0; i < 16; ++i) xg[i * 64 + m - 64] = v[16 * ci + i];
        }
        tc_epi_sync();
        if (q < 2) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int b = 16 * ci + i;
            if (b < d.B) {
              const float g = v[16 * ci + i], uu = xg[i * 64 + m];
              const float hv = g / (1.0f + expf(-g)) * uu;
              d.out[(size_t)b * d.N + feat] = hv;
              if (d.out_hl) {
                const uint16_t hi = f32_to_bf16_bits(hv);
                const uint16_t lo = f32_to_bf16_bits(hv - bf16_bits_to_f32(hi));
                *reinterpret_cast<uint16_t*>(d.out_hl + dense_act_offset(d.out_np, 2 * b, feat)) = hi;
                *reinterpret_cast<uint16_t*>(d.out_hl + dense_act_offset(d.out_np, 2 * b + 1, feat)) =
                    lo;
              }
            }
          }
        }
        ++fin;
      }
    } else {
      const int row = tile * 128 + m;
      if (row < d.N) {
        if (d.hilo) {
#pragma unroll
          for (int b = 0; b < kTcDenseMaxN / 2; ++b)
            if (b < d.B) d.out[(size_t)b * d.N + row] = v[2 * b] + v[2 * b + 1];
        } else {
#pragma unroll
          for (int b = 0; b < kTcDenseMaxN; ++b)
            if (b < d.B) d.out[(size_t)b * d.N + row] = v[b];
        }
      }
    }
    u = ue;
  }
}

// Shared-expert bf16 weights [rows][K] (row-major) -> 128-row tiles of the
// layout above.  GLU: rows are the gate half then the up half (rows / 2
// each), and tile T takes gate rows 64T..64T+63 then the matching up rows.
static __global__ void dense_relayout_kernel(const uint16_t* src, int64_t rows, int K, int glu,
                                             uint8_t* dst) {
  const int64_t G = K / 8, total = rows * G;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / G;
    const int g = (int)(i - r * G);
    int64_t T, mrow;
    if (glu) {
      const int64_t half = rows / 2, j = r < half ? r : r - half;
      T = j / 64;
      mrow = j % 64 + (r < half ? 0 : 64);
    } else {
      T = r / 128;
      mrow = r % 128;
    }
    const uint4 v = *reinterpret_cast<const uint4*>(src + r * K + (int64_t)g * 8);
    *reinterpret_cast<uint4*>(dst + dense_w_offset(K, (int)T, (int)mrow, 8 * g)) = v;
  }
}

// Wait until the last use of every stage has been consumed, so no copy is
// still landing in this CTA's shared memory when it exits.
__device__ __forceinline__ void tc_drain(uint64_t* empty, int NS, uint32_t stage, int* status) {
  for (int b = 0; b < NS && (uint32_t)b < stage; ++b) {
    const uint32_t uses = (stage - (uint32_t)b + (uint32_t)NS - 1) / (uint32_t)NS;
    mbar_wait(&empty[b], (uses - 1) & 1u, status);
  }
}

// ---------------------------------------------------------------------------
// The kernel.  FC1 (GLU): the dense gate/up pass on x, which the predecessor
// kernels do not write, then the routed gate/up pass once top-k's tables are
// in.  FC2: the dense down pass first, its weight copies requested before
// FC1 is waited for (they fill the gap while FC1's last CTAs drain), then the
// routed down pass.  Warp 6 builds the routed run table as soon as the
// predecessor's tables are visible, while the other roles are still in the
// dense pass.
// ---------------------------------------------------------------------------
constexpr int kTcThreads = 224;

__host__ __device__ inline size_t tc_kernel_smem(int NS, int stage_bytes, int E, int K,
                                                 bool rowscale) {
  return (size_t)NS * stage_bytes + (size_t)NS * 16 + tc_smem_bytes(E, K, rowscale);
}

template <bool GLU>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_kernel(const TcArgs b, const TcDense dn, const __grid_constant__ CUtensorMap xmap) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  trace_begin(b.trace, b.trace_id);
  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)b.NS * b.stage_bytes);
  uint64_t* empty = full + b.NS;
  const TcSmem t = tc_smem(reinterpret_cast<uint8_t*>(empty + b.NS), b.K, b.rowscale != 0);
  if (threadIdx.x == 0) {
    for (int i = 0; i < b.NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&t.acc_full[i], 1);
      mbar_init(&t.acc_empty[i], 4);
      mbar_init(&t.sfb_full[i], 1);
      mbar_init(&t.sfb_empty[i], 1);
    }
    mbar_init(t.sched, 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(t.tbase);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t T = *t.tbase;
  if (b.rowscale && warp >= 2 && warp < 6) {
    // per-row activation scales: the MMAs multiply by 1 (code 127) and the
    // epilogue applies each plane's scale
    const uint32_t col = kTcSfaCol + (uint32_t)b.NS * ((uint32_t)b.KC / 32);
    tmem_st2(T + ((uint32_t)(32 * (warp & 3)) << 16) + col, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
    tmem_wait_st();
    tc_fence_before();
  }
  // the constant columns are written before any MMA is issued
  __syncthreads();
  tc_fence_after();
  pdl_launch_dependents();
  uint32_t stage = 0;
  int jobs = 0, fin = 0;
  if (warp == 0) {
    if (lane == 0) {
      dense_produce(dn, &xmap, stages, full, empty, b.NS, b.stage_bytes, stage, b.status, !GLU);
      if (GLU) pdl_wait_prerequisites();
      tc_produce(b, t, stages, full, empty, stage);
      tc_drain(empty, b.NS, stage, b.status);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      dense_mma(dn, t, T, stages, full, empty, b.NS, b.stage_bytes, stage, jobs, b.status);
      pdl_wait_prerequisites();
      tc_mma(b, t, T, stages, full, empty, stage, jobs);
    }
    __syncwarp();
  } else if (warp < 6) {
    const int q = warp & 3;
    dense_epilogue<GLU>(dn, t, T, q, lane, jobs, fin, b.status);
    pdl_wait_prerequisites();
    tc_epilogue<GLU>(b, t, T, q, lane, jobs, fin);
  } else {
    pdl_wait_prerequisites();
    tc_schedule(b, t, lane);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(T);
  trace_end(b.trace, b.trace_id);
}

// ---------------------------------------------------------------------------
// Router on the tensor cores (tensor-core expert path): the logits as a dense
// pass (router weights in 128-row tiles, the last one zero-padded, x through
// the tensor map), and the x activation planes of the routed FC1, one
// plane-0 code per row (planes.cuh): this CTA's share of the B * K/32
// blocks, each row it touches getting its max |x| from all five plane warps.
// ---------------------------------------------------------------------------
struct TcXPlanes {
  const uint16_t* x;   // [B][K] bf16
  int B, K;
  uint8_t* xq;         // planes [B][4 K], or null
  uint8_t* xq_code;    // plane-0 code per row
  int f8;              // 1: the planes hold x's MXFP8 rounding
};

// Warps 2..6 only (named barrier 3).
__device__ __forceinline__ void tc_plane_sync() { asm volatile("bar.sync 3, 160;" ::: "memory"); }

__device__ __forceinline__ void tc_xplanes(const TcXPlanes& p, int cta, int ncta, int wi, int lane,
                                           unsigned* slots) {
  constexpr int NW = 5;
  const int nb = p.K / 32, total = p.B * nb;
  const int lo = (int)((long long)total * cta / ncta);
  const int hi = (int)((long long)total * (cta + 1) / ncta);
  for (int row = lo / nb; lo < hi && row <= (hi - 1) / nb; ++row) {
    const uint16_t* xrow = p.x + (size_t)row * p.K;
    const uint32_t mx = row_amax_bits(xrow, p.K, wi * 32 + lane, NW * 32, p.f8);
    if (lane == 0) slots[wi] = mx;
    tc_plane_sync();
    uint32_t amax = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) amax = max(amax, slots[w]);
    tc_plane_sync();
    const int c0 = planes_code0(__uint_as_float(amax));
    if (wi == 0 && lane == 0) p.xq_code[row] = (uint8_t)c0;
    const int b0 = max(lo, row * nb) - row * nb, b1 = min(hi, (row + 1) * nb) - row * nb;
    for (int blk = b0 + wi; blk < b1; blk += NW) {
      float v = bf16_bits_to_f32(xrow[blk * 32 + lane]);
      if (p.f8) v = mxfp8_round1(v);
      planes_block_c(v, lane, p.xq + (size_t)row * planes_row_bytes(p.K) + blk * 128, c0);
    }
  }
}

__global__ void __launch_bounds__(kTcThreads, 1)
    tc_router_kernel(const TcDense dn, const __grid_constant__ CUtensorMap xmap,
                     const TcXPlanes xp, int NS, int stage_bytes, int* status,
                     unsigned long long* trace) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  trace_begin(trace, 0);
  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)NS * stage_bytes);
  uint64_t* empty = full + NS;
  const TcSmem t = tc_smem(reinterpret_cast<uint8_t*>(empty + NS), dn.K, true);
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&t.acc_full[i], 1);
      mbar_init(&t.acc_empty[i], 4);
    }
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(t.tbase);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t T = *t.tbase;
  pdl_launch_dependents();
  uint32_t stage = 0;
  int jobs = 0, fin = 0;
  if (warp == 0) {
    if (lane == 0) {
      dense_produce(dn, &xmap, stages, full, empty, NS, stage_bytes, stage, status, false);
      tc_drain(empty, NS, stage, status);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) dense_mma(dn, t, T, stages, full, empty, NS, stage_bytes, stage, jobs, status);
    __syncwarp();
  } else {
    // the x planes on the CTAs past the dense pass's (all of them when the
    // pass takes the whole grid), then the epilogues
    const int G = dense_ctas(dn), spare = (int)gridDim.x - G;
    unsigned* slots = reinterpret_cast<unsigned*>(t.xchg);
    if (xp.xq) {
      if (spare > 0) {
        if ((int)blockIdx.x >= G) tc_xplanes(xp, blockIdx.x - G, spare, warp - 2, lane, slots);
      } else {
        tc_xplanes(xp, blockIdx.x, gridDim.x, warp - 2, lane, slots);
      }
    }
    if (warp < 6) dense_epilogue<false>(dn, t, T, warp & 3, lane, jobs, fin, status);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(T);
  trace_end(trace, 0);
}

}  // namespace moe
