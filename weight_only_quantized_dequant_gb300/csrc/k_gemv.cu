// Dequant-GEMV / small-batch GEMM on CUDA cores (batch 1..4), INT8 per-tensor
// and outlier-aware INT4.
//
// What is computed (per output row i and batch row b):
//   INT8  ("Open Origin - ELG Stream Layer", INT8 Quantization & Direct
//          Mapping; FP16 On-The-Fly GPU Reconstruction):
//          y = scale * sum_j q_ij x_j
//   INT4  ("On-The-Fly Weight Synthesizer (OTF-LLM Engine)", Architecture &
//          Key Innovations diagram and items 1 and 3):
//          y = sum_{t<n_out} w_out_it x_perm[t] + s_i * sum_t' q_it' x_perm[n_out+t']
// Every product is exact in fp32 (an integer code of at most 8 bits times an
// fp16 input) and products are summed in fp32; no fp16 weight is formed.
//
// Design (HBM-bound stream; on GB300 the ALU and FMA pipes and the shared
// memory pipe are close behind, so every instruction per weight counts):
//  * x is gathered through the permutation into shared memory once per CTA,
//    in fp16.  Codes become exact fp16 integers two at a time: one LOP3 puts
//    a nibble pair (or, via PRMT, a byte pair) under the 0x6400 exponent and
//    one packed fp16 subtract removes the offset.  Products use the
//    mixed-precision fma.rn.f32.f16 (fp16 x fp16, exact, added in fp32; one
//    full-rate instruction), so no code or input is ever widened to fp32.
//    Staged chunks are padded by 16 bytes (conflict-free for the 8 lanes of a
//    128-bit phase), so every shared read is a per-lane base plus an
//    immediate offset.
//  * A warp computes R rows at once: each staged granule is read once for
//    all R rows, halving the shared-memory traffic per weight.
//  * Each warp streams its rows' codes through its own ring of shared-memory
//    stages, filled by bulk copies (cp.async.bulk completing on an mbarrier)
//    one stage ahead of the stage it computes; each warp requests its first
//    stage before the wait for the previous kernel.
//  * CTAs own contiguous, equal row ranges; the grid is the SM count times
//    the resident CTAs per SM.
#include "qz_internal.cuh"

namespace qz {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int64_t kPrefetchBytes = 64 * 1024;  // sequence kernel: next product's rows per CTA

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// Weight loads.  Device-resident weights go through the non-coherent path
// (codes arrive by bulk copies); weights read in place from mapped pinned host
// memory (ZC, zero-copy) use plain global loads.
template <bool ZC>
__device__ __forceinline__ uint4 ld_w4(const uint4 *p) {
  if constexpr (ZC) {
    uint4 r;
    asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
  } else {
    return ld_stream(p);
  }
}

template <bool ZC>
__device__ __forceinline__ float ld_wf(const float *p) {
  if constexpr (ZC) {
    float v;
    asm volatile("ld.global.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
  } else {
    return __ldg(p);
  }
}

template <bool ZC>
__device__ __forceinline__ int ld_wi(const int32_t *p) {
  if constexpr (ZC) {
    int v;
    asm volatile("ld.global.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
  } else {
    return __ldg(p);
  }
}

__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// (a & b) ^ c in one LOP3 (truth table 0x6A).
__device__ __forceinline__ uint32_t and_xor(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// c0 += q.lo * x.lo, c1 += q'.lo * x.hi, c2 += q.hi * y.lo, c3 += q'.hi * y.hi
// with fp16 pairs q, q', x, y and fp32 accumulators (fma.rn.f32.f16).
__device__ __forceinline__ void fhfma4(float &c0, float &c1, float &c2, float &c3, uint32_t q,
                                       uint32_t qq, uint32_t x, uint32_t y) {
  asm("{\n\t.reg .f16 q0,q1,r0,r1,x0,x1,y0,y1;\n\t"
      "mov.b32 {q0,q1}, %4;\n\tmov.b32 {r0,r1}, %5;\n\t"
      "mov.b32 {x0,x1}, %6;\n\tmov.b32 {y0,y1}, %7;\n\t"
      "fma.rn.f32.f16 %0, q0, x0, %0;\n\tfma.rn.f32.f16 %1, r0, x1, %1;\n\t"
      "fma.rn.f32.f16 %2, q1, y0, %2;\n\tfma.rn.f32.f16 %3, r1, y1, %3;\n\t}"
      : "+f"(c0), "+f"(c1), "+f"(c2), "+f"(c3)
      : "r"(q), "r"(qq), "r"(x), "r"(y));
}

// c0 += q.lo * x.lo, c1 += q.hi * x.hi
__device__ __forceinline__ void fhfma2(float &c0, float &c1, uint32_t q, uint32_t x) {
  asm("{\n\t.reg .f16 q0,q1,x0,x1;\n\t"
      "mov.b32 {q0,q1}, %2;\n\tmov.b32 {x0,x1}, %3;\n\t"
      "fma.rn.f32.f16 %0, q0, x0, %0;\n\tfma.rn.f32.f16 %1, q1, x1, %1;\n\t}"
      : "+f"(c0), "+f"(c1)
      : "r"(q), "r"(x));
}

__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Accumulators of one row and batch row: [0],[2] collect unscaled products,
// [1],[3] products of codes taken at 16x (INT4 odd nibbles); the background
// sum is (a0 + a2) + (a1 + a3) / 16.
using Acc4 = float[4];

// 32 nibbles of one chunk of each of R rows against the staged fp16 input at
// byte offset `o` (8 inputs per 16-byte granule).  In a word of 8 nibbles
// (elements e0..e7 at bits 4e..4e+3):
//   (w & 0x000F000F) ^ 0x64086408 = fp16 pair (1024 + q0 + 8, 1024 + q4 + 8)
//   (w & 0x00F000F0) ^ 0x64806480 = (1152 + 16 q1, 1152 + 16 q5)
// and the same on w >> 8 for e2,e6 and e3,e7; subtracting 1032 resp. 1152
// leaves q resp. 16 q exactly.
template <int B, int R>
__device__ __forceinline__ void int4_chunk(const uint4 (&v)[R], const void *xs, uint32_t o,
                                           uint32_t bstride, Acc4 (&acc)[R][B]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {  // word k: elements 8k .. 8k+7 = granule k
    uint4 xv[B];
#pragma unroll
    for (int b = 0; b < B; ++b)
      xv[b] = *reinterpret_cast<const uint4 *>(reinterpret_cast<const char *>(xs) + o + k * 16 +
                                               b * bstride);
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
      const uint32_t w = k == 0 ? v[rr].x : k == 1 ? v[rr].y : k == 2 ? v[rr].z : v[rr].w;
      const uint32_t w8 = w >> 8;
      const uint32_t qa = hsub2_bits(and_xor(w, 0x000F000Fu, 0x64086408u), 0x64086408u);
      const uint32_t qb = hsub2_bits(and_xor(w, 0x00F000F0u, 0x64806480u), 0x64806480u);
      const uint32_t qc = hsub2_bits(and_xor(w8, 0x000F000Fu, 0x64086408u), 0x64086408u);
      const uint32_t qd = hsub2_bits(and_xor(w8, 0x00F000F0u, 0x64806480u), 0x64806480u);
#pragma unroll
      for (int b = 0; b < B; ++b) {
        // xv.x = (x0,x1), .y = (x2,x3), .z = (x4,x5), .w = (x6,x7)
        fhfma4(acc[rr][b][0], acc[rr][b][1], acc[rr][b][2], acc[rr][b][3], qa, qb, xv[b].x,
               xv[b].z);
        fhfma4(acc[rr][b][0], acc[rr][b][1], acc[rr][b][2], acc[rr][b][3], qc, qd, xv[b].y,
               xv[b].w);
      }
    }
  }
}

// 16 int8 codes of one chunk of each of R rows.  XOR 0x80 makes each byte the
// offset-binary u = q + 128; PRMT puts two of them under the 0x6400 exponent
// (fp16 1024 + u) and subtracting 1152 leaves q exactly.
template <int B, int R>
__device__ __forceinline__ void int8_chunk(const uint4 (&v)[R], const void *xs, uint32_t o,
                                           uint32_t bstride, Acc4 (&acc)[R][B]) {
#pragma unroll
  for (int k2 = 0; k2 < 2; ++k2) {  // words 2k2, 2k2+1: elements 8k2 .. 8k2+7
    uint4 xv[B];
#pragma unroll
    for (int b = 0; b < B; ++b)
      xv[b] = *reinterpret_cast<const uint4 *>(reinterpret_cast<const char *>(xs) + o + k2 * 16 +
                                               b * bstride);
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
      const uint32_t w0 = (k2 == 0 ? v[rr].x : v[rr].z) ^ 0x80808080u;
      const uint32_t w1 = (k2 == 0 ? v[rr].y : v[rr].w) ^ 0x80808080u;
      const uint32_t q01 = hsub2_bits(__byte_perm(w0, 0x64646464u, 0x4140), 0x64806480u);
      const uint32_t q23 = hsub2_bits(__byte_perm(w0, 0x64646464u, 0x4342), 0x64806480u);
      const uint32_t q45 = hsub2_bits(__byte_perm(w1, 0x64646464u, 0x4140), 0x64806480u);
      const uint32_t q67 = hsub2_bits(__byte_perm(w1, 0x64646464u, 0x4342), 0x64806480u);
#pragma unroll
      for (int b = 0; b < B; ++b) {
        fhfma2(acc[rr][b][0], acc[rr][b][2], q01, xv[b].x);
        fhfma2(acc[rr][b][0], acc[rr][b][2], q23, xv[b].y);
        fhfma2(acc[rr][b][0], acc[rr][b][2], q45, xv[b].z);
        fhfma2(acc[rr][b][0], acc[rr][b][2], q67, xv[b].w);
      }
    }
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------------------
// Bulk-copy ring.  Each warp streams its rows' codes through kNS stages of
// shared memory: lane 0 issues cp.async.bulk copies (global -> shared, with
// an mbarrier transaction count) kNS-1 stages ahead of the stage the lanes
// are computing, so a warp keeps its next rows in flight without holding
// them in registers.  A stage is RPS rounds (32 chunks of 16 bytes) of each
// of the warp's R rows.  Every wait is bounded in time.
// ---------------------------------------------------------------------------
__device__ int g_gemv_error = 0;  // 1 if a bounded wait gave up (read by qz_device_error)

constexpr uint32_t kRoundBytes = 512;          // 32 chunks x 16 bytes
constexpr unsigned long long kWaitNs = 2000000000ull;

template <int B>
struct Ring {
  static constexpr int NS = 2;                 // stages per warp
  static constexpr int R = B == 1 ? 2 : 1;     // rows per warp
  static constexpr int RPS = B == 1 ? 4 : 2;   // rounds per stage
  static constexpr int MINB = 1;               // CTAs per SM the registers allow
  static constexpr uint32_t STAGE_ROW = RPS * kRoundBytes;  // bytes of one row in a stage
};
// gemv_smem_bytes sizes every B > 1 by Ring<2>
static_assert(Ring<3>::NS == Ring<2>::NS && Ring<3>::R == Ring<2>::R &&
                  Ring<3>::STAGE_ROW == Ring<2>::STAGE_ROW && Ring<4>::NS == Ring<2>::NS &&
                  Ring<4>::R == Ring<2>::R && Ring<4>::STAGE_ROW == Ring<2>::STAGE_ROW,
              "one ring shape for all batches > 1");

__device__ __forceinline__ uint32_t smem_u32(const void *ptr) {
  return (uint32_t)__cvta_generic_to_shared(ptr);
}

__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait; on timeout the error word is set and false returned.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try(bar, parity)) return true;
  const unsigned long long t0 = gtimer();
  for (;;) {
    if (mbar_try(bar, parity)) return true;
    if (gtimer() - t0 > kWaitNs) {
      atomicExch(&g_gemv_error, 1);
      return false;
    }
  }
}

// After a warp gave up a wait: stages first..issued-1 of its ring may still
// have bulk copies in flight.  Stage i lives in slot i % NS and completes
// phase i / NS of that slot's barrier, so each is waited for (bounded) on its
// own parity before the CTA's shared memory can be handed to another CTA.
template <int NS>
__device__ __forceinline__ void ring_drain(uint32_t bar_w, int first, int issued) {
  const unsigned long long t0 = gtimer();
  for (int i = first; i < issued; ++i) {
    const uint32_t bar = bar_w + (uint32_t)(i % NS) * 8u;
    const uint32_t parity = (uint32_t)(i / NS) & 1u;
    while (!mbar_try(bar, parity)) {
      if (gtimer() - t0 > kWaitNs) return;
    }
  }
}

// Row boundaries of the grouped matrices, kept in registers (32-bit rows:
// the host limits a launch to < 2^31 rows).
struct Bounds {
  int end[QZ_MAX_GROUP];
  int n;
};

// Row r of the launch -> (matrix, row inside it).
__device__ __forceinline__ void locate(const Bounds &bd, int r, int &m, int &i) {
  m = 0;
#pragma unroll
  for (int t = 0; t < QZ_MAX_GROUP - 1; ++t) m += (t < bd.n - 1 && r >= bd.end[t]) ? 1 : 0;
  int lo = 0;
#pragma unroll
  for (int t = 0; t < QZ_MAX_GROUP - 1; ++t) lo = (t < m) ? bd.end[t] : lo;
  i = r - lo;
}

// W: warps per CTA (16, or 20 at batch 1 when shared memory allows).
// ZC (batch 1): the weights (codes, outliers, scales, permutation) may be in
// mapped pinned host memory; every lane then reads its chunks of each round
// with plain loads, without the bulk-copy ring (whose engine is not asked to
// read host memory), and the permutation is read from where it lies.
template <bool INT4, int B, int W, bool ZC = false>
__global__ void __launch_bounds__(W * 32, Ring<B>::MINB)
    gemv_kernel(const __grid_constant__ GemvParams p) {
  static_assert(!ZC || B == 1, "zero-copy reads at batch 1 only");
  constexpr int kWarps = W, kThreads = W * 32;
  constexpr int R = Ring<B>::R, NS = Ring<B>::NS, kRPS = Ring<B>::RPS;
  constexpr uint32_t kStageRow = Ring<B>::STAGE_ROW;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  constexpr int EPC = INT4 ? 32 : 16;      // fp16 inputs per code chunk
  constexpr uint32_t CS = EPC * 2 + 16;    // staged bytes per chunk (padded by 16)
  const int cpr = p.cpr;
  const int Jw = (cpr + 31) >> 5;          // rounds of 32 chunks per row
  const int staged = (Jw > 0 ? Jw : 1) * 32;
  const uint32_t bstride = (uint32_t)staged * CS;  // bytes per batch row
  const uint32_t ostride = (uint32_t)p.ocpr * 16;  // outlier input bytes per batch row
  __half *xs = reinterpret_cast<__half *>(smem_raw);
  __half *xo = reinterpret_cast<__half *>(smem_raw + B * bstride);
  uint8_t *ring = smem_raw + (((size_t)B * bstride + (size_t)B * ostride + 127) & ~(size_t)127);
  uint64_t *bars =
      reinterpret_cast<uint64_t *>(ring + (ZC ? 0 : (size_t)kWarps * NS * R * kStageRow));

  const int64_t r0 = p.total_rows * blockIdx.x / gridDim.x;
  const int64_t r1 = p.total_rows * (blockIdx.x + 1) / gridDim.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // No L2 prefetch of the CTA's first rows: measured, a 16-256 KiB prefetch
  // before the wait gained nothing (16 KiB) or lost 5-10% (the ring's own
  // first stages are already requested before the wait).
  if (lane == 0) {
    for (int st = 0; st < NS; ++st)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bars[warp * NS + st]))
                   : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // ---- each warp: row groups of R rows, streamed through its ring -----------
  Bounds bd;
#pragma unroll
  for (int t = 0; t < QZ_MAX_GROUP; ++t) bd.end[t] = (int)p.row_end[t];
  bd.n = p.n_mats;
  const int rlo = (int)r0, rhi = (int)r1;
  const int first = rlo + warp * R;
  constexpr int stride = kWarps * R;
  const bool has_rows = first < rhi;  // warps without rows still join the barrier
  const int P = has_rows ? (rhi - first + stride - 1) / stride : 0;  // row groups of this warp
  const int SPR = (Jw + kRPS - 1) / kRPS;             // stages per row group
  const int items = P * SPR;
  const uint32_t lane_off = (uint32_t)lane * CS;
  constexpr uint32_t kRound = 32u * CS;  // staged bytes per round of 32 chunks
  // Ring slots are laid out stage-major ([stage][warp]): slot st of this
  // warp at ring_w + st * slot_stride.  Only the first stage of every warp
  // is requested before the input is staged, so the second stages of all
  // warps form one free block meanwhile (used for the permutation table).
  constexpr uint32_t slot_stride = (uint32_t)kWarps * R * kStageRow;
  const uint32_t ring_w = smem_u32(ring) + (uint32_t)warp * R * kStageRow;
  const uint32_t bar_w = smem_u32(&bars[warp * NS]);

  // Producer state (tracked by every lane so control flow stays uniform;
  // only lane 0 issues): next stage to fill = row group pg, stage psj of it,
  // ring slot pst; pptr = the rows' code pointers of group pg.
  int pg = 0, psj = 0, pst = 0;
  int pleft = items;
  const uint8_t *pptr[R];
  auto prow_setup = [&](int gidx) {
    const int rb = first + gidx * stride;
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
      const int rc = rb + rr < rhi ? rb + rr : rhi - 1;  // past the end: alias a valid row
      int m, i;
      locate(bd, rc, m, i);
      pptr[rr] = p.codes[m] + (int64_t)i * p.ld_codes[m];
    }
  };
  auto issue_next = [&]() {
    if (lane == 0) {
      const int j0 = psj * kRPS;
      const int span = cpr - 32 * j0 < 32 * kRPS ? cpr - 32 * j0 : 32 * kRPS;  // chunks
      const uint32_t bytes = (uint32_t)span * 16u;
      const uint32_t bar = bar_w + pst * 8;
      asm volatile(
          "{\n\t.reg .b64 t;\n\t"
          "mbarrier.arrive.expect_tx.shared::cta.b64 t, [%0], %1;\n\t}" ::"r"(bar),
          "r"(bytes * R)
          : "memory");
#pragma unroll
      for (int rr = 0; rr < R; ++rr) {
        const uint32_t dst = ring_w + (uint32_t)pst * slot_stride + (uint32_t)rr * kStageRow;
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
                "r"(dst),
            "l"(pptr[rr] + j0 * kRoundBytes), "r"(bytes), "r"(bar)
            : "memory");
      }
    }
    --pleft;
    pst = pst + 1 == NS ? 0 : pst + 1;
    if (++psj == SPR) {
      psj = 0;
      if (++pg < P) prow_setup(pg);
    }
  };

  // The first stages are issued before the wait: weights are static, so
  // under programmatic overlap they stream in during the previous kernel.
  // With the permutation read before the wait, its first loads go out
  // before these copies (measured against the copies first: 70B-shaped step
  // +0.9%, 3B +1.5%).
  auto issue_first = [&]() {
    if constexpr (!ZC) {
      if (items > 0) prow_setup(0);
      for (int it = 0; it < NS - 1 && pleft > 0; ++it) issue_next();
    }
  };

  // INT4: the permutation (static) goes into the free ring block before the
  // wait, read with coalesced 16-byte loads, as 16-bit entries (K <= 57344):
  // background entry t' at pb[t'], outlier entry t at pb[kb_pad + t].  The
  // gather after the wait then needs no global round trip for it.
  uint16_t *pb = reinterpret_cast<uint16_t *>(ring + slot_stride);
  const int elems = staged * EPC;           // staged inputs per batch row (multiple of 8)
  // (measured: pays for K > 4096; at smaller K the gather after the wait is
  // short and the extra barrier costs more than it saves)
  const bool perm_smem = !ZC && INT4 && NS == 2 && p.K > 4096 &&
                         (size_t)(elems + p.ocpr * 8) * 2 <= slot_stride;
  if (INT4 && perm_smem) {
    const int K = p.K, n_out = p.n_out;
    auto place = [&](int e, int v) {
      if (e < n_out) pb[elems + e] = (uint16_t)v;
      else pb[e - n_out] = (uint16_t)v;
    };
    // the first batch of loads goes out before the ring's first stages
    constexpr int kPermBatch = 8;
    const int nv = K / 4;
    bool issued = false;
#pragma unroll 1
    for (int c0 = threadIdx.x; c0 < nv; c0 += kPermBatch * kThreads) {
      int4 v[kPermBatch];
#pragma unroll
      for (int u = 0; u < kPermBatch; ++u) {
        const int c = c0 + u * kThreads;
        v[u] = c < nv ? __ldg(reinterpret_cast<const int4 *>(p.perm) + c) : make_int4(0, 0, 0, 0);
      }
      if (!issued) {
        issue_first();
        issued = true;
      }
#pragma unroll
      for (int u = 0; u < kPermBatch; ++u) {
        const int c = c0 + u * kThreads;
        if (c < nv) {
          place(4 * c, v[u].x);
          place(4 * c + 1, v[u].y);
          place(4 * c + 2, v[u].z);
          place(4 * c + 3, v[u].w);
        }
      }
    }
    if (!issued) issue_first();
    for (int e = 4 * nv + threadIdx.x; e < K; e += kThreads) place(e, __ldg(p.perm + e));
    for (int t = p.kb + threadIdx.x; t < elems; t += kThreads) pb[t] = 0xFFFFu;
    for (int t = n_out + threadIdx.x; t < p.ocpr * 8; t += kThreads) pb[elems + t] = 0xFFFFu;
  } else {
    issue_first();
  }

  asm volatile("griddepcontrol.wait;" ::: "memory");
  // let the next kernel on the stream get scheduled as SMs free up
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (INT4 && perm_smem) __syncthreads();

  // ---- stage x (gathered through perm for INT4) in shared memory, fp16 ----
  // Eight consecutive inputs per step and thread: eight perm entries, eight
  // independent gathers, one 16-byte shared store (8 inputs never straddle a
  // staged chunk); INT8 inputs are read in order.  With the permutation in
  // shared memory each thread issues the gathers of kGroupsP steps before it
  // stores any of them, for INT8 the loads of kGroups steps (measured at
  // the step: 2 gathers 0.1-0.3% ahead of 4 and 1.1-1.5% ahead of 8, 1 the
  // same as 2; the INT8 loads lose about 1% with 2 instead of 4).
  const __half hzero = __ushort_as_half((unsigned short)0);
  const int step8 = kThreads * 8;
  constexpr int kGroups = 4;
  if (INT4 && perm_smem) {
    constexpr int kGroupsP = 2;
#pragma unroll 1
    for (int b = 0; b < B; ++b) {
      const __half *xb = p.x + b * p.ldx;
#pragma unroll 1
      for (int g0 = threadIdx.x * 8; g0 < elems; g0 += kGroupsP * step8) {
        uint4 v[kGroupsP];
#pragma unroll
        for (int gi = 0; gi < kGroupsP; ++gi) {
          const int e0 = g0 + gi * step8;
          uint32_t h[8];
          if (e0 < elems) {
            const uint4 q = *reinterpret_cast<const uint4 *>(pb + e0);
            const uint32_t qq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t lo = qq[k] & 0xFFFFu, hi = qq[k] >> 16;
              h[2 * k] = lo != 0xFFFFu ? __half_as_ushort(__ldg(xb + lo)) : 0u;
              h[2 * k + 1] = hi != 0xFFFFu ? __half_as_ushort(__ldg(xb + hi)) : 0u;
            }
          } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) h[k] = 0u;
          }
          v[gi] = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                             h[6] | (h[7] << 16));
        }
#pragma unroll
        for (int gi = 0; gi < kGroupsP; ++gi) {
          const int e0 = g0 + gi * step8;
          if (e0 < elems)
            *reinterpret_cast<uint4 *>(reinterpret_cast<char *>(xs) + b * bstride + (e0 / EPC) * CS +
                                       (e0 % EPC) * 2) = v[gi];
        }
      }
#pragma unroll 1
      for (int e = threadIdx.x; e < p.ocpr * 8; e += kThreads) {
        const uint32_t src = pb[elems + e];
        xo[b * ostride / 2 + e] = src != 0xFFFFu ? __ldg(xb + src) : hzero;
      }
    }
  } else if constexpr (INT4) {
#pragma unroll 1
    for (int b = 0; b < B; ++b) {
      const __half *xb = p.x + b * p.ldx;
#pragma unroll 1
      for (int e0 = threadIdx.x * 8; e0 < elems; e0 += step8) {
        int idx[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) idx[k] = e0 + k < p.kb ? ld_wi<ZC>(p.perm + p.n_out + e0 + k) : -1;
        __half v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = idx[k] >= 0 ? xb[idx[k]] : hzero;
        uint32_t h[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          h[k] = (uint32_t)__half_as_ushort(v[2 * k]) | ((uint32_t)__half_as_ushort(v[2 * k + 1]) << 16);
        *reinterpret_cast<uint4 *>(reinterpret_cast<char *>(xs) + b * bstride + (e0 / EPC) * CS +
                                   (e0 % EPC) * 2) = make_uint4(h[0], h[1], h[2], h[3]);
      }
#pragma unroll 1
      for (int e = threadIdx.x; e < p.ocpr * 8; e += kThreads)
        xo[b * ostride / 2 + e] = e < p.n_out ? xb[ld_wi<ZC>(p.perm + e)] : hzero;
    }
  } else {
    // INT8: inputs in order, eight per thread and step as one 16-byte load
    // where x is 16-byte aligned, the loads of kGroups steps out before any
    // is stored (measured: with eight 2-byte loads per thread, each
    // warp-wide request spanning 512 bytes, INT8 decode steps ran 2-3%
    // slower).
#pragma unroll 1
    for (int b = 0; b < B; ++b) {
      const __half *xb = p.x + b * p.ldx;
      const bool vec = (reinterpret_cast<uintptr_t>(xb) & 15u) == 0;
      char *xsb = reinterpret_cast<char *>(xs) + b * bstride;
#pragma unroll 1
      for (int g0 = threadIdx.x * 8; g0 < elems; g0 += kGroups * step8) {
        uint4 v[kGroups];
#pragma unroll
        for (int gi = 0; gi < kGroups; ++gi) {
          const int e = g0 + gi * step8;
          if (vec && e + 8 <= p.kb) {
            if constexpr (ZC) v[gi] = *reinterpret_cast<const uint4 *>(xb + e);
            else v[gi] = __ldg(reinterpret_cast<const uint4 *>(xb + e));
          } else {
            uint32_t h[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              h[k] = e + k < p.kb ? (uint32_t)__half_as_ushort(xb[e + k]) : 0u;
            v[gi] = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                               h[6] | (h[7] << 16));
          }
        }
#pragma unroll
        for (int gi = 0; gi < kGroups; ++gi) {
          const int e = g0 + gi * step8;  // 8 inputs never straddle a staged chunk
          if (e < elems) *reinterpret_cast<uint4 *>(xsb + (e / EPC) * CS + (e % EPC) * 2) = v[gi];
        }
      }
    }
  }
  __syncthreads();
  if (!has_rows) return;  // no barrier follows

  Acc4 acc[R][B];
#pragma unroll
  for (int rr = 0; rr < R; ++rr)
#pragma unroll
    for (int b = 0; b < B; ++b) acc[rr][b][0] = acc[rr][b][1] = acc[rr][b][2] = acc[rr][b][3] = 0.f;

  bool ok = true;
  int cst = 0;            // consumer ring slot
  uint32_t cphase = 0;    // parity of the slot's current use
  int cidx = 0;           // stages consumed (ring position of the consumer)
  int fail_at = -1;       // first stage whose wait gave up
  for (int g = 0; g < P; ++g) {
    // rows of this group: matrix, row, scale, first outlier chunk
    const int rb = first + g * stride;
    int mrow[R], irow[R];
    float srow[R];
    bool live[R];
    uint4 ov[R];  // first outlier chunk of each row, loaded now, used at the end
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
      live[rr] = rb + rr < rhi;
      locate(bd, live[rr] ? rb + rr : rhi - 1, mrow[rr], irow[rr]);
      srow[rr] = INT4 ? ld_wf<ZC>(p.scale[mrow[rr]] + irow[rr]) : ld_wf<ZC>(p.scale[mrow[rr]]);
      ov[rr] = make_uint4(0, 0, 0, 0);
      if (INT4 && lane < p.ocpr)
        ov[rr] = ld_w4<ZC>(reinterpret_cast<const uint4 *>(
                               p.w_out[mrow[rr]] + (int64_t)irow[rr] * p.ld_out[mrow[rr]]) +
                           lane);
    }
    for (int sj = 0; sj < SPR; ++sj) {
      if constexpr (ZC) {
        // every lane loads its chunk of each round of the stage in place
        uint4 v[kRPS][R];
#pragma unroll
        for (int u = 0; u < kRPS; ++u) {
          const int c = (sj * kRPS + u) * 32 + lane;  // chunk of the row
#pragma unroll
          for (int rr = 0; rr < R; ++rr)
            v[u][rr] = c < cpr ? ld_w4<true>(reinterpret_cast<const uint4 *>(
                                     p.codes[mrow[rr]] + (int64_t)irow[rr] * p.ld_codes[mrow[rr]]) +
                                 c)
                               : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kRPS; ++u) {
          const int j = sj * kRPS + u;
          if (j < Jw) {  // warp-uniform
            const uint32_t o = lane_off + (uint32_t)j * kRound;
            if constexpr (INT4) int4_chunk<B, R>(v[u], xs, o, bstride, acc);
            else int8_chunk<B, R>(v[u], xs, o, bstride, acc);
          }
        }
        continue;
      }
      if (ok && pleft > 0) {
        // the slot being refilled was read by every lane before the last
        // __syncwarp; order those reads before the async-proxy write
        if (lane == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        issue_next();
      }
      if (ok) {
        ok = mbar_wait(bar_w + cst * 8, cphase);
        if (!ok) fail_at = cidx;
      }
      if (ok) {
        // Lanes whose chunk lies past the row's end read stale (finite) codes
        // of the slot; their staged inputs are zero, so they add exact zeros.
        const uint32_t sbase = ring_w + (uint32_t)cst * slot_stride + lane * 16;
#pragma unroll
        for (int u = 0; u < kRPS; ++u) {
          const int j = sj * kRPS + u;
          if (j < Jw) {  // warp-uniform
            uint4 v[R];
#pragma unroll
            for (int rr = 0; rr < R; ++rr) {
              const uint32_t a = sbase + (uint32_t)rr * kStageRow + u * kRoundBytes;
              asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                           : "=r"(v[rr].x), "=r"(v[rr].y), "=r"(v[rr].z), "=r"(v[rr].w)
                           : "r"(a));
            }
            const uint32_t o = lane_off + (uint32_t)j * kRound;
            if constexpr (INT4) int4_chunk<B, R>(v, xs, o, bstride, acc);
            else int8_chunk<B, R>(v, xs, o, bstride, acc);
          }
        }
      }
      __syncwarp();
      ++cidx;
      if (++cst == NS) {
        cst = 0;
        cphase ^= 1u;
      }
    }
    // ---- row epilogue: outliers, scale, reduction, store --------------------
    float outl[R][B][2];
#pragma unroll
    for (int rr = 0; rr < R; ++rr)
#pragma unroll
      for (int b = 0; b < B; ++b) outl[rr][b][0] = outl[rr][b][1] = 0.0f;
    if constexpr (INT4) {
#pragma unroll
      for (int rr = 0; rr < R; ++rr) {
        const uint4 *orow = reinterpret_cast<const uint4 *>(p.w_out[mrow[rr]] +
                                                            (int64_t)irow[rr] * p.ld_out[mrow[rr]]);
#pragma unroll 1
        for (int c = lane; c < p.ocpr; c += 32) {
          const uint4 v = c == lane ? ov[rr] : ld_w4<ZC>(orow + c);
#pragma unroll
          for (int b = 0; b < B; ++b) {
            const uint4 xv = *reinterpret_cast<const uint4 *>(
                reinterpret_cast<const char *>(xo) + b * ostride + c * 16);
            fhfma2(outl[rr][b][0], outl[rr][b][1], v.x, xv.x);
            fhfma2(outl[rr][b][0], outl[rr][b][1], v.y, xv.y);
            fhfma2(outl[rr][b][0], outl[rr][b][1], v.z, xv.z);
            fhfma2(outl[rr][b][0], outl[rr][b][1], v.w, xv.w);
          }
        }
      }
    }
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const float bg = (acc[rr][b][0] + acc[rr][b][2]) + (acc[rr][b][1] + acc[rr][b][3]) * 0.0625f;
        // y = s_i * background + outliers, combined per lane, one reduction
        const float yl = warp_sum(fmaf(srow[rr], bg, outl[rr][b][0] + outl[rr][b][1]));
        if (lane == 0 && live[rr]) p.y[mrow[rr]][b * p.ldy[mrow[rr]] + irow[rr]] = __float2half_rn(yl);
        acc[rr][b][0] = acc[rr][b][1] = acc[rr][b][2] = acc[rr][b][3] = 0.f;
      }
    }
  }
  // A warp that gave up a wait may still have copies in flight into its
  // ring; give them a bounded time to land before the CTA's shared memory goes.
  if (!ZC && !ok && lane == 0) ring_drain<NS>(bar_w, fail_at, items - pleft);
}

// ---------------------------------------------------------------------------
// Sequence kernel: up to kMaxSeq dependent batch-1 products in one launch.
// Product k reads its x only after every CTA has stored its rows of products
// 0..k-1 (a grid-wide barrier on a counter in caller memory), so x of k may be
// the y of an earlier product.  The weight ring is not drained at the
// barriers: the producers run into the next product's rows (weights are
// static), and thread 0 pulls the next product's first rows into L2 while the
// current one is computed.  Same per-row arithmetic as gemv_kernel<INT4, 1, W>.
// The grid must be co-resident (one CTA per SM; every wait is bounded).
// ---------------------------------------------------------------------------
template <bool INT4>
__global__ void __launch_bounds__(kThreads, 1) gemv_seq_kernel(const __grid_constant__ SeqParams sp) {
  constexpr int B = 1;
  constexpr int R = Ring<1>::R, NS = Ring<1>::NS, kRPS = Ring<1>::RPS;
  constexpr uint32_t kStageRow = Ring<1>::STAGE_ROW;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  constexpr int EPC = INT4 ? 32 : 16;      // fp16 inputs per code chunk
  constexpr uint32_t CS = EPC * 2 + 16;    // staged bytes per chunk (padded by 16)
  constexpr uint32_t kRound = 32u * CS;    // staged bytes per round of 32 chunks
  constexpr int stride = kWarps * R;
  __half *xs = reinterpret_cast<__half *>(smem_raw);
  uint8_t *ring = smem_raw + sp.xs_bytes;                       // 128-aligned by the host
  uint64_t *bars = reinterpret_cast<uint64_t *>(ring + (size_t)kWarps * NS * R * kStageRow);
  int *abort_flag = reinterpret_cast<int *>(bars + kWarps * NS);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = (int)gridDim.x;

  // This warp's share of product k: rows [rlo, rhi) of the CTA, groups of R
  // rows starting at `first`, P groups of SPR stages.
  struct Work {
    int rlo, rhi, first, P, SPR, Jw;
  };
  auto plan = [&](int k) {
    const GemvParams &p = sp.t[k];
    Work w;
    w.rlo = (int)(p.total_rows * blockIdx.x / G);
    w.rhi = (int)(p.total_rows * (blockIdx.x + 1) / G);
    w.first = w.rlo + warp * R;
    w.P = w.first < w.rhi ? (w.rhi - w.first + stride - 1) / stride : 0;
    w.Jw = (p.cpr + 31) >> 5;
    w.SPR = (w.Jw + kRPS - 1) / kRPS;
    return w;
  };
  auto prefetch_rows = [&](int k) {  // the first 64 KiB of this CTA's rows of product k
    const GemvParams &p = sp.t[k];
    const int64_t r0 = p.total_rows * blockIdx.x / G, r1 = p.total_rows * (blockIdx.x + 1) / G;
    int64_t budget = kPrefetchBytes, r = r0;
    for (int m = 0; m < p.n_mats && budget > 0 && r < r1; ++m) {
      const int64_t m_lo = m ? p.row_end[m - 1] : 0, m_hi = p.row_end[m];
      if (r >= m_hi) continue;
      const int64_t e = r1 < m_hi ? r1 : m_hi;
      int64_t bytes = (e - r) * p.ld_codes[m];
      if (bytes > budget) bytes = budget;
      bytes &= ~(int64_t)15;
      if (bytes > 0) prefetch_l2(p.codes[m] + (r - m_lo) * p.ld_codes[m], (uint32_t)bytes);
      budget -= bytes;
      r = e;
    }
  };
  if (threadIdx.x == 0) {
    prefetch_rows(0);
    *abort_flag = 0;
  }
  if (lane == 0) {
    for (int st = 0; st < NS; ++st)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bars[warp * NS + st]))
                   : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  const uint32_t ring_w = smem_u32(ring) + (uint32_t)warp * NS * R * kStageRow;
  const uint32_t bar_w = smem_u32(&bars[warp * NS]);

  // Producer state, across products: product pk, row group pg, stage psj,
  // ring slot pst, stages left in product pk, stages issued in all.
  int pk = 0, pg = 0, psj = 0, pst = 0, pleft = 0, issued = 0;
  Work pw = plan(0);
  Bounds pbd;
  const uint8_t *pptr[R];
  auto prow_setup = [&]() {
    const GemvParams &p = sp.t[pk];
    const int rb = pw.first + pg * stride;
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
      const int rc = rb + rr < pw.rhi ? rb + rr : pw.rhi - 1;  // past the end: alias a valid row
      int m, i;
      locate(pbd, rc, m, i);
      pptr[rr] = p.codes[m] + (int64_t)i * p.ld_codes[m];
    }
  };
  auto enter = [&](int k) {  // producer moves to the first product >= k with stages for it
    for (pk = k; pk < sp.n; ++pk) {
      pw = plan(pk);
      if (pw.P > 0) break;
    }
    pg = psj = 0;
    pleft = pk < sp.n ? pw.P * pw.SPR : 0;
    if (pleft > 0) {
#pragma unroll
      for (int t = 0; t < QZ_MAX_GROUP; ++t) pbd.end[t] = (int)sp.t[pk].row_end[t];
      pbd.n = sp.t[pk].n_mats;
      prow_setup();
    }
  };
  auto issue_next = [&]() {
    if (lane == 0) {
      const int cpr = sp.t[pk].cpr;
      const int j0 = psj * kRPS;
      const int span = cpr - 32 * j0 < 32 * kRPS ? cpr - 32 * j0 : 32 * kRPS;  // chunks
      const uint32_t bytes = (uint32_t)span * 16u;
      const uint32_t bar = bar_w + pst * 8;
      asm volatile(
          "{\n\t.reg .b64 t;\n\t"
          "mbarrier.arrive.expect_tx.shared::cta.b64 t, [%0], %1;\n\t}" ::"r"(bar),
          "r"(bytes * R)
          : "memory");
#pragma unroll
      for (int rr = 0; rr < R; ++rr) {
        if (bytes == 0) break;  // no codes: the arrival alone completes the stage
        const uint32_t dst = ring_w + (uint32_t)(pst * R + rr) * kStageRow;
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
                "r"(dst),
            "l"(pptr[rr] + j0 * kRoundBytes), "r"(bytes), "r"(bar)
            : "memory");
      }
    }
    pst = pst + 1 == NS ? 0 : pst + 1;
    ++issued;
    if (--pleft == 0) {
      enter(pk + 1);
    } else if (++psj == pw.SPR) {
      psj = 0;
      ++pg;
      prow_setup();
    }
  };
  auto any_left = [&]() { return pk < sp.n && pleft > 0; };

  enter(0);
  for (int it = 0; it < NS - 1 && any_left(); ++it) issue_next();

  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const __half hzero = __ushort_as_half((unsigned short)0);
  Acc4 acc[R][B];
#pragma unroll
  for (int rr = 0; rr < R; ++rr) acc[rr][0][0] = acc[rr][0][1] = acc[rr][0][2] = acc[rr][0][3] = 0.f;
  bool ok = true;
  int cst = 0;            // consumer ring slot
  uint32_t cphase = 0;    // parity of the slot's current use
  int cidx = 0;           // stages consumed (ring position of the consumer)
  int fail_at = -1;       // first stage not consumed after an abort

  for (int k = 0; k < sp.n; ++k) {
    const GemvParams &p = sp.t[k];
    const Work w = plan(k);
    const int staged = (w.Jw > 0 ? w.Jw : 1) * 32;
    const uint32_t bstride = (uint32_t)staged * CS;
    __half *xo = reinterpret_cast<__half *>(smem_raw + bstride);
    // ---- wait until every CTA has stored its rows of products < k ----------
    if (k > 0) {
      __syncthreads();  // this CTA's stores of product k-1 precede the arrival
      if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(sp.sync, 1u);
        const unsigned target = (unsigned)(k * G);
        const unsigned long long t0 = gtimer();
        unsigned v = 0;
        for (;;) {
          asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(sp.sync) : "memory");
          if (v >= target) break;
          if (gtimer() - t0 > kWaitNs) {
            atomicExch(&g_gemv_error, 1);
            *(volatile int *)abort_flag = 1;
            break;
          }
        }
        if (k + 1 < sp.n) prefetch_rows(k + 1);
      }
      __syncthreads();
      if (*(volatile int *)abort_flag && ok) {
        ok = false;
        fail_at = cidx;
      }
    } else if (threadIdx.x == 0 && sp.n > 1) {
      prefetch_rows(1);
    }
    // ---- stage x of product k (L1 bypassed: it may be an earlier product's y)
    const int elems = staged * EPC;
    const __half *xb = p.x;
    if (ok) {
#pragma unroll 1
      for (int e0 = threadIdx.x * 8; e0 < elems; e0 += kThreads * 8) {
        uint32_t h[4];
        __half v[8];
        if constexpr (INT4) {
          int idx[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) idx[q] = e0 + q < p.kb ? __ldg(p.perm + p.n_out + e0 + q) : -1;
#pragma unroll
          for (int q = 0; q < 8; ++q) v[q] = idx[q] >= 0 ? __ldcg(xb + idx[q]) : hzero;
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) v[q] = e0 + q < p.kb ? __ldcg(xb + e0 + q) : hzero;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          h[q] = (uint32_t)__half_as_ushort(v[2 * q]) | ((uint32_t)__half_as_ushort(v[2 * q + 1]) << 16);
        *reinterpret_cast<uint4 *>(reinterpret_cast<char *>(xs) + (e0 / EPC) * CS + (e0 % EPC) * 2) =
            make_uint4(h[0], h[1], h[2], h[3]);
      }
      if constexpr (INT4) {
#pragma unroll 1
        for (int e = threadIdx.x; e < p.ocpr * 8; e += kThreads)
          xo[e] = e < p.n_out ? __ldcg(xb + __ldg(p.perm + e)) : hzero;
      }
    }
    __syncthreads();

    Bounds bd;
#pragma unroll
    for (int t = 0; t < QZ_MAX_GROUP; ++t) bd.end[t] = (int)p.row_end[t];
    bd.n = p.n_mats;
    const uint32_t lane_off = (uint32_t)lane * CS;
    for (int g = 0; g < w.P; ++g) {
      const int rb = w.first + g * stride;
      int mrow[R], irow[R];
      float srow[R];
      bool live[R];
      uint4 ov[R];
#pragma unroll
      for (int rr = 0; rr < R; ++rr) {
        live[rr] = rb + rr < w.rhi;
        locate(bd, live[rr] ? rb + rr : w.rhi - 1, mrow[rr], irow[rr]);
        srow[rr] = INT4 ? __ldg(p.scale[mrow[rr]] + irow[rr]) : __ldg(p.scale[mrow[rr]]);
        ov[rr] = make_uint4(0, 0, 0, 0);
        if (INT4 && lane < p.ocpr)
          ov[rr] = ld_stream(reinterpret_cast<const uint4 *>(
                                 p.w_out[mrow[rr]] + (int64_t)irow[rr] * p.ld_out[mrow[rr]]) +
                             lane);
      }
      for (int sj = 0; sj < w.SPR; ++sj) {
        if (ok && any_left()) {
          if (lane == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          issue_next();
        }
        if (ok) {
          ok = mbar_wait(bar_w + cst * 8, cphase);
          if (!ok) fail_at = cidx;
        }
        if (ok) {
          const uint32_t sbase = ring_w + (uint32_t)cst * R * kStageRow + lane * 16;
#pragma unroll
          for (int u = 0; u < kRPS; ++u) {
            const int j = sj * kRPS + u;
            if (j < w.Jw) {  // warp-uniform
              uint4 v[R];
#pragma unroll
              for (int rr = 0; rr < R; ++rr) {
                const uint32_t a = sbase + (uint32_t)rr * kStageRow + u * kRoundBytes;
                asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                             : "=r"(v[rr].x), "=r"(v[rr].y), "=r"(v[rr].z), "=r"(v[rr].w)
                             : "r"(a));
              }
              const uint32_t o = lane_off + (uint32_t)j * kRound;
              if constexpr (INT4) int4_chunk<B, R>(v, xs, o, bstride, acc);
              else int8_chunk<B, R>(v, xs, o, bstride, acc);
            }
          }
        }
        __syncwarp();
        ++cidx;
        if (++cst == NS) {
          cst = 0;
          cphase ^= 1u;
        }
      }
      float outl[R][2];
#pragma unroll
      for (int rr = 0; rr < R; ++rr) outl[rr][0] = outl[rr][1] = 0.0f;
      if constexpr (INT4) {
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
          const uint4 *orow = reinterpret_cast<const uint4 *>(p.w_out[mrow[rr]] +
                                                              (int64_t)irow[rr] * p.ld_out[mrow[rr]]);
#pragma unroll 1
          for (int c = lane; c < p.ocpr; c += 32) {
            const uint4 v = c == lane ? ov[rr] : ld_stream(orow + c);
            const uint4 xv = *reinterpret_cast<const uint4 *>(reinterpret_cast<const char *>(xo) + c * 16);
            fhfma2(outl[rr][0], outl[rr][1], v.x, xv.x);
            fhfma2(outl[rr][0], outl[rr][1], v.y, xv.y);
            fhfma2(outl[rr][0], outl[rr][1], v.z, xv.z);
            fhfma2(outl[rr][0], outl[rr][1], v.w, xv.w);
          }
        }
      }
#pragma unroll
      for (int rr = 0; rr < R; ++rr) {
        const float bg = (acc[rr][0][0] + acc[rr][0][2]) + (acc[rr][0][1] + acc[rr][0][3]) * 0.0625f;
        const float yl = warp_sum(fmaf(srow[rr], bg, outl[rr][0] + outl[rr][1]));
        if (lane == 0 && live[rr] && ok) p.y[mrow[rr]][irow[rr]] = __float2half_rn(yl);
        acc[rr][0][0] = acc[rr][0][1] = acc[rr][0][2] = acc[rr][0][3] = 0.f;
      }
    }
  }
  // ---- the last CTA past the final product resets the counter ---------------
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned old = atomicAdd(sp.sync, 1u);
    if (old == (unsigned)(sp.n * G - 1)) atomicExch(sp.sync, 0u);
  }
  // A warp that gave up a wait may still have copies in flight into its
  // ring; give them a bounded time to land before the CTA's shared memory goes.
  if (!ok && lane == 0) ring_drain<NS>(bar_w, fail_at, issued);
}

// Shared memory of gemv_kernel with W warps: staged inputs, then the ring
// and its barriers as the kernel carves them (Ring<B> is the same for every
// B > 1).
size_t gemv_smem_bytes_w(bool int4, int B, const GemvParams &p, int W, bool zc = false) {
  const size_t cs = int4 ? 80 : 48;  // padded staged fp16 bytes per chunk
  const size_t rounds = p.cpr > 0 ? (size_t)(p.cpr + 31) / 32 : 1;
  const size_t staged = (rounds * 32 * cs + (int4 ? (size_t)p.ocpr * 16 : 0)) * (size_t)B;
  const size_t NS = B == 1 ? Ring<1>::NS : Ring<2>::NS;
  const size_t R = B == 1 ? Ring<1>::R : Ring<2>::R;
  const size_t stage_row = B == 1 ? Ring<1>::STAGE_ROW : Ring<2>::STAGE_ROW;
  const size_t ring = zc ? 0 : (size_t)W * NS * R * stage_row;
  return ((staged + 127) & ~(size_t)127) + ring + (size_t)W * NS * 8;
}

template <bool INT4, int B, int W, bool ZC = false>
qz_status launch_w(const GemvParams &p, const DeviceInfo &di, cudaStream_t s) {
  constexpr int R = Ring<B>::R;
  auto kern = gemv_kernel<INT4, B, W, ZC>;
  const size_t smem = gemv_smem_bytes_w(INT4, B, p, W, ZC);
  if (smem > (size_t)di.max_smem_optin) return QZ_ERR_UNSUPPORTED;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return cuda_status(e);
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, W * 32, smem);
  if (e != cudaSuccess) return cuda_status(e);
  if (occ < 1) return QZ_ERR_UNSUPPORTED;
  // Whole waves only: every SM gets the same number of CTAs (and CTAs equal
  // row ranges), so no SM carries a second CTA while another idles.
  int64_t per_sm = occ;
  while (per_sm > 1 && (int64_t)di.sms * per_sm * W * R > p.total_rows * 2) --per_sm;
  int64_t grid = (int64_t)di.sms * per_sm;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(W * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.overlap ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return cuda_status(e);
  return launch_status();
}

// Batch 1 takes 20 warps per CTA when their rings fit in shared memory:
// more bytes in flight per SM (measured on GB300: Gemma INT8 +1%, 3B INT4
// +5%, 70B INT4 +2%; 24 warps lost 1% on Gemma).  Batches 2..4 keep 16.
template <bool INT4, int B>
qz_status launch_t(const GemvParams &p, cudaStream_t s) {
  DeviceInfo di;
  qz_status st = device_info(&di);
  if (st != QZ_OK) return st;
  const size_t cap = (size_t)di.max_smem_optin;
  if constexpr (B == 1)
    if (gemv_smem_bytes_w(INT4, B, p, 20) <= cap) return launch_w<INT4, B, 20>(p, di, s);
  return launch_w<INT4, B, 16>(p, di, s);
}

}  // namespace

// The 16-warp size: the least any batch-1..4 launch needs (the path choice
// between CUDA cores and tensor cores tests this).
size_t gemv_smem_bytes(bool int4, int B, const GemvParams &p) {
  return gemv_smem_bytes_w(int4, B, p, kWarps);
}

size_t gemv_seq_smem_bytes(bool int4, const SeqParams &sp, uint32_t *xs_bytes) {
  const size_t cs = int4 ? 80 : 48;
  size_t xsb = 0;
  for (int k = 0; k < sp.n; ++k) {
    const size_t rounds = sp.t[k].cpr > 0 ? (size_t)(sp.t[k].cpr + 31) / 32 : 1;
    const size_t need = rounds * 32 * cs + (int4 ? (size_t)sp.t[k].ocpr * 16 : 0);
    if (need > xsb) xsb = need;
  }
  xsb = (xsb + 127) & ~(size_t)127;
  if (xs_bytes) *xs_bytes = (uint32_t)xsb;
  const size_t ring = (size_t)kWarps * Ring<1>::NS * Ring<1>::R * Ring<1>::RPS * kRoundBytes;
  return xsb + ring + (size_t)kWarps * Ring<1>::NS * 8 + 16;
}

qz_status launch_gemv_seq(bool int4, SeqParams &sp, cudaStream_t s) {
  DeviceInfo di;
  qz_status st = device_info(&di);
  if (st != QZ_OK) return st;
  const size_t smem = gemv_seq_smem_bytes(int4, sp, &sp.xs_bytes);
  if (smem > (size_t)di.max_smem_optin) return QZ_ERR_UNSUPPORTED;
  auto kern = int4 ? gemv_seq_kernel<true> : gemv_seq_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_status(e);
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem);
  if (e != cudaSuccess) return cuda_status(e);
  if (occ < 1) return QZ_ERR_UNSUPPORTED;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)di.sms);  // one CTA per SM: all resident for the barriers
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = sp.t[0].overlap ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, sp);
  if (e != cudaSuccess) return cuda_status(e);
  return launch_status();
}

qz_status read_gemv_error(int *code, int clear) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_gemv_error, sizeof(int));
  if (e != cudaSuccess) return cuda_status(e);
  if (clear && v) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_gemv_error, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_status(e);
  }
  *code = v;
  return QZ_OK;
}

// Batch-1 product with the weights read in place (zero-copy), 20 warps.
qz_status launch_gemv_mapped(bool int4, const GemvParams &p, cudaStream_t s) {
  DeviceInfo di;
  qz_status st = device_info(&di);
  if (st != QZ_OK) return st;
  return int4 ? launch_w<true, 1, 20, true>(p, di, s) : launch_w<false, 1, 20, true>(p, di, s);
}

size_t gemv_mapped_smem_bytes(bool int4, const GemvParams &p) {
  return gemv_smem_bytes_w(int4, 1, p, 20, true);
}

qz_status launch_gemv(bool int4, int B, const GemvParams &p, cudaStream_t s) {
  if (int4) {
    switch (B) {
      case 1: return launch_t<true, 1>(p, s);
      case 2: return launch_t<true, 2>(p, s);
      case 3: return launch_t<true, 3>(p, s);
      case 4: return launch_t<true, 4>(p, s);
    }
  } else {
    switch (B) {
      case 1: return launch_t<false, 1>(p, s);
      case 2: return launch_t<false, 2>(p, s);
      case 3: return launch_t<false, 3>(p, s);
      case 4: return launch_t<false, 4>(p, s);
    }
  }
  return QZ_ERR_UNSUPPORTED;
}

}  // namespace qz
