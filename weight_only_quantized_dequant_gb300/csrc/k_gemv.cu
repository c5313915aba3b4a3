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
//    as fp32 and, for INT4, pre-scaled by 16^-(t' mod 4) so that one LOP3
//    turns a nibble into the fp32 number 2^23 + (q+8)*16^p and one packed
//    subtract leaves q*16^p exactly.  Staged chunks are padded by 16 bytes
//    (conflict-free for the 8 lanes of a 128-bit phase), so every shared read
//    is a per-lane base plus an immediate offset.
//  * A warp computes R rows at once: each staged granule is read once for
//    all R rows, halving the shared-memory traffic per weight.
//  * Loads are software-pipelined in registers: the next group of chunks
//    (possibly of the next rows) is issued before the current one is
//    consumed, and each warp bulk-prefetches its following rows into L2.
//  * Products use the sm_100+ packed fp32x2 add/FMA (two weights per issue).
//  * CTAs own contiguous, equal row ranges; the grid is the SM count times
//    the resident CTAs per SM.
#include "qz_internal.cuh"

namespace qz {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int64_t kPrefetchBytes = 64 * 1024;  // per CTA, issued before the wait

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
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

__device__ __forceinline__ float4 lds(const float4 *base, uint32_t byte_off) {
  return *reinterpret_cast<const float4 *>(reinterpret_cast<const char *>(base) + byte_off);
}

// Outlier inputs: granule g (0/1) of outlier chunk c, XOR-swizzled.
__device__ __forceinline__ int ogidx(int c, int g) { return c * 2 + (g ^ ((c >> 2) & 1)); }

// 32 nibbles of one chunk of each of R rows against the staged input at byte
// offset `o` (granule g at o + 16 g).  For nibble p (0..3) of a half-word,
// (w & 0xF<<4p) ^ (0x4B000000 | 8<<4p) is 2^23 + (q+8)*16^p; subtracting
// 2^23 + 8*16^p leaves q*16^p, and the staged input is x*16^-p.
template <int B, int R>
__device__ __forceinline__ void int4_chunk(const uint4 (&v)[R], const float4 *xs, uint32_t o,
                                           uint32_t bstride, float2 (&acc)[R][B][2]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float4 xv[B];
#pragma unroll
      for (int b = 0; b < B; ++b) xv[b] = lds(xs, o + (2 * k + h) * 16 + b * bstride);
#pragma unroll
      for (int rr = 0; rr < R; ++rr) {
        const uint32_t w = k == 0 ? v[rr].x : k == 1 ? v[rr].y : k == 2 ? v[rr].z : v[rr].w;
        const uint32_t ww = h ? (w >> 16) : w;
        const float f0 = __uint_as_float(and_xor(ww, 0x000Fu, 0x4B000008u));
        const float f1 = __uint_as_float(and_xor(ww, 0x00F0u, 0x4B000080u));
        const float f2 = __uint_as_float(and_xor(ww, 0x0F00u, 0x4B000800u));
        const float f3 = __uint_as_float(and_xor(ww, 0xF000u, 0x4B008000u));
        const float2 qa = __fadd2_rn(make_float2(f0, f1),
                                     make_float2(-8388616.0f, -8388736.0f));
        const float2 qb = __fadd2_rn(make_float2(f2, f3),
                                     make_float2(-8390656.0f, -8421376.0f));
#pragma unroll
        for (int b = 0; b < B; ++b) {
          acc[rr][b][0] = __ffma2_rn(qa, make_float2(xv[b].x, xv[b].y), acc[rr][b][0]);
          acc[rr][b][1] = __ffma2_rn(qb, make_float2(xv[b].z, xv[b].w), acc[rr][b][1]);
        }
      }
    }
  }
}

// 16 int8 codes of one chunk of each of R rows.  XOR 0x80 makes each byte the
// offset-binary u = q + 128; PRMT drops it into the low byte of 2^23's bit
// pattern, and subtracting 2^23 + 128 leaves q exactly.
template <int B, int R>
__device__ __forceinline__ void int8_chunk(const uint4 (&v)[R], const float4 *xs, uint32_t o,
                                           uint32_t bstride, float2 (&acc)[R][B][2]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float4 xv[B];
#pragma unroll
    for (int b = 0; b < B; ++b) xv[b] = lds(xs, o + k * 16 + b * bstride);
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
      const uint32_t w =
          (k == 0 ? v[rr].x : k == 1 ? v[rr].y : k == 2 ? v[rr].z : v[rr].w) ^ 0x80808080u;
      const float f0 = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440));
      const float f1 = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7441));
      const float f2 = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7442));
      const float f3 = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7443));
      const float2 qa = __fadd2_rn(make_float2(f0, f1),
                                   make_float2(-8388736.0f, -8388736.0f));
      const float2 qb = __fadd2_rn(make_float2(f2, f3),
                                   make_float2(-8388736.0f, -8388736.0f));
#pragma unroll
      for (int b = 0; b < B; ++b) {
        acc[rr][b][0] = __ffma2_rn(qa, make_float2(xv[b].x, xv[b].y), acc[rr][b][0]);
        acc[rr][b][1] = __ffma2_rn(qb, make_float2(xv[b].z, xv[b].w), acc[rr][b][1]);
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
// them in registers.  A stage is kRPS rounds (32 chunks of 16 bytes) of each
// of the warp's R rows.  Every wait is bounded in time.
// ---------------------------------------------------------------------------
__device__ int g_gemv_error = 0;  // 1 if a bounded wait gave up (read by qz_device_error)

constexpr int kRPS = 2;                        // rounds per stage
constexpr uint32_t kRoundBytes = 512;          // 32 chunks x 16 bytes
constexpr uint32_t kStageRow = kRPS * kRoundBytes;
constexpr unsigned long long kWaitNs = 2000000000ull;

template <int B>
struct Ring {
  static constexpr int NS = B == 1 ? 3 : 2;    // stages per warp
  static constexpr int R = B == 1 ? 2 : 1;     // rows per warp
};

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

// Row r of the launch -> (matrix, row inside it).
__device__ __forceinline__ void locate(const GemvParams &p, int64_t r, int &m, int64_t &i) {
  m = 0;
#pragma unroll
  for (int t = 0; t < QZ_MAX_GROUP - 1; ++t) m += (t < p.n_mats - 1 && r >= p.row_end[t]) ? 1 : 0;
  i = r - (m ? p.row_end[m - 1] : 0);
}

template <bool INT4, int B>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_kernel(const __grid_constant__ GemvParams p) {
  constexpr int R = Ring<B>::R, NS = Ring<B>::NS;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  constexpr int GPC = INT4 ? 8 : 4;        // 16-byte granules per code chunk
  constexpr int EPC = GPC * 4;             // inputs per code chunk
  constexpr uint32_t CS = (GPC + 1) * 16;  // staged bytes per chunk (padded)
  const int cpr = p.cpr;
  const int Jw = (cpr + 31) >> 5;          // rounds of 32 chunks per row
  const int staged = (Jw > 0 ? Jw : 1) * 32;
  const uint32_t bstride = (uint32_t)staged * CS;  // bytes per batch row
  const int ostride = p.ocpr * 2;          // outlier granules per batch row
  float4 *xs = reinterpret_cast<float4 *>(smem_raw);
  float4 *xo = reinterpret_cast<float4 *>(smem_raw + B * bstride);
  uint8_t *ring = smem_raw + (((size_t)B * bstride + (size_t)B * ostride * 16 + 127) & ~(size_t)127);
  uint64_t *bars = reinterpret_cast<uint64_t *>(ring + (size_t)kWarps * NS * R * kStageRow);

  const int64_t r0 = p.total_rows * blockIdx.x / gridDim.x;
  const int64_t r1 = p.total_rows * (blockIdx.x + 1) / gridDim.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // The first rows of this CTA are pulled into L2 right away.  With
  // programmatic overlap this CTA may start while the previous kernel on the
  // stream is still running; the weights are static by the caller's promise,
  // and x (which that kernel may produce) is only read after the wait.
  if (threadIdx.x == 0) {
    int64_t budget = kPrefetchBytes;
    int64_t r = r0;
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
  }
  if (lane == 0) {
    for (int st = 0; st < NS; ++st)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bars[warp * NS + st]))
                   : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // let the next kernel on the stream get scheduled as SMs free up
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ---- stage x (gathered through perm for INT4) in shared memory ---------
  float *xsf = reinterpret_cast<float *>(xs);
  const int elems = staged * EPC;
#pragma unroll 1
  for (int b = 0; b < B; ++b) {
    const __half *xb = p.x + b * p.ldx;
#pragma unroll 1
    for (int e = threadIdx.x; e < elems; e += kThreads) {
      float val = 0.0f;
      if (e < p.kb) {
        if constexpr (INT4) {
          const int ch = __ldg(p.perm + p.n_out + e);
          const float sc = (e & 3) == 0   ? 1.0f
                           : (e & 3) == 1 ? 0.0625f
                           : (e & 3) == 2 ? 0.00390625f
                                          : 0.000244140625f;
          val = __half2float(xb[ch]) * sc;  // exact: power-of-two scaling
        } else {
          val = __half2float(xb[e]);
        }
      }
      const int c = e / EPC, u = e % EPC;
      xsf[(b * bstride + c * CS + (u >> 2) * 16) / 4 + (u & 3)] = val;
    }
    if constexpr (INT4) {
      float *xof = reinterpret_cast<float *>(xo);
#pragma unroll 1
      for (int e = threadIdx.x; e < ostride * 4; e += kThreads) {
        const float val = e < p.n_out ? __half2float(xb[__ldg(p.perm + e)]) : 0.0f;
        xof[(b * ostride + ogidx(e >> 3, (e & 7) >> 2)) * 4 + (e & 3)] = val;
      }
    }
  }
  __syncthreads();

  // ---- each warp: row groups of R rows, streamed through its ring -----------
  const int64_t first = r0 + (int64_t)warp * R;
  const int64_t stride = (int64_t)kWarps * R;
  if (first >= r1) return;  // no barrier follows
  const int64_t P = (r1 - first + stride - 1) / stride;  // row groups of this warp
  const int SPR = (Jw + kRPS - 1) / kRPS;                 // stages per row group
  const int64_t items = P * SPR;
  const uint32_t lane_off = (uint32_t)lane * CS;
  constexpr uint32_t kRound = 32u * CS;  // staged bytes per round of 32 chunks
  const uint32_t ring_w = smem_u32(ring) + (uint32_t)warp * NS * R * kStageRow;
  const uint32_t bar_w = smem_u32(&bars[warp * NS]);

  // lane 0: copy stage `it` (row group it / SPR, rounds from (it % SPR) * kRPS)
  auto issue = [&](int64_t it) {
    const int64_t k = it / SPR;
    const int j0 = (int)(it - k * SPR) * kRPS;
    const int st = (int)(it % NS);
    const int span = cpr - 32 * j0 < 32 * kRPS ? cpr - 32 * j0 : 32 * kRPS;  // chunks
    const uint32_t bytes = (uint32_t)span * 16u;
    const uint32_t bar = bar_w + st * 8;
    asm volatile(
        "{\n\t.reg .b64 t;\n\t"
        "mbarrier.arrive.expect_tx.shared::cta.b64 t, [%0], %1;\n\t}" ::"r"(bar),
        "r"(bytes * R)
        : "memory");
    const int64_t rb = first + k * stride;
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
      const int64_t rc = rb + rr < r1 ? rb + rr : r1 - 1;  // past the end: alias a valid row
      int m;
      int64_t i;
      locate(p, rc, m, i);
      const uint8_t *src = p.codes[m] + i * p.ld_codes[m] + (size_t)j0 * kRoundBytes;
      const uint32_t dst = ring_w + (uint32_t)(st * R + rr) * kStageRow;
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
              "r"(dst),
          "l"(src), "r"(bytes), "r"(bar)
          : "memory");
    }
  };

  if (lane == 0)
    for (int64_t it = 0; it < NS - 1 && it < items; ++it) issue(it);

  float2 acc[R][B][2];
#pragma unroll
  for (int rr = 0; rr < R; ++rr)
#pragma unroll
    for (int b = 0; b < B; ++b) acc[rr][b][0] = acc[rr][b][1] = make_float2(0.f, 0.f);

  bool ok = true;
  int64_t k = 0;   // row group
  int sj = 0;      // stage inside the row group
  const int64_t groups_total = P;
  for (int64_t g = 0; g < groups_total; ++g) {
    // rows of this group: scales, matrix, and the outlier rows into L2
    const int64_t rb = first + g * stride;
    int mrow[R];
    int64_t irow[R];
    float srow[R];
    bool live[R];
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
      live[rr] = rb + rr < r1;
      locate(p, live[rr] ? rb + rr : r1 - 1, mrow[rr], irow[rr]);
      srow[rr] = INT4 ? __ldg(p.scale[mrow[rr]] + irow[rr]) : __ldg(p.scale[mrow[rr]]);
      if (INT4 && p.ocpr && lane == 8 + rr)
        prefetch_l2(p.w_out[mrow[rr]] + irow[rr] * p.ld_out[mrow[rr]], (uint32_t)p.ocpr * 16u);
    }
    for (sj = 0; sj < SPR; ++sj) {
      const int64_t it = g * SPR + sj;
      if (ok && lane == 0 && it + NS - 1 < items) {
        // the stage being refilled was read by every lane before the last
        // __syncwarp; order those reads before the async-proxy write
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        issue(it + NS - 1);
      }
      const int st = (int)(it % NS);
      if (ok) ok = mbar_wait(bar_w + st * 8, (uint32_t)((it / NS) & 1));
      if (ok) {
        const uint32_t sbase = ring_w + (uint32_t)st * R * kStageRow;
#pragma unroll
        for (int u = 0; u < kRPS; ++u) {
          const int j = sj * kRPS + u;
          if (j < Jw) {  // warp-uniform
            const bool in = lane + 32 * j < cpr;
            uint4 v[R];
#pragma unroll
            for (int rr = 0; rr < R; ++rr) {
              v[rr] = make_uint4(0, 0, 0, 0);
              if (in) {
                const uint32_t a = sbase + (uint32_t)rr * kStageRow + u * kRoundBytes + lane * 16;
                asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                             : "=r"(v[rr].x), "=r"(v[rr].y), "=r"(v[rr].z), "=r"(v[rr].w)
                             : "r"(a));
              }
            }
            const uint32_t o = lane_off + (uint32_t)j * kRound;
            if constexpr (INT4) int4_chunk<B, R>(v, xs, o, bstride, acc);
            else int8_chunk<B, R>(v, xs, o, bstride, acc);
          }
        }
      }
      __syncwarp();
    }
    (void)k;
    // ---- row epilogue: outliers, scale, reduction, store --------------------
    float outl[R][B];
#pragma unroll
    for (int rr = 0; rr < R; ++rr)
#pragma unroll
      for (int b = 0; b < B; ++b) outl[rr][b] = 0.0f;
    if constexpr (INT4) {
#pragma unroll
      for (int rr = 0; rr < R; ++rr) {
        const uint4 *orow =
            reinterpret_cast<const uint4 *>(p.w_out[mrow[rr]] + irow[rr] * p.ld_out[mrow[rr]]);
#pragma unroll 1
        for (int c = lane; c < p.ocpr; c += 32) {
          const uint4 v = ld_stream(orow + c);
          const float2 h0 = __half22float2(*reinterpret_cast<const __half2 *>(&v.x));
          const float2 h1 = __half22float2(*reinterpret_cast<const __half2 *>(&v.y));
          const float2 h2 = __half22float2(*reinterpret_cast<const __half2 *>(&v.z));
          const float2 h3 = __half22float2(*reinterpret_cast<const __half2 *>(&v.w));
#pragma unroll
          for (int b = 0; b < B; ++b) {
            const float4 xa = xo[b * ostride + ogidx(c, 0)];
            const float4 xc = xo[b * ostride + ogidx(c, 1)];
            float a = outl[rr][b];
            a = fmaf(h0.x, xa.x, a); a = fmaf(h0.y, xa.y, a);
            a = fmaf(h1.x, xa.z, a); a = fmaf(h1.y, xa.w, a);
            a = fmaf(h2.x, xc.x, a); a = fmaf(h2.y, xc.y, a);
            a = fmaf(h3.x, xc.z, a); a = fmaf(h3.y, xc.w, a);
            outl[rr][b] = a;
          }
        }
      }
    }
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const float bg =
            (acc[rr][b][0].x + acc[rr][b][0].y) + (acc[rr][b][1].x + acc[rr][b][1].y);
        // y = s_i * background + outliers, combined per lane, one reduction
        const float yl = warp_sum(fmaf(srow[rr], bg, outl[rr][b]));
        if (lane == 0 && live[rr]) p.y[mrow[rr]][b * p.ldy + irow[rr]] = __float2half_rn(yl);
        acc[rr][b][0] = acc[rr][b][1] = make_float2(0.f, 0.f);
      }
    }
  }
  // A warp that gave up a wait still has copies in flight into its ring;
  // give them a bounded time to land before the CTA's shared memory goes.
  if (!ok && lane == 0) {
    for (int st = 0; st < NS; ++st) {
      const unsigned long long t0 = gtimer();
      while (!mbar_try(bar_w + st * 8, 0) && !mbar_try(bar_w + st * 8, 1) &&
             gtimer() - t0 < kWaitNs) {
      }
    }
  }
}

template <bool INT4, int B>
qz_status launch_t(const GemvParams &p, cudaStream_t s) {
  constexpr int R = Ring<B>::R;
  auto kern = gemv_kernel<INT4, B>;
  DeviceInfo di;
  qz_status st = device_info(&di);
  if (st != QZ_OK) return st;
  const size_t smem = gemv_smem_bytes(INT4, B, p);
  if (smem > (size_t)di.max_smem_optin) return QZ_ERR_UNSUPPORTED;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return cuda_status(e);
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem);
  if (e != cudaSuccess) return cuda_status(e);
  if (occ < 1) return QZ_ERR_UNSUPPORTED;
  // Whole waves only: every SM gets the same number of CTAs (and CTAs equal
  // row ranges), so no SM carries a second CTA while another idles.
  int64_t per_sm = occ;
  while (per_sm > 1 && (int64_t)di.sms * per_sm * kWarps * R > p.total_rows * 2) --per_sm;
  int64_t grid = (int64_t)di.sms * per_sm;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
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

}  // namespace

size_t gemv_smem_bytes(bool int4, int B, const GemvParams &p) {
  const size_t cs = int4 ? 144 : 80;  // padded staged bytes per chunk
  const size_t rounds = p.cpr > 0 ? (size_t)(p.cpr + 31) / 32 : 1;
  const size_t staged = (rounds * 32 * cs + (int4 ? (size_t)p.ocpr * 32 : 0)) * (size_t)B;
  const size_t R = B == 1 ? 2 : 1, NS = B == 1 ? 3 : 2;
  const size_t ring = (size_t)kWarps * NS * R * kStageRow;
  return ((staged + 127) & ~(size_t)127) + ring + (size_t)kWarps * NS * 8;
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
