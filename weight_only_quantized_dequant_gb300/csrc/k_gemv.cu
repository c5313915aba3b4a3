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
// Design (HBM-bound stream):
//  * x is gathered through the permutation into shared memory once per CTA,
//    converted to fp32 and, for INT4, pre-scaled by 16^-(t' mod 4) so that a
//    nibble can be turned into an exact fp32 multiple of 16^p with one LOP3
//    (OR-ing it into the mantissa of 2^23) and one packed subtract.
//  * Each warp streams whole rows with 16-byte non-allocating loads, four
//    chunks per lane in flight; shared-memory reads of x are swizzled so the
//    eight lanes of each 128-bit phase hit distinct banks.
//  * Products use the sm_100+ packed fp32x2 add/FMA (two weights per issue).
//  * CTAs own contiguous, equal row ranges; the grid is the SM count times
//    the resident CTAs per SM.
#include "qz_internal.cuh"

namespace qz {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 6;  // 16-byte chunks per lane in flight
constexpr int64_t kPrefetchBytes = 64 * 1024;  // per CTA, issued before the wait

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// Index of 16-byte granule g of code chunk c in the staged input.  GPC is the
// number of granules per chunk (8 for INT4: 32 nibbles -> 32 floats; 4 for
// INT8: 16 bytes -> 16 floats; 2 for the fp16 outliers: 8 halves -> 8 floats).
// Lane L reads chunk c = L + 32u, so the XOR keeps the 8 lanes of one LDS.128
// phase on distinct bank groups.
template <int GPC>
__device__ __forceinline__ int gidx(int c, int g) {
  if constexpr (GPC == 8) return c * 8 + (g ^ (c & 7));
  else if constexpr (GPC == 4) return c * 4 + (g ^ ((c >> 1) & 3));
  else return c * 2 + (g ^ ((c >> 2) & 1));
}

// (a & b) ^ c in one LOP3 (truth table 0x6A).
__device__ __forceinline__ uint32_t and_xor(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Shared-memory read of one staged granule (4 fp32 inputs) at a byte offset.
__device__ __forceinline__ float4 lds(const float4 *base, uint32_t byte_off) {
  return *reinterpret_cast<const float4 *>(reinterpret_cast<const char *>(base) + byte_off);
}

// 32 nibbles of one chunk against the staged (pre-scaled) input.
// For nibble p (0..3) of a half-word, (w & 0xF<<4p) ^ (0x4B000000 | 8<<4p) is
// the fp32 number 2^23 + (q+8)*16^p; subtracting 2^23 + 8*16^p leaves q*16^p
// exactly, and the input was staged as x*16^-p, so each FMA adds q*x exactly.
// goff[g] is the lane's byte offset of granule g inside its chunk (the swizzle
// only depends on the lane), cbase the byte offset of the chunk, bstride the
// bytes between batch rows of the staged input.
template <int B>
__device__ __forceinline__ void int4_chunk(const uint4 v, const float4 *xs,
                                           const uint32_t (&goff)[8], uint32_t cbase,
                                           uint32_t bstride, float2 (&acc)[B][2]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t ww = h ? (w[k] >> 16) : w[k];
      const float f0 = __uint_as_float(and_xor(ww, 0x000Fu, 0x4B000008u));
      const float f1 = __uint_as_float(and_xor(ww, 0x00F0u, 0x4B000080u));
      const float f2 = __uint_as_float(and_xor(ww, 0x0F00u, 0x4B000800u));
      const float f3 = __uint_as_float(and_xor(ww, 0xF000u, 0x4B008000u));
      const float2 qa = __fadd2_rn(make_float2(f0, f1),
                                   make_float2(-8388616.0f, -8388736.0f));
      const float2 qb = __fadd2_rn(make_float2(f2, f3),
                                   make_float2(-8390656.0f, -8421376.0f));
      const uint32_t o = cbase + goff[2 * k + h];
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const float4 xv = lds(xs, o + b * bstride);
        acc[b][0] = __ffma2_rn(qa, make_float2(xv.x, xv.y), acc[b][0]);
        acc[b][1] = __ffma2_rn(qb, make_float2(xv.z, xv.w), acc[b][1]);
      }
    }
  }
}

// 16 int8 codes of one chunk.  XOR 0x80 makes each byte the offset-binary
// u = q + 128; PRMT drops it into the low byte of 2^23's bit pattern, and
// subtracting 2^23 + 128 leaves q exactly.
template <int B>
__device__ __forceinline__ void int8_chunk(const uint4 v, const float4 *xs,
                                           const uint32_t (&goff)[8], uint32_t cbase,
                                           uint32_t bstride, float2 (&acc)[B][2]) {
  const uint32_t w[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u,
                         v.z ^ 0x80808080u, v.w ^ 0x80808080u};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float f0 = __uint_as_float(__byte_perm(w[k], 0x4B000000u, 0x7440));
    const float f1 = __uint_as_float(__byte_perm(w[k], 0x4B000000u, 0x7441));
    const float f2 = __uint_as_float(__byte_perm(w[k], 0x4B000000u, 0x7442));
    const float f3 = __uint_as_float(__byte_perm(w[k], 0x4B000000u, 0x7443));
    const float2 qa = __fadd2_rn(make_float2(f0, f1),
                                 make_float2(-8388736.0f, -8388736.0f));
    const float2 qb = __fadd2_rn(make_float2(f2, f3),
                                 make_float2(-8388736.0f, -8388736.0f));
    const uint32_t o = cbase + goff[k];
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const float4 xv = lds(xs, o + b * bstride);
      acc[b][0] = __ffma2_rn(qa, make_float2(xv.x, xv.y), acc[b][0]);
      acc[b][1] = __ffma2_rn(qb, make_float2(xv.z, xv.w), acc[b][1]);
    }
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <bool INT4, int B>
__global__ void __launch_bounds__(kThreads, (B == 1 ? 2 : 1))
    gemv_kernel(const __grid_constant__ GemvParams p) {
  extern __shared__ float4 smem[];
  constexpr int GPC = INT4 ? 8 : 4;       // granules per code chunk
  constexpr int EPC = GPC * 4;            // elements per code chunk
  const int cps = p.cpr > 32 ? p.cpr : 32;  // staged chunks (>= 32: one per lane)
  const int gstride = cps * GPC;          // background granules per batch row
  const int ostride = p.ocpr * 2;         // outlier granules per batch row
  float4 *xs = smem;
  float4 *xo = smem + B * gstride;

  const int64_t r0 = p.total_rows * blockIdx.x / gridDim.x;
  const int64_t r1 = p.total_rows * (blockIdx.x + 1) / gridDim.x;

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
      if (bytes > 0) {
        const uint8_t *src = p.codes[m] + (r - m_lo) * p.ld_codes[m];
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"((uint32_t)bytes)
                     : "memory");
      }
      budget -= bytes;
      r = e;
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // let the next kernel on the stream get scheduled as SMs free up
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ---- stage x (gathered through perm for INT4) in shared memory ---------
  float *xsf = reinterpret_cast<float *>(xs);
  const int elems = cps * EPC;
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
      xsf[(b * gstride + gidx<GPC>(c, u >> 2)) * 4 + (u & 3)] = val;
    }
    if constexpr (INT4) {
      float *xof = reinterpret_cast<float *>(xo);
#pragma unroll 1
      for (int e = threadIdx.x; e < ostride * 4; e += kThreads) {
        const float val = e < p.n_out ? __half2float(xb[__ldg(p.perm + e)]) : 0.0f;
        xof[(b * ostride + gidx<2>(e >> 3, (e & 7) >> 2)) * 4 + (e & 3)] = val;
      }
    }
  }
  __syncthreads();

  // ---- one warp per row ----------------------------------------------------
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Lane L reads chunks c = L + 32j.  The staging swizzle of a granule only
  // depends on c's low bits, i.e. on the lane, so the byte offsets of the
  // GPC granules inside a chunk are fixed per lane.
  uint32_t goff[8];
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const int sw = GPC == 8 ? (lane & 7) : ((lane >> 1) & 3);
    goff[g] = (uint32_t)((lane * GPC + ((g % GPC) ^ sw)) * 16);
  }
  const uint32_t bstride = (uint32_t)gstride * 16u;
  constexpr uint32_t kChunkStep = 32u * GPC * 16u;  // bytes between a lane's chunks
  // Warp-uniform trip counts: rounds where every lane has a chunk run without
  // predicates; the last partial round (if any) runs predicated, and lanes
  // past the row's end load zero codes against a valid staged slot (at least
  // 32 chunks are always staged), so they add exact zeros.  No divergence.
  const int cpr = p.cpr;
  const int Jfull = cpr >> 5;             // rounds in which all 32 lanes have a chunk
  const int Jw = (cpr + 31) >> 5;         // all rounds
  const int64_t total_rows = p.total_rows;
  (void)total_rows;
#pragma unroll 1
  for (int64_t r = r0 + warp; r < r1; r += kWarps) {
    int m = 0;
#pragma unroll
    for (int t = 0; t < QZ_MAX_GROUP - 1; ++t)
      m += (t < p.n_mats - 1 && r >= p.row_end[t]) ? 1 : 0;
    const int64_t i = r - (m ? p.row_end[m - 1] : 0);
    const float s = INT4 ? __ldg(p.scale[m] + i) : __ldg(p.scale[m]);
    const int64_t ldc = p.ld_codes[m];
    const uint4 *row = reinterpret_cast<const uint4 *>(p.codes[m] + i * ldc) + lane;
    // Bulk-prefetch the warp's next row into L2 while this one is computed:
    // DRAM keeps streaming independently of this warp's load-use latency.
    // (Skipped when the next row belongs to the next matrix of a group.)
    if (lane == 0 && cpr > 0 && r + kWarps < r1 && r + kWarps < p.row_end[m]) {
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                       p.codes[m] + (i + kWarps) * ldc),
                   "r"((uint32_t)cpr * 16u)
                   : "memory");
      if (INT4 && p.ocpr)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                         p.w_out[m] + (i + kWarps) * p.ld_out[m]),
                     "r"((uint32_t)p.ocpr * 16u)
                     : "memory");
    }

    float2 acc[B][2];
#pragma unroll
    for (int b = 0; b < B; ++b) acc[b][0] = acc[b][1] = make_float2(0.f, 0.f);

    int j = 0;
    uint32_t cbase = 0;
    const uint4 *rp = row;
#pragma unroll 1
    for (; j + kUnroll <= Jfull; j += kUnroll, cbase += kUnroll * kChunkStep, rp += 32 * kUnroll) {
      uint4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) v[u] = ld_stream(rp + 32 * u);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if constexpr (INT4) int4_chunk<B>(v[u], xs, goff, cbase + u * kChunkStep, bstride, acc);
        else int8_chunk<B>(v[u], xs, goff, cbase + u * kChunkStep, bstride, acc);
      }
    }
    if (j < Jw) {  // tail: at most kUnroll rounds, the last one possibly partial
      uint4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        v[u] = (j + u < Jw && lane + 32 * (j + u) < cpr) ? ld_stream(rp + 32 * u)
                                                         : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if (j + u < Jw) {  // warp-uniform
          const uint32_t cb = lane + 32 * (j + u) < cpr ? cbase + u * kChunkStep : 0u;
          if constexpr (INT4) int4_chunk<B>(v[u], xs, goff, cb, bstride, acc);
          else int8_chunk<B>(v[u], xs, goff, cb, bstride, acc);
        }
      }
    }

    float outl[B];
#pragma unroll
    for (int b = 0; b < B; ++b) outl[b] = 0.0f;
    if constexpr (INT4) {
      const uint4 *orow = reinterpret_cast<const uint4 *>(p.w_out[m] + i * p.ld_out[m]);
#pragma unroll 1
      for (int c = lane; c < p.ocpr; c += 32) {
        const uint4 v = ld_stream(orow + c);
        const float2 h0 = __half22float2(*reinterpret_cast<const __half2 *>(&v.x));
        const float2 h1 = __half22float2(*reinterpret_cast<const __half2 *>(&v.y));
        const float2 h2 = __half22float2(*reinterpret_cast<const __half2 *>(&v.z));
        const float2 h3 = __half22float2(*reinterpret_cast<const __half2 *>(&v.w));
#pragma unroll
        for (int b = 0; b < B; ++b) {
          const float4 xa = xo[b * ostride + gidx<2>(c, 0)];
          const float4 xc = xo[b * ostride + gidx<2>(c, 1)];
          float a = outl[b];
          a = fmaf(h0.x, xa.x, a); a = fmaf(h0.y, xa.y, a);
          a = fmaf(h1.x, xa.z, a); a = fmaf(h1.y, xa.w, a);
          a = fmaf(h2.x, xc.x, a); a = fmaf(h2.y, xc.y, a);
          a = fmaf(h3.x, xc.z, a); a = fmaf(h3.y, xc.w, a);
          outl[b] = a;
        }
      }
    }

#pragma unroll
    for (int b = 0; b < B; ++b) {
      float bgs = (acc[b][0].x + acc[b][0].y) + (acc[b][1].x + acc[b][1].y);
      bgs = warp_sum(bgs);
      float os = INT4 ? warp_sum(outl[b]) : 0.0f;
      if (lane == 0) p.y[m][b * p.ldy + i] = __float2half_rn(fmaf(s, bgs, os));
    }
  }
}

template <bool INT4, int B>
qz_status launch_t(const GemvParams &p, cudaStream_t s) {
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
  while (per_sm > 1 && (int64_t)di.sms * per_sm * kWarps > p.total_rows * 2) --per_sm;
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
  const size_t gpc = int4 ? 8 : 4;
  const size_t cps = p.cpr > 32 ? (size_t)p.cpr : 32;
  const size_t per_b = (cps * gpc + (int4 ? (size_t)p.ocpr * 2 : 0)) * 16;
  return per_b * (size_t)B;
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
