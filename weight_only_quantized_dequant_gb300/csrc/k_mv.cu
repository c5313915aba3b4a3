// Dequant-GEMV for small batches (2..8) with the multiply-adds on warp-level
// MMA.
//
// What is computed (per output row i and batch row b), as in k_gemv.cu:
//   INT8  ("Open Origin - ELG Stream Layer", INT8 Quantization & Direct
//          Mapping; FP16 On-The-Fly GPU Reconstruction):
//          y = scale * sum_j q_ij x_j
//   INT4  ("On-The-Fly Weight Synthesizer (OTF-LLM Engine)", Architecture &
//          Key Innovations diagram and items 1 and 3):
//          y = sum_{t<n_out} w_out_it x_perm[t] + s_i * sum_t' q_it' x_perm[n_out+t']
// Codes become exact fp16 integers in registers (no fp16 weight array is ever
// formed); every product of an exact code with an fp16 input is exact and
// products are summed in fp32 (MMA accumulators).
//
// Why MMA: the product is HBM-bound at ~0.5 byte per INT4 weight, so a GB300
// SM must retire ~42 weights per clock.  On the CUDA cores each weight costs
// one fp32 FMA per input row, which runs out of issue slots from two rows on.
// One mma.sync.m16n8k16 (16 rows x 16 inputs x 8 input rows) takes 256
// weights times up to 8 input rows off the issue path; what is left per
// weight is the conversion (one LOP3 and one packed fp16 subtract per two
// INT4 codes) and a share of one shared-memory read, whatever the batch.
//
// Layout of the work:
//  * The weights are the MMA's A operand (16 rows of a tile); the inputs are
//    its B operand, one batch row per column (columns >= B repeat the last
//    row and are discarded).  The order in which a dot product visits its
//    inputs is free, so each thread's registers are used in the order the
//    bit tricks produce them, and the input is staged in shared memory in
//    that same order (the permutation gather lands there directly).
//  * One producer warp streams the weights through a ring of shared-memory
//    stages (16 rows x a run of 64-byte K blocks, one bulk copy per row
//    piece, completing on an mbarrier).  Whole rows, or long pieces of rows,
//    per copy keep HBM efficient; the copies carry an L2 evict-first hint so
//    that the small, reused tensors (permutations, inputs, outputs) stay in
//    L2 while the weights stream past.
//  * A stage holds TP 16-row tiles (1 or 2); the eight consumer warps split
//    into TP groups, each splitting the K blocks of its tile; a tile's parts
//    are added in shared memory by the last warp of its group to finish it,
//    in warp order (the result does not depend on timing), or stored
//    directly when one warp owns the tile.
//  * Batches 9..16 were tried with two 8-column blocks per converted weight
//    fragment (inputs of 16 rows staged in shared memory): slower than the
//    tensor-core GEMM on 30 of the 32 launches of the 3B/7B/70B/Gemma layers
//    (7B o at batch 16: 31.9 against 15.4 us), so batches above 8 stay there.
//  * INT4 inputs are first copied contiguously into shared memory (into ring
//    slots that the producer fills only after the input is staged) and then
//    gathered there through the permutation, which is read with coalesced
//    loads before the wait for the previous kernel.
#include <cstring>

#include "qz_internal.cuh"

namespace qz {
namespace {

constexpr int kKB = 64;                     // bytes per row of one K block
constexpr int kConsumers = 8;               // consumer warps
constexpr int kProducers = 2;               // producer warps (issue alternate stages)
constexpr int kMaxThreads = (kConsumers + kProducers) * 32;
constexpr int kPermWords = 6;               // gather words whose perm a thread loads early
constexpr unsigned long long kMvWaitNs = 2000000000ull;
constexpr uint32_t kSleepHintNs = 100000;   // one suspended try_wait: at most 0.1 ms
constexpr int kEarlyStages = 2;             // ring stages issued before the first input is staged
constexpr uint32_t kNoInput = 0xFFFFu;      // permutation entry that reads a zero
constexpr int kOutPerThread = 3;            // outlier entries per consumer thread (n_out <= 768)

__device__ int g_mv_error = 0;  // 1 if a bounded wait gave up (read by qz_device_error)

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

// try_wait with a suspend-time hint: a thread whose phase is not complete
// sleeps until it completes (or the hint runs out) instead of spinning, so
// waiting warps leave the issue slots to the warps that compute.
__device__ __forceinline__ bool mbar_try_sleep(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSleepHintNs)
      : "memory");
  return ok != 0;
}

// Bounded wait; on timeout the error word is set and false returned.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_sleep(bar, parity)) return true;
  const unsigned long long t0 = gtimer();
  for (;;) {
    if (mbar_try_sleep(bar, parity)) return true;
    if (gtimer() - t0 > kMvWaitNs) {
      atomicExch(&g_mv_error, 1);
      return false;
    }
  }
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}

// (a & b) ^ c in one LOP3 (truth table 0x6A).
__device__ __forceinline__ uint32_t and_xor(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// D += A * B, m16n8k16, fp16 operands, fp32 accumulators.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Row boundaries of the grouped matrices (32-bit rows: the host limits a
// launch to < 2^31 rows).
__device__ __forceinline__ void locate(const GemvParams &p, int r, int &m, int &i) {
  m = 0;
#pragma unroll
  for (int t = 0; t < QZ_MAX_GROUP - 1; ++t) m += (t < p.n_mats - 1 && r >= (int)p.row_end[t]) ? 1 : 0;
  int lo = 0;
#pragma unroll
  for (int t = 0; t < QZ_MAX_GROUP - 1; ++t) lo = (t < m) ? (int)p.row_end[t] : lo;
  i = r - lo;
}

// One INT4 K block (64 bytes = 128 codes of each of the tile's rows g and
// g + 8; this thread's 16-byte chunk cg / cg8) against the staged input.
// In a word of 8 nibbles (elements e0..e7 at bits 4e..4e+3):
//   (w & 0x000F000F) ^ 0x64086408 = fp16 pair (1024 + q0 + 8, 1024 + q4 + 8)
//   (w & 0x00F000F0) ^ 0x64806480 = (1152 + 16 q1, 1152 + 16 q5)
// and the same on w >> 8 for e2,e6 and e3,e7; subtracting 1032 resp. 1152
// leaves q resp. 16 q exactly.  Pairs (e0,e4),(e2,e6) feed the "even" MMA,
// the 16x pairs (e1,e5),(e3,e7) the "odd" one; the staged 16-byte input word
// holds x in the order e0,e4,e2,e6,e1,e5,e3,e7.
__device__ __forceinline__ void int4_block(const uint4 &cg, const uint4 &cg8, uint32_t xa,
                                           float (&de0)[4], float (&dd0)[4], float (&de1)[4],
                                           float (&dd1)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    // words 0, 2 and 1, 3 accumulate in separate chains (MMA latency)
    float(&de)[4] = (j & 1) ? de1 : de0;
    float(&dd)[4] = (j & 1) ? dd1 : dd0;
    const uint32_t w = j == 0 ? cg.x : j == 1 ? cg.y : j == 2 ? cg.z : cg.w;
    const uint32_t v = j == 0 ? cg8.x : j == 1 ? cg8.y : j == 2 ? cg8.z : cg8.w;
    const uint4 xv = lds128(xa + j * 64);
    const uint32_t w8 = w >> 8, v8 = v >> 8;
    const uint32_t p0 = hsub2_bits(and_xor(w, 0x000F000Fu, 0x64086408u), 0x64086408u);
    const uint32_t q0 = hsub2_bits(and_xor(v, 0x000F000Fu, 0x64086408u), 0x64086408u);
    const uint32_t p2 = hsub2_bits(and_xor(w8, 0x000F000Fu, 0x64086408u), 0x64086408u);
    const uint32_t q2 = hsub2_bits(and_xor(v8, 0x000F000Fu, 0x64086408u), 0x64086408u);
    mma16816(de, p0, q0, p2, q2, xv.x, xv.y);
    const uint32_t p1 = hsub2_bits(and_xor(w, 0x00F000F0u, 0x64806480u), 0x64806480u);
    const uint32_t q1 = hsub2_bits(and_xor(v, 0x00F000F0u, 0x64806480u), 0x64806480u);
    const uint32_t p3 = hsub2_bits(and_xor(w8, 0x00F000F0u, 0x64806480u), 0x64806480u);
    const uint32_t q3 = hsub2_bits(and_xor(v8, 0x00F000F0u, 0x64806480u), 0x64806480u);
    mma16816(dd, p1, q1, p3, q3, xv.z, xv.w);
  }
}

// One INT8 K block (64 codes of rows g and g + 8; this thread's 16 codes of
// each).  XOR 0x80 makes each byte the offset-binary u = q + 128; PRMT puts
// two of them under the 0x6400 exponent (fp16 1024 + u) and subtracting 1152
// leaves q exactly.  Codes (0,1) of a word are k, k+1 of the MMA, (2,3) are
// k+8, k+9; the staged input word holds x in natural order.
__device__ __forceinline__ void int8_block(const uint4 &cg, const uint4 &cg8, uint32_t xa,
                                           float (&d0)[4], float (&d1)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float(&d)[4] = (j & 1) ? d1 : d0;  // two accumulator chains (MMA latency)
    const uint32_t w = (j == 0 ? cg.x : j == 1 ? cg.y : j == 2 ? cg.z : cg.w) ^ 0x80808080u;
    const uint32_t v = (j == 0 ? cg8.x : j == 1 ? cg8.y : j == 2 ? cg8.z : cg8.w) ^ 0x80808080u;
    const uint2 xv = lds64(xa + j * 32);
    const uint32_t a0 = hsub2_bits(__byte_perm(w, 0x64646464u, 0x4140), 0x64806480u);
    const uint32_t a1 = hsub2_bits(__byte_perm(v, 0x64646464u, 0x4140), 0x64806480u);
    const uint32_t a2 = hsub2_bits(__byte_perm(w, 0x64646464u, 0x4342), 0x64806480u);
    const uint32_t a3 = hsub2_bits(__byte_perm(v, 0x64646464u, 0x4342), 0x64806480u);
    mma16816(d, a0, a1, a2, a3, xv.x, xv.y);
  }
}

// ---- stage one product's input (fp16) in shared memory ------------------
// INT4 codes: input t' = 8 wd + e goes to K block wd / 16, word wd % 4,
// chunk (wd / 4) % 4, slot pos(e) of e0,e4,e2,e6,e1,e5,e3,e7; outlier input t
// to byte 2t of its row.  INT8: input t = 4 wd + e to K block wd / 16, word
// wd % 4, chunk (wd / 4) % 4, slot e.  Inputs are read through L2 (they may
// have been written by another CTA of this launch).
__device__ __forceinline__ uint32_t int4_word_off(int wd) {
  return (uint32_t)(wd >> 4) * 256u + (uint32_t)(wd & 3) * 64u + (uint32_t)((wd >> 2) & 3) * 16u;
}
__device__ __forceinline__ uint32_t int8_word_off(int wd) {
  return (uint32_t)(wd >> 4) * 128u + (uint32_t)(wd & 3) * 32u + (uint32_t)((wd >> 2) & 3) * 8u;
}

// The permutation of product p, read with coalesced 16-byte loads into
// shared memory as 16-bit entries (K <= 57344 < 2^16): background entries
// perm[n_out + t'] at pb[t'] (the staged-input region, still free), padded
// with kNoInput up to the staged width; outlier entries perm[t] at po16[t]
// (the staged outlier region).  Then every thread takes the entries of its
// gather words with one 16-byte shared read per word, and its outlier
// entries.  Ends at a consumer barrier; the caller must pass another before
// anything is written over pb/po16.
__device__ __forceinline__ void load_perm(uint8_t *smem, const MvLaunch &L, const GemvParams &p,
                                          const MvProduct &pr, int tid, int T,
                                          uint32_t (&pp)[kPermWords][4], int (&po)[kOutPerThread]) {
  uint16_t *pb = reinterpret_cast<uint16_t *>(smem);
  uint16_t *po16 = reinterpret_cast<uint16_t *>(smem + L.xo_off);
  const int K = p.K, n_out = p.n_out, nwb = pr.Kb * 16;
  auto place = [&](int e, int v) {
    if (e < n_out) po16[e] = (uint16_t)v;
    else pb[e - n_out] = (uint16_t)v;
  };
  const int nv = K / 4;
#pragma unroll 4
  for (int c = tid; c < nv; c += T) {
    const int4 v = __ldg(reinterpret_cast<const int4 *>(p.perm) + c);
    place(4 * c, v.x);
    place(4 * c + 1, v.y);
    place(4 * c + 2, v.z);
    place(4 * c + 3, v.w);
  }
  for (int e = 4 * nv + tid; e < K; e += T) place(e, __ldg(p.perm + e));
  for (int t = p.kb + tid; t < nwb * 8; t += T) pb[t] = kNoInput;
  asm volatile("bar.sync 1, %0;" ::"r"(T) : "memory");
#pragma unroll
  for (int i = 0; i < kPermWords; ++i) {
    const int wd = tid + i * T;
    uint4 q = make_uint4(kNoInput | (kNoInput << 16), kNoInput | (kNoInput << 16),
                         kNoInput | (kNoInput << 16), kNoInput | (kNoInput << 16));
    if (wd < nwb) q = *reinterpret_cast<const uint4 *>(pb + 8 * wd);
    pp[i][0] = q.x;
    pp[i][1] = q.y;
    pp[i][2] = q.z;
    pp[i][3] = q.w;
  }
#pragma unroll
  for (int i = 0; i < kOutPerThread; ++i) {
    const int t = tid + i * T;
    po[i] = t < n_out ? (int)po16[t] : -1;
  }
}

__device__ __forceinline__ uint4 pack_word(const uint32_t (&h)[8]) {
  // slots e0,e4,e2,e6,e1,e5,e3,e7 of the word
  return make_uint4(h[0] | (h[4] << 16), h[2] | (h[6] << 16), h[1] | (h[5] << 16),
                    h[3] | (h[7] << 16));
}

// ---- stage one product's input (fp16) in shared memory ------------------
template <bool INT4>
__device__ __forceinline__ void stage_input(uint8_t *smem, const MvLaunch &L, const GemvParams &p,
                                            const MvProduct &pr, int tid, int T,
                                            const uint32_t (&pp)[kPermWords][4],
                                            const int (&po)[kOutPerThread]) {
  const int B = L.B;
  const int nwb = pr.Kb * 16;
  if constexpr (INT4) {
    uint16_t *pb = reinterpret_cast<uint16_t *>(smem);
    const bool raw = pr.raw;
    uint8_t *rawp = smem + L.raw_off;
    if (raw) {
      // the input rows, contiguous, into shared memory (16-byte loads when
      // the rows allow)
      const int K = p.K;
      const bool vec = ((uintptr_t)p.x % 16u == 0) && (B == 1 || p.ldx % 8 == 0);
      for (int b = 0; b < B; ++b) {
        const __half *xb = p.x + b * p.ldx;
        uint16_t *rb = reinterpret_cast<uint16_t *>(rawp + (size_t)b * pr.rawstride);
        const int nv = vec ? K / 8 : 0;
#pragma unroll 4
        for (int c = tid; c < nv; c += T)
          reinterpret_cast<uint4 *>(rb)[c] = __ldcg(reinterpret_cast<const uint4 *>(xb) + c);
        for (int e = nv * 8 + tid; e < K; e += T) rb[e] = __half_as_ushort(__ldcg(xb + e));
      }
    }
    // (raw: the copy is complete; both: every thread holds its entries, so
    // the entry tables may be written over)
    asm volatile("bar.sync 1, %0;" ::"r"(T) : "memory");
    auto fetch = [&](int b, uint32_t idx) -> uint32_t {
      if (idx == kNoInput) return 0u;
      if (raw) return reinterpret_cast<const uint16_t *>(rawp + (size_t)b * pr.rawstride)[idx];
      return __half_as_ushort(__ldcg(p.x + b * p.ldx + idx));
    };
    for (int b = 0; b < B; ++b) {
      uint8_t *xsb = smem + (size_t)b * pr.bstride;
      uint4 v[kPermWords];
#pragma unroll
      for (int i = 0; i < kPermWords; ++i) {
        uint32_t h[8];
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {
          h[2 * e2] = fetch(b, pp[i][e2] & 0xFFFFu);
          h[2 * e2 + 1] = fetch(b, pp[i][e2] >> 16);
        }
        v[i] = pack_word(h);
      }
#pragma unroll
      for (int i = 0; i < kPermWords; ++i) {
        const int wd = tid + i * T;
        if (wd < nwb) *reinterpret_cast<uint4 *>(xsb + int4_word_off(wd)) = v[i];
      }
    }
    // words beyond the ones whose entries are in registers (K above ~20k
    // inputs): one pass of T words (16 whole K blocks) at a time, entries
    // read from pb before any word of the pass is written over them
    for (int base = kPermWords * T; base < nwb; base += T) {
      const int wd = base + tid;
      uint4 q = make_uint4(0, 0, 0, 0);
      if (wd < nwb) q = *reinterpret_cast<const uint4 *>(pb + 8 * wd);
      asm volatile("bar.sync 1, %0;" ::"r"(T) : "memory");
      if (wd < nwb) {
        const uint32_t e2s[4] = {q.x, q.y, q.z, q.w};
        for (int b = 0; b < B; ++b) {
          uint32_t h[8];
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            h[2 * e2] = fetch(b, e2s[e2] & 0xFFFFu);
            h[2 * e2 + 1] = fetch(b, e2s[e2] >> 16);
          }
          *reinterpret_cast<uint4 *>(smem + (size_t)b * pr.bstride + int4_word_off(wd)) = pack_word(h);
        }
      }
    }
    // outliers: input t < Ko * 32 at byte 2t of each batch row
    for (int b = 0; b < B; ++b) {
      uint16_t *xo = reinterpret_cast<uint16_t *>(smem + L.xo_off + (size_t)b * pr.ostride);
#pragma unroll
      for (int i = 0; i < kOutPerThread; ++i) {
        const int t = tid + i * T;
        if (t < pr.Ko * 32) xo[t] = po[i] >= 0 ? (uint16_t)fetch(b, (uint32_t)po[i]) : (uint16_t)0;
      }
    }
  } else {
    constexpr int kW8 = 8;  // words (4 inputs each) per thread loaded at once
    for (int b = 0; b < B; ++b) {
      const __half *xb = p.x + b * p.ldx;
      uint8_t *xsb = smem + (size_t)b * pr.bstride;
#pragma unroll 1
      for (int w0 = tid; w0 < nwb; w0 += kW8 * T) {
        uint2 v[kW8];
#pragma unroll
        for (int i = 0; i < kW8; ++i) {
          uint32_t h[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int t = 4 * (w0 + i * T) + e;
            h[e] = t < p.K ? __half_as_ushort(__ldcg(xb + t)) : 0u;
          }
          v[i] = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
        }
#pragma unroll
        for (int i = 0; i < kW8; ++i) {
          const int wd = w0 + i * T;
          if (wd < nwb) *reinterpret_cast<uint2 *>(xsb + int8_word_off(wd)) = v[i];
        }
      }
    }
  }
}

// TP: 16-row tiles per ring stage; the W consumer warps split into TP
// groups of WT = W / TP, group q owning tile q of every stage, its warps
// taking alternate K blocks of it.  A CTA's rows are cut into super-tiles of
// at most 16 TP rows (evenly), each super-tile into TP tiles (evenly).
template <bool INT4, int TP>
__global__ void __launch_bounds__(kMaxThreads, 1) mv_kernel(const __grid_constant__ MvLaunch L) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int W = kConsumers;                     // consumer warps; warps W.. produce
  constexpr int WT = W / TP;                        // warps per tile
  static_assert(W % TP == 0, "tiles per stage must divide the consumer warps");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;
  const int B = L.B;
  const int G = (int)gridDim.x;  // CTAs: each owns rows [total*b/G, total*(b+1)/G)
  const int NS = L.ns;
  const uint32_t slot_bytes = L.slot_bytes;
  const uint32_t ring = smem_u32(smem + L.ring_off);
  const uint32_t full = smem_u32(smem + L.bar_off);      // NS barriers: stage landed
  const uint32_t empty = full + 8u * NS;                  // NS barriers: stage released
  const uint32_t xready = empty + 8u * NS;                // the first input is staged
  const int nslot = NS + 1;                               // tile-partial slots
  float *part = reinterpret_cast<float *>(smem + L.part_off);
  int *cnt = reinterpret_cast<int *>(smem + L.cnt_off);

  if (threadIdx.x == 0) {
    for (int st = 0; st < NS; ++st) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(full + 8 * st) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(empty + 8 * st), "r"(W) : "memory");
    }
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(xready) : "memory");
    for (int i = 0; i < nslot * TP; ++i) cnt[i] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp >= W) {
    // ---- producers: the stages of every product, one after another; stage
    // S is issued by producer warp S % kProducers (one warp's bulk-copy
    // issue does not keep up with short row pieces).  Lanes 0..15 copy the
    // outlier piece of row `lane` of each tile of the stage, lanes 16..31
    // the code piece of row lane - 16.  Weights only: they never wait for
    // the previous kernel or for earlier products.
    const int pw = warp - W;
    bool xr = false;  // the first input has been staged
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    bool ok = true;
    int S = 0, slot = 0, round = 0;  // stage count, ring slot, times the ring went round
    {
      const GemvParams &p = L.t;
      const MvProduct &pr = L.pr;
      const int64_t r0 = p.total_rows * blockIdx.x / G;
      const int rows = (int)(p.total_rows * (blockIdx.x + 1) / G - r0);
      const int Tc = (rows + 16 * TP - 1) / (16 * TP);
      const int Ko = pr.Ko, Kc = pr.Ko + pr.Kb;
      const uint32_t P = pr.pitch;
      int te = 0;
      for (int t = 0; t < Tc && ok; ++t) {
        const int ts = te;
        te = rows * (t + 1) / Tc;
        const int live = te - ts;  // rows of the super-tile
        const int row = lane & 15;
        int m[TP], i[TP];
        bool lv[TP];
#pragma unroll
        for (int q = 0; q < TP; ++q) {  // this lane's row of tile q
          const int q0 = live * q / TP, nq = live * (q + 1) / TP - q0;
          lv[q] = row < nq;
          m[q] = i[q] = 0;
          if (lv[q]) locate(p, (int)r0 + ts + q0 + row, m[q], i[q]);
        }
        for (int j = 0; j < pr.nst; ++j) {
          if (S % kProducers != pw) {  // another producer's stage
            ++S;
            if (++slot == NS) {
              slot = 0;
              ++round;
            }
            continue;
          }
          if (round > 0) {
            ok = mbar_wait(empty + 8u * slot, (uint32_t)(round - 1) & 1u);
            if (!ok) break;
          }
          // The first stages go out at once; the rest only after the first
          // input has been staged, so that the input's loads, which every
          // consumer waits for, do not queue behind a whole ring of weights.
          if (S >= L.early && !xr) {
            ok = mbar_wait(xready, 0u);
            if (!ok) break;
            xr = true;
          }
          const int ka = j * pr.skc, kz = ka + pr.skc < Kc ? ka + pr.skc : Kc;
          // outlier K blocks [ka, min(kz, Ko)), code K blocks [max(ka, Ko), kz)
          const int oa = ka, oz = kz < Ko ? kz : Ko;
          const int ca = ka > Ko ? ka : Ko, cz = kz;
          int ob = oz > oa ? (oz - oa) * kKB : 0;
          if (ob > p.ocpr * 16 - oa * kKB) ob = p.ocpr * 16 - oa * kKB;
          int cb = cz > ca ? (cz - ca) * kKB : 0;
          if (cb > p.cpr * 16 - (ca - Ko) * kKB) cb = p.cpr * 16 - (ca - Ko) * kKB;
          if (ob < 0) ob = 0;
          if (cb < 0) cb = 0;
          const uint32_t fb = full + 8u * slot;
          if (lane == 0)
            asm volatile(
                "{\n\t.reg .b64 st;\n\t"
                "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(fb),
                "r"((uint32_t)((ob + cb) * live))
                : "memory");
          const bool is_code = lane >= 16;
          const int nb = is_code ? cb : ob;
          if (nb > 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
#pragma unroll
          for (int q = 0; q < TP; ++q) {
            if (lv[q] && nb > 0) {
              const uint8_t *src =
                  is_code ? p.codes[m[q]] + (int64_t)i[q] * p.ld_codes[m[q]] + (ca - Ko) * kKB
                          : reinterpret_cast<const uint8_t *>(p.w_out[m[q]] +
                                                              (int64_t)i[q] * p.ld_out[m[q]]) +
                                oa * kKB;
              const uint32_t dst = ring + (uint32_t)slot * slot_bytes +
                                   (uint32_t)(16 * q + row) * P +
                                   (uint32_t)((is_code ? ca : oa) - ka) * kKB;
              asm volatile(
                  "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                  " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
                  "l"(src), "r"((uint32_t)nb), "r"(fb), "l"(policy)
                  : "memory");
            }
          }
          ++S;
          if (++slot == NS) {
            slot = 0;
            ++round;
          }
        }
      }
    }
    // Before the CTA's shared memory can go, every copy issued must have
    // landed: wait (bounded) for the last stage issued to each slot.
    if (lane == 0) {
      const unsigned long long t0 = gtimer();
      for (int i = S - NS > 0 ? S - NS : 0; i < S; ++i)
        while (!mbar_try(full + 8u * (i % NS), (uint32_t)(i / NS) & 1u))
          if (gtimer() - t0 > kMvWaitNs) break;
    }
    return;
  }

  // ---- consumers -------------------------------------------------------
  constexpr int T = W * 32;
  const int tid = threadIdx.x;
  const int bsel = g < B ? g : B - 1;               // this thread's B-operand column
  uint32_t pp[kPermWords][4];
  int po[kOutPerThread];
  float de[4], dd[4], de1[4], dd1[4], dout[4];
  int mrow[2] = {0, 0}, irow[2] = {0, 0};
  bool live[2] = {false, false};
  float srow[2] = {0.f, 0.f};
  bool ok = true;
  int slot = 0, ps = 0;  // ring slot, tile-partial slot
  uint32_t phase = 0;
  {
    const GemvParams &p = L.t;
    const MvProduct &pr = L.pr;
    // permutation entries first: static, so read before the wait
    if constexpr (INT4) load_perm(smem, L, p, pr, tid, T, pp, po);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    stage_input<INT4>(smem, L, p, pr, tid, T, pp, po);
    asm volatile("bar.sync 1, %0;" ::"r"(T) : "memory");  // consumer warps only
    if (tid == 0)
      asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(xready)
                   : "memory");

    const uint32_t xrow = smem_u32(smem) + (uint32_t)bsel * pr.bstride;
    const uint32_t orow = smem_u32(smem + L.xo_off) + (uint32_t)bsel * pr.ostride;
    const int64_t r0 = p.total_rows * blockIdx.x / G;
    const int rows = (int)(p.total_rows * (blockIdx.x + 1) / G - r0);
    const int Tc = (rows + 16 * TP - 1) / (16 * TP);
    const int Ko = pr.Ko, Kc = pr.Ko + pr.Kb;
    const int NST = pr.nst, SKc = pr.skc;
    const uint32_t P = pr.pitch;
    const int q = warp / WT, phi = warp % WT;  // this warp's tile of a stage, its K phase
    int ts = 0, te = 0;
    for (int t = 0; t < Tc && ok; ++t) {
      ts = te;
      te = rows * (t + 1) / Tc;
      const int q0 = ts + (te - ts) * q / TP;            // first row of tile q
      const int nq = ts + (te - ts) * (q + 1) / TP - q0;  // its rows (0..16)
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // the tile's rows, scales, fresh accumulators
        const int rr = g + 8 * h;
        live[h] = rr < nq;
        locate(p, (int)r0 + q0 + (live[h] ? rr : (nq > 0 ? nq - 1 : 0)), mrow[h], irow[h]);
        srow[h] = INT4 ? __ldg(p.scale[mrow[h]] + irow[h]) : __ldg(p.scale[mrow[h]]);
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) de[c] = dd[c] = de1[c] = dd1[c] = dout[c] = 0.f;
      for (int j = 0; j < NST; ++j) {
        ok = mbar_wait(full + 8u * slot, phase);
        if (!ok) break;
        const int ka = j * SKc, kz = ka + SKc < Kc ? ka + SKc : Kc;
        const uint32_t sb = ring + (uint32_t)slot * slot_bytes + (uint32_t)(16 * q + g) * P +
                            (uint32_t)tig * 16u;
        int kk = ka + phi;                            // this warp's K blocks: kk, kk + WT, ...
        if constexpr (INT4) {
#pragma unroll 1
          for (; kk < kz && kk < Ko; kk += WT) {      // outlier columns (fp16)
            const uint32_t a_off = (uint32_t)(kk - ka) * kKB;
            uint4 a = lds128(sb + a_off), a8 = lds128(sb + 8 * P + a_off);
            if (kk * 4 + tig >= p.ocpr) a = a8 = make_uint4(0, 0, 0, 0);  // past the row's outliers
            const uint4 xv = lds128(orow + (uint32_t)kk * kKB + tig * 16u);
            mma16816(dout, a.x, a8.x, a.y, a8.y, xv.x, xv.y);
            mma16816(dout, a.z, a8.z, a.w, a8.w, xv.z, xv.w);
          }
        }
        {
          uint32_t a_addr = sb + (uint32_t)(kk - ka) * kKB;
          uint32_t x_addr = INT4 ? xrow + (uint32_t)(kk - Ko) * 256u + tig * 16u
                                 : xrow + (uint32_t)kk * 128u + tig * 8u;
#pragma unroll 2
          for (; kk < kz; kk += WT) {
            const uint4 a = lds128(a_addr), a8 = lds128(a_addr + 8 * P);
            if constexpr (INT4)
              int4_block(a, a8, x_addr, de, dd, de1, dd1);
            else
              int8_block(a, a8, x_addr, de, de1);
            a_addr += (uint32_t)WT * kKB;
            x_addr += (uint32_t)WT * (INT4 ? 256u : 128u);
          }
        }
        __syncwarp();
        if (lane == 0)  // this warp is done with the stage
          asm volatile(
              "{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(
                  empty + 8u * slot)
              : "memory");
        if (++slot == NS) {
          slot = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if constexpr (WT == 1) {
        // ---- tile epilogue, one warp per tile: its outputs straight out
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int col = 2 * tig + c, ci = 2 * h + c;
            const float e = de[ci] + de1[ci], o = dd[ci] + dd1[ci];
            const float v = INT4 ? fmaf(srow[h], e + 0.0625f * o, dout[ci]) : srow[h] * e;
            if (col < B && live[h])
              p.y[mrow[h]][col * p.ldy[mrow[h]] + irow[h]] = __float2half_rn(v);
          }
      } else {
        // ---- tile epilogue: this warp's part of every output of the tile,
        // then the last of the tile's warps to arrive adds the parts in warp
        // order ---------------------------------------------------------
        float *pw = part + ((size_t)ps * W + warp) * 16 * B;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int col = 2 * tig + c, ci = 2 * h + c;
            const float e = de[ci] + de1[ci], o = dd[ci] + dd1[ci];
            const float v = INT4 ? fmaf(srow[h], e + 0.0625f * o, dout[ci]) : srow[h] * e;
            if (col < B) pw[(g + 8 * h) * B + col] = v;
          }
        __threadfence_block();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomicAdd(&cnt[ps * TP + q], 1) == WT - 1;
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          __threadfence_block();
          const int rr = lane & 15;
          if (rr < nq) {
            int m, i;
            locate(p, (int)r0 + q0 + rr, m, i);
            for (int col = lane >> 4; col < B; col += 2) {
              float acc = 0.f;
              for (int w = q * WT; w < q * WT + WT; ++w)
                acc += part[(((size_t)ps * W + w) * 16 + rr) * B + col];
              p.y[m][col * p.ldy[m] + i] = __float2half_rn(acc);
            }
          }
          __syncwarp();
          if (lane == 0) cnt[ps * TP + q] = 0;
        }
        if (++ps == nslot) ps = 0;
      }
    }
  }
}

}  // namespace

namespace {

constexpr int kMaxStages = 6;
// Row pieces per stage tried in turn (bytes): whole rows up to the first,
// then shorter pieces until the ring fits.
constexpr int kRowCaps[] = {4352, 3456, 2688, 2112, 1600, 1344, 1088, 832, 576, 320, 64};

// Shared-memory layout and shapes of a launch.  raw: copy INT4 inputs
// contiguously before the gather.  Returns the bytes of shared memory, or 0
// if no ring of min_ns stages fits.
size_t mv_layout(bool int4, const GemvParams &p, int B, int raw, int cap, int min_ns, int tp,
                 size_t avail, MvLaunch &L) {
  L.B = B;
  L.tp = tp;
  MvProduct &pr = L.pr;
  pr.Ko = int4 ? (p.ocpr + 3) / 4 : 0;
  pr.Kb = (p.cpr + 3) / 4;
  const int Kc = pr.Ko + pr.Kb;
  const int kmax = cap / kKB > 0 ? cap / kKB : 1;
  pr.nst = (Kc + kmax - 1) / kmax;
  pr.skc = (Kc + pr.nst - 1) / pr.nst;
  // stage rows 64 mod 128 bytes apart: rows g and g + 1 of one read phase
  // fall in different bank halves
  pr.pitch = (uint32_t)pr.skc * kKB;
  if (pr.pitch % 128u == 0) pr.pitch += 64u;
  // batch rows of the staged inputs: 64 (16-byte reads) resp. 32 (8-byte
  // reads) mod 128 bytes apart, so one read phase meets distinct banks
  pr.bstride = (uint32_t)pr.Kb * (int4 ? 256u : 128u) + (int4 ? 64u : 32u);
  pr.ostride = (uint32_t)pr.Ko * kKB;
  if (pr.ostride % 128u == 0) pr.ostride += 64u;
  pr.raw = int4 && raw;
  pr.rawstride = (uint32_t)((p.K * 2 + 15) / 16 * 16);
  const size_t xs = (size_t)B * pr.bstride, xo = int4 ? (size_t)B * pr.ostride : 0;
  const size_t rw = pr.raw ? (size_t)B * pr.rawstride : 0;
  const size_t slot = (size_t)16 * tp * pr.pitch;
  L.slot_bytes = (uint32_t)slot;
  // The contiguous input copy borrows the ring's last slots, which the
  // producer fills only after the input is staged.
  const int raw_slots = (int)((rw + slot - 1) / slot);
  size_t off = xs;
  L.xo_off = (uint32_t)off;
  off += xo;
  off = (off + 127) & ~(size_t)127;
  L.ring_off = (uint32_t)off;
  for (int ns = kMaxStages; ns >= min_ns; --ns) {
    if (ns <= raw_slots) break;  // at least one slot left for the early stages
    L.raw_off = (uint32_t)(off + (size_t)(ns - raw_slots) * slot);
    L.early = ns - raw_slots < kEarlyStages ? ns - raw_slots : kEarlyStages;
    size_t o = off + (size_t)ns * slot;
    const size_t bar = o;
    o += (size_t)ns * 16 + 16;
    const size_t prt = o;  // tile parts, when several warps share a tile
    if (kConsumers / tp > 1) o += (size_t)(ns + 1) * kConsumers * 16 * B * sizeof(float);
    const size_t cn = o;
    o += (size_t)(ns + 1) * tp * sizeof(int);
    o = (o + 15) & ~(size_t)15;
    if (o <= avail) {
      L.ns = ns;
      L.bar_off = (uint32_t)bar;
      L.part_off = (uint32_t)prt;
      L.cnt_off = (uint32_t)cn;
      return o;
    }
  }
  return 0;
}

// Launch shapes, as measured on every grouped launch of the 3B/7B/70B INT4
// and Gemma INT8 layers at batches 2, 4 and 8:
//  * Two tiles per stage when a CTA holds at most kTwoTileRows rows and a
//    stage still holds whole rows (INT4) or at least half of every row
//    (INT8): there the per-tile setup and the sum of eight warps' parts cost
//    more than the ring stages of 32 rows do.  Otherwise one tile per stage
//    (the 70B launches, the long-row down projections); four or eight tiles
//    per stage lost everywhere (their stages leave too few bytes in flight).
//  * One tile per stage: whole rows in two or more stages when they fit,
//    else three or more stages of the longest pieces, then two.
//  * Inputs copied to shared memory before the gather whenever that fits.
constexpr int64_t kTwoTileRows = 200;
constexpr uint32_t kMinPiece = 576;  // bytes of a row per stage, unless whole rows

size_t mv_plan(bool int4, const GemvParams &p, int B, const DeviceInfo &di, MvLaunch &L) {
  const size_t avail = (size_t)di.max_smem_optin;
  const int64_t tiles = (p.total_rows + 15) / 16;
  const int64_t grid = tiles < di.sms ? tiles : di.sms;
  const int64_t R = (p.total_rows + grid - 1) / grid;  // rows of a CTA
  if (R <= kTwoTileRows)
    for (int raw = int4 ? 1 : 0; raw >= 0; --raw)
      for (int cap : kRowCaps) {
        const size_t smem = mv_layout(int4, p, B, raw, cap, 2, 2, avail, L);
        if (smem && L.pr.nst <= (int4 ? 1 : 2)) return smem;
      }
  const int row = (int4 ? (p.ocpr + 3) / 4 + (p.cpr + 3) / 4 : (p.cpr + 3) / 4) * kKB;
  for (int raw = int4 ? 1 : 0; raw >= 0; --raw) {
    const size_t smem = mv_layout(int4, p, B, raw, row, 2, 1, avail, L);
    if (smem) return smem;
  }
  for (int raw = int4 ? 1 : 0; raw >= 0; --raw)
    for (int min_ns = 3; min_ns >= 2; --min_ns)
      for (int cap : kRowCaps) {
        const size_t smem = mv_layout(int4, p, B, raw, cap, min_ns, 1, avail, L);
        // pieces shorter than kMinPiece stream poorly: leave those launches
        // to the tensor-core GEMM
        if (smem && (L.pr.nst == 1 || (uint32_t)L.pr.skc * kKB >= kMinPiece)) return smem;
      }
  return 0;
}

template <bool INT4>
qz_status launch_mv_t(const GemvParams &p, int B, cudaStream_t s) {
  DeviceInfo di;
  qz_status st = device_info(&di);
  if (st != QZ_OK) return st;
  MvLaunch L;
  memset(&L, 0, sizeof(L));
  L.t = p;
  const size_t smem = mv_plan(INT4, p, B, di, L);
  if (!smem) return QZ_ERR_UNSUPPORTED;
  auto kern = L.tp == 2 ? mv_kernel<INT4, 2> : mv_kernel<INT4, 1>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_status(e);
  const int64_t tiles = (p.total_rows + 15) / 16;
  const int64_t grid = tiles < di.sms ? tiles : di.sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)kMaxThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.overlap ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, L);
  if (e != cudaSuccess) return cuda_status(e);
  return launch_status();
}

}  // namespace

bool mv_fits(bool int4, int B, const GemvParams &p) {
  if (B < 1 || B > kMvMaxBatch) return false;
  DeviceInfo di;
  if (device_info(&di) != QZ_OK) return false;
  MvLaunch L;
  return mv_plan(int4, p, B, di, L) != 0;
}

qz_status launch_mv(bool int4, int B, const GemvParams &p, cudaStream_t s) {
  return int4 ? launch_mv_t<true>(p, B, s) : launch_mv_t<false>(p, B, s);
}

qz_status read_mv_error(int *code, int clear) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_mv_error, sizeof(int));
  if (e != cudaSuccess) return cuda_status(e);
  if (clear && v) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_mv_error, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_status(e);
  }
  *code = v;
  return QZ_OK;
}

}  // namespace qz
