// Tensor-core dequant-GEMM (tcgen05 + TMEM) for batches the CUDA-core GEMV
// does not cover: B > 4, or B in 2..4 when the staged inputs exceed shared
// memory.  Same math as the GEMV ("Open Origin - ELG Stream Layer", INT8
// Quantization & Direct Mapping; "On-The-Fly Weight Synthesizer (OTF-LLM
// Engine)", Architecture & Key Innovations: outlier product + background
// product), now a dense contraction Y[b][i] = sum_k A[i][k] * X[b][k]:
//
//  * A (weights) is the MMA's M side, in tiles of 128 output rows.  Producer
//    warps turn packed codes into exact fp16 integers in registers (INT4: one
//    LOP3 onto the 0x6400 exponent and one packed subtract or fused
//    multiply-add per nibble pair, no shifts for half of the pairs; INT8: one
//    PRMT per byte pair) and store them into tensor memory, where the MMA
//    reads A.  No fp16 weight tensor exists in HBM.
//  * B (activations, N = batch rounded up to 16) is gathered through the
//    permutation once per call into the canonical K-major layout, in the k
//    order the nibble conversion produces, and streamed into shared memory.
//  * tcgen05.mma (kind::f16, fp32 accumulate) into two TMEM accumulators:
//    outlier channels and INT4 background, so that the per-row scale
//    multiplies the background only: y = D_out + s_i * D_bg.  Issuing one
//    MMA costs its thread about 60 SM clocks whatever N is (measured: one
//    thread, 2048 weights per instruction), so two threads in two warps issue
//    alternate work units into accumulators of their own, and the epilogue
//    adds the two in issuer order.  Per-unit ring positions are counters,
//    not divisions: the issuing threads run serial code.
//  * Schedules of the (tile, K tile) work units of all matrices of the call,
//    chosen per call by a cost model: persistent stream-K (one contiguous
//    range per CTA, one CTA per SM, so every SM gets the same number of MMAs
//    whatever the tile count; a tile cut between CTAs is finished by the
//    last of its CTAs to arrive, which adds the fp32 partials in CTA order),
//    a cluster of S CTAs per tile that split its K tiles and add their
//    partials in rank order through distributed shared memory (few tiles),
//    or persistent whole tiles (no workspace).  All are deterministic.
//  * Up to batch 32 the accumulators are double-buffered, so the epilogue
//    warps drain one tile while the MMAs of the next run (above that tensor
//    memory holds one buffer per issuer beside four A stages).  Every wait is
//    bounded in time and reports a timeout through a device flag.
#include <cuda.h>

#include <cstring>
#include <atomic>
#include <mutex>

#include "qz_internal.cuh"

namespace qz {

// Device-side error word of the library (0 = none).  Written only when a
// bounded wait gives up; read and cleared by qz_device_error().
__device__ int g_device_error = 0;

namespace {

constexpr int kM = 128;         // weight rows per tile (MMA M)
constexpr int kKT = 128;        // K elements per work unit (one pipeline stage)
constexpr int kMaxAStages = 6;  // A stages in tensor memory (64 columns each)
constexpr uint32_t kTmemCols = 512;    // 2 x (outlier, background) accumulators, A above
constexpr int kProducers = 256;  // 8 warps: two groups of 4 (alternate units), one thread per row
constexpr int kGroupWarps = 4;   // converter warps that fill one A stage
constexpr int kEpiWarp = kProducers / 32;     // warps 8-11 drain the accumulators
constexpr int kMmaWarp = kEpiWarp + 4;        // warp 12 issues the MMAs of even units
constexpr int kCodeWarp = kMmaWarp + 1;       // warp 13 fills the code ring
constexpr int kLoadWarp = kMmaWarp + 2;       // warp 14 fills the activation ring
constexpr int kMma2Warp = kMmaWarp + 3;       // warp 15 issues the MMAs of odd units
constexpr int kMaxIssuers = 2;
constexpr int kThreadsTc = kProducers + 256;
constexpr int kEpiThreads = 128;
constexpr int kMaxBStages = 8;                // activation ring depth (smem permitting)
constexpr size_t kBRingBytes = 80 * 1024;     // shared memory given to that ring
constexpr int kMaxCtas = 160;   // persistent grid cap (partial slots in the workspace)
constexpr int kMinUnits = 4;    // work units per CTA at least (its fixed start-up cost)
constexpr uint32_t kLBO = 128;   // bytes between core matrices along K
constexpr uint32_t kSBO = 2048;  // bytes between 8-row groups (kKT/8 * 128)
constexpr unsigned long long kWaitNs = 2000000000ull;  // 2 s per wait
// Raw-code ring: K tiles of packed codes (kM rows x ROWB bytes, one 2D
// tensor copy each) in flight ahead of the fp16 A stages.
template <bool INT4>
struct RawRing {
  static constexpr int DEPTH = INT4 ? 8 : 4;        // K tiles in flight
  static constexpr int ROWB = INT4 ? kKT / 2 : kKT;  // packed bytes per row per K tile
  static constexpr int BYTES = DEPTH * kM * ROWB;
};
constexpr int kMaxRaw = 8;
constexpr int kBarBytes = 1024;  // mbarriers and flags at the start of shared memory
// Schedules of the (tile, K tile) work units over the CTAs.
constexpr int kWhole = 0;    // persistent, ranges of whole tiles (no workspace)
constexpr int kStreamK = 1;  // persistent, even ranges of units; cut tiles finished in L2
constexpr int kCluster = 2;  // a cluster of S CTAs per tile splits K; reduced in DSMEM

struct TcParams {
  CUtensorMap codes_map[QZ_MAX_GROUP];  // 2D: [rows][ld_codes bytes], box kM x ROWB
  GemvParams g;
  int B;                // batch rows
  int Np;               // MMA N: B rounded up to 16
  int nbs;              // stages of the activation ring
  int nsa;              // A stages in tensor memory
  int nmma;             // MMA-issuing threads (1 or 2), each with its own accumulators
  int nbuf;             // accumulator buffers (1 or 2) per issuer
  uint32_t a_base;      // first TMEM column of the A stages (nbuf * nmma * 2 Np)
  const uint8_t *ws;    // gathered activations, one canonical B tile per K tile (or null)
  float *part;          // partials of cut tiles: [kMaxCtas][2][4 quarters][Np/4][32][4] fp32
  unsigned *cnt;        // arrivals per cut tile and TMEM lane quarter, by its first CTA
  int ko;               // K tiles of the outlier block
  int kbt;              // K tiles of the background block
  int KT;               // K tiles per tile: ko + kbt
  int tiles;            // row tiles of all matrices
  int U;                // work units: tiles * KT
  int G;                // CTAs (persistent grid)
  int split;            // schedule: kWhole, kStreamK or kCluster
  int S;                // kCluster: CTAs per tile (cluster size), each 1/S of its K tiles
  int n_tiles[QZ_MAX_GROUP];
  int tile_end[QZ_MAX_GROUP];
  int64_t mat_rows[QZ_MAX_GROUP];
};


__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
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

// Wait for the phase of the given parity; false (and the error flag set) if
// it does not complete within kWaitNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int *abort_flag) {
  if (mbar_try(bar, parity)) return true;
  const unsigned long long t0 = gtimer();
  for (;;) {
    if (mbar_try(bar, parity)) return true;
    if (*(volatile int *)abort_flag) return false;
    if (gtimer() - t0 > kWaitNs) {
      atomicExch(&g_device_error, 1);
      *(volatile int *)abort_flag = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// 16 bytes from global memory through L2 only (not L1).
__device__ __forceinline__ float4 ld_cg_f4(const float4 *p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

// Canonical K-major, no-swizzle shared-memory matrix descriptor.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFF) >> 4);
  d |= (uint64_t)(kLBO >> 4) << 16;
  d |= (uint64_t)(kSBO >> 4) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version
  return d;                // base offset 0, relative LBO, no swizzle
}

// Instruction descriptor: kind::f16, A = B = f16, D = f32, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// The eight MMAs of one unit (K slots 0..127): D (TMEM) += A[:, 16k:16k+16] *
// B[16k:16k+16, :], A in TMEM at a0 + 8k (lane = row, 2 fp16 of K per column),
// B in shared memory with its descriptor's low word advanced by 16 per step
// (the address field, in 16-byte units, cannot carry: shared memory is below
// 256 KB); only the first may start the accumulator (acc0 == 0).  One asm
// block keeps the issuing thread's instructions per MMA to three.
__device__ __forceinline__ void mma8_f16_ta(uint32_t d, uint32_t a0, uint32_t blo, uint32_t bhi,
                                            uint32_t idesc, uint32_t acc0) {
  asm volatile(
      "{\n\t.reg .pred p0, p1;\n\t.reg .b64 b;\n\t.reg .b32 lo, a;\n\t"
      "setp.ne.b32 p0, %5, 0;\n\t"
      "setp.eq.b32 p1, %5, %5;\n\t"
      "mov.b64 b, {%2, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], b, %4, p0;\n\t"
      "add.u32 a, %1, 8;\n\tadd.u32 lo, %2, 16;\n\tmov.b64 b, {lo, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, p1;\n\t"
      "add.u32 a, %1, 16;\n\tadd.u32 lo, %2, 32;\n\tmov.b64 b, {lo, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, p1;\n\t"
      "add.u32 a, %1, 24;\n\tadd.u32 lo, %2, 48;\n\tmov.b64 b, {lo, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, p1;\n\t"
      "add.u32 a, %1, 32;\n\tadd.u32 lo, %2, 64;\n\tmov.b64 b, {lo, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, p1;\n\t"
      "add.u32 a, %1, 40;\n\tadd.u32 lo, %2, 80;\n\tmov.b64 b, {lo, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, p1;\n\t"
      "add.u32 a, %1, 48;\n\tadd.u32 lo, %2, 96;\n\tmov.b64 b, {lo, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, p1;\n\t"
      "add.u32 a, %1, 56;\n\tadd.u32 lo, %2, 112;\n\tmov.b64 b, {lo, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, p1;\n\t}" ::"r"(d),
      "r"(a0), "r"(blo), "r"(bhi), "r"(idesc), "r"(acc0));
}

// 32 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 16 consecutive fp32 TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Byte offset of (row r, k-slot c) in a canonical tile.
__device__ __forceinline__ uint32_t core_off(int r, int c) {
  return (uint32_t)((r >> 3) * kSBO + (c >> 3) * kLBO + (r & 7) * 16 + (c & 7) * 2);
}

// The nibble conversion below yields k slots in the order 0,4,1,5,2,6,3,7 of
// every group of 8 elements; the activations are staged in the same order.
__device__ __forceinline__ int slot_elem(int c) {
  const int s = c & 7;
  return (c & ~7) + ((s & 1) ? 4 + (s >> 1) : (s >> 1));
}

// Position in a ring of n slots that advances by one per work unit: the slot
// and the parity of its current round (slot = q mod n, parity = (q / n) & 1),
// kept without run-time divisions on the serial path of the issuing threads.
struct RingPos {
  int slot = 0;
  uint32_t parity = 0;
  __device__ __forceinline__ void next(int n) {
    if (++slot == n) {
      slot = 0;
      parity ^= 1u;
    }
  }
};

// (tile, K tile) of a work unit, advanced by one unit at a time.
struct UnitPos {
  int t, kt;
  __device__ __forceinline__ UnitPos(int u, int KT) : t(u / KT), kt(u - (u / KT) * KT) {}
  __device__ __forceinline__ void next(int KT) {
    if (++kt == KT) {
      kt = 0;
      ++t;
    }
  }
};

// Whether the issuer w (of W in {1, 2}) owns a unit among K tiles [a, b) of
// tile t: units alternate between issuers by their position in the CTA's range.
__device__ __forceinline__ bool issuer_has(int W, int w, int t, int a, int b, int KT, int u_begin) {
  if (b <= a) return false;
  if (W == 1 || b - a >= 2) return true;
  return ((t * KT + a - u_begin) & 1) == w;
}

// a * b + c on fp16 pairs (one rounding).
__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  __half2 r = __hfma2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b),
                      *reinterpret_cast<__half2 *>(&c));
  return *reinterpret_cast<uint32_t *>(&r);
}

__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
  return *reinterpret_cast<uint32_t *>(&r);
}

// Work-unit range [start(c), start(c+1)) of CTA c: an even cut of the U
// units (a tile may span CTAs), 1/S of one tile's K tiles, or whole tiles.
__device__ __forceinline__ int range_start(const TcParams &tp, int c) {
  if (tp.split == kStreamK) return (int)((int64_t)c * tp.U / tp.G);
  if (tp.split == kCluster) return (c / tp.S) * tp.KT + tp.KT * (c % tp.S) / tp.S;
  return (int)((int64_t)c * tp.tiles / tp.G) * tp.KT;
}

// The CTA whose range holds unit u (split schedule).
__device__ __forceinline__ int unit_owner(const TcParams &tp, int u) {
  return (int)((((int64_t)u + 1) * tp.G - 1) / tp.U);
}

struct TileInfo {
  int m;           // matrix of the group
  int64_t row0;    // first row of the tile in that matrix
  int64_t nrows;   // rows of that matrix
};

__device__ __forceinline__ TileInfo tile_info(const TcParams &tp, int t) {
  int m = 0;
#pragma unroll
  for (int i = 0; i < QZ_MAX_GROUP - 1; ++i) m += (i < tp.g.n_mats - 1 && t >= tp.tile_end[i]) ? 1 : 0;
  TileInfo r;
  r.m = m;
  r.row0 = (int64_t)(t - (m ? tp.tile_end[m - 1] : 0)) * kM;
  r.nrows = tp.mat_rows[m];
  return r;
}

// Slot of CTA q's partial of tile t: 0 if t is the first tile of its range.
__device__ __forceinline__ int part_slot(const TcParams &tp, int q, int t) {
  return t == range_start(tp, q) / tp.KT ? 0 : 1;
}

// Bounded wait that ignores the abort flag: used to let this CTA's own bulk
// copies land before it exits after an abort.
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = gtimer();
  while (!mbar_try(bar, parity))
    if (gtimer() - t0 > kWaitNs) return;
}

template <bool INT4>
__global__ void __launch_bounds__(kThreadsTc, 1) tc_gemm_kernel(const __grid_constant__ TcParams tp) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const GemvParams &p = tp.g;
  // 1024-byte aligned carve-up
  uint8_t *base = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int bBytes = tp.Np * kKT * 2;
  const int NB = tp.nbs, NA = tp.nsa, KT = tp.KT, Np = tp.Np;
  // [barriers | activation ring | raw-code ring | ...]; under the cluster
  // schedule, once a CTA's MMAs are done its rings hold its partial
  uint64_t *bars = reinterpret_cast<uint64_t *>(base);
  uint8_t *b_st = base + kBarBytes;                  // NB * bBytes
  uint8_t *raw = b_st + NB * bBytes;                 // RawRing<INT4>::BYTES
  uint64_t *full = bars, *empty = bars + kMaxAStages;
  uint64_t *bfull = bars + 2 * kMaxAStages, *bempty = bfull + kMaxBStages;
  uint64_t *rfull = bempty + kMaxBStages, *rempty = rfull + kMaxRaw;
  uint64_t *dfull = rempty + kMaxRaw, *dempty = dfull + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(dempty + 2);
  int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = (int)blockIdx.x;
  const int u_begin = range_start(tp, cta), u_end = range_start(tp, cta + 1);

  // Code loader state, carried from the prologue into its main loop: the
  // loader sets up its own ring barriers, only arrives at the start-up
  // barrier (named barrier 1) and issues the first ring of code copies while
  // the other warps set up the rest and warp 0 allocates tensor memory.
  // The ring is split between the two converter groups: group g owns slots
  // g, g + 2, ..., so that every slot has one consumer that takes its
  // copies in order (an mbarrier wait tells phases apart by parity only).
  constexpr int DR = RawRing<INT4>::DEPTH, RB = RawRing<INT4>::ROWB, DRG = DR / 2;
  static_assert(DR % 2 == 0, "the code ring splits evenly between the two groups");
  int cl_n0 = 0, cl_n1 = 0;  // copies issued per group
  int cl_u = u_begin, cl_t = 0, cl_kt = 0;
  auto issue_codes = [&](int slot, int t, int kt) {
    const uint32_t bar = smem_u32(&rfull[slot]);
    const TileInfo ti = tile_info(tp, t);
    const uint64_t cmap = reinterpret_cast<uint64_t>(&tp.codes_map[ti.m]);
    const int x = INT4 ? (kt - tp.ko) * RB : kt * RB;
    asm volatile(
        "{\n\t.reg .b64 t;\n\t"
        "mbarrier.arrive.expect_tx.shared::cta.b64 t, [%0], %1;\n\t}" ::"r"(bar),
        "r"((uint32_t)(kM * RB))
        : "memory");
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(raw) + (uint32_t)slot * (kM * RB)),
        "l"(cmap), "r"(x), "r"((int)ti.row0), "r"(bar)
        : "memory");
  };
  uint32_t tmem = 0;
  if (warp == kCodeWarp) {
    if (lane == 0) {
      for (int s = 0; s < kMaxRaw; ++s) {
        mbar_init(smem_u32(&rfull[s]), 1);
        mbar_init(smem_u32(&rempty[s]), kGroupWarps);
      }
      *abort_flag = 0;  // (thread 0 writes the same; this warp may poll it first)
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    asm volatile("bar.arrive 1, %0;" ::"n"(kThreadsTc) : "memory");
    if (lane == 0) {  // in unit order, until the next unit's sub-ring is full
      UnitPos up(u_begin, KT);
      for (; cl_u < u_end; ++cl_u) {
        const int t = up.t, kt = up.kt;
        const int g = (cl_u - u_begin) & 1, c = g ? cl_n1 : cl_n0;
        if (kt >= tp.ko && c == DRG) break;
        up.next(KT);
        if (kt < tp.ko) continue;  // outlier units read fp16 rows directly
        issue_codes(g + 2 * c, t, kt);
        if (g)
          ++cl_n1;
        else
          ++cl_n0;
      }
      cl_t = up.t;
      cl_kt = up.kt;
    }
  } else {
    if (tid == 0) {
      for (int s = 0; s < kMaxAStages; ++s) {
        mbar_init(smem_u32(&full[s]), kGroupWarps);  // one arrival per converter warp of a group
        mbar_init(smem_u32(&empty[s]), 1);
      }
      for (int s = 0; s < kMaxBStages; ++s) {
        mbar_init(smem_u32(&bfull[s]), 1);
        mbar_init(smem_u32(&bempty[s]), 1);
      }
      for (int s = 0; s < 2; ++s) {
        mbar_init(smem_u32(&dfull[s]), (uint32_t)tp.nmma);
        mbar_init(smem_u32(&dempty[s]), kEpiThreads);
      }
      *abort_flag = 0;
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(tmem_slot)),
                   "r"(kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    asm volatile("bar.sync 1, %0;" ::"n"(kThreadsTc) : "memory");
    fence_after();
    tmem = *tmem_slot;
  }
  // TMEM columns: issuer w's accumulators in buffer d at
  // [2 Np (d W + w), 2 Np (d W + w) + 2 Np) (outlier then background), A
  // stages from tp.a_base = 2 Np W nbuf.
  const int W = tp.nmma, NBUF = tp.nbuf;

  if (warp < kEpiWarp) {
    // ------------------------------------------------------ producers ----
    // Two groups of 4 warps (one per TMEM lane quarter) take alternate units:
    // group g the units at positions q = g (mod 2), so that every wait and
    // arrival of a group covers a whole unit's conversion.  Thread = one row
    // of the tile: its 128 codes of the unit become 64 fp16 pairs in two
    // halves of 32 TMEM columns of its own lane, one tcgen05.st each.
    const int g = warp >> 2, r = (warp & 3) * 32 + lane;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    // Background (INT4) or all (INT8) K tiles arrive as packed codes in the
    // raw ring (filled by the code loader warp); each thread converts its row.
    const uint32_t raw_me = smem_u32(raw) + (uint32_t)r * RB;
    // Weights only: no wait for the preceding kernel (under programmatic
    // launch the caller guarantees that nothing in flight writes them).
    int n = 0;       // code tiles this group has taken from its sub-ring
    int t_cur = -1;  // tile of the previous unit of this group
    TileInfo ti = {0, 0, 0};
    // This group visits only its own units, positions q = g, g + 2, ...
    // (A stage q mod NA: NA is even, so the group's stages are its own).
    int s = g % NA;                // A stage of the unit
    uint32_t aph = 0;              // parity of the stage's current round
    UnitPos up(u_begin + g, KT);   // (tile, K tile) of the unit
    const int n_units = u_end - u_begin;
    for (int q = g; q < n_units; q += 2) {
      const int t = up.t, kt = up.kt;
      const int s_here = s;
      const uint32_t aph_here = aph;
      up.kt += 2;
      while (up.kt >= KT) {
        up.kt -= KT;
        ++up.t;
      }
      s += 2;
      if (s >= NA) {
        s -= NA;
        aph ^= 1u;
      }
      const bool outl = INT4 && kt < tp.ko;
      if (q >= NA) {
        const bool ok = mbar_wait(smem_u32(&empty[s_here]), aph_here ^ 1u, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) break;
        fence_after();  // the MMAs that read this A stage are complete
      }
      if (t != t_cur) {
        ti = tile_info(tp, t);
        t_cur = t;
      }
      const int64_t grow = ti.row0 + r;
      const bool live = grow < ti.nrows;
      const uint32_t acol = tmem + lane_base + tp.a_base + (uint32_t)s_here * (kKT / 2);
      uint32_t o[32];  // fp16 pairs of k slots 2j, 2j+1 of one half (64 slots)
      if (outl) {
        const uint4 *src = reinterpret_cast<const uint4 *>(p.w_out[ti.m] + grow * p.ld_out[ti.m]);
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          const int t0 = kt * kKT + h * (kKT / 2);
#pragma unroll
          for (int kg = 0; kg < 8; ++kg) {
            const int tt = t0 + kg * 8;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (live && tt < p.n_out) {
              v = __ldg(src + tt / 8);
              // zero the slots past n_out inside the last group
              const int valid = p.n_out - tt;
              if (valid < 8) {
                uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 8; ++e)
                  if (e >= valid) w[e >> 1] &= (e & 1) ? 0x0000FFFFu : 0xFFFF0000u;
                v = make_uint4(w[0], w[1], w[2], w[3]);
              }
            }
            o[4 * kg] = v.x;
            o[4 * kg + 1] = v.y;
            o[4 * kg + 2] = v.z;
            o[4 * kg + 3] = v.w;
          }
          tmem_st32(acol + (uint32_t)h * 32, o);
        }
      } else {
        const int slot = g + 2 * (n % DRG);
        const bool ok = mbar_wait(smem_u32(&rfull[slot]), (n / DRG) & 1, abort_flag);
        ++n;
        if (!__all_sync(0xffffffffu, ok)) break;
        const uint32_t rsrc = raw_me + (uint32_t)slot * (kM * RB);
        if (INT4) {
          uint4 qv[4];  // the row's 64 code bytes (chunk c at c ^ ((r / 2) % 4): 64-byte swizzle)
#pragma unroll
          for (int c = 0; c < 4; ++c)
            asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(qv[c].x), "=r"(qv[c].y), "=r"(qv[c].z), "=r"(qv[c].w)
                         : "r"(rsrc + 16u * ((uint32_t)c ^ (((uint32_t)r >> 1) & 3u))));
          __syncwarp();  // the warp's codes are in registers
          if (lane == 0) mbar_arrive(smem_u32(&rempty[slot]));
          const uint32_t bias = 0x64086408u;  // 1032 in both halves after the XOR
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t words[8] = {qv[2 * h].x,     qv[2 * h].y,     qv[2 * h].z,
                                       qv[2 * h].w,     qv[2 * h + 1].x, qv[2 * h + 1].y,
                                       qv[2 * h + 1].z, qv[2 * h + 1].w};
#pragma unroll
            for (int kg = 0; kg < 8; ++kg) {
              const uint32_t w = words[kg];
              // Nibble pairs at bits 0-3 / 16-19: 1024 + (q+8) - 1032 = q.
              // Pairs at bits 4-7 / 20-23 are masked in place: 1024 + 16 (q+8),
              // then x/16 - 72 = q in one fused step (every value a small
              // integer, exact in fp16).  One shift by 8 serves the upper two
              // pairs.  Elements past kb hold zero nibbles (q = 0) from the
              // row padding, rows past N zeros; slot order 0,4,1,5,2,6,3,7
              // (pairs (e0,e4), (e1,e5), ...).
              const uint32_t w8 = w >> 8;
              o[4 * kg] = hsub2_u32((w & 0x000F000Fu) ^ bias, bias);
              o[4 * kg + 1] = hfma2_u32((w & 0x00F000F0u) ^ 0x64806480u, 0x2C002C00u, 0xD480D480u);
              o[4 * kg + 2] = hsub2_u32((w8 & 0x000F000Fu) ^ bias, bias);
              o[4 * kg + 3] = hfma2_u32((w8 & 0x00F000F0u) ^ 0x64806480u, 0x2C002C00u, 0xD480D480u);
            }
            if (!live) {
#pragma unroll
              for (int j = 0; j < 32; ++j) o[j] = 0;
            }
            tmem_st32(acol + (uint32_t)h * 32, o);
          }
        } else {
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            uint4 vv[4];  // 64 code bytes of this half (chunk k at k ^ (r % 8): 128-byte swizzle)
#pragma unroll
            for (int c = 0; c < 4; ++c)
              asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                           : "=r"(vv[c].x), "=r"(vv[c].y), "=r"(vv[c].z), "=r"(vv[c].w)
                           : "r"(rsrc + 16u * ((uint32_t)(4 * h + c) ^ ((uint32_t)r & 7u))));
            if (h == 1) {
              __syncwarp();  // the warp's codes are in registers
              if (lane == 0) mbar_arrive(smem_u32(&rempty[slot]));
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint32_t w[4] = {vv[c].x ^ 0x80808080u, vv[c].y ^ 0x80808080u,
                                     vv[c].z ^ 0x80808080u, vv[c].w ^ 0x80808080u};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                // 0x64 above each offset-binary byte: 1024 + (q + 128); minus 1152
                o[8 * c + 2 * k] = hsub2_u32(__byte_perm(w[k], 0x64646464u, 0x4140), 0x64806480u);
                o[8 * c + 2 * k + 1] = hsub2_u32(__byte_perm(w[k], 0x64646464u, 0x4342), 0x64806480u);
              }
            }
            if (!live) {
#pragma unroll
              for (int j = 0; j < 32; ++j) o[j] = 0;
            }
            tmem_st32(acol + (uint32_t)h * 32, o);
          }
        }
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      fence_before();
      __syncwarp();  // every lane's tensor-memory stores are complete
      if (lane == 0) mbar_arrive(smem_u32(&full[s_here]));
    }
  } else if (warp < kMmaWarp) {
    // ------------------------------------------------------- epilogue ----
    // Thread = one row of the tile (its TMEM lane).  Segment j of this CTA
    // (its units of one tile) sits in accumulator buffer j % 2.
    const int qtr = warp - kEpiWarp;  // == warp % 4: the TMEM lane quarter it may read
    const int r = qtr * 32 + lane;
    const uint32_t lane_base = (uint32_t)(qtr * 32) << 16;
    // Adds the partials of cut tile t (CTAs c_lo..c_hi, in that order) for
    // this lane quarter and stores the rows.  Each lane reads its own float4s
    // of every partial straight from L2 (ld.global.cg: other SMs wrote them
    // and L1 is not coherent with them), two partials per round trip, so the
    // sum needs no shared memory and runs as soon as the count says so.
    auto finish_tile = [&](int t, int c_lo, int c_hi) {
      const TileInfo ti = tile_info(tp, t);
      const int64_t grow = ti.row0 + r;
      const bool live = grow < ti.nrows;
      __half *yrow = p.y[ti.m] + grow;
      const int64_t ldy = p.ldy[ti.m];
      auto part = [&](int k) {  // CTA k's partial of this lane quarter: float4 (n / 4, lane)
        return reinterpret_cast<const float4 *>(
                   tp.part + (size_t)((k * 2 + part_slot(tp, k, t)) * 4 + qtr) * Np * 32) +
               lane;
      };
      for (int n0 = 0; n0 < tp.B; n0 += 16) {  // 16 columns: 4 float4 per partial
        float4 acc[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[q] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        for (int k = c_lo; k <= c_hi; k += 2) {
          const bool two = k + 1 <= c_hi;
          const float4 *pa = part(k) + (n0 / 4) * 32;
          const float4 *pb = part(two ? k + 1 : k) + (n0 / 4) * 32;
          float4 va[4], vb[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) va[q] = ld_cg_f4(pa + q * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q) vb[q] = two ? ld_cg_f4(pb + q * 32) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            acc[q].x += va[q].x;
            acc[q].y += va[q].y;
            acc[q].z += va[q].z;
            acc[q].w += va[q].w;
          }
          if (two) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              acc[q].x += vb[q].x;
              acc[q].y += vb[q].y;
              acc[q].z += vb[q].z;
              acc[q].w += vb[q].w;
            }
          }
        }
        if (live) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float e[4] = {acc[q].x, acc[q].y, acc[q].z, acc[q].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int n = n0 + 4 * q + i;
              if (n < tp.B) yrow[(int64_t)n * ldy] = __float2half_rn(e[i]);
            }
          }
        }
      }
    };
    asm volatile("griddepcontrol.wait;" ::: "memory");
    int j = 0;
    for (int u = u_begin; u < u_end; ++j) {
      const int t = u / KT;
      const int k0 = u - t * KT;
      const int seg_end = u_end < (t + 1) * KT ? u_end : (t + 1) * KT;
      const int k1 = seg_end - t * KT;
      u = seg_end;
      const TileInfo ti = tile_info(tp, t);
      const int64_t grow = ti.row0 + r;
      const bool live = grow < ti.nrows;
      const int kso = k1 < tp.ko ? k1 : tp.ko;  // outlier K tiles of the segment: [k0, kso)
      const int ksb = k0 > tp.ko ? k0 : tp.ko;  // background K tiles: [ksb, k1)
      bool has_out[kMaxIssuers], has_bg[kMaxIssuers];
#pragma unroll
      for (int w = 0; w < kMaxIssuers; ++w) {
        has_out[w] = INT4 && w < W && issuer_has(W, w, t, k0, kso, KT, u_begin);
        has_bg[w] = w < W && issuer_has(W, w, t, ksb, k1, KT, u_begin);
      }
      const bool cut = !(k0 == 0 && k1 == KT);
      float s_i = 1.0f;
      if (live) s_i = INT4 ? __ldg(p.scale[ti.m] + grow) : __ldg(p.scale[ti.m]);
      __half *yrow = p.y[ti.m] + grow;
      const int64_t ldy = p.ldy[ti.m];
      const int db = NBUF == 2 ? (j & 1) : 0;
      const bool ok = mbar_wait(smem_u32(&dfull[db]), (NBUF == 2 ? (j >> 1) : j) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      fence_after();
      const uint32_t dcol = tmem + lane_base + (uint32_t)(db * W * 2 * Np);
      // partial of a cut tile: float4 (n / 4, lane) of its (slot, quarter) block
      float4 *mine = nullptr;
      float *mine_c = reinterpret_cast<float *>(b_st) + r;  // kCluster: [n][kM] in its own rings
      if (cut && tp.split != kCluster)
        mine = reinterpret_cast<float4 *>(
                   tp.part + (size_t)((cta * 2 + part_slot(tp, cta, t)) * 4 + qtr) * Np * 32) +
               lane;
      for (int c0 = 0; c0 < Np; c0 += 16) {
        float y[16], o[16];  // y: background sum, then the result
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) y[jj] = o[jj] = 0.0f;
#pragma unroll
        for (int w = 0; w < kMaxIssuers; ++w) {  // issuers' partials, in issuer order
          float v[16];
          const uint32_t col = dcol + (uint32_t)(w * 2 * Np);
          if (has_bg[w]) {
            tmem_ld16(col + (uint32_t)Np + c0, v);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) y[jj] += v[jj];
          }
          if (has_out[w]) {
            tmem_ld16(col + c0, v);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) o[jj] += v[jj];
          }
        }
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) y[jj] = fmaf(s_i, y[jj], o[jj]);  // this CTA's units of the tile
        if (!cut) {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj)
            if (live && c0 + jj < tp.B) yrow[(int64_t)(c0 + jj) * ldy] = __float2half_rn(y[jj]);
        } else if (tp.split == kCluster) {  // this CTA's only segment; its rings are free
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) mine_c[(c0 + jj) * kM] = y[jj];
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            mine[(c0 / 4 + q) * 32] = make_float4(y[4 * q], y[4 * q + 1], y[4 * q + 2], y[4 * q + 3]);
        }
      }
      fence_before();
      mbar_arrive(smem_u32(&dempty[db]));  // the MMAs may reuse this buffer
      if (!cut || tp.split == kCluster) continue;
      // Publish the partial (release: the warp's stores, ordered by the warp
      // barrier, before the count); the warp that brings the count of its
      // lane quarter to the number of contributors adds them all in CTA order.
      const int c_lo = unit_owner(tp, t * KT), c_hi = unit_owner(tp, (t + 1) * KT - 1);
      __syncwarp();
      unsigned prev = 0;
      if (lane == 0)
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                     : "=r"(prev)
                     : "l"(tp.cnt + c_lo * 4 + qtr)
                     : "memory");
      prev = __shfl_sync(0xffffffffu, prev, 0);
      if (prev != (unsigned)(c_hi - c_lo)) continue;
      __syncwarp();  // lane 0's acquire, then every lane's loads of the partials
      finish_tile(t, c_lo, c_hi);
    }
  } else if (warp == kMmaWarp || warp == kMma2Warp) {
    // ---------------------------------------------------- MMA issuers ---
    // One thread per issuing warp; issuer w takes the units at positions
    // q = w (mod W) of the CTA's range into its own accumulators, so that the
    // serial issue cost of each tcgen05.mma is paid by W threads in parallel.
    // Every issuer commits once per segment to the accumulator-full barrier
    // (W arrivals), after the drain of that buffer's previous segment.
    const int w = warp == kMmaWarp ? 0 : 1;
    if (lane == 0 && w < W) {
      asm volatile("griddepcontrol.wait;" ::: "memory");
      const uint32_t idesc = idesc_f16(kM, Np);
      // This issuer visits only its own units (positions q = w, w + W, ...).
      // Segment j of the range is tile t0 + j; the issuer enters every
      // segment in order (waiting for the drain of that buffer's previous
      // segment) and commits each one's accumulator-full barrier once, right
      // after its last own unit there, or on leaving a segment it had no unit
      // in, so that the barrier sees W arrivals per segment.
      const int n_units = u_end - u_begin;
      const int t0 = u_begin / KT, j_last = n_units > 0 ? (u_end - 1) / KT - t0 : -1;
      int jc = -1;       // segment entered
      bool cm = false;   // its accumulator-full barrier committed
      uint32_t dcol = 0;
      int db = 0;
      bool seen_out = false, seen_bg = false;  // this issuer's first unit of each kind in the segment
      bool ok = true;
      auto enter_through = [&](int jq) {  // move to segment jq, closing the ones left
        while (jc < jq) {
          if (jc >= 0 && !cm) mma_commit(smem_u32(&dfull[db]));
          ++jc;
          cm = false;
          db = NBUF == 2 ? (jc & 1) : 0;
          dcol = (uint32_t)((db * W + w) * 2 * Np);
          seen_out = seen_bg = false;
          if (jc >= NBUF) {
            if (!mbar_wait(smem_u32(&dempty[db]), ((NBUF == 2 ? (jc >> 1) : jc) - 1) & 1, abort_flag)) {
              ok = false;
              return;
            }
            fence_after();
          }
        }
      };
      UnitPos up(u_begin + w, KT);  // (tile, K tile) of position q
      int s = w % NA, sb = w % NB;
      uint32_t aph = 0, bph = 0;
      for (int q = w; q < n_units && ok; q += W) {
        const int kt = up.kt;
        enter_through(up.t - t0);
        if (!ok) break;
        if (!mbar_wait(smem_u32(&full[s]), aph, abort_flag)) break;
        if (!mbar_wait(smem_u32(&bfull[sb]), bph, abort_flag)) break;
        fence_after();
        const bool outl = kt < tp.ko;
        const uint32_t a0 = tmem + tp.a_base + (uint32_t)s * (kKT / 2);
        const uint32_t b0 = smem_u32(b_st + sb * bBytes);
        const uint32_t d = tmem + dcol + (outl ? 0u : (uint32_t)Np);
        const bool first = outl ? !seen_out : !seen_bg;
        if (outl)
          seen_out = true;
        else
          seen_bg = true;
        static_assert(kKT / 16 == 8 && 2 * kLBO / 16 == 16, "mma8_f16_ta covers one unit");
        const uint64_t bd = sdesc(b0);
        mma8_f16_ta(d, a0, (uint32_t)bd, (uint32_t)(bd >> 32), idesc, first ? 0u : 1u);
        mma_commit(smem_u32(&empty[s]));
        mma_commit(smem_u32(&bempty[sb]));
        if (q + W >= n_units || kt + W >= KT) {  // its last unit of this segment
          mma_commit(smem_u32(&dfull[db]));
          cm = true;
        }
        // next own position: W units on
        up.kt += W;
        while (up.kt >= KT) {
          up.kt -= KT;
          ++up.t;
        }
        s += W;
        if (s >= NA) {
          s -= NA;
          aph ^= 1u;
        }
        sb += W;
        if (sb >= NB) {
          sb -= NB;
          bph ^= 1u;
        }
      }
      if (ok) {  // the segments after its last unit, and the last one's barrier
        enter_through(j_last);
        if (ok && jc >= 0 && !cm) mma_commit(smem_u32(&dfull[db]));
      }
    }
  } else if (warp == kCodeWarp) {
    // ------------------------------------------------------ code loader ---
    // Packed codes of the background (INT4) or all (INT8) K tiles of this
    // CTA's units, one 2D tensor copy of kM rows x ROWB bytes each, DR ahead
    // of the converters.  The codes are static: no wait for earlier kernels.
    if (lane == 0) {
      // (the first copies went out in the prologue)
      int n0 = cl_n0, n1 = cl_n1;
      UnitPos up(u_begin, KT);
      up.t = cl_t;
      up.kt = cl_kt;
      for (int u = cl_u; u < u_end; ++u) {
        const int t = up.t, kt = up.kt;
        up.next(KT);
        if (kt < tp.ko) continue;  // outlier units read fp16 rows directly
        const int g = (u - u_begin) & 1, c = g ? n1 : n0;
        const int slot = g + 2 * (c % DRG);
        if (c >= DRG) {
          if (!mbar_wait(smem_u32(&rempty[slot]), ((c / DRG) - 1) & 1, abort_flag)) break;
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        issue_codes(slot, t, kt);
        if (g)
          ++n1;
        else
          ++n0;
      }
      if (*(volatile int *)abort_flag)  // let the copies in flight land
        for (int g = 0; g < 2; ++g) {
          const int ng = g ? n1 : n0;
          for (int c = ng > DRG ? ng - DRG : 0; c < ng; ++c)
            mbar_drain(smem_u32(&rfull[g + 2 * (c % DRG)]), (c / DRG) & 1);
        }
    }
  } else if (warp == kLoadWarp) {
    // ------------------------------------------------ activation loader ---
    // Np x kKT activations per unit, NB units ahead of the MMAs.  With a
    // workspace the tile was gathered once per call by tc_xprep_kernel and
    // arrives by one bulk copy; without one this warp gathers it.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    int q = 0;
    RingPos bp;
    UnitPos up(u_begin, KT);
    for (int u = u_begin; u < u_end; ++u, ++q) {
      const int kt = up.kt;
      const int sb = bp.slot;
      const uint32_t bph = bp.parity;
      up.next(KT);
      bp.next(NB);
      if (q >= NB) {
        const bool ok = mbar_wait(smem_u32(&bempty[sb]), bph ^ 1u, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      uint8_t *Bt = b_st + sb * bBytes;
      const uint32_t bar = smem_u32(&bfull[sb]);
      if (tp.ws) {
        if (lane == 0) {
          asm volatile(
              "{\n\t.reg .b64 t;\n\t"
              "mbarrier.arrive.expect_tx.shared::cta.b64 t, [%0], %1;\n\t}" ::"r"(bar),
              "r"((uint32_t)bBytes)
              : "memory");
          asm volatile(
              "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
              "[%3];" ::"r"(smem_u32(Bt)),
              "l"(tp.ws + (size_t)kt * bBytes), "r"((uint32_t)bBytes), "r"(bar)
              : "memory");
        }
      } else {
        const bool outl = kt < tp.ko;
        for (int idx = lane; idx < Np * kKT; idx += 32) {
          const int c = idx % kKT, n = idx / kKT;
          __half v = __float2half_rn(0.0f);
          if (n < tp.B) {
            const __half *xb = p.x + (int64_t)n * p.ldx;
            if (INT4 && outl) {
              const int tt = kt * kKT + c;
              if (tt < p.n_out) v = xb[__ldg(p.perm + tt)];
            } else if (INT4) {
              const int e = (kt - tp.ko) * kKT + slot_elem(c);
              if (e < p.kb) v = xb[__ldg(p.perm + p.n_out + e)];
            } else {
              const int e = kt * kKT + c;
              if (e < p.K) v = xb[e];
            }
          }
          *reinterpret_cast<__half *>(Bt + core_off(n, c)) = v;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(bar);
      }
    }
    if (tp.ws && lane == 0 && *(volatile int *)abort_flag)  // let the copies in flight land
      for (int k = q > NB ? q - NB : 0; k < q; ++k) mbar_drain(smem_u32(&bfull[k % NB]), (k / NB) & 1);
  }

  __syncwarp();
  if (tp.split == kCluster && tp.S > 1) {
    // Cluster reduction through distributed shared memory: each CTA holds
    // the partial of its K tiles, [n][row] fp32 at the start of its rings;
    // CTA k adds rows [k kM / S, (k + 1) kM / S) over the S CTAs in rank
    // order and stores them.
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
    const int S = tp.S, rank = cta % S, t = cta / S;
    const TileInfo ti = tile_info(tp, t);
    const int rlo = kM * rank / S, nr = kM * (rank + 1) / S - rlo;
    const uint32_t local = smem_u32(b_st);
    for (int e = tid; e < nr * tp.B; e += kThreadsTc) {
      const int n = e / nr, rr = rlo + e % nr;
      const uint32_t off = (uint32_t)(n * kM + rr) * 4u;
      float v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q)  // all S loads in flight, then the sum in rank order
        if (q < S) {
          uint32_t ra;
          asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(local + off), "r"(q));
          asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v[q]) : "r"(ra));
        }
      float acc = 0.0f;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (q < S) acc += v[q];
      const int64_t grow = ti.row0 + rr;
      if (grow < ti.nrows) p.y[ti.m][(int64_t)n * p.ldy[ti.m] + grow] = __float2half_rn(acc);
    }
    // keep every CTA's shared memory alive until all remote reads are done
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                 : "memory");
}

// The B operand of every K tile, gathered through the permutation (INT4:
// in the k order of the nibble conversion) into the canonical K-major layout,
// one contiguous tile of Np x 64 fp16 per K tile.  One CTA per (K tile, 16
// batch rows).
template <bool INT4>
__global__ void __launch_bounds__(256) tc_xprep_kernel(const __grid_constant__ TcParams tp,
                                                       uint8_t *ws) {
  const GemvParams &p = tp.g;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int kt = blockIdx.x;
  // the arrival counters of the cut tiles start every call at zero
  if (kt == 0 && blockIdx.y == 0 && tp.cnt)
    for (int i = threadIdx.x; i < 4 * tp.G; i += blockDim.x) tp.cnt[i] = 0u;
  const int bBytes = tp.Np * kKT * 2;
  uint8_t *tile = ws + (size_t)kt * bBytes;
  const bool outl = kt < tp.ko;
  // Eight elements per thread and step, all eight loads issued before the
  // one 16-byte store: the compiler cannot prove that the workspace does not
  // alias the inputs, so loads and stores mixed in one loop stay in order.
  // this CTA's batch rows: [16 y, 16 y + 16)
  const int total = (blockIdx.y + 1) * 16 * kKT;
  for (int base = blockIdx.y * 16 * kKT + threadIdx.x * 8; base < total; base += 256 * 8) {
    __half v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int idx = base + k;             // 8 consecutive k slots of one row n
      const int c = idx % kKT, n = idx / kKT;
      v[k] = __ushort_as_half((unsigned short)0);
      if (n < tp.B) {
        const __half *xb = p.x + (int64_t)n * p.ldx;
        if (INT4 && outl) {
          const int t = kt * kKT + c;
          if (t < p.n_out) v[k] = xb[__ldg(p.perm + t)];
        } else if (INT4) {
          const int e = (kt - tp.ko) * kKT + slot_elem(c);
          if (e < p.kb) v[k] = xb[__ldg(p.perm + p.n_out + e)];
        } else {
          const int e = kt * kKT + c;
          if (e < p.K) v[k] = xb[e];
        }
      }
    }
    // slots c .. c+7 (c a multiple of 8) are one 16-byte core-matrix row
    const int c = base % kKT, n = base / kKT;
    uint32_t h[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      h[k] = (uint32_t)__half_as_ushort(v[2 * k]) | ((uint32_t)__half_as_ushort(v[2 * k + 1]) << 16);
    *reinterpret_cast<uint4 *>(tile + core_off(n, c)) = make_uint4(h[0], h[1], h[2], h[3]);
  }
}

}  // namespace

static size_t tc_part_bytes(int64_t Np) { return (size_t)2 * kMaxCtas * Np * kM * sizeof(float); }

size_t tc_workspace_bytes(bool int4, int64_t B, int64_t K, int64_t n_out) {
  const int64_t Np = (B + 15) / 16 * 16;
  const int64_t tiles = int4 ? (n_out + kKT - 1) / kKT + (K - n_out + kKT - 1) / kKT
                             : (K + kKT - 1) / kKT;
  // gathered activations, then the partials of cut tiles (two per CTA), then
  // one arrival counter per CTA and TMEM lane quarter
  return (size_t)(tiles * Np * kKT * 2) + tc_part_bytes(Np) + (size_t)kMaxCtas * 4 * sizeof(unsigned);
}

// Stages of the activation ring for a batch of Np (MMA N) columns.
static int tc_b_stages(int Np) {
  const size_t per = (size_t)Np * kKT * 2;
  const size_t n = kBRingBytes / per;
  return (int)(n < (size_t)kMaxBStages ? n : (size_t)kMaxBStages);
}

size_t tc_smem_bytes(bool int4, int Np) {
  // barriers, activation ring, raw-code ring; the host launches with the
  // device's whole per-CTA maximum (one CTA per SM, which holds all 512 TMEM
  // columns), the space past the rings staging the cut-tile reduction
  return 1024 + kBarBytes + (size_t)tc_b_stages(Np) * Np * kKT * 2 +
         (int4 ? RawRing<true>::BYTES : RawRing<false>::BYTES);
}

namespace {

// cuTensorMapEncodeTiled, found once through the runtime's driver entry point
// (the library does not link the driver API).
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// The packed codes of one matrix as a 2D byte tensor [rows][ld bytes], read
// in boxes of kM rows x row_bytes bytes (rows past the end read as zeros).
// The copy swizzles the 16-byte chunks of each row (64- or 128-byte pattern,
// the row's own size), so that the converter threads, one row each, read a
// chunk column without shared-memory bank conflicts.
qz_status codes_map(CUtensorMap *map, const uint8_t *codes, int64_t ld, int64_t rows,
                    int row_bytes) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return QZ_ERR_CUDA;
  const cuuint64_t dim[2] = {(cuuint64_t)ld, (cuuint64_t)rows};
  const cuuint64_t stride[1] = {(cuuint64_t)ld};
  const cuuint32_t box[2] = {(cuuint32_t)row_bytes, (cuuint32_t)kM};
  const cuuint32_t estride[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(codes), dim,
                        stride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        row_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                        : row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                          : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? QZ_OK : QZ_ERR_INVALID_ARG;
}

}  // namespace

// Clusters of S CTAs of the GEMM kernel that the GPU holds at once (one CTA
// per SM; GPCs whose SM count is not a multiple of S strand some SMs).
// Asked of the runtime once per device, format and S.
template <typename Kern>
qz_status tc_resident_clusters(bool int4, Kern kern, int S, size_t smem, int sms, int *out) {
  if (S == 1) {
    *out = sms;
    return QZ_OK;
  }
  constexpr int kDev = 16;
  // 0 = not asked yet, -1 = not launchable; threads that race ask the
  // runtime twice and store the same answer
  static std::atomic<int> cache[kDev][2][4];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e);
  const int si = S == 2 ? 1 : (S == 4 ? 2 : 3);
  if (dev < 0 || dev >= kDev) {
    *out = 0;
    return QZ_OK;
  }
  std::atomic<int> &c = cache[dev][int4 ? 1 : 0][si];
  int v = c.load(std::memory_order_relaxed);
  if (v == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)S);
    cfg.blockDim = dim3(kThreadsTc);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute a;
    a.id = cudaLaunchAttributeClusterDimension;
    a.val.clusterDim.x = (unsigned)S;
    a.val.clusterDim.y = 1;
    a.val.clusterDim.z = 1;
    cfg.attrs = &a;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();  // not a sticky error: this S is just not used
      n = -1;
    }
    v = n > 0 ? n : -1;
    c.store(v, std::memory_order_relaxed);
  }
  *out = v > 0 ? v : 0;
  return QZ_OK;
}

qz_status launch_tc(bool int4, int B, const GemvParams &g, const int64_t *mat_rows,
                    void *workspace, size_t workspace_bytes, cudaStream_t s) {
  DeviceInfo di;
  qz_status st = device_info(&di);
  if (st != QZ_OK) return st;
  TcParams tp;
  memset(&tp, 0, sizeof(tp));
  tp.g = g;
  tp.B = B;
  tp.Np = (B + 15) / 16 * 16;
  tp.nbs = tc_b_stages(tp.Np);
  // Two MMA issuers with double-buffered accumulators where tensor memory
  // leaves at least 4 A stages, else single-buffered, else one issuer.
  tp.nmma = 1;
  tp.nbuf = 2;
  for (int cand = 0; cand < 3; ++cand) {
    const int W = cand < 2 ? 2 : 1, nb = cand == 1 ? 1 : 2;
    const int64_t a_base = (int64_t)nb * W * 2 * tp.Np;
    if ((kTmemCols - a_base) / (kKT / 2) >= 4 || cand == 2) {
      tp.nmma = W;
      tp.nbuf = nb;
      break;
    }
  }
  tp.a_base = (uint32_t)(tp.nbuf * tp.nmma * 2 * tp.Np);
  tp.nsa = (int)((kTmemCols - tp.a_base) / (kKT / 2));
  if (tp.nsa > kMaxAStages) tp.nsa = kMaxAStages;
  // Even, so that each A stage is filled by one converter group and read by
  // one issuer, in order (mbarrier waits tell phases apart by parity only).
  tp.nsa &= ~1;
  tp.ko = int4 ? (g.n_out + kKT - 1) / kKT : 0;
  tp.kbt = int4 ? (g.kb + kKT - 1) / kKT : (g.K + kKT - 1) / kKT;
  tp.KT = tp.ko + tp.kbt;
  tp.ws = nullptr;
  if (workspace) {
    const size_t xbytes = tc_workspace_bytes(int4, B, g.K, g.n_out) - tc_part_bytes(tp.Np) -
                          (size_t)kMaxCtas * 4 * sizeof(unsigned);
    if (workspace_bytes < tc_workspace_bytes(int4, B, g.K, g.n_out)) return QZ_ERR_INVALID_ARG;
    if ((uintptr_t)workspace & 15u) return QZ_ERR_ALIGNMENT;
    tp.ws = reinterpret_cast<const uint8_t *>(workspace);
    tp.part = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(workspace) + xbytes);
    tp.cnt = reinterpret_cast<unsigned *>(reinterpret_cast<uint8_t *>(workspace) + xbytes +
                                          tc_part_bytes(tp.Np));
  }
  for (int m = 0; m < g.n_mats; ++m)
    if (tp.kbt > 0) {
      st = codes_map(&tp.codes_map[m], g.codes[m], g.ld_codes[m], mat_rows[m],
                     int4 ? RawRing<true>::ROWB : RawRing<false>::ROWB);
      if (st != QZ_OK) return st;
    }
  int64_t tiles = 0;
  for (int m = 0; m < QZ_MAX_GROUP; ++m) {
    tp.mat_rows[m] = m < g.n_mats ? mat_rows[m] : 0;
    tp.n_tiles[m] = m < g.n_mats ? (int)((mat_rows[m] + kM - 1) / kM) : 0;
    tiles += tp.n_tiles[m];
    tp.tile_end[m] = (int)tiles;
  }
  if (tiles == 0 || tp.KT == 0) return QZ_OK;
  if (tiles * tp.KT > (int64_t)INT32_MAX) return QZ_ERR_UNSUPPORTED;
  tp.tiles = (int)tiles;
  tp.U = (int)(tiles * tp.KT);
  if (tc_smem_bytes(int4, tp.Np) > (size_t)di.max_smem_optin) return QZ_ERR_UNSUPPORTED;
  // 200 KB: below the SM's total, so that a small kernel launched before
  // this one (the input gather) can still run beside it under programmatic
  // launch; the cluster schedule stages its partial ([B][kM] fp32) in the rings
  const size_t smem = (size_t)di.max_smem_optin < (size_t)200 * 1024 ? (size_t)di.max_smem_optin
                                                                      : (size_t)200 * 1024;
  if (smem < tc_smem_bytes(int4, tp.Np)) return QZ_ERR_UNSUPPORTED;
  auto kern = int4 ? tc_gemm_kernel<true> : tc_gemm_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_status(e);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
  if (e != cudaSuccess) return cuda_status(e);

  // Schedule.  Estimated times in microseconds, fitted to GB300 timings of
  // an earlier build of this kernel (units now cost about half as much; the
  // choices were re-checked against forced schedules and still pick the
  // faster one): a launch costs kStart (start-up to the first MMA and the
  // drain after the last), a unit 0.9 (8 MMAs); stream-K adds the L2
  // reduction of its cut tiles, a cluster of S > 1 its shared-memory
  // reduction, and clusters come in waves of what fits on the GPCs at once.
  const int gmax = di.sms < kMaxCtas ? di.sms : kMaxCtas;
  const double kStart = 3.5, kUnit = 0.9;
  double best = 1e30;
  int best_mode = kWhole, best_S = 1;
  {
    const int per = (tp.tiles + gmax - 1) / gmax;  // whole tiles per CTA
    best = kStart + kUnit * per * tp.KT;
  }
  if (tp.ws) {
    const int want = tp.U / kMinUnits;
    const int G = want < 1 ? 1 : (want < gmax ? want : gmax);
    const int per = (tp.U + G - 1) / G;
    const bool cuts = !(tp.U % G == 0 && (tp.U / G) % tp.KT == 0);
    const double t = kStart + kUnit * per + (cuts ? 5.5 + tp.B / 16.0 : 0.0);
    if (t < best) {
      best = t;
      best_mode = kStreamK;
    }
  }
  for (int S = 1; S <= 8; S *= 2) {
    if (S > 1 && tp.KT < 2 * S) break;
    int clusters = 0;
    st = tc_resident_clusters(int4, kern, S, smem, di.sms, &clusters);
    if (st != QZ_OK) return st;
    if (clusters < 1) continue;
    const int waves = (tp.tiles + clusters - 1) / clusters;
    const double t = waves * (kStart + kUnit * ((tp.KT + S - 1) / S) +
                              (S > 1 ? 1.0 + tp.B / 40.0 : 0.0));
    if (t < best - 1e-9) {
      best = t;
      best_mode = kCluster;
      best_S = S;
    }
  }
  tp.split = best_mode;
  tp.S = best_S;
  if (best_mode == kStreamK) {
    const int want = tp.U / kMinUnits;
    tp.G = want < 1 ? 1 : (want < gmax ? want : gmax);
  } else if (best_mode == kCluster) {
    tp.G = tp.tiles * tp.S;
    tp.cnt = nullptr;  // no cut-tile counters (and none to clear)
  } else {
    tp.G = tp.tiles < gmax ? tp.tiles : gmax;
    tp.cnt = nullptr;
  }

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)tp.G);
  cfg.blockDim = dim3(kThreadsTc);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (g.overlap) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  const int n_pdl = na;
  if (tp.split == kCluster) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = (unsigned)tp.S;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  if (tp.ws) {  // gather the activations once (and clear the counters), then the GEMM
    cudaLaunchConfig_t pc = {};
    pc.gridDim = dim3((unsigned)tp.KT, (unsigned)(tp.Np / 16));
    pc.blockDim = dim3(256);
    pc.stream = s;
    pc.attrs = attr;
    pc.numAttrs = n_pdl;
    auto prep = int4 ? tc_xprep_kernel<true> : tc_xprep_kernel<false>;
    e = cudaLaunchKernelEx(&pc, prep, tp, reinterpret_cast<uint8_t *>(workspace));
    if (e != cudaSuccess) return cuda_status(e);
  }
  e = cudaLaunchKernelEx(&cfg, kern, tp);
  if (e != cudaSuccess) return cuda_status(e);
  return launch_status();
}

qz_status read_device_error(int *code, int clear) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int));
  if (e != cudaSuccess) return cuda_status(e);
  if (clear && v) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_status(e);
  }
  *code = v;
  return QZ_OK;
}

}  // namespace qz

// ---------------------------------------------------------------------------
// Allocation-free batched INT4-outlier product.
//
// Some callers cannot allocate device memory at the point where they run the
// product: code that runs while a CUDA graph is being captured (cudaMalloc is
// not a capturable operation), plugins that live inside a host application
// which owns the device memory budget and hands out no allocator, and
// real-time loops that must not touch the allocator after start-up.  For them
// the tensor-core path's gathered-input workspace lives in a library-owned,
// fixed-size device array instead of caller memory.  Every GPU that loads the
// library holds this array until the process exits.
// ---------------------------------------------------------------------------
namespace qz {
namespace {

constexpr size_t kNoAllocScratchBytes = QZ_NOALLOC_SCRATCH_BYTES;  // the header's stated limit
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array on the current device.  The name of a
// __device__ array is only a host-side stand-in in host code, so its address
// is looked up once per device with that device current.
qz_status noalloc_scratch(void **out) {
  constexpr int kMaxDev = 64;
  static void *addr[kMaxDev];
  static cudaError_t err[kMaxDev];
  static std::once_flag once[kMaxDev];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e);
  if (dev < 0 || dev >= kMaxDev) return QZ_ERR_UNSUPPORTED;
  std::call_once(once[dev], [&] {
    err[dev] = cudaGetSymbolAddress(&addr[dev], g_noalloc_scratch);
  });
  if (err[dev] != cudaSuccess) return cuda_status(err[dev]);
  *out = addr[dev];
  return QZ_OK;
}

}  // namespace
}  // namespace qz

extern "C" qz_status qz_gemm_int4_outlier_noalloc(const qz_int4o_weight *w, int64_t B,
                                                  const qz_half *X, int64_t ldx, qz_half *Y,
                                                  int64_t ldy, qz_stream s) {
  // The batch and weight-size checks come first, in the order and with the
  // statuses of qz_gemm_int4_outlier, so that only the scratch limit below
  // can make the two calls answer differently.
  if (!w) return QZ_ERR_INVALID_ARG;
  if (w->N < 1 || w->K < 1 || w->n_out < 0 || w->n_out > w->K) return QZ_ERR_INVALID_ARG;
  if (B < 1) return QZ_ERR_INVALID_ARG;
  if (B > QZ_MAX_BATCH) return QZ_ERR_UNSUPPORTED;
  const size_t need = qz_gemm_workspace_bytes(B, w->K, w->n_out);
  if (need == 0) return QZ_ERR_INVALID_ARG;  // not reached: B, K and n_out are in range
  if (need > qz::kNoAllocScratchBytes) return QZ_ERR_UNSUPPORTED;
  void *scratch = nullptr;
  qz_status st = qz::noalloc_scratch(&scratch);
  if (st != QZ_OK) return st;
  // The existing entry point with the scratch array as its workspace: the
  // gather kernel rewrites every byte of the tiles it uses, so nothing needs
  // clearing between calls.
  return qz_gemm_int4_outlier(w, B, X, ldx, Y, ldy, scratch, qz::kNoAllocScratchBytes, s);
}
