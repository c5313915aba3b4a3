// Quantize / pack kernels.  All decisions that produce integers are taken in
// fp32 with IEEE division (__fdiv_rn) and round-half-to-even (rintf); there
// is no fast-math anywhere in the library, so codes are bit-reproducible.
//
//  * INT8 per tensor: "Open Origin - ELG Stream Layer", Technical
//    Architecture, INT8 Quantization & Direct Mapping (scale = max|W|/127,
//    q = round(W/scale)).
//  * Saliency, outlier selection, INT4 split/quantize/pack: "On-The-Fly
//    Weight Synthesizer (OTF-LLM Engine)", Architecture & Key Innovations
//    (diagram; key innovation 3: top-1% channels by |W| x |X_profile| kept in
//    FP16 behind global_perm_idx; background INT4 in [-7,7], zero-point 0,
//    2:1 packing into uint8).
#include "qz_internal.cuh"

namespace qz {
namespace {

// |h| of an fp16 bit pattern as an order-preserving integer (finite values).
__device__ __forceinline__ uint32_t abs_bits(uint16_t h) { return h & 0x7FFFu; }

__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// --------------------------------------------------------------- INT8 -----
// Pass 1: max |W| over the tensor.  Each warp folds its maximum into *amax
// (the bit pattern of a non-negative fp32 number orders like an unsigned int).
__global__ void int8_absmax_kernel(const __half *__restrict__ W, int64_t N,
                                   int64_t K, int64_t ldw,
                                   unsigned int *amax) {
  const int64_t vpr = (K + 7) / 8;  // 8-half vectors per row holding data
  const int64_t total = N * vpr;
  uint32_t m = 0;
  for (int64_t v = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; v < total;
       v += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = v / vpr, j0 = (v % vpr) * 8;
    const uint4 d = __ldg(reinterpret_cast<const uint4 *>(W + i * ldw + j0));
    const uint16_t *h = reinterpret_cast<const uint16_t *>(&d);
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (j0 + e < K) m = max(m, abs_bits(h[e]));
  }
  // fp16 magnitude -> fp32 bits (exact), then reduce.
  uint32_t f = __float_as_uint(__half2float(__ushort_as_half((uint16_t)m)));
  f = warp_max_u32(f);
  if ((threadIdx.x & 31) == 0 && f) atomicMax(amax, f);
}

// Pass 2: q = clamp(rint(fp32(W) / s), -127, 127) with s = amax / 127.  Each
// thread writes one 16-byte run of q; columns K..ldq-1 are written as 0.
__global__ void int8_quant_kernel(const __half *__restrict__ W, int64_t N,
                                  int64_t K, int64_t ldw, int8_t *__restrict__ q,
                                  int64_t ldq, const float *amax_in) {
  const float amax = *amax_in;
  const float s = __fdiv_rn(amax, 127.0f);
  const int64_t rpr = ldq / 16;
  const int64_t total = N * rpr;
  for (int64_t v = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; v < total;
       v += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = v / rpr, j0 = (v % rpr) * 16;
    uint32_t out[4] = {0, 0, 0, 0};
    if (s != 0.0f) {
#pragma unroll
      for (int half8 = 0; half8 < 2; ++half8) {
        const int64_t jb = j0 + 8 * half8;
        if (jb >= K) break;
        const uint4 d = __ldg(reinterpret_cast<const uint4 *>(W + i * ldw + jb));
        const __half *h = reinterpret_cast<const __half *>(&d);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          int code = 0;
          if (jb + e < K) {
            float r = rintf(__fdiv_rn(__half2float(h[e]), s));
            r = fminf(fmaxf(r, -127.0f), 127.0f);
            code = (int)r;
          }
          const int byte = 8 * half8 + e;
          out[byte >> 2] |= (uint32_t)(code & 0xFF) << (8 * (byte & 3));
        }
      }
    }
    *reinterpret_cast<uint4 *>(q + i * ldq + j0) = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

// Pass 3: the stored scale.
__global__ void int8_scale_kernel(float *scale) {
  *scale = __fdiv_rn(*scale, 127.0f);
}

// ----------------------------------------------------------- saliency ----
// |fp16| in units of 2^-24 as an exact integer.
__device__ __forceinline__ uint64_t fp16_units(uint16_t h) {
  const uint32_t e = (h >> 10) & 0x1F, m = h & 0x3FF;
  return e == 0 ? (uint64_t)m : ((uint64_t)(1024 + m) << (e - 1));
}

// Each thread sums 8 adjacent columns over a slab of rows; slabs are added
// into colsum with 64-bit integer atomics (exact, order-independent).
constexpr int kSalRows = 256;
__global__ void saliency_kernel(const __half *__restrict__ W, int64_t N,
                                int64_t K, int64_t ldw,
                                unsigned long long *colsum) {
  const int64_t v = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const int64_t j0 = v * 8;
  if (j0 >= K) return;
  const int64_t i0 = (int64_t)blockIdx.y * kSalRows;
  const int64_t i1 = min(N, i0 + kSalRows);
  uint64_t acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int64_t i = i0; i < i1; ++i) {
    const uint4 d = __ldg(reinterpret_cast<const uint4 *>(W + i * ldw + j0));
    const uint16_t *h = reinterpret_cast<const uint16_t *>(&d);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] += fp16_units(h[e]);
  }
#pragma unroll
  for (int e = 0; e < 8; ++e)
    if (j0 + e < K && acc[e]) atomicAdd(colsum + j0 + e, (unsigned long long)acc[e]);
}

// ----------------------------------------------------------- selection ---
// score_j = fp64(colsum_j) * fp64(|x_profile_j|), one RN multiply.  Scores
// are >= +0, so their fp64 bit patterns order exactly like the values; the
// ranking compares them as unsigned integers.
__device__ __forceinline__ unsigned long long score_key(const int64_t *colsum,
                                                        const float *xp, int64_t j) {
  const double sc = __dmul_rn(__ll2double_rn(colsum[j]), (double)fabsf(xp[j]));
  return (unsigned long long)__double_as_longlong(sc);
}

// rank_j = #{i : s_i > s_j} + #{i < j : s_i == s_j}; channel j is an outlier
// iff rank_j < n_out.  The flag is parked in perm[j] for the next kernel.
constexpr int kSelThreads = 256;
__global__ void __launch_bounds__(kSelThreads)
    select_flag_kernel(const int64_t *__restrict__ colsum,
                       const float *__restrict__ xp, int64_t K, int64_t n_out,
                       int32_t *perm) {
  __shared__ unsigned long long tile[kSelThreads];
  const int64_t j = blockIdx.x * (int64_t)kSelThreads + threadIdx.x;
  const unsigned long long sj = j < K ? score_key(colsum, xp, j) : 0ull;
  int64_t rank = 0;
  for (int64_t base = 0; base < K; base += kSelThreads) {
    const int64_t i = base + threadIdx.x;
    tile[threadIdx.x] = i < K ? score_key(colsum, xp, i) : 0ull;
    __syncthreads();
    const int lim = (int)(K - base < kSelThreads ? K - base : kSelThreads);
    for (int t = 0; t < lim; ++t) {
      const unsigned long long si = tile[t];
      rank += (si > sj) || (si == sj && base + t < j);
    }
    __syncthreads();
  }
  if (j < K) perm[j] = rank < n_out ? 1 : 0;
}

// One CTA: outliers get positions 0..n_out-1 and the rest n_out..K-1, both in
// ascending channel order (an exclusive scan of the flags).
constexpr int kScanThreads = 1024;
__global__ void __launch_bounds__(kScanThreads)
    select_perm_kernel(int64_t K, int64_t n_out, int32_t *perm) {
  extern __shared__ uint32_t bits[];  // K flag bits
  __shared__ int32_t counts[kScanThreads];
  const int64_t words = (K + 31) / 32;
  for (int64_t w = threadIdx.x; w < words; w += kScanThreads) bits[w] = 0;
  __syncthreads();
  for (int64_t j = threadIdx.x; j < K; j += kScanThreads)
    if (perm[j]) atomicOr(&bits[j >> 5], 1u << (j & 31));
  __syncthreads();
  // thread t owns the contiguous range [lo, hi)
  const int64_t per = (K + kScanThreads - 1) / kScanThreads;
  const int64_t lo0 = (int64_t)threadIdx.x * per;
  const int64_t lo = lo0 < K ? lo0 : K, hi = lo + per < K ? lo + per : K;
  int32_t cnt = 0;
  for (int64_t j = lo; j < hi; ++j) cnt += (bits[j >> 5] >> (j & 31)) & 1;
  counts[threadIdx.x] = cnt;
  __syncthreads();
  // exclusive scan over 1024 counts (Hillis-Steele on a copy)
  for (int o = 1; o < kScanThreads; o <<= 1) {
    const int32_t add = threadIdx.x >= o ? counts[threadIdx.x - o] : 0;
    __syncthreads();
    counts[threadIdx.x] += add;
    __syncthreads();
  }
  int64_t outl_before = counts[threadIdx.x] - cnt;  // outliers in [0, lo)
  for (int64_t j = lo; j < hi; ++j) {
    const bool f = (bits[j >> 5] >> (j & 31)) & 1;
    const int64_t pos = f ? outl_before : n_out + (j - outl_before);
    perm[pos] = (int32_t)j;
    outl_before += f;
  }
}

// ----------------------------------------------------------- perm check --
__global__ void __launch_bounds__(1024)
    check_perm_kernel(const int32_t *__restrict__ perm, int64_t K, int32_t *flag) {
  extern __shared__ uint32_t seen[];
  __shared__ int bad_range, bad_dup;
  const int64_t words = (K + 31) / 32;
  if (threadIdx.x == 0) bad_range = bad_dup = 0;
  for (int64_t w = threadIdx.x; w < words; w += blockDim.x) seen[w] = 0;
  __syncthreads();
  for (int64_t t = threadIdx.x; t < K; t += blockDim.x) {
    const int32_t v = perm[t];
    if (v < 0 || v >= K) {
      bad_range = 1;
    } else {
      const uint32_t bit = 1u << (v & 31);
      if (atomicOr(&seen[v >> 5], bit) & bit) bad_dup = 1;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) *flag = bad_range ? 1 : (bad_dup ? 2 : 0);
}

// ----------------------------------------------------------- INT4 --------
// One CTA per row (grid-stride): the row is staged in shared memory, the
// outlier columns are copied bit-exactly, the background max is reduced,
// s_i = max/7, and codes are rounded, clamped and packed four bytes per
// thread.  All padding is written as zero.
constexpr int kQ4Threads = 256;
__global__ void __launch_bounds__(kQ4Threads)
    int4o_quant_kernel(const __half *__restrict__ W, int64_t ldw,
                       const int32_t *__restrict__ perm, int64_t N, int64_t K,
                       int64_t n_out, __half *__restrict__ w_out, int64_t ld_out,
                       uint8_t *__restrict__ q4, int64_t ld_q4,
                       float *__restrict__ scale) {
  extern __shared__ uint4 rowbuf4[];
  __shared__ uint32_t red[kQ4Threads / 32];
  const uint16_t *rowbuf = reinterpret_cast<const uint16_t *>(rowbuf4);
  const int64_t vpr = (K + 7) / 8;
  for (int64_t i = blockIdx.x; i < N; i += gridDim.x) {
    for (int64_t v = threadIdx.x; v < vpr; v += kQ4Threads)
      rowbuf4[v] = __ldg(reinterpret_cast<const uint4 *>(W + i * ldw) + v);
    __syncthreads();
    // outliers, bit-exact, zero padded to ld_out
    for (int64_t t = threadIdx.x; t < ld_out; t += kQ4Threads) {
      const uint16_t h = t < n_out ? rowbuf[__ldg(perm + t)] : (uint16_t)0;
      reinterpret_cast<uint16_t *>(w_out)[i * ld_out + t] = h;
    }
    // background max |W|
    uint32_t m = 0;
    for (int64_t t = n_out + threadIdx.x; t < K; t += kQ4Threads)
      m = max(m, abs_bits(rowbuf[__ldg(perm + t)]));
    m = warp_max_u32(m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    uint32_t mm = 0;
#pragma unroll
    for (int w = 0; w < kQ4Threads / 32; ++w) mm = max(mm, red[w]);
    const float amax = __half2float(__ushort_as_half((uint16_t)mm));
    const float s = __fdiv_rn(amax, 7.0f);
    // quantize + pack: thread handles bytes 4*v .. 4*v+3
    const int64_t kb = K - n_out;
    for (int64_t v = threadIdx.x; v < ld_q4 / 4; v += kQ4Threads) {
      uint32_t word = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int64_t tp = 8 * v + e;  // background element index
        int code = 0;
        if (tp < kb && s != 0.0f) {
          const float wv = __half2float(__ushort_as_half(rowbuf[__ldg(perm + n_out + tp)]));
          float r = rintf(__fdiv_rn(wv, s));
          r = fminf(fmaxf(r, -7.0f), 7.0f);
          code = (int)r;
        }
        word |= (uint32_t)(code & 0xF) << (4 * e);
      }
      reinterpret_cast<uint32_t *>(q4 + i * ld_q4)[v] = word;
    }
    if (threadIdx.x == 0) scale[i] = s;
    __syncthreads();  // rowbuf and red are reused by the next row
  }
}

int grid_for(int64_t work, int threads, int sms) {
  int64_t g = (work + threads - 1) / threads;
  const int64_t cap = (int64_t)sms * 8;
  if (g > cap) g = cap;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace

qz_status launch_quantize_int8(const __half *W, int64_t N, int64_t K, int64_t ldw,
                               int8_t *q, int64_t ldq, float *scale, cudaStream_t s) {
  DeviceInfo di;
  qz_status st = device_info(&di);
  if (st != QZ_OK) return st;
  cudaError_t e = cudaMemsetAsync(scale, 0, sizeof(float), s);
  if (e != cudaSuccess) return cuda_status(e);
  int_fast64_t vecs = N * ((K + 7) / 8);
  int8_absmax_kernel<<<grid_for(vecs, 256, di.sms), 256, 0, s>>>(
      W, N, K, ldw, reinterpret_cast<unsigned int *>(scale));
  if ((st = launch_status()) != QZ_OK) return st;
  int8_quant_kernel<<<grid_for(N * (ldq / 16), 256, di.sms), 256, 0, s>>>(
      W, N, K, ldw, q, ldq, scale);
  if ((st = launch_status()) != QZ_OK) return st;
  int8_scale_kernel<<<1, 1, 0, s>>>(scale);
  return launch_status();
}

qz_status launch_saliency(const __half *W, int64_t N, int64_t K, int64_t ldw,
                          int64_t *colsum, cudaStream_t s) {
  const int64_t vecs = (K + 7) / 8;
  dim3 grid((unsigned)((vecs + 127) / 128), (unsigned)((N + kSalRows - 1) / kSalRows));
  saliency_kernel<<<grid, 128, 0, s>>>(W, N, K, ldw,
                                       reinterpret_cast<unsigned long long *>(colsum));
  return launch_status();
}

qz_status launch_select(const int64_t *colsum, const float *xprof, int64_t K,
                        int64_t n_out, int32_t *perm, cudaStream_t s) {
  select_flag_kernel<<<(unsigned)((K + kSelThreads - 1) / kSelThreads), kSelThreads, 0, s>>>(
      colsum, xprof, K, n_out, perm);
  qz_status st = launch_status();
  if (st != QZ_OK) return st;
  const size_t smem = (size_t)((K + 31) / 32) * 4;
  cudaError_t e = cudaFuncSetAttribute(select_perm_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_status(e);
  select_perm_kernel<<<1, kScanThreads, smem, s>>>(K, n_out, perm);
  return launch_status();
}

qz_status launch_check_perm(const int32_t *perm, int64_t K, int32_t *flag, cudaStream_t s) {
  const size_t smem = (size_t)((K + 31) / 32) * 4;
  cudaError_t e = cudaFuncSetAttribute(check_perm_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_status(e);
  check_perm_kernel<<<1, 1024, smem, s>>>(perm, K, flag);
  return launch_status();
}

qz_status launch_quantize_int4o(const __half *W, int64_t ldw, const int32_t *perm,
                                int64_t N, int64_t K, int64_t n_out, __half *w_out,
                                int64_t ld_out, uint8_t *q4, int64_t ld_q4, float *scale,
                                cudaStream_t s) {
  DeviceInfo di;
  qz_status st = device_info(&di);
  if (st != QZ_OK) return st;
  const size_t smem = (size_t)((K + 7) / 8) * 16;
  if (smem > (size_t)di.max_smem_optin) return QZ_ERR_UNSUPPORTED;
  cudaError_t e = cudaFuncSetAttribute(int4o_quant_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_status(e);
  int64_t grid = N < (int64_t)di.sms * 8 ? N : (int64_t)di.sms * 8;
  int4o_quant_kernel<<<(unsigned)grid, kQ4Threads, smem, s>>>(W, ldw, perm, N, K, n_out,
                                                              w_out, ld_out, q4, ld_q4, scale);
  return launch_status();
}

}  // namespace qz
