// Lookup of rows of an INT8 vocabulary table, reconstructed to fp16.
//
// "On-The-Fly Weight Synthesizer (OTF-LLM Engine)", key innovation 4 keeps the
// vocabulary table (embed_tokens) in INT8; a looked-up row is reconstructed
// as in "Open Origin - ELG Stream Layer", FP16 On-The-Fly GPU Reconstruction:
// out[b][j] = fp16(q[tokens[b]][j] * scale).  The product of the 8-bit code
// and the fp32 scale is rounded once, to the nearest fp16 (ties to even):
// the fp32 product is taken toward zero and its sticky bit (whether the
// remainder, exact by FMA, is nonzero) is forced into the last bit, i.e.
// rounding to odd, which makes the later fp32 -> fp16 rounding correct
// (Boldo and Melquiond, "Emulation of FMA and correctly rounded sums: proved
// algorithms using rounding to odd", IEEE Trans. Computers 57(4), 2008:
// round-to-odd at p + 2 or more bits followed by round-to-nearest at p bits
// equals one round-to-nearest; here 24 >= 11 + 2).
//
// The row is a contiguous run of K bytes (HBM-bound, a few KB per token):
// each thread converts 8 codes, one 8-byte load and one 16-byte store.
#include "qz_internal.cuh"

namespace qz {
namespace {

constexpr int kEmbedThreads = 128;

__device__ int g_embed_error = 0;  // 2 if a token lay outside the table (qz_device_error)

__device__ __forceinline__ uint32_t round_once_bits(int q, float s) {
  const float qf = (float)q;
  const float p = __fmul_rz(qf, s);        // truncated product
  const float e = __fmaf_rn(qf, s, -p);    // exact remainder q*s - p
  uint32_t b = __float_as_uint(p);
  if (e != 0.0f) b |= 1u;                  // round to odd
  return (uint32_t)__half_as_ushort(__float2half_rn(__uint_as_float(b)));
}

__global__ void __launch_bounds__(kEmbedThreads)
    embed_int8_kernel(const int8_t *__restrict__ q, int64_t ldq, const float *__restrict__ scale,
                      int64_t V, int64_t K, const int32_t *__restrict__ tokens, int64_t B,
                      __half *__restrict__ out, int64_t ldo) {
  const int64_t j0 = ((int64_t)blockIdx.x * kEmbedThreads + threadIdx.x) * 8;
  const float s = __ldg(scale);
  for (int64_t b = blockIdx.y; b < B; b += gridDim.y) {
    const int32_t t = __ldg(tokens + b);
    const bool valid = t >= 0 && (int64_t)t < V;
    if (!valid && blockIdx.x == 0 && threadIdx.x == 0) atomicOr(&g_embed_error, 2);
    if (j0 >= K) continue;
    const int8_t *row = q + (valid ? (int64_t)t : 0) * ldq + j0;
    __half *o = out + b * ldo + j0;
    if (j0 + 8 <= K) {
      uint2 v = make_uint2(0, 0);
      if (valid) v = __ldg(reinterpret_cast<const uint2 *>(row));  // ldq % 16 == 0
      uint32_t h[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t w = k < 2 ? v.x : v.y;
        const int sh = (k & 1) * 16;
        const int q0 = (int)(int8_t)((w >> sh) & 0xFFu);
        const int q1 = (int)(int8_t)((w >> (sh + 8)) & 0xFFu);
        h[k] = round_once_bits(q0, s) | (round_once_bits(q1, s) << 16);
      }
      *reinterpret_cast<uint4 *>(o) = make_uint4(h[0], h[1], h[2], h[3]);  // ldo % 8 == 0
    } else {
      for (int64_t j = 0; j < K - j0; ++j)
        o[j] = __ushort_as_half((unsigned short)round_once_bits(valid ? row[j] : 0, s));
    }
  }
}

}  // namespace

qz_status launch_embed_int8(const int8_t *q, int64_t ldq, const float *scale, int64_t V, int64_t K,
                            const int32_t *tokens, int64_t B, __half *out, int64_t ldo,
                            cudaStream_t s) {
  if (B == 0) return QZ_OK;
  const int64_t per_block = (int64_t)kEmbedThreads * 8;
  const int64_t gx = (K + per_block - 1) / per_block;
  const int64_t gy = B < 65535 ? B : 65535;
  embed_int8_kernel<<<dim3((unsigned)gx, (unsigned)gy), kEmbedThreads, 0, s>>>(q, ldq, scale, V, K,
                                                                              tokens, B, out, ldo);
  return launch_status();
}

qz_status read_embed_error(int *code, int clear) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_embed_error, sizeof(int));
  if (e != cudaSuccess) return cuda_status(e);
  if (clear && v) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_embed_error, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_status(e);
  }
  *code = v;
  return QZ_OK;
}

}  // namespace qz
