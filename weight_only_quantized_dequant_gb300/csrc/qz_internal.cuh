// Internal declarations shared by the translation units of libqz.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/qz.h"

namespace qz {

// ---------------------------------------------------------------- errors --
// Record a CUDA error for qz_last_cuda_error() and map it to a status.
qz_status cuda_status(cudaError_t e);
// cudaGetLastError() after a launch, mapped to a status.
inline qz_status launch_status() { return cuda_status(cudaGetLastError()); }

// Per-device facts, cached on first use (current device).
struct DeviceInfo {
  int sms = 0;
  int max_smem_optin = 0;  // bytes of dynamic shared memory one CTA may use
};
qz_status device_info(DeviceInfo *out);

// ------------------------------------------------------------ GEMV (CUDA cores)
// One launch reads up to QZ_MAX_GROUP matrices that share the input.
// Row r of the launch belongs to matrix m with row_end[m-1] <= r < row_end[m].
struct GemvParams {
  const __half *x;  // [B][ldx], original channel order
  int64_t ldx;
  const int32_t *perm;  // INT4 only: [K]
  int K, n_out, kb;     // INT8: n_out = 0, kb = K
  int cpr;              // 16-byte chunks per row of the code array that hold data
  int ocpr;             // 16-byte chunks per row of w_out that hold data (INT4)
  int n_mats;
  int64_t total_rows;
  int64_t row_end[QZ_MAX_GROUP];
  const uint8_t *codes[QZ_MAX_GROUP];  // int8 codes or packed nibbles
  int64_t ld_codes[QZ_MAX_GROUP];      // bytes between rows
  const __half *w_out[QZ_MAX_GROUP];   // INT4 outlier block
  int64_t ld_out[QZ_MAX_GROUP];        // halves between rows
  const float *scale[QZ_MAX_GROUP];    // INT8: [1]; INT4: [N]
  __half *y[QZ_MAX_GROUP];             // [B][ldy]
  int64_t ldy[QZ_MAX_GROUP];          // row stride of each y
  int overlap;  // programmatic dependent launch + weight prefetch before the wait
};

// Up to QZ_MAX_SEQ dependent batch-1 products in one launch (grid barrier
// between products on the counter *sync, which starts and ends at 0).
struct SeqParams {
  GemvParams t[QZ_MAX_SEQ];
  int n;
  unsigned int *sync;
  uint32_t xs_bytes;  // shared bytes reserved for the staged input (set by the launcher)
};
qz_status launch_gemv_seq(bool int4, SeqParams &sp, cudaStream_t s);

// Per-host-thread launch option set by qz_set_overlap().
int overlap_enabled();

// Shared-memory bytes the CUDA-core kernel needs for batch B.
size_t gemv_smem_bytes(bool int4, int B, const GemvParams &p);
// Enqueue the CUDA-core GEMV for batch 1 <= B <= 4.
qz_status launch_gemv(bool int4, int B, const GemvParams &p, cudaStream_t s);
// Batch-1 CUDA-core GEMV reading the weights in place, where they may lie in
// mapped pinned host memory (zero-copy); its shared-memory bytes.
qz_status launch_gemv_mapped(bool int4, const GemvParams &p, cudaStream_t s);
size_t gemv_mapped_smem_bytes(bool int4, const GemvParams &p);

// Warp-MMA GEMV (mma.sync on dequantized codes) for batch 1..kMvMaxBatch.
constexpr int kMvMaxBatch = 8;
struct MvProduct {  // shapes of the product, chosen by the host
  int Ko, Kb;         // 64-byte K blocks per row: outliers (INT4), codes
  int nst, skc;       // ring stages per 16-row tile, K blocks per stage
  uint32_t pitch;     // bytes between the rows of a stage
  uint32_t bstride;   // staged input bytes per batch row (codes' inputs)
  uint32_t ostride;   // staged outlier-input bytes per batch row
  uint32_t rawstride; // contiguous input bytes per batch row (raw)
  int raw;            // INT4: input copied to shared memory, then gathered
};
struct MvLaunch {
  GemvParams t;
  MvProduct pr;
  int B;
  int tp;                // 16-row tiles per ring stage (1 or 2)
  int ns;                // ring stages
  int early;             // stages issued before the input is staged
  uint32_t slot_bytes;   // bytes of one ring stage
  uint32_t xo_off, raw_off, ring_off, bar_off, part_off, cnt_off;  // shared-memory offsets
};
// Whether a batch-B product fits the kernel's shared memory.
bool mv_fits(bool int4, int B, const GemvParams &p);
qz_status launch_mv(bool int4, int B, const GemvParams &p, cudaStream_t s);
qz_status read_mv_error(int *code, int clear);

// Tensor-core (tcgen05) GEMM for any batch 1..64; rows of each matrix are
// p.row_end differences.
size_t tc_smem_bytes(bool int4, int Np);
size_t tc_workspace_bytes(bool int4, int64_t B, int64_t K, int64_t n_out);
qz_status launch_tc(bool int4, int B, const GemvParams &p, const int64_t *mat_rows,
                    void *workspace, size_t workspace_bytes, cudaStream_t s);
qz_status read_device_error(int *code, int clear);
qz_status read_gemv_error(int *code, int clear);
qz_status read_embed_error(int *code, int clear);

// INT8 vocabulary-table lookup (rows of q reconstructed to fp16).
qz_status launch_embed_int8(const int8_t *q, int64_t ldq, const float *scale, int64_t V, int64_t K,
                            const int32_t *tokens, int64_t B, __half *out, int64_t ldo,
                            cudaStream_t s);

// ------------------------------------------------------------ quantizers ---
qz_status launch_quantize_int8(const __half *W, int64_t N, int64_t K,
                               int64_t ldw, int8_t *q, int64_t ldq,
                               float *scale, cudaStream_t s);
qz_status launch_saliency(const __half *W, int64_t N, int64_t K, int64_t ldw,
                          int64_t *colsum, cudaStream_t s);
qz_status launch_select(const int64_t *colsum, const float *xprof, int64_t K,
                        int64_t n_out, int32_t *perm, cudaStream_t s);
qz_status launch_check_perm(const int32_t *perm, int64_t K, int32_t *flag,
                            cudaStream_t s);
qz_status launch_quantize_int4o(const __half *W, int64_t ldw,
                                const int32_t *perm, int64_t N, int64_t K,
                                int64_t n_out, __half *w_out, int64_t ld_out,
                                uint8_t *q4, int64_t ld_q4, float *scale,
                                cudaStream_t s);

}  // namespace qz
