// extern "C" entry points of libqz: argument validation, then one launcher.
// Validation never touches the GPU, so an invalid call enqueues nothing.
#include <mutex>

#include <cstring>

#include "qz_internal.cuh"

namespace qz {

static thread_local int g_last_cuda_error = 0;
static thread_local int g_overlap = 0;

int overlap_enabled() { return g_overlap; }

qz_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return QZ_OK;
  g_last_cuda_error = (int)e;
  return QZ_ERR_CUDA;
}

qz_status device_info(DeviceInfo *out) {
  constexpr int kMaxDev = 64;
  static DeviceInfo cache[kMaxDev];
  static std::once_flag once[kMaxDev];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e);
  if (dev < 0 || dev >= kMaxDev) return QZ_ERR_UNSUPPORTED;
  cudaError_t err = cudaSuccess;
  std::call_once(once[dev], [&] {
    DeviceInfo d;
    err = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (err == cudaSuccess)
      err = cudaDeviceGetAttribute(&d.max_smem_optin,
                                   cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cache[dev] = d;
  });
  if (err != cudaSuccess) return cuda_status(err);
  if (cache[dev].sms <= 0) return QZ_ERR_CUDA;
  *out = cache[dev];
  return QZ_OK;
}

namespace {

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Shared checks of a matrix argument: non-null, 16-B aligned, rows of
// ld*elem bytes that are a multiple of 16, ld >= cols.
qz_status check_mat(const void *p, int64_t rows, int64_t cols, int64_t ld, int elem) {
  if (!p || rows < 1 || cols < 1 || ld < cols) return QZ_ERR_INVALID_ARG;
  if (!aligned16(p) || (ld * elem) % 16 != 0) return QZ_ERR_ALIGNMENT;
  return QZ_OK;
}

#define QZ_TRY(expr)               \
  do {                             \
    qz_status _st = (expr);        \
    if (_st != QZ_OK) return _st;  \
  } while (0)

constexpr int64_t kMaxGemvK = 57344;

qz_status check_int8_weight(const qz_int8_weight *w) {
  if (!w) return QZ_ERR_INVALID_ARG;
  QZ_TRY(check_mat(w->q, w->N, w->K, w->ldq, 1));
  if (!w->scale) return QZ_ERR_INVALID_ARG;
  if (w->K > kMaxGemvK || w->N > ((int64_t)1 << 30)) return QZ_ERR_UNSUPPORTED;
  return QZ_OK;
}

qz_status check_int4o_weight(const qz_int4o_weight *w) {
  if (!w) return QZ_ERR_INVALID_ARG;
  if (w->N < 1 || w->K < 1 || w->n_out < 0 || w->n_out > w->K) return QZ_ERR_INVALID_ARG;
  const int64_t kb = w->K - w->n_out;
  if (!w->perm || !w->scale) return QZ_ERR_INVALID_ARG;
  if (w->n_out > 0 && !w->w_out) return QZ_ERR_INVALID_ARG;
  if (kb > 0 && !w->q4) return QZ_ERR_INVALID_ARG;
  if (w->ld_out < w->n_out || w->ld_q4 < (kb + 1) / 2) return QZ_ERR_INVALID_ARG;
  if (w->ld_out % 8 || w->ld_q4 % 16) return QZ_ERR_ALIGNMENT;
  if ((w->w_out && !aligned16(w->w_out)) || (w->q4 && !aligned16(w->q4)) ||
      !aligned16(w->scale) || !aligned16(w->perm))
    return QZ_ERR_ALIGNMENT;
  if (w->K > kMaxGemvK || w->N > ((int64_t)1 << 30)) return QZ_ERR_UNSUPPORTED;
  return QZ_OK;
}

// Activation/output vectors are read and written one element at a time, so
// they only need the 2-byte alignment of fp16.
qz_status check_vec(const void *x, int64_t B, int64_t len, int64_t ld) {
  if (!x || B < 1 || len < 1 || (B > 1 && ld < len)) return QZ_ERR_INVALID_ARG;
  if ((uintptr_t)x & 1u) return QZ_ERR_ALIGNMENT;
  return QZ_OK;
}

// Fill the per-matrix part of the launch for INT8.
void fill_int8(GemvParams &p, const qz_int8_weight *ws, int n) {
  p.perm = nullptr;
  p.K = (int)ws[0].K;
  p.n_out = 0;
  p.kb = p.K;
  p.cpr = (int)((ws[0].K + 15) / 16);
  p.ocpr = 0;
  p.n_mats = n;
  int64_t rows = 0;
  for (int m = 0; m < QZ_MAX_GROUP; ++m) {
    if (m < n) {
      rows += ws[m].N;
      p.codes[m] = reinterpret_cast<const uint8_t *>(ws[m].q);
      p.ld_codes[m] = ws[m].ldq;
      p.scale[m] = ws[m].scale;
    } else {
      p.codes[m] = nullptr;
      p.ld_codes[m] = 0;
      p.scale[m] = nullptr;
    }
    p.w_out[m] = nullptr;
    p.ld_out[m] = 0;
    p.row_end[m] = rows;
    p.y[m] = nullptr;
  }
  p.total_rows = rows;
}

void fill_int4o(GemvParams &p, const qz_int4o_weight *ws, int n) {
  p.perm = ws[0].perm;
  p.K = (int)ws[0].K;
  p.n_out = (int)ws[0].n_out;
  p.kb = p.K - p.n_out;
  p.cpr = (int)(((p.kb + 1) / 2 + 15) / 16);
  p.ocpr = (p.n_out + 7) / 8;
  p.n_mats = n;
  int64_t rows = 0;
  for (int m = 0; m < QZ_MAX_GROUP; ++m) {
    if (m < n) {
      rows += ws[m].N;
      p.codes[m] = ws[m].q4;
      p.ld_codes[m] = ws[m].ld_q4;
      p.w_out[m] = reinterpret_cast<const __half *>(ws[m].w_out);
      p.ld_out[m] = ws[m].ld_out;
      p.scale[m] = ws[m].scale;
    } else {
      p.codes[m] = nullptr;
      p.ld_codes[m] = 0;
      p.w_out[m] = nullptr;
      p.ld_out[m] = 0;
      p.scale[m] = nullptr;
    }
    p.row_end[m] = rows;
    p.y[m] = nullptr;
  }
  p.total_rows = rows;
}

qz_status gemm_common(bool int4, GemvParams &p, int64_t B, const qz_half *X, int64_t ldx,
                      qz_half *const *Ys, const int64_t *ldys, int n, void *ws, size_t ws_bytes,
                      cudaStream_t s) {
  p.x = reinterpret_cast<const __half *>(X);
  p.overlap = overlap_enabled();
  p.ldx = B > 1 ? ldx : 0;
  for (int m = 0; m < QZ_MAX_GROUP; ++m) p.ldy[m] = (B > 1 && m < n) ? ldys[m] : 0;
  for (int m = 0; m < n; ++m) p.y[m] = reinterpret_cast<__half *>(Ys[m]);
  DeviceInfo di;
  QZ_TRY(device_info(&di));
  // a workspace, when given, is checked whatever path the call then takes
  if (ws) {
    if (ws_bytes < tc_workspace_bytes(int4, B, p.K, p.n_out)) return QZ_ERR_INVALID_ARG;
    if ((uintptr_t)ws & 15u) return QZ_ERR_ALIGNMENT;
  }
  // Batch 1 runs on the CUDA-core GEMV (one fp32 FMA per weight keeps pace
  // with HBM at one input row); batches 2..8 on the warp-MMA GEMV, where the
  // CUDA cores would need one FMA per weight and input row.  Either takes
  // the call when its staged inputs fit in shared memory; larger batches are
  // dense enough for the tcgen05 GEMM, which also takes the small batches at
  // the few K too large to stage (its inputs stream in tiles).
  if (B == 1 && gemv_smem_bytes(int4, 1, p) <= (size_t)di.max_smem_optin)
    return launch_gemv(int4, 1, p, s);
  if (B <= kMvMaxBatch && mv_fits(int4, (int)B, p)) return launch_mv(int4, (int)B, p, s);
  if (B <= 4 && gemv_smem_bytes(int4, (int)B, p) <= (size_t)di.max_smem_optin)
    return launch_gemv(int4, (int)B, p, s);
  int64_t rows[QZ_MAX_GROUP];
  for (int m = 0; m < QZ_MAX_GROUP; ++m)
    rows[m] = m < n ? p.row_end[m] - (m ? p.row_end[m - 1] : 0) : 0;
  return launch_tc(int4, (int)B, p, rows, ws, ws_bytes, s);
}

template <typename W, typename Fill, typename Check>
qz_status sequence_common(bool int4, const W *ws, const int *counts, int n,
                          const qz_half *const *x, qz_half *const *ys, uint32_t *sync,
                          cudaStream_t s, Fill fill, Check check) {
  if (!ws || !counts || !x || !ys || !sync || n < 1) return QZ_ERR_INVALID_ARG;
  if (n > QZ_MAX_SEQ) return QZ_ERR_UNSUPPORTED;
  if (((uintptr_t)sync & 3u) != 0) return QZ_ERR_ALIGNMENT;
  SeqParams sp;
  memset(&sp, 0, sizeof(sp));
  int off = 0;
  for (int k = 0; k < n; ++k) {
    const int c = counts[k];
    if (c < 1) return QZ_ERR_INVALID_ARG;
    if (c > QZ_MAX_GROUP) return QZ_ERR_UNSUPPORTED;
    for (int m = 0; m < c; ++m) {
      QZ_TRY(check(ws[off + m], ws[off]));
      QZ_TRY(check_vec(ys[off + m], 1, ws[off + m].N, 0));
    }
    QZ_TRY(check_vec(x[k], 1, ws[off].K, 0));
    GemvParams &p = sp.t[k];
    fill(p, ws + off, c);
    p.x = reinterpret_cast<const __half *>(x[k]);
    p.ldx = 0;
    p.overlap = overlap_enabled();
    for (int m = 0; m < QZ_MAX_GROUP; ++m) p.ldy[m] = 0;
    for (int m = 0; m < c; ++m) p.y[m] = reinterpret_cast<__half *>(ys[off + m]);
    off += c;
  }
  sp.n = n;
  sp.sync = reinterpret_cast<unsigned int *>(sync);
  return launch_gemv_seq(int4, sp, s);
}
// The address under which the device reads a weight buffer in place: device
// memory, or host memory that is pinned and mapped (unified addressing).
// Pageable or unknown memory is refused, so nothing is launched on it.
qz_status device_view(const void *ptr, const void **dev) {
  if (!ptr) {
    *dev = nullptr;
    return QZ_OK;
  }
  cudaPointerAttributes a;
  const cudaError_t e = cudaPointerGetAttributes(&a, ptr);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return QZ_ERR_INVALID_ARG;
  }
  if (a.type == cudaMemoryTypeUnregistered || !a.devicePointer) return QZ_ERR_INVALID_ARG;
  *dev = a.devicePointer;
  return QZ_OK;
}

template <typename T>
qz_status device_view_t(T *&ptr) {
  const void *d = nullptr;
  QZ_TRY(device_view(ptr, &d));
  ptr = reinterpret_cast<T *>(const_cast<void *>(d));
  return QZ_OK;
}

// Batch-1 grouped product with the weights read in place (zero-copy).
qz_status mapped_common(bool int4, GemvParams &p, const qz_half *x, qz_half *const *ys, int n,
                        cudaStream_t s) {
  p.x = reinterpret_cast<const __half *>(x);
  p.overlap = overlap_enabled();
  p.ldx = 0;
  for (int m = 0; m < QZ_MAX_GROUP; ++m) p.ldy[m] = 0;
  for (int m = 0; m < n; ++m) p.y[m] = reinterpret_cast<__half *>(ys[m]);
  DeviceInfo di;
  QZ_TRY(device_info(&di));
  if (gemv_mapped_smem_bytes(int4, p) > (size_t)di.max_smem_optin) return QZ_ERR_UNSUPPORTED;
  return launch_gemv_mapped(int4, p, s);
}

}  // namespace
}  // namespace qz

using namespace qz;

extern "C" {

const char *qz_status_string(qz_status st) {
  switch (st) {
    case QZ_OK: return "QZ_OK";
    case QZ_ERR_INVALID_ARG: return "QZ_ERR_INVALID_ARG";
    case QZ_ERR_ALIGNMENT: return "QZ_ERR_ALIGNMENT";
    case QZ_ERR_UNSUPPORTED: return "QZ_ERR_UNSUPPORTED";
    case QZ_ERR_CUDA: return "QZ_ERR_CUDA";
    case QZ_ERR_IO: return "QZ_ERR_IO";
    case QZ_ERR_DATA: return "QZ_ERR_DATA";
  }
  return "QZ_ERR_UNKNOWN";
}

int qz_version(void) { return 1 * 10000 + 0 * 100 + 0; }

int qz_last_cuda_error(void) { return g_last_cuda_error; }

qz_status qz_set_overlap(int enable) {
  if (enable != 0 && enable != 1) return QZ_ERR_INVALID_ARG;
  g_overlap = enable;
  return QZ_OK;
}

int qz_get_overlap(void) { return g_overlap; }

qz_status qz_device_error(int *code, int clear) {
  if (!code || (clear != 0 && clear != 1)) return QZ_ERR_INVALID_ARG;
  int a = 0, b = 0, c = 0, d = 0;
  QZ_TRY(read_device_error(&a, clear));
  QZ_TRY(read_gemv_error(&b, clear));
  QZ_TRY(read_embed_error(&c, clear));
  QZ_TRY(read_mv_error(&d, clear));
  *code = a | b | c | d;
  return QZ_OK;
}

// ------------------------------------------------------------------ INT8 --
qz_status qz_quantize_int8(const qz_half *W, int64_t N, int64_t K, int64_t ldw, int8_t *q,
                           int64_t ldq, float *scale, qz_stream s) {
  QZ_TRY(check_mat(W, N, K, ldw, 2));
  QZ_TRY(check_mat(q, N, K, ldq, 1));
  if (!scale) return QZ_ERR_INVALID_ARG;
  if (((uintptr_t)scale & 3u) != 0) return QZ_ERR_ALIGNMENT;
  return launch_quantize_int8(reinterpret_cast<const __half *>(W), N, K, ldw, q, ldq, scale,
                              (cudaStream_t)s);
}

qz_status qz_gemv_int8(const qz_int8_weight *w, const qz_half *x, qz_half *y, qz_stream s) {
  return qz_gemm_int8(w, 1, x, 0, y, 0, nullptr, 0, s);
}

qz_status qz_gemm_int8(const qz_int8_weight *w, int64_t B, const qz_half *X, int64_t ldx,
                       qz_half *Y, int64_t ldy, void *workspace, size_t workspace_bytes,
                       qz_stream s) {
  QZ_TRY(check_int8_weight(w));
  if (B < 1) return QZ_ERR_INVALID_ARG;
  if (B > QZ_MAX_BATCH) return QZ_ERR_UNSUPPORTED;
  QZ_TRY(check_vec(X, B, w->K, ldx));
  QZ_TRY(check_vec(Y, B, w->N, ldy));
  GemvParams p;
  fill_int8(p, w, 1);
  qz_half *ys[1] = {Y};
  return gemm_common(false, p, B, X, ldx, ys, &ldy, 1, workspace, workspace_bytes,
                     (cudaStream_t)s);
}

qz_status qz_embed_int8(const qz_int8_weight *table, const int32_t *tokens, int64_t B,
                        qz_half *out, int64_t ldo, qz_stream s) {
  if (!table || B < 0) return QZ_ERR_INVALID_ARG;
  QZ_TRY(check_mat(table->q, table->N, table->K, table->ldq, 1));
  if (!table->scale) return QZ_ERR_INVALID_ARG;
  if (B == 0) return QZ_OK;
  if (!tokens) return QZ_ERR_INVALID_ARG;
  if (((uintptr_t)tokens & 3u) != 0) return QZ_ERR_ALIGNMENT;
  QZ_TRY(check_mat(out, B, table->K, ldo, 2));
  return launch_embed_int8(table->q, table->ldq, table->scale, table->N, table->K, tokens, B,
                           reinterpret_cast<__half *>(out), ldo, (cudaStream_t)s);
}

qz_status qz_gemv_int8_grouped(const qz_int8_weight *ws, int n, const qz_half *x,
                               qz_half *const *ys, qz_stream s) {
  if (!ws || !ys || n < 1) return QZ_ERR_INVALID_ARG;
  if (n > QZ_MAX_GROUP) return QZ_ERR_UNSUPPORTED;
  for (int m = 0; m < n; ++m) {
    QZ_TRY(check_int8_weight(&ws[m]));
    if (ws[m].K != ws[0].K) return QZ_ERR_INVALID_ARG;
    QZ_TRY(check_vec(ys[m], 1, ws[m].N, 0));
  }
  QZ_TRY(check_vec(x, 1, ws[0].K, 0));
  GemvParams p;
  fill_int8(p, ws, n);
  return gemm_common(false, p, 1, x, 0, ys, nullptr, n, nullptr, 0, (cudaStream_t)s);
}

qz_status qz_gemm_int8_grouped(const qz_int8_weight *ws, int n, int64_t B, const qz_half *X,
                               int64_t ldx, qz_half *const *Ys, const int64_t *ldys,
                               void *workspace, size_t workspace_bytes, qz_stream s) {
  if (!ws || !Ys || !ldys || n < 1 || B < 1) return QZ_ERR_INVALID_ARG;
  if (n > QZ_MAX_GROUP || B > QZ_MAX_BATCH) return QZ_ERR_UNSUPPORTED;
  for (int m = 0; m < n; ++m) {
    QZ_TRY(check_int8_weight(&ws[m]));
    if (ws[m].K != ws[0].K) return QZ_ERR_INVALID_ARG;
    QZ_TRY(check_vec(Ys[m], B, ws[m].N, ldys[m]));
  }
  QZ_TRY(check_vec(X, B, ws[0].K, ldx));
  GemvParams p;
  fill_int8(p, ws, n);
  return gemm_common(false, p, B, X, ldx, Ys, ldys, n, workspace, workspace_bytes,
                     (cudaStream_t)s);
}

size_t qz_gemm_workspace_bytes(int64_t B, int64_t K, int64_t n_out) {
  if (B < 1 || B > QZ_MAX_BATCH || K < 1 || n_out < 0 || n_out > K) return 0;
  // n_out = 0 gives the INT8 size (ceil(K/64) tiles of the gathered input)
  return tc_workspace_bytes(true, B, K, n_out);
}

// ------------------------------------------------------------------ INT4 --
qz_status qz_int4o_layout(int64_t N, int64_t K, int64_t n_out, int64_t *ld_out,
                          int64_t *ld_q4) {
  if (N < 1 || K < 1 || n_out < 0 || n_out > K || !ld_out || !ld_q4) return QZ_ERR_INVALID_ARG;
  const int64_t kb = K - n_out;
  *ld_out = (n_out + 7) / 8 * 8;
  *ld_q4 = ((kb + 1) / 2 + 15) / 16 * 16;
  return QZ_OK;
}

qz_status qz_saliency_accumulate(const qz_half *W, int64_t N, int64_t K, int64_t ldw,
                                 int64_t *colsum, qz_stream s) {
  QZ_TRY(check_mat(W, N, K, ldw, 2));
  if (!colsum) return QZ_ERR_INVALID_ARG;
  if (((uintptr_t)colsum & 7u) != 0) return QZ_ERR_ALIGNMENT;
  if (N > (int64_t)65535 * 256) return QZ_ERR_UNSUPPORTED;
  return launch_saliency(reinterpret_cast<const __half *>(W), N, K, ldw, colsum,
                         (cudaStream_t)s);
}

qz_status qz_select_outliers(const int64_t *colsum, const float *x_profile, int64_t K,
                             int64_t n_out, int32_t *perm, qz_stream s) {
  if (!colsum || !x_profile || !perm || K < 1 || n_out < 0 || n_out > K)
    return QZ_ERR_INVALID_ARG;
  if (((uintptr_t)colsum & 7u) || ((uintptr_t)x_profile & 3u) || ((uintptr_t)perm & 3u))
    return QZ_ERR_ALIGNMENT;
  if (K > ((int64_t)1 << 20)) return QZ_ERR_UNSUPPORTED;
  return launch_select(colsum, x_profile, K, n_out, perm, (cudaStream_t)s);
}

qz_status qz_check_perm(const int32_t *perm, int64_t K, int32_t *flag, qz_stream s) {
  if (!perm || !flag || K < 1) return QZ_ERR_INVALID_ARG;
  if (((uintptr_t)perm & 3u) || ((uintptr_t)flag & 3u)) return QZ_ERR_ALIGNMENT;
  if (K > ((int64_t)1 << 20)) return QZ_ERR_UNSUPPORTED;
  return launch_check_perm(perm, K, flag, (cudaStream_t)s);
}

qz_status qz_quantize_int4_outlier(const qz_half *W, int64_t ldw, const int32_t *perm,
                                   int64_t N, int64_t K, int64_t n_out, qz_half *w_out,
                                   int64_t ld_out, uint8_t *q4, int64_t ld_q4, float *scale,
                                   qz_stream s) {
  QZ_TRY(check_mat(W, N, K, ldw, 2));
  if (!perm || !scale || n_out < 0 || n_out > K) return QZ_ERR_INVALID_ARG;
  const int64_t kb = K - n_out;
  if ((n_out > 0 && !w_out) || (kb > 0 && !q4)) return QZ_ERR_INVALID_ARG;
  if (ld_out < n_out || ld_q4 < (kb + 1) / 2) return QZ_ERR_INVALID_ARG;
  if (ld_out % 8 || ld_q4 % 16 || (w_out && !aligned16(w_out)) || (q4 && !aligned16(q4)) ||
      ((uintptr_t)perm & 3u) || ((uintptr_t)scale & 3u))
    return QZ_ERR_ALIGNMENT;
  if ((ld_out > 0 && !w_out) || (ld_q4 > 0 && !q4)) return QZ_ERR_INVALID_ARG;
  if (K > ((int64_t)1 << 17)) return QZ_ERR_UNSUPPORTED;
  return launch_quantize_int4o(reinterpret_cast<const __half *>(W), ldw, perm, N, K, n_out,
                               reinterpret_cast<__half *>(w_out), ld_out, q4, ld_q4, scale,
                               (cudaStream_t)s);
}

qz_status qz_gemv_int4_outlier(const qz_int4o_weight *w, const qz_half *x, qz_half *y,
                               qz_stream s) {
  return qz_gemm_int4_outlier(w, 1, x, 0, y, 0, nullptr, 0, s);
}

qz_status qz_gemm_int4_outlier(const qz_int4o_weight *w, int64_t B, const qz_half *X,
                               int64_t ldx, qz_half *Y, int64_t ldy, void *workspace,
                               size_t workspace_bytes, qz_stream s) {
  QZ_TRY(check_int4o_weight(w));
  if (B < 1) return QZ_ERR_INVALID_ARG;
  if (B > QZ_MAX_BATCH) return QZ_ERR_UNSUPPORTED;
  QZ_TRY(check_vec(X, B, w->K, ldx));
  QZ_TRY(check_vec(Y, B, w->N, ldy));
  GemvParams p;
  fill_int4o(p, w, 1);
  qz_half *ys[1] = {Y};
  return gemm_common(true, p, B, X, ldx, ys, &ldy, 1, workspace, workspace_bytes,
                     (cudaStream_t)s);
}

qz_status qz_gemm_int4_outlier_grouped(const qz_int4o_weight *ws, int n, int64_t B,
                                       const qz_half *X, int64_t ldx, qz_half *const *Ys,
                                       const int64_t *ldys, void *workspace,
                                       size_t workspace_bytes, qz_stream s) {
  if (!ws || !Ys || !ldys || n < 1 || B < 1) return QZ_ERR_INVALID_ARG;
  if (n > QZ_MAX_GROUP || B > QZ_MAX_BATCH) return QZ_ERR_UNSUPPORTED;
  for (int m = 0; m < n; ++m) {
    QZ_TRY(check_int4o_weight(&ws[m]));
    if (ws[m].K != ws[0].K || ws[m].n_out != ws[0].n_out || ws[m].perm != ws[0].perm)
      return QZ_ERR_INVALID_ARG;
    QZ_TRY(check_vec(Ys[m], B, ws[m].N, ldys[m]));
  }
  QZ_TRY(check_vec(X, B, ws[0].K, ldx));
  GemvParams p;
  fill_int4o(p, ws, n);
  return gemm_common(true, p, B, X, ldx, Ys, ldys, n, workspace, workspace_bytes,
                     (cudaStream_t)s);
}

qz_status qz_gemv_int8_grouped_mapped(const qz_int8_weight *ws, int n, const qz_half *x,
                                      qz_half *const *ys, qz_stream s) {
  if (!ws || !ys || n < 1) return QZ_ERR_INVALID_ARG;
  if (n > QZ_MAX_GROUP) return QZ_ERR_UNSUPPORTED;
  qz_int8_weight v[QZ_MAX_GROUP];
  for (int m = 0; m < n; ++m) {
    QZ_TRY(check_int8_weight(&ws[m]));
    if (ws[m].K != ws[0].K) return QZ_ERR_INVALID_ARG;
    QZ_TRY(check_vec(ys[m], 1, ws[m].N, 0));
    v[m] = ws[m];
    QZ_TRY(device_view_t(v[m].q));
    QZ_TRY(device_view_t(v[m].scale));
  }
  QZ_TRY(check_vec(x, 1, ws[0].K, 0));
  GemvParams p;
  fill_int8(p, v, n);
  return mapped_common(false, p, x, ys, n, (cudaStream_t)s);
}

qz_status qz_gemv_int4_outlier_grouped_mapped(const qz_int4o_weight *ws, int n,
                                              const qz_half *x, qz_half *const *ys,
                                              qz_stream s) {
  if (!ws || !ys || n < 1) return QZ_ERR_INVALID_ARG;
  if (n > QZ_MAX_GROUP) return QZ_ERR_UNSUPPORTED;
  qz_int4o_weight v[QZ_MAX_GROUP];
  for (int m = 0; m < n; ++m) {
    QZ_TRY(check_int4o_weight(&ws[m]));
    if (ws[m].K != ws[0].K || ws[m].n_out != ws[0].n_out || ws[m].perm != ws[0].perm)
      return QZ_ERR_INVALID_ARG;
    QZ_TRY(check_vec(ys[m], 1, ws[m].N, 0));
    v[m] = ws[m];
    QZ_TRY(device_view_t(v[m].perm));
    QZ_TRY(device_view_t(v[m].w_out));
    QZ_TRY(device_view_t(v[m].q4));
    QZ_TRY(device_view_t(v[m].scale));
  }
  QZ_TRY(check_vec(x, 1, ws[0].K, 0));
  GemvParams p;
  fill_int4o(p, v, n);
  return mapped_common(true, p, x, ys, n, (cudaStream_t)s);
}

qz_status qz_gemv_int4_outlier_grouped(const qz_int4o_weight *ws, int n, const qz_half *x,
                                       qz_half *const *ys, qz_stream s) {
  if (!ws || !ys || n < 1) return QZ_ERR_INVALID_ARG;
  if (n > QZ_MAX_GROUP) return QZ_ERR_UNSUPPORTED;
  for (int m = 0; m < n; ++m) {
    QZ_TRY(check_int4o_weight(&ws[m]));
    if (ws[m].K != ws[0].K || ws[m].n_out != ws[0].n_out || ws[m].perm != ws[0].perm)
      return QZ_ERR_INVALID_ARG;
    QZ_TRY(check_vec(ys[m], 1, ws[m].N, 0));
  }
  QZ_TRY(check_vec(x, 1, ws[0].K, 0));
  GemvParams p;
  fill_int4o(p, ws, n);
  return gemm_common(true, p, 1, x, 0, ys, nullptr, n, nullptr, 0, (cudaStream_t)s);
}


qz_status qz_gemv_int8_sequence(const qz_int8_weight *ws, const int *counts, int n,
                                const qz_half *const *x, qz_half *const *ys, uint32_t *sync,
                                qz_stream s) {
  return sequence_common(
      false, ws, counts, n, x, ys, sync, (cudaStream_t)s,
      [](GemvParams &p, const qz_int8_weight *w, int c) { fill_int8(p, w, c); },
      [](const qz_int8_weight &w, const qz_int8_weight &w0) -> qz_status {
        QZ_TRY(check_int8_weight(&w));
        return w.K == w0.K ? QZ_OK : QZ_ERR_INVALID_ARG;
      });
}

qz_status qz_gemv_int4_outlier_sequence(const qz_int4o_weight *ws, const int *counts, int n,
                                        const qz_half *const *x, qz_half *const *ys,
                                        uint32_t *sync, qz_stream s) {
  return sequence_common(
      true, ws, counts, n, x, ys, sync, (cudaStream_t)s,
      [](GemvParams &p, const qz_int4o_weight *w, int c) { fill_int4o(p, w, c); },
      [](const qz_int4o_weight &w, const qz_int4o_weight &w0) -> qz_status {
        QZ_TRY(check_int4o_weight(&w));
        return (w.K == w0.K && w.n_out == w0.n_out && w.perm == w0.perm) ? QZ_OK
                                                                          : QZ_ERR_INVALID_ARG;
      });
}

}  // extern "C"
