/*
 * qz.h - C ABI of libqz: weight-only quantized dequant-GEMV/GEMM for one GB300.
 *
 * The operations follow three web pages about serving a decoder LLM from
 * compressed weights:
 *   [ELG]  "Open Origin - ELG Stream Layer" (INT8 layer paging),
 *   [OTF]  "On-The-Fly Weight Synthesizer (OTF-LLM Engine)" (outlier-aware INT4),
 *   [NTR]  "NTransformer" summary (tiered layer streaming with custom GEMV).
 * Each entry point below names the section of the page that defines it.
 *
 * Conventions for every call
 *   - Pointers are DEVICE pointers unless the comment says host.
 *   - The caller allocates and owns every buffer.  The library never allocates
 *     or frees device memory and keeps no pointer to caller memory between
 *     calls (the pager keeps the pointers it is given until it is destroyed).
 *   - fp16 data is passed as qz_half: the bit pattern of an IEEE-754 binary16.
 *   - Matrices are row-major.  ld* is the distance between rows in ELEMENTS
 *     of the array's own type (bytes for int8/uint8 arrays).
 *   - Every call that launches GPU work is asynchronous on the given stream
 *     (NULL = the legacy default stream).  Outputs are valid once the stream
 *     has reached the call.  Calls that overlap on the GPU and write the same
 *     output race.
 *   - Arguments are validated on the host before anything is enqueued: a call
 *     that returns an error has enqueued nothing (QZ_ERR_CUDA excepted: the
 *     launch itself failed, and cudaGetLastError's code is kept in
 *     qz_last_cuda_error(), per host thread).
 *   - Alignment: every device pointer of a MATRIX (W, q, q4, w_out) must be
 *     16-byte aligned and its ld* must make rows 16-byte multiples (ld % 8 == 0
 *     for fp16, ld % 16 == 0 for int8/uint8); activation and output vectors
 *     (x, X, y, Y) need only the 2-byte alignment of fp16, with any ld >= the
 *     row length.  Violations return QZ_ERR_ALIGNMENT.
 *   - Inputs must be finite.  Non-finite weights or profiles give unspecified
 *     (but memory-safe) results.
 *   - No exception, abort or device trap is ever raised by the library.
 */
#ifndef QZ_H
#define QZ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *qz_stream; /* the same type as cudaStream_t */
typedef uint16_t qz_half;              /* IEEE-754 binary16 bit pattern */

typedef enum {
  QZ_OK = 0,
  QZ_ERR_INVALID_ARG = 1, /* null pointer, negative or inconsistent size */
  QZ_ERR_ALIGNMENT = 2,   /* pointer or leading dimension breaks the 16-B rule */
  QZ_ERR_UNSUPPORTED = 3, /* valid but outside what the kernels handle (see call) */
  QZ_ERR_CUDA = 4,        /* a CUDA launch/enqueue failed; see qz_last_cuda_error */
  QZ_ERR_IO = 5,          /* pager host-side failure (copy enqueue, event) */
  QZ_ERR_DATA = 6         /* data check failed (qz_check_perm) */
} qz_status;

/* Human-readable name of a status; never NULL. */
const char *qz_status_string(qz_status st);
/* Library version as major*10000 + minor*100 + patch. */
int qz_version(void);
/* The cudaError_t of the last QZ_ERR_CUDA returned on this host thread. */
int qz_last_cuda_error(void);

/* Launch overlap for the GEMV/GEMM entry points, per host thread (off by
 * default).  When on, each product kernel is launched with programmatic
 * dependent launch: it may start while the preceding kernel on the stream is
 * still running, starts loading (GEMV: the first ring stage of each warp) or
 * already converts (tensor-core GEMM) the first weight tiles of each CTA, and
 * waits for that kernel (griddepcontrol.wait) before it reads x or writes y.
 * The caller promises that no work still in flight on the stream writes the
 * WEIGHTS of the call (q/q4/w_out/scale/perm); inputs and outputs keep normal
 * stream order.  Returns QZ_ERR_INVALID_ARG unless enable is 0 or 1. */
qz_status qz_set_overlap(int enable);
/* The current host thread's overlap setting (0 or 1). */
int qz_get_overlap(void);

/* The library's device error word, a bit set: 1 if a kernel gave up a
 * bounded wait (its output is then incomplete); 2 if qz_embed_int8 met a
 * token outside its table (that row was written as zeros).  0 if neither
 * happened since the last clear.  Synchronous (reads device memory);
 * clear = 1 resets it.  Not for use during stream capture. */
qz_status qz_device_error(int *code, int clear);

/* Largest batch the GEMM entry points accept. */
#define QZ_MAX_BATCH 64
/* Largest number of matrices in one grouped launch. */
#define QZ_MAX_GROUP 4
/* Largest number of products in one sequence call (qz_gemv_*_sequence). */
#define QZ_MAX_SEQ 4

/* ======================================================================
 * INT8, one scale per tensor  [ELG "Technical Architecture > INT8
 * Quantization & Direct Mapping": scale = max|W| / 127, q = round(W/scale);
 * "FP16 On-The-Fly GPU Reconstruction": w = q * scale]
 * ====================================================================== */

/* Quantize an fp16 matrix W [N][ldw] to q [N][ldq] int8 and one fp32 scale.
 *   scale = fp32(max |W|) / 127 (IEEE fp32 divide, round to nearest even);
 *   q     = clamp(rint(fp32(W) / scale), -127, 127), rint = half-to-even;
 *   an all-zero W gives scale = 0 and q = 0.
 * Columns K..ldq-1 of q are written as 0.  *scale is used as the running
 * maximum while the call runs, so no other work may read it until the
 * stream has passed this call.  N, K >= 1; ldw >= K; ldq >= K. */
qz_status qz_quantize_int8(const qz_half *W, int64_t N, int64_t K, int64_t ldw,
                           int8_t *q, int64_t ldq, float *scale, qz_stream s);

/* A quantized INT8 matrix as the GEMV calls read it (a host struct holding
 * device pointers).  Bytes q[i][K..ldq) are never used in a product. */
typedef struct {
  const int8_t *q;     /* [N][ldq] codes */
  const float *scale;  /* [1] per-tensor scale */
  int64_t N, K, ldq;
} qz_int8_weight;

/* y[i] = fp16( scale * sum_j q[i][j] * x[j] ), fp32 accumulation, products of
 * the exact integer code with the fp16 input; no fp16 weight is formed.
 * x [K], y [N].  K <= 57344.  The CUDA-core kernel stages the input in
 * shared memory; at the largest K, where it does not fit, the call runs on the
 * tensor-core kernel instead (same result bound). */
qz_status qz_gemv_int8(const qz_int8_weight *w, const qz_half *x, qz_half *y,
                       qz_stream s);

/* Y[b][i] = fp16( scale * sum_j q[i][j] * X[b][j] ) for b < B.
 * X [B][ldx], Y [B][ldy]; 1 <= B <= QZ_MAX_BATCH.  The path depends on the
 * shape, never the result bound: B = 1 as qz_gemv_int8; B = 2..8 on the
 * warp-MMA kernel (mma.sync on the exact codes, fp32 accumulation) when the
 * batch's fp16 inputs and a ring of weight stages fit in shared memory
 * (roughly 2*B*K bytes well under 227 KiB); otherwise, and for B > 8, on
 * the tensor cores (tcgen05, fp16 x fp16 products of the exact codes, fp32
 * accumulation in tensor memory). */
qz_status qz_gemm_int8(const qz_int8_weight *w, int64_t B, const qz_half *X,
                       int64_t ldx, qz_half *Y, int64_t ldy, void *workspace,
                       size_t workspace_bytes, qz_stream s);

/* Device workspace the batched calls use on the tensor-core path: the
 * permuted inputs are gathered once per call into tensor-core tiles there,
 * then streamed into the GEMM by bulk copies; behind them lie the fp32
 * partial sums of output tiles whose K range is cut between SMs (at most two
 * per SM) and their arrival counters, so that every SM gets the same share
 * of the call's work.  B inputs of K channels with n_out outlier channels (0
 * for INT8); 0 for invalid sizes.  Host only; the size does not depend on N
 * or the device.  The workspace argument of qz_gemm_* may be NULL (the
 * tensor-core kernel then gathers its inputs itself and gives each SM whole
 * 128-row tiles only, much more slowly); if given it must be 16-byte aligned
 * and at least this many bytes (checked whatever path the call takes:
 * QZ_ERR_INVALID_ARG if short, QZ_ERR_ALIGNMENT if misaligned, before
 * anything is enqueued), caller-owned, and not used by other work while the
 * call runs.  Only the tensor-core path uses it.  Results with and without a
 * workspace agree within the products' rounding bound, not bit for bit (the
 * fp32 partial sums are added in a different order). */
size_t qz_gemm_workspace_bytes(int64_t B, int64_t K, int64_t n_out);

/* n matrices (1 <= n <= QZ_MAX_GROUP) that read the same input x, in one
 * launch (q/k/v, gate/up).  Each keeps its own scale.  ws: host array of n
 * structs with equal K; ys: host array of n device pointers. */
qz_status qz_gemv_int8_grouped(const qz_int8_weight *ws, int n,
                               const qz_half *x, qz_half *const *ys,
                               qz_stream s);

/* The batched form of qz_gemv_int8_grouped: n matrices (1 <= n <=
 * QZ_MAX_GROUP) of equal K read the same inputs X [B][ldx] in one call, and
 * Ys[m] [B][ldys[m]] receives matrix m's outputs.  Ys and ldys are host
 * arrays of n entries.  Batch limits, the CUDA-core/tensor-core choice and
 * the workspace are those of qz_gemm_int8 (one workspace serves the whole
 * group: qz_gemm_workspace_bytes(B, K, 0)). */
qz_status qz_gemm_int8_grouped(const qz_int8_weight *ws, int n, int64_t B,
                               const qz_half *X, int64_t ldx, qz_half *const *Ys,
                               const int64_t *ldys, void *workspace,
                               size_t workspace_bytes, qz_stream s);

/* Rows of an INT8 vocabulary table (embed_tokens) as fp16 activations
 * [OTF "Architecture & Key Innovations", key innovation 4: vocabulary
 * lookup tables compressed to INT8; ELG "FP16 On-The-Fly GPU
 * Reconstruction": q * scale as fp16]:
 *   out[b][j] = fp16(q[tokens[b]][j] * scale), b < B, j < K,
 * the exact product rounded once to the nearest fp16, ties to even.
 * table: the quantized [V][K] table (V = table->N), as qz_quantize_int8
 * makes it (one scale per tensor); any K.  tokens: device int32 [B], 4-byte
 * aligned.  out: device fp16 [B][ldo], 16-byte aligned, ldo >= K, ldo a
 * multiple of 8.  B >= 0 (B = 0 enqueues nothing).  A token outside [0, V)
 * is not read: its row of out is written as zeros and bit 2 of the device
 * error word (qz_device_error) is set.
 * With tied word embeddings the same table is the output projection
 * (lm_head): qz_gemv_int8(table, h, logits) gives
 * logits[v] = scale * sum_j q[v][j] h[j]. */
qz_status qz_embed_int8(const qz_int8_weight *table, const int32_t *tokens,
                        int64_t B, qz_half *out, int64_t ldo, qz_stream s);

/* ======================================================================
 * Outlier-aware INT4  [OTF "Architecture & Key Innovations": diagram and
 * key innovation 3 (global_perm_idx; top-1% channels by |W| x |X_profile|
 * kept in FP16; background INT4 in [-7,7], zero-point 0, 2:1 uint8 packing;
 * output = outlier product + background product); key innovation 1 (packed
 * weights dequantized in registers, no fp16 weight tensor)]
 *
 * Format of one [N][K] matrix with n_out outlier channels, kb = K - n_out:
 *   perm  int32 [K]          : permuted input t reads x[perm[t]]; t < n_out
 *                              are the outliers (global_perm_idx);
 *   w_out fp16  [N][ld_out]  : w_out[i][t] = W[i][perm[t]], t < n_out;
 *   q4    uint8 [N][ld_q4]   : background code of permuted input n_out + t'
 *                              in byte t'/2, low nibble if t' even, as the
 *                              two's-complement nibble (values -7..7);
 *   scale fp32  [N]          : s_i = fp32(max_t' |W[i][perm[n_out+t']]|) / 7.
 * ld_out = roundup(n_out, 8), ld_q4 = roundup(ceil(kb/2), 16); padding is 0.
 * ====================================================================== */

/* Row strides of the format (host only, no GPU work).  ld_out/ld_q4: host. */
qz_status qz_int4o_layout(int64_t N, int64_t K, int64_t n_out, int64_t *ld_out,
                          int64_t *ld_q4);

/* colsum[j] += sum_i |W[i][j]| * 2^24, exactly, as int64 (every fp16 value
 * is an integer multiple of 2^-24, so the sum is order-independent).  Call it
 * once per matrix that shares the permutation; the caller zeroes colsum. */
qz_status qz_saliency_accumulate(const qz_half *W, int64_t N, int64_t K,
                                 int64_t ldw, int64_t *colsum, qz_stream s);

/* Build global_perm_idx from colsum [K] and the activation profile
 * x_profile [K] (fp32): score_j = fp64(colsum[j]) * fp64(|x_profile[j]|); the
 * n_out channels of highest score (ties: lower j first) come first, in
 * ascending j, then the rest in ascending j.  0 <= n_out <= K <= 2^20.
 * perm [K] int32 is also used as working storage during the call. */
qz_status qz_select_outliers(const int64_t *colsum, const float *x_profile,
                             int64_t K, int64_t n_out, int32_t *perm,
                             qz_stream s);

/* *flag = 0 if perm [K] is a permutation of 0..K-1, 1 if an entry is out of
 * range, 2 if an entry repeats.  K <= 2^20.  The host reads flag after the
 * stream reaches the call; QZ_ERR_DATA is the host's verdict for flag != 0. */
qz_status qz_check_perm(const int32_t *perm, int64_t K, int32_t *flag,
                        qz_stream s);

/* Quantize W [N][ldw] fp16 with the given perm into the format above.
 * w_out may be NULL when n_out == 0.  ld_out/ld_q4 must be at least the
 * values of qz_int4o_layout and keep the 16-B rule; all padding is written
 * as 0.  Each CTA stages one fp16 row of W in shared memory, so K is limited
 * by the device's opt-in shared memory per block: 2 * roundup(K, 8) bytes
 * must fit (K <= 116224 on GB300's 227 KiB); beyond that, and beyond
 * K = 2^17 on any device, the call returns QZ_ERR_UNSUPPORTED. */
qz_status qz_quantize_int4_outlier(const qz_half *W, int64_t ldw,
                                   const int32_t *perm, int64_t N, int64_t K,
                                   int64_t n_out, qz_half *w_out,
                                   int64_t ld_out, uint8_t *q4, int64_t ld_q4,
                                   float *scale, qz_stream s);

/* One quantized INT4-outlier matrix (host struct holding device pointers). */
typedef struct {
  int64_t N, K, n_out, ld_out, ld_q4;
  const int32_t *perm;
  const qz_half *w_out; /* may be NULL when n_out == 0 */
  const uint8_t *q4;
  const float *scale;
} qz_int4o_weight;

/* y[i] = fp16( sum_{t<n_out} w_out[i][t] * x[perm[t]]
 *            + s_i * sum_{t'} q[i][t'] * x[perm[n_out+t']] )
 * fp32 accumulation of exact products; x is gathered through perm into
 * shared memory inside the kernel.  x [K] in ORIGINAL channel order, y [N].
 * K <= 57344. */
qz_status qz_gemv_int4_outlier(const qz_int4o_weight *w, const qz_half *x,
                               qz_half *y, qz_stream s);

/* The same for a batch: X [B][ldx], Y [B][ldy], 1 <= B <= QZ_MAX_BATCH; the
 * same choice of kernels as qz_gemm_int8.  Every kernel keeps the outlier
 * and background products apart and combines them as y = D_out + s_i * D_bg. */
qz_status qz_gemm_int4_outlier(const qz_int4o_weight *w, int64_t B,
                               const qz_half *X, int64_t ldx, qz_half *Y,
                               int64_t ldy, void *workspace,
                               size_t workspace_bytes, qz_stream s);

/* Allocation-free variant of qz_gemm_int4_outlier.  The pages have no
 * counterpart; it exists for callers that cannot allocate device memory at
 * the point of the call (code running during CUDA-graph capture, where
 * cudaMalloc is not allowed; plugins inside a host application that owns the
 * device memory budget; loops that must not touch an allocator after
 * start-up).  Instead of a caller workspace it uses a library-owned static
 * device array of QZ_NOALLOC_SCRATCH_BYTES, which every GPU that loads the
 * library holds until the process exits; it allocates nothing itself.
 * Limit: qz_gemm_workspace_bytes(B, K, n_out) must not exceed
 * QZ_NOALLOC_SCRATCH_BYTES (e.g. B = 64 up to K ~ 48k), else
 * QZ_ERR_UNSUPPORTED.  All calls share the array (it keeps the last call's
 * contents, every call rewrites what it reads): calls that overlap on the
 * GPU, on any stream, race.  The first call on a device looks the array's
 * device address up (cudaGetSymbolAddress) and should come before any stream
 * capture.  Same arguments and result as qz_gemm_int4_outlier otherwise. */
#define QZ_NOALLOC_SCRATCH_BYTES (16u << 20)
qz_status qz_gemm_int4_outlier_noalloc(const qz_int4o_weight *w, int64_t B,
                                       const qz_half *X, int64_t ldx,
                                       qz_half *Y, int64_t ldy, qz_stream s);

/* n matrices sharing one input and one permutation (same perm pointer, K and
 * n_out), one launch.  ws: host array; ys: host array of device pointers. */
qz_status qz_gemv_int4_outlier_grouped(const qz_int4o_weight *ws, int n,
                                       const qz_half *x, qz_half *const *ys,
                                       qz_stream s);

/* The batched form of qz_gemv_int4_outlier_grouped: n matrices sharing K,
 * n_out and perm read X [B][ldx]; Ys[m] [B][ldys[m]] receives matrix m's
 * outputs (host arrays of n entries).  Otherwise as qz_gemm_int4_outlier;
 * one workspace of qz_gemm_workspace_bytes(B, K, n_out) bytes serves the
 * group. */
qz_status qz_gemm_int4_outlier_grouped(const qz_int4o_weight *ws, int n, int64_t B,
                                       const qz_half *X, int64_t ldx,
                                       qz_half *const *Ys, const int64_t *ldys,
                                       void *workspace, size_t workspace_bytes,
                                       qz_stream s);

/* ======================================================================
 * Dependent products in one launch  [no counterpart on the pages: a decoder
 * layer's four products (q,k,v; o; gate,up; down) run back to back, each
 * reading the previous one's result through the layer glue, so one launch
 * per layer replaces four]
 *
 * n batch-1 grouped products (1 <= n <= QZ_MAX_SEQ) run in order in one
 * launch: product k multiplies the next counts[k] matrices of ws (equal K;
 * for INT4 also equal n_out and perm, as in the grouped calls) with x[k] and
 * stores them to the next counts[k] entries of ys.  Product k reads x[k] only
 * after every output of products 0..k-1 has been stored, so x[k] may be one
 * of those outputs.  Results equal the separate grouped calls bit for bit.
 *   ws, ys: host arrays of sum(counts) entries; counts, x: host arrays of n.
 *   sync: device uint32, 4-byte aligned, 0 before the first call; every call
 *   that completes leaves it 0.  Calls that can be in flight at the same time
 *   (for example consecutive calls under qz_set_overlap) need different
 *   words; after a device error (qz_device_error) it must be zeroed again.
 * The launch holds one CTA on every SM and its CTAs wait on one another
 * (bounded in time, reported through qz_device_error), so it must not share
 * the GPU with work that keeps SMs busy indefinitely.
 * ====================================================================== */
qz_status qz_gemv_int8_sequence(const qz_int8_weight *ws, const int *counts, int n,
                                const qz_half *const *x, qz_half *const *ys,
                                uint32_t *sync, qz_stream s);
qz_status qz_gemv_int4_outlier_sequence(const qz_int4o_weight *ws, const int *counts,
                                        int n, const qz_half *const *x,
                                        qz_half *const *ys, uint32_t *sync,
                                        qz_stream s);

/* ======================================================================
 * Zero-copy products  ["Open Origin - ELG Stream Layer", Technical
 * Architecture > INT8 Quantization & Direct Mapping: INT8 tensors kept in a
 * pre-allocated pinned memory pool and reached by zero-copy DMA; "NTransformer"
 * summary, 3-Tier Adaptive Caching, Tier B: layers kept in pinned RAM]
 *
 * The batch-1 grouped products with the weights read in place by the GPU:
 * every weight buffer of ws (codes, scales, and for INT4 outliers and perm)
 * may be pinned host memory mapped into the device's address space
 * (cudaHostAlloc, or cudaHostRegister with cudaHostRegisterMapped; under
 * unified addressing the host pointer is the device pointer) or device
 * memory.  Each call asks the runtime for the device address of every buffer
 * (cudaPointerGetAttributes); pageable or unknown memory gives
 * QZ_ERR_INVALID_ARG and nothing is launched.  x and ys are device memory.
 * Results equal the device-resident calls bit for bit; only the way codes
 * are read differs (plain loads by every lane, over the host link, instead
 * of bulk copies).  The host memory must stay pinned and unchanged until the
 * stream has passed the call.  Same sizes and errors as the grouped calls.
 * ====================================================================== */
qz_status qz_gemv_int8_grouped_mapped(const qz_int8_weight *ws, int n,
                                      const qz_half *x, qz_half *const *ys,
                                      qz_stream s);
qz_status qz_gemv_int4_outlier_grouped_mapped(const qz_int4o_weight *ws, int n,
                                              const qz_half *x,
                                              qz_half *const *ys, qz_stream s);

/* ======================================================================
 * Layer pager  [ELG "Key Features" 2 (prefetch, transfer, reconstruct,
 * purge) and 3 (a second CUDA stream copies layer N+1 while layer N
 * computes); NTR "3-Tier Adaptive Caching", Tier B (pinned RAM, H2D DMA)]
 *
 * Double-buffers packed layers from pinned host memory into two device
 * slots owned by the caller.  acquire(L) makes the compute stream wait until
 * layer L is in its slot and starts the copy of layer L+1 into the other
 * slot (after the compute that last used that slot, recorded by release);
 * release(L) marks the end of the compute work that reads layer L.  Layers
 * must be acquired in order 0, 1, ..., n-1 (then 0 again for the next pass).
 * The "purge" of the page becomes slot reuse: nothing is freed in the loop.
 * ====================================================================== */
typedef struct qz_pager qz_pager;

/* host_layers: host array of n_layers pinned host pointers; bytes: host
 * array of their sizes (each <= slot_bytes, multiple of 16); slot0/slot1:
 * device buffers of slot_bytes each.  The pager creates its own events; it
 * is destroyed with qz_pager_destroy.  *out receives the handle (host). */
qz_status qz_pager_create(const void *const *host_layers, const size_t *bytes,
                          int n_layers, void *slot0, void *slot1,
                          size_t slot_bytes, qz_stream copy_stream,
                          qz_stream compute_stream, qz_pager **out);
/* *dev_ptr (host) receives the device slot that holds `layer`. */
qz_status qz_pager_acquire(qz_pager *p, int layer, const void **dev_ptr);
qz_status qz_pager_release(qz_pager *p, int layer);
/* Waits for the pager's copies to finish, then frees its host state. */
qz_status qz_pager_destroy(qz_pager *p);

/* Host-side fault injection for tests: make the copy enqueue of layer
 * `layer` (at its next prefetch) fail as if cudaMemcpyAsync had failed.
 * The pager then drains its copy stream and acquire returns QZ_ERR_IO.
 * layer = -1 clears the injection.  Touches no GPU state. */
qz_status qz_pager_inject_copy_failure(qz_pager *p, int layer);

#ifdef __cplusplus
}
#endif
#endif /* QZ_H */
