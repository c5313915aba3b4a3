// Layer pager: double-buffered host->device streaming of packed layers.
//
// "Open Origin - ELG Stream Layer", Key Features 2 (prefetch from the pinned
// RAM pool, transfer over the bus, reconstruct on the GPU, purge) and 3 (a
// second CUDA stream copies layer N+1 while layer N computes); "NTransformer"
// summary, 3-Tier Adaptive Caching, Tier B (pinned RAM streamed by H2D DMA).
//
// Two device slots alternate.  Ordering is by CUDA events only (no host
// waits in the steady state, no device spin-waits):
//   copy stream:    wait freed[k] -> memcpy(slot k <- layer) -> record copied[k]
//   compute stream: wait copied[k] -> (caller's kernels) -> record freed[k]
// The page's "purge" becomes slot reuse: nothing is freed inside the loop.
#include <cuda_runtime.h>

#include <new>
#include <vector>

#include "../../include/qz.h"

namespace qz {
qz_status cuda_status(cudaError_t e);
}

struct qz_pager {
  std::vector<const void *> host;
  std::vector<size_t> bytes;
  void *slot[2] = {nullptr, nullptr};
  size_t slot_bytes = 0;
  cudaStream_t copy = nullptr, compute = nullptr;
  cudaEvent_t copied[2] = {nullptr, nullptr};
  cudaEvent_t freed[2] = {nullptr, nullptr};
  int slot_layer[2] = {-1, -1};   // layer held (or being copied) in each slot
  bool in_use[2] = {false, false};  // acquired and not yet released
  bool freed_valid[2] = {false, false};
  int expected = 0;               // next layer acquire accepts
  int cur_slot = -1;              // slot of the last acquired layer
  int inject_layer = -1;
  qz_status sticky = QZ_OK;
};

namespace {

// Enqueue the copy of `layer` into slot k on the copy stream.
qz_status enqueue_copy(qz_pager *p, int k, int layer) {
  if (p->inject_layer == layer) {
    // Injected failure: behave as a failed enqueue.  Drain what is in flight
    // so the caller sees a quiet copy stream, then report the failure.
    p->inject_layer = -1;
    cudaStreamSynchronize(p->copy);
    p->slot_layer[k] = -1;
    return QZ_ERR_IO;
  }
  cudaError_t e = cudaSuccess;
  if (p->freed_valid[k]) e = cudaStreamWaitEvent(p->copy, p->freed[k], 0);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(p->slot[k], p->host[layer], p->bytes[layer], cudaMemcpyHostToDevice,
                        p->copy);
  if (e == cudaSuccess) e = cudaEventRecord(p->copied[k], p->copy);
  if (e != cudaSuccess) {
    qz::cuda_status(e);
    cudaStreamSynchronize(p->copy);
    p->slot_layer[k] = -1;
    return QZ_ERR_IO;
  }
  p->slot_layer[k] = layer;
  return QZ_OK;
}

}  // namespace

extern "C" {

qz_status qz_pager_create(const void *const *host_layers, const size_t *bytes, int n_layers,
                          void *slot0, void *slot1, size_t slot_bytes, qz_stream copy_stream,
                          qz_stream compute_stream, qz_pager **out) {
  if (!host_layers || !bytes || n_layers < 1 || !slot0 || !slot1 || !out || slot0 == slot1)
    return QZ_ERR_INVALID_ARG;
  if (((uintptr_t)slot0 & 15u) || ((uintptr_t)slot1 & 15u)) return QZ_ERR_ALIGNMENT;
  for (int l = 0; l < n_layers; ++l) {
    if (!host_layers[l] || bytes[l] == 0 || bytes[l] > slot_bytes) return QZ_ERR_INVALID_ARG;
    if (bytes[l] % 16 || ((uintptr_t)host_layers[l] & 15u)) return QZ_ERR_ALIGNMENT;
  }
  qz_pager *p = new (std::nothrow) qz_pager;
  if (!p) return QZ_ERR_IO;
  p->host.assign(host_layers, host_layers + n_layers);
  p->bytes.assign(bytes, bytes + n_layers);
  p->slot[0] = slot0;
  p->slot[1] = slot1;
  p->slot_bytes = slot_bytes;
  p->copy = (cudaStream_t)copy_stream;
  p->compute = (cudaStream_t)compute_stream;
  for (int k = 0; k < 2; ++k) {
    cudaError_t e = cudaEventCreateWithFlags(&p->copied[k], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->freed[k], cudaEventDisableTiming);
    if (e != cudaSuccess) {
      qz::cuda_status(e);
      for (int j = 0; j < 2; ++j) {
        if (p->copied[j]) cudaEventDestroy(p->copied[j]);
        if (p->freed[j]) cudaEventDestroy(p->freed[j]);
      }
      delete p;
      return QZ_ERR_CUDA;
    }
  }
  *out = p;
  return QZ_OK;
}

qz_status qz_pager_acquire(qz_pager *p, int layer, const void **dev_ptr) {
  if (!p || !dev_ptr) return QZ_ERR_INVALID_ARG;
  if (p->sticky != QZ_OK) return p->sticky;
  const int n = (int)p->host.size();
  if (layer != p->expected) return QZ_ERR_INVALID_ARG;
  // slot that holds (or will hold) this layer
  int k = -1;
  for (int j = 0; j < 2; ++j)
    if (p->slot_layer[j] == layer) k = j;
  if (k < 0) {
    k = p->cur_slot < 0 ? 0 : 1 - p->cur_slot;
    if (p->in_use[k]) return QZ_ERR_INVALID_ARG;  // previous user not released
    qz_status st = enqueue_copy(p, k, layer);
    if (st != QZ_OK) return p->sticky = st;
  }
  cudaError_t e = cudaStreamWaitEvent(p->compute, p->copied[k], 0);
  if (e != cudaSuccess) return qz::cuda_status(e);
  p->in_use[k] = true;
  p->cur_slot = k;
  p->expected = (layer + 1) % n;
  // prefetch the next layer into the other slot while this one computes
  const int next = (layer + 1) % n;
  const int o = 1 - k;
  if (n > 1 && p->slot_layer[o] != next && !p->in_use[o]) {
    qz_status st = enqueue_copy(p, o, next);
    if (st != QZ_OK) return p->sticky = st;
  }
  *dev_ptr = p->slot[k];
  return QZ_OK;
}

qz_status qz_pager_release(qz_pager *p, int layer) {
  if (!p) return QZ_ERR_INVALID_ARG;
  int k = -1;
  for (int j = 0; j < 2; ++j)
    if (p->slot_layer[j] == layer && p->in_use[j]) k = j;
  if (k < 0) return QZ_ERR_INVALID_ARG;
  cudaError_t e = cudaEventRecord(p->freed[k], p->compute);
  if (e != cudaSuccess) return qz::cuda_status(e);
  p->freed_valid[k] = true;
  p->in_use[k] = false;
  return QZ_OK;
}

qz_status qz_pager_inject_copy_failure(qz_pager *p, int layer) {
  if (!p || layer < -1 || layer >= (int)p->host.size()) return QZ_ERR_INVALID_ARG;
  p->inject_layer = layer;
  return QZ_OK;
}

qz_status qz_pager_destroy(qz_pager *p) {
  if (!p) return QZ_ERR_INVALID_ARG;
  cudaError_t first = cudaStreamSynchronize(p->copy);
  for (int k = 0; k < 2; ++k) {
    cudaError_t e = cudaEventDestroy(p->copied[k]);
    if (first == cudaSuccess) first = e;
    e = cudaEventDestroy(p->freed[k]);
    if (first == cudaSuccess) first = e;
  }
  delete p;
  return first == cudaSuccess ? QZ_OK : qz::cuda_status(first);
}

}  // extern "C"
