"""Python API over libqz.  PyTorch supplies device memory and streams only:
every step of quantization and every product runs in the library's kernels.

Names follow the C ABI (include/qz.h): ``quantize_int8``, ``gemv_int8``,
``gemm_int8``, ``gemv_int8_grouped``, ``saliency_accumulate``,
``select_outliers``, ``check_perm``, ``quantize_int4_outlier``,
``gemv_int4_outlier``, ``gemm_int4_outlier``, ``gemv_int4_outlier_grouped``
and the ``Pager``.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _lib
from ._lib import Int4oWeight, Int8Weight, QzError  # noqa: F401


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _round_up(v: int, m: int) -> int:
    return -(-v // m) * m


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("libqz works on CUDA tensors only (no CPU fallback)")


def set_overlap(enable: bool) -> None:
    """Programmatic dependent launch for this host thread's product calls
    (see qz_set_overlap): only when no in-flight work writes the weights."""
    _lib.call("qz_set_overlap", 1 if enable else 0)


def get_overlap() -> bool:
    return bool(_lib.load().qz_get_overlap())


def device_error(clear: bool = True) -> int:
    """The library's device error word (1 = a kernel gave up a bounded wait)."""
    v = ctypes.c_int()
    _lib.call("qz_device_error", ctypes.byref(v), 1 if clear else 0)
    return v.value


# ------------------------------------------------------------------ INT8 ---
@dataclass
class Int8Matrix:
    """Per-tensor INT8 matrix: q [N, ldq] int8 (columns >= K are 0), scale [1]."""
    q: torch.Tensor
    scale: torch.Tensor
    N: int
    K: int

    @property
    def ldq(self) -> int:
        return self.q.stride(0)

    def struct(self) -> Int8Weight:
        return Int8Weight(self.q.data_ptr(), self.scale.data_ptr(), self.N, self.K, self.ldq)

    def tensors(self):
        return (self.q, self.scale)

    def nbytes(self) -> int:
        """Algorithmic bytes: N*K codes + one fp32 scale."""
        return self.N * self.K + 4

    def padded_bytes(self) -> int:
        """Bytes as stored: N*ldq codes (rows padded to 16 bytes) + the scale."""
        return self.N * self.ldq + 4


def quantize_int8(W: torch.Tensor, stream=None) -> Int8Matrix:
    """scale = max|W|/127, q = round(W/scale) (half-to-even), on the GPU."""
    _need_cuda(W)
    assert W.dtype == torch.float16 and W.dim() == 2
    N, K = W.shape
    if W.stride(1) != 1 or W.stride(0) % 8 or W.data_ptr() % 16:
        W = _padded_fp16(W)
    q = torch.empty((N, _round_up(K, 16)), dtype=torch.int8, device=W.device)
    scale = torch.empty((1,), dtype=torch.float32, device=W.device)
    _lib.call("qz_quantize_int8", W.data_ptr(), N, K, W.stride(0), q.data_ptr(), q.stride(0),
              scale.data_ptr(), _stream(stream))
    return Int8Matrix(q, scale, N, K)


def _padded_fp16(W: torch.Tensor) -> torch.Tensor:
    """Copy W into rows padded to a multiple of 8 halves (16 bytes)."""
    N, K = W.shape
    buf = torch.zeros((N, _round_up(K, 8)), dtype=W.dtype, device=W.device)
    buf[:, :K] = W
    return buf


def _vec_out(x: torch.Tensor, N: int, B: int | None = None) -> torch.Tensor:
    if B is None:
        return torch.empty((N,), dtype=torch.float16, device=x.device)
    return torch.empty((B, N), dtype=torch.float16, device=x.device)


def gemv_int8(w: Int8Matrix, x: torch.Tensor, y: torch.Tensor | None = None, stream=None):
    """y = fp16(scale * q @ x) for one input vector x [K]."""
    _need_cuda(x)
    y = _vec_out(x, w.N) if y is None else y
    _lib.call("qz_gemv_int8", ctypes.byref(w.struct()), x.data_ptr(), y.data_ptr(),
              _stream(stream))
    return y


def gemm_workspace_bytes(B: int, K: int, n_out: int = 0) -> int:
    """Device workspace of the tensor-core path for B inputs of K channels."""
    return int(_lib.load().qz_gemm_workspace_bytes(B, K, n_out))


def _workspace(X: torch.Tensor, K: int, n_out: int, workspace):
    """The caller's workspace, a fresh one (B > 4), or None."""
    B = X.shape[0]
    if workspace is False:  # explicitly none: the kernel gathers its inputs itself
        return None, 0
    if workspace is None:
        if B <= 4:
            return None, 0
        nbytes = gemm_workspace_bytes(B, K, n_out)
        workspace = torch.empty((nbytes,), dtype=torch.uint8, device=X.device)
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


def gemm_int8(w: Int8Matrix, X: torch.Tensor, Y: torch.Tensor | None = None, stream=None,
              workspace=None):
    """Y [B, N] = fp16(scale * X @ q^T) for X [B, K], B <= 64.  workspace: a
    uint8 device tensor of gemm_workspace_bytes(B, K) bytes (allocated here if
    None and B > 4; False to let the tensor-core kernel gather by itself)."""
    _need_cuda(X)
    B = X.shape[0]
    Y = _vec_out(X, w.N, B) if Y is None else Y
    wp, wb = _workspace(X, w.K, 0, workspace)
    _lib.call("qz_gemm_int8", ctypes.byref(w.struct()), B, X.data_ptr(), X.stride(0),
              Y.data_ptr(), Y.stride(0), wp, wb, _stream(stream))
    return Y


def gemv_int8_grouped(ws, x: torch.Tensor, ys=None, stream=None):
    """One launch for matrices sharing the input x (q/k/v, gate/up)."""
    _need_cuda(x)
    n = len(ws)
    ys = [_vec_out(x, w.N) for w in ws] if ys is None else ys
    arr = (Int8Weight * n)(*[w.struct() for w in ws])
    yp = (ctypes.c_void_p * n)(*[y.data_ptr() for y in ys])
    _lib.call("qz_gemv_int8_grouped", arr, n, x.data_ptr(), yp, _stream(stream))
    return ys


def embed_int8(table: Int8Matrix, tokens: torch.Tensor, out: torch.Tensor | None = None,
               stream=None) -> torch.Tensor:
    """out [B, K] fp16 = rows tokens[b] of the INT8 table, each q * scale
    rounded once to fp16.  tokens: int32 device tensor [B].  A token outside
    [0, V) gives a zero row and sets bit 2 of device_error()."""
    _need_cuda(tokens)
    assert tokens.dtype == torch.int32 and tokens.dim() == 1 and tokens.is_contiguous()
    B = tokens.shape[0]
    if out is None:
        buf = torch.empty((B, _round_up(table.K, 8)), dtype=torch.float16, device=tokens.device)
        out = buf[:, :table.K]
    _lib.call("qz_embed_int8", ctypes.byref(table.struct()), tokens.data_ptr(), B,
              out.data_ptr(), out.stride(0) if B > 0 else _round_up(table.K, 8), _stream(stream))
    return out


# ------------------------------------------------------------------ INT4 ---
def int4o_layout(N: int, K: int, n_out: int) -> tuple[int, int]:
    """(ld_out halves, ld_q4 bytes) of the packed INT4-outlier format."""
    a, b = ctypes.c_int64(), ctypes.c_int64()
    _lib.call("qz_int4o_layout", N, K, n_out, ctypes.byref(a), ctypes.byref(b))
    return a.value, b.value


def default_n_out(K: int) -> int:
    """Top-1% outlier channels, rounded up: ceil(K / 100)."""
    return (K + 99) // 100


@dataclass
class Int4oMatrix:
    """Outlier-aware INT4 matrix (format in include/qz.h)."""
    perm: torch.Tensor     # int32 [K]
    w_out: torch.Tensor    # fp16 [N, ld_out]
    q4: torch.Tensor       # uint8 [N, ld_q4]
    scale: torch.Tensor    # fp32 [N]
    N: int
    K: int
    n_out: int

    @property
    def ld_out(self) -> int:
        return self.w_out.shape[1]

    @property
    def ld_q4(self) -> int:
        return self.q4.shape[1]

    def struct(self) -> Int4oWeight:
        return Int4oWeight(self.N, self.K, self.n_out, self.ld_out, self.ld_q4,
                           self.perm.data_ptr(),
                           self.w_out.data_ptr() if self.ld_out else None,
                           self.q4.data_ptr() if self.ld_q4 else None,
                           self.scale.data_ptr())

    def tensors(self):
        return (self.perm, self.w_out, self.q4, self.scale)

    def nbytes(self) -> int:
        """Algorithmic bytes: packed codes + fp16 outliers + fp32 row scales."""
        kb = self.K - self.n_out
        return self.N * ((kb + 1) // 2 + 2 * self.n_out + 4)

    def padded_bytes(self) -> int:
        return self.N * (self.ld_q4 + 2 * self.ld_out + 4)


def saliency_accumulate(W: torch.Tensor, colsum: torch.Tensor, stream=None) -> torch.Tensor:
    """colsum[j] += sum_i |W_ij| in units of 2^-24 (exact int64)."""
    _need_cuda(W, colsum)
    if W.stride(1) != 1 or W.stride(0) % 8 or W.data_ptr() % 16:
        W = _padded_fp16(W)
    N, K = W.shape
    _lib.call("qz_saliency_accumulate", W.data_ptr(), N, K, W.stride(0), colsum.data_ptr(),
              _stream(stream))
    return colsum


def select_outliers(colsum: torch.Tensor, x_profile: torch.Tensor, n_out: int,
                    stream=None) -> torch.Tensor:
    """global_perm_idx: top-n_out channels by colsum*|x_profile|, then the rest."""
    _need_cuda(colsum, x_profile)
    K = colsum.shape[0]
    perm = torch.empty((K,), dtype=torch.int32, device=colsum.device)
    _lib.call("qz_select_outliers", colsum.data_ptr(), x_profile.data_ptr(), K, n_out,
              perm.data_ptr(), _stream(stream))
    return perm


def check_perm(perm: torch.Tensor, stream=None) -> int:
    """0 if perm is a bijection of 0..K-1, 1 out of range, 2 duplicate (syncs)."""
    _need_cuda(perm)
    flag = torch.full((1,), -1, dtype=torch.int32, device=perm.device)
    _lib.call("qz_check_perm", perm.data_ptr(), perm.shape[0], flag.data_ptr(),
              _stream(stream))
    return int(flag.item())


def quantize_int4_outlier(W: torch.Tensor, perm: torch.Tensor, n_out: int,
                          stream=None) -> Int4oMatrix:
    """Split W by perm into fp16 outliers + per-row INT4 background, packed."""
    _need_cuda(W, perm)
    assert W.dtype == torch.float16 and W.dim() == 2
    N, K = W.shape
    if W.stride(1) != 1 or W.stride(0) % 8 or W.data_ptr() % 16:
        W = _padded_fp16(W)
    ld_out, ld_q4 = int4o_layout(N, K, n_out)
    dev = W.device
    w_out = torch.empty((N, ld_out), dtype=torch.float16, device=dev)
    q4 = torch.empty((N, ld_q4), dtype=torch.uint8, device=dev)
    scale = torch.empty((N,), dtype=torch.float32, device=dev)
    _lib.call("qz_quantize_int4_outlier", W.data_ptr(), W.stride(0), perm.data_ptr(), N, K,
              n_out, w_out.data_ptr() if ld_out else None, ld_out,
              q4.data_ptr() if ld_q4 else None, ld_q4, scale.data_ptr(), _stream(stream))
    return Int4oMatrix(perm, w_out, q4, scale, N, K, n_out)


def gemv_int4_outlier(w: Int4oMatrix, x: torch.Tensor, y: torch.Tensor | None = None,
                      stream=None):
    """y = fp16(W_out @ x[perm[:n_out]] + s * (Q @ x[perm[n_out:]])), x [K]."""
    _need_cuda(x)
    y = _vec_out(x, w.N) if y is None else y
    _lib.call("qz_gemv_int4_outlier", ctypes.byref(w.struct()), x.data_ptr(), y.data_ptr(),
              _stream(stream))
    return y


def gemm_int4_outlier(w: Int4oMatrix, X: torch.Tensor, Y: torch.Tensor | None = None,
                      stream=None, workspace=None):
    """Y [B, N] for X [B, K]; workspace as for gemm_int8."""
    _need_cuda(X)
    B = X.shape[0]
    Y = _vec_out(X, w.N, B) if Y is None else Y
    wp, wb = _workspace(X, w.K, w.n_out, workspace)
    _lib.call("qz_gemm_int4_outlier", ctypes.byref(w.struct()), B, X.data_ptr(), X.stride(0),
              Y.data_ptr(), Y.stride(0), wp, wb, _stream(stream))
    return Y


def gemv_int4_outlier_grouped(ws, x: torch.Tensor, ys=None, stream=None):
    _need_cuda(x)
    n = len(ws)
    ys = [_vec_out(x, w.N) for w in ws] if ys is None else ys
    arr = (Int4oWeight * n)(*[w.struct() for w in ws])
    yp = (ctypes.c_void_p * n)(*[y.data_ptr() for y in ys])
    _lib.call("qz_gemv_int4_outlier_grouped", arr, n, x.data_ptr(), yp, _stream(stream))
    return ys


def gemv_mapped(ws, x: torch.Tensor, ys=None, stream=None):
    """Batch-1 grouped product with the weights read in place (zero-copy,
    qz_gemv_*_grouped_mapped): the matrices' tensors may be pinned host
    tensors (or device tensors).  ws: Int8Matrix or Int4oMatrix list sharing
    K (INT4: and the permutation); x and ys on the GPU."""
    _need_cuda(x)
    n = len(ws)
    ys = [_vec_out(x, w.N) for w in ws] if ys is None else ys
    for w in ws:
        for t in w.tensors():
            if t.numel() and not (t.is_cuda or t.is_pinned()):
                raise ValueError("zero-copy weights must be device or pinned host tensors")
    int8 = isinstance(ws[0], Int8Matrix)
    arr = ((Int8Weight if int8 else Int4oWeight) * n)(*[w.struct() for w in ws])
    yp = (ctypes.c_void_p * n)(*[y.data_ptr() for y in ys])
    fn = "qz_gemv_int8_grouped_mapped" if int8 else "qz_gemv_int4_outlier_grouped_mapped"
    _lib.call(fn, arr, n, x.data_ptr(), yp, _stream(stream))
    return ys


def _grouped_gemm(fn: str, struct_t, ws, X: torch.Tensor, Ys, stream, workspace, n_out: int):
    _need_cuda(X)
    n, B = len(ws), X.shape[0]
    Ys = [_vec_out(X, w.N, B) for w in ws] if Ys is None else Ys
    arr = (struct_t * n)(*[w.struct() for w in ws])
    yp = (ctypes.c_void_p * n)(*[y.data_ptr() for y in Ys])
    ld = (ctypes.c_int64 * n)(*[y.stride(0) for y in Ys])
    wp, wb = _workspace(X, ws[0].K, n_out, workspace)
    _lib.call(fn, arr, n, B, X.data_ptr(), X.stride(0), yp, ld, wp, wb, _stream(stream))
    return Ys


def gemm_int8_grouped(ws, X: torch.Tensor, Ys=None, stream=None, workspace=None):
    """Ys[m] [B, N_m] for X [B, K] and n matrices sharing K, in one call."""
    return _grouped_gemm("qz_gemm_int8_grouped", Int8Weight, ws, X, Ys, stream, workspace, 0)


def gemm_int4_outlier_grouped(ws, X: torch.Tensor, Ys=None, stream=None, workspace=None):
    """Ys[m] [B, N_m] for X [B, K] and n matrices sharing K, n_out and perm."""
    return _grouped_gemm("qz_gemm_int4_outlier_grouped", Int4oWeight, ws, X, Ys, stream,
                         workspace, ws[0].n_out)


def gemv_sequence(groups, xs, ys=None, sync: torch.Tensor | None = None, stream=None):
    """Dependent batch-1 grouped products in one launch: product k multiplies
    the matrices groups[k] with xs[k] into ys[k]; xs[k] may be an output of an
    earlier product.  sync: a zeroed device int32 word (left zero); concurrent
    calls need different words.  Returns ys (list of lists)."""
    _need_cuda(*xs)
    n = len(groups)
    ys = [[_vec_out(xs[k], w.N) for w in g] for k, g in enumerate(groups)] if ys is None else ys
    flat = [w for g in groups for w in g]
    int8 = isinstance(flat[0], Int8Matrix)
    arr = ((Int8Weight if int8 else Int4oWeight) * len(flat))(*[w.struct() for w in flat])
    counts = (ctypes.c_int * n)(*[len(g) for g in groups])
    xp = (ctypes.c_void_p * n)(*[x.data_ptr() for x in xs])
    yp = (ctypes.c_void_p * len(flat))(*[y.data_ptr() for yy in ys for y in yy])
    if sync is None:
        sync = torch.zeros((1,), dtype=torch.int32, device=xs[0].device)
    fn = "qz_gemv_int8_sequence" if int8 else "qz_gemv_int4_outlier_sequence"
    _lib.call(fn, arr, counts, n, xp, yp, sync.data_ptr(), _stream(stream))
    return ys


# ----------------------------------------------------------------- Pager ---
class Pager:
    """Double-buffered host->device layer streaming (qz_pager_*).

    host_layers: pinned uint8 CPU tensors (one per layer); slots: two uint8
    device tensors of equal size.  The tensors must outlive the pager.
    """

    def __init__(self, host_layers, slots, copy_stream, compute_stream):
        self._keep = (list(host_layers), list(slots))
        n = len(host_layers)
        ptrs = (ctypes.c_void_p * n)(*[h.data_ptr() for h in host_layers])
        sizes = (ctypes.c_size_t * n)(*[h.numel() for h in host_layers])
        out = ctypes.c_void_p()
        _lib.call("qz_pager_create", ptrs, sizes, n, slots[0].data_ptr(), slots[1].data_ptr(),
                  slots[0].numel(), copy_stream.cuda_stream, compute_stream.cuda_stream,
                  ctypes.byref(out))
        self._h = out
        self.slots = slots

    def acquire(self, layer: int) -> int:
        p = ctypes.c_void_p()
        _lib.call("qz_pager_acquire", self._h, layer, ctypes.byref(p))
        return p.value

    def release(self, layer: int) -> None:
        _lib.call("qz_pager_release", self._h, layer)

    def inject_copy_failure(self, layer: int) -> None:
        _lib.call("qz_pager_inject_copy_failure", self._h, layer)

    def close(self) -> None:
        if self._h:
            _lib.call("qz_pager_destroy", self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
