"""The allocation-free batched product (qz_gemm_int4_outlier_noalloc).

It serves callers that cannot allocate device memory where they run the
product (during CUDA-graph capture, inside a host application that owns the
device memory, in loops that must not touch an allocator): its tensor-core
workspace is a fixed library-owned device array.  The test calls it through
the C ABI twice in a row and checks each result against the workspace entry
point qz_gemm_int4_outlier (bit-identical, same kernels) and against the CPU
oracle's bound.  This file sorts last so a failure here never hides others.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import qz_oracle as O
from weight_only_quantized_dequant_gb300 import synthetic as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_only_quantized_dequant_gb300 import _lib, build
    build.build()
    return _lib.load()


def test_noalloc_matches_workspace_entry_point_twice(lib):
    import weight_only_quantized_dequant_gb300 as qz
    N, K, n_out, B = 1000, 4096, 41, 64
    W = S.weight(N, K, 9900, device="cuda")
    prof = S.x_profile(K, n_out, 9901, device="cuda")
    colsum = torch.zeros((K,), dtype=torch.int64, device="cuda")
    qz.saliency_accumulate(W, colsum)
    perm = qz.select_outliers(colsum, prof, n_out)
    w = qz.quantize_int4_outlier(W, perm, n_out)
    X = S.activation(B, K, 9902, device="cuda")
    ref = qz.gemm_int4_outlier(w, X)          # caller-provided workspace
    torch.cuda.synchronize()
    wo, q4, s = O.int4o_quantize(W.cpu().numpy(), perm.cpu().numpy(), n_out)
    y_ref, a_ref = O.int4o_product_ref(wo, q4, s, perm.cpu().numpy(), n_out, K, X.cpu().numpy())
    tol = O.tolerance(y_ref, a_ref)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        Y = torch.full((B, N), float("nan"), dtype=torch.float16, device="cuda")
        st = lib.qz_gemm_int4_outlier_noalloc(ctypes.byref(w.struct()), B, X.data_ptr(),
                                              X.stride(0), Y.data_ptr(), Y.stride(0), stream)
        assert st == 0, f"call {call}: status {st}"
        torch.cuda.synchronize()
        assert qz.device_error() == 0
        assert torch.equal(Y, ref), f"call {call} differs from the workspace entry point"
        err = np.abs(Y.float().cpu().numpy().astype(np.float64) - y_ref)
        assert (err <= tol).all(), f"call {call} outside the oracle bound"


def _int4_matrix(N, K, n_out, seed):
    import weight_only_quantized_dequant_gb300 as qz
    W = S.weight(N, K, seed, device="cuda")
    prof = S.x_profile(K, n_out, seed + 1, device="cuda")
    colsum = torch.zeros((K,), dtype=torch.int64, device="cuda")
    qz.saliency_accumulate(W, colsum)
    perm = qz.select_outliers(colsum, prof, n_out)
    w = qz.quantize_int4_outlier(W, perm, n_out)
    wo, q4, s = O.int4o_quantize(W.cpu().numpy(), perm.cpu().numpy(), n_out)
    return w, (wo, q4, s, perm.cpu().numpy())


def _call(lib, w, X, Y, stream):
    B = X.shape[0]
    return lib.qz_gemm_int4_outlier_noalloc(ctypes.byref(w.struct()), B, X.data_ptr(),
                                            X.stride(0), Y.data_ptr(), Y.stride(0), stream)


def test_noalloc_cut_tile_counters_restart_twice(lib):
    """One ragged 128-row tile at K = 28672, batch 16: the tile's K range is
    cut between many SMs, whose partial sums and arrival counters live in
    the shared scratch array.  Two calls in a row give the bits of the
    workspace entry point (so the counters start each call at zero) and
    stay inside the oracle bound."""
    import weight_only_quantized_dequant_gb300 as qz
    N, K, n_out, B = 100, 28672, 287, 16
    w, (wo, q4, s, pn) = _int4_matrix(N, K, n_out, 9920)
    X = S.activation(B, K, 9922, device="cuda")
    ref = qz.gemm_int4_outlier(w, X)
    torch.cuda.synchronize()
    y_ref, a_ref = O.int4o_product_ref(wo, q4, s, pn, n_out, K, X.cpu().numpy())
    tol = O.tolerance(y_ref, a_ref)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        Y = torch.full((B, N), float("nan"), dtype=torch.float16, device="cuda")
        assert _call(lib, w, X, Y, stream) == 0
        torch.cuda.synchronize()
        assert qz.device_error() == 0
        assert torch.equal(Y, ref), f"call {call} differs from the workspace entry point"
        err = np.abs(Y.float().cpu().numpy().astype(np.float64) - y_ref)
        assert (err <= tol).all(), f"call {call} outside the oracle bound"


def test_noalloc_call_captured_in_a_graph(lib):
    """After one ordinary call (which looks the scratch address up), a call
    captured in a CUDA graph and replayed twice matches the oracle."""
    import weight_only_quantized_dequant_gb300 as qz
    N, K, n_out, B = 700, 4096, 41, 16
    w, (wo, q4, s, pn) = _int4_matrix(N, K, n_out, 9930)
    X = S.activation(B, K, 9932, device="cuda")
    Y = torch.zeros((B, N), dtype=torch.float16, device="cuda")
    assert _call(lib, w, X, Y, torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    first = Y.clone()
    y_ref, a_ref = O.int4o_product_ref(wo, q4, s, pn, n_out, K, X.cpu().numpy())
    tol = O.tolerance(y_ref, a_ref)
    cs = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cs):
        st = _call(lib, w, X, Y, cs.cuda_stream)
    assert st == 0
    for rep in range(2):
        Y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert qz.device_error() == 0
        assert torch.equal(Y, first), f"replay {rep} differs from the uncaptured call"
        err = np.abs(Y.float().cpu().numpy().astype(np.float64) - y_ref)
        assert (err <= tol).all(), f"replay {rep} outside the oracle bound"


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    import weight_only_quantized_dequant_gb300 as qz
    # B = 64 at K = 57344 needs ~7.4 MB of gathered inputs plus ~10.5 MB of
    # partial tiles, beyond the 16 MiB array
    K, n_out, B = 57344, 574, 64
    assert lib.qz_gemm_workspace_bytes(B, K, n_out) > (16 << 20)
    W = S.weight(8, K, 9910, device="cuda")
    perm = torch.arange(K, dtype=torch.int32, device="cuda")
    w = qz.quantize_int4_outlier(W, perm, n_out)
    X = torch.zeros((B, K), dtype=torch.float16, device="cuda")
    Y = torch.zeros((B, 8), dtype=torch.float16, device="cuda")
    st = lib.qz_gemm_int4_outlier_noalloc(ctypes.byref(w.struct()), B, X.data_ptr(), K,
                                          Y.data_ptr(), 8, None)
    assert st == 3  # QZ_ERR_UNSUPPORTED, nothing enqueued
    # batch outside 1..QZ_MAX_BATCH: the statuses of qz_gemm_int4_outlier
    for b, want in ((0, 1), (-1, 1), (65, 3)):
        st = lib.qz_gemm_int4_outlier_noalloc(ctypes.byref(w.struct()), b, X.data_ptr(), K,
                                              Y.data_ptr(), 8, None)
        assert st == want, (b, st)
        st = lib.qz_gemm_int4_outlier(ctypes.byref(w.struct()), b, X.data_ptr(), K,
                                      Y.data_ptr(), 8, None, 0, None)
        assert st == want, (b, st)
