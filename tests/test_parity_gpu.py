"""CUDA path vs the CPU oracle, element by element, on seeded inputs.

Bit-exact: INT8 codes and scale, saliency sums, the permutation, INT4 codes,
row scales, outlier copies and every padding byte.  Products: within
|y - y_ref| <= 1e-3 * sum_j |w_ij x_j| + 1 fp16 ulp(y_ref), y_ref in fp64 on
the same reconstructed weights.
"""
import numpy as np
import pytest
import torch

from oracle import qz_oracle as O
from weight_only_quantized_dequant_gb300 import synthetic as S

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_only_quantized_dequant_gb300 import build
    build.build()


def qz():
    import weight_only_quantized_dequant_gb300 as m
    return m


def assert_close(y_gpu, y_ref, a_ref, what=""):
    y = y_gpu.float().cpu().numpy().astype(np.float64).reshape(y_ref.shape)
    tol = O.tolerance(y_ref, a_ref)
    err = np.abs(y - y_ref)
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())}/{bad.size} outside tolerance; "
                           f"worst err/tol {float((err / tol).max()):.3g}")
    return float((err / tol).max())


def padded_rows(X: torch.Tensor) -> torch.Tensor:
    """View of X whose rows start on 16-byte boundaries."""
    B, K = X.shape
    Kp = -(-K // 8) * 8
    buf = torch.zeros((B, Kp), dtype=X.dtype, device=X.device)
    buf[:, :K] = X
    return buf[:, :K]


# ----------------------------------------------------------------- INT8 ---
def test_tiny_int8_256():
    W, x = S.tiny_int8_inputs()
    w = qz().quantize_int8(W.to(DEV))
    y = qz().gemv_int8(w, x[0].to(DEV))
    q_ref, s_ref = O.int8_quantize(W.numpy())
    assert np.array_equal(w.q.cpu().numpy()[:, :256], q_ref)
    assert w.scale.item() == float(s_ref)
    y_ref, a_ref = O.int8_product_ref(q_ref, s_ref, x.numpy())
    assert_close(y, y_ref[0], a_ref[0], "tiny int8")


# (96, 14336): batch 1 at 20 warps per CTA; (100, 28672): at 16 (20 do not fit in
# shared memory); (8, 57344): staging too large, tensor cores at every batch
INT8_SHAPES = [(1, 1), (3, 34), (37, 100), (257, 1000), (1024, 4096), (96, 14336), (100, 28672),
               (8, 57344)]


@pytest.mark.parametrize("N,K", INT8_SHAPES)
def test_int8_quantize_bit_exact(N, K):
    W = S.weight(N, K, 1000 + N + K, device=DEV)
    w = qz().quantize_int8(W)
    q_ref, s_ref = O.int8_quantize(W.cpu().numpy())
    q = w.q.cpu().numpy()
    assert w.scale.item() == float(s_ref)
    assert np.array_equal(q[:, :K], q_ref)
    assert not q[:, K:].any()


BATCHES = [1, 2, 3, 4, 5, 8, 16, 24, 33, 64]


@pytest.mark.parametrize("N,K", INT8_SHAPES)
@pytest.mark.parametrize("B", BATCHES)
def test_int8_gemm(N, K, B):
    """B <= 4 on CUDA cores (tensor cores when the staged inputs do not fit
    in shared memory), B > 4 on the tensor cores."""
    W = S.weight(N, K, 2000 + N + K, device=DEV)
    X = padded_rows(S.activation(B, K, 3000 + B, device=DEV))
    w = qz().quantize_int8(W)
    Y = qz().gemv_int8(w, X[0]).unsqueeze(0) if B == 1 else qz().gemm_int8(w, X)
    assert qz().device_error() == 0
    q_ref, s_ref = O.int8_quantize(W.cpu().numpy())
    y_ref, a_ref = O.int8_product_ref(q_ref, s_ref, X.cpu().numpy())
    assert_close(Y, y_ref, a_ref, f"int8 N={N} K={K} B={B}")


def two_byte_aligned_rows(X: torch.Tensor) -> torch.Tensor:
    """Copy of X whose first row starts 2 bytes past a 16-byte boundary and
    whose rows are K + 1 fp16 apart (so no row is 16-byte aligned at K % 8 ==
    0): the inputs' fp16 alignment is all the interface promises."""
    B, K = X.shape
    buf = torch.zeros((B * (K + 1) + 8,), dtype=X.dtype, device=X.device)
    out = buf[1:1 + B * (K + 1)].view(B, K + 1)[:, :K]
    out.copy_(X)
    assert out.data_ptr() % 16 == 2
    return out


@pytest.mark.parametrize("N,K", [(37, 100), (257, 1000), (1024, 4096), (96, 14336)])
@pytest.mark.parametrize("B", [1, 3])
def test_int8_inputs_only_two_byte_aligned(N, K, B):
    """The GEMV reads inputs 16 bytes at a time where they are 16-byte aligned
    and element by element otherwise; both give the oracle's result."""
    W = S.weight(N, K, 2100 + N + K, device=DEV)
    X = two_byte_aligned_rows(S.activation(B, K, 3100 + B, device=DEV))
    w = qz().quantize_int8(W)
    Y = qz().gemv_int8(w, X[0]).unsqueeze(0) if B == 1 else qz().gemm_int8(w, X)
    assert qz().device_error() == 0
    q_ref, s_ref = O.int8_quantize(W.cpu().numpy())
    y_ref, a_ref = O.int8_product_ref(q_ref, s_ref, X.cpu().numpy())
    assert_close(Y, y_ref, a_ref, f"int8 2-byte-aligned x N={N} K={K} B={B}")


def test_int8_zero_matrix():
    W = torch.zeros((5, 40), dtype=torch.float16, device=DEV)
    w = qz().quantize_int8(W)
    assert w.scale.item() == 0.0 and not w.q.any()
    y = qz().gemv_int8(w, S.activation(1, 40, 5, device=DEV)[0])
    assert not y.float().abs().sum().item()


def test_int8_grouped_matches_separate():
    K = 3584
    Ns = [4096, 2048, 2048]
    Ws = [S.weight(n, K, 50 + i, device=DEV) for i, n in enumerate(Ns)]
    x = S.activation(1, K, 60, device=DEV)
    ws = [qz().quantize_int8(W) for W in Ws]
    ys = qz().gemv_int8_grouped(ws, x[0])
    for W, y in zip(Ws, ys):
        q_ref, s_ref = O.int8_quantize(W.cpu().numpy())
        y_ref, a_ref = O.int8_product_ref(q_ref, s_ref, x.cpu().numpy())
        assert_close(y, y_ref[0], a_ref[0], "grouped int8")


# ------------------------------------------------------- INT4 quantizer ---
@pytest.mark.parametrize("N,K", [(1, 1), (3, 34), (300, 1000), (700, 3072), (64, 28672)])
def test_saliency_exact(N, K):
    Ws = [S.weight(N, K, 70 + i, device=DEV) for i in range(2)]
    colsum = torch.zeros((K,), dtype=torch.int64, device=DEV)
    for W in Ws:
        qz().saliency_accumulate(W, colsum)
    ref = O.saliency_fixed([W.cpu().numpy() for W in Ws])
    assert np.array_equal(colsum.cpu().numpy(), ref)


@pytest.mark.parametrize("K", [1, 7, 300, 3072, 28672])
def test_select_outliers_exact_with_ties(K):
    g = torch.Generator().manual_seed(K)
    colsum = torch.randint(0, 6, (K,), generator=g, dtype=torch.int64)
    prof = torch.tensor([0.5, 1.0, -1.0, 2.0])[torch.randint(0, 4, (K,), generator=g)]
    for n_out in sorted({0, 1, (K + 99) // 100, K // 2, K}):
        perm = qz().select_outliers(colsum.to(DEV), prof.to(DEV), n_out)
        ref = O.select_outliers(colsum.numpy(), prof.numpy(), n_out)
        assert np.array_equal(perm.cpu().numpy(), ref), (K, n_out)


def test_select_outliers_realistic_profile():
    K, n_out = 11008, 111
    W = S.weight(512, K, 90, device=DEV)
    prof = S.x_profile(K, n_out, 91, device=DEV)
    colsum = torch.zeros((K,), dtype=torch.int64, device=DEV)
    qz().saliency_accumulate(W, colsum)
    perm = qz().select_outliers(colsum, prof, n_out)
    ref = O.select_outliers(O.saliency_fixed(W.cpu().numpy()), prof.cpu().numpy(), n_out)
    assert np.array_equal(perm.cpu().numpy(), ref)


def test_check_perm_flags():
    K = 1000
    p = torch.randperm(K, generator=torch.Generator().manual_seed(1)).to(torch.int32)
    assert qz().check_perm(p.to(DEV)) == 0
    dup = p.clone()
    dup[5] = dup[6]
    assert qz().check_perm(dup.to(DEV)) == 2
    oob = p.clone()
    oob[7] = K
    assert qz().check_perm(oob.to(DEV)) == 1
    neg = p.clone()
    neg[0] = -1
    assert qz().check_perm(neg.to(DEV)) == 1


INT4_SHAPES = [(1, 1, 0), (1, 1, 1), (3, 34, 1), (5, 34, 0), (7, 34, 34), (64, 520, 6),
               (300, 3072, 31), (129, 4096, 41), (64, 11008, 111), (16, 28672, 287),
               (8, 57344, 574)]


def _int4_inputs(N, K, n_out, seed):
    W = S.weight(N, K, seed, device=DEV)
    prof = S.x_profile(K, max(n_out, 0), seed + 1, device=DEV)
    colsum = torch.zeros((K,), dtype=torch.int64, device=DEV)
    qz().saliency_accumulate(W, colsum)
    perm = qz().select_outliers(colsum, prof, n_out)
    return W, prof, perm


@pytest.mark.parametrize("N,K,n_out", INT4_SHAPES)
def test_int4_quantize_bit_exact(N, K, n_out):
    W, prof, perm = _int4_inputs(N, K, n_out, 4000 + K + n_out)
    w = qz().quantize_int4_outlier(W, perm, n_out)
    Wn = W.cpu().numpy()
    perm_ref = O.select_outliers(O.saliency_fixed(Wn), prof.cpu().numpy(), n_out)
    assert np.array_equal(perm.cpu().numpy(), perm_ref)
    wo, q4, s = O.int4o_quantize(Wn, perm_ref, n_out)
    assert np.array_equal(w.w_out.cpu().numpy().view(np.uint16), wo.view(np.uint16))
    assert np.array_equal(w.q4.cpu().numpy(), q4)
    assert np.array_equal(w.scale.cpu().numpy().view(np.uint32), s.view(np.uint32))


@pytest.mark.parametrize("N,K,n_out", INT4_SHAPES)
@pytest.mark.parametrize("B", BATCHES)
def test_int4_gemm(N, K, n_out, B):
    W, prof, perm = _int4_inputs(N, K, n_out, 5000 + K + n_out)
    w = qz().quantize_int4_outlier(W, perm, n_out)
    X = padded_rows(S.activation(B, K, 6000 + B, device=DEV))
    Y = qz().gemv_int4_outlier(w, X[0]).unsqueeze(0) if B == 1 else qz().gemm_int4_outlier(w, X)
    assert qz().device_error() == 0
    wo, q4, s = O.int4o_quantize(W.cpu().numpy(), perm.cpu().numpy(), n_out)
    y_ref, a_ref = O.int4o_product_ref(wo, q4, s, perm.cpu().numpy(), n_out, K, X.cpu().numpy())
    assert_close(Y, y_ref, a_ref, f"int4 N={N} K={K} n_out={n_out} B={B}")


@pytest.mark.parametrize("N,K,n_out", [(64, 520, 6), (129, 4096, 41), (64, 11008, 111)])
@pytest.mark.parametrize("B", [1, 3, 16])
def test_int4_inputs_only_two_byte_aligned(N, K, n_out, B):
    """INT4 products with inputs at fp16 alignment only (see the INT8 case)."""
    W, prof, perm = _int4_inputs(N, K, n_out, 5100 + K + n_out)
    w = qz().quantize_int4_outlier(W, perm, n_out)
    X = two_byte_aligned_rows(S.activation(B, K, 6100 + B, device=DEV))
    Y = qz().gemv_int4_outlier(w, X[0]).unsqueeze(0) if B == 1 else qz().gemm_int4_outlier(w, X)
    assert qz().device_error() == 0
    wo, q4, s = O.int4o_quantize(W.cpu().numpy(), perm.cpu().numpy(), n_out)
    y_ref, a_ref = O.int4o_product_ref(wo, q4, s, perm.cpu().numpy(), n_out, K, X.cpu().numpy())
    assert_close(Y, y_ref, a_ref, f"int4 2-byte-aligned x N={N} K={K} n_out={n_out} B={B}")


def test_int4_grouped_matches_separate():
    K, n_out = 4096, 41
    Ns = [4096, 1024, 1024]
    Ws = [S.weight(n, K, 150 + i, device=DEV) for i, n in enumerate(Ns)]
    prof = S.x_profile(K, n_out, 160, device=DEV)
    colsum = torch.zeros((K,), dtype=torch.int64, device=DEV)
    for W in Ws:
        qz().saliency_accumulate(W, colsum)
    perm = qz().select_outliers(colsum, prof, n_out)
    ws = [qz().quantize_int4_outlier(W, perm, n_out) for W in Ws]
    x = S.activation(1, K, 170, device=DEV)
    ys = qz().gemv_int4_outlier_grouped(ws, x[0])
    pn = perm.cpu().numpy()
    for W, y in zip(Ws, ys):
        wo, q4, s = O.int4o_quantize(W.cpu().numpy(), pn, n_out)
        y_ref, a_ref = O.int4o_product_ref(wo, q4, s, pn, n_out, K, x.cpu().numpy())
        assert_close(y, y_ref[0], a_ref[0], "grouped int4")


@pytest.mark.parametrize("fmt", ["int8", "int4o"])
@pytest.mark.parametrize("B", [3, 16, 64])
def test_batched_grouped_matches_oracle(fmt, B):
    """One grouped batched call over 3 matrices of different heights sharing
    the input (and, for INT4, the permutation); outputs with padded strides
    of their own; every output against the oracle."""
    K, n_out = 1000, 10
    Ns = [300, 129, 64]
    Ws = [S.weight(n, K, 9500 + i, device=DEV) for i, n in enumerate(Ns)]
    X = padded_rows(S.activation(B, K, 9510 + B, device=DEV))
    Ys = [torch.full((B, n + 8 * (i + 1)), 3.0, dtype=torch.float16, device=DEV)[:, :n]
          for i, n in enumerate(Ns)]
    if fmt == "int8":
        ws = [qz().quantize_int8(W) for W in Ws]
        qz().gemm_int8_grouped(ws, X, Ys)
    else:
        prof = S.x_profile(K, n_out, 9520, device=DEV)
        colsum = torch.zeros((K,), dtype=torch.int64, device=DEV)
        for W in Ws:
            qz().saliency_accumulate(W, colsum)
        perm = qz().select_outliers(colsum, prof, n_out)
        ws = [qz().quantize_int4_outlier(W, perm, n_out) for W in Ws]
        qz().gemm_int4_outlier_grouped(ws, X, Ys)
    assert qz().device_error() == 0
    Xn = X.cpu().numpy()
    for i, (W, Y) in enumerate(zip(Ws, Ys)):
        Wn = W.cpu().numpy()
        if fmt == "int8":
            q_ref, s_ref = O.int8_quantize(Wn)
            y_ref, a_ref = O.int8_product_ref(q_ref, s_ref, Xn)
        else:
            pn = perm.cpu().numpy()
            wo, q4, s = O.int4o_quantize(Wn, pn, n_out)
            y_ref, a_ref = O.int4o_product_ref(wo, q4, s, pn, n_out, K, Xn)
        assert_close(Y, y_ref, a_ref, f"grouped {fmt} B={B} m={i}")
        full = Y.as_strided((B, Y.stride(0)), (Y.stride(0), 1)).cpu()
        assert (full[:, Ns[i]:] == 3.0).all()   # the padding of each row untouched


@pytest.mark.parametrize("fmt", ["int8", "int4o"])
@pytest.mark.parametrize("B", [5, 64])
def test_tensor_core_without_workspace(fmt, B):
    """The tensor-core kernel also works without a workspace (it gathers the
    permuted inputs itself and gives each CTA whole tiles).  Both forms are
    checked against the oracle and each repeats its own bits; they differ
    from each other only in the order in which fp32 partial sums are added."""
    N, K = 300, 3072
    X = S.activation(B, K, 9100 + B, device=DEV)
    if fmt == "int8":
        W = S.weight(N, K, 9101, device=DEV)
        w = qz().quantize_int8(W)
        run = lambda ws: qz().gemm_int8(w, X, workspace=ws)
        q_ref, s_ref = O.int8_quantize(W.cpu().numpy())
        y_ref, a_ref = O.int8_product_ref(q_ref, s_ref, X.cpu().numpy())
    else:
        W, prof, perm = _int4_inputs(N, K, 31, 9102)
        w = qz().quantize_int4_outlier(W, perm, 31)
        run = lambda ws: qz().gemm_int4_outlier(w, X, workspace=ws)
        pn = perm.cpu().numpy()
        wo, q4, s = O.int4o_quantize(W.cpu().numpy(), pn, 31)
        y_ref, a_ref = O.int4o_product_ref(wo, q4, s, pn, 31, K, X.cpu().numpy())
    for ws in (False, None):
        a = run(ws)
        b = run(ws)
        assert qz().device_error() == 0
        assert torch.equal(a, b), f"workspace={ws} not repeatable"
        assert_close(a, y_ref, a_ref, f"{fmt} B={B} workspace={ws}")


@pytest.mark.parametrize("B", [16, 64])
def test_tensor_core_grouped_large_int4(B):
    """q,k,v-sized grouped call (84 row tiles, ragged ends) at K = 4096: the
    persistent schedule cuts tiles between SMs, also across the matrix
    boundaries; every output of the three matrices against the oracle."""
    K, n_out = 4096, 41
    Ns = [4096, 4096 + 300, 2048 + 77]
    Ws = [S.weight(n, K, 9600 + i, device=DEV) for i, n in enumerate(Ns)]
    prof = S.x_profile(K, n_out, 9610, device=DEV)
    colsum = torch.zeros((K,), dtype=torch.int64, device=DEV)
    for W in Ws:
        qz().saliency_accumulate(W, colsum)
    perm = qz().select_outliers(colsum, prof, n_out)
    ws = [qz().quantize_int4_outlier(W, perm, n_out) for W in Ws]
    X = S.activation(B, K, 9620 + B, device=DEV)
    Ys = qz().gemm_int4_outlier_grouped(ws, X)
    assert qz().device_error() == 0
    pn = perm.cpu().numpy()
    Xn = X.cpu().numpy()
    for i, (W, Y) in enumerate(zip(Ws, Ys)):
        wo, q4, s = O.int4o_quantize(W.cpu().numpy(), pn, n_out)
        y_ref, a_ref = O.int4o_product_ref(wo, q4, s, pn, n_out, K, Xn)
        assert_close(Y, y_ref, a_ref, f"grouped int4 large B={B} m={i}")


@pytest.mark.parametrize("B", [16, 64])
def test_tensor_core_grouped_large_int8(B):
    """gate,up-sized grouped INT8 call (225 row tiles, ragged ends, K = 3584):
    every output against the oracle."""
    K = 3584
    Ns = [14336 - 77, 14336 + 45]
    Ws = [S.weight(n, K, 9700 + i, device=DEV) for i, n in enumerate(Ns)]
    ws = [qz().quantize_int8(W) for W in Ws]
    X = S.activation(B, K, 9720 + B, device=DEV)
    Ys = qz().gemm_int8_grouped(ws, X)
    assert qz().device_error() == 0
    Xn = X.cpu().numpy()
    for i, (W, Y) in enumerate(zip(Ws, Ys)):
        q_ref, s_ref = O.int8_quantize(W.cpu().numpy())
        y_ref, a_ref = O.int8_product_ref(q_ref, s_ref, Xn)
        assert_close(Y, y_ref, a_ref, f"grouped int8 large B={B} m={i}")


def test_tensor_core_workspace_validation():
    """A workspace one byte short, or not 16-byte aligned, is refused before
    anything is enqueued (the output stays untouched); the exact size works."""
    import ctypes
    from weight_only_quantized_dequant_gb300 import _lib
    lib = _lib.load()
    N, K, B = 300, 1024, 16
    w = qz().quantize_int8(S.weight(N, K, 9170, device=DEV))
    X = S.activation(B, K, 9171, device=DEV)
    need = qz().gemm_workspace_bytes(B, K, 0)
    ws = torch.empty((need + 32,), dtype=torch.uint8, device=DEV)
    Y = torch.full((B, N), 7.0, dtype=torch.float16, device=DEV)
    f = lib.qz_gemm_int8
    st = f(ctypes.byref(w.struct()), B, X.data_ptr(), K, Y.data_ptr(), N, ws.data_ptr(),
           need - 1, None)
    assert st == 1  # QZ_ERR_INVALID_ARG
    st = f(ctypes.byref(w.struct()), B, X.data_ptr(), K, Y.data_ptr(), N, ws.data_ptr() + 8,
           need, None)
    assert st == 2  # QZ_ERR_ALIGNMENT
    torch.cuda.synchronize()
    assert (Y == 7.0).all()
    st = f(ctypes.byref(w.struct()), B, X.data_ptr(), K, Y.data_ptr(), N, ws.data_ptr(), need,
           None)
    assert st == 0
    torch.cuda.synchronize()
    assert qz().device_error() == 0
    ref = qz().gemm_int8(w, X)  # the same call through the binding
    assert torch.equal(Y, ref)


@pytest.mark.parametrize("fmt", ["int8", "int4o"])
def test_tensor_core_more_tiles_than_sms_without_workspace(fmt):
    """160 row tiles and no workspace: persistent CTAs take whole tiles, some
    two in a row (the accumulators alternate), every output checked."""
    N, K, B, n_out = 160 * 128 - 37, 1024, 16, 11
    X = S.activation(B, K, 9160, device=DEV)
    if fmt == "int8":
        W = S.weight(N, K, 9161, device=DEV)
        w = qz().quantize_int8(W)
        Y = qz().gemm_int8(w, X, workspace=False)
        q_ref, s_ref = O.int8_quantize(W.cpu().numpy())
        y_ref, a_ref = O.int8_product_ref(q_ref, s_ref, X.cpu().numpy())
    else:
        W, prof, perm = _int4_inputs(N, K, n_out, 9162)
        w = qz().quantize_int4_outlier(W, perm, n_out)
        Y = qz().gemm_int4_outlier(w, X, workspace=False)
        pn = perm.cpu().numpy()
        wo, q4, s = O.int4o_quantize(W.cpu().numpy(), pn, n_out)
        y_ref, a_ref = O.int4o_product_ref(wo, q4, s, pn, n_out, K, X.cpu().numpy())
    assert qz().device_error() == 0
    assert_close(Y, y_ref, a_ref, f"{fmt} 160 tiles, no workspace")


@pytest.mark.parametrize("fmt", ["int8", "int4o"])
def test_tensor_core_one_tile_cut_between_many_ctas(fmt):
    """One ragged 128-row tile at K = 28672: its K tiles are cut between
    dozens of CTAs and the last to arrive adds all their partials.  Two
    calls on one workspace give the same bits (the counters restart)."""
    N, K, B, n_out = 100, 28672, 16, 287
    X = S.activation(B, K, 9150, device=DEV)
    if fmt == "int8":
        W = S.weight(N, K, 9151, device=DEV)
        w = qz().quantize_int8(W)
        ws = torch.empty((qz().gemm_workspace_bytes(B, K, 0),), dtype=torch.uint8, device=DEV)
        run = lambda: qz().gemm_int8(w, X, workspace=ws)
        q_ref, s_ref = O.int8_quantize(W.cpu().numpy())
        y_ref, a_ref = O.int8_product_ref(q_ref, s_ref, X.cpu().numpy())
    else:
        W, prof, perm = _int4_inputs(N, K, n_out, 9152)
        w = qz().quantize_int4_outlier(W, perm, n_out)
        ws = torch.empty((qz().gemm_workspace_bytes(B, K, n_out),), dtype=torch.uint8, device=DEV)
        run = lambda: qz().gemm_int4_outlier(w, X, workspace=ws)
        pn = perm.cpu().numpy()
        wo, q4, s = O.int4o_quantize(W.cpu().numpy(), pn, n_out)
        y_ref, a_ref = O.int4o_product_ref(wo, q4, s, pn, n_out, K, X.cpu().numpy())
    a = run()
    b = run()
    assert qz().device_error() == 0
    assert torch.equal(a, b)
    assert_close(a, y_ref, a_ref, f"{fmt} one tile cut")


def test_tensor_core_7b_batch64_full_matrix():
    """The 7B gate projection (11008 x 4096) at batch 64 on the tensor
    cores, every output checked."""
    N, K, n_out, B = 11008, 4096, 41, 64
    W, prof, perm = _int4_inputs(N, K, n_out, 8800)
    w = qz().quantize_int4_outlier(W, perm, n_out)
    X = S.activation(B, K, 8801, device=DEV)
    Y = qz().gemm_int4_outlier(w, X)
    assert qz().device_error() == 0
    wo, q4, s = O.int4o_quantize(W.cpu().numpy(), perm.cpu().numpy(), n_out)
    y_ref, a_ref = O.int4o_product_ref(wo, q4, s, perm.cpu().numpy(), n_out, K, X.cpu().numpy())
    assert_close(Y, y_ref, a_ref, "7b gate b64")


# ------------------------------------------------------ launch overlap ----
def test_overlap_graph_matches_plain_launches():
    """A decode step captured with programmatic dependent launch gives the
    same bits as plain launches, for both formats (two layers each)."""
    import weight_only_quantized_dequant_gb300 as m
    from weight_only_quantized_dequant_gb300 import stack as ST
    for name in ("gemma2_9b_int8", "llama_7b_int4o"):
        st = ST.LayerStack(S.WORKLOADS[name], layers=2)
        st.run_step()
        torch.cuda.synchronize()
        ref = [y.clone() for ys in st.y for yy in ys for y in yy]
        for y in [y for ys in st.y for yy in ys for y in yy]:
            y.fill_(0)
        g = st.capture(overlap=True)
        for y in [y for ys in st.y for yy in ys for y in yy]:
            y.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        got = [y for ys in st.y for yy in ys for y in yy]
        assert all(torch.equal(a, b) for a, b in zip(ref, got)), name
    assert m.get_overlap() is False


# --------------------------------------------------- full-size matrices ---
@pytest.mark.slow
def test_full_gemma_layer_int8():
    """Every matrix of one Gemma-2-9B-shaped layer: codes bit-exact and the
    grouped launches of the decode step within tolerance."""
    wl = S.WORKLOADS["gemma2_9b_int8"]
    mats = {}
    for m in S.MATS:
        N, K = wl.shape(m)
        W = S.weight(N, K, S.matrix_seed(wl, 0, m), device=DEV)
        mats[m] = (W, qz().quantize_int8(W))
    for g, names in enumerate(S.GROUPS):
        K = wl.shape(names[0])[1]
        x = S.activation(1, K, S.input_seed(wl, 0, g), device=DEV)
        ys = qz().gemv_int8_grouped([mats[m][1] for m in names], x[0])
        for m, y in zip(names, ys):
            W, w = mats[m]
            q_ref, s_ref = O.int8_quantize(W.cpu().numpy())
            assert w.scale.item() == float(s_ref)
            assert np.array_equal(w.q.cpu().numpy()[:, :K], q_ref)
            y_ref, a_ref = O.int8_product_ref(q_ref, s_ref, x.cpu().numpy())
            assert_close(y, y_ref[0], a_ref[0], f"gemma {m}")


@pytest.mark.slow
def test_full_70b_down_proj_int4_sampled():
    """The largest matrix (8192 x 28672): saliency and permutation exact over
    the whole matrix; codes and outputs checked on 64 sampled rows."""
    N, K = 8192, 28672
    n_out = O.default_n_out(K)
    W = S.weight(N, K, 77, device=DEV)
    prof = S.x_profile(K, n_out, 78, device=DEV)
    colsum = torch.zeros((K,), dtype=torch.int64, device=DEV)
    qz().saliency_accumulate(W, colsum)
    perm = qz().select_outliers(colsum, prof, n_out)
    w = qz().quantize_int4_outlier(W, perm, n_out)
    x = S.activation(1, K, 79, device=DEV)
    y = qz().gemv_int4_outlier(w, x[0])
    Wn = W.cpu().numpy()
    assert np.array_equal(colsum.cpu().numpy(), O.saliency_fixed(Wn))
    pn = O.select_outliers(O.saliency_fixed(Wn), prof.cpu().numpy(), n_out)
    assert np.array_equal(perm.cpu().numpy(), pn)
    rows = np.random.default_rng(0).choice(N, 64, replace=False)
    wo, q4, s = O.int4o_quantize(Wn[rows], pn, n_out)
    assert np.array_equal(w.q4.cpu().numpy()[rows], q4)
    assert np.array_equal(w.w_out.cpu().numpy()[rows].view(np.uint16), wo.view(np.uint16))
    assert np.array_equal(w.scale.cpu().numpy()[rows], s)
    y_ref, a_ref = O.int4o_product_ref(wo, q4, s, pn, n_out, K, x.cpu().numpy())
    assert_close(y[rows], y_ref[0], a_ref[0], "70b down sampled")


@pytest.mark.slow
def test_full_70b_gate_up_grouped_int4_sampled():
    """The largest batch-1 launch of the 70B layer: gate and up (2 x 28672 x
    8192, one permutation table from both matrices' saliency) in one grouped
    call.  Saliency and permutation exact; codes and outputs checked on 64
    sampled rows of each matrix plus the rows at both ends."""
    N, K = 28672, 8192
    n_out = O.default_n_out(K)
    Ws = [S.weight(N, K, 81 + i, device=DEV) for i in range(2)]
    prof = S.x_profile(K, n_out, 83, device=DEV)
    colsum = torch.zeros((K,), dtype=torch.int64, device=DEV)
    for W in Ws:
        qz().saliency_accumulate(W, colsum)
    perm = qz().select_outliers(colsum, prof, n_out)
    ws = [qz().quantize_int4_outlier(W, perm, n_out) for W in Ws]
    x = S.activation(1, K, 84, device=DEV)
    ys = qz().gemv_int4_outlier_grouped(ws, x[0])
    assert qz().device_error() == 0
    sal = sum(O.saliency_fixed(W.cpu().numpy()) for W in Ws)
    assert np.array_equal(colsum.cpu().numpy(), sal)
    pn = O.select_outliers(sal, prof.cpu().numpy(), n_out)
    assert np.array_equal(perm.cpu().numpy(), pn)
    rng = np.random.default_rng(1)
    for i, (W, w, y) in enumerate(zip(Ws, ws, ys)):
        rows = np.unique(np.concatenate([rng.choice(N, 64, replace=False),
                                         [0, 1, 15, 16, N - 17, N - 16, N - 1]]))
        wo, q4, sc = O.int4o_quantize(W[torch.from_numpy(rows).to(DEV)].cpu().numpy(), pn, n_out)
        assert np.array_equal(w.q4.cpu().numpy()[rows], q4)
        assert np.array_equal(w.scale.cpu().numpy()[rows], sc)
        y_ref, a_ref = O.int4o_product_ref(wo, q4, sc, pn, n_out, K, x.cpu().numpy())
        assert_close(y[rows], y_ref[0], a_ref[0], f"70b gate+up sampled m={i}")


def test_full_70b_gate_up_grouped_int8_sampled():
    """The largest batch-1 launch of the 70B-shaped INT8 stack: gate and up
    (2 x 28672 x 8192) in one grouped call.  The per-tensor scale and the
    codes of sampled rows against the oracle quantizer run on each whole
    matrix; outputs on 64 sampled rows of each matrix plus the rows at both
    ends."""
    N, K = 28672, 8192
    Ws = [S.weight(N, K, 91 + i, device=DEV) for i in range(2)]
    ws = [qz().quantize_int8(W) for W in Ws]
    x = S.activation(1, K, 94, device=DEV)
    ys = qz().gemv_int8_grouped(ws, x[0])
    assert qz().device_error() == 0
    rng = np.random.default_rng(2)
    for i, (W, w, y) in enumerate(zip(Ws, ws, ys)):
        q_ref, s_ref = O.int8_quantize(W.cpu().numpy())
        assert w.scale.item() == float(s_ref)
        rows = np.unique(np.concatenate([rng.choice(N, 64, replace=False),
                                         [0, 1, 15, 16, N - 17, N - 16, N - 1]]))
        q_rows = w.q[torch.from_numpy(rows).to(DEV)].cpu().numpy()[:, :K]
        assert np.array_equal(q_rows, q_ref[rows])
        y_ref, a_ref = O.int8_product_ref(q_ref[rows], s_ref, x.cpu().numpy())
        assert_close(y[rows], y_ref[0], a_ref[0], f"70b int8 gate+up sampled m={i}")


@pytest.mark.parametrize("fmt,Ns,K,n_out", [("int4o", [7300, 7301], 3000, 31),
                                             ("int4o", [14600], 8200, 83),
                                             ("int8", [14593], 1000, 0),
                                             ("int8", [7000, 7601], 4100, 0)])
def test_batch1_many_rows_against_oracle(fmt, Ns, K, n_out):
    """Batch-1 grouped launches with many rows per CTA (97): ragged row
    pairs and ring stages, rows not a multiple of a ring stage, an odd
    outlier count, two matrices in one launch; every output against the
    oracle."""
    Ws = [S.weight(n, K, 9950 + i + K, device=DEV) for i, n in enumerate(Ns)]
    x = S.activation(1, K, 9960 + K, device=DEV)
    if fmt == "int8":
        ws = [qz().quantize_int8(W) for W in Ws]
        ys = qz().gemv_int8_grouped(ws, x[0])
    else:
        prof = S.x_profile(K, n_out, 9970 + K, device=DEV)
        colsum = torch.zeros((K,), dtype=torch.int64, device=DEV)
        for W in Ws:
            qz().saliency_accumulate(W, colsum)
        perm = qz().select_outliers(colsum, prof, n_out)
        ws = [qz().quantize_int4_outlier(W, perm, n_out) for W in Ws]
        ys = qz().gemv_int4_outlier_grouped(ws, x[0])
    assert qz().device_error() == 0
    xn = x.cpu().numpy()
    for i, (W, y) in enumerate(zip(Ws, ys)):
        Wn = W.cpu().numpy()
        if fmt == "int8":
            q_ref, s_ref = O.int8_quantize(Wn)
            y_ref, a_ref = O.int8_product_ref(q_ref, s_ref, xn)
        else:
            pn = perm.cpu().numpy()
            wo, q4, sc = O.int4o_quantize(Wn, pn, n_out)
            y_ref, a_ref = O.int4o_product_ref(wo, q4, sc, pn, n_out, K, xn)
        assert_close(y, y_ref[0], a_ref[0], f"many rows {fmt} K={K} m={i}")


# ----------------------------------------------------------------- pager ---
def test_pager_streams_layers_and_reports_injected_failure():
    import weight_only_quantized_dequant_gb300 as m
    K, N, L = 1024, 512, 5
    ws, hosts = [], []
    for l in range(L):
        W = S.weight(N, K, 300 + l, device=DEV)
        w = m.quantize_int8(W)
        ws.append(w)
        # one packed layer = q bytes then the scale, padded to 16 bytes
        blob = torch.zeros((N * w.ldq + 16,), dtype=torch.uint8)
        blob[: N * w.ldq] = w.q.cpu().view(torch.uint8).reshape(-1)
        blob[N * w.ldq: N * w.ldq + 4] = w.scale.cpu().view(torch.uint8)
        hosts.append(blob.pin_memory())
    slots = [torch.empty((hosts[0].numel(),), dtype=torch.uint8, device=DEV) for _ in range(2)]
    copy_s, comp_s = torch.cuda.Stream(), torch.cuda.Stream()
    x = S.activation(1, K, 400, device=DEV)[0]
    ref = [m.gemv_int8(w, x) for w in ws]
    torch.cuda.synchronize()
    # the oracle's product of each layer, from the seeded fp16 weights
    oref = []
    for l in range(L):
        q_ref, s_ref = O.int8_quantize(S.weight(N, K, 300 + l, device=DEV).cpu().numpy())
        oref.append(O.int8_product_ref(q_ref, s_ref, x.cpu().numpy()[None]))
    pager = m.Pager(hosts, slots, copy_s, comp_s)
    outs = [torch.empty((N,), dtype=torch.float16, device=DEV) for _ in range(L)]
    for rnd in range(2):
        for l in range(L):
            ptr = pager.acquire(l)
            slot = slots[0] if ptr == slots[0].data_ptr() else slots[1]
            assert ptr in (slots[0].data_ptr(), slots[1].data_ptr())
            wq = m.Int8Matrix(slot[: N * ws[l].ldq].view(torch.int8).view(N, ws[l].ldq),
                              slot[N * ws[l].ldq: N * ws[l].ldq + 4].view(torch.float32), N, K)
            with torch.cuda.stream(comp_s):
                m.gemv_int8(wq, x, outs[l], stream=comp_s)
            pager.release(l)
        comp_s.synchronize()
        for l in range(L):
            assert_close(outs[l], oref[l][0][0], oref[l][1][0], f"paged layer {l} pass {rnd}")
            assert torch.equal(outs[l], ref[l]), (rnd, l)
    # host-side injected copy failure: acquire reports QZ_ERR_IO, nothing hangs
    pager.inject_copy_failure(2)
    with pytest.raises(m.QzError) as ei:
        for l in range(L):
            pager.acquire(l)
            pager.release(l)
    assert ei.value.name == "QZ_ERR_IO"
    pager.close()
    torch.cuda.synchronize()


# ----------------------------------------------------- sequence launches ----
@pytest.mark.parametrize("fmt", ["int8", "int4o"])
def test_sequence_chain_against_oracle(fmt):
    """Three dependent products in one launch, each reading the previous
    one's output: every product against the oracle on the inputs it read
    (x0, then the launch's own y0, then y1); the barrier word left at zero and
    reusable; the separate grouped calls agree within the same bound."""
    K0, N0, N1, N2 = 3072, 1536, 1024, 700
    shapes = [(N0, K0), (N1, N0), (N2, N1), (N2 + 64, N1)]
    Ws = [S.weight(n, k, 9900 + i, device=DEV) for i, (n, k) in enumerate(shapes)]
    x0 = S.activation(1, K0, 9910, device=DEV)[0]
    if fmt == "int8":
        ws = [qz().quantize_int8(W) for W in Ws]
        grouped = qz().gemv_int8_grouped
    else:
        ws = []
        perms = {}
        for i, W in enumerate(Ws):
            K = W.shape[1]
            n_out = O.default_n_out(K)
            key = (K, i >= 2)              # products 2 and 3 share one permutation
            if key not in perms:
                colsum = torch.zeros((K,), dtype=torch.int64, device=DEV)
                for j in ([2, 3] if i >= 2 else [i]):
                    qz().saliency_accumulate(Ws[j], colsum)
                perms[key] = qz().select_outliers(colsum, S.x_profile(K, n_out, 9920 + i,
                                                                      device=DEV), n_out)
            ws.append(qz().quantize_int4_outlier(W, perms[key], n_out))
        grouped = qz().gemv_int4_outlier_grouped
    # chain: y0 = W0 x0; y1 = W1 y0; (y2, y3) = (W2, W3) y1
    y0 = torch.empty((N0,), dtype=torch.float16, device=DEV)
    y1 = torch.empty((N1,), dtype=torch.float16, device=DEV)
    y2 = torch.empty((N2,), dtype=torch.float16, device=DEV)
    y3 = torch.empty((N2 + 64,), dtype=torch.float16, device=DEV)
    sync = torch.zeros((1,), dtype=torch.int32, device=DEV)
    for _ in range(2):                      # the second call reuses the barrier word
        qz().gemv_sequence([[ws[0]], [ws[1]], [ws[2], ws[3]]], [x0, y0, y1],
                           [[y0], [y1], [y2, y3]], sync=sync)
        assert qz().device_error() == 0
        assert int(sync.item()) == 0

    def ref(i, x):
        Wn, xn = Ws[i].cpu().numpy(), x.cpu().numpy()[None]
        if fmt == "int8":
            q_ref, s_ref = O.int8_quantize(Wn)
            return O.int8_product_ref(q_ref, s_ref, xn)
        pn = ws[i].perm.cpu().numpy()
        wo, q4, s = O.int4o_quantize(Wn, pn, ws[i].n_out)
        return O.int4o_product_ref(wo, q4, s, pn, ws[i].n_out, Wn.shape[1], xn)

    for i, (y, x) in enumerate(((y0, x0), (y1, y0), (y2, y1), (y3, y1))):
        y_ref, a_ref = ref(i, x)
        assert_close(y, y_ref[0], a_ref[0], f"sequence {fmt} product {i}")
    # the separate grouped calls on the same inputs: within the bound too
    r0 = grouped([ws[0]], x0)[0]
    r1 = grouped([ws[1]], y0)[0]
    r2, r3 = grouped([ws[2], ws[3]], y1)
    for i, (r, x) in enumerate(((r0, x0), (r1, y0), (r2, y1), (r3, y1))):
        y_ref, a_ref = ref(i, x)
        assert_close(r, y_ref[0], a_ref[0], f"grouped {fmt} product {i}")
