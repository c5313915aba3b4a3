"""Zero-copy products: weights in pinned host memory read in place by the GPU
(the pages' pinned pool reached by zero-copy DMA).  Same bits as the
device-resident launch, and within the oracle's bound."""
import ctypes

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
    bad = np.abs(y - y_ref) > tol
    assert not bad.any(), f"{what}: {int(bad.sum())}/{bad.size} outside tolerance"


def _pinned(t: torch.Tensor) -> torch.Tensor:
    return t.cpu().pin_memory()


def test_int8_grouped_from_pinned_host():
    K, Ns = 3584, [4096, 2048, 2048]
    Ws = [S.weight(n, K, 9600 + i, device=DEV) for i, n in enumerate(Ns)]
    dev = [qz().quantize_int8(W) for W in Ws]
    host = [qz().Int8Matrix(_pinned(w.q), _pinned(w.scale), w.N, w.K) for w in dev]
    x = S.activation(1, K, 9610, device=DEV)[0]
    y_dev = qz().gemv_int8_grouped(dev, x)
    y_map = qz().gemv_mapped(host, x)
    y_dmap = qz().gemv_mapped(dev, x)          # device tensors through the same entry
    assert qz().device_error() == 0
    for i, W in enumerate(Ws):
        assert torch.equal(y_map[i], y_dev[i]) and torch.equal(y_dmap[i], y_dev[i])
        q_ref, s_ref = O.int8_quantize(W.cpu().numpy())
        y_ref, a_ref = O.int8_product_ref(q_ref, s_ref, x.cpu().numpy()[None])
        assert_close(y_map[i], y_ref[0], a_ref[0], f"mapped int8 m={i}")


@pytest.mark.parametrize("K,n_out", [(3072, 31), (8192, 82), (1000, 0)])
def test_int4_grouped_from_pinned_host(K, n_out):
    Ns = [1024, 1536]
    Ws = [S.weight(n, K, 9700 + i + K, device=DEV) for i, n in enumerate(Ns)]
    colsum = torch.zeros((K,), dtype=torch.int64, device=DEV)
    for W in Ws:
        qz().saliency_accumulate(W, colsum)
    perm = qz().select_outliers(colsum, S.x_profile(K, n_out, 9710, device=DEV), n_out)
    dev = [qz().quantize_int4_outlier(W, perm, n_out) for W in Ws]
    hperm = _pinned(perm)
    host = [qz().Int4oMatrix(hperm, _pinned(w.w_out), _pinned(w.q4), _pinned(w.scale),
                             w.N, w.K, w.n_out) for w in dev]
    x = S.activation(1, K, 9720, device=DEV)[0]
    y_dev = qz().gemv_int4_outlier_grouped(dev, x)
    y_map = qz().gemv_mapped(host, x)
    y_dmap = qz().gemv_mapped(dev, x)          # device tensors through the same entry
    assert qz().device_error() == 0
    assert all(torch.equal(a, b) for a, b in zip(y_dmap, y_dev))
    pn = perm.cpu().numpy()
    for i, W in enumerate(Ws):
        assert torch.equal(y_map[i], y_dev[i])
        wo, q4, s = O.int4o_quantize(W.cpu().numpy(), pn, n_out)
        y_ref, a_ref = O.int4o_product_ref(wo, q4, s, pn, n_out, K, x.cpu().numpy()[None])
        assert_close(y_map[i], y_ref[0], a_ref[0], f"mapped int4 K={K} m={i}")


def test_pageable_host_weights_are_refused():
    from weight_only_quantized_dequant_gb300 import _lib
    K, N = 256, 64
    w = qz().quantize_int8(S.weight(N, K, 9800, device=DEV))
    q_pageable = w.q.cpu()                      # not pinned
    with pytest.raises(ValueError):
        qz().gemv_mapped([qz().Int8Matrix(q_pageable, _pinned(w.scale), N, K)],
                         torch.zeros((K,), dtype=torch.float16, device=DEV))
    # the C ABI itself refuses it too (no launch)
    lib = _lib.load()
    ws = (_lib.Int8Weight * 1)(_lib.Int8Weight(q_pageable.data_ptr(), w.scale.data_ptr(),
                                               N, K, q_pageable.stride(0)))
    y = torch.empty((N,), dtype=torch.float16, device=DEV)
    x = torch.zeros((K,), dtype=torch.float16, device=DEV)
    ys = (ctypes.c_void_p * 1)(y.data_ptr())
    assert lib.qz_gemv_int8_grouped_mapped(ws, 1, x.data_ptr(), ys, None) == 1  # INVALID_ARG
