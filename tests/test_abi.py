"""The C ABI on the host: the library loads, exports every function that
include/qz.h declares, and validates arguments before touching the GPU.
No GPU needed (no call here reaches a launch)."""
import ctypes
import os
import re

import pytest

from oracle import qz_oracle as O
from weight_only_quantized_dequant_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qz.h")

OK, INVAL, ALIGN, UNSUP = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_lib.LIB_PATH):
        from weight_only_quantized_dequant_gb300 import build
        build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qz_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ["qz_quantize_int8", "qz_gemv_int8", "qz_gemm_int8", "qz_gemv_int8_grouped",
                 "qz_int4o_layout", "qz_saliency_accumulate", "qz_select_outliers",
                 "qz_check_perm", "qz_quantize_int4_outlier", "qz_gemv_int4_outlier",
                 "qz_gemm_int4_outlier", "qz_gemv_int4_outlier_grouped", "qz_pager_create",
                 "qz_pager_acquire", "qz_pager_release", "qz_pager_destroy"]:
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding knows every one of them
    assert set(declared_functions()) <= set(_lib._SIGS)


def test_struct_layouts():
    assert ctypes.sizeof(_lib.Int8Weight) == 40
    assert ctypes.sizeof(_lib.Int4oWeight) == 72


def test_overlap_setting_is_per_thread_and_validated(lib):
    import threading
    assert lib.qz_get_overlap() == 0
    assert lib.qz_set_overlap(2) == INVAL
    assert lib.qz_set_overlap(1) == OK and lib.qz_get_overlap() == 1
    seen = []
    t = threading.Thread(target=lambda: seen.append(lib.qz_get_overlap()))
    t.start()
    t.join()
    assert seen == [0]
    assert lib.qz_set_overlap(0) == OK and lib.qz_get_overlap() == 0


def test_workspace_bytes(lib):
    # ceil(n_out/128) + ceil((K-n_out)/128) tiles of Np x 128 fp16 (Np = B
    # rounded up to 16), then fp32 partials of two 128-row tiles for each of
    # at most 160 CTAs, then 160 x 4 arrival counters
    def extra(Np):
        return 2 * 160 * Np * 128 * 4 + 160 * 4 * 4
    assert lib.qz_gemm_workspace_bytes(64, 4096, 41) == (1 + 32) * 64 * 128 * 2 + extra(64)
    assert lib.qz_gemm_workspace_bytes(5, 100, 0) == 1 * 16 * 128 * 2 + extra(16)
    assert lib.qz_gemm_workspace_bytes(5, 300, 0) == 3 * 16 * 128 * 2 + extra(16)
    assert lib.qz_gemm_workspace_bytes(33, 300, 0) == 3 * 48 * 128 * 2 + extra(48)
    assert lib.qz_gemm_workspace_bytes(65, 100, 0) == 0
    assert lib.qz_gemm_workspace_bytes(1, 100, 101) == 0


def test_version_and_status_strings(lib):
    assert lib.qz_version() >= 10000
    for code, name in _lib.STATUS.items():
        assert lib.qz_status_string(code).decode() == name
    assert lib.qz_status_string(99).decode() == "QZ_ERR_UNKNOWN"


@pytest.mark.parametrize("K,n_out", [(1, 0), (1, 1), (34, 1), (3072, 31), (4096, 41),
                                     (8192, 82), (11008, 111), (28672, 287), (57344, 574)])
def test_layout_matches_oracle(lib, K, n_out):
    a, b = ctypes.c_int64(), ctypes.c_int64()
    assert lib.qz_int4o_layout(7, K, n_out, ctypes.byref(a), ctypes.byref(b)) == OK
    assert (a.value, b.value) == O.int4o_layout(K, n_out)


def test_layout_rejects_bad_sizes(lib):
    a, b = ctypes.c_int64(), ctypes.c_int64()
    assert lib.qz_int4o_layout(7, 10, 11, ctypes.byref(a), ctypes.byref(b)) == INVAL
    assert lib.qz_int4o_layout(0, 10, 1, ctypes.byref(a), ctypes.byref(b)) == INVAL
    assert lib.qz_int4o_layout(7, 10, -1, ctypes.byref(a), ctypes.byref(b)) == INVAL
    assert lib.qz_int4o_layout(7, 10, 1, None, ctypes.byref(b)) == INVAL


# Fake device addresses: validation only inspects their values.
P = 0x10000  # 16-byte aligned
PU = 0x10008  # 8-byte aligned only


def test_quantize_int8_validation(lib):
    f = lib.qz_quantize_int8
    assert f(None, 4, 16, 16, P, 16, P, None) == INVAL
    assert f(P, 4, 16, 8, P, 16, P, None) == INVAL            # ldw < K
    assert f(P, 4, 16, 16, P, 16, None, None) == INVAL        # no scale
    assert f(PU, 4, 16, 16, P, 16, P, None) == ALIGN          # W misaligned
    assert f(P, 4, 16, 20, P, 16, P, None) == ALIGN           # ldw*2 % 16
    assert f(P, 4, 16, 16, P, 24, P, None) == ALIGN           # ldq % 16
    assert f(P, 0, 16, 16, P, 16, P, None) == INVAL


def _w8(N=8, K=32, ldq=32, q=P, scale=P):
    return _lib.Int8Weight(q, scale, N, K, ldq)


def test_gemv_int8_validation(lib):
    w = _w8()
    assert lib.qz_gemv_int8(None, P, P, None) == INVAL
    assert lib.qz_gemv_int8(ctypes.byref(w), None, P, None) == INVAL
    assert lib.qz_gemv_int8(ctypes.byref(w), P, None, None) == INVAL
    assert lib.qz_gemv_int8(ctypes.byref(w), P + 1, P, None) == ALIGN     # odd fp16 pointer
    assert lib.qz_gemv_int8(ctypes.byref(_w8(ldq=40)), P, P, None) == ALIGN
    assert lib.qz_gemv_int8(ctypes.byref(_w8(ldq=16)), P, P, None) == INVAL
    assert lib.qz_gemv_int8(ctypes.byref(_w8(K=57360, ldq=57360)), P, P, None) == UNSUP
    assert lib.qz_gemm_int8(ctypes.byref(w), 65, P, 32, P, 8, None, 0, None) == UNSUP
    assert lib.qz_gemm_int8(ctypes.byref(w), 0, P, 32, P, 8, None, 0, None) == INVAL
    assert lib.qz_gemm_int8(ctypes.byref(w), 2, P, 16, P, 8, None, 0, None) == INVAL  # ldx < K
    assert lib.qz_gemm_int8(ctypes.byref(w), 2, P, 32, P + 1, 8, None, 0, None) == ALIGN


def test_embed_int8_validation(lib):
    w = _w8()                                     # V = 8 rows of K = 32
    E = lib.qz_embed_int8
    assert E(None, P, 1, P, 32, None) == INVAL
    assert E(ctypes.byref(w), P, -1, P, 32, None) == INVAL
    assert E(ctypes.byref(w), None, 0, None, 0, None) == OK       # B = 0: nothing to do
    assert E(ctypes.byref(w), None, 1, P, 32, None) == INVAL
    assert E(ctypes.byref(w), P + 2, 1, P, 32, None) == ALIGN     # tokens need 4-byte alignment
    assert E(ctypes.byref(w), P, 2, P + 2, 32, None) == ALIGN     # out rows start on 16 bytes
    assert E(ctypes.byref(w), P, 2, P, 36, None) == ALIGN         # ldo a multiple of 8
    assert E(ctypes.byref(w), P, 2, P, 16, None) == INVAL         # ldo < K
    assert E(ctypes.byref(_w8(ldq=40)), P, 1, P, 32, None) == ALIGN
    bad = _lib.Int8Weight(P, None, 4, 32, 32)
    assert E(ctypes.byref(bad), P, 1, P, 32, None) == INVAL        # no scale


def test_grouped_int8_validation(lib):
    ws = (_lib.Int8Weight * 5)(*[_w8() for _ in range(5)])
    ys = (ctypes.c_void_p * 5)(*[P] * 5)
    assert lib.qz_gemv_int8_grouped(ws, 5, P, ys, None) == UNSUP
    assert lib.qz_gemv_int8_grouped(ws, 0, P, ys, None) == INVAL
    bad = (_lib.Int8Weight * 2)(_w8(K=32), _w8(K=48, ldq=48))
    assert lib.qz_gemv_int8_grouped(bad, 2, P, ys, None) == INVAL


def test_grouped_gemm_validation(lib):
    ws = (_lib.Int8Weight * 5)(*[_w8() for _ in range(5)])
    ys = (ctypes.c_void_p * 5)(*[P] * 5)
    ld = (ctypes.c_int64 * 5)(*[8] * 5)
    G = lib.qz_gemm_int8_grouped
    assert G(ws, 5, 3, P, 32, ys, ld, None, 0, None) == UNSUP
    assert G(ws, 2, 65, P, 32, ys, ld, None, 0, None) == UNSUP
    assert G(ws, 2, 0, P, 32, ys, ld, None, 0, None) == INVAL
    assert G(ws, 2, 3, P, 32, ys, None, None, 0, None) == INVAL
    assert G(ws, 2, 3, P, 16, ys, ld, None, 0, None) == INVAL        # ldx < K
    bad_ld = (ctypes.c_int64 * 2)(8, 4)                                 # ldy < N
    assert G(ws, 2, 3, P, 32, ys, bad_ld, None, 0, None) == INVAL
    bad = (_lib.Int8Weight * 2)(_w8(K=32), _w8(K=48, ldq=48))
    assert G(bad, 2, 3, P, 48, ys, ld, None, 0, None) == INVAL
    w4 = (_lib.Int4oWeight * 2)(_w4(), _w4(perm=P + 16))
    assert lib.qz_gemm_int4_outlier_grouped(w4, 2, 3, P, 64, ys, ld, None, 0, None) == INVAL


def test_sequence_validation(lib):
    ws = (_lib.Int8Weight * 6)(*[_w8() for _ in range(6)])
    ys = (ctypes.c_void_p * 6)(*[P] * 6)
    xs = (ctypes.c_void_p * 5)(*[P] * 5)
    F = lib.qz_gemv_int8_sequence
    one = (ctypes.c_int * 5)(1, 1, 1, 1, 1)
    assert F(ws, one, 5, xs, ys, P, None) == UNSUP              # more than QZ_MAX_SEQ
    assert F(ws, one, 0, xs, ys, P, None) == INVAL
    assert F(ws, one, 2, xs, ys, None, None) == INVAL           # no barrier word
    assert F(ws, one, 2, xs, ys, P + 2, None) == ALIGN          # barrier word 4-byte aligned
    zero = (ctypes.c_int * 2)(1, 0)
    assert F(ws, zero, 2, xs, ys, P, None) == INVAL             # empty product
    five = (ctypes.c_int * 1)(5)
    assert F(ws, five, 1, xs, ys, P, None) == UNSUP              # more than QZ_MAX_GROUP
    bad = (_lib.Int8Weight * 2)(_w8(K=32), _w8(K=48, ldq=48))
    two = (ctypes.c_int * 1)(2)
    assert F(bad, two, 1, xs, ys, P, None) == INVAL              # K differs inside a product
    w4 = (_lib.Int4oWeight * 2)(_w4(), _w4(perm=P + 16))
    assert lib.qz_gemv_int4_outlier_sequence(w4, two, 1, xs, ys, P, None) == INVAL


def test_mapped_validation(lib):
    """The zero-copy entry points check sizes, alignment and the shared
    permutation like the grouped calls, then refuse any weight buffer the
    runtime cannot name a device address for (here: memory no CUDA context
    knows), all before anything is launched."""
    M8, M4 = lib.qz_gemv_int8_grouped_mapped, lib.qz_gemv_int4_outlier_grouped_mapped
    ws = (_lib.Int8Weight * 5)(*[_w8() for _ in range(5)])
    ys = (ctypes.c_void_p * 5)(*[P] * 5)
    assert M8(ws, 5, P, ys, None) == UNSUP
    assert M8(ws, 0, P, ys, None) == INVAL
    bad = (_lib.Int8Weight * 2)(_w8(K=32), _w8(K=48, ldq=48))
    assert M8(bad, 2, P, ys, None) == INVAL
    mis = (_lib.Int8Weight * 1)(_w8(ldq=40))
    assert M8(mis, 1, P, ys, None) == ALIGN
    unknown = (_lib.Int8Weight * 2)(_w8(), _w8())
    assert M8(unknown, 2, P, ys, None) == INVAL               # no device address for P
    w4 = (_lib.Int4oWeight * 2)(_w4(), _w4(perm=P + 16))
    assert M4(w4, 2, P, ys, None) == INVAL                   # perm must be shared
    w4 = (_lib.Int4oWeight * 1)(_w4(q4=PU))
    assert M4(w4, 1, P, ys, None) == ALIGN
    w4 = (_lib.Int4oWeight * 2)(_w4(), _w4())
    assert M4(w4, 2, P, ys, None) == INVAL                   # no device address for P


def _w4(N=8, K=64, n_out=1, perm=P, w_out=P, q4=P, scale=P, ld_out=None, ld_q4=None):
    lo, lq = O.int4o_layout(K, min(n_out, K))
    return _lib.Int4oWeight(N, K, n_out, lo if ld_out is None else ld_out,
                            lq if ld_q4 is None else ld_q4, perm, w_out, q4, scale)


def test_gemv_int4_validation(lib):
    g = lambda w: lib.qz_gemv_int4_outlier(ctypes.byref(w), P, P, None)  # noqa: E731
    assert g(_w4(n_out=65)) == INVAL
    assert g(_w4(perm=None)) == INVAL
    assert g(_w4(w_out=None)) == INVAL                        # n_out > 0 needs w_out
    assert g(_w4(q4=None)) == INVAL
    assert g(_w4(ld_q4=16)) == INVAL                          # < ceil(kb/2)
    assert g(_w4(ld_out=12)) == ALIGN
    assert g(_w4(ld_q4=40)) == ALIGN
    assert g(_w4(q4=PU)) == ALIGN
    assert g(_w4(K=57345)) == UNSUP
    w = _w4()
    assert lib.qz_gemm_int4_outlier(ctypes.byref(w), 65, P, 64, P, 8, None, 0, None) == UNSUP


def test_grouped_int4_requires_shared_perm(lib):
    ws = (_lib.Int4oWeight * 2)(_w4(), _w4(perm=P + 0x100))
    ys = (ctypes.c_void_p * 2)(P, P)
    assert lib.qz_gemv_int4_outlier_grouped(ws, 2, P, ys, None) == INVAL
    ws = (_lib.Int4oWeight * 2)(_w4(), _w4(n_out=2))
    assert lib.qz_gemv_int4_outlier_grouped(ws, 2, P, ys, None) == INVAL


def test_quantizer_int4_validation(lib):
    f = lib.qz_quantize_int4_outlier
    lo, lq = O.int4o_layout(64, 1)
    assert f(P, 64, P, 8, 64, 65, P, lo, P, lq, P, None) == INVAL   # n_out > K
    assert f(P, 64, P, 8, 64, 1, None, lo, P, lq, P, None) == INVAL
    assert f(P, 64, P, 8, 64, 1, P, lo, P, 16, P, None) == INVAL    # ld_q4 too small
    assert f(P, 64, P, 8, 64, 1, P, 12, P, lq, P, None) == ALIGN
    assert f(P, 64, None, 8, 64, 1, P, lo, P, lq, P, None) == INVAL
    assert f(P, 64, P, 8, 1 << 17 + 1, 1, P, lo, P, lq, P, None) != OK
    assert lib.qz_select_outliers(P, P, (1 << 20) + 1, 1, P, None) == UNSUP
    assert lib.qz_select_outliers(P, P, 10, 11, P, None) == INVAL
    assert lib.qz_select_outliers(PU + 4, P, 10, 1, P, None) == ALIGN
    assert lib.qz_check_perm(None, 10, P, None) == INVAL
    assert lib.qz_saliency_accumulate(P, 4, 16, 16, PU + 4, None) == ALIGN


def test_pager_create_validation(lib):
    hp = (ctypes.c_void_p * 2)(P, P + 0x1000)
    sz = (ctypes.c_size_t * 2)(256, 256)
    out = ctypes.c_void_p()
    f = lib.qz_pager_create
    assert f(hp, sz, 2, P, P, 256, None, None, ctypes.byref(out)) == INVAL     # same slot
    assert f(hp, sz, 2, P, P + 0x800, 128, None, None, ctypes.byref(out)) == INVAL
    assert f(hp, sz, 0, P, P + 0x800, 256, None, None, ctypes.byref(out)) == INVAL
    assert f(hp, sz, 2, PU, P + 0x800, 256, None, None, ctypes.byref(out)) == ALIGN
    sz_bad = (ctypes.c_size_t * 2)(250, 256)
    assert f(hp, sz_bad, 2, P, P + 0x800, 256, None, None, ctypes.byref(out)) == ALIGN
    assert lib.qz_pager_acquire(None, 0, ctypes.byref(out)) == INVAL
    assert lib.qz_pager_release(None, 0) == INVAL
    assert lib.qz_pager_destroy(None) == INVAL


def test_python_api_refuses_cpu_tensors():
    import torch
    import weight_only_quantized_dequant_gb300 as qz
    with pytest.raises(ValueError):
        qz.quantize_int8(torch.zeros((4, 16), dtype=torch.float16))
