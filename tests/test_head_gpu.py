"""The steps either side of the decoder stack, CUDA path vs the CPU oracle:
the INT8 vocabulary-table lookup (bit-exact fp16 rows) and the output
projection (lm_head) over the 128256 x 3072 table, tied (the INT8 table
itself) and untied (outlier-aware INT4), on sampled rows.
"""
from fractions import Fraction

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
    assert not bad.any(), f"{what}: {int(bad.sum())}/{bad.size} outside tolerance"


def _bits(a) -> np.ndarray:
    return np.asarray(a).view(np.uint16)


def _table(q: np.ndarray, scale: float):
    """An Int8Matrix holding the given codes and scale (rows padded to 16)."""
    V, K = q.shape
    ldq = -(-K // 16) * 16
    qp = np.zeros((V, ldq), np.int8)
    qp[:, :K] = q
    return qz().Int8Matrix(torch.from_numpy(qp).to(DEV),
                           torch.tensor([scale], dtype=torch.float32, device=DEV), V, K)


# ------------------------------------------------------------- lookup ----
@pytest.mark.parametrize("V,K,B", [(1, 1, 1), (40, 29, 7), (300, 1000, 33), (64, 4096, 5)])
def test_embed_bit_exact_after_gpu_quantize(V, K, B):
    W = S.weight(V, K, 9100 + K, device=DEV)
    table = qz().quantize_int8(W)
    tok = S.tokens(B, V, 9200 + B, device=DEV)
    out = qz().embed_int8(table, tok)
    assert qz().device_error() == 0
    q_ref, s_ref = O.int8_quantize(W.cpu().numpy())
    ref = O.int8_embed(q_ref, s_ref, tok.cpu().numpy())
    assert np.array_equal(_bits(out.cpu().numpy()), _bits(ref))


def _trap_scales():
    """fp32 scales for which an fp32 product q * s falls on an fp16 midpoint
    that the exact product is not on (found by exact rational search)."""
    out = []
    for qv in range(3, 128, 2):
        for mid in (1 + 2 ** -11, 1 + 3 * 2 ** -11, 1.5 + 2 ** -11, 64 + 2 ** -5):
            s = np.float32(mid / qv)
            for _ in range(3):
                exact = qv * Fraction(float(s))
                if float(np.float32(np.float32(qv) * s)) == mid and exact != Fraction(mid):
                    out.append(float(s))
                s = np.nextafter(s, np.float32(1))
    return sorted(set(out))


def test_embed_every_code_ties_and_fp32_traps():
    """All 255 codes against scales that put products on fp16 midpoints
    (ties to even) or within an fp32 rounding of one (one rounding only)."""
    scales = [1 + 2 ** -11, 1 + 3 * 2 ** -11, 2.0 ** -7, 0.0, 1e-3] + _trap_scales()[:24]
    assert len(scales) >= 20
    q = np.arange(-127, 128, dtype=np.int8).reshape(1, 255)
    for s in scales:
        table = _table(np.repeat(q, 3, axis=0), s)
        tok = torch.tensor([2, 0, 1, 0], dtype=torch.int32, device=DEV)
        out = qz().embed_int8(table, tok)
        ref = O.int8_embed(np.repeat(q, 3, axis=0), np.float32(s), [2, 0, 1, 0])
        assert np.array_equal(_bits(out.cpu().numpy()), _bits(ref)), f"scale {s!r}"


def test_embed_out_of_range_tokens_flagged_and_zeroed():
    W = S.weight(50, 64, 9300, device=DEV)
    table = qz().quantize_int8(W)
    qz().device_error(clear=True)
    tok = torch.tensor([-1, 50, 7, 2 ** 31 - 1, 49], dtype=torch.int32, device=DEV)
    out = qz().embed_int8(table, tok)
    err = qz().device_error(clear=True)
    assert err & 2
    o = out.cpu().numpy()
    assert not o[[0, 1, 3]].any()
    q_ref, s_ref = O.int8_quantize(W.cpu().numpy())
    ref = O.int8_embed(q_ref, s_ref, [7, 49])
    assert np.array_equal(_bits(o[[2, 4]]), _bits(ref))
    assert qz().device_error() == 0


def test_embed_empty_batch_and_strided_output():
    W = S.weight(20, 24, 9400, device=DEV)
    table = qz().quantize_int8(W)
    empty = qz().embed_int8(table, torch.empty((0,), dtype=torch.int32, device=DEV))
    assert empty.shape == (0, 24)
    buf = torch.full((3, 40), 7.0, dtype=torch.float16, device=DEV)
    tok = torch.tensor([3, 19, 0], dtype=torch.int32, device=DEV)
    qz().embed_int8(table, tok, out=buf[:, :24])
    q_ref, s_ref = O.int8_quantize(W.cpu().numpy())
    ref = O.int8_embed(q_ref, s_ref, [3, 19, 0])
    got = buf.cpu().numpy()
    assert np.array_equal(_bits(got[:, :24]), _bits(ref))
    assert (got[:, 24:] == 7.0).all()               # beyond K untouched


# --------------------------------------------- vocabulary-sized head ----
@pytest.mark.slow
def test_llama32_3b_head_tied_and_untied():
    """128256 x 3072: lookup of 64 tokens bit-exact; tied lm_head (the INT8
    table) and untied INT4-outlier lm_head on 256 sampled rows."""
    hd = S.HEADS["llama32_3b_head"]
    V, H = hd.vocab, hd.hidden
    W = S.weight(V, H, hd.seed_base, device=DEV)
    table = qz().quantize_int8(W)
    tok = S.tokens(64, V, hd.seed_base + 4, device=DEV)
    tok[0], tok[1] = 0, V - 1
    emb = qz().embed_int8(table, tok)
    h = S.activation(1, H, hd.seed_base + 3, device=DEV)
    logits = qz().gemv_int8(table, h[0])
    assert qz().device_error() == 0
    Wn = W.cpu().numpy()
    del W
    q_ref, s_ref = O.int8_quantize(Wn)
    assert table.scale.item() == float(s_ref)
    ref = O.int8_embed(q_ref, s_ref, tok.cpu().numpy())
    assert np.array_equal(_bits(emb.cpu().numpy()), _bits(ref))
    rows = np.random.default_rng(1).choice(V, 256, replace=False)
    rows[:2] = [0, V - 1]
    assert np.array_equal(table.q.cpu().numpy()[rows, :H], q_ref[rows])
    y_ref, a_ref = O.int8_product_ref(q_ref[rows], s_ref, h.cpu().numpy())
    assert_close(logits[rows], y_ref[0], a_ref[0], "tied lm_head")
    del Wn, q_ref

    # untied: its own outlier-aware INT4 matrix
    n_out = O.default_n_out(H)
    W2 = S.weight(V, H, hd.seed_base + 1, device=DEV)
    prof = S.x_profile(H, n_out, hd.seed_base + 2, device=DEV)
    colsum = torch.zeros((H,), dtype=torch.int64, device=DEV)
    qz().saliency_accumulate(W2, colsum)
    perm = qz().select_outliers(colsum, prof, n_out)
    w4 = qz().quantize_int4_outlier(W2, perm, n_out)
    y4 = qz().gemv_int4_outlier(w4, h[0])
    assert qz().device_error() == 0
    W2n = W2.cpu().numpy()
    del W2
    sal = O.saliency_fixed(W2n)
    assert np.array_equal(colsum.cpu().numpy(), sal)
    pn = O.select_outliers(sal, prof.cpu().numpy(), n_out)
    assert np.array_equal(perm.cpu().numpy(), pn)
    wo, q4, s = O.int4o_quantize(W2n[rows], pn, n_out)
    assert np.array_equal(w4.q4.cpu().numpy()[rows], q4)
    y_ref, a_ref = O.int4o_product_ref(wo, q4, s, pn, n_out, H, h.cpu().numpy())
    assert_close(y4[rows], y_ref[0], a_ref[0], "untied int4 lm_head")
