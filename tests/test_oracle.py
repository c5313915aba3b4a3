"""Pins of the CPU oracle against things other than itself.

Closed forms worked out by hand (scale equations of "Open Origin - ELG Stream
Layer", INT8 Quantization & Direct Mapping; the diagram and key innovation 3
of "On-The-Fly Weight Synthesizer (OTF-LLM Engine)"), exact-rational brute
force on tiny inputs, invariants, and the byte counts the pages print
(tests/golden/page_byte_counts.json).  No GPU needed.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import qz_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f16(a):
    return np.asarray(a, np.float16)


# ----------------------------------------------------------------- INT8 ----
def test_int8_hand_scale_one_rne_ties():
    # max|W| = 127 -> scale = 127/127 = 1 exactly, so q = round-half-even(W).
    W = f16([[127.0, -2.5, 3.5, 0.5, -0.5], [1.5, 126.5, -127.0, 2.25, -3.75]])
    q, s = O.int8_quantize(W)
    assert s == np.float32(1.0)
    assert q.tolist() == [[127, -2, 4, 0, 0], [2, 126, -127, 2, -4]]


def test_int8_hand_negative_max_half_scale():
    # max|W| comes from a negative entry: |-63.5| -> scale 0.5; q = rint(2W).
    W = f16([[-63.5, 10.25], [0.75, 31.75]])
    q, s = O.int8_quantize(W)
    assert s == np.float32(0.5)
    assert q.tolist() == [[-127, 20], [2, 64]]   # 20.5 -> 20, 1.5 -> 2, 63.5 -> 64


def test_int8_zero_tensor():
    q, s = O.int8_quantize(np.zeros((3, 5), np.float16))
    assert s == 0 and not q.any()


def _rint_exact(fr: Fraction) -> int:
    """Round a rational to the nearest integer, ties to even."""
    fl = fr.numerator // fr.denominator
    rem = fr - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        return fl + 1
    return fl


@pytest.mark.parametrize("seed", range(4))
def test_int8_against_exact_rationals(seed):
    """scale = fp32(max|W|/127) and q within rounding of the exact quotient."""
    rng = np.random.default_rng(seed)
    W = f16(rng.standard_t(4, size=(5, 7)) * 0.02)
    q, s = O.int8_quantize(W)
    amax = max(abs(Fraction(float(v))) for v in W.ravel())
    # fp32 rounding of the exact quotient amax / 127 (relative error <= 2^-24)
    assert abs(Fraction(float(s)) - amax / 127) <= (amax / 127) * Fraction(1, 2 ** 24)
    for i in range(W.shape[0]):
        for j in range(W.shape[1]):
            exact = Fraction(float(W[i, j])) / Fraction(float(s))
            # the fp32 quotient may only move the result across a tie
            assert abs(q[i, j] - exact) <= Fraction(1, 2) + Fraction(128, 2 ** 24)
            if abs(exact - _rint_exact(exact)) < Fraction(1, 2) - Fraction(1, 2 ** 16):
                assert q[i, j] == _rint_exact(exact)
    # the largest magnitude maps to +-127
    i, j = np.unravel_index(np.argmax(np.abs(W.astype(np.float32))), W.shape)
    assert abs(int(q[i, j])) == 127


def test_int8_invariants_random():
    rng = np.random.default_rng(7)
    W = f16(rng.standard_t(4, size=(64, 96)) * 0.02)
    q, s = O.int8_quantize(W)
    assert np.abs(q.astype(int)).max() == 127
    err = np.abs(W.astype(np.float64) - q.astype(np.float64) * float(s))
    assert (err <= float(s) / 2 * (1 + 2 ** -16)).all()


def test_int8_product_brute_force_exact():
    """y = sum_j (q_ij * s) x_j, checked with exact rationals, non-square."""
    rng = np.random.default_rng(3)
    W = f16(rng.normal(0, 0.02, size=(3, 5)))
    X = f16(rng.normal(0, 1, size=(2, 5)))
    q, s = O.int8_quantize(W)
    y, a = O.int8_product_ref(q, s, X)
    assert y.shape == (2, 3)
    S = Fraction(float(s))
    for b in range(2):
        for i in range(3):
            exact = sum(int(q[i, j]) * S * Fraction(float(X[b, j])) for j in range(5))
            mag = sum(abs(int(q[i, j]) * S * Fraction(float(X[b, j]))) for j in range(5))
            assert abs(Fraction(y[b, i]) - exact) <= mag * Fraction(1, 2 ** 50)
            assert abs(Fraction(a[b, i]) - mag) <= mag * Fraction(1, 2 ** 50)


# ------------------------------------------------------ INT8 embedding ----
_F16_POS = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16)   # every finite value >= 0
_F16_POS64 = _F16_POS.astype(np.float64)                             # exact


def _nearest_fp16(v: Fraction) -> np.float16:
    """Round an exact rational to fp16 by brute force: the two finite fp16
    neighbours of |v| are compared with exact arithmetic; ties go to the
    neighbour with the even bit pattern."""
    a = abs(v)
    k = int(np.searchsorted(_F16_POS64, float(a), side="left"))
    cands = [c for c in (k - 1, k, k + 1) if 0 <= c < _F16_POS.size]
    best = min(cands, key=lambda c: (abs(Fraction(float(_F16_POS64[c])) - a), c & 1))
    h = _F16_POS[best]
    return np.float16(-h) if v < 0 else h


def test_embed_hand_ties_to_even():
    # scale 1 + 2^-11 is an fp16 midpoint between 1 and 1 + 2^-10 -> 1 (even);
    # 1 + 3*2^-11 lies between 1 + 2^-10 and 1 + 2^-9 -> 1 + 2^-9 (even).
    q = np.array([[1, -1, 0], [2, 127, -127]], np.int8)
    out = O.int8_embed(q, np.float32(1 + 2 ** -11), [0])
    assert out.tolist() == [[1.0, -1.0, 0.0]]
    out = O.int8_embed(q, np.float32(1 + 3 * 2 ** -11), [0, 0])
    assert out.tolist() == [[1 + 2 ** -9, -(1 + 2 ** -9), 0.0]] * 2
    # 2 * (1 + 2^-11) = 2 + 2^-10, midpoint between 2 and 2 + 2^-9 -> 2
    out = O.int8_embed(q, np.float32(1 + 2 ** -11), [1])
    assert out[0, 0] == 2.0
    assert out.dtype == np.float16


def test_embed_single_rounding_not_via_fp32():
    """A product that an fp32 multiply would round onto an fp16 midpoint must
    still round to the fp16 neighbour the exact value is nearer to."""
    found = 0
    for qv in range(3, 128, 2):
        for mid in (1 + 2 ** -11, 1 + 3 * 2 ** -11, 1.5 + 2 ** -11):
            s = np.float32(mid / qv)
            for _ in range(4):
                exact = qv * Fraction(float(s))
                naive = np.float32(np.float32(qv) * s)
                if float(naive) == mid and exact != Fraction(mid):
                    want = _nearest_fp16(exact)
                    got = O.int8_embed(np.array([[qv]], np.int8), s, [0])[0, 0]
                    assert got == want and got.view(np.uint16) == want.view(np.uint16)
                    found += np.float16(naive) != want   # the fp32 path would be wrong
                s = np.nextafter(s, np.float32(1))
    assert found >= 3


def test_embed_brute_force_nearest_and_special_cases():
    rng = np.random.default_rng(11)
    W = f16(rng.standard_t(4, size=(40, 24)) * 0.02)
    q, s = O.int8_quantize(W)
    tokens = [5, 0, 39, 5]
    out = O.int8_embed(q, s, tokens)
    assert out.shape == (4, 24) and out.dtype == np.float16
    S = Fraction(float(s))
    for b, t in enumerate(tokens):
        for j in range(24):
            want = _nearest_fp16(int(q[t, j]) * S)
            assert out[b, j].view(np.uint16) == want.view(np.uint16) or (want == 0 and out[b, j] == 0)
    assert (out[0] == out[3]).all()
    # the fp16 rows are within half an fp16 ulp of the reconstruction q * s
    exact = O.int8_dequant(q[tokens], s)
    assert (np.abs(out.astype(np.float64) - exact) <= O.fp16_ulp(exact) / 2).all()
    # zero table: scale 0, rows 0
    qz, sz = O.int8_quantize(np.zeros((3, 8), np.float16))
    assert (O.int8_embed(qz, sz, [2, 1]) == 0).all()
    with pytest.raises(AssertionError):
        O.int8_embed(q, s, [40])


# ------------------------------------------------------------- INT4 parts --
def test_saliency_hand():
    # column sums of |W| over rows, in units of 2^-24; includes the smallest
    # fp16 subnormal 2^-24 (one unit) and a non-square shape.
    W = f16([[1.0, -2.0, 0.25], [0.5, 2.0 ** -24, -0.25]])
    c = O.saliency_fixed(W)
    assert c.tolist() == [3 * 2 ** 23, 2 * 2 ** 24 + 1, 2 ** 23]
    c2 = O.saliency_fixed([W, W])
    assert (c2 == 2 * c).all()


def test_select_hand_ties_and_abs_profile():
    # scores = colsum * |x_profile| = [10, 50, 50, 70, 40]; top-2 = {3, 1}
    # (1 beats 2 on the tie: lower index); perm lists outliers then the rest,
    # each ascending.
    colsum = np.array([10, 50, 50, 7, 20], np.int64)
    prof = np.array([1.0, 1.0, 1.0, 10.0, -2.0], np.float32)
    perm = O.select_outliers(colsum, prof, 2)
    assert perm.tolist() == [1, 3, 0, 2, 4]
    assert O.select_outliers(colsum, prof, 0).tolist() == [0, 1, 2, 3, 4]
    assert O.select_outliers(colsum, prof, 5).tolist() == [0, 1, 2, 3, 4]


@pytest.mark.parametrize("seed", range(6))
def test_select_brute_force(seed):
    rng = np.random.default_rng(seed)
    K = int(rng.integers(1, 40))
    n_out = int(rng.integers(0, K + 1))
    colsum = rng.integers(0, 6, size=K).astype(np.int64)     # many ties
    prof = rng.choice([0.5, 1.0, -1.0, 2.0], size=K).astype(np.float32)
    perm = O.select_outliers(colsum, prof, n_out)
    keyed = sorted(range(K), key=lambda j: (-(int(colsum[j]) * abs(float(prof[j]))), j))
    want = sorted(keyed[:n_out]) + sorted(keyed[n_out:])
    assert perm.tolist() == want


def test_layout_and_row_bytes():
    # K=4096 -> n_out 41, kb 4055, 2028 packed bytes -> ld 2032; ld_out 48
    assert O.default_n_out(4096) == 41
    assert O.int4o_layout(4096, 41) == (48, 2032)
    assert O.int4o_row_bytes(4096, 41) == 2028 + 82 + 4
    # K=28672 -> 287 outliers, kb 28385 (odd) -> 14193 bytes -> ld 14208
    assert O.default_n_out(28672) == 287
    assert O.int4o_layout(28672, 287) == (288, 14208)
    assert O.int4o_layout(5, 5) == (8, 0)
    assert O.int4o_layout(5, 0) == (0, 16)


def test_int4_hand_quantize_pack_product():
    # K=6, n_out=1, perm puts channel 4 first.  Row 0 background (perm order
    # 0,1,2,3,5) = [3.5,-7,1.5,2.5,-0.5]: max 7 -> s=1 -> q=[4,-7,2,2,0];
    # nibbles 0x4,0x9,0x2,0x2,0x0 -> bytes 0x94, 0x22, 0x00.  Row 1 has a zero
    # background -> s=0, q=0.
    W = f16([[3.5, -7.0, 1.5, 2.5, 100.0, -0.5], [0, 0, 0, 0, -2.0, 0]])
    perm = np.array([4, 0, 1, 2, 3, 5], np.int32)
    w_out, q4, s = O.int4o_quantize(W, perm, 1)
    assert w_out.shape == (2, 8) and q4.shape == (2, 16)
    assert w_out[:, 0].tolist() == [100.0, -2.0] and not w_out[:, 1:].any()
    assert s.tolist() == [1.0, 0.0]
    assert q4[0, :3].tolist() == [0x94, 0x22, 0x00] and not q4[0, 3:].any()
    assert not q4[1].any()
    # y0 = 100*0.5 + (4*1 - 7*2 + 2*3 + 2*4 + 0*(-1)) = 54 ; y1 = -2*0.5 = -1
    x = f16([[1, 2, 3, 4, 0.5, -1]])
    y, a = O.int4o_product_ref(w_out, q4, s, perm, 1, 6, x)
    assert y.tolist() == [[54.0, -1.0]]
    assert a.tolist() == [[50 + 4 + 14 + 6 + 8, 1.0]]
    yp = O.int4o_product_permuted(w_out, q4, s, perm, 1, 6, x)
    assert yp.tolist() == [[54.0, -1.0]]


@pytest.mark.parametrize("kb", [1, 2, 7, 32, 33])
def test_pack_unpack_round_trip(kb):
    rng = np.random.default_rng(kb)
    q = rng.integers(-7, 8, size=(3, kb)).astype(np.int8)
    packed = O.pack_int4(q)
    assert packed.shape == (3, (kb + 1) // 2)
    assert (O.unpack_int4(packed, kb) == q).all()
    if kb % 2:
        assert not (packed[:, -1] >> 4).any()      # the odd tail nibble is 0
    # byte m = low nibble 2m, high nibble 2m+1, two's complement
    assert packed[0, 0] == ((int(q[0, 0]) & 15) | (((int(q[0, 1]) & 15) << 4) if kb > 1 else 0))


def _int4_case(seed, N=9, K=37, n_out=None):
    rng = np.random.default_rng(seed)
    W = f16(rng.standard_t(4, size=(N, K)) * 0.02)
    prof = np.abs(rng.normal(size=K)).astype(np.float32)
    n_out = O.default_n_out(K) if n_out is None else n_out
    perm = O.select_outliers(O.saliency_fixed(W), prof, n_out)
    return W, perm, n_out


@pytest.mark.parametrize("seed", range(4))
def test_int4_invariants(seed):
    W, perm, n_out = _int4_case(seed, N=11, K=53, n_out=3)
    N, K = W.shape
    w_out, q4, s = O.int4o_quantize(W, perm, n_out)
    # perm is a bijection
    assert sorted(perm.tolist()) == list(range(K))
    # outliers reproduced exactly in fp16, bitwise
    assert (w_out[:, :n_out].view(np.uint16) == W[:, perm[:n_out]].view(np.uint16)).all()
    kb = K - n_out
    q = O.unpack_int4(q4, kb).astype(np.int64)
    assert np.abs(q).max() <= 7
    bg = W[:, perm[n_out:]].astype(np.float64)
    for i in range(N):
        assert abs(q[i]).max() == 7                         # max attained per row
        assert (np.abs(bg[i] - q[i] * float(s[i])) <= float(s[i]) / 2 * (1 + 2 ** -16)).all()
        assert float(s[i]) == float(np.float32(np.float32(np.abs(bg[i]).max()) / np.float32(7)))
    # padding is zero
    assert not q4[:, (kb + 1) // 2:].any()
    assert not w_out[:, n_out:].any()


@pytest.mark.parametrize("seed", range(3))
def test_int4_permuted_equals_unpermuted(seed):
    W, perm, n_out = _int4_case(seed, N=13, K=64, n_out=5)
    w_out, q4, s = O.int4o_quantize(W, perm, n_out)
    X = f16(np.random.default_rng(seed + 100).normal(size=(3, 64)))
    y, _ = O.int4o_product_ref(w_out, q4, s, perm, n_out, 64, X)
    yp = O.int4o_product_permuted(w_out, q4, s, perm, n_out, 64, X)
    assert np.allclose(y, yp, rtol=1e-12, atol=1e-12)


def test_int4_all_outliers_is_plain_fp16_gemv():
    W, perm, _ = _int4_case(5, N=6, K=16)
    w_out, q4, s = O.int4o_quantize(W, perm, 16)
    assert q4.shape[1] == 0 and not s.any()
    X = f16(np.random.default_rng(1).normal(size=(2, 16)))
    y, _ = O.int4o_product_ref(w_out, q4, s, perm, 16, 16, X)
    plain = np.einsum("bk,nk->bn", X.astype(np.float64), W.astype(np.float64))
    assert np.allclose(y, plain, rtol=1e-13, atol=1e-15)


def test_int4_no_outliers_is_per_row_int4():
    W, _, _ = _int4_case(6, N=5, K=20)
    perm = np.arange(20, dtype=np.int32)
    w_out, q4, s = O.int4o_quantize(W, perm, 0)
    assert w_out.shape[1] == 0
    What = O.int4o_dequant(w_out, q4, s, perm, 0, 20)
    for i in range(5):
        si = float(s[i])
        assert si == float(np.float32(np.float32(np.abs(W[i].astype(np.float32)).max()) / np.float32(7)))
        assert (np.abs(W[i].astype(np.float64) - What[i]) <= si / 2 * (1 + 2 ** -16)).all()


def test_int4_product_brute_force_exact():
    W, perm, n_out = _int4_case(9, N=4, K=10, n_out=2)
    w_out, q4, s = O.int4o_quantize(W, perm, n_out)
    X = f16(np.random.default_rng(2).normal(size=(2, 10)))
    y, _ = O.int4o_product_ref(w_out, q4, s, perm, n_out, 10, X)
    q = O.unpack_int4(q4, 10 - n_out)
    for b in range(2):
        for i in range(4):
            exact = Fraction(0)
            for t in range(10):
                xv = Fraction(float(X[b, perm[t]]))
                if t < n_out:
                    exact += Fraction(float(w_out[i, t])) * xv
                else:
                    exact += int(q[i, t - n_out]) * Fraction(float(s[i])) * xv
            assert abs(Fraction(y[b, i]) - exact) <= abs(exact) * Fraction(1, 2 ** 48) + Fraction(1, 2 ** 70)


# ---------------------------------------------------------- tolerance -----
def test_fp16_ulp_closed_forms():
    v = np.array([1.0, 1.5, 2.0, 65504.0, 2.0 ** -14, 1e-6, 0.0, -3.0])
    want = [2 ** -10, 2 ** -10, 2 ** -9, 32.0, 2 ** -24, 2 ** -24, 2 ** -24, 2 ** -9]
    assert O.fp16_ulp(v).tolist() == want


def test_tolerance_hand_values():
    """The acceptance bound 1e-3 * sum_j |w_ij x_j| + 1 fp16 ulp of y_ref,
    evaluated by hand: a normal, a negative, a subnormal and a zero y_ref,
    the largest finite fp16, and a zero magnitude sum (ulp alone)."""
    y_ref = np.array([1.0, -3.0, 1e-6, 0.0, 65504.0, 0.75])
    abs_ref = np.array([2.0, 10.0, 0.5, 0.0, 70000.0, 0.0])
    want = [2e-3 + 2 ** -10,        # ulp(1) = 2^-10
            1e-2 + 2 ** -9,         # ulp(3) = 2^-9
            5e-4 + 2 ** -24,        # subnormal: spacing 2^-24
            2 ** -24,               # zero: the subnormal spacing
            70.0 + 32.0,            # ulp(65504) = 32
            2 ** -11]               # ulp(0.75) = 2^-11, no magnitude term
    got = O.tolerance(y_ref, abs_ref)
    assert np.allclose(got, want, rtol=1e-15, atol=0)
    # the relative term is 1e-3, not 1e-2 or 1e-4: an error of 1.5e-3 on a
    # magnitude sum of 1 at y_ref = 0 fails, 0.9e-3 passes
    assert 1.5e-3 > O.tolerance(np.array([0.0]), np.array([1.0]))[0]
    assert 0.9e-3 < O.tolerance(np.array([0.0]), np.array([1.0]))[0]


# ------------------------------------------------- byte counts (pages) ----
def _golden():
    with open(os.path.join(GOLDEN, "page_byte_counts.json")) as f:
        return json.load(f)


def test_int8_pool_matches_elg_7_75_gb():
    g = _golden()["int8_pool_gemma2_9b"]
    h, qo, kv, it = g["hidden"], g["q_out"], g["kv_out"], g["inter"]
    shapes = [(qo, h), (kv, h), (kv, h), (h, qo), (it, h), (it, h), (h, it)]
    per_layer = sum(O.int8_weight_bytes(n, k) - 4 for n, k in shapes)  # codes only
    assert per_layer == 198_180_864
    total = g["layers"] * per_layer
    assert abs(total / 2 ** 30 - g["printed"]) <= g["half_unit"]


def test_base_vram_matches_elg_1_71_gb():
    g = _golden()["base_vram_gemma2_9b"]
    assert abs(g["vocab"] * g["hidden"] * 2 / 2 ** 30 - g["printed"]) <= g["half_unit"]


def test_perm_tables_match_otf_1_6_mb():
    g = _golden()["perm_tables_llama32_3b"]
    per_layer = 4 * (g["hidden"] + g["q_out"] + g["inter"])
    assert abs(g["layers"] * per_layer / 1e6 - g["printed"]) <= g["half_unit"]


def test_70b_stack_bytes():
    # 70B shapes at the packed format: 441,006,080 bytes per layer
    h, qo, kv, it = 8192, 8192, 1024, 28672
    shapes = [(qo, h), (kv, h), (kv, h), (h, qo), (it, h), (it, h), (h, it)]
    per = sum(O.int4o_weight_bytes(n, k, O.default_n_out(k)) for n, k in shapes)
    assert per == 441_006_080
