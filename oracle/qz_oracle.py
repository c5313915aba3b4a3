"""CPU oracle for weight-only quantized dequant-GEMV (numpy, fp64 products).

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module.  It shares no code
with the CUDA library (no kernels, headers, tables or helpers); the two meet
only on the seeded inputs of ``weight_only_quantized_dequant_gb300.synthetic``.

Every function below is the plain definition of one step of the method, in the
order the pages give it, with no blocking or fusion:

* INT8 per-tensor quantization, "Open Origin - ELG Stream Layer", section
  "Technical Architecture > INT8 Quantization & Direct Mapping" (the scale and
  round equations), and its reconstruction, section "FP16 On-The-Fly GPU
  Reconstruction" (the one-line cast-and-multiply).
* Outlier-aware INT4, "On-The-Fly Weight Synthesizer (OTF-LLM Engine)",
  section "Architecture & Key Innovations": the diagram (permutation, 1% FP16
  outlier channels, 99% INT4 background in [-7, +7] with zero-point 0 and 2:1
  packing, outlier product + background product) and key innovation 3 (top-1%
  channels ranked by |W| x |X_profile|, one static permutation).

Where the pages leave a step open, the reading taken is stated at the step.

Pinning: every function here is checked by ``tests/test_oracle.py`` against
hand-derived closed forms, brute force on tiny inputs and invariants.  The
pages print no worked numeric example, so the accuracy claims of the pages
("maintaining precision", "100% accuracy retention") are parity unpinned; they
need trained models and are not tested.
"""
from __future__ import annotations

import numpy as np

INT8_QMAX = 127          # ELG Stream Layer, scale equation: max|W| / 127
INT4_QMAX = 7            # OTF-LLM diagram: background range [-7 ... +7]
FIXED_POINT_BITS = 24    # every finite fp16 value is an integer multiple of 2^-24


# --------------------------------------------------------------------------
# INT8 per-tensor (ELG Stream Layer, "INT8 Quantization & Direct Mapping")
# --------------------------------------------------------------------------
def int8_quantize(W: np.ndarray) -> tuple[np.ndarray, np.float32]:
    """scale = max|W| / 127 and q = round(W / scale), one scale per tensor.

    Readings: the scale is one fp32 number per weight matrix (the page writes a
    single max over |W| even though its prose says "per-parameter"); the divide
    is an IEEE fp32 division of fp32(W) by the fp32 scale, not a multiply by a
    reciprocal; ``round`` is round-half-to-even (the page's own code runs on
    torch, whose round is half-to-even); the clip to [-127, 127] only matters
    at fp edges; an all-zero tensor gets scale 0 and q = 0 (no divide).
    """
    W = np.asarray(W)
    assert W.dtype == np.float16 and W.ndim == 2
    w32 = W.astype(np.float32)
    amax = np.float32(np.max(np.abs(w32))) if w32.size else np.float32(0.0)
    scale = np.float32(amax / np.float32(INT8_QMAX))
    if scale == 0:
        return np.zeros(W.shape, np.int8), np.float32(0.0)
    q = np.rint(w32 / scale)                       # fp32 / fp32 is IEEE RN
    q = np.clip(q, -INT8_QMAX, INT8_QMAX).astype(np.int8)
    return q, scale


def int8_dequant(q: np.ndarray, scale) -> np.ndarray:
    """Reconstruction q * scale ("FP16 On-The-Fly GPU Reconstruction").

    Reading: the reconstructed weight is the exact product q * scale (fp64);
    the page rounds it to fp16, which would spend half of the output tolerance
    on that rounding alone, so the kernels factor the scale out instead and
    the oracle keeps the exact value.
    """
    return np.asarray(q, np.float64) * np.float64(np.float32(scale))


def int8_embed(q: np.ndarray, scale, tokens) -> np.ndarray:
    """Rows of an INT8 vocabulary table, reconstructed to fp16.

    "On-The-Fly Weight Synthesizer (OTF-LLM Engine)", key innovation 4 keeps
    the vocabulary lookup table (embed_tokens) in INT8; the reconstruction is
    the ELG Stream Layer one ("FP16 On-The-Fly GPU Reconstruction"): q * scale
    as fp16.  Readings: the table is quantized like any other matrix (one fp32
    scale per tensor, int8_quantize); a looked-up row is the exact product
    q * scale (int8_dequant) rounded once to the nearest fp16, ties to even.
    Here the row leaves the method as an fp16 activation, so the one rounding
    is the output's own.  tokens: int array of row indices, each in [0, V).
    """
    q = np.asarray(q)
    tokens = np.asarray(tokens, np.int64).reshape(-1)
    assert q.ndim == 2 and np.all((tokens >= 0) & (tokens < q.shape[0]))
    exact = int8_dequant(q[tokens], scale)          # exact in fp64 (7 x 24 bits)
    return exact.astype(np.float16)                 # one round to nearest even


# --------------------------------------------------------------------------
# Outlier-aware INT4 (OTF-LLM, "Architecture & Key Innovations")
# --------------------------------------------------------------------------
def default_n_out(K: int) -> int:
    """Number of FP16 outlier channels for K inputs: ceil(K / 100).

    Reading of "Top-1%": at least 1% of the channels are kept.
    """
    return (K + 99) // 100


def int4o_layout(K: int, n_out: int) -> tuple[int, int]:
    """Row strides (ld_out in halves, ld_q4 in bytes) of the packed format.

    Reading: rows are padded so that every row starts on a 16-byte boundary:
    ld_out = n_out rounded up to 8 halves, ld_q4 = ceil((K - n_out) / 2)
    rounded up to 16 bytes.  Padding holds zeros.
    """
    assert 0 <= n_out <= K
    kb = K - n_out
    ld_out = -(-n_out // 8) * 8
    ld_q4 = -(-((kb + 1) // 2) // 16) * 16
    return ld_out, ld_q4


def saliency_fixed(Ws) -> np.ndarray:
    """Per-input-channel weight magnitude, summed over output rows.

    The |W| factor of the ranking score of key innovation 3, reduced over the
    output rows of every matrix that shares the permutation (reading: one
    permutation per input space and layer; L1 over rows).  The sum is exact:
    each fp16 magnitude times 2^24 is an integer, and the result is returned
    in those units as int64, so its value does not depend on summation order.
    """
    if isinstance(Ws, np.ndarray):
        Ws = [Ws]
    K = Ws[0].shape[1]
    total = np.zeros(K, np.int64)
    for W in Ws:
        assert W.dtype == np.float16 and W.shape[1] == K
        units = np.abs(W.astype(np.float64)) * float(1 << FIXED_POINT_BITS)
        total += units.astype(np.int64).sum(axis=0, dtype=np.int64)
    return total


def outlier_scores(colsum: np.ndarray, x_profile: np.ndarray) -> np.ndarray:
    """Score |W| x |X_profile| per channel: fp64(colsum) * fp64(|x_profile|).

    colsum is in units of 2^-24; the common factor does not change the order.
    Both factors convert exactly or with one RN rounding, and the product is
    one fp64 RN multiply.
    """
    c = np.asarray(colsum, np.int64).astype(np.float64)
    xp = np.abs(np.asarray(x_profile, np.float32)).astype(np.float64)
    return c * xp


def select_outliers(colsum: np.ndarray, x_profile: np.ndarray, n_out: int) -> np.ndarray:
    """global_perm_idx: the n_out top-scoring channels first, then the rest.

    Reading: ties in the score go to the lower channel index; inside each of
    the two groups channels keep ascending original order (the pages fix no
    order, and any order gives the same product).  Returns int32 [K] with
    xp[t] = x[perm[t]].
    """
    K = colsum.shape[0]
    assert 0 <= n_out <= K
    score = outlier_scores(colsum, x_profile)
    idx = np.arange(K)
    order = np.lexsort((idx, -score))           # score descending, index ascending
    outl = np.sort(order[:n_out])
    rest = np.sort(order[n_out:])
    return np.concatenate([outl, rest]).astype(np.int32)


def int4o_quantize(W: np.ndarray, perm: np.ndarray, n_out: int):
    """Split W along the permuted channels into FP16 outliers + packed INT4.

    Outliers: w_out[i, t] = W[i, perm[t]] for t < n_out, bit-exact fp16.
    Background (t >= n_out): per output row i, s_i = max|W_bg[i]| / 7 (fp32
    IEEE divide) and q = clip(round(W / s_i), -7, 7) with round-half-to-even,
    zero-point 0.  Reading: the scale is per output row and its max runs over
    the background only (excluding outliers is their purpose); a zero row
    gets s_i = 0 and q = 0.
    Packing (2:1 into uint8): background element t' goes to byte t' // 2, the
    low nibble when t' is even, as the two's-complement nibble q & 0xF.
    Returns (w_out fp16 [N, ld_out], q4 uint8 [N, ld_q4], s fp32 [N]).
    """
    W = np.asarray(W)
    assert W.dtype == np.float16 and W.ndim == 2
    N, K = W.shape
    perm = np.asarray(perm, np.int64)
    ld_out, ld_q4 = int4o_layout(K, n_out)
    kb = K - n_out

    Wp = W[:, perm]                                   # permuted channel order
    w_out = np.zeros((N, ld_out), np.float16)
    w_out[:, :n_out] = Wp[:, :n_out]

    bg = Wp[:, n_out:].astype(np.float32)
    if kb:
        amax = np.max(np.abs(bg), axis=1).astype(np.float32)
    else:
        amax = np.zeros(N, np.float32)
    s = (amax / np.float32(INT4_QMAX)).astype(np.float32)
    q = np.zeros((N, kb), np.int8)
    nz = s != 0
    if kb and nz.any():
        r = np.rint(bg[nz] / s[nz, None])             # fp32 / fp32 is IEEE RN
        q[nz] = np.clip(r, -INT4_QMAX, INT4_QMAX).astype(np.int8)
    q4 = np.zeros((N, ld_q4), np.uint8)
    q4[:, : (kb + 1) // 2] = pack_int4(q)
    return w_out, q4, s


def pack_int4(q: np.ndarray) -> np.ndarray:
    """Two signed 4-bit values per byte: element 2m low nibble, 2m+1 high."""
    q = np.asarray(q, np.int8)
    N, kb = q.shape
    nib = (q.astype(np.int16) & 0xF).astype(np.uint8)
    if kb % 2:
        nib = np.concatenate([nib, np.zeros((N, 1), np.uint8)], axis=1)
    return (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)


def unpack_int4(q4: np.ndarray, kb: int) -> np.ndarray:
    """Inverse of pack_int4: the first kb signed values of each row."""
    q4 = np.asarray(q4, np.uint8)
    lo = (q4 & 0xF).astype(np.int16)
    hi = (q4 >> 4).astype(np.int16)
    both = np.empty((q4.shape[0], 2 * q4.shape[1]), np.int16)
    both[:, 0::2] = lo
    both[:, 1::2] = hi
    both = np.where(both >= 8, both - 16, both)
    return both[:, :kb].astype(np.int8)


def int4o_dequant(w_out, q4, s, perm, n_out: int, K: int) -> np.ndarray:
    """Reconstructed weight in ORIGINAL channel order, fp64 [N, K].

    Outlier columns are the fp16 values themselves; background columns are the
    exact products q * s_i.
    """
    perm = np.asarray(perm, np.int64)
    N = q4.shape[0]
    kb = K - n_out
    What = np.zeros((N, K), np.float64)
    What[:, perm[:n_out]] = np.asarray(w_out)[:, :n_out].astype(np.float64)
    qb = unpack_int4(q4, kb).astype(np.float64)
    What[:, perm[n_out:]] = qb * np.asarray(s, np.float32).astype(np.float64)[:, None]
    return What


# --------------------------------------------------------------------------
# Products
# --------------------------------------------------------------------------
def product_ref(What: np.ndarray, X: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """y_ref = What @ x in fp64, and the magnitude sum |What| @ |x|.

    What is the reconstructed weight [N, K]; X is fp16 [B, K] (or [K]).
    Returns (y_ref [B, N], abs_ref [B, N]) in fp64.
    """
    X = np.asarray(X)
    x64 = np.atleast_2d(X.astype(np.float64))
    y = x64 @ What.T
    a = np.abs(x64) @ np.abs(What).T
    return y, a


def int8_product_ref(q, scale, X):
    """y = (q * scale) . x for the INT8 per-tensor format."""
    return product_ref(int8_dequant(q, scale), X)


def int4o_product_ref(w_out, q4, s, perm, n_out, K, X):
    """Outlier FP16 product + INT4 background product, in original order."""
    return product_ref(int4o_dequant(w_out, q4, s, perm, n_out, K), X)


def int4o_product_permuted(w_out, q4, s, perm, n_out, K, X):
    """The same product computed the way the diagram draws it.

    x is permuted with global_perm_idx, the outlier block multiplies the first
    n_out permuted inputs, the background block (q * s_i) multiplies the rest,
    and the two products are added.  Equal to int4o_product_ref up to fp64
    rounding order; used as an invariant.
    """
    perm = np.asarray(perm, np.int64)
    x64 = np.atleast_2d(np.asarray(X).astype(np.float64))
    xp = x64[:, perm]
    kb = K - n_out
    y_out = xp[:, :n_out] @ np.asarray(w_out)[:, :n_out].astype(np.float64).T
    qb = unpack_int4(q4, kb).astype(np.float64)
    y_bg = (xp[:, n_out:] @ qb.T) * np.asarray(s, np.float32).astype(np.float64)[None, :]
    return y_out + y_bg


# --------------------------------------------------------------------------
# Acceptance bound
# --------------------------------------------------------------------------
def fp16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of fp16 numbers at |v| (2^-24 below the normal range)."""
    a = np.abs(np.asarray(v, np.float64))
    out = np.full(a.shape, 2.0 ** -24)
    norm = a >= 2.0 ** -14
    e = np.floor(np.log2(np.where(norm, a, 1.0)))
    out[norm] = 2.0 ** (e[norm] - 10)
    return out


def tolerance(y_ref: np.ndarray, abs_ref: np.ndarray) -> np.ndarray:
    """|y - y_ref| <= 1e-3 * sum_j |w_ij x_j| + 1 fp16 ulp of y_ref."""
    return 1e-3 * np.asarray(abs_ref, np.float64) + fp16_ulp(y_ref)


# --------------------------------------------------------------------------
# Byte accounting of the formats (algorithmic bytes: no padding)
# --------------------------------------------------------------------------
def int8_weight_bytes(N: int, K: int) -> int:
    """N*K int8 codes plus one fp32 scale."""
    return N * K + 4


def int4o_row_bytes(K: int, n_out: int) -> int:
    """ceil(kb/2) packed bytes + 2*n_out fp16 outlier bytes + 4 (fp32 scale)."""
    kb = K - n_out
    return (kb + 1) // 2 + 2 * n_out + 4


def int4o_weight_bytes(N: int, K: int, n_out: int) -> int:
    return N * int4o_row_bytes(K, n_out)
