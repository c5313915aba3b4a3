"""The bench's byte accounting (the numerator of every GB/s it reports), on
CPU: the matrix classes' algorithmic byte counts agree with the oracle's, and
per decoder layer they come to the counts derived from the published model
dimensions (codes, fp16 outliers and fp32 scales; no padding)."""
import torch

from oracle import qz_oracle as O
from weight_only_quantized_dequant_gb300 import api
from weight_only_quantized_dequant_gb300 import synthetic as S

# per layer, all 7 matrices: INT8 codes + one fp32 scale each; INT4-outlier
# ceil(kb/2) packed bytes + 2 n_out outlier bytes + 4 scale bytes per row
LAYER_BYTES = {
    "gemma2_9b_int8": 198_180_864 + 7 * 4,
    "llama32_3b_int4o": 51_975_168,
    "llama_7b_int4o": 104_422_400,
    "llama_70b_int4o": 441_006_080,
}


def _matrix(fmt: str, N: int, K: int):
    """A matrix object of the binding with empty CPU tensors (only its sizes
    matter to the byte count)."""
    if fmt == "int8":
        return api.Int8Matrix(torch.empty((0,)), torch.empty((1,)), N, K)
    n_out = O.default_n_out(K)
    return api.Int4oMatrix(torch.empty((K,), dtype=torch.int32), torch.empty((0, 0)),
                           torch.empty((0, 0)), torch.empty((N,)), N, K, n_out)


def test_layer_bytes_match_the_published_dimensions():
    for name, want in LAYER_BYTES.items():
        wl = S.WORKLOADS[name]
        oracle_bytes = 0
        binding_bytes = 0
        for m in S.MATS:
            N, K = wl.shape(m)
            if wl.fmt == "int8":
                oracle_bytes += O.int8_weight_bytes(N, K)
            else:
                oracle_bytes += O.int4o_weight_bytes(N, K, O.default_n_out(K))
            binding_bytes += _matrix(wl.fmt, N, K).nbytes()
        assert oracle_bytes == want, name
        assert binding_bytes == want, name


def test_int4o_bytes_per_weight_near_half():
    """About 0.516 bytes per weight at K = 4096 (1% fp16 outliers)."""
    K, N = 4096, 1
    b = O.int4o_weight_bytes(N, K, O.default_n_out(K))
    assert abs(b / K - 0.516) < 0.002
