"""Streaming quantizer on the GPU: checkpoint file -> packed pool file, bit for
bit the layers built in memory, and the INT8 codes against the oracle run on
the memory-mapped fp16 weights."""
import numpy as np
import pytest
import torch

from oracle import qz_oracle as O
from weight_only_quantized_dequant_gb300 import checkpoint as C
from weight_only_quantized_dequant_gb300 import stack as ST
from weight_only_quantized_dequant_gb300 import synthetic as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_only_quantized_dequant_gb300 import build
    build.build()


@pytest.mark.parametrize("name,layers", [("llama32_3b_int4o", 2), ("gemma2_9b_int8", 1)])
def test_stream_quantize_matches_in_memory_build(tmp_path, name, layers):
    wl = S.WORKLOADS[name]
    ck = str(tmp_path / "w.safetensors")
    pool = str(tmp_path / "w.qz")
    C.write_synthetic_checkpoint(ck, wl, layers)
    stats = C.quantize_stream(ck, wl, layers, pool)
    assert stats["layers"] == layers
    hdr, blobs = C.load_pool(pool)
    ps = ST.PagedStack(wl, n_layers=layers, distinct=layers)
    for a, b in zip(blobs, ps.blobs):
        assert torch.equal(a, b)
    # a stack streamed from the reloaded pool gives the same outputs
    ps2 = ST.PagedStack(wl, n_layers=layers, blobs=blobs)
    ps.run_step()
    ps2.run_step()
    torch.cuda.synchronize()
    for g in range(len(S.GROUPS)):
        for y1, y2 in zip(ps.y[layers - 1][g], ps2.y[layers - 1][g]):
            assert torch.equal(y1, y2)
    ps.close()
    ps2.close()


def test_stream_int8_codes_against_oracle(tmp_path):
    """Every INT8 matrix of a Gemma layer streamed from disk equals the
    oracle's quantization of the same memory-mapped fp16 weights."""
    wl = S.WORKLOADS["gemma2_9b_int8"]
    ck = str(tmp_path / "g.safetensors")
    pool = str(tmp_path / "g.qz")
    C.write_synthetic_checkpoint(ck, wl, 1)
    C.quantize_stream(ck, wl, 1, pool)
    hdr, blobs = C.load_pool(pool)
    f = C.SafetensorsFile(ck)
    parts = {(k, p): (o, n, sh) for k, p, o, n, _, sh in hdr["layout"]}
    blob = blobs[0].numpy()
    for m in S.MATS:
        W = np.array(f.array(C.tensor_name(0, m)))
        q_ref, s_ref = O.int8_quantize(W)
        o, n, sh = parts[(m, "q")]
        q = blob[o:o + n].view(np.int8).reshape(sh)
        assert np.array_equal(q[:, :W.shape[1]], q_ref)
        assert not q[:, W.shape[1]:].any()
        o, n, sh = parts[(m, "scale")]
        assert blob[o:o + n].view(np.float32)[0] == s_ref
    f.close()
