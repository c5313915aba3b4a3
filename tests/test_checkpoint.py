"""The offline side on the host: the checkpoint file format the streaming
quantizer reads, and the packed pool file it writes.  No GPU needed."""
import json
import os
import struct

import numpy as np
import pytest
import torch

from weight_only_quantized_dequant_gb300 import checkpoint as C
from weight_only_quantized_dequant_gb300 import stack as ST
from weight_only_quantized_dequant_gb300 import synthetic as S


def test_checkpoint_layout_by_hand(tmp_path):
    """The file is the safetensors layout: u64 LE header length, JSON header
    (8-byte padded), then the tensors back to back in the header's order."""
    wl = S.WORKLOADS["tiny_int8"]
    path = str(tmp_path / "tiny.safetensors")
    size = C.write_synthetic_checkpoint(path, wl, 1, device="cpu")
    raw = open(path, "rb").read()
    assert len(raw) == size
    (n,) = struct.unpack("<Q", raw[:8])
    assert n % 8 == 0
    hdr = json.loads(raw[8:8 + n])
    assert hdr.pop("__metadata__")["workload"] == "tiny_int8"
    assert sorted(hdr) == sorted(C.tensor_name(0, m) for m in S.MATS)
    ends = sorted(e["data_offsets"] for e in hdr.values())
    assert ends[0][0] == 0 and all(a[1] == b[0] for a, b in zip(ends, ends[1:]))
    assert 8 + n + ends[-1][1] == size
    e = hdr["model.layers.0.mlp.down_proj.weight"]
    assert e["dtype"] == "F16" and e["shape"] == [256, 256]
    b, en = e["data_offsets"]
    W = np.frombuffer(raw[8 + n + b:8 + n + en], dtype=np.float16).reshape(256, 256)
    want = S.weight(256, 256, S.matrix_seed(wl, 0, "down"), device="cpu", dist=wl.dist).numpy()
    assert np.array_equal(W.view(np.uint16), want.view(np.uint16))


def test_reader_views_and_bad_files(tmp_path):
    wl = S.WORKLOADS["tiny_int8"]
    path = str(tmp_path / "tiny.safetensors")
    C.write_synthetic_checkpoint(path, wl, 1, device="cpu")
    ck = C.SafetensorsFile(path)
    assert ck.metadata["format"] == "pt"
    for m in S.MATS:
        a = ck.array(C.tensor_name(0, m))
        want = S.weight(*wl.shape(m), S.matrix_seed(wl, 0, m), device="cpu", dist=wl.dist)
        assert a.dtype == np.float16 and np.array_equal(a.view(np.uint16),
                                                       want.numpy().view(np.uint16))
        assert not a.flags.writeable               # a view of the read-only mapping
    ck.close()
    bad = str(tmp_path / "bad.safetensors")
    with open(bad, "wb") as f:
        f.write(struct.pack("<Q", 1 << 40) + b"{}")
    with pytest.raises(ValueError):
        C.SafetensorsFile(bad)


@pytest.mark.parametrize("name", ["llama32_3b_int4o", "gemma2_9b_int8"])
def test_pool_file_round_trip(tmp_path, name):
    wl = S.WORKLOADS[name]
    layout, nb = ST.blob_layout(wl)
    path = str(tmp_path / "pool.qz")
    w = C.PoolWriter(path, wl, 3)
    rng = np.random.default_rng(5)
    blobs = [torch.from_numpy(rng.integers(0, 256, nb, dtype=np.uint8)) for _ in range(3)]
    for b in blobs:
        w.write(b)
    w.close()
    hdr = C.read_pool_header(path)
    assert hdr["layers"] == 3 and hdr["blob_bytes"] == nb and hdr["data_start"] % 4096 == 0
    assert hdr["slot_bytes"] % 4096 == 0 and hdr["slot_bytes"] >= nb
    assert [tuple(e[:4]) for e in hdr["layout"]] == [(k, p, o, n) for k, p, o, n, _, _ in layout]
    assert os.path.getsize(path) == hdr["data_start"] + 3 * hdr["slot_bytes"]
    _, got = C.load_pool(path, pin=False)
    assert all(torch.equal(a, b) for a, b in zip(got, blobs))
    _, one = C.load_pool(path, layers=[2], pin=False)
    assert torch.equal(one[0], blobs[2])
    with pytest.raises(IndexError):
        C.load_pool(path, layers=[3], pin=False)


def test_pool_file_rejects_foreign_and_short_files(tmp_path):
    p = str(tmp_path / "x.qz")
    with open(p, "wb") as f:
        f.write(b"NOTAPOOL" + b"\0" * 64)
    with pytest.raises(ValueError):
        C.read_pool_header(p)
    wl = S.WORKLOADS["llama32_3b_int4o"]
    w = C.PoolWriter(str(tmp_path / "short.qz"), wl, 2)
    w.write(torch.zeros((ST.blob_layout(wl)[1],), dtype=torch.uint8))
    with pytest.raises(AssertionError):
        w.close()                                 # one layer short
    w._f.close()
    with pytest.raises(ValueError):
        C.load_pool(str(tmp_path / "short.qz"), layers=[1], pin=False)
