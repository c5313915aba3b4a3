"""The offline side of the path: weights streamed from a checkpoint file on
disk, quantized layer by layer on the GPU, and the packed pool written to (and
read back from) a file.

"On-The-Fly Weight Synthesizer (OTF-LLM Engine)", key innovation 2: the
quantizer memory-maps the checkpoint (safetensors.safe_open) and streams it
layer by layer, so host memory stays small.  "Open Origin - ELG Stream Layer",
INT8 Quantization & Direct Mapping: the INT8 tensors go into a pre-allocated
pinned pool that the GPU reads by DMA.

No trained checkpoint exists on this machine, so `write_synthetic_checkpoint`
writes the seeded synthetic weights of a workload in the safetensors layout
(8-byte little-endian header length, JSON header of name -> dtype, shape and
data offsets, then the raw data), with Llama-style tensor names.

Host memory held by `quantize_stream`: one pinned staging buffer of the
largest matrix (fp16) and one pinned blob of a packed layer; the checkpoint
pages come and go through the page cache.

Pool file: b"QZPOOL01", a little-endian u64 header length, a JSON header
(workload, format, layer count, blob size, alignment, the blob layout), zero
padding to 4096 bytes, then one packed layer per 4096-aligned slot.
"""
from __future__ import annotations

import json
import mmap
import os
import struct

import numpy as np
import torch

from . import api
from . import synthetic as S
from .stack import Layer, blob_layout

_HF = {"q": "self_attn.q_proj", "k": "self_attn.k_proj", "v": "self_attn.v_proj",
       "o": "self_attn.o_proj", "gate": "mlp.gate_proj", "up": "mlp.up_proj",
       "down": "mlp.down_proj"}
_ST_DTYPES = {"F16": np.float16, "F32": np.float32, "I8": np.int8, "U8": np.uint8,
              "I32": np.int32}
POOL_MAGIC = b"QZPOOL01"
POOL_ALIGN = 4096


def tensor_name(layer: int, m: str) -> str:
    return f"model.layers.{layer}.{_HF[m]}.weight"


def _round(n: int, a: int) -> int:
    return (n + a - 1) // a * a


# ------------------------------------------------------------ checkpoint ---
def write_synthetic_checkpoint(path: str, wl: S.Workload, layers: int, device="cuda") -> int:
    """Write the seeded fp16 weights of the first `layers` layers as a
    safetensors file; returns its size in bytes.  One matrix at a time is
    generated (on `device`) and written."""
    entries, off = {}, 0
    for l in range(layers):
        for m in S.MATS:
            N, K = wl.shape(m)
            entries[tensor_name(l, m)] = {"dtype": "F16", "shape": [N, K],
                                          "data_offsets": [off, off + 2 * N * K]}
            off += 2 * N * K
    entries["__metadata__"] = {"format": "pt", "workload": wl.name}
    hdr = json.dumps(entries, separators=(",", ":")).encode()
    hdr += b" " * ((-len(hdr)) % 8)
    with open(path, "wb") as f:
        f.write(struct.pack("<Q", len(hdr)))
        f.write(hdr)
        for l in range(layers):
            for m in S.MATS:
                W = S.weight(*wl.shape(m), S.matrix_seed(wl, l, m), device=device, dist=wl.dist)
                f.write(W.cpu().numpy().tobytes())
                del W
    return 8 + len(hdr) + off


class SafetensorsFile:
    """Read-only memory map of a safetensors file; tensors are zero-copy
    numpy views of the mapping."""

    def __init__(self, path: str):
        self._f = open(path, "rb")
        self._mm = mmap.mmap(self._f.fileno(), 0, access=mmap.ACCESS_READ)
        (n,) = struct.unpack_from("<Q", self._mm, 0)
        if n > len(self._mm) - 8:
            raise ValueError("safetensors header length past the end of the file")
        self.header = json.loads(bytes(self._mm[8:8 + n]).decode("utf-8"))
        self.metadata = self.header.pop("__metadata__", {})
        self._base = 8 + n

    def names(self):
        return list(self.header)

    def array(self, name: str) -> np.ndarray:
        e = self.header[name]
        dt = np.dtype(_ST_DTYPES[e["dtype"]])
        b, en = e["data_offsets"]
        count = (en - b) // dt.itemsize
        shape = tuple(e["shape"])
        if count != int(np.prod(shape)) or self._base + en > len(self._mm):
            raise ValueError(f"bad extent for {name}")
        return np.frombuffer(self._mm, dtype=dt, count=count, offset=self._base + b).reshape(shape)

    def close(self):
        """Unmap now if no view is alive, else when the last view goes."""
        try:
            self._mm.close()
        except BufferError:
            pass
        self._f.close()


# ------------------------------------------------------------- pool file ---
class PoolWriter:
    def __init__(self, path: str, wl: S.Workload, layers: int):
        self.layout, self.blob_bytes = blob_layout(wl)
        self.slot = _round(self.blob_bytes, POOL_ALIGN)
        hdr = {"workload": wl.name, "format": wl.fmt, "layers": layers,
               "blob_bytes": self.blob_bytes, "slot_bytes": self.slot, "align": POOL_ALIGN,
               "layout": [[k, p, o, n, str(dt).replace("torch.", ""), list(sh)]
                          for k, p, o, n, dt, sh in self.layout]}
        body = json.dumps(hdr, separators=(",", ":")).encode()
        self.data_start = _round(16 + len(body), POOL_ALIGN)
        self._f = open(path, "wb")
        self._f.write(POOL_MAGIC + struct.pack("<Q", len(body)) + body)
        self._f.write(b"\0" * (self.data_start - 16 - len(body)))
        self.layers, self.written = layers, 0

    def write(self, blob: torch.Tensor) -> None:
        assert blob.numel() == self.blob_bytes and self.written < self.layers
        self._f.write(blob.numpy().tobytes())
        self._f.write(b"\0" * (self.slot - self.blob_bytes))
        self.written += 1

    def close(self) -> None:
        assert self.written == self.layers, "pool file short of layers"
        self._f.close()


def read_pool_header(path: str) -> dict:
    with open(path, "rb") as f:
        head = f.read(16)
        if head[:8] != POOL_MAGIC:
            raise ValueError("not a packed pool file")
        (n,) = struct.unpack("<Q", head[8:16])
        hdr = json.loads(f.read(n).decode("utf-8"))
    hdr["data_start"] = _round(16 + n, hdr["align"])
    return hdr


def load_pool(path: str, layers: list[int] | None = None,
              pin: bool = True) -> tuple[dict, list[torch.Tensor]]:
    """Read packed layers (all, or the listed ones) into host blobs, pinned
    unless pin is False."""
    hdr = read_pool_header(path)
    want = range(hdr["layers"]) if layers is None else layers
    blobs = []
    with open(path, "rb", buffering=0) as f:
        for l in want:
            if not 0 <= l < hdr["layers"]:
                raise IndexError(l)
            blob = torch.empty((hdr["blob_bytes"],), dtype=torch.uint8, pin_memory=pin)
            f.seek(hdr["data_start"] + l * hdr["slot_bytes"])
            view = memoryview(blob.numpy())
            got = 0
            while got < hdr["blob_bytes"]:
                n = f.readinto(view[got:])
                if not n:
                    raise ValueError("pool file truncated")
                got += n
            blobs.append(blob)
    return hdr, blobs


# ------------------------------------------------- streaming quantizer ---
def quantize_stream(ckpt_path: str, wl: S.Workload, layers: int, pool_path: str,
                    device="cuda") -> dict:
    """Quantize `layers` layers of the checkpoint into a pool file, one layer
    at a time: every matrix goes page cache -> pinned staging -> device, is
    quantized there by the library (INT8 per tensor, or saliency, outlier
    selection and INT4 packing per input space), and the packed layer goes
    device -> pinned blob -> file."""
    ck = SafetensorsFile(ckpt_path)
    writer = PoolWriter(pool_path, wl, layers)
    biggest = max(wl.shape(m)[0] * wl.shape(m)[1] for m in S.MATS)
    staging = torch.empty((biggest,), dtype=torch.float16).pin_memory()
    blob = torch.zeros((writer.blob_bytes,), dtype=torch.uint8).pin_memory()  # padding stays 0
    dev = torch.device(device)
    read_bytes = 0
    for l in range(layers):
        Ws = {}
        for m in S.MATS:
            a = ck.array(tensor_name(l, m))
            st = staging[:a.size].view(a.shape)
            st.numpy()[...] = a                      # page cache -> pinned
            read_bytes += a.nbytes
            del a
            Ws[m] = st.to(dev, non_blocking=True)
            torch.cuda.current_stream(dev).synchronize()  # staging is reused next
        layer = Layer({})
        if wl.fmt == "int8":
            for m in S.MATS:
                layer.mats[m] = api.quantize_int8(Ws[m])
        else:
            for table, members in S.PERM_TABLES.items():
                K = wl.shape(members[0])[1]
                n_out = api.default_n_out(K)
                colsum = torch.zeros((K,), dtype=torch.int64, device=dev)
                for m in members:
                    api.saliency_accumulate(Ws[m], colsum)
                prof = S.x_profile(K, n_out, S.profile_seed(wl, l, table), device=dev)
                layer.perms[table] = api.select_outliers(colsum, prof, n_out)
                for m in members:
                    layer.mats[m] = api.quantize_int4_outlier(Ws[m], layer.perms[table], n_out)
        del Ws
        for key, part, o, nb, dt, shape in writer.layout:
            t = layer.perms[key] if part == "perm" else getattr(layer.mats[key], part)
            blob[o:o + nb].copy_(t.reshape(-1).view(torch.uint8), non_blocking=True)
        torch.cuda.current_stream(dev).synchronize()
        writer.write(blob)
    writer.close()
    ck.close()
    return {"layers": layers, "checkpoint_bytes": read_bytes,
            "pool_bytes": layers * writer.blob_bytes,
            "host_buffer_bytes": staging.numel() * 2 + blob.numel()}
