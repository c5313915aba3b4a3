"""Decoder-layer stack driver: one decode step = every quantized linear of
every layer, four dependent launches per layer ({q,k,v}, {o}, {gate,up},
{down}; matrices of one group share their input and run in one launch).

The pages give no glue between the linears (attention, norms, activations are
not part of the weight path), so each group reads its own seeded input
vector.  Weights are generated, quantized and packed on the GPU by the
library's own kernels; the fp16 originals are dropped after quantization.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

from . import api
from . import synthetic as S


@dataclass
class Layer:
    mats: dict                      # name -> Int8Matrix | Int4oMatrix
    perms: dict = field(default_factory=dict)


class LayerStack:
    def __init__(self, wl: S.Workload, layers: int | None = None, batch: int = 1,
                 device="cuda", keep_fp16: bool = False):
        self.wl = wl
        self.n_layers = wl.layers if layers is None else layers
        self.batch = batch
        self.device = torch.device(device)
        self.layers: list[Layer] = []
        self.fp16: list[dict] = []          # only if keep_fp16 (tests)
        self.profiles: list[dict] = []
        for l in range(self.n_layers):
            self.layers.append(self._build_layer(l, keep_fp16))
        self._alloc_io()
        self.workspace = None
        if batch > 1:  # one workspace for every batched call of the step
            nb = max(api.gemm_workspace_bytes(batch, K, api.default_n_out(K) if wl.fmt == "int4o" else 0)
                     for K in {wl.shape(m)[1] for m in S.MATS})
            self.workspace = torch.empty((nb,), dtype=torch.uint8, device=self.device)

    # ------------------------------------------------------------ build ---
    def _build_layer(self, l: int, keep_fp16: bool) -> Layer:
        wl, dev = self.wl, self.device
        Ws = {m: S.weight(*wl.shape(m), S.matrix_seed(wl, l, m), device=dev, dist=wl.dist)
              for m in S.MATS}
        if keep_fp16:
            self.fp16.append({m: W.cpu() for m, W in Ws.items()})
        layer = Layer({})
        if wl.fmt == "int8":
            for m in S.MATS:
                layer.mats[m] = api.quantize_int8(Ws[m])
        else:
            profs = {}
            for table, members in S.PERM_TABLES.items():
                K = wl.shape(members[0])[1]
                n_out = api.default_n_out(K)
                colsum = torch.zeros((K,), dtype=torch.int64, device=dev)
                for m in members:
                    api.saliency_accumulate(Ws[m], colsum)
                prof = S.x_profile(K, n_out, S.profile_seed(wl, l, table), device=dev)
                profs[table] = prof
                perm = api.select_outliers(colsum, prof, n_out)
                layer.perms[table] = perm
                for m in members:
                    layer.mats[m] = api.quantize_int4_outlier(Ws[m], perm, n_out)
            if keep_fp16:
                self.profiles.append({t: p.cpu() for t, p in profs.items()})
        del Ws
        return layer

    def _alloc_io(self):
        B, dev = self.batch, self.device
        self.x = []   # [layer][group] -> [B, K] fp16
        self.y = []   # [layer][group] -> list of [B, N] fp16
        for l in range(self.n_layers):
            xs, ys = [], []
            for g, names in enumerate(S.GROUPS):
                K = self.wl.shape(names[0])[1]
                xs.append(S.activation(B, K, S.input_seed(self.wl, l, g), device=dev))
                ys.append([torch.empty((B, self.wl.shape(m)[0]), dtype=torch.float16, device=dev)
                           for m in names])
            self.x.append(xs)
            self.y.append(ys)

    # ------------------------------------------------------------- run ----
    def launches_per_step(self) -> int:
        """Kernel launches of one step: one per group; on the tensor-core path
        (batch > 4) each group adds the launch that gathers its inputs."""
        per_group = 1 if self.batch <= 4 else 2
        return self.n_layers * len(S.GROUPS) * per_group

    def run_group(self, l: int, g: int, stream=None):
        names = S.GROUPS[g]
        mats = [self.layers[l].mats[m] for m in names]
        x, ys = self.x[l][g], self.y[l][g]
        int8 = self.wl.fmt == "int8"
        if self.batch == 1:
            outs = [y[0] for y in ys]
            if len(mats) == 1:
                fn = api.gemv_int8 if int8 else api.gemv_int4_outlier
                fn(mats[0], x[0], outs[0], stream=stream)
            else:
                fn = api.gemv_int8_grouped if int8 else api.gemv_int4_outlier_grouped
                fn(mats, x[0], outs, stream=stream)
        elif len(mats) == 1:
            fn = api.gemm_int8 if int8 else api.gemm_int4_outlier
            fn(mats[0], x, ys[0], stream=stream, workspace=self.workspace)
        else:
            fn = api.gemm_int8_grouped if int8 else api.gemm_int4_outlier_grouped
            fn(mats, x, ys, stream=stream, workspace=self.workspace)

    def run_step(self, stream=None):
        for l in range(self.n_layers):
            for g in range(len(S.GROUPS)):
                self.run_group(l, g, stream)

    def capture(self, overlap: bool = True) -> torch.cuda.CUDAGraph:
        """CUDA graph of one decode step (all layers).  With overlap, each
        launch may start while the previous one drains (weights are static
        during decode)."""
        prev = api.get_overlap()
        api.set_overlap(overlap)
        try:
            return self._capture()
        finally:
            api.set_overlap(prev)

    def _capture(self) -> torch.cuda.CUDAGraph:
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):
            self.run_step(s)          # warm-up outside capture
        torch.cuda.current_stream(self.device).wait_stream(s)
        torch.cuda.synchronize(self.device)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            self.run_step(s)
        return graph

    # --------------------------------------------------------- accounting --
    def weight_bytes_per_layer(self) -> int:
        """Algorithmic bytes of one layer's weights (codes, outliers, scales)."""
        return sum(w.nbytes() for w in self.layers[0].mats.values())

    def io_bytes_per_layer(self) -> int:
        """Input and output vectors (+ the permutation tables for INT4)."""
        B, wl = self.batch, self.wl
        b = 0
        for names in S.GROUPS:
            K = wl.shape(names[0])[1]
            b += 2 * B * K + sum(2 * B * wl.shape(m)[0] for m in names)
            if wl.fmt == "int4o":
                b += 4 * K
        return b

    def bytes_per_step(self) -> int:
        return self.n_layers * (self.weight_bytes_per_layer() + self.io_bytes_per_layer())

    def h2d_bytes_per_step(self) -> int:
        return sum(x.numel() * 2 for xs in self.x for x in xs)

    def d2h_bytes_per_step(self) -> int:
        return sum(y.numel() * 2 for ys in self.y for yy in ys for y in yy)


# ---------------------------------------------------------------- paging ---
def _align16(n: int) -> int:
    return (n + 15) // 16 * 16


class PagedStack:
    """A stack whose packed layers live in pinned host memory and stream
    through the pager into two device slots ("Open Origin - ELG Stream
    Layer", Key Features 2-3; "NTransformer", Tier B).

    distinct: number of distinct host layers actually built; layer l of the
    n_layers-deep stack reuses host blob l % distinct (bounds pinned memory).
    """

    def __init__(self, wl: S.Workload, n_layers: int | None = None, distinct: int = 4,
                 device="cuda"):
        self.wl = wl
        self.n_layers = wl.layers if n_layers is None else n_layers
        self.distinct = min(distinct, self.n_layers)
        self.device = torch.device(device)
        src = LayerStack(wl, layers=self.distinct, device=device)
        self.x, self.y = src.x, src.y
        # one blob layout shared by every layer (same shapes)
        self.layout = []  # (kind, name, offset, nbytes, dtype, shape)
        off = 0
        lay0 = src.layers[0]
        if wl.fmt == "int8":
            for m in S.MATS:
                w = lay0.mats[m]
                for part, t in (("q", w.q), ("scale", w.scale)):
                    self.layout.append((m, part, off, t.numel() * t.element_size(), t.dtype,
                                        tuple(t.shape)))
                    off = _align16(off + t.numel() * t.element_size())
        else:
            for table in S.PERM_TABLES:
                t = lay0.perms[table]
                self.layout.append((table, "perm", off, t.numel() * 4, t.dtype, tuple(t.shape)))
                off = _align16(off + t.numel() * 4)
            for m in S.MATS:
                w = lay0.mats[m]
                for part, t in (("w_out", w.w_out), ("q4", w.q4), ("scale", w.scale)):
                    nb = t.numel() * t.element_size()
                    self.layout.append((m, part, off, nb, t.dtype, tuple(t.shape)))
                    off = _align16(off + nb)
        self.blob_bytes = _align16(off)
        self.blobs = []
        for l in range(self.distinct):
            blob = torch.zeros((self.blob_bytes,), dtype=torch.uint8).pin_memory()
            lay = src.layers[l]
            for key, part, o, nb, dt, shape in self.layout:
                if part == "perm":
                    t = lay.perms[key]
                else:
                    t = getattr(lay.mats[key], part)
                blob[o:o + nb] = t.reshape(-1).view(torch.uint8).cpu()
            self.blobs.append(blob)
        self.weight_bytes_per_layer = src.weight_bytes_per_layer()
        self.io_bytes_per_layer = src.io_bytes_per_layer()
        del src
        self.slots = [torch.empty((self.blob_bytes,), dtype=torch.uint8, device=self.device)
                      for _ in range(2)]
        self.copy_stream = torch.cuda.Stream(device=self.device)
        self.compute_stream = torch.cuda.Stream(device=self.device)
        hosts = [self.blobs[l % self.distinct] for l in range(self.n_layers)]
        self.pager = api.Pager(hosts, self.slots, self.copy_stream, self.compute_stream)
        self._views = [self._mats_in(slot) for slot in self.slots]

    def _mats_in(self, slot: torch.Tensor) -> dict:
        """The layer's matrices as views into a device slot."""
        parts, perms = {}, {}
        for key, part, o, nb, dt, shape in self.layout:
            t = slot[o:o + nb].view(dt).view(shape)
            if part == "perm":
                perms[key] = t
            else:
                parts.setdefault(key, {})[part] = t
        mats = {}
        for m in S.MATS:
            N, K = self.wl.shape(m)
            if self.wl.fmt == "int8":
                mats[m] = api.Int8Matrix(parts[m]["q"], parts[m]["scale"], N, K)
            else:
                table = next(t for t, mem in S.PERM_TABLES.items() if m in mem)
                mats[m] = api.Int4oMatrix(perms[table], parts[m]["w_out"], parts[m]["q4"],
                                          parts[m]["scale"], N, K, api.default_n_out(K))
        return mats

    def run_step(self):
        """All n_layers layers once, each acquired from the pager."""
        cs = self.compute_stream
        int8 = self.wl.fmt == "int8"
        for l in range(self.n_layers):
            ptr = self.pager.acquire(l)
            mats = self._views[0 if ptr == self.slots[0].data_ptr() else 1]
            xs, ys = self.x[l % self.distinct], self.y[l % self.distinct]
            for g, names in enumerate(S.GROUPS):
                ws = [mats[m] for m in names]
                outs = [y[0] for y in ys[g]]
                if len(ws) == 1:
                    (api.gemv_int8 if int8 else api.gemv_int4_outlier)(ws[0], xs[g][0], outs[0],
                                                                       stream=cs)
                else:
                    (api.gemv_int8_grouped if int8 else api.gemv_int4_outlier_grouped)(
                        ws, xs[g][0], outs, stream=cs)
            self.pager.release(l)

    def close(self):
        self.pager.close()


# ------------------------------------------------------------ tiering ---
class TieredStack:
    """Tier A + tier B on one GPU ("NTransformer" summary, 3-Tier Adaptive
    Caching: VRAM-resident layers, then layers streamed from pinned RAM by
    host-to-device DMA): the first `resident` layers live in device memory,
    the others stay in pinned host memory and stream through the pager into
    two device slots.  Host layers: `distinct` packed blobs reused cyclically,
    as in PagedStack.  Both tiers run on the pager's compute stream.
    """

    def __init__(self, wl: S.Workload, resident: int, n_layers: int | None = None,
                 distinct: int = 4, device="cuda"):
        self.wl = wl
        self.n_layers = wl.layers if n_layers is None else n_layers
        self.resident = max(0, min(resident, self.n_layers))
        self.device = torch.device(device)
        self.host = PagedStack(wl, n_layers=max(1, self.n_layers - self.resident),
                               distinct=distinct, device=device)
        self.dev = LayerStack(wl, layers=self.resident, device=device) if self.resident else None
        self.weight_bytes_per_layer = self.host.weight_bytes_per_layer
        self.io_bytes_per_layer = self.host.io_bytes_per_layer

    def bytes_per_step(self) -> int:
        return self.n_layers * (self.weight_bytes_per_layer + self.io_bytes_per_layer)

    @property
    def stream(self):
        """The stream a step runs on (the pager's compute stream)."""
        return self.host.compute_stream

    def run_step(self):
        s = self.stream
        for l in range(self.resident):
            for g in range(len(S.GROUPS)):
                self.dev.run_group(l, g, s)
        if self.n_layers > self.resident:
            self.host.run_step()

    def close(self):
        self.host.close()
