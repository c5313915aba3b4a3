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


def make_io(wl: S.Workload, layers: int, batch: int, device):
    """Seeded inputs and output buffers of every group of `layers` layers:
    x[layer][group] = [B, K] fp16, y[layer][group] = list of [B, N] fp16."""
    xs_all, ys_all = [], []
    for l in range(layers):
        xs, ys = [], []
        for g, names in enumerate(S.GROUPS):
            K = wl.shape(names[0])[1]
            xs.append(S.activation(batch, K, S.input_seed(wl, l, g), device=device))
            ys.append([torch.empty((batch, wl.shape(m)[0]), dtype=torch.float16, device=device)
                       for m in names])
        xs_all.append(xs)
        ys_all.append(ys)
    return xs_all, ys_all


class LayerStack:
    def __init__(self, wl: S.Workload, layers: int | None = None, batch: int = 1,
                 device="cuda", keep_fp16: bool = False, fused: bool = False):
        """fused: at batch 1, run each layer's four products as one sequence
        launch (api.gemv_sequence) instead of four launches."""
        self.wl = wl
        self.fused = fused and batch == 1
        self.n_layers = wl.layers if layers is None else layers
        self.batch = batch
        self.device = torch.device(device)
        self.layers: list[Layer] = []
        self.fp16: list[dict] = []          # only if keep_fp16 (tests)
        self.profiles: list[dict] = []
        for l in range(self.n_layers):
            self.layers.append(self._build_layer(l, keep_fp16))
        self._alloc_io()
        # barrier words of the sequence launches (consecutive layers alternate)
        self.sync = torch.zeros((2,), dtype=torch.int32, device=self.device)
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
        self.x, self.y = make_io(self.wl, self.n_layers, self.batch, self.device)

    # ------------------------------------------------------------- run ----
    def launches_per_step(self) -> int:
        """Kernel launches of one step: one per group (one per layer when
        fused); on the tensor-core path (batch > 4) each group adds the launch
        that gathers its inputs."""
        if self.fused:
            return self.n_layers
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

    def run_layer_fused(self, l: int, stream=None):
        """The layer's four products as one dependent sequence launch."""
        mats = self.layers[l].mats
        groups = [[mats[m] for m in names] for names in S.GROUPS]
        xs = [x[0] for x in self.x[l]]
        ys = [[y[0] for y in yy] for yy in self.y[l]]
        api.gemv_sequence(groups, xs, ys, sync=self.sync[l % 2:l % 2 + 1], stream=stream)

    def run_step(self, stream=None):
        for l in range(self.n_layers):
            if self.fused:
                self.run_layer_fused(l, stream)
                continue
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

    def padded_weight_bytes_per_layer(self) -> int:
        """Bytes of one layer's weights as stored (rows padded to 16 bytes)."""
        return sum(w.padded_bytes() for w in self.layers[0].mats.values())

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


def _pad_bytes(wl: S.Workload, m: str) -> int:
    """Padding bytes of matrix m in its packed parts (not algorithmic bytes)."""
    N, K = wl.shape(m)
    if wl.fmt == "int8":
        return N * (_align16(K) - K)
    n_out = api.default_n_out(K)
    ld_out, ld_q4 = api.int4o_layout(N, K, n_out)
    return N * (2 * (ld_out - n_out) + ld_q4 - (K - n_out + 1) // 2)


def _io_bytes(wl: S.Workload, batch: int) -> int:
    """Input and output vectors of one layer (+ the permutation tables for INT4)."""
    b = 0
    for names in S.GROUPS:
        K = wl.shape(names[0])[1]
        b += 2 * batch * K + sum(2 * batch * wl.shape(m)[0] for m in names)
        if wl.fmt == "int4o":
            b += 4 * K
    return b


def blob_layout(wl: S.Workload):
    """Layout of one packed layer in a contiguous blob (host pool, device
    slot, pool file): a list of (key, part, offset, nbytes, dtype, shape),
    16-byte aligned parts, and the blob size.  INT8: q and scale of every
    matrix; INT4: the permutation of every input space, then w_out, q4 and
    scale of every matrix."""
    layout, off = [], 0

    def add(key, part, dtype, shape):
        nonlocal off
        nb = int(torch.empty((), dtype=dtype).element_size())
        for d in shape:
            nb *= d
        layout.append((key, part, off, nb, dtype, tuple(shape)))
        off = _align16(off + nb)

    if wl.fmt == "int8":
        for m in S.MATS:
            N, K = wl.shape(m)
            add(m, "q", torch.int8, (N, _align16(K)))
            add(m, "scale", torch.float32, (1,))
    else:
        for table, members in S.PERM_TABLES.items():
            add(table, "perm", torch.int32, (wl.shape(members[0])[1],))
        for m in S.MATS:
            N, K = wl.shape(m)
            ld_out, ld_q4 = api.int4o_layout(N, K, api.default_n_out(K))
            add(m, "w_out", torch.float16, (N, ld_out))
            add(m, "q4", torch.uint8, (N, ld_q4))
            add(m, "scale", torch.float32, (N,))
    return layout, _align16(off)


def pack_layer(layer: "Layer", layout, blob: torch.Tensor) -> None:
    """Copy a quantized layer's tensors into a host blob at their offsets."""
    for key, part, o, nb, dt, shape in layout:
        t = layer.perms[key] if part == "perm" else getattr(layer.mats[key], part)
        assert t.dtype == dt and tuple(t.shape) == shape, (key, part, t.shape, shape)
        blob[o:o + nb] = t.reshape(-1).view(torch.uint8).cpu()


class PagedStack:
    """A stack whose packed layers live in pinned host memory and stream
    through the pager into two device slots ("Open Origin - ELG Stream
    Layer", Key Features 2-3; "NTransformer", Tier B).

    distinct: number of distinct host layers actually built; layer l of the
    n_layers-deep stack reuses host blob l % distinct (bounds pinned memory).
    """

    def __init__(self, wl: S.Workload, n_layers: int | None = None, distinct: int = 4,
                 device="cuda", blobs: list | None = None):
        """blobs: packed host layers to stream instead of building them (for
        example from a pool file, checkpoint.load_pool); pinned uint8 tensors
        in the layout of blob_layout(wl)."""
        self.wl = wl
        self.n_layers = wl.layers if n_layers is None else n_layers
        self.device = torch.device(device)
        # one blob layout shared by every layer (same shapes)
        self.layout, self.blob_bytes = blob_layout(wl)
        if blobs is None:
            self.distinct = min(distinct, self.n_layers)
            src = LayerStack(wl, layers=self.distinct, device=device)
            self.blobs = []
            for l in range(self.distinct):
                blob = torch.zeros((self.blob_bytes,), dtype=torch.uint8).pin_memory()
                pack_layer(src.layers[l], self.layout, blob)
                self.blobs.append(blob)
            del src
        else:
            assert all(b.numel() == self.blob_bytes and b.is_pinned() for b in blobs)
            self.distinct = min(len(blobs), self.n_layers)
            self.blobs = list(blobs[:self.distinct])
        self.x, self.y = make_io(wl, self.distinct, 1, self.device)
        self.weight_bytes_per_layer = sum(
            nb for key, part, o, nb, dt, shape in self.layout if part != "perm") - sum(
            _pad_bytes(wl, m) for m in S.MATS)
        self.io_bytes_per_layer = _io_bytes(wl, 1)
        self.slots = [torch.empty((self.blob_bytes,), dtype=torch.uint8, device=self.device)
                      for _ in range(2)]
        self.copy_stream = torch.cuda.Stream(device=self.device)
        self.compute_stream = torch.cuda.Stream(device=self.device)
        # the inputs were generated on the current stream: order both streams after it
        cur = torch.cuda.current_stream(self.device)
        self.copy_stream.wait_stream(cur)
        self.compute_stream.wait_stream(cur)
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

    def run_layer(self, mats: dict, hl: int, stream):
        """The four group launches of one layer whose matrices are `mats`
        (views into a device slot), on the inputs and outputs of host layer
        hl."""
        int8 = self.wl.fmt == "int8"
        xs, ys = self.x[hl], self.y[hl]
        for g, names in enumerate(S.GROUPS):
            ws = [mats[m] for m in names]
            outs = [y[0] for y in ys[g]]
            if len(ws) == 1:
                (api.gemv_int8 if int8 else api.gemv_int4_outlier)(ws[0], xs[g][0], outs[0],
                                                                   stream=stream)
            else:
                (api.gemv_int8_grouped if int8 else api.gemv_int4_outlier_grouped)(
                    ws, xs[g][0], outs, stream=stream)

    def run_step(self):
        """All n_layers layers once, each acquired from the pager."""
        for l in range(self.n_layers):
            ptr = self.pager.acquire(l)
            mats = self._views[0 if ptr == self.slots[0].data_ptr() else 1]
            self.run_layer(mats, l % self.distinct, self.compute_stream)
            self.pager.release(l)

    def close(self):
        self.pager.close()


# ------------------------------------------------------------ tiering ---
class TieredStack:
    """Tier A + tier B on one GPU ("NTransformer" summary, 3-Tier Adaptive
    Caching: VRAM-resident layers, then layers kept in pinned RAM): the first
    `resident` layers live in device memory, the others stay in pinned host
    memory and are either streamed through the pager into two device slots
    (mode "paged": host-to-device DMA) or read in place by the zero-copy GEMV
    (mode "zero_copy": the ELG page's pinned pool reached by zero-copy DMA).
    Host layers: `distinct` packed blobs reused cyclically, as in PagedStack.
    Both tiers run on the pager's compute stream.
    """

    def __init__(self, wl: S.Workload, resident: int, n_layers: int | None = None,
                 distinct: int = 4, device="cuda", mode: str = "paged"):
        assert mode in ("paged", "zero_copy")
        self.wl, self.mode = wl, mode
        self.n_layers = wl.layers if n_layers is None else n_layers
        self.resident = max(0, min(resident, self.n_layers))
        self.device = torch.device(device)
        self.host = PagedStack(wl, n_layers=max(1, self.n_layers - self.resident),
                               distinct=distinct, device=device)
        self.dev = LayerStack(wl, layers=self.resident, device=device) if self.resident else None
        # the resident layers were quantized on the current stream; the step
        # runs on the pager's compute stream, which must not start before them
        self.host.compute_stream.wait_stream(torch.cuda.current_stream(self.device))
        # zero-copy: the matrices as views into the pinned host blobs
        self._host_views = ([self.host._mats_in(b) for b in self.host.blobs]
                            if mode == "zero_copy" else None)
        self.weight_bytes_per_layer = self.host.weight_bytes_per_layer
        self.io_bytes_per_layer = self.host.io_bytes_per_layer

    def bytes_per_step(self) -> int:
        return self.n_layers * (self.weight_bytes_per_layer + self.io_bytes_per_layer)

    @property
    def stream(self):
        """The stream a step runs on (the pager's compute stream)."""
        return self.host.compute_stream

    def _run_host_layer_in_place(self, j: int, stream):
        """Layer j of tier B (0-based within the tier), read in place."""
        hl = j % self.host.distinct
        mats = self._host_views[hl]
        xs, ys = self.host.x[hl], self.host.y[hl]
        for g, names in enumerate(S.GROUPS):
            api.gemv_mapped([mats[m] for m in names], xs[g][0], [y[0] for y in ys[g]],
                            stream=stream)

    def run_step(self):
        s = self.stream
        for l in range(self.resident):
            for g in range(len(S.GROUPS)):
                self.dev.run_group(l, g, s)
        if self.n_layers <= self.resident:
            return
        if self.mode == "zero_copy":
            for j in range(self.n_layers - self.resident):
                self._run_host_layer_in_place(j, s)
        else:
            self.host.run_step()

    def close(self):
        self.host.close()
