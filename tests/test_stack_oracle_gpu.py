"""Whole decode steps against the CPU oracle, element by element.

The per-matrix parity tests check each kernel; these check what a stack
binds together: which weights, permutation table and input each launch of a
decode step reads, and where its outputs land.  For every layer of the step
the oracle re-derives the layer from the seeded fp16 weights (quantization,
saliency, outlier selection, packing), checks the stack's codes bit for bit,
and bounds every output by |y - y_ref| <= 1e-3 sum_j |w_ij x_j| + 1 fp16 ulp.

Covered: LayerStack.run_step() and its captured graph with programmatic
dependent launch (Gemma-2-9B INT8 and the 7B INT4-outlier shapes), the
paged Gemma stack (layers streamed from pinned host memory through the
pager, "Open Origin - ELG Stream Layer", Key Features 1-3) and a tiered 3B
stack with both tiers in use ("NTransformer" summary, 3-Tier Adaptive
Caching, tiers A and B), tier B paged or read in place (zero-copy).
"""
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


_CACHE = {}


def oracle_layer(wl: S.Workload, l: int):
    """The oracle's view of layer l of workload wl: per matrix its codes and,
    for the layer's seeded group inputs (batch 1), (y_ref, a_ref)."""
    key = (wl.name, l)
    if key in _CACHE:
        return _CACHE[key]
    Ws = {m: S.weight(*wl.shape(m), S.matrix_seed(wl, l, m), device=DEV, dist=wl.dist)
          .cpu().numpy() for m in S.MATS}
    codes, refs, perms = {}, {}, {}
    if wl.fmt == "int8":
        for m in S.MATS:
            codes[m] = O.int8_quantize(Ws[m])
    else:
        for table, members in S.PERM_TABLES.items():
            K = wl.shape(members[0])[1]
            n_out = O.default_n_out(K)
            colsum = O.saliency_fixed([Ws[m] for m in members])
            prof = S.x_profile(K, n_out, S.profile_seed(wl, l, table), device=DEV).cpu().numpy()
            perms[table] = O.select_outliers(colsum, prof, n_out)
            for m in members:
                codes[m] = O.int4o_quantize(Ws[m], perms[table], n_out)
    for g, names in enumerate(S.GROUPS):
        K = wl.shape(names[0])[1]
        x = S.activation(1, K, S.input_seed(wl, l, g), device=DEV).cpu().numpy()
        for m in names:
            if wl.fmt == "int8":
                q, s = codes[m]
                refs[m] = O.int8_product_ref(q, s, x)
            else:
                table = next(t for t, mem in S.PERM_TABLES.items() if m in mem)
                wo, q4, s = codes[m]
                refs[m] = O.int4o_product_ref(wo, q4, s, perms[table], O.default_n_out(K), K, x)
    out = {"codes": codes, "refs": refs, "perms": perms}
    _CACHE[key] = out
    return out


def check_codes(wl, layer_mats, layer_perms, ref):
    """The stack's quantized layer equals the oracle's bit for bit."""
    for m in S.MATS:
        w = layer_mats[m]
        N, K = wl.shape(m)
        if wl.fmt == "int8":
            q, s = ref["codes"][m]
            assert w.scale.item() == float(s), m
            assert np.array_equal(w.q.cpu().numpy()[:, :K], q), m
        else:
            wo, q4, s = ref["codes"][m]
            assert np.array_equal(w.q4.cpu().numpy(), q4), m
            assert np.array_equal(w.w_out.cpu().numpy().view(np.uint16), wo.view(np.uint16)), m
            assert np.array_equal(w.scale.cpu().numpy(), s), m
    for table, p in layer_perms.items():
        assert np.array_equal(p.cpu().numpy(), ref["perms"][table]), table


def check_outputs(ys_layer, ref, what):
    """ys_layer[g][k]: [1, N] (or [N]) outputs of group g, matrix k."""
    worst = 0.0
    for g, names in enumerate(S.GROUPS):
        for m, y in zip(names, ys_layer[g]):
            y_ref, a_ref = ref["refs"][m]
            got = y.float().cpu().numpy().astype(np.float64).reshape(y_ref.shape)
            tol = O.tolerance(y_ref, a_ref)
            err = np.abs(got - y_ref)
            bad = err > tol
            assert not bad.any(), (f"{what} {m}: {int(bad.sum())}/{bad.size} outside the bound,"
                                   f" worst err/tol {float((err / tol).max()):.3g}")
            worst = max(worst, float((err / tol).max()))
    return worst


def _clear(ys):
    for yl in ys:
        for yy in yl:
            for y in yy:
                y.fill_(float("nan"))


@pytest.mark.parametrize("name", ["gemma2_9b_int8", "llama_7b_int4o"])
def test_layer_stack_step_and_graph_against_oracle(name):
    """Two layers: the plain step and the step captured with programmatic
    dependent launch, every output of every group against the oracle."""
    from weight_only_quantized_dequant_gb300 import stack as ST
    wl = S.WORKLOADS[name]
    st = ST.LayerStack(wl, layers=2)
    torch.cuda.synchronize()
    for l in range(2):
        check_codes(wl, st.layers[l].mats, st.layers[l].perms, oracle_layer(wl, l))
    _clear(st.y)
    st.run_step()
    torch.cuda.synchronize()
    import weight_only_quantized_dequant_gb300 as qz
    assert qz.device_error() == 0
    for l in range(2):
        check_outputs(st.y[l], oracle_layer(wl, l), f"{name} step layer {l}")
    plain = [y.clone() for yl in st.y for yy in yl for y in yy]
    g = st.capture(overlap=True)
    _clear(st.y)
    g.replay()
    torch.cuda.synchronize()
    assert qz.device_error() == 0
    for l in range(2):
        check_outputs(st.y[l], oracle_layer(wl, l), f"{name} graph layer {l}")
    got = [y for yl in st.y for yy in yl for y in yy]
    assert all(torch.equal(a, b) for a, b in zip(plain, got))


def test_paged_gemma_step_against_oracle():
    """The Gemma INT8 stack as the ELG page runs it: 3 layer positions
    streamed from 2 distinct pinned host layers through the pager (layer
    position p reads host layer p % 2), twice over.  After each pass every
    output of both host layers against the oracle; the packed host layers
    against the oracle's codes."""
    from weight_only_quantized_dequant_gb300 import stack as ST
    wl = S.WORKLOADS["gemma2_9b_int8"]
    ps = ST.PagedStack(wl, n_layers=3, distinct=2)
    try:
        torch.cuda.synchronize()
        for l in range(2):
            ref = oracle_layer(wl, l)
            for key, part, o, nb, dt, shape in ps.layout:
                t = ps.blobs[l][o:o + nb].view(dt).view(shape).numpy()
                q, s = ref["codes"][key]
                if part == "q":
                    assert np.array_equal(t[:, :wl.shape(key)[1]], q), key
                    assert not t[:, wl.shape(key)[1]:].any(), key
                else:
                    assert t[0] == s, key
        # positions 0 and 2 read host layer 0 and write the same outputs;
        # the second pass starts over at position 0 (slot reuse, wrap-around)
        for rnd in range(2):
            _clear(ps.y)
            torch.cuda.synchronize()       # the step runs on the pager's stream
            ps.run_step()
            ps.compute_stream.synchronize()
            for hl in range(2):
                check_outputs(ps.y[hl], oracle_layer(wl, hl), f"paged gemma pass {rnd} layer {hl}")
    finally:
        ps.close()


def test_tiered_3b_step_both_tiers_against_oracle():
    """A 3-layer 3B INT4-outlier stack with layer 0 resident in device memory
    (tier A) and layers 1-2 streamed from pinned host memory (tier B, two
    distinct host layers): every output of both tiers against the oracle."""
    from weight_only_quantized_dequant_gb300 import stack as ST
    import weight_only_quantized_dequant_gb300 as qz
    wl = S.WORKLOADS["llama32_3b_int4o"]
    ts = ST.TieredStack(wl, resident=1, n_layers=3, distinct=2)
    try:
        _clear(ts.dev.y)
        _clear(ts.host.y)
        torch.cuda.synchronize()           # the step runs on the pager's stream
        ts.run_step()
        ts.stream.synchronize()
        assert qz.device_error() == 0
        # tier A: resident layer 0 (weights and inputs of layer 0)
        check_codes(wl, ts.dev.layers[0].mats, ts.dev.layers[0].perms, oracle_layer(wl, 0))
        check_outputs(ts.dev.y[0], oracle_layer(wl, 0), "tiered 3b resident layer 0")
        # tier B: positions 1 and 2 read host layers 0 and 1
        for hl in range(2):
            check_outputs(ts.host.y[hl], oracle_layer(wl, hl), f"tiered 3b host layer {hl}")
    finally:
        ts.close()


def test_tiered_3b_zero_copy_step_against_oracle():
    """The same 3-layer 3B stack with tier B read in place from pinned host
    memory by the zero-copy GEMV ("Open Origin - ELG Stream Layer", INT8
    Quantization & Direct Mapping, zero-copy DMA; "NTransformer", Tier B):
    every output of both tiers against the oracle."""
    from weight_only_quantized_dequant_gb300 import stack as ST
    import weight_only_quantized_dequant_gb300 as qz
    wl = S.WORKLOADS["llama32_3b_int4o"]
    ts = ST.TieredStack(wl, resident=1, n_layers=3, distinct=2, mode="zero_copy")
    try:
        _clear(ts.dev.y)
        _clear(ts.host.y)
        torch.cuda.synchronize()
        ts.run_step()
        ts.stream.synchronize()
        assert qz.device_error() == 0
        check_outputs(ts.dev.y[0], oracle_layer(wl, 0), "zero-copy tiered 3b resident layer 0")
        for hl in range(2):
            check_outputs(ts.host.y[hl], oracle_layer(wl, hl), f"zero-copy tiered 3b host layer {hl}")
    finally:
        ts.close()


def test_fused_stack_graph_against_oracle():
    """A decode step of two Gemma layers captured as one sequence launch per
    layer (with programmatic overlap), replayed three times: every output
    against the oracle; the barrier words left at zero."""
    from weight_only_quantized_dequant_gb300 import stack as ST
    import weight_only_quantized_dequant_gb300 as qz
    wl = S.WORKLOADS["gemma2_9b_int8"]
    b = ST.LayerStack(wl, layers=2, fused=True)
    g = b.capture(overlap=True)
    _clear(b.y)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert qz.device_error() == 0
    assert not b.sync.any()
    for l in range(2):
        check_outputs(b.y[l], oracle_layer(wl, l), f"fused gemma layer {l}")
