"""The tensor-core path's first call in a process made inside a CUDA-graph
capture: its one-time host queries (cluster occupancy per schedule) must not
break the capture, and the replayed graph must give the product the oracle
gives.  Runs in a child process so that nothing was launched before."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import numpy as np, torch
import weight_only_quantized_dequant_gb300 as qz
from weight_only_quantized_dequant_gb300 import synthetic as S
from oracle import qz_oracle as O
N, K, B, n_out = 700, 3072, 16, 31
W = S.weight(N, K, 9800, device="cuda")
colsum = torch.zeros((K,), dtype=torch.int64, device="cuda")
qz.saliency_accumulate(W, colsum)
perm = qz.select_outliers(colsum, S.x_profile(K, n_out, 9801, device="cuda"), n_out)
w = qz.quantize_int4_outlier(W, perm, n_out)
X = S.activation(B, K, 9802, device="cuda")
Y = torch.zeros((B, N), dtype=torch.float16, device="cuda")
ws = torch.empty((qz.gemm_workspace_bytes(B, K, n_out),), dtype=torch.uint8, device="cuda")
torch.cuda.synchronize()
s = torch.cuda.Stream()
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g, stream=s):
    qz.gemm_int4_outlier(w, X, Y, stream=s, workspace=ws)
g.replay()
torch.cuda.synchronize()
assert qz.device_error() == 0
pn = perm.cpu().numpy()
wo, q4, sc = O.int4o_quantize(W.cpu().numpy(), pn, n_out)
y_ref, a_ref = O.int4o_product_ref(wo, q4, sc, pn, n_out, K, X.cpu().numpy())
err = np.abs(Y.float().cpu().numpy().astype(np.float64) - y_ref)
assert (err <= O.tolerance(y_ref, a_ref)).all()
print("ok")
"""


def test_first_tensor_core_call_inside_graph_capture():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_only_quantized_dequant_gb300 import build
    build.build()
    out = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, capture_output=True, text=True,
                         timeout=300)
    assert out.returncode == 0 and out.stdout.strip().endswith("ok"), out.stderr[-2000:]
