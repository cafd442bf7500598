"""First calls in a fresh process.

Kernel launch settings that persist inside a process (the per-function opt-in to more than
48 KB of shared memory) must be made by the call that needs them, not left to an earlier call
with a larger shape. Each case runs the whole path once in a new Python process, on a shape
whose kernels need such settings, and checks the mask and the output against the oracle.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

CODE = r"""
import sys
sys.path.insert(0, {root!r})
sys.path.insert(0, {tests!r})
import numpy as np
import torch
import oracle as O
import workloads as WL
import free_sparse_swiglu_stage1_b300 as P
from gpu_helpers import check_band, check_y, cuda, random_layer

d, F, B = {d}, {F}, {B}
lay = random_layer(d, F, seed=77)
ws = P.prox_workspace(d, F, B)
x = WL.make_random_tokens(B, d, seed=78)
k = P.prox_k_for(0.7, F)
idx = torch.empty((B, k), dtype=torch.int32, device="cuda")
y = P.prox_ffn_forward(lay.packed, cuda(x), 0.7, 0.5, ws, idx_out=idx).cpu().numpy()
assert P.prox_get_status(ws) == 0
idx = idx.cpu().numpy()
for b in sorted({{0, B - 1}}):
    st = O.stage1_token(lay.o, x[b], 0.5)
    check_band(st["sigma"], k, idx[b])
    y_ref, _ = O.stage2_exact(x[b], lay.o.w_gate, lay.o.w_up, lay.o.w_down, idx[b])
    check_y(y[b], y_ref)
yd = P.prox_dense_ffn(lay.packed, cuda(x), ws).cpu().numpy()
check_y(yd[0], O.dense_ffn(x[0], lay.o.w_gate, lay.o.w_up, lay.o.w_down))
print("ok")
"""


@pytest.mark.parametrize("d,F,B", [(4096, 1024, 1), (4096, 1024, 4), (8192, 512, 2),
                                   (16384, 256, 1)])
def test_first_call_in_fresh_process(d, F, B):
    code = CODE.format(root=ROOT, tests=HERE, d=d, F=F, B=B)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-4000:]
