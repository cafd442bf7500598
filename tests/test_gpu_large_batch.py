"""Batches above one tile (PROX_MAX_BATCH = 16 tokens) through the C ABI: every token against
the oracle (its own input set and mask, technical summary "Significance and Claims": large-batch
serving is the method's open limitation, so a large call runs tile by tile), and every tile
bit-identical to a tile-sized call of its own.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
import free_sparse_swiglu_stage1_b300 as P
from gpu_helpers import check_band, check_y, cuda, workload_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def layer_1024():
    return workload_layer(1, 0)


def _tiles(B):
    return [(t0, min(16, B - t0)) for t0 in range(0, B, 16)]


@pytest.mark.parametrize("B", [17, 21, 40])
def test_forward_every_token_vs_oracle(layer_1024, B):
    lay = layer_1024
    s, s_in = 0.5, 0.5
    x = WL.make_tokens(1, range(100, 100 + B))
    ws = P.prox_workspace(lay.d, lay.F, B)
    assert ws.nbytes == P.prox_workspace_bytes(lay.d, lay.F, 16)
    k = O.k_for(s, lay.F)
    idx = torch.empty((B, k), dtype=torch.int32, device="cuda")
    y = P.prox_ffn_forward(lay.packed, cuda(x), s, s_in, ws, idx_out=idx)
    assert P.prox_get_status(ws) == 0
    y, idx = y.cpu().numpy(), idx.cpu().numpy()
    for b in range(B):
        check_band(O.stage1_token(lay.o, x[b], s_in)["sigma"], k, idx[b])
        y_ref, _ = O.stage2_exact(x[b], lay.o.w_gate, lay.o.w_up, lay.o.w_down, idx[b])
        check_y(y[b], y_ref)
    # each tile is exactly a call of its own size
    for t0, nb in _tiles(B):
        wt = P.prox_workspace(lay.d, lay.F, nb)
        it = torch.empty((nb, k), dtype=torch.int32, device="cuda")
        yt = P.prox_ffn_forward(lay.packed, cuda(x[t0:t0 + nb]), s, s_in, wt, idx_out=it)
        np.testing.assert_array_equal(it.cpu().numpy(), idx[t0:t0 + nb])
        np.testing.assert_array_equal(yt.cpu().numpy().view(np.uint32), y[t0:t0 + nb].view(np.uint32))


def test_mask_given_and_dense_vs_oracle(layer_1024):
    lay = layer_1024
    B, s, s_in = 35, 0.7, 0.5
    x = WL.make_tokens(1, range(200, 200 + B))
    ws = P.prox_workspace(lay.d, lay.F, B)
    k = O.k_for(s, lay.F)
    idx = P.prox_build_mask(lay.packed, cuda(x), s, s_in, ws)
    idx_np = idx.cpu().numpy()
    for b in range(B):
        check_band(O.stage1_token(lay.o, x[b], s_in)["sigma"], k, idx_np[b])
    # Stage 2 over a given mask, and the dense FFN, tile by tile
    y = P.prox_sparse_ffn(lay.packed, cuda(x), idx, ws).cpu().numpy()
    yd = P.prox_dense_ffn(lay.packed, cuda(x), ws).cpu().numpy()
    assert P.prox_get_status(ws) == 0
    for b in range(B):
        y_ref, _ = O.stage2_exact(x[b], lay.o.w_gate, lay.o.w_up, lay.o.w_down, idx_np[b])
        check_y(y[b], y_ref)
        check_y(yd[b], O.dense_ffn(x[b], lay.o.w_gate, lay.o.w_up, lay.o.w_down))


def test_host_entry_point_matches_device(layer_1024):
    lay = layer_1024
    B, s, s_in = 19, 0.5, 0.5
    x = WL.make_tokens(1, range(300, 300 + B))
    ws = P.prox_workspace(lay.d, lay.F, B)
    y_dev = P.prox_ffn_forward(lay.packed, cuda(x), s, s_in, ws).cpu().numpy()
    y_host = P.prox_ffn_forward_host(lay.packed, torch.from_numpy(x).pin_memory(), s, s_in, ws)
    np.testing.assert_array_equal(y_host.numpy().view(np.uint32), y_dev.view(np.uint32))


def test_full_size_batch_32_sampled():
    """The 4096 x 14336 layer at 32 tokens (two full tiles), sampled tokens of both tiles."""
    lay = workload_layer(3, 0)
    B, s, s_in = 32, 0.7, 0.5
    x = WL.make_tokens(3, range(B))
    ws = P.prox_workspace(lay.d, lay.F, B)
    k = O.k_for(s, lay.F)
    idx = torch.empty((B, k), dtype=torch.int32, device="cuda")
    y = P.prox_ffn_forward(lay.packed, cuda(x), s, s_in, ws, idx_out=idx).cpu().numpy()
    assert P.prox_get_status(ws) == 0
    idx = idx.cpu().numpy()
    for b in (0, 15, 16, 31):
        check_band(O.stage1_token(lay.o, x[b], s_in)["sigma"], k, idx[b])
        y_ref, _ = O.stage2_exact(x[b], lay.o.w_gate, lay.o.w_up, lay.o.w_down, idx[b])
        check_y(y[b], y_ref)


def test_limits(layer_1024):
    lay = layer_1024
    assert P.prox_workspace_bytes(lay.d, lay.F, P.MAX_TOKENS) == P.prox_workspace_bytes(lay.d, lay.F, 16)
    assert P.prox_workspace_bytes(lay.d, lay.F, P.MAX_TOKENS + 1) == 0
    ws = P.prox_workspace(lay.d, lay.F, 16)
    x = torch.zeros((P.MAX_TOKENS + 1, lay.d), device="cuda")
    with pytest.raises(P.ProxError):
        P.prox_ffn_forward(lay.packed, x, 0.5, 0.5, ws)
    # a workspace sized for fewer tokens than one tile is refused for a larger call
    small = P.prox_workspace(lay.d, lay.F, 2)
    with pytest.raises(P.ProxError):
        P.prox_ffn_forward(lay.packed, torch.zeros((20, lay.d), device="cuda"), 0.5, 0.5, small)
