"""Batch Stage 2 on the tensor cores (batches of 9 to 16 tokens).

A batch runs one tcgen05 kernel over the union of its tokens' masks: gate/up and down
projections as bf16 MMAs with fp32 accumulation, activations split into bf16 pairs. Every
token's output must match the oracle's exact Stage 2 over that token's own mask (channels of
other tokens contribute nothing to it) within the Stage-2 tolerance. Cases: several output
tiles and a ragged union, a union smaller than the grid (most blocks own no channel), equal
masks, the dense FFN and sparsity 0, slices of more than 128 channels (two and three M-tiles
of the gate/up contraction), and agreement with the single-token CUDA-core path.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
import free_sparse_swiglu_stage1_b300 as P
from gpu_helpers import Layer, check_band, check_y, cuda, random_layer, ws_for

pytestmark = pytest.mark.gpu


def _oracle_masks(lay, x, sparsity, s_in):
    outs = [O.ffn_token(lay.o, x[b], sparsity, s_in) for b in range(len(x))]
    return np.stack([o["idx"] for o in outs]).astype(np.int32), [o["y"] for o in outs]


@pytest.mark.parametrize("d,F", [(1024, 2816), (1152, 4096), (384, 352)])
@pytest.mark.parametrize("batch", [9, 12, 16])
def test_given_masks(d, F, batch):
    lay = random_layer(d, F, seed=d + F + batch)
    x = WL.make_random_tokens(batch, d, seed=400 + batch)
    idx, y_ref = _oracle_masks(lay, x, 0.7, 0.5)
    ws = ws_for(lay, batch)
    y = P.prox_sparse_ffn(lay.packed, cuda(x), cuda(idx), ws).cpu().numpy()
    assert P.prox_get_status(ws) == 0
    for b in range(batch):
        check_y(y[b], y_ref[b])


def test_union_smaller_than_grid():
    """Three channels per token: most blocks own no channel and contribute zeros."""
    lay = random_layer(1024, 2816, seed=401)
    x = WL.make_random_tokens(9, 1024, seed=402)
    idx, y_ref = _oracle_masks(lay, x, 0.999, 0.5)
    ws = ws_for(lay, 9)
    y = P.prox_sparse_ffn(lay.packed, cuda(x), cuda(idx), ws).cpu().numpy()
    assert P.prox_get_status(ws) == 0
    for b in range(9):
        check_y(y[b], y_ref[b])


def test_equal_masks_and_zero_tokens():
    """Every token selects the same channels; two tokens are all zero (y = 0 exactly)."""
    lay = random_layer(1024, 2816, seed=403)
    x = WL.make_random_tokens(16, 1024, seed=404)
    x[3] = 0.0
    x[11] = 0.0
    k = O.k_for(0.7, 2816)
    one = np.sort(np.random.default_rng(405).choice(2816, k, replace=False)).astype(np.int32)
    idx = np.tile(one, (16, 1))
    ws = ws_for(lay, 16)
    y = P.prox_sparse_ffn(lay.packed, cuda(x), cuda(idx), ws).cpu().numpy()
    assert P.prox_get_status(ws) == 0
    for b in range(16):
        y_b, _ = O.stage2_exact(x[b], lay.o.w_gate, lay.o.w_up, lay.o.w_down, one)
        check_y(y[b], y_b)
    assert not y[3].any() and not y[11].any()


def test_dense_and_sparsity_zero():
    lay = random_layer(1024, 2816, seed=406)
    x = WL.make_random_tokens(16, 1024, seed=407)
    ws = ws_for(lay, 16)
    yd = P.prox_dense_ffn(lay.packed, cuda(x), ws).cpu().numpy()
    y0 = P.prox_ffn_forward(lay.packed, cuda(x), 0.0, 0.5, ws).cpu().numpy()
    assert P.prox_get_status(ws) == 0
    for b in (0, 7, 15):
        check_y(yd[b], O.dense_ffn(x[b], lay.o.w_gate, lay.o.w_up, lay.o.w_down))
    np.testing.assert_array_equal(yd, y0)


@pytest.mark.parametrize("d,F,sparsity", [(256, 20480, 0.5), (128, 53248, 0.0)])
def test_long_slices(d, F, sparsity):
    """More than 128 union channels per block: two (d_ff 20480) and three (d_ff 53248,
    dense) passes of the gate/up contraction, and K-chunks of the down projection."""
    lay = random_layer(d, F, seed=d + F)
    x = WL.make_random_tokens(16, d, seed=408)
    ws = ws_for(lay, 16)
    if sparsity == 0.0:
        y = P.prox_dense_ffn(lay.packed, cuda(x), ws).cpu().numpy()
        refs = {b: O.dense_ffn(x[b], lay.o.w_gate, lay.o.w_up, lay.o.w_down) for b in (0, 9, 15)}
    else:
        k = O.k_for(sparsity, F)
        rng = np.random.default_rng(409)
        idx = np.stack([np.sort(rng.choice(F, k, replace=False)) for _ in range(16)]).astype(np.int32)
        y = P.prox_sparse_ffn(lay.packed, cuda(x), cuda(idx), ws).cpu().numpy()
        refs = {b: O.stage2_exact(x[b], lay.o.w_gate, lay.o.w_up, lay.o.w_down, idx[b])[0]
                for b in (0, 9, 15)}
    assert P.prox_get_status(ws) == 0
    for b, y_ref in refs.items():
        check_y(y[b], y_ref)


def test_forward_matches_single_tokens():
    """The whole path at batch 16 (masks per 4-token tile, one tensor-core Stage 2) against
    the single-token path (CUDA cores), token by token, and the masks against the oracle."""
    lay = random_layer(2048, 5632, seed=410)
    x = WL.make_random_tokens(16, 2048, seed=411)
    ws = ws_for(lay, 16)
    k = O.k_for(0.7, 5632)
    idx = torch.empty((16, k), dtype=torch.int32, device="cuda")
    yb = P.prox_ffn_forward(lay.packed, cuda(x), 0.7, 0.5, ws, idx_out=idx).cpu().numpy()
    assert P.prox_get_status(ws) == 0
    idx = idx.cpu().numpy()
    ws1 = ws_for(lay, 1)
    for b in range(16):
        i1 = torch.empty((1, k), dtype=torch.int32, device="cuda")
        y1 = P.prox_ffn_forward(lay.packed, cuda(x[b:b + 1]), 0.7, 0.5, ws1, idx_out=i1)
        np.testing.assert_array_equal(i1.cpu().numpy()[0], idx[b])
        check_y(yb[b], y1.cpu().numpy()[0])
    for b in (0, 15):
        check_band(O.stage1_token(lay.o, x[b], 0.5)["sigma"], k, idx[b])


def test_deterministic():
    lay = random_layer(1024, 2816, seed=412)
    x = cuda(WL.make_random_tokens(16, 1024, seed=413))
    ws = ws_for(lay, 16)
    a = P.prox_ffn_forward(lay.packed, x, 0.7, 0.5, ws)
    b = P.prox_ffn_forward(lay.packed, x, 0.7, 0.5, ws)
    assert torch.equal(a, b)
