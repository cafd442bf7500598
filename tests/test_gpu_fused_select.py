"""The single-token Stage-2 variant that selects its own channels.

This variant folds the top-k into the front of the Stage-2 kernel: every block bulk-loads the
salience and Stage 1's histogram of it, finds the bin of the k-th value, starts copying the
channels above that bin, and resolves the winners inside the bin while those copies are in
flight. It is reached through the prox_debug_fused_forward hook, which also returns the
selected channels. The selected set must be exactly the mask prox_build_mask returns (the same
ranking rule on the same salience), the output must agree with the two-step path (mask, then
Stage 2 over it) and with the oracle, and ties must go to the lower channel index.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
import free_sparse_swiglu_stage1_b300 as P
from gpu_helpers import Layer, check_band, check_y, cuda, random_layer, workload_layer, ws_for

pytestmark = pytest.mark.gpu


def _check_fused(lay, x, sparsity, s_in):
    ws = ws_for(lay, 1)
    xg = cuda(x)
    k = O.k_for(sparsity, lay.F)
    y_f, sel = P.prox_debug_fused_forward(lay.packed, xg, sparsity, s_in, ws)
    mask = P.prox_build_mask(lay.packed, xg, sparsity, s_in, ws)
    y_two = P.prox_sparse_ffn(lay.packed, xg, mask, ws)
    assert P.prox_get_status(ws) == 0
    sel = sel.cpu().numpy()
    mask = mask.cpu().numpy()[0]
    assert sel.min() >= 0, "a selected slot was not written"
    np.testing.assert_array_equal(np.sort(sel), mask)
    # the sure channels, then the boundary winners: two ascending runs
    breaks = np.nonzero(np.diff(sel) < 0)[0]
    assert len(breaks) <= 1
    y_f = y_f.cpu().numpy()[0]
    check_y(y_f, y_two.cpu().numpy()[0])
    y_ref, _ = O.stage2_exact(x[0], lay.o.w_gate, lay.o.w_up, lay.o.w_down, mask)
    check_y(y_f, y_ref)
    y_plain = P.prox_ffn_forward(lay.packed, xg, sparsity, s_in, ws).cpu().numpy()[0]
    check_y(y_plain, y_f)
    return sel, mask


@pytest.mark.parametrize("d,F", [(1024, 2816), (4096, 1024), (2048, 1056), (1152, 4096)])
@pytest.mark.parametrize("sparsity", [0.5, 0.7, 0.9, 0.999])
def test_fused_selection_equals_mask(d, F, sparsity):
    lay = random_layer(d, F, seed=d + F)
    x = WL.make_random_tokens(1, d, seed=31 + int(sparsity * 1000))
    sel, mask = _check_fused(lay, x, sparsity, 0.5)
    st = O.stage1_token(lay.o, x[0], 0.5)
    check_band(st["sigma"], O.k_for(sparsity, F), mask)


def test_fused_selection_all_ties():
    """Zero input: every salience is 0, so the mask is the first k channels."""
    lay = random_layer(1024, 2816, seed=41)
    x = np.zeros((1, 1024), np.float32)
    sel, mask = _check_fused(lay, x, 0.7, 0.5)
    np.testing.assert_array_equal(mask, np.arange(O.k_for(0.7, 2816)))


def test_fused_selection_identical_channels():
    """Every channel has the same weights, so every salience is equal and the lowest k
    channel indices win."""
    mats = WL.make_random_layer(1024, 1024, seed=42)
    for n in ("w_gate", "w_up"):
        mats[n][:] = mats[n][0].clone()
    mats["w_down"][:] = mats["w_down"][:, :1].clone()
    lay = Layer(mats)
    x = WL.make_random_tokens(1, 1024, seed=43)
    sel, mask = _check_fused(lay, x, 0.5, 0.5)
    np.testing.assert_array_equal(mask, np.arange(512))


def test_fused_selection_llama3_8b_layer():
    """The benchmarked layer (4096 x 14336, 70% / 50%) at full size."""
    lay = workload_layer(3, 0)
    x = WL.make_tokens(3, range(2))
    for t in range(2):
        _check_fused(lay, x[t:t + 1], 0.7, 0.5)


def test_fused_selection_wide_layer():
    """d_ff above 16384 takes the 64-keys-per-thread variant."""
    lay = random_layer(1024, 20480, seed=44)
    x = WL.make_random_tokens(1, 1024, seed=45)
    _check_fused(lay, x, 0.7, 0.5)
