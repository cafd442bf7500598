"""Decode through a stack of independently seeded Prox FFN layers with a unit-gain RMSNorm
between them (the 32-layer Llama-3-8B-shaped stack among the workloads).

Every layer runs on the GPU from the previous layer's GPU output, as in decoding; each layer
is then checked against the oracle given that same input: the mask against the oracle's
salience (tie band), y against the oracle's exact Stage 2 over the GPU mask, and the next
input against the oracle's RMSNorm of the GPU output. A full-length chain runs on a small
layer shape (32 layers, so the stack's depth is covered); the 4096 x 14336 shape runs a
shorter chain of its own seeded layers.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
import free_sparse_swiglu_stage1_b300 as P
from gpu_helpers import Layer, check_band, check_y, cuda

pytestmark = pytest.mark.gpu


def _run_chain(layers, x0, sparsity, s_in, eps=1e-6):
    d, F = layers[0].d, layers[0].F
    ws = P.prox_workspace(d, F, 1)
    k = O.k_for(sparsity, F)
    x = cuda(x0)
    for li, lay in enumerate(layers):
        idx = torch.empty((1, k), dtype=torch.int32, device="cuda")
        y = P.prox_ffn_forward(lay.packed, x, sparsity, s_in, ws, idx_out=idx)
        x_next = P.prox_rmsnorm(y, eps)
        assert P.prox_get_status(ws) == 0
        xin = x.cpu().numpy()[0]
        idx_h = idx.cpu().numpy()[0]
        st = O.stage1_token(lay.o, xin, s_in)
        check_band(st["sigma"], k, idx_h)
        y_ref, _ = O.stage2_exact(xin, lay.o.w_gate, lay.o.w_up, lay.o.w_down, idx_h)
        y_h = y.cpu().numpy()[0]
        check_y(y_h, y_ref)
        np.testing.assert_allclose(x_next.cpu().numpy()[0], O.rmsnorm(y_h[None], eps)[0],
                                   rtol=2e-6, atol=1e-7)
        assert np.all(np.isfinite(y_h)), f"layer {li}"
        x = x_next
    return x


def test_stack_of_32_small_layers():
    layers = [Layer(WL.make_random_layer(1024, 2816, seed=5000 + li)) for li in range(32)]
    x0 = WL.make_random_tokens(1, 1024, seed=5100)
    _run_chain(layers, x0, 0.7, 0.5)


def test_stack_llama3_8b_layers():
    layers = [Layer(WL.make_layer(4, li)) for li in range(3)]
    x0 = WL.make_tokens(4, [0])
    _run_chain(layers, x0, 0.7, 0.5)


def test_stack_llama3_8b_all_32_layers():
    """The whole 32-layer 4096 x 14336 stack for one token: each layer is built, run from the
    previous layer's GPU output, checked against the oracle and released before the next one,
    so host and device memory hold one layer at a time."""
    k = O.k_for(0.7, 14336)
    ws = P.prox_workspace(4096, 14336, 1)
    x = cuda(WL.make_tokens(4, [1]))
    for li in range(32):
        lay = Layer(WL.make_layer(4, li))
        idx = torch.empty((1, k), dtype=torch.int32, device="cuda")
        y = P.prox_ffn_forward(lay.packed, x, 0.7, 0.5, ws, idx_out=idx)
        x_next = P.prox_rmsnorm(y, 1e-6)
        assert P.prox_get_status(ws) == 0
        xin = x.cpu().numpy()[0]
        idx_h = idx.cpu().numpy()[0]
        check_band(O.stage1_token(lay.o, xin, 0.5)["sigma"], k, idx_h)
        y_ref, _ = O.stage2_exact(xin, lay.o.w_gate, lay.o.w_up, lay.o.w_down, idx_h)
        y_h = y.cpu().numpy()[0]
        check_y(y_h, y_ref)
        np.testing.assert_allclose(x_next.cpu().numpy()[0], O.rmsnorm(y_h[None], 1e-6)[0],
                                   rtol=2e-6, atol=1e-7)
        x = x_next
        del lay
