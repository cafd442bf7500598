"""Split layers and the sliding window of device-resident proxies, through the C ABI: a split
layer computes exactly what its packed layer computes (same kernels, same bits), and a layer
stack run through a window of fewer slots than layers, with the proxies paged in from pinned
host memory, gives bit for bit the stack run on resident layers (technical summary,
"Significance and Claims": sliding-window schemes for the proxies' memory).
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
import free_sparse_swiglu_stage1_b300 as P
from gpu_helpers import check_band, check_y, cuda, workload_layer

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.cpu().numpy().view(np.uint32)


@pytest.fixture(scope="module")
def stack():
    return [workload_layer(1, l) for l in range(5)]


@pytest.mark.parametrize("B", [1, 4])
def test_split_layer_bit_identical(stack, B):
    lay = stack[0]
    split = P.prox_split_packed(lay.packed, proxy_on_host=False)
    x = cuda(WL.make_tokens(1, range(B)))
    ws = P.prox_workspace(lay.d, lay.F, B)
    k = P.prox_k_for(0.5, lay.F)
    i0 = torch.empty((B, k), dtype=torch.int32, device="cuda")
    i1 = torch.empty_like(i0)
    y0 = P.prox_ffn_forward(lay.packed, x, 0.5, 0.5, ws, idx_out=i0)
    y1 = P.prox_ffn_forward(split, x, 0.5, 0.5, ws, idx_out=i1)
    assert P.prox_get_status(ws) == 0
    np.testing.assert_array_equal(i0.cpu().numpy(), i1.cpu().numpy())
    np.testing.assert_array_equal(_bits(y0), _bits(y1))
    np.testing.assert_array_equal(_bits(P.prox_dense_ffn(lay.packed, x, ws)),
                                  _bits(P.prox_dense_ffn(split, x, ws)))
    # the split rows and proxy are the packed buffer's two regions
    pb = P.prox_proxy_bytes(lay.d, lay.F)
    full = lay.packed.buffer.cpu().numpy()
    np.testing.assert_array_equal(split.proxy_buffer.cpu().numpy(), full[:pb])
    rb = P.prox_rows_bytes(lay.d, lay.F)
    np.testing.assert_array_equal(split.buffer.cpu().numpy()[: lay.F * 6 * lay.d],
                                  full[pb: pb + lay.F * 6 * lay.d])
    assert rb >= lay.F * 6 * lay.d


def test_proxy_in_host_memory_is_refused(stack):
    lay = stack[0]
    split = P.prox_split_packed(lay.packed, proxy_on_host=True)
    ws = P.prox_workspace(lay.d, lay.F, 1)
    with pytest.raises(P.ProxError):
        P.prox_ffn_forward(split, torch.zeros((1, lay.d), device="cuda"), 0.5, 0.5, ws)


def _run_stack(layers, xs, s, s_in, ws, window=None):
    """Decode tokens one after another through the stack (RMSNorm between layers); returns
    every layer's output per token."""
    outs = []
    for x in xs:
        h = cuda(x[None])
        per = []
        for l, lay in enumerate(layers):
            desc = window.acquire(l) if window is not None else lay
            y = P.prox_ffn_forward(desc, h, s, s_in, ws)
            if window is not None:
                window.release(l)
            per.append(y.clone())
            h = P.prox_rmsnorm(y)
        outs.append(per)
    return outs


@pytest.mark.parametrize("slots", [1, 2, 3, 5, 7])
def test_window_stack_bit_identical(stack, slots):
    s, s_in = 0.5, 0.5
    xs = WL.make_tokens(1, range(3))
    lay0 = stack[0]
    ws = P.prox_workspace(lay0.d, lay0.F, 1)
    want = _run_stack([l.packed for l in stack], xs, s, s_in, ws)
    splits = [P.prox_split_packed(l.packed, proxy_on_host=True) for l in stack]
    win = P.ProxyWindow(splits, slots)
    got = _run_stack(splits, xs, s, s_in, ws, window=win)
    torch.cuda.synchronize()
    assert P.prox_get_status(ws) == 0
    for t in range(len(xs)):
        for l in range(len(stack)):
            np.testing.assert_array_equal(_bits(got[t][l]), _bits(want[t][l]))
    copies, nbytes = win.stats()
    L, visits = len(stack), len(stack) * len(xs)
    if slots >= L:
        assert copies == L                      # every proxy copied once, then resident
    else:
        assert visits <= copies <= visits + slots
    assert nbytes == copies * P.prox_proxy_bytes(lay0.d, lay0.F)
    win.close()


def test_window_first_layer_vs_oracle(stack):
    """The first layer of a windowed stack against the oracle (mask in the tie band, y within
    the Stage-2 tolerance)."""
    lay = stack[0]
    splits = [P.prox_split_packed(l.packed, proxy_on_host=True) for l in stack[:2]]
    win = P.ProxyWindow(splits, 1)
    x = WL.make_tokens(1, [7])
    ws = P.prox_workspace(lay.d, lay.F, 1)
    k = P.prox_k_for(0.7, lay.F)
    idx = torch.empty((1, k), dtype=torch.int32, device="cuda")
    y = P.prox_ffn_forward(win.acquire(0), cuda(x), 0.7, 0.5, ws, idx_out=idx)
    win.release(0)
    idx = idx.cpu().numpy()[0]
    check_band(O.stage1_token(lay.o, x[0], 0.5)["sigma"], k, idx)
    y_ref, _ = O.stage2_exact(x[0], lay.o.w_gate, lay.o.w_up, lay.o.w_down, idx)
    check_y(y.cpu().numpy()[0], y_ref)
    win.close()


def test_window_full_size_layers():
    """Three 4096 x 14336 layers through a one-slot window: bit-identical to resident layers."""
    layers = [workload_layer(3, l) for l in range(3)]
    lay0 = layers[0]
    ws = P.prox_workspace(lay0.d, lay0.F, 1)
    xs = WL.make_tokens(3, range(2))
    want = _run_stack([l.packed for l in layers], xs, 0.7, 0.5, ws)
    splits = [P.prox_split_packed(l.packed, proxy_on_host=True) for l in layers]
    win = P.ProxyWindow(splits, 1)
    got = _run_stack(splits, xs, 0.7, 0.5, ws, window=win)
    torch.cuda.synchronize()
    assert P.prox_get_status(ws) == 0
    for t in range(len(xs)):
        for l in range(len(layers)):
            np.testing.assert_array_equal(_bits(got[t][l]), _bits(want[t][l]))
    visits = len(xs) * len(layers)
    assert visits <= win.stats()[0] <= visits + 1   # plus the lookahead after the last release
    win.close()
