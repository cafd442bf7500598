"""Parity of the CUDA path (through the C ABI) with the CPU oracle, element by element.

Bars: packed codes and scales bit-exact; activation codes, scales and int32 proxy
accumulators bit-exact; masks exact outside the 1e-6 tie band of the k-th salience;
Stage-2 outputs given the same mask within max|err| <= 2e-2 max|y| and rel-L2 <= 5e-3.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
import free_sparse_swiglu_stage1_b300 as P
from gpu_helpers import (check_band, check_y, cuda, decode_packed, random_layer, workload_layer,
                         ws_for)

pytestmark = pytest.mark.gpu

# (d_model, d_ff): several channel blocks, a ragged last block (d_ff % 128 != 0), one group
SHAPES = [(1024, 2816), (384, 352), (128, 32), (2048, 1056)]


@pytest.fixture(scope="module", params=SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
def layer(request):
    d, F = request.param
    return random_layer(d, F, seed=d * 31 + F)


def _tokens(n, d, seed, kind="student_t"):
    return WL.make_random_tokens(n, d, seed, kind=kind)


def test_pack_bitwise(layer):
    dec = decode_packed(layer.packed.buffer.cpu().numpy(), layer.d, layer.F)
    np.testing.assert_array_equal(dec["q_gate"], layer.o.q_gate)
    np.testing.assert_array_equal(dec["q_up"], layer.o.q_up)
    np.testing.assert_array_equal(dec["sw_gate_bits"], layer.o.sw_gate.view(np.uint16))
    np.testing.assert_array_equal(dec["sw_up_bits"], layer.o.sw_up.view(np.uint16))
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(dec["rows"][:, 0, :], bits(layer.mats["w_gate"]))
    np.testing.assert_array_equal(dec["rows"][:, 1, :], bits(layer.mats["w_up"]))
    np.testing.assert_array_equal(dec["rows"][:, 2, :], bits(layer.mats["w_down"]).T)


# batches past one token tile (4 tokens at these widths) take the tensor-core Stage 1
@pytest.mark.parametrize("batch,s_in", [(1, 0.5), (3, 0.5), (2, 0.0), (1, 0.9), (6, 0.5),
                                        (16, 0.3)])
def test_stage1_integers_bitexact(layer, batch, s_in):
    ws = ws_for(layer, batch)
    x = _tokens(batch, layer.d, seed=batch * 7 + int(s_in * 10))
    out = P.prox_debug_stage1(layer.packed, cuda(x), s_in, ws)
    assert P.prox_get_status(ws) == 0
    got = {k: v.cpu().numpy() for k, v in out.items()}
    for b in range(batch):
        st = O.stage1_token(layer.o, x[b], s_in)
        np.testing.assert_array_equal(got["qx"][b].astype(np.int32), st["qx"])
        np.testing.assert_array_equal(got["sx"][b].view(np.uint32), st["sx"].view(np.uint32))
        np.testing.assert_array_equal(got["acc_gate"][b], st["A_gate"])
        np.testing.assert_array_equal(got["acc_up"][b], st["A_up"])
        ref = st["sigma"]
        np.testing.assert_allclose(got["salience"][b], ref, rtol=2e-6, atol=1e-30)


@pytest.mark.parametrize("batch,sparsity,s_in", [(1, 0.5, 0.5), (1, 0.7, 0.5), (1, 0.9, 0.3),
                                                 (4, 0.7, 0.5), (5, 0.5, 0.5), (2, 0.99, 0.5)])
def test_mask_and_forward(layer, batch, sparsity, s_in):
    ws = ws_for(layer, batch)
    x = _tokens(batch, layer.d, seed=100 + batch)
    k = O.k_for(sparsity, layer.F)
    idx_mask = P.prox_build_mask(layer.packed, cuda(x), sparsity, s_in, ws).cpu().numpy()
    idx_fwd = torch.empty((batch, k), dtype=torch.int32, device="cuda")
    y = P.prox_ffn_forward(layer.packed, cuda(x), sparsity, s_in, ws, idx_out=idx_fwd)
    y = y.cpu().numpy()
    idx_fwd = idx_fwd.cpu().numpy()
    assert P.prox_get_status(ws) == 0
    np.testing.assert_array_equal(idx_mask, idx_fwd)
    for b in range(batch):
        st = O.stage1_token(layer.o, x[b], s_in)
        check_band(st["sigma"], k, idx_fwd[b])
        y_ref, _ = O.stage2_exact(x[b], layer.o.w_gate, layer.o.w_up, layer.o.w_down, idx_fwd[b])
        check_y(y[b], y_ref)


@pytest.mark.parametrize("batch", [1, 2, 4, 7])
def test_stage2_given_oracle_mask(layer, batch):
    ws = ws_for(layer, batch)
    x = _tokens(batch, layer.d, seed=200 + batch)
    k = O.k_for(0.7, layer.F)
    outs = [O.ffn_token(layer.o, x[b], 0.7, 0.5) for b in range(batch)]
    idx = np.stack([o["idx"] for o in outs]).astype(np.int32)
    y = P.prox_sparse_ffn(layer.packed, cuda(x), cuda(idx), ws).cpu().numpy()
    assert P.prox_get_status(ws) == 0
    assert idx.shape == (batch, k)
    for b in range(batch):
        check_y(y[b], outs[b]["y"])


def test_dense_and_sparsity_zero(layer):
    ws = ws_for(layer, 2)
    x = _tokens(2, layer.d, seed=300)
    yd = P.prox_dense_ffn(layer.packed, cuda(x), ws).cpu().numpy()
    y0 = P.prox_ffn_forward(layer.packed, cuda(x), 0.0, 0.5, ws).cpu().numpy()
    for b in range(2):
        check_y(yd[b], O.dense_ffn(x[b], layer.o.w_gate, layer.o.w_up, layer.o.w_down))
    np.testing.assert_array_equal(yd, y0)


def test_union_bitexact():
    rng = np.random.default_rng(5)
    F, k, B = 1000, 300, 4
    idx = np.stack([np.sort(rng.choice(F, k, replace=False)) for _ in range(B)]).astype(np.int32)
    ws = P.prox_workspace(1024, F - F % 32, 1)
    u, bits = P.prox_debug_union(cuda(idx), F, ws)
    U, B_ref = O.batch_union(list(idx), F)
    np.testing.assert_array_equal(u.cpu().numpy(), U)
    bits = bits.cpu().numpy().view(np.uint32)
    for b in range(B):
        np.testing.assert_array_equal((bits >> b) & 1, B_ref[b].astype(np.uint32))


def test_rmsnorm():
    y = np.random.default_rng(6).normal(0, 3, (3, 4096)).astype(np.float32)
    out = P.prox_rmsnorm(cuda(y), 1e-6).cpu().numpy()
    np.testing.assert_allclose(out, O.rmsnorm(y, 1e-6), rtol=2e-6, atol=1e-7)


# ----------------------------------------------------------------------------- invariants

def test_error_isolation():
    """Proxy values reach the output only through the mask (technical summary, Stage 1
    "Error Isolation"): Stage 2 never reads the proxies, and the full path's output equals
    Stage 2 over the mask it built."""
    lay = random_layer(1024, 2816, seed=11)
    ws = ws_for(lay, 1)
    x = cuda(_tokens(1, 1024, seed=12))
    k = O.k_for(0.7, lay.F)
    idx = torch.empty((1, k), dtype=torch.int32, device="cuda")
    y_fwd = P.prox_ffn_forward(lay.packed, x, 0.7, 0.5, ws, idx_out=idx)
    y_s2 = P.prox_sparse_ffn(lay.packed, x, idx, ws)
    assert torch.equal(y_fwd, y_s2)
    proxy_bytes = lay.d * lay.F + (lay.d // 128) * lay.F * 4   # codes + scales (contiguous here)
    lay.packed.buffer[:proxy_bytes] = torch.randint(0, 256, (proxy_bytes,), dtype=torch.uint8,
                                                   device="cuda")
    y_corrupt = P.prox_sparse_ffn(lay.packed, x, idx, ws)
    assert torch.equal(y_s2, y_corrupt)
    assert P.prox_get_status(ws) == 0


def test_determinism_and_nesting():
    lay = random_layer(1024, 2816, seed=13)
    ws = ws_for(lay, 3)
    x = cuda(_tokens(3, 1024, seed=14))
    a = P.prox_ffn_forward(lay.packed, x, 0.7, 0.5, ws)
    b = P.prox_ffn_forward(lay.packed, x, 0.7, 0.5, ws)
    assert torch.equal(a, b)
    m70 = P.prox_build_mask(lay.packed, x, 0.7, 0.5, ws).cpu().numpy()
    m50 = P.prox_build_mask(lay.packed, x, 0.5, 0.5, ws).cpu().numpy()
    for t in range(3):
        assert set(m70[t].tolist()) <= set(m50[t].tolist())


def test_batch_matches_single_tokens():
    lay = random_layer(1024, 2816, seed=15)
    x = _tokens(6, 1024, seed=16)
    wsb = ws_for(lay, 6)
    yb = P.prox_ffn_forward(lay.packed, cuda(x), 0.7, 0.5, wsb).cpu().numpy()
    ws1 = ws_for(lay, 1)
    for t in range(6):
        y1 = P.prox_ffn_forward(lay.packed, cuda(x[t:t + 1]), 0.7, 0.5, ws1).cpu().numpy()
        check_y(yb[t], y1[0])


# ----------------------------------------------------------------------------- edge cases

def test_edge_cases():
    lay = random_layer(256, 96, seed=17)
    ws = ws_for(lay, 16)
    # all-zero input: every salience is 0, the mask is the first k channels, y is 0
    k = O.k_for(0.5, 96)
    idx = torch.empty((1, k), dtype=torch.int32, device="cuda")
    y = P.prox_ffn_forward(lay.packed, torch.zeros((1, 256), device="cuda"), 0.5, 0.5, ws,
                           idx_out=idx)
    assert torch.count_nonzero(y) == 0
    np.testing.assert_array_equal(idx.cpu().numpy()[0], np.arange(k))
    # equal magnitudes everywhere: ties go to the lowest indices
    xe = np.where(np.arange(256) % 3 == 0, 1.0, -1.0).astype(np.float32)[None]
    out = P.prox_debug_stage1(lay.packed, cuda(xe), 0.5, ws)
    st = O.stage1_token(lay.o, xe[0], 0.5)
    np.testing.assert_array_equal(out["qx"].cpu().numpy()[0].astype(np.int32), st["qx"])
    assert np.all(st["qx"][128:] == 0) and np.all(np.abs(st["qx"][:128]) == 127)
    # extreme k and k_in, the largest batch
    x = _tokens(16, 256, seed=18)
    for sparsity, s_in in ((0.999, 0.5), (0.01, 0.999), (0.5, 0.0)):
        kk = O.k_for(sparsity, 96)
        idx = torch.empty((16, kk), dtype=torch.int32, device="cuda")
        y = P.prox_ffn_forward(lay.packed, cuda(x), sparsity, s_in, ws, idx_out=idx).cpu().numpy()
        idx = idx.cpu().numpy()
        for b in (0, 5, 15):
            st = O.stage1_token(lay.o, x[b], s_in)
            check_band(st["sigma"], kk, idx[b])
            y_ref, _ = O.stage2_exact(x[b], lay.o.w_gate, lay.o.w_up, lay.o.w_down, idx[b])
            check_y(y[b], y_ref)
    assert P.prox_get_status(ws) == 0


def test_wide_rows_and_long_channels():
    """d_model 16384 (four 16-byte chunks per thread) and d_model 8192 with two tokens."""
    for d, F, B in ((16384, 256, 1), (8192, 512, 2)):
        lay = random_layer(d, F, seed=d + F)
        ws = ws_for(lay, B)
        x = _tokens(B, d, seed=19)
        k = O.k_for(0.7, F)
        idx = torch.empty((B, k), dtype=torch.int32, device="cuda")
        y = P.prox_ffn_forward(lay.packed, cuda(x), 0.7, 0.5, ws, idx_out=idx).cpu().numpy()
        idx = idx.cpu().numpy()
        for b in range(B):
            st = O.stage1_token(lay.o, x[b], 0.5)
            check_band(st["sigma"], k, idx[b])
            y_ref, _ = O.stage2_exact(x[b], lay.o.w_gate, lay.o.w_up, lay.o.w_down, idx[b])
            check_y(y[b], y_ref)


def test_bounded_wait_reports_timeout():
    """A wait that nothing completes gives up, reports PROX_ERR_TIMEOUT through the status
    word, and leaves the context usable."""
    lay = random_layer(256, 96, seed=20)
    ws = ws_for(lay, 1)
    P.prox_debug_wait_timeout(ws, 200_000)
    assert P.prox_get_status(ws) == -4
    assert P.prox_get_status(ws) == 0
    y = P.prox_dense_ffn(lay.packed, cuda(_tokens(1, 256, seed=21)), ws)
    torch.cuda.synchronize()
    assert torch.isfinite(y).all()


def test_host_entry_point():
    lay = random_layer(1024, 2816, seed=22)
    ws = ws_for(lay, 2)
    x = _tokens(2, 1024, seed=23)
    xh = torch.from_numpy(x).pin_memory()
    yh = P.prox_ffn_forward_host(lay.packed, xh, 0.7, 0.5, ws)
    yd = P.prox_ffn_forward(lay.packed, cuda(x), 0.7, 0.5, ws).cpu()
    assert torch.equal(yh, yd)


# ----------------------------------------------------------------------------- full sizes

@pytest.mark.parametrize("batch", [1, 2, 4, 8, 16])
def test_llama3_8b_layer_full_size(batch):
    """The benchmarked layer (4096 x 14336, 70% channel / 50% input sparsity), checked on
    sampled tokens of the batch one by one."""
    lay = workload_layer(3, 0)
    x = WL.make_tokens(3, range(batch))
    ws = ws_for(lay, batch)
    k = O.k_for(0.7, lay.F)
    idx = torch.empty((batch, k), dtype=torch.int32, device="cuda")
    y = P.prox_ffn_forward(lay.packed, cuda(x), 0.7, 0.5, ws, idx_out=idx).cpu().numpy()
    idx = idx.cpu().numpy()
    assert P.prox_get_status(ws) == 0
    for b in sorted({0, batch // 2, batch - 1}):
        st = O.stage1_token(lay.o, x[b], 0.5)
        check_band(st["sigma"], k, idx[b])
        y_ref, _ = O.stage2_exact(x[b], lay.o.w_gate, lay.o.w_up, lay.o.w_down, idx[b])
        check_y(y[b], y_ref)


def test_llama2_7b_sparsity_sweep_full_size():
    lay = workload_layer(2, 0)
    x = WL.make_tokens(2, range(2))
    ws = ws_for(lay, 1)
    for sparsity in (0.0, 0.5, 0.7, 0.9):
        k = O.k_for(sparsity, lay.F)
        for t in range(2):
            idx = torch.empty((1, k), dtype=torch.int32, device="cuda")
            y = P.prox_ffn_forward(lay.packed, cuda(x[t:t + 1]), sparsity, 0.5, ws, idx_out=idx)
            idx = idx.cpu().numpy()[0]
            if sparsity > 0:
                check_band(O.stage1_token(lay.o, x[t], 0.5)["sigma"], k, idx)
            y_ref, _ = O.stage2_exact(x[t], lay.o.w_gate, lay.o.w_up, lay.o.w_down, idx)
            check_y(y.cpu().numpy()[0], y_ref)


def test_llama2_70b_batch8_full_size():
    lay = workload_layer(5, 0)
    x = WL.make_tokens(5, range(8))
    ws = ws_for(lay, 8)
    k = O.k_for(0.7, lay.F)
    idx = torch.empty((8, k), dtype=torch.int32, device="cuda")
    y = P.prox_ffn_forward(lay.packed, cuda(x), 0.7, 0.5, ws, idx_out=idx).cpu().numpy()
    idx = idx.cpu().numpy()
    for b in (0, 7):
        st = O.stage1_token(lay.o, x[b], 0.5)
        check_band(st["sigma"], k, idx[b])
        y_ref, _ = O.stage2_exact(x[b], lay.o.w_gate, lay.o.w_up, lay.o.w_down, idx[b])
        check_y(y[b], y_ref)


def test_channel_permutation_equivariance():
    """Renumbering the intermediate channels (rows of W_gate and W_up, columns of W_down, by
    one permutation) renumbers the salience, the mask and nothing else: the salience of a
    channel does not depend on its position (bitwise), the mask is the renumbered mask, and y
    is unchanged up to the order of the fp32 sums."""
    d, F = 1024, 2816
    mats = WL.make_random_layer(d, F, seed=24)
    perm = np.random.default_rng(25).permutation(F)
    inv = np.argsort(perm)
    pm = {"w_gate": mats["w_gate"][torch.from_numpy(perm)].contiguous(),
          "w_up": mats["w_up"][torch.from_numpy(perm)].contiguous(),
          "w_down": mats["w_down"][:, torch.from_numpy(perm)].contiguous()}
    from gpu_helpers import Layer
    lay, lay_p = Layer(mats), Layer(pm)
    ws = ws_for(lay, 1)
    x = _tokens(1, d, seed=26)
    s = P.prox_debug_stage1(lay.packed, cuda(x), 0.5, ws)["salience"].cpu().numpy()[0]
    s_p = P.prox_debug_stage1(lay_p.packed, cuda(x), 0.5, ws)["salience"].cpu().numpy()[0]
    np.testing.assert_array_equal(s_p, s[perm])
    k = O.k_for(0.7, F)
    idx = P.prox_build_mask(lay.packed, cuda(x), 0.7, 0.5, ws).cpu().numpy()[0]
    idx_p = P.prox_build_mask(lay_p.packed, cuda(x), 0.7, 0.5, ws).cpu().numpy()[0]
    if len(np.unique(s)) == F:   # no exact ties: the renumbered mask is unique
        np.testing.assert_array_equal(idx_p, np.sort(inv[idx]))
    y = P.prox_ffn_forward(lay.packed, cuda(x), 0.7, 0.5, ws).cpu().numpy()[0]
    y_p = P.prox_ffn_forward(lay_p.packed, cuda(x), 0.7, 0.5, ws).cpu().numpy()[0]
    assert P.prox_get_status(ws) == 0
    check_y(y_p, y)
    y_ref, _ = O.stage2_exact(x[0], lay.o.w_gate, lay.o.w_up, lay.o.w_down, idx)
    check_y(y_p, y_ref)
    assert len(idx) == k
