"""Stage 2 over FP8 (E4M3) weights (technical summary, "Experimental Results",
Compatibility: Prox is orthogonal to weight quantization such as FP8), through the C ABI.

The packed FP8 codes and row scales must equal the oracle's bit for bit; the proxies, hence the
masks, must be those of the bf16 packing; y must match the oracle's exact Stage 2 over the
dequantized FP8 weights within the Stage-2 tolerance (the same arithmetic as the bf16 path:
exact products, fp32 accumulation). Stage 2 over FP8 rows runs in the single-token kernel; a
batch runs token by token and gives each token's single-token result bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle as O
import oracle.fp8_weights as F8
import workloads as WL
import free_sparse_swiglu_stage1_b300 as P
from gpu_helpers import check_band, check_y, cuda, ws_for

pytestmark = pytest.mark.gpu


class Fp8Layer:
    def __init__(self, mats):
        self.mats = mats
        dev = {k: v.cuda() for k, v in mats.items() if k.startswith("w_")}
        self.packed = P.prox_pack_weights(dev["w_gate"], dev["w_up"], dev["w_down"], fp8=True)
        self.packed_bf16 = P.prox_pack_weights(dev["w_gate"], dev["w_up"], dev["w_down"])
        self.o = O.prepare_layer(*(mats[k].float().numpy() for k in ("w_gate", "w_up", "w_down")))
        self.f8 = F8.fp8_layer(self.o.w_gate, self.o.w_up, self.o.w_down)
        self.d, self.F = self.packed.d_model, self.packed.d_ff


@pytest.fixture(scope="module", params=[(1024, 2816), (384, 352), (2048, 1056)],
                ids=lambda s: f"{s[0]}x{s[1]}")
def layer(request):
    d, F = request.param
    return Fp8Layer(WL.make_random_layer(d, F, seed=d + 3 * F))


def test_fp8_pack_bitwise(layer):
    d, F = layer.d, layer.F
    buf = layer.packed.buffer.cpu().numpy()
    assert layer.packed.desc.format == P.FORMAT_FP8
    a = lambda v: (v + 255) // 256 * 256
    G = d // 128
    # the proxies (codes, then scales; not the alignment padding after them) are those of the
    # bf16 packing
    ref = layer.packed_bf16.buffer.cpu().numpy()
    np.testing.assert_array_equal(buf[: d * F], ref[: d * F])
    np.testing.assert_array_equal(buf[a(d * F): a(d * F) + G * F * 4], ref[a(d * F): a(d * F) + G * F * 4])
    ro = a(a(d * F) + G * F * 4)
    rb = 3 * d + 16
    rows = buf[ro: ro + F * rb].reshape(F, rb)
    f8 = layer.f8
    np.testing.assert_array_equal(rows[:, :d], F8.e4m3_bits(f8["q_gate"]))
    np.testing.assert_array_equal(rows[:, d:2 * d], F8.e4m3_bits(f8["q_up"]))
    np.testing.assert_array_equal(rows[:, 2 * d:3 * d], F8.e4m3_bits(f8["q_down"]))
    sc = rows[:, 3 * d:].copy().view(np.float32)
    np.testing.assert_array_equal(sc[:, 0], f8["s_gate"])
    np.testing.assert_array_equal(sc[:, 1], f8["s_up"])
    np.testing.assert_array_equal(sc[:, 2], f8["s_down"])
    assert not sc[:, 3].any()


def test_fp8_given_mask_and_forward(layer):
    ws = ws_for(layer, 1)
    for t in range(3):
        x = WL.make_random_tokens(1, layer.d, seed=70 + t)
        out = O.ffn_token(layer.o, x[0], 0.7, 0.5)
        idx = out["idx"].astype(np.int32)[None]
        y = P.prox_sparse_ffn(layer.packed, cuda(x), cuda(idx), ws).cpu().numpy()[0]
        y_ref, _ = O.stage2_exact(x[0], layer.f8["w_gate"], layer.f8["w_up"], layer.f8["w_down"], idx[0])
        check_y(y, y_ref)
        # the whole path: the mask is the bf16 packing's (same proxies)
        k = O.k_for(0.7, layer.F)
        i8 = torch.empty((1, k), dtype=torch.int32, device="cuda")
        i16 = torch.empty((1, k), dtype=torch.int32, device="cuda")
        yf = P.prox_ffn_forward(layer.packed, cuda(x), 0.7, 0.5, ws, idx_out=i8).cpu().numpy()[0]
        P.prox_ffn_forward(layer.packed_bf16, cuda(x), 0.7, 0.5, ws, idx_out=i16)
        assert torch.equal(i8, i16)
        i8 = i8.cpu().numpy()[0]
        check_band(out["sigma"], k, i8)
        y_ref, _ = O.stage2_exact(x[0], layer.f8["w_gate"], layer.f8["w_up"], layer.f8["w_down"], i8)
        check_y(yf, y_ref)
    assert P.prox_get_status(ws) == 0


def test_fp8_dense_and_batches(layer):
    B = 5
    ws = ws_for(layer, B)
    x = WL.make_random_tokens(B, layer.d, seed=80)
    yd = P.prox_dense_ffn(layer.packed, cuda(x[:1]), ws).cpu().numpy()[0]
    check_y(yd, O.dense_ffn(x[0], layer.f8["w_gate"], layer.f8["w_up"], layer.f8["w_down"]))
    # a batch goes token by token: each row equals the single-token call bit for bit
    k = O.k_for(0.7, layer.F)
    idx = torch.empty((B, k), dtype=torch.int32, device="cuda")
    y = P.prox_ffn_forward(layer.packed, cuda(x), 0.7, 0.5, ws, idx_out=idx)
    ydb = P.prox_dense_ffn(layer.packed, cuda(x), ws)
    yg = P.prox_sparse_ffn(layer.packed, cuda(x), idx, ws)
    bits = lambda t: t.cpu().numpy().view(np.uint32)
    for b in range(B):
        y1 = P.prox_ffn_forward(layer.packed, cuda(x[b:b + 1]), 0.7, 0.5, ws)
        np.testing.assert_array_equal(bits(y[b:b + 1]), bits(y1))
        np.testing.assert_array_equal(bits(ydb[b:b + 1]), bits(P.prox_dense_ffn(layer.packed, cuda(x[b:b + 1]), ws)))
        np.testing.assert_array_equal(bits(yg[b:b + 1]), bits(y1))
    y_np, idx_np = y.cpu().numpy(), idx.cpu().numpy()
    for b in (0, B - 1):
        y_ref, _ = O.stage2_exact(x[b], layer.f8["w_gate"], layer.f8["w_up"], layer.f8["w_down"], idx_np[b])
        check_y(y_np[b], y_ref)
    # masks need no Stage 2: the bf16 packing's, from the batch kernels
    m8 = P.prox_build_mask(layer.packed, cuda(x), 0.7, 0.5, ws)
    m16 = P.prox_build_mask(layer.packed_bf16, cuda(x), 0.7, 0.5, ws)
    assert torch.equal(m8, m16)
    assert P.prox_get_status(ws) == 0


def test_fp8_llama3_layer_full_size():
    lay = Fp8Layer(WL.make_layer(3, 0))
    ws = ws_for(lay, 1)
    x = WL.make_tokens(3, range(2))
    k = O.k_for(0.7, lay.F)
    for t in range(2):
        idx = torch.empty((1, k), dtype=torch.int32, device="cuda")
        y = P.prox_ffn_forward(lay.packed, cuda(x[t:t + 1]), 0.7, 0.5, ws, idx_out=idx).cpu().numpy()[0]
        idx = idx.cpu().numpy()[0]
        check_band(O.stage1_token(lay.o, x[t], 0.5)["sigma"], k, idx)
        y_ref, _ = O.stage2_exact(x[t], lay.f8["w_gate"], lay.f8["w_up"], lay.f8["w_down"], idx)
        check_y(y, y_ref)
    assert P.prox_get_status(ws) == 0
