"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Every check here compares the oracle with an independent source: exact rational arithmetic,
a library routine (torch fp64), brute force over all subsets, a closed form, or a number the
pages print. A plausible slip in the oracle (a dropped term, a wrong sign or index, a
transposed operand, gate and up swapped, a wrong rounding) fails at least one of them.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------- exact rounding

def _floor_log2(m: Fraction) -> int:
    e = m.numerator.bit_length() - m.denominator.bit_length()
    while Fraction(2) ** e > m:
        e -= 1
    while Fraction(2) ** (e + 1) <= m:
        e += 1
    return e


def _rint_half_even(fr: Fraction) -> int:
    fl = fr.numerator // fr.denominator
    rem = fr - fl
    if rem > Fraction(1, 2):
        return fl + 1
    if rem < Fraction(1, 2):
        return fl
    return fl if fl % 2 == 0 else fl + 1


def _round_float(fr: Fraction, mant: int, emin: int, max_finite: Fraction):
    """Round an exact rational to an IEEE binary format, nearest-even, with subnormals."""
    if fr == 0:
        return Fraction(0)
    sign = -1 if fr < 0 else 1
    m = abs(fr)
    e = max(_floor_log2(m), emin)
    ulp = Fraction(2) ** (e - mant)
    r = _rint_half_even(m / ulp) * ulp
    if r > max_finite:
        return sign * math.inf
    return sign * r


F32_MAX = Fraction((2 ** 24 - 1) * 2 ** 104)
F16_MAX = Fraction(65504)


def r32(fr):
    return _round_float(fr, 23, -126, F32_MAX)


def r16(fr):
    return _round_float(fr, 10, -14, F16_MAX)


def _exact_weight_quant(row_group):
    """Reading of the weight proxy re-derived with exact rationals for one group."""
    vals = [Fraction(float(v)) for v in row_group]
    a = max(abs(v) for v in vals)
    sw = r16(r32(a / 7))
    if sw == 0:
        return [0] * len(vals), sw
    q = [max(-7, min(7, _rint_half_even(r32(v / sw)))) for v in vals]
    return q, sw


def _bf16_values(rng, n, lo_exp=-12, hi_exp=2):
    """n random bf16 values (as fp32) spread over several binades."""
    mant = rng.integers(0, 128, n)
    ex = rng.integers(lo_exp, hi_exp, n)
    sign = rng.choice([-1.0, 1.0], n)
    return (sign * (1.0 + mant / 128.0) * np.exp2(ex)).astype(np.float32)


# ----------------------------------------------------------------------------- k rounding

def test_k_for_fixed_values():
    # Values fixed by the workload shapes: d_ff 2816 at 50% keeps 1408 channels (stated with
    # the 1024 x 2816 workload); 14336 and 11008 at 70%; 4096 inputs at 50%.
    assert O.k_for(0.5, 2816) == 1408
    assert O.k_for(0.7, 14336) == 4301
    assert O.k_for(0.7, 11008) == 3302
    assert O.k_for(0.9, 11008) == 1101
    assert O.k_for(0.5, 4096) == 2048
    assert O.k_for(0.0, 14336) == 14336
    assert O.k_for(0.99999, 10) == 1          # clamped below
    ks = [O.k_for(s, 1000) for s in np.linspace(0, 0.999, 200)]
    assert all(a >= b for a, b in zip(ks, ks[1:]))


# ----------------------------------------------------------------------------- SiLU

def test_silu_against_library_and_identities():
    z = np.random.default_rng(0).normal(0, 6, 4096)
    ref = torch.nn.functional.silu(torch.from_numpy(z)).numpy()
    np.testing.assert_allclose(O.silu(z), ref, rtol=1e-14, atol=1e-300)
    np.testing.assert_allclose(O.silu(z) - O.silu(-z), z, rtol=1e-12, atol=1e-12)
    assert O.silu(np.array([0.0]))[0] == 0.0
    assert O.silu(np.array([-800.0]))[0] == 0.0


# ----------------------------------------------------------------------------- weight proxy

def test_weight_quant_exact_rational_all_bf16_of_a_binade():
    rng = np.random.default_rng(1)
    rows = []
    all_binade = (1.0 + np.arange(128) / 128.0)           # every bf16 value in [1, 2)
    for scale_exp in (-10, -6, -3, 0, 3):
        r = all_binade * np.exp2(scale_exp) * rng.choice([-1.0, 1.0], 128)
        rows.append(rng.permutation(r))
    for _ in range(6):
        rows.append(_bf16_values(rng, 128))
    # explicit ties: max 7 -> sw = 1 exactly, then w/sw = n + 1/2 must round to even
    tie = np.zeros(128)
    tie[:6] = [7.0, 2.5, 3.5, -0.5, 1.5, -2.5]
    rows.append(tie)
    rows.append(np.zeros(128))                               # all-zero group -> sw = 0, q = 0
    w = np.array(rows, dtype=np.float32)
    w = np.concatenate([w, w[:, ::-1]], axis=1)              # two groups per row
    q, sw = O.quantize_weight_proxy(w, 128)
    for j in range(w.shape[0]):
        for g in range(2):
            qe, swe = _exact_weight_quant(w[j, g * 128:(g + 1) * 128])
            assert Fraction(float(sw[g, j])) == swe, (j, g)
            assert list(q[j, g * 128:(g + 1) * 128]) == qe, (j, g)
    t = len(rows) - 2
    assert list(q[t, :6]) == [7, 2, 4, 0, 2, -2]


def test_weight_quant_bounds_and_symmetry():
    rng = np.random.default_rng(2)
    w = _bf16_values(rng, 64 * 512).reshape(64, 512)
    q, sw = O.quantize_weight_proxy(w, 128)
    q2, sw2 = O.quantize_weight_proxy(-w, 128)
    np.testing.assert_array_equal(q2, -q)
    np.testing.assert_array_equal(sw2, sw)
    swf = np.repeat(sw.T.astype(np.float64), 128, axis=1)      # [F, d]
    err = np.abs(w.astype(np.float64) - q * swf)
    unclamped = np.abs(w / swf) <= 7.0
    assert np.all(err[unclamped] <= swf[unclamped] / 2 * (1 + 1e-6))
    wg = np.abs(w.reshape(64, 4, 128))
    amax_pos = wg.argmax(axis=2)
    qg = np.abs(q.reshape(64, 4, 128))
    assert np.all(np.take_along_axis(qg, amax_pos[..., None], 2) == 7)


# ----------------------------------------------------------------------------- inputs

def _brute_topk(values, k):
    """Lexicographically first k-subset among those with the largest sum (exact ints)."""
    n = len(values)
    best, best_set = None, None
    for c in itertools.combinations(range(n), k):
        s = sum(values[i] for i in c)
        if best is None or s > best:
            best, best_set = s, c
    return best_set


def test_select_inputs_brute_force_with_ties():
    rng = np.random.default_rng(3)
    for _ in range(60):
        d = int(rng.integers(3, 11))
        k = int(rng.integers(1, d + 1))
        mags = rng.integers(0, 4, d)
        x = (mags * rng.choice([-1, 1], d)).astype(np.float32)
        assert tuple(O.select_inputs(x, k)) == _brute_topk([int(m) for m in mags], k)


def test_select_inputs_matches_torch_topk():
    rng = np.random.default_rng(4)
    x = rng.standard_t(4, 4096).astype(np.float32)
    for k in (1, 100, 2048, 4095, 4096):
        ref = torch.topk(torch.from_numpy(np.abs(x)), k).indices.numpy()
        assert set(O.select_inputs(x, k)) == set(ref.tolist())


def _exact_act_quant(xg):
    vals = [Fraction(float(v)) for v in xg]
    b = max(abs(v) for v in vals)
    sx = r32(b / 127)
    if sx == 0:
        return [0] * len(vals), sx
    return [max(-127, min(127, _rint_half_even(r32(v / sx)))) for v in vals], sx


def test_activation_quant_exact_rational_and_bounds():
    rng = np.random.default_rng(5)
    x = rng.standard_t(4, 1024).astype(np.float32)
    x[7] = 0.0
    x[300:310] *= 30.0
    kept = O.select_inputs(x, 512)
    qx, sx = O.quantize_activations(x, kept, 128)
    xh = np.zeros_like(x)
    xh[kept] = x[kept]
    for g in range(8):
        qe, sxe = _exact_act_quant(xh[g * 128:(g + 1) * 128])
        assert Fraction(float(sx[g])) == sxe
        assert list(qx[g * 128:(g + 1) * 128]) == qe
    sxf = np.repeat(sx.astype(np.float64), 128)
    assert np.all(np.abs(xh - qx * sxf) <= sxf / 2 * (1 + 1e-6))
    assert np.all(qx[np.setdiff1d(np.arange(1024), kept)] == 0)
    # a group with nothing kept quantizes to zero with a zero scale
    qz, sz = O.quantize_activations(np.ones(256, np.float32), np.arange(128), 128)
    assert sz[1] == 0 and np.all(qz[128:] == 0) and np.all(qz[:128] == 127)


# ----------------------------------------------------------------------------- accumulators

def test_proxy_accumulators_pure_python():
    rng = np.random.default_rng(6)
    d, F = 256, 5
    q = rng.integers(-7, 8, (F, d)).astype(np.int8)
    qx = rng.integers(-127, 128, d).astype(np.int32)
    A = O.proxy_accumulators(qx, q, 128)
    for g in range(2):
        for j in range(F):
            s = 0
            for i in range(g * 128, (g + 1) * 128):
                s += int(qx[i]) * int(q[j][i])
            assert A[g][j] == s


# ----------------------------------------------------------------------------- lossless pipeline

def _lossless_layer(rng, d, F):
    """Weights exactly q * 2^e per (channel, group), |q| <= 7 with one |q| = 7 per group, so
    the INT4 proxy is exact; W_down is plain random bf16."""
    G = d // 128
    mats, qs, es = {}, {}, {}
    for name in ("w_gate", "w_up"):
        q = rng.integers(-7, 8, (F, d))
        pos = rng.integers(0, 128, (F, G)) + 128 * np.arange(G)[None, :]
        np.put_along_axis(q, pos, rng.choice([-7, 7], (F, G)), axis=1)
        e = rng.integers(-9, -4, (F, G))
        mats[name] = (q * np.exp2(np.repeat(e, 128, axis=1))).astype(np.float32)
        qs[name], es[name] = q, e
    mats["w_down"] = _bf16_values(rng, d * F, -9, -5).reshape(d, F)
    return mats, qs, es


def _lossless_tokens(rng, d):
    """x exactly qx * 2^f per group with one |qx| = 127 per group; distinct magnitudes at the
    top so the input selection has no tie at any k used below."""
    G = d // 128
    while True:
        qx = rng.integers(-126, 127, d)
        pos = rng.integers(0, 128, G) + 128 * np.arange(G)
        qx[pos] = rng.choice([-127, 127], G)
        f = rng.integers(-6, -1, G)
        x = (qx * np.exp2(np.repeat(f, 128))).astype(np.float32)
        mags = np.sort(np.abs(x))[::-1]
        k_in = O.k_for(0.5, d)
        if mags[k_in - 1] != mags[k_in]:
            return x, qx, f


@pytest.mark.parametrize("input_sparsity", [0.0, 0.5])
def test_lossless_proxy_equals_exact_swiglu_ranking(input_sparsity):
    rng = np.random.default_rng(7 + int(input_sparsity * 10))
    d, F = 512, 96
    mats, qs, es = _lossless_layer(rng, d, F)
    layer = O.prepare_layer(mats["w_gate"], mats["w_up"], mats["w_down"])
    np.testing.assert_array_equal(layer.q_gate, qs["w_gate"])
    np.testing.assert_array_equal(layer.q_up, qs["w_up"])
    np.testing.assert_array_equal(layer.sw_gate.astype(np.float64), np.exp2(es["w_gate"]).T)
    for _ in range(4):
        x, qx_true, f = _lossless_tokens(rng, d)
        k_in = O.k_for(input_sparsity, d)
        st = O.stage1_token(layer, x, input_sparsity)
        kept_ref = torch.topk(torch.from_numpy(np.abs(x)), k_in).indices.numpy()
        assert set(st["kept"].tolist()) == set(kept_ref.tolist())
        np.testing.assert_array_equal(st["qx"][st["kept"]], qx_true[st["kept"]])
        # exact SwiGLU on the sparse input, by torch in fp64
        xh = torch.zeros(d, dtype=torch.float64)
        xh[kept_ref] = torch.from_numpy(x.astype(np.float64))[kept_ref]
        g = torch.from_numpy(mats["w_gate"].astype(np.float64)) @ xh
        u = torch.from_numpy(mats["w_up"].astype(np.float64)) @ xh
        s_ref = (torch.nn.functional.silu(g) * u).abs().numpy()
        np.testing.assert_allclose(st["g_t"], g.numpy(), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(st["u_t"], u.numpy(), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(st["sigma"], s_ref, rtol=1e-11, atol=1e-13)
        for sparsity in (0.3, 0.5, 0.7, 0.9):
            k = O.k_for(sparsity, F)
            srt = np.sort(s_ref)[::-1]
            if k < F and (srt[k - 1] - srt[k]) <= 1e-9 * srt[k - 1]:
                continue
            ref = torch.topk(torch.from_numpy(s_ref), k).indices.numpy()
            assert set(O.channel_mask(st["sigma"], k).tolist()) == set(ref.tolist())


def test_channel_mask_brute_force_with_ties():
    rng = np.random.default_rng(8)
    for _ in range(80):
        F = int(rng.integers(2, 12))
        k = int(rng.integers(1, F + 1))
        sig = rng.integers(0, 5, F)
        got = tuple(O.channel_mask(sig.astype(np.float64), k))
        assert got == _brute_topk([int(v) for v in sig], k)
        assert list(got) == sorted(got)


# ----------------------------------------------------------------------------- Stage 2 / whole path

def _torch_ffn(x, mats, mask=None):
    X = torch.from_numpy(np.asarray(x, np.float64))
    Wg = torch.from_numpy(mats["w_gate"].astype(np.float64))
    Wu = torch.from_numpy(mats["w_up"].astype(np.float64))
    Wd = torch.from_numpy(mats["w_down"].astype(np.float64))
    s = torch.nn.functional.silu(Wg @ X) * (Wu @ X)
    if mask is not None:
        s = s * torch.from_numpy(mask.astype(np.float64))
    return (Wd @ s).numpy()


def _random_mats(rng, d, F):
    return {"w_gate": _bf16_values(rng, F * d, -9, -5).reshape(F, d),
            "w_up": _bf16_values(rng, F * d, -9, -5).reshape(F, d),
            "w_down": _bf16_values(rng, d * F, -9, -5).reshape(d, F)}


def test_sparsity_zero_is_dense_swiglu():
    rng = np.random.default_rng(9)
    d, F = 256, 200
    mats = _random_mats(rng, d, F)
    layer = O.prepare_layer(mats["w_gate"], mats["w_up"], mats["w_down"])
    x = rng.standard_t(4, d).astype(np.float32)
    out = O.ffn_token(layer, x, 0.0, 0.5)
    ref = _torch_ffn(x, mats)
    np.testing.assert_allclose(out["y"], ref, rtol=1e-11, atol=1e-14 * np.abs(ref).max())
    np.testing.assert_allclose(O.dense_ffn(x, **mats), ref, rtol=1e-11,
                               atol=1e-14 * np.abs(ref).max())


def test_stage2_is_dense_ffn_with_masked_intermediate():
    rng = np.random.default_rng(10)
    d, F = 256, 300
    mats = _random_mats(rng, d, F)
    layer = O.prepare_layer(mats["w_gate"], mats["w_up"], mats["w_down"])
    for sparsity in (0.5, 0.7, 0.9):
        x = rng.standard_t(4, d).astype(np.float32)
        out = O.ffn_token(layer, x, sparsity, 0.5)
        assert len(out["idx"]) == O.k_for(sparsity, F)
        mask = np.zeros(F)
        mask[out["idx"]] = 1
        ref = _torch_ffn(x, mats, mask)
        np.testing.assert_allclose(out["y"], ref, rtol=1e-10, atol=1e-13 * np.abs(ref).max())
        # an arbitrary mask, too
        idx = np.sort(rng.choice(F, 37, replace=False))
        y, _ = O.stage2_exact(x, mats["w_gate"], mats["w_up"], mats["w_down"], idx)
        m2 = np.zeros(F)
        m2[idx] = 1
        np.testing.assert_allclose(y, _torch_ffn(x, mats, m2), rtol=1e-10, atol=1e-15)


def test_quantized_mask_recalls_exact_mask():
    """Sanity, not parity: the pages print no recall figure. A correct int4 proxy with half
    the inputs kept recovers most of the exact top-k; a sign, index or operand slip in the
    proxy path drops recall to chance level (~ 1 - sparsity)."""
    rng = np.random.default_rng(11)
    d, F = 1024, 1024
    mats = {k: v for k, v in _random_mats(rng, d, F).items()}
    layer = O.prepare_layer(mats["w_gate"], mats["w_up"], mats["w_down"])
    recalls = []
    for _ in range(4):
        x = rng.standard_t(4, d).astype(np.float32)
        out = O.ffn_token(layer, x, 0.5, 0.5)
        X = x.astype(np.float64)
        s = np.abs(O.silu(mats["w_gate"] @ X) * (mats["w_up"] @ X))
        exact = set(np.argsort(-s)[:out["k"]].tolist())
        recalls.append(len(exact & set(out["idx"].tolist())) / out["k"])
    assert np.mean(recalls) > 0.8


def test_batch_union_against_dense_masks():
    rng = np.random.default_rng(12)
    F = 500
    idxs = [np.sort(rng.choice(F, int(rng.integers(1, 200)), replace=False)) for _ in range(5)]
    U, bits = O.batch_union(idxs, F)
    dense = np.zeros((5, F), bool)
    for b, ix in enumerate(idxs):
        dense[b, ix] = True
    anyb = dense.any(axis=0)
    np.testing.assert_array_equal(U, np.nonzero(anyb)[0])
    np.testing.assert_array_equal(bits, dense[:, anyb])


def test_rmsnorm_closed_form():
    rng = np.random.default_rng(13)
    y = rng.normal(0, 3, (3, 4096))
    out = O.rmsnorm(y, 1e-6)
    m = np.mean(y * y, axis=1)
    np.testing.assert_allclose(np.mean(out * out, axis=1), m / (m + 1e-6), rtol=1e-12)
    np.testing.assert_allclose(out / np.linalg.norm(out, axis=1, keepdims=True),
                               y / np.linalg.norm(y, axis=1, keepdims=True), rtol=1e-12)


def test_proxy_overhead_matches_pages():
    with open(os.path.join(GOLDEN, "proxy_overhead.json")) as f:
        gold = json.load(f)
    model_bytes = gold["params"] * gold["bytes_per_param"]
    frac = gold["n_layers"] * O.proxy_storage_bytes(gold["d_model"], gold["d_ff"]) / model_bytes
    assert abs(frac - gold["claim_fraction"]) <= gold["tolerance"], frac
    # the alternatives the reading rejects fall outside the pages' figure
    d, F, L = gold["d_model"], gold["d_ff"], gold["n_layers"]
    all_three = L * (O.proxy_storage_bytes(d, F) * 3 / 2) / model_bytes
    int8_gate_up = L * (2 * d * F + 2 * (d // 128) * F * 2) / model_bytes
    assert all_three - gold["claim_fraction"] > gold["tolerance"]
    assert int8_gate_up - gold["claim_fraction"] > gold["tolerance"]


def test_proxy_storage_counts_the_quantizers_outputs():
    """The proxy bytes of a layer are what the quantizer produces: two int4 codes per (input,
    channel) pair, one for W_gate and one for W_up, packed two to a byte, plus both projections'
    fp16 group scales (counted from the arrays quantize_weight_proxy returns)."""
    rng = np.random.default_rng(14)
    for d, F in ((256, 96), (384, 160)):
        wg = rng.normal(0, 0.02, (F, d)).astype(np.float32)
        wu = rng.normal(0, 0.02, (F, d)).astype(np.float32)
        qg, sg = O.quantize_weight_proxy(wg, 128)
        qu, su = O.quantize_weight_proxy(wu, 128)
        nibbles = qg.size + qu.size                       # one 4-bit code each
        assert O.proxy_storage_bytes(d, F) == nibbles // 2 + sg.nbytes + su.nbytes
