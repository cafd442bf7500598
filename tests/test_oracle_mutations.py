"""Plants plausible mistakes in the oracle, one at a time and on the CPU only, and checks that the
oracle's pins catch every one of them: the pins of tests/test_oracle_pins.py,
tests/test_fp8_oracle.py and tests/test_sparsity_allocation.py (except the tests that compare
the library with the oracle, which are not independent of the product). The unmodified oracle
passes every pin. Each mistake is a one-line change of one oracle function, written out below.
"""
import contextlib
import inspect
import math

import numpy as np
import pytest

import oracle as O
import oracle.fp8_weights as F8
import oracle.prox_oracle as PO
import oracle.sparsity_allocation as SA
import test_fp8_oracle as PINS_FP8
import test_oracle_pins as PINS
import test_sparsity_allocation as PINS_ALLOC

_silu = PO.silu


def _pins():
    """(name, zero-argument call) for every independent pin, parametrizations expanded."""
    out = []
    for mod in (PINS, PINS_FP8, PINS_ALLOC):
        for name, fn in sorted(vars(mod).items()):
            if not name.startswith("test_") or not callable(fn) or "library" in name:
                continue
            marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
            if not marks:
                if inspect.signature(fn).parameters:
                    continue   # needs fixtures: not a pure pin
                out.append((name, fn))
                continue
            argnames, values = marks[0].args[0], marks[0].args[1]
            argnames = [a.strip() for a in argnames.split(",")] if isinstance(argnames, str) else argnames
            for v in values:
                args = v if len(argnames) > 1 else (v,)
                out.append((f"{name}{list(args)}", lambda fn=fn, args=args: fn(*args)))
    return out


def _failures():
    bad = []
    for name, call in _pins():
        try:
            call()
        except Exception:   # an assertion, or the mutation broke the call itself
            bad.append(name)
    return bad


@contextlib.contextmanager
def _planted(module, attr, fn):
    """Replace module.attr (and its re-export in the oracle package) for the duration."""
    old = getattr(module, attr)
    pkg_old = getattr(O, attr, None)
    setattr(module, attr, fn)
    if pkg_old is old:
        setattr(O, attr, fn)
    try:
        yield
    finally:
        setattr(module, attr, old)
        if pkg_old is old:
            setattr(O, attr, old)


# ------------------------------------------------------------------ the mistakes

def k_for_no_half(sparsity, n):                      # floor without the +0.5
    return int(min(max(math.floor((1.0 - float(sparsity)) * n), 1), n))


def silu_wrong_sign(z):                              # z * sigmoid(-z)
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(z))


def _weight_proxy(w, group, divisor, lo):
    w = np.asarray(w, dtype=np.float32)
    F, d = w.shape
    G = d // group
    wg = w.reshape(F, G, group)
    a = np.max(np.abs(wg), axis=2)
    sw16 = (a / np.float32(divisor)).astype(np.float16)
    sw = sw16.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.rint(wg / sw[:, :, None])
    q = np.where(sw[:, :, None] == 0, 0.0, np.clip(r, lo, 7))
    return q.astype(np.int8).reshape(F, d), np.ascontiguousarray(sw16.T)


def weight_scale_over_8(w, group=PO.GROUP):         # scale max|w| / 8
    return _weight_proxy(w, group, 8.0, -7)


def weight_truncated(w, group=PO.GROUP):            # codes truncated instead of rounded
    w = np.asarray(w, dtype=np.float32)
    F, d = w.shape
    G = d // group
    wg = w.reshape(F, G, group)
    sw16 = (np.max(np.abs(wg), axis=2) / np.float32(7.0)).astype(np.float16)
    sw = sw16.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.trunc(wg / sw[:, :, None])
    q = np.where(sw[:, :, None] == 0, 0.0, np.clip(r, -7, 7))
    return q.astype(np.int8).reshape(F, d), np.ascontiguousarray(sw16.T)


def select_ties_high(x, k_in):                       # equal magnitudes to the higher index
    x = np.asarray(x)
    d = x.shape[0]
    order = np.lexsort((-np.arange(d), -np.abs(x.astype(np.float64))))
    return np.sort(order[:k_in]).astype(np.int64)


def select_signed(x, k_in):                          # largest x instead of largest |x|
    x = np.asarray(x)
    d = x.shape[0]
    order = np.lexsort((np.arange(d), -x.astype(np.float64)))
    return np.sort(order[:k_in]).astype(np.int64)


def _act_quant(x, kept, group, divisor, sparse=True):
    x = np.asarray(x, dtype=np.float32)
    d = x.shape[0]
    G = d // group
    xh = np.zeros(d, np.float32)
    if sparse:
        xh[kept] = x[kept]
    else:
        xh[:] = x
    xg = xh.reshape(G, group)
    sx = (np.max(np.abs(xg), axis=1) / np.float32(divisor)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.rint(xg / sx[:, None])
    qx = np.where(sx[:, None] == 0, 0.0, np.clip(r, -127, 127))
    return qx.astype(np.int32).reshape(d), sx


def act_scale_over_128(x, kept, group=PO.GROUP):    # scale max|x| / 128
    return _act_quant(x, kept, group, 128.0)


def act_keeps_rejected(x, kept, group=PO.GROUP):    # input sparsity not applied
    return _act_quant(x, kept, group, 127.0, sparse=False)


def acc_shifted_groups(qx, q, group=PO.GROUP):      # group g summed over inputs shifted by one
    F, d = q.shape
    G = d // group
    A = np.empty((G, F), np.int64)
    qx64 = np.asarray(qx, dtype=np.int64)
    for g in range(G):
        sl = np.arange(g * group + 1, (g + 1) * group + 1) % d
        A[g] = q[:, sl].astype(np.int64) @ qx64[sl]
    return A


def _salience(A_gate, A_up, sx, sw_gate, sw_up, form):
    G, F = A_gate.shape
    g_t = np.zeros(F, np.float64)
    u_t = np.zeros(F, np.float64)
    for g in range(G):
        sxg = np.float64(sx[g])
        g_t = g_t + (sxg * sw_gate[g].astype(np.float64)) * A_gate[g].astype(np.float64)
        u_t = u_t + (sxg * sw_up[g].astype(np.float64)) * A_up[g].astype(np.float64)
    sigma = np.abs(form(g_t, u_t))
    return sigma, g_t, u_t


def salience_without_silu(A_gate, A_up, sx, sw_gate, sw_up):      # |g~ u~|
    return _salience(A_gate, A_up, sx, sw_gate, sw_up, lambda g, u: g * u)


def salience_gate_and_up_swapped(A_gate, A_up, sx, sw_gate, sw_up):   # |SiLU(u~) g~|
    return _salience(A_gate, A_up, sx, sw_gate, sw_up, lambda g, u: _silu(u) * g)


def mask_ties_high(sigma, k):                        # equal saliences to the higher index
    sigma = np.asarray(sigma, dtype=np.float64)
    F = sigma.shape[0]
    order = np.lexsort((-np.arange(F), -sigma))
    return np.sort(order[:k]).astype(np.int64)


def stage2_silu_on_up(x, w_gate, w_up, w_down, idx):   # SiLU on the up projection
    x64 = np.asarray(x, dtype=np.float64)
    idx = np.asarray(idx, dtype=np.int64)
    g = np.asarray(w_gate, dtype=np.float64)[idx] @ x64
    u = np.asarray(w_up, dtype=np.float64)[idx] @ x64
    s = _silu(u) * g
    return np.asarray(w_down, dtype=np.float64)[:, idx] @ s, s


def rmsnorm_eps_outside(y, eps=1e-6):                # y / (sqrt(mean y^2) + eps)
    y = np.asarray(y, dtype=np.float64)
    return y / (np.sqrt(np.mean(y * y, axis=-1, keepdims=True)) + eps)


def union_is_intersection(idx_list, n):              # the tokens' common channels only
    sets = [set(int(v) for v in np.asarray(ix).ravel()) for ix in idx_list]
    U = np.array(sorted(set.intersection(*sets)) if sets else [], dtype=np.int64)
    bits = np.array([[int(u) in s for u in U] for s in sets], dtype=bool).reshape(len(sets), len(U))
    return U, bits


def storage_scales_once(d_model, d_ff, group=PO.GROUP):   # one projection's scales counted
    G = d_model // group
    return d_model * d_ff + G * d_ff * 2


def e4m3_round_truncating(v):                        # mantissa truncated instead of rounded
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    a = np.abs(v)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, F8.E4M3_MIN_EXP)
    quantum = np.exp2(e - 3)
    r = np.minimum(np.floor(a / quantum) * quantum, F8.E4M3_MAX)
    return np.copysign(r, v) * (a > 0)


def e4m3_bits_bias_8(q):                             # exponent bias 8 instead of 7
    q = np.asarray(q, dtype=np.float64)
    a = np.abs(q)
    sign = np.signbit(q).astype(np.uint8) << 7
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    normal = (e >= F8.E4M3_MIN_EXP) & (a > 0)
    e = np.maximum(e, F8.E4M3_MIN_EXP)
    m = np.where(normal, a / np.exp2(e) - 1.0, a / np.exp2(F8.E4M3_MIN_EXP)) * 8.0
    code = (np.where(normal, e + 8, 0).astype(np.int64) << 3) | np.rint(m).astype(np.int64)
    return sign | (code & 0x7F).astype(np.uint8)


def fp8_rows_scale_447(w):                           # row scale max|w| / 447
    w = np.asarray(w, dtype=np.float32)
    s = (np.max(np.abs(w), axis=1) / np.float32(447.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = (w / s[:, None]).astype(np.float32)
    return np.where(s[:, None] == 0, 0.0, F8.e4m3_round(np.nan_to_num(t))), s


def allocate_without_input_floor(cost, d_model, d_ff, target, anchor=0.7, min_input_kept=0.3):
    return _allocate(cost, d_model, d_ff, target, anchor, 1e-9)   # the 30% floor dropped


_allocate = SA.allocate_sparsity


def allocate_channels_off_anchor(cost, d_model, d_ff, target, anchor=0.7, min_input_kept=0.3):
    return _allocate(cost, d_model, d_ff, target, anchor + 0.05, min_input_kept)


MUTATIONS = [
    (PO, "k_for", k_for_no_half),
    (PO, "silu", silu_wrong_sign),
    (PO, "quantize_weight_proxy", weight_scale_over_8),
    (PO, "quantize_weight_proxy", weight_truncated),
    (PO, "select_inputs", select_ties_high),
    (PO, "select_inputs", select_signed),
    (PO, "quantize_activations", act_scale_over_128),
    (PO, "quantize_activations", act_keeps_rejected),
    (PO, "proxy_accumulators", acc_shifted_groups),
    (PO, "proxy_salience", salience_without_silu),
    (PO, "proxy_salience", salience_gate_and_up_swapped),
    (PO, "channel_mask", mask_ties_high),
    (PO, "stage2_exact", stage2_silu_on_up),
    (PO, "rmsnorm", rmsnorm_eps_outside),
    (PO, "batch_union", union_is_intersection),
    (PO, "proxy_storage_bytes", storage_scales_once),
    (F8, "e4m3_round", e4m3_round_truncating),
    (F8, "e4m3_bits", e4m3_bits_bias_8),
    (F8, "quantize_rows_e4m3", fp8_rows_scale_447),
    (SA, "allocate_sparsity", allocate_without_input_floor),
    (SA, "allocate_sparsity", allocate_channels_off_anchor),
]


def test_unmodified_oracle_passes_every_pin():
    assert _failures() == []


@pytest.mark.parametrize("module,attr,mistake", MUTATIONS, ids=[m[2].__name__ for m in MUTATIONS])
def test_planted_mistake_is_caught(module, attr, mistake):
    with _planted(module, attr, mistake):
        caught = _failures()
    assert caught, f"no pin catches {mistake.__name__} in {attr}"
