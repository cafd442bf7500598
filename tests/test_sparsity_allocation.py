"""Sparsity allocation (technical summary, "Sparsity Allocation"): the oracle's rule pinned by
hand-computed cases and by a brute-force search over every (kept inputs, kept channels) pair,
and the library's host-side call (prox_choose_sparsity) equal to the oracle everywhere.

Reading (the pages give no formula): effective sparsity = 1 - C with C the sparse path's cost
relative to the dense FFN, proxy included; the channels stay at the 70% anchor while the
budget allows, Stage 1 keeps at least 30% of the inputs.
"""
import ctypes
import math

import numpy as np
import pytest

import oracle as O
from free_sparse_swiglu_stage1_b300 import _lib

LLAMA3 = (4096, 14336)


def test_byte_cost_model_llama3():
    c = O.byte_cost_model(*LLAMA3)
    # one byte of gate+up codes per channel and kept input; 32 groups x 2 fp16 scales; three
    # bf16 rows per channel; the dense FFN reads 3 x 4096 x 14336 bf16 values
    assert c == {"in_cost": 14336.0, "fixed_cost": 1835008.0, "ch_cost": 24576.0,
                 "dense_cost": 352321536.0}


@pytest.mark.parametrize("target,k_in,k", [
    (0.6, 2329, 4301),    # channels at the anchor, inputs fill the budget
    (0.3, 4096, 7571),    # every input fits: the rest buys channels beyond the anchor
    (0.75, 1229, 2792),   # the 30%-of-inputs floor binds: channels drop below the anchor
])
def test_llama3_hand_computed(target, k_in, k):
    """Worked by hand from the byte model: budget (1 - t) x 352321536 bytes, 4301 channels at
    the anchor (24576 bytes each), 1835008 bytes of scales, 14336 bytes per kept input, at
    least ceil(0.3 x 4096) = 1229 inputs."""
    s1, s2, eff = O.allocate_sparsity(O.byte_cost_model(*LLAMA3), *LLAMA3, target)
    assert O.k_for(s1, 4096) == k_in and O.k_for(s2, 14336) == k
    assert eff >= target
    assert math.isclose(eff, 1 - (14336 * k_in + 1835008 + 24576 * k) / 352321536, rel_tol=1e-15)


def _brute(cost, d, F, target, anchor, keep):
    """The rule stated by enumerating every (k_in, k) pair and the cost in exact rationals."""
    from fractions import Fraction as Q
    budget = (1 - Q(target)) * Q(cost["dense_cost"])

    def fits(a, b):
        return Q(cost["in_cost"]) * a + Q(cost["fixed_cost"]) + Q(cost["ch_cost"]) * b <= budget

    k_min = max(1, min(d, math.ceil(Q(keep) * d)))
    ka = O.k_for(anchor, F)
    at_anchor = [a for a in range(1, d + 1) if fits(a, ka)]
    if at_anchor and max(at_anchor) >= k_min:
        a = max(at_anchor)
        if a == d:
            return d, max(b for b in range(1, F + 1) if fits(d, b))
        return a, ka
    bs = [b for b in range(1, F + 1) if fits(k_min, b)]
    return (k_min, max(bs)) if bs else None


def test_brute_force_small_layers():
    rng = np.random.default_rng(3)
    cases = 0
    for d, F in ((256, 64), (384, 96), (128, 32)):
        for trial in range(60):
            if trial % 2:
                cost = O.byte_cost_model(d, F)
            else:   # a measured-time-like model with fractional costs
                cost = {"in_cost": float(rng.uniform(0.5, 3)), "fixed_cost": float(rng.uniform(0, 50)),
                        "ch_cost": float(rng.uniform(2, 20)), "dense_cost": 0.0}
                cost["dense_cost"] = cost["ch_cost"] * F * float(rng.uniform(1.0, 1.3))
            target = float(rng.uniform(0, 0.95))
            anchor = float(rng.choice([0.5, 0.7, 0.9]))
            keep = float(rng.choice([0.3, 0.5]))
            got = O.allocate_sparsity(cost, d, F, target, anchor, keep)
            want = _brute(cost, d, F, target, anchor, keep)
            if want is None:
                assert got is None
                continue
            assert got is not None
            assert (O.k_for(got[0], d), O.k_for(got[1], F)) == want, (d, F, target, anchor, keep)
            cases += 1
    assert cases > 100


def test_properties_llama3():
    cost = O.byte_cost_model(*LLAMA3)
    prev = None
    for t in np.linspace(0.0, 0.8, 81):
        s1, s2, eff = O.allocate_sparsity(cost, *LLAMA3, float(t))
        k_in, k = O.k_for(s1, 4096), O.k_for(s2, 14336)
        assert eff >= t - 1e-12
        assert k_in >= 1229                     # at least 30% of the inputs kept
        if 1229 < k_in < 4096:
            assert k == 4301                    # channels at the anchor
        # the quantity the rule fills last cannot grow by one within the budget: inputs while
        # the channels sit at the anchor, otherwise channels
        if k == 4301 and k_in < 4096:
            assert O.normalized_cost(cost, k_in + 1, k) > 1 - t
        elif k < 14336:
            assert O.normalized_cost(cost, k_in, k + 1) > 1 - t
        if prev is not None:                    # a higher target never keeps more
            assert k_in <= prev[0] and k <= prev[1]
        prev = (k_in, k)


def test_library_matches_oracle():
    L = _lib.lib()
    for d, F in (LLAMA3, (4096, 11008), (8192, 28672), (1024, 2816), (256, 64)):
        cm = _lib.prox_cost_model()
        assert L.prox_cost_model_bytes(d, F, ctypes.byref(cm)) == 0
        oc = O.byte_cost_model(d, F)
        assert (cm.in_cost, cm.fixed_cost, cm.ch_cost, cm.dense_cost) == \
            (oc["in_cost"], oc["fixed_cost"], oc["ch_cost"], oc["dense_cost"])
        for t in np.linspace(0.0, 0.95, 39):
            for anchor in (0.5, 0.7):
                s1, s2, eff = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
                rc = L.prox_choose_sparsity(ctypes.byref(cm), d, F, float(t), anchor, 0.3,
                                            ctypes.byref(s1), ctypes.byref(s2), ctypes.byref(eff))
                want = O.allocate_sparsity(oc, d, F, float(t), anchor, 0.3)
                if want is None:
                    assert rc == -6
                    continue
                assert rc == 0
                assert (s1.value, s2.value, eff.value) == want
                assert L.prox_k_for(s1.value, d) == O.k_for(want[0], d)
                assert L.prox_k_for(s2.value, F) == O.k_for(want[1], F)


def test_library_rejects_bad_arguments():
    L = _lib.lib()
    cm = _lib.prox_cost_model(1.0, 0.0, 1.0, 10.0)
    out = ctypes.c_double()
    assert L.prox_choose_sparsity(None, 256, 64, 0.5, 0.7, 0.3, None, None, None) == -1
    assert L.prox_choose_sparsity(ctypes.byref(cm), 256, 64, 1.0, 0.7, 0.3, None, None, None) == -1
    assert L.prox_choose_sparsity(ctypes.byref(cm), 256, 64, 0.5, 1.0, 0.3, None, None, None) == -1
    assert L.prox_choose_sparsity(ctypes.byref(cm), 256, 64, 0.5, 0.7, 0.0, None, None, None) == -1
    bad = _lib.prox_cost_model(0.0, 0.0, 1.0, 10.0)
    assert L.prox_choose_sparsity(ctypes.byref(bad), 256, 64, 0.5, 0.7, 0.3, ctypes.byref(out),
                                  None, None) == -1
    assert L.prox_cost_model_bytes(100, 64, ctypes.byref(cm)) == -1


def test_cost_model_fit_recovers_a_linear_model():
    """The fit against numpy's least squares, on exact and on noisy synthetic measurements."""
    from free_sparse_swiglu_stage1_b300 import prox_cost_model_fit
    rng = np.random.default_rng(7)
    k_in = np.array([2048, 4096, 2048, 1229, 3000, 1500], float)
    k = np.array([4301, 4301, 8602, 1434, 6000, 3000], float)
    a, b, c = 2.5e-3, 9.0, 3.1e-3
    t = a * k_in + b + c * k
    m = prox_cost_model_fit(k_in, k, t, 60.0)
    assert math.isclose(m.in_cost, a, rel_tol=1e-9) and math.isclose(m.fixed_cost, b, rel_tol=1e-9)
    assert math.isclose(m.ch_cost, c, rel_tol=1e-9) and m.dense_cost == 60.0
    tn = t + rng.normal(0, 0.3, len(t))
    m = prox_cost_model_fit(k_in, k, tn, 60.0)
    want = np.linalg.lstsq(np.stack([k_in, np.ones_like(k_in), k], 1), tn, rcond=None)[0]
    np.testing.assert_allclose([m.in_cost, m.fixed_cost, m.ch_cost], want, rtol=1e-9, atol=1e-12)


def test_cost_model_fit_guards():
    from free_sparse_swiglu_stage1_b300 import ProxError, prox_cost_model_fit
    # a term the times do not depend on is raised to min_cost, so allocation still accepts it
    m = prox_cost_model_fit([1, 2, 3, 4], [10, 10, 20, 20], [5, 5, 5, 5], 10.0, min_cost=1e-6)
    assert m.in_cost == 1e-6 and m.ch_cost == 1e-6 and math.isclose(m.fixed_cost, 5.0)
    with pytest.raises(ProxError):   # all points on one line: the coefficients are not determined
        prox_cost_model_fit([1, 2, 3], [1, 2, 3], [1, 2, 3], 10.0)
    with pytest.raises(ProxError):
        prox_cost_model_fit([1, 2], [1, 2], [1, 2], 10.0)
    with pytest.raises(ProxError):
        prox_cost_model_fit([1, 2, 3], [3, 1, 2], [1, 2, 3], 0.0)
