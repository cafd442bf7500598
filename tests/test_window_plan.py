"""The proxy window's slot policy (prox_debug_window_plan: the policy alone, on the host),
checked against what the window must guarantee: an acquired layer is in the slot it was given,
a slot in use is never overwritten, decode order keeps every layer copied ahead of its visit,
and a window as large as the stack copies every layer once (technical summary, "Significance
and Claims": sliding-window schemes for the proxies' memory; the reading is in the header)."""
import random

import pytest

from free_sparse_swiglu_stage1_b300 import prox_debug_window_plan


def _replay(n_layers, n_slots, ops):
    """Runs the policy and checks every op against a model of the slot contents built from
    the copy log alone. Returns (slots, copies)."""
    slots, copies, n = prox_debug_window_plan(n_layers, n_slots, ops)
    assert n == len(copies)
    held = [None] * n_slots
    busy = {}                        # layer -> slot, while acquired
    by_op = {}
    for op, s, layer in copies:
        by_op.setdefault(op, []).append((s, layer))
    for i, op in enumerate(ops):
        layer = op if op >= 0 else -1 - op
        if op < 0:                   # a release happens before its copies
            if layer in busy:
                assert slots[i] == busy.pop(layer)
            else:
                assert slots[i] == -1
        for s, m in by_op.get(i, []):
            assert 0 <= s < n_slots
            assert s not in busy.values(), f"op {i}: copy into slot {s} in use"
            assert m not in held, f"op {i}: layer {m} copied twice into the window"
            held[s] = m
        if op >= 0:
            if slots[i] < 0:
                # refused only when every slot is in use by an acquired layer
                assert len(busy) == n_slots
                continue
            assert held[slots[i]] == layer, f"op {i}: layer {layer} not in slot {slots[i]}"
            busy[layer] = slots[i]
    return slots, copies


@pytest.mark.parametrize("L,S", [(6, 2), (5, 3), (32, 4), (7, 1), (3, 8), (4, 4)])
def test_decode_order(L, S):
    steps = 3
    ops = []
    for _ in range(steps):
        for l in range(L):
            ops += [l, -1 - l]
    slots, copies = _replay(L, S, ops)
    if S >= L:
        assert len(copies) == L      # every layer once, then resident for good
        return
    # one copy per visit, plus the window's lookahead at the end
    assert steps * L <= len(copies) <= steps * L + S
    if S >= 2:
        # after the first visit every layer was copied at an earlier op than its acquire
        first = {}
        for op, s, layer in copies:
            first.setdefault((layer, op), True)
        for i, op in enumerate(ops):
            if op >= 0 and i > 0:
                assert all(o != i for o, _, _ in copies), f"acquire at op {i} had to copy"


def test_all_slots_in_use_is_refused():
    slots, _ = _replay(4, 2, [0, 1, 2, -1 - 0, 2])
    assert slots[2] == -1 and slots[4] >= 0


def test_release_of_a_layer_not_acquired():
    slots, _ = _replay(4, 2, [-1 - 3, 0, -1 - 1, -1 - 0, -1 - 0])
    assert slots[0] == -1 and slots[2] == -1 and slots[4] == -1


def test_random_orders():
    rng = random.Random(5)
    for trial in range(300):
        L = rng.randint(1, 9)
        S = rng.randint(1, 5)
        ops, held = [], []
        for _ in range(rng.randint(1, 60)):
            if held and (rng.random() < 0.5 or len(held) >= S):
                ops.append(-1 - held.pop(rng.randrange(len(held))))
            else:
                l = rng.randrange(L)
                if l not in held:
                    ops.append(l)
                    held.append(l)
        slots, _ = _replay(L, S, ops)
