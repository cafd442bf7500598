"""Oracle of the sparsity-allocation step (test infrastructure only, like the rest of oracle/).

What it follows: "Prox: Training-Free FFN Activation Sparsity via Approximate
Intermediate-Channel Salience in LLMs", technical summary, "Methodology: The Prox Framework",
subsection "Sparsity Allocation": the channel (Stage 2) sparsity s2 is anchored around 70%, the
input (Stage 1) sparsity s1 keeps at least 30% of the inputs, and a cost model picks s1 and s2
for a target effective sparsity, with the overhead of the quantized proxy counted.

The pages give no formula. Reading used here (R11):
  cost    C(k_in, k) = (in_cost k_in + fixed_cost + ch_cost k) / dense_cost, the sparse path's
          cost of one token relative to the dense FFN's; by default the costs are HBM bytes
          (byte_cost_model), a caller may pass measured times instead.
  target  effective sparsity = 1 - C: the share of the dense cost the sparse path saves,
          after paying for the proxy. A target t means C <= 1 - t.
  rule    keep the channels at the anchor (k = k_for(anchor, F)) and keep as many inputs as
          the budget allows; if that is every input, spend the rest on channels (more
          channels than the anchor); if it is fewer than the floor ceil(min_input_kept d),
          keep the floor and drop channels below the anchor to fit. Sparsities are returned as
          s1 = 1 - k_in / d, s2 = 1 - k / F, which the kept-count rule maps back to k_in, k.
Pinned in tests/test_sparsity_allocation.py by hand-computed cases and a brute-force search
over every (k_in, k) pair of small layers.
"""
from __future__ import annotations

import math

from .prox_oracle import GROUP, k_for


def byte_cost_model(d_model: int, d_ff: int, group: int = GROUP) -> dict:
    """Per-token HBM bytes of the path's parts: one byte of INT4 gate+up codes per (kept input,
    channel), the fp16 group scales of both proxies, three bf16 rows (6 d bytes) per selected
    channel; the dense FFN reads every channel's rows."""
    G = d_model // group
    return {"in_cost": float(d_ff), "fixed_cost": float(4 * G * d_ff),
            "ch_cost": float(6 * d_model), "dense_cost": float(6 * d_model * d_ff)}


def normalized_cost(cost: dict, k_in: int, k: int) -> float:
    return (cost["in_cost"] * k_in + cost["fixed_cost"] + cost["ch_cost"] * k) / cost["dense_cost"]


def allocate_sparsity(cost: dict, d_model: int, d_ff: int, target: float, anchor: float = 0.7,
                      min_input_kept: float = 0.3):
    """(input_sparsity, sparsity, effective_sparsity) for a target effective sparsity, by the
    rule of reading R11; None when no allocation fits the budget."""
    d, F = d_model, d_ff
    budget = (1.0 - target) * cost["dense_cost"]
    k_in_min = max(1, min(d, math.ceil(min_input_kept * d)))
    k_anchor = k_for(anchor, F)
    k_in = math.floor((budget - cost["fixed_cost"] - cost["ch_cost"] * k_anchor) / cost["in_cost"])
    if k_in >= d:
        k_in = d
        k = min(F, math.floor((budget - cost["fixed_cost"] - cost["in_cost"] * d) / cost["ch_cost"]))
    elif k_in >= k_in_min:
        k = k_anchor
    else:
        k_in = k_in_min
        k = math.floor((budget - cost["fixed_cost"] - cost["in_cost"] * k_in) / cost["ch_cost"])
        if k < 1:
            return None
    s1 = 1.0 - k_in / d
    s2 = 1.0 - k / F
    return s1, s2, 1.0 - normalized_cost(cost, k_in, k)
