"""Oracle of Stage 2 over FP8 weights (test infrastructure only, like the rest of oracle/).

What it follows: "Prox: Training-Free FFN Activation Sparsity via Approximate
Intermediate-Channel Salience in LLMs", technical summary, "Experimental Results",
Compatibility: Prox is orthogonal to weight quantization such as FP8. Stage 2 ("Exact Sparse
Computation") then multiplies the masked channels with the quantized weights in place of the
bf16 ones; Stage 1 keeps its INT4 proxies of the original weights.

Reading (R12; the pages name FP8 only): OCP FP8 E4M3 ("e4m3fn": 4 exponent bits, bias 7,
3 mantissa bits, no infinities, largest finite 448) with one fp32 scale per weight row, the
rows being W_gate[j, :], W_up[j, :] and W_down[:, j] of channel j:
    s = fp32(max |w|) / 448      (binary32 divide)
    q = e4m3(fp32(w) / s)         (binary32 divide, round to nearest even, saturating at 448)
    q = 0 where s = 0
and the dequantized weight is q * s (exact in fp64). A quotient that rounds to zero keeps
its sign, as IEEE rounding does (a tiny negative weight has code 0x80, value -0). Stage 2
over FP8 weights is stage2_exact over the dequantized matrices.
Pinned in tests/test_fp8_oracle.py: the value set against the format's closed-form
definition, the rounding against torch's float8_e4m3fn cast, saturation, and the row scale.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_EXP = -6    # smallest normal exponent; subnormals are multiples of 2^-9


def e4m3_round(v) -> np.ndarray:
    """Nearest E4M3 value of each element (ties to the even mantissa), saturated at +-448, as
    fp64. Inputs are binary32 values."""
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    a = np.abs(v)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, E4M3_MIN_EXP)
    quantum = np.exp2(e - 3)                    # 3 mantissa bits
    r = np.rint(a / quantum) * quantum          # exact scaling by a power of two; RNE
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, v) * (a > 0)


def e4m3_bits(q) -> np.ndarray:
    """The 8-bit codes of E4M3 values (sign | exponent << 3 | mantissa)."""
    q = np.asarray(q, dtype=np.float64)
    a = np.abs(q)
    sign = np.signbit(q).astype(np.uint8) << 7   # a negative zero keeps its sign bit
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    normal = e >= E4M3_MIN_EXP
    e = np.maximum(e, E4M3_MIN_EXP)
    normal &= a > 0                             # zero is the subnormal with mantissa 0
    m = np.where(normal, a / np.exp2(e) - 1.0, a / np.exp2(E4M3_MIN_EXP)) * 8.0
    exp_field = np.where(normal, e + 7, 0)
    code = (exp_field.astype(np.int64) << 3) | np.rint(m).astype(np.int64)
    return sign | code.astype(np.uint8)


def quantize_rows_e4m3(w) -> tuple[np.ndarray, np.ndarray]:
    """Per-row FP8 E4M3 quantization of w [R, n] (exact bf16 values): returns
    (q [R, n] fp64 E4M3 values, s [R] float32 row scales), reading R12."""
    w = np.asarray(w, dtype=np.float32)
    a = np.max(np.abs(w), axis=1)
    s = (a / np.float32(E4M3_MAX)).astype(np.float32)        # binary32 divide
    with np.errstate(divide="ignore", invalid="ignore"):
        t = (w / s[:, None]).astype(np.float32)               # binary32 divide
    q = np.where(s[:, None] == 0, 0.0, e4m3_round(np.nan_to_num(t)))
    return q, s


def fp8_layer(w_gate, w_up, w_down) -> dict:
    """The FP8 copy of one layer's Stage-2 weights: codes, scales and dequantized matrices
    (W_down is quantized per column, i.e. per channel)."""
    qg, sg = quantize_rows_e4m3(w_gate)
    qu, su = quantize_rows_e4m3(w_up)
    qd, sd = quantize_rows_e4m3(np.asarray(w_down, dtype=np.float32).T)
    return {"q_gate": qg, "s_gate": sg, "q_up": qu, "s_up": su, "q_down": qd, "s_down": sd,
            "w_gate": qg * sg[:, None].astype(np.float64),
            "w_up": qu * su[:, None].astype(np.float64),
            "w_down": (qd * sd[:, None].astype(np.float64)).T}
