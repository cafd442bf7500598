"""Plain CPU oracle for the Prox two-stage sparse SwiGLU FFN (decode, one layer).

TEST INFRASTRUCTURE ONLY. The test-suite, the smoke check and the benchmark's CPU-baseline
leg are the only code allowed to import or run this module. The CUDA product path never
calls it, and the two share no code: no kernels, headers, helpers, tables or constants.

What it follows: "Prox: Training-Free FFN Activation Sparsity via Approximate
Intermediate-Channel Salience in LLMs" -- the authors' abstract, and the technical summary
("Methodology: The Prox Framework", subsections "Stage 1: Lightweight Proxy Construction"
and "Stage 2: Exact Sparse Computation").

Notation. g = W_gate x, u = W_up x, a = SiLU(g) (the pages' gate activation h),
s = a * u (the pages' intermediate state s = u (.) h), y = W_down s. Proxy quantities carry
the suffix _t (the pages' tilde). F = d_ff channels, d = d_model inputs, G = d / group.

Arithmetic. fp64 throughout, except the two quantizers, whose reading fixes binary32
divisions and a binary16 scale; those run in exactly those formats (numpy float32/float16,
IEEE round-to-nearest-even), so the integer codes they produce are unique.

Readings of what the pages leave open (the pages only say "input sparsity", "INT4
proxy weights", "magnitude ranking"):
  R1  k = clamp(floor((1 - s) * n + 0.5), 1, n) in IEEE double, for channels (s = sparsity,
      n = F) and for inputs (s = input sparsity, n = d).
  R2  Input sparsity keeps the k_in largest |x_i|; equal magnitudes go to the lower index.
      Stage 1 then sees x_hat (x on kept entries, 0 elsewhere). Stage 2 uses the dense x.
  R3  Proxy weights: symmetric int4, group of 128 inputs along d per channel, codes in
      [-7, 7], scale sw = fp16(fp32(max|w|) / 7), q = clamp(rint(fp32(w) / fp32(sw)), -7, 7),
      q = 0 when sw == 0. Only W_gate and W_up get proxies.
  R4  Activations for the integer proxy product: per group of 128, sx = fp32(max|x_hat|)/127
      (binary32), qx = clamp(rint(x_hat / sx), -127, 127), qx = 0 when sx == 0. The pages
      never mention this step; integer accumulation needs integer activations.
  R5  A[g, j] = sum_{i in g} qx_i q[j, i] exactly; g_t[j] = sum_g (sx_g sw[g, j]) A[g, j]
      (each term is exact in fp64, summed over g in order); same for u_t.
  R6  Salience sigma_j = |SiLU(g_t[j]) * u_t[j]|, SiLU(z) = z / (1 + exp(-z)).
  R7  Mask: the k channels with the largest sigma, equal values to the lower index, given
      as ascending indices.
  R8  Stage 2: for j in the mask, g_j and u_j from the bf16 weights and the dense x;
      s_j = SiLU(g_j) u_j; y = sum_j s_j W_down[:, j].
  R9  A batch is a set of independent tokens, each with its own input set and mask.

What pins each function (tests/test_oracle_pins.py; no pin re-types the formula):
  k_for                  values fixed by the workload shapes; clamping; monotonicity.
  quantize_weight_proxy  exact-rational re-derivation over all bf16 of a binade; error and
                         symmetry bounds; lossless on weights that are int4 x 2^e.
  select_inputs          torch.topk on distinct magnitudes; brute force with ties.
  quantize_activations   exact-rational re-derivation; error bound; lossless on int8 x 2^e.
  proxy_accumulators     pure-Python loops on small shapes.
  proxy_salience,
  channel_mask           lossless construction: the quantized pipeline equals a torch fp64
                         SwiGLU and torch.topk; brute force over all C(F, k) masks.
  stage2_exact, ffn      sparsity 0 equals the dense torch fp64 SwiGLU FFN; any mask equals
                         the dense FFN with s multiplied by that 0/1 mask.
  batch_union            brute-force set union.
  rmsnorm                closed form of the mean square.
  proxy_storage_bytes    the pages' ~12% proxy memory overhead (tests/golden).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

GROUP = 128
Q_W_MAX = 7      # int4 symmetric range [-7, 7]    (reading R3)
Q_X_MAX = 127    # int8 symmetric range [-127, 127] (reading R4)


def k_for(sparsity: float, n: int) -> int:
    """Number of items kept at a given sparsity (reading R1)."""
    k = math.floor((1.0 - float(sparsity)) * n + 0.5)
    return int(min(max(k, 1), n))


def silu(z: np.ndarray) -> np.ndarray:
    """SiLU(z) = z * sigmoid(z) in fp64 (the SwiGLU gate activation)."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


# --------------------------------------------------------------------------------------
# Stage 1 -- "Input Sparsity & Quantization"
# --------------------------------------------------------------------------------------

def quantize_weight_proxy(w: np.ndarray, group: int = GROUP):
    """INT4 proxy of one projection [Prox, technical summary, Stage 1, "Input Sparsity &
    Quantization": quantized proxy weights (INT4) for the up and gate projections].

    w: [F, d] bf16 values held exactly in fp32 (nn.Linear layout, row j = channel j).
    Returns (q [F, d] int8 in [-7, 7], sw [G, F] float16), reading R3.
    """
    w = np.asarray(w, dtype=np.float32)
    F, d = w.shape
    if d % group:
        raise ValueError("d must be a multiple of the group size")
    G = d // group
    wg = w.reshape(F, G, group)
    a = np.max(np.abs(wg), axis=2)                        # exact
    sw16 = (a / np.float32(7.0)).astype(np.float16)       # binary32 divide, RNE to binary16
    sw = sw16.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.rint(wg / sw[:, :, None])                  # binary32 divide, ties to even
    q = np.clip(r, -Q_W_MAX, Q_W_MAX)
    q = np.where(sw[:, :, None] == 0, 0.0, q)
    return q.astype(np.int8).reshape(F, d), np.ascontiguousarray(sw16.T)


def select_inputs(x: np.ndarray, k_in: int) -> np.ndarray:
    """Input sparsity [Stage 1, "Input Sparsity & Quantization": input sparsity on the FFN
    input x]: ascending indices of the k_in largest |x_i|, ties to the lower index (R2)."""
    x = np.asarray(x)
    d = x.shape[0]
    mag = np.abs(x.astype(np.float64))
    order = np.lexsort((np.arange(d), -mag))
    return np.sort(order[:k_in]).astype(np.int64)


def quantize_activations(x: np.ndarray, kept: np.ndarray, group: int = GROUP):
    """int8 per-group codes of the sparse input x_hat (reading R4).

    Returns (qx [d] int32, sx [G] float32). Entries outside `kept` are zero.
    """
    x = np.asarray(x, dtype=np.float32)
    d = x.shape[0]
    G = d // group
    xh = np.zeros(d, np.float32)
    xh[kept] = x[kept]
    xg = xh.reshape(G, group)
    b = np.max(np.abs(xg), axis=1)
    sx = (b / np.float32(127.0)).astype(np.float32)      # binary32 divide
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.rint(xg / sx[:, None])                     # binary32 divide, ties to even
    qx = np.clip(r, -Q_X_MAX, Q_X_MAX)
    qx = np.where(sx[:, None] == 0, 0.0, qx)
    return qx.astype(np.int32).reshape(d), sx


def proxy_accumulators(qx: np.ndarray, q: np.ndarray, group: int = GROUP) -> np.ndarray:
    """Integer proxy projection per group: A[g, j] = sum_{i in g} qx_i q[j, i] (exact int64)
    [Stage 1, "Proxy Activation": proxy activations from the quantized weights and the
    sparse input]. Rejected inputs have qx_i = 0 and add nothing."""
    F, d = q.shape
    G = d // group
    A = np.empty((G, F), np.int64)
    qx64 = np.asarray(qx, dtype=np.int64)
    for g in range(G):
        sl = slice(g * group, (g + 1) * group)
        A[g] = q[:, sl].astype(np.int64) @ qx64[sl]
    if A.size and np.abs(A).max() > group * Q_X_MAX * Q_W_MAX:
        raise AssertionError("accumulator out of the int32 design range")
    return A


def proxy_salience(A_gate, A_up, sx, sw_gate, sw_up):
    """Proxy activations and salience [Stage 1, "Proxy Activation" and "Mask Generation":
    s_t = u_t (.) h_t, ranked by magnitude]. Readings R5, R6.

    Returns (sigma [F], g_t [F], u_t [F]) in fp64.
    """
    G, F = A_gate.shape
    g_t = np.zeros(F, np.float64)
    u_t = np.zeros(F, np.float64)
    for g in range(G):
        sxg = np.float64(sx[g])
        g_t = g_t + (sxg * sw_gate[g].astype(np.float64)) * A_gate[g].astype(np.float64)
        u_t = u_t + (sxg * sw_up[g].astype(np.float64)) * A_up[g].astype(np.float64)
    sigma = np.abs(silu(g_t) * u_t)
    return sigma, g_t, u_t


def channel_mask(sigma: np.ndarray, k: int) -> np.ndarray:
    """Shared channel mask m_s [Stage 1, "Mask Generation"; abstract: the mask is built from
    the magnitude ranking of the intermediate state's entries]: ascending indices of the k
    largest sigma, equal values to the lower index (R7)."""
    sigma = np.asarray(sigma, dtype=np.float64)
    F = sigma.shape[0]
    order = np.lexsort((np.arange(F), -sigma))
    return np.sort(order[:k]).astype(np.int64)


# --------------------------------------------------------------------------------------
# Stage 2 -- "Exact Sparse Computation"
# --------------------------------------------------------------------------------------

def stage2_exact(x, w_gate, w_up, w_down, idx):
    """Exact sparse FFN over the masked channels [Stage 2: "Exact Projections" with the
    original full-precision weights; "Final Output": the down projection sparsified by the
    same mask]. Reading R8. Returns (y [d] fp64, s [k] fp64)."""
    x64 = np.asarray(x, dtype=np.float64)
    idx = np.asarray(idx, dtype=np.int64)
    g = np.asarray(w_gate, dtype=np.float64)[idx] @ x64
    u = np.asarray(w_up, dtype=np.float64)[idx] @ x64
    s = silu(g) * u
    y = np.asarray(w_down, dtype=np.float64)[:, idx] @ s
    return y, s


def dense_ffn(x, w_gate, w_up, w_down) -> np.ndarray:
    """Dense SwiGLU FFN y = W_down (SiLU(W_gate x) * (W_up x)) [technical summary, "Problem
    Statement": s = u (.) h], fp64."""
    x64 = np.asarray(x, dtype=np.float64)
    g = np.asarray(w_gate, dtype=np.float64) @ x64
    u = np.asarray(w_up, dtype=np.float64) @ x64
    return np.asarray(w_down, dtype=np.float64) @ (silu(g) * u)


# --------------------------------------------------------------------------------------
# Whole path
# --------------------------------------------------------------------------------------

@dataclass
class OracleLayer:
    """Weights of one layer as exact fp32 copies of the bf16 values, plus the proxies."""
    w_gate: np.ndarray   # [F, d]
    w_up: np.ndarray     # [F, d]
    w_down: np.ndarray   # [d, F]
    q_gate: np.ndarray   # [F, d] int8
    q_up: np.ndarray     # [F, d] int8
    sw_gate: np.ndarray  # [G, F] float16
    sw_up: np.ndarray    # [G, F] float16
    group: int = GROUP

    @property
    def d_model(self) -> int:
        return self.w_gate.shape[1]

    @property
    def d_ff(self) -> int:
        return self.w_gate.shape[0]


def prepare_layer(w_gate, w_up, w_down, group: int = GROUP) -> OracleLayer:
    """Offline step: build the INT4 proxies of W_gate and W_up (W_down gets none)."""
    w_gate = np.ascontiguousarray(w_gate, dtype=np.float32)
    w_up = np.ascontiguousarray(w_up, dtype=np.float32)
    w_down = np.ascontiguousarray(w_down, dtype=np.float32)
    q_g, sw_g = quantize_weight_proxy(w_gate, group)
    q_u, sw_u = quantize_weight_proxy(w_up, group)
    return OracleLayer(w_gate, w_up, w_down, q_g, q_u, sw_g, sw_u, group)


def stage1_token(layer: OracleLayer, x, input_sparsity: float) -> dict:
    """Stage 1 for one token up to the salience (R2 .. R6)."""
    d = layer.d_model
    k_in = k_for(input_sparsity, d)
    kept = select_inputs(x, k_in)
    qx, sx = quantize_activations(x, kept, layer.group)
    A_g = proxy_accumulators(qx, layer.q_gate, layer.group)
    A_u = proxy_accumulators(qx, layer.q_up, layer.group)
    sigma, g_t, u_t = proxy_salience(A_g, A_u, sx, layer.sw_gate, layer.sw_up)
    return dict(k_in=k_in, kept=kept, qx=qx, sx=sx, A_gate=A_g, A_up=A_u,
                sigma=sigma, g_t=g_t, u_t=u_t)


def ffn_token(layer: OracleLayer, x, sparsity: float, input_sparsity: float) -> dict:
    """Prox forward for one token: Stage 1 mask, then exact Stage 2 over it.

    At sparsity 0 every channel is kept and Stage 1 does not change the result.
    """
    F = layer.d_ff
    k = k_for(sparsity, F)
    out = stage1_token(layer, x, input_sparsity)
    idx = channel_mask(out["sigma"], k) if k < F else np.arange(F, dtype=np.int64)
    y, s = stage2_exact(x, layer.w_gate, layer.w_up, layer.w_down, idx)
    out.update(k=k, idx=idx, y=y, s=s)
    return out


def ffn_batch(layer: OracleLayer, X, sparsity: float, input_sparsity: float) -> list[dict]:
    """A batch of independent tokens (R9): each token has its own inputs and mask."""
    return [ffn_token(layer, X[b], sparsity, input_sparsity) for b in range(len(X))]


def batch_union(idx_list, n: int):
    """Union of per-token channel sets as an ascending list, plus membership bits[b][u]."""
    sets = [set(int(v) for v in np.asarray(ix).ravel()) for ix in idx_list]
    U = np.array(sorted(set().union(*sets)) if sets else [], dtype=np.int64)
    bits = np.array([[int(u) in s for u in U] for s in sets], dtype=bool).reshape(len(sets), len(U))
    if len(U) and (U.min() < 0 or U.max() >= n):
        raise ValueError("channel index out of range")
    return U, bits


def rmsnorm(y, eps: float = 1e-6) -> np.ndarray:
    """Unit-gain RMSNorm between stacked layers: y / sqrt(mean(y^2) + eps), fp64."""
    y = np.asarray(y, dtype=np.float64)
    return y / np.sqrt(np.mean(y * y, axis=-1, keepdims=True) + eps)


def proxy_storage_bytes(d_model: int, d_ff: int, group: int = GROUP) -> int:
    """Bytes of the Stage-1 proxies of one layer: int4 codes of W_gate and W_up (one byte per
    (input, channel) pair for both) plus their fp16 group scales."""
    G = d_model // group
    return d_model * d_ff + 2 * G * d_ff * 2
