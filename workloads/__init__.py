"""Seeded synthetic inputs for the Prox sparse SwiGLU FFN decode path.

This module only draws random numbers. It holds none of the method's arithmetic, so the
CPU oracle and the CUDA path can both be fed from it without sharing any code.

The pages measure on trained LLMs (Qwen3, Llama-3, Mistral, Gemma-3) with downstream and
perplexity suites [Prox, technical summary, "Key Contributions" and "Experimental Results"].
Neither the trained weights nor those datasets are available, so seeded synthetic tensors
with the same layer shapes stand in for them. Five workloads are defined:

  1  d=1024, F=2816, W ~ N(0, 0.02^2); x ~ N(0,1) with 1% of entries (seeded positions)
     scaled x20; channel sparsity 0.5, input sparsity 0.5; 64 tokens, batch 1.
  2  Llama-2-7B FFN shape 4096 x 11008; W ~ N(0, 0.02^2) times a per-channel factor
     c_j ~ LogNormal(0, 0.5) applied to W_gate row j, W_up row j and W_down column j;
     x ~ Student-t(nu=4); channel sparsity 0 / 0.5 / 0.7 / 0.9, input sparsity 0.5.
  3  Llama-3-8B FFN shape 4096 x 14336; W ~ N(0, 0.02^2); x ~ Student-t(4); channel
     sparsity 0.7, input sparsity 0.5; batch 1, 2, 4, 8, 16.
  4  32 independently seeded layers of workload 3; 256 consecutive tokens, batch 1.
  5  Llama-2-70B FFN shape 8192 x 28672; W ~ N(0, 0.01^2) times LogNormal(0, 0.5) per
     channel; x ~ Student-t(3); channel sparsity 0.5 / 0.7 / 0.8 / 0.9; batch 1 and 8.

Seeds: layer weights use 1000*workload + layer, tokens use 1_000_000 + 1000*workload + t.
Weights are drawn in fp32 and rounded to bf16 (round to nearest even, done by torch).
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np
import torch

__all__ = [
    "Workload", "WORKLOADS", "layer_seed", "token_seed", "make_layer", "make_tokens",
    "make_random_layer", "make_random_tokens",
]

_CHUNKS = 16  # fixed chunking of every large draw: results never depend on thread count


@dataclass(frozen=True)
class Workload:
    key: int
    name: str
    d_model: int
    d_ff: int
    w_std: float
    channel_lognormal: float | None   # sigma of the per-channel LogNormal(0, sigma) factor
    x_kind: str                       # "normal_outliers" or "student_t"
    x_df: float | None                # Student-t degrees of freedom
    sparsities: tuple[float, ...]
    input_sparsity: float
    batches: tuple[int, ...]
    tokens: int
    layers: int


WORKLOADS: dict[int, Workload] = {
    1: Workload(1, "ffn-1024x2816", 1024, 2816, 0.02, None, "normal_outliers", None,
                (0.5,), 0.5, (1,), 64, 1),
    2: Workload(2, "llama2-7b-ffn-4096x11008", 4096, 11008, 0.02, 0.5, "student_t", 4.0,
                (0.0, 0.5, 0.7, 0.9), 0.5, (1,), 64, 1),
    3: Workload(3, "llama3-8b-ffn-4096x14336", 4096, 14336, 0.02, None, "student_t", 4.0,
                (0.7,), 0.5, (1, 2, 4, 8, 16), 64, 1),
    4: Workload(4, "llama3-8b-ffn-stack32-4096x14336", 4096, 14336, 0.02, None, "student_t",
                4.0, (0.7,), 0.5, (1,), 256, 32),
    5: Workload(5, "llama2-70b-ffn-8192x28672", 8192, 28672, 0.01, 0.5, "student_t", 3.0,
                (0.5, 0.7, 0.8, 0.9), 0.5, (1, 8), 64, 1),
}


def layer_seed(workload: int, layer: int) -> int:
    return 1000 * workload + layer


def token_seed(workload: int, token: int) -> int:
    return 1_000_000 + 1000 * workload + token


def _normal_f32(seed_words: tuple[int, ...], n: int) -> np.ndarray:
    """n standard normals in fp32, drawn in fixed chunks from spawned PCG64 streams."""
    out = np.empty(n, np.float32)
    kids = np.random.SeedSequence(list(seed_words)).spawn(_CHUNKS)
    bounds = [(i * n // _CHUNKS, (i + 1) * n // _CHUNKS) for i in range(_CHUNKS)]

    def fill(i: int) -> None:
        a, b = bounds[i]
        if b > a:
            np.random.Generator(np.random.PCG64(kids[i])).standard_normal(
                out=out[a:b], dtype=np.float32)

    if n >= 1 << 20:
        with ThreadPoolExecutor(max_workers=8) as ex:
            list(ex.map(fill, range(_CHUNKS)))
    else:
        for i in range(_CHUNKS):
            fill(i)
    return out


def make_random_layer(d_model: int, d_ff: int, seed: int, w_std: float = 0.02,
                      channel_lognormal: float | None = None) -> dict[str, torch.Tensor]:
    """One SwiGLU FFN layer in nn.Linear layout, bf16 on the CPU.

    Returns w_gate [F, d], w_up [F, d], w_down [d, F] and, when a per-channel factor is
    drawn, its values as "channel_scale" [F] (fp32, for reference only).
    """
    F, d = d_ff, d_model
    mats = {}
    for mid, name, shape in ((0, "w_gate", (F, d)), (1, "w_up", (F, d)), (2, "w_down", (d, F))):
        z = _normal_f32((seed, mid), math.prod(shape)).reshape(shape)
        z *= np.float32(w_std)
        mats[name] = z
    out: dict[str, torch.Tensor] = {}
    if channel_lognormal is not None:
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 3])))
        c = np.exp(rng.standard_normal(F) * channel_lognormal).astype(np.float32)
        mats["w_gate"] *= c[:, None]
        mats["w_up"] *= c[:, None]
        mats["w_down"] *= c[None, :]
        out["channel_scale"] = torch.from_numpy(c)
    for name in ("w_gate", "w_up", "w_down"):
        out[name] = torch.from_numpy(mats[name]).to(torch.bfloat16)
    return out


def make_layer(workload: int, layer: int = 0) -> dict[str, torch.Tensor]:
    """The seeded layer `layer` of workload `workload` (see the module docstring)."""
    w = WORKLOADS[workload]
    return make_random_layer(w.d_model, w.d_ff, layer_seed(workload, layer), w.w_std,
                             w.channel_lognormal)


def _one_token(w: Workload, seed: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    d = w.d_model
    if w.x_kind == "normal_outliers":
        x = rng.standard_normal(d)
        n_out = max(1, round(0.01 * d))
        pos = rng.choice(d, size=n_out, replace=False)
        x[pos] *= 20.0
    elif w.x_kind == "student_t":
        x = rng.standard_t(w.x_df, size=d)
    else:
        raise ValueError(w.x_kind)
    return x.astype(np.float32)


def make_tokens(workload: int, tokens) -> np.ndarray:
    """FFN inputs x [len(tokens), d] fp32 for the given token numbers of a workload."""
    w = WORKLOADS[workload]
    toks = list(tokens)
    if not toks:
        return np.zeros((0, w.d_model), np.float32)
    return np.stack([_one_token(w, token_seed(workload, t)) for t in toks])


def make_random_tokens(n: int, d_model: int, seed: int, kind: str = "student_t",
                       df: float = 4.0) -> np.ndarray:
    """n seeded fp32 inputs of width d_model for custom (test) shapes."""
    w = Workload(0, "custom", d_model, 0, 0.0, None, kind, df, (), 0.0, (), n, 1)
    return np.stack([_one_token(w, seed * 7919 + t) for t in range(n)]) if n else \
        np.zeros((0, d_model), np.float32)
