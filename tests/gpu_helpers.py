"""Shared helpers of the GPU parity tests: build a layer for both sides from the seeded
generators, decode the documented packed layout, and the tolerance rules."""
import numpy as np
import torch

import oracle as O
import workloads as WL
import free_sparse_swiglu_stage1_b300 as P

DEV = "cuda"

# Stage-2 tolerance (given the same mask): bf16 weights, fp32 accumulation
Y_MAXERR = 2e-2
Y_RELL2 = 5e-3
# mask tie band: channels whose salience lies within this relative distance of the k-th
# value may be swapped for one another
BAND = 1e-6


class Layer:
    def __init__(self, mats: dict):
        self.mats = mats
        self.dev = {k: v.to(DEV) for k, v in mats.items() if k.startswith("w_")}
        self.packed = P.prox_pack_weights(self.dev["w_gate"], self.dev["w_up"], self.dev["w_down"])
        self.o = O.prepare_layer(*(mats[k].float().numpy() for k in ("w_gate", "w_up", "w_down")))
        self.d, self.F = self.packed.d_model, self.packed.d_ff


def random_layer(d, F, seed, std=0.02, lognormal=None) -> Layer:
    return Layer(WL.make_random_layer(d, F, seed, std, lognormal))


def workload_layer(key, layer=0) -> Layer:
    return Layer(WL.make_layer(key, layer))


def decode_packed(buf: np.ndarray, d: int, F: int) -> dict:
    """Splits a packed buffer by the layout documented in include/prox.h."""
    a = lambda v: (v + 255) // 256 * 256
    G = d // 128
    codes = buf[: d * F].reshape(d, F)
    so = a(d * F)
    scales = buf[so: so + G * F * 4].view(np.uint32).reshape(G, F)
    ro = a(so + G * F * 4)
    rows = buf[ro: ro + F * 3 * d * 2].view(np.uint16).reshape(F, 3, d)
    return {
        "q_gate": (codes & 0xF).astype(np.int16).T - 8,
        "q_up": (codes >> 4).astype(np.int16).T - 8,
        "sw_gate_bits": (scales & 0xFFFF).astype(np.uint16),
        "sw_up_bits": (scales >> 16).astype(np.uint16),
        "rows": rows,
    }


def check_band(sigma: np.ndarray, k: int, idx) -> None:
    """GPU mask vs the oracle salience: exactly k ascending channels, containing every
    channel clearly above the k-th oracle value and none clearly below it. Among the
    channels whose oracle salience equals the k-th value exactly, the ones taken must be the
    lowest indices (the ranking rule gives equal values to the lower channel index)."""
    idx = np.asarray(idx, dtype=np.int64)
    assert len(idx) == k
    assert np.all(np.diff(idx) > 0), "mask not strictly ascending"
    assert idx.min() >= 0 and idx.max() < len(sigma)
    sk = np.sort(sigma)[::-1][k - 1]
    got = set(idx.tolist())
    must = set(np.nonzero(sigma > sk * (1 + BAND))[0].tolist())
    must_not = set(np.nonzero(sigma < sk * (1 - BAND))[0].tolist())
    assert must <= got, f"missing {len(must - got)} channels above the band"
    assert not (must_not & got), f"{len(must_not & got)} channels below the band selected"
    ties = np.nonzero(sigma == sk)[0]          # ascending
    if len(ties) > 1:
        taken = np.array([j in got for j in ties.tolist()])
        n = int(taken.sum())
        assert taken[:n].all() and not taken[n:].any(), \
            "equal saliences not taken lowest index first"


def check_y(y_gpu: np.ndarray, y_ref: np.ndarray) -> None:
    y_gpu = np.asarray(y_gpu, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    scale = np.abs(y_ref).max()
    err = np.abs(y_gpu - y_ref)
    if scale == 0:
        assert err.max() == 0
        return
    assert err.max() <= Y_MAXERR * scale, f"max err {err.max() / scale:.3e} of max|y|"
    rel = np.linalg.norm(y_gpu - y_ref) / np.linalg.norm(y_ref)
    assert rel <= Y_RELL2, f"relative L2 {rel:.3e}"


def ws_for(layer: Layer, batch: int):
    return P.prox_workspace(layer.d, layer.F, batch)


def cuda(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV)
