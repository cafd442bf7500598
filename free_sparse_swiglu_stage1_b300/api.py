"""Python binding of the Prox C ABI with the same names as include/prox.h.

Argument marshalling only: torch tensors supply device memory and streams, and every step
of the computation runs in libprox.so's kernels. Tensors must be contiguous; x and y are
fp32 [batch, d_model], weights bf16 in nn.Linear layout, masks int32 [batch, k].
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _lib
from ._lib import ProxError, prox_cost_model, prox_packed

GROUP = 128
MAX_BATCH = 16      # tokens per tile (one pass of the batch kernels)
MAX_TOKENS = 1024   # tokens per call; larger calls run tile by tile


def _stream(stream, device) -> int:
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t: torch.Tensor, dtype: torch.dtype, name: str, ndim: int | None = None) -> int:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions")
    return t.data_ptr()


FORMAT_BF16 = 0
FORMAT_FP8 = 1


def prox_packed_bytes(d_model: int, d_ff: int, group: int = GROUP) -> int:
    return int(_lib.lib().prox_packed_bytes(d_model, d_ff, group))


def prox_packed_bytes_fp8(d_model: int, d_ff: int, group: int = GROUP) -> int:
    return int(_lib.lib().prox_packed_bytes_fp8(d_model, d_ff, group))


def prox_workspace_bytes(d_model: int, d_ff: int, batch: int) -> int:
    return int(_lib.lib().prox_workspace_bytes(d_model, d_ff, batch))


def prox_k_for(sparsity: float, n: int) -> int:
    return int(_lib.lib().prox_k_for(float(sparsity), int(n)))


def prox_cost_model_bytes(d_model: int, d_ff: int) -> prox_cost_model:
    """The HBM-byte cost model of a layer shape (see include/prox.h)."""
    out = prox_cost_model()
    _lib.check(_lib.lib().prox_cost_model_bytes(d_model, d_ff, ctypes.byref(out)),
               "prox_cost_model_bytes")
    return out


def prox_cost_model_fit(k_in, k, t, dense_t: float, min_cost: float = 1e-9) -> prox_cost_model:
    """The cost model t = in_cost k_in + fixed_cost + ch_cost k fitted to measured times."""
    n = len(t)
    if len(k_in) != n or len(k) != n:
        raise ValueError("k_in, k and t must have the same length")
    arr = lambda v: (ctypes.c_double * max(n, 1))(*[float(x) for x in v])
    out = prox_cost_model()
    _lib.check(_lib.lib().prox_cost_model_fit(arr(k_in), arr(k), arr(t), n, float(dense_t),
                                              float(min_cost), ctypes.byref(out)),
               "prox_cost_model_fit")
    return out


def prox_choose_sparsity(cost: prox_cost_model, d_model: int, d_ff: int, target: float,
                         anchor: float = 0.7, min_input_kept: float = 0.3):
    """(input_sparsity, sparsity, effective_sparsity) for a target effective sparsity."""
    s1, s2, eff = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    _lib.check(_lib.lib().prox_choose_sparsity(ctypes.byref(cost), d_model, d_ff, float(target),
                                               float(anchor), float(min_input_kept),
                                               ctypes.byref(s1), ctypes.byref(s2),
                                               ctypes.byref(eff)), "prox_choose_sparsity")
    return s1.value, s2.value, eff.value


@dataclass
class PackedLayer:
    """A packed layer: the device buffer and its C descriptor."""
    buffer: torch.Tensor
    desc: prox_packed
    d_model: int
    d_ff: int

    @property
    def ref(self):
        return ctypes.byref(self.desc)


@dataclass
class Workspace:
    buffer: torch.Tensor
    d_model: int
    d_ff: int
    batch: int

    @property
    def ptr(self) -> int:
        return self.buffer.data_ptr()

    @property
    def nbytes(self) -> int:
        return self.buffer.numel()


def prox_workspace(d_model: int, d_ff: int, batch: int, device=None, stream=None) -> Workspace:
    """Allocates (torch) and initialises a workspace for calls up to this shape."""
    device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(device):
        n = prox_workspace_bytes(d_model, d_ff, batch)
        if n == 0:
            raise ValueError("invalid shape for a workspace")
        buf = torch.empty(n, dtype=torch.uint8, device=device)
        ws = Workspace(buf, d_model, d_ff, batch)
        prox_workspace_init(ws, stream)
    return ws


def prox_workspace_init(ws: Workspace, stream=None) -> None:
    _lib.check(_lib.lib().prox_workspace_init(ws.ptr, ws.nbytes, _stream(stream, ws.buffer.device)),
               "prox_workspace_init")


def prox_pack_weights(w_gate: torch.Tensor, w_up: torch.Tensor, w_down: torch.Tensor,
                      group: int = GROUP, stream=None, fp8: bool = False) -> PackedLayer:
    """Packs one layer; with fp8 the Stage-2 rows are kept as FP8 E4M3 with row scales
    (prox_pack_weights_fp8)."""
    F, d = w_gate.shape
    if tuple(w_up.shape) != (F, d) or tuple(w_down.shape) != (d, F):
        raise ValueError("expected w_gate, w_up [d_ff, d_model] and w_down [d_model, d_ff]")
    pg = _dev(w_gate, torch.bfloat16, "w_gate", 2)
    pu = _dev(w_up, torch.bfloat16, "w_up", 2)
    pd = _dev(w_down, torch.bfloat16, "w_down", 2)
    n = (prox_packed_bytes_fp8 if fp8 else prox_packed_bytes)(d, F, group)
    if n == 0:
        raise ValueError(f"unsupported layer shape d_model={d}, d_ff={F}")
    buf = torch.empty(n, dtype=torch.uint8, device=w_gate.device)
    desc = prox_packed()
    name = "prox_pack_weights_fp8" if fp8 else "prox_pack_weights"
    _lib.check(getattr(_lib.lib(), name)(pg, pu, pd, d, F, group, buf.data_ptr(), n,
                                         _stream(stream, w_gate.device), ctypes.byref(desc)), name)
    return PackedLayer(buf, desc, d, F)


def prox_proxy_bytes(d_model: int, d_ff: int, group: int = GROUP) -> int:
    return int(_lib.lib().prox_proxy_bytes(d_model, d_ff, group))


def prox_rows_bytes(d_model: int, d_ff: int, group: int = GROUP, fp8: bool = False) -> int:
    return int(_lib.lib().prox_rows_bytes(d_model, d_ff, group, FORMAT_FP8 if fp8 else FORMAT_BF16))


@dataclass
class SplitLayer(PackedLayer):
    """A packed layer split into device-resident rows (buffer) and its proxy (proxy_buffer:
    pinned host memory, or device memory)."""
    proxy_buffer: torch.Tensor | None = None


def prox_split_packed(layer: PackedLayer, proxy_on_host: bool = True, stream=None) -> SplitLayer:
    """Copies the layer's rows to a device buffer of their own and its proxy to pinned host
    memory (or, with proxy_on_host=False, to a device buffer); waits for the copies, so the
    full packed buffer may be dropped afterwards."""
    d, F = layer.d_model, layer.d_ff
    fp8 = layer.desc.format == FORMAT_FP8
    rb, pb = prox_rows_bytes(d, F, fp8=fp8), prox_proxy_bytes(d, F)
    dev = layer.buffer.device
    rows = torch.empty(rb, dtype=torch.uint8, device=dev)
    proxy = (torch.empty(pb, dtype=torch.uint8, pin_memory=True) if proxy_on_host
             else torch.empty(pb, dtype=torch.uint8, device=dev))
    desc = prox_packed()
    st = _stream(stream, dev)
    _lib.check(_lib.lib().prox_split_packed(layer.ref, rows.data_ptr(), rb, proxy.data_ptr(), pb, st,
                                            ctypes.byref(desc)), "prox_split_packed")
    torch.cuda.current_stream(dev).synchronize() if stream is None else stream.synchronize()
    return SplitLayer(rows, desc, d, F, proxy)


class ProxyWindow:
    """A sliding window of n_slots device-resident proxies over a stack of split layers
    (prox_window_*). Usage per layer visit: window.acquire(l) -> a descriptor whose proxy
    points at the slot; run the layer's calls; window.release(l)."""

    def __init__(self, layers: list[SplitLayer], n_slots: int, device=None):
        if not layers:
            raise ValueError("a window needs at least one layer")
        d, F = layers[0].d_model, layers[0].d_ff
        if any((l.d_model, l.d_ff) != (d, F) for l in layers):
            raise ValueError("every layer of a window has one shape")
        if any(l.proxy_buffer is None or l.proxy_buffer.is_cuda for l in layers):
            raise ValueError("the layers' proxies must be in host memory")
        self.layers = layers
        self.device = torch.device(device) if device is not None else layers[0].buffer.device
        pb = prox_proxy_bytes(d, F)
        self.slots = torch.empty(n_slots * pb, dtype=torch.uint8, device=self.device)
        ptrs = (ctypes.c_void_p * len(layers))(*[l.proxy_buffer.data_ptr() for l in layers])
        self._handle = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            _lib.check(_lib.lib().prox_window_create(len(layers), n_slots, d, F, ptrs,
                                                     self.slots.data_ptr(), self.slots.numel(),
                                                     ctypes.byref(self._handle)),
                       "prox_window_create")
        self._descs = [prox_packed.from_buffer_copy(l.desc) for l in layers]

    def acquire(self, layer: int, stream=None) -> PackedLayer:
        desc = self._descs[layer]
        _lib.check(_lib.lib().prox_window_acquire(self._handle, layer, ctypes.byref(desc),
                                                  _stream(stream, self.device)),
                   "prox_window_acquire")
        src = self.layers[layer]
        return PackedLayer(src.buffer, desc, src.d_model, src.d_ff)

    def release(self, layer: int, stream=None) -> None:
        _lib.check(_lib.lib().prox_window_release(self._handle, layer, _stream(stream, self.device)),
                   "prox_window_release")

    def stats(self) -> tuple[int, int]:
        c, b = ctypes.c_uint64(), ctypes.c_uint64()
        _lib.check(_lib.lib().prox_window_stats(self._handle, ctypes.byref(c), ctypes.byref(b)),
                   "prox_window_stats")
        return int(c.value), int(b.value)

    def close(self) -> None:
        if self._handle:
            _lib.lib().prox_window_destroy(self._handle)
            self._handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def prox_debug_window_plan(n_layers: int, n_slots: int, ops: list[int], copy_cap: int = 4096):
    """The window's slot policy on the host alone: (slot per op, [(op, slot, layer)] copies)."""
    n = len(ops)
    arr = (ctypes.c_int * max(n, 1))(*ops)
    slots = (ctypes.c_int * max(n, 1))()
    log = (ctypes.c_int * (3 * max(copy_cap, 1)))()
    nc = ctypes.c_int()
    _lib.check(_lib.lib().prox_debug_window_plan(n_layers, n_slots, arr, n, slots, log, copy_cap,
                                                 ctypes.byref(nc)), "prox_debug_window_plan")
    copies = [(log[3 * i], log[3 * i + 1], log[3 * i + 2]) for i in range(min(nc.value, copy_cap))]
    return list(slots)[:n], copies, nc.value


def _x(layer: PackedLayer, x: torch.Tensor) -> tuple[int, int]:
    if x.dim() == 1:
        x = x.view(1, -1)
    if x.shape[1] != layer.d_model:
        raise ValueError("x must be [batch, d_model]")
    return _dev(x, torch.float32, "x", 2), x.shape[0]


def prox_build_mask(layer: PackedLayer, x: torch.Tensor, sparsity: float, input_sparsity: float,
                    ws: Workspace, idx_out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    px, B = _x(layer, x)
    k = prox_k_for(sparsity, layer.d_ff)
    if idx_out is None:
        idx_out = torch.empty((B, k), dtype=torch.int32, device=x.device)
    _dev(idx_out, torch.int32, "idx_out")
    if idx_out.numel() != B * k:
        raise ValueError(f"idx_out must hold [batch, {k}]")
    _lib.check(_lib.lib().prox_build_mask(layer.ref, px, B, float(sparsity), float(input_sparsity),
                                          idx_out.data_ptr(), ws.ptr, ws.nbytes,
                                          _stream(stream, x.device)), "prox_build_mask")
    return idx_out


def prox_sparse_ffn(layer: PackedLayer, x: torch.Tensor, idx: torch.Tensor, ws: Workspace,
                    y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    px, B = _x(layer, x)
    if idx.dim() == 1:
        idx = idx.view(1, -1)
    pi = _dev(idx, torch.int32, "idx", 2)
    if idx.shape[0] != B:
        raise ValueError("idx must be [batch, k]")
    if y is None:
        y = torch.empty((B, layer.d_model), dtype=torch.float32, device=x.device)
    py = _dev(y, torch.float32, "y")
    _lib.check(_lib.lib().prox_sparse_ffn(layer.ref, px, B, pi, idx.shape[1], py, ws.ptr, ws.nbytes,
                                          _stream(stream, x.device)), "prox_sparse_ffn")
    return y


def prox_sparse_ffn_noalloc(layer: PackedLayer, x: torch.Tensor, idx: torch.Tensor,
                            y: torch.Tensor | None = None, stream=None,
                            wait_status: bool = False) -> torch.Tensor:
    """prox_sparse_ffn with the library's own fixed device scratch instead of a workspace
    (for callers that cannot allocate one). With wait_status, waits and raises on a device
    error."""
    px, B = _x(layer, x)
    if idx.dim() == 1:
        idx = idx.view(1, -1)
    pi = _dev(idx, torch.int32, "idx", 2)
    if idx.shape[0] != B:
        raise ValueError("idx must be [batch, k]")
    if y is None:
        y = torch.empty((B, layer.d_model), dtype=torch.float32, device=x.device)
    py = _dev(y, torch.float32, "y")
    st = ctypes.c_int(0)
    _lib.check(_lib.lib().prox_sparse_ffn_noalloc(layer.ref, px, B, pi, idx.shape[1], py,
                                                  ctypes.byref(st) if wait_status else None,
                                                  _stream(stream, x.device)),
               "prox_sparse_ffn_noalloc")
    _lib.check(st.value, "prox_sparse_ffn_noalloc (device status)")
    return y


def prox_ffn_forward(layer: PackedLayer, x: torch.Tensor, sparsity: float, input_sparsity: float,
                     ws: Workspace, y: torch.Tensor | None = None,
                     idx_out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    px, B = _x(layer, x)
    if y is None:
        y = torch.empty((B, layer.d_model), dtype=torch.float32, device=x.device)
    py = _dev(y, torch.float32, "y")
    pi = None
    if idx_out is not None:
        pi = _dev(idx_out, torch.int32, "idx_out")
        if idx_out.numel() != B * prox_k_for(sparsity, layer.d_ff):
            raise ValueError("idx_out must hold [batch, k]")
    _lib.check(_lib.lib().prox_ffn_forward(layer.ref, px, B, float(sparsity), float(input_sparsity),
                                           py, pi, ws.ptr, ws.nbytes, _stream(stream, x.device)),
               "prox_ffn_forward")
    return y


def prox_ffn_forward_host(layer: PackedLayer, x_host: torch.Tensor, sparsity: float,
                          input_sparsity: float, ws: Workspace,
                          y_host: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Host fp32 input and output (pinned memory recommended); waits for completion."""
    if x_host.is_cuda or x_host.dtype != torch.float32 or not x_host.is_contiguous():
        raise ValueError("x_host must be a contiguous fp32 CPU tensor")
    xh = x_host.view(-1, layer.d_model)
    B = xh.shape[0]
    if y_host is None:
        y_host = torch.empty((B, layer.d_model), dtype=torch.float32, pin_memory=True)
    if y_host.is_cuda or y_host.dtype != torch.float32 or not y_host.is_contiguous():
        raise ValueError("y_host must be a contiguous fp32 CPU tensor")
    _lib.check(_lib.lib().prox_ffn_forward_host(layer.ref, xh.data_ptr(), B, float(sparsity),
                                                float(input_sparsity), y_host.data_ptr(), ws.ptr,
                                                ws.nbytes, _stream(stream, ws.buffer.device)),
               "prox_ffn_forward_host")
    return y_host


def prox_dense_ffn(layer: PackedLayer, x: torch.Tensor, ws: Workspace,
                   y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    px, B = _x(layer, x)
    if y is None:
        y = torch.empty((B, layer.d_model), dtype=torch.float32, device=x.device)
    py = _dev(y, torch.float32, "y")
    _lib.check(_lib.lib().prox_dense_ffn(layer.ref, px, B, py, ws.ptr, ws.nbytes,
                                         _stream(stream, x.device)), "prox_dense_ffn")
    return y


def prox_rmsnorm(y: torch.Tensor, eps: float = 1e-6, out: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
    if y.dim() == 1:
        y = y.view(1, -1)
    py = _dev(y, torch.float32, "y", 2)
    if out is None:
        out = torch.empty_like(y)
    po = _dev(out, torch.float32, "out")
    _lib.check(_lib.lib().prox_rmsnorm(py, po, y.shape[0], y.shape[1], float(eps),
                                       _stream(stream, y.device)), "prox_rmsnorm")
    return out


def prox_get_status(ws: Workspace, stream=None) -> int:
    return int(_lib.lib().prox_get_status(ws.ptr, _stream(stream, ws.buffer.device)))


def prox_launch_count() -> int:
    """Kernel launches the library has enqueued in this process (graph captures count once)."""
    return int(_lib.lib().prox_launch_count())


def prox_error_string(code: int) -> str:
    return _lib.error_string(code)


def prox_debug_stage1(layer: PackedLayer, x: torch.Tensor, input_sparsity: float, ws: Workspace,
                      stream=None) -> dict:
    """Integer intermediates of Stage 1: qx [B,d] int8, sx [B,G] fp32, acc_gate / acc_up
    [B,G,F] int32 and the salience [B,F] fp32."""
    px, B = _x(layer, x)
    d, F = layer.d_model, layer.d_ff
    G = d // GROUP
    dev = x.device
    out = {"qx": torch.empty((B, d), dtype=torch.int8, device=dev),
           "sx": torch.empty((B, G), dtype=torch.float32, device=dev),
           "acc_gate": torch.empty((B, G, F), dtype=torch.int32, device=dev),
           "acc_up": torch.empty((B, G, F), dtype=torch.int32, device=dev),
           "salience": torch.empty((B, F), dtype=torch.float32, device=dev)}
    _lib.check(_lib.lib().prox_debug_stage1(
        layer.ref, px, B, float(input_sparsity), out["qx"].data_ptr(), out["sx"].data_ptr(),
        out["acc_gate"].data_ptr(), out["acc_up"].data_ptr(), out["salience"].data_ptr(), ws.ptr,
        ws.nbytes, _stream(stream, dev)), "prox_debug_stage1")
    return out


def prox_debug_fused_forward(layer: PackedLayer, x: torch.Tensor, sparsity: float,
                             input_sparsity: float, ws: Workspace, stream=None):
    """(y [1, d], selected channels [k]) of the single-token path whose Stage 2 selects its
    channels itself; the channels come as the sure ones then the boundary winners."""
    px, B = _x(layer, x)
    if B != 1:
        raise ValueError("one token")
    k = prox_k_for(sparsity, layer.d_ff)
    y = torch.empty((1, layer.d_model), dtype=torch.float32, device=x.device)
    sel = torch.full((k,), -1, dtype=torch.int32, device=x.device)
    _lib.check(_lib.lib().prox_debug_fused_forward(layer.ref, px, float(sparsity),
                                                   float(input_sparsity), y.data_ptr(),
                                                   sel.data_ptr(), ws.ptr, ws.nbytes,
                                                   _stream(stream, x.device)),
               "prox_debug_fused_forward")
    return y, sel


def prox_debug_union(idx: torch.Tensor, d_ff: int, ws: Workspace, stream=None):
    """(union [n] int32, bits [n] uint32-as-int32) of the rows of idx [batch, k]."""
    pi = _dev(idx, torch.int32, "idx", 2)
    B, k = idx.shape
    dev = idx.device
    u = torch.empty(d_ff, dtype=torch.int32, device=dev)
    bits = torch.empty(d_ff, dtype=torch.int32, device=dev)
    cnt = torch.zeros(1, dtype=torch.int32, device=dev)
    _lib.check(_lib.lib().prox_debug_union(pi, B, k, d_ff, u.data_ptr(), bits.data_ptr(),
                                           cnt.data_ptr(), ws.ptr, ws.nbytes, _stream(stream, dev)),
               "prox_debug_union")
    n = int(cnt.item())
    return u[:n], bits[:n]


def prox_debug_wait_timeout(ws: Workspace, spin_cycles: int, stream=None) -> None:
    _lib.check(_lib.lib().prox_debug_wait_timeout(ws.ptr, ws.nbytes, int(spin_cycles),
                                                  _stream(stream, ws.buffer.device)),
               "prox_debug_wait_timeout")


__all__ = [
    "GROUP", "MAX_BATCH", "MAX_TOKENS", "ProxyWindow", "SplitLayer", "prox_proxy_bytes",
    "prox_rows_bytes", "prox_split_packed", "prox_debug_window_plan", "prox_cost_model_fit", "PackedLayer", "ProxError", "Workspace", "prox_build_mask",
    "prox_choose_sparsity", "prox_cost_model", "prox_cost_model_bytes",
    "prox_debug_fused_forward", "prox_debug_stage1", "prox_debug_union", "prox_debug_wait_timeout", "prox_dense_ffn",
    "prox_error_string", "prox_ffn_forward", "prox_ffn_forward_host", "prox_get_status",
    "prox_launch_count", "prox_packed_bytes_fp8", "FORMAT_BF16", "FORMAT_FP8",
    "prox_k_for", "prox_pack_weights", "prox_packed_bytes", "prox_rmsnorm", "prox_sparse_ffn",
    "prox_sparse_ffn_noalloc",
    "prox_workspace", "prox_workspace_bytes", "prox_workspace_init",
]
