"""prox_sparse_ffn_noalloc, the entry point that allocates nothing, against prox_sparse_ffn.

Some callers cannot give the library a workspace: they run where device allocation is not
allowed or not affordable (a serving runtime that reserved all device memory for its own
pool, a latency-critical loop that cannot take cudaMalloc's implicit synchronization). For
them the library keeps the Stage-2 scratch in a fixed device array of its own. These tests
call that entry point through the C ABI twice in a row, with different inputs each time, and
check every output against the workspace entry point and against the oracle's exact Stage 2
over the same mask, within the Stage-2 tolerance. Batches larger than one token tile (6 and 9
tokens at d_model 1024, tiles of 4) run several tiles one after another through the same
shared array. A request larger than the fixed array must be refused before anything is
launched.
"""
import ctypes

import pytest
import torch

import oracle as O
import workloads as WL
import free_sparse_swiglu_stage1_b300 as P
from free_sparse_swiglu_stage1_b300 import _lib
from gpu_helpers import check_y, cuda, random_layer, ws_for

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d,F,batch", [(1024, 2816, 1), (4096, 1024, 1), (1024, 2816, 2),
                                       (1024, 2816, 6), (1024, 2816, 9)])
def test_noalloc_matches_workspace_entry_point(d, F, batch):
    lay = random_layer(d, F, seed=d + F + batch)
    ws = ws_for(lay, batch)
    L = _lib.lib()
    stream = torch.cuda.current_stream().cuda_stream
    k = P.prox_k_for(0.7, F)
    for call in range(2):
        x = cuda(WL.make_random_tokens(batch, d, seed=900 + call))
        idx = P.prox_build_mask(lay.packed, x, 0.7, 0.5, ws)
        y_ref = P.prox_sparse_ffn(lay.packed, x, idx, ws)
        y = torch.full_like(y_ref, float("nan"))
        status = ctypes.c_int(-99)
        rc = L.prox_sparse_ffn_noalloc(lay.packed.ref, x.data_ptr(), batch, idx.data_ptr(), k,
                                       y.data_ptr(), ctypes.byref(status), stream)
        assert rc == 0, P.prox_error_string(rc)
        assert status.value == 0, P.prox_error_string(status.value)
        got, ref = y.cpu().numpy(), y_ref.cpu().numpy()
        xh, idxh = x.cpu().numpy(), idx.cpu().numpy()
        for b in range(batch):
            check_y(got[b], ref[b])
            y_o, _ = O.stage2_exact(xh[b], lay.o.w_gate, lay.o.w_up, lay.o.w_down, idxh[b])
            check_y(got[b], y_o)
    assert P.prox_get_status(ws) == 0


def test_noalloc_refuses_requests_beyond_its_scratch():
    # two tokens of d_model 8192 need SMs * 2 * 8192 * 4 bytes of partial sums, over 8 MiB
    L = _lib.lib()
    stream = torch.cuda.current_stream().cuda_stream
    buf = torch.empty(256, dtype=torch.uint8, device="cuda")
    desc = _lib.prox_packed()
    desc.d_model, desc.d_ff, desc.group = 8192, 28672, 128
    desc.base = buf.data_ptr()
    desc.bytes = P.prox_packed_bytes(8192, 28672)
    x = torch.zeros((2, 8192), device="cuda")
    y = torch.empty_like(x)
    idx = torch.zeros((2, 4), dtype=torch.int32, device="cuda")
    rc = L.prox_sparse_ffn_noalloc(ctypes.byref(desc), x.data_ptr(), 2, idx.data_ptr(), 4,
                                   y.data_ptr(), None, stream)
    assert rc == -2, P.prox_error_string(rc)
