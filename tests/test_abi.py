"""The C ABI without a GPU: the library loads, exports every function include/prox.h
declares, and rejects bad arguments on the host before any launch."""
import ctypes

import pytest

import oracle as O
from free_sparse_swiglu_stage1_b300 import _lib

E_ARG, E_WS = -1, -2
FAKE = 1 << 20          # an aligned address that is never dereferenced (validation fails first)


@pytest.fixture(scope="module")
def L():
    return _lib.lib()


def test_exports_every_declared_symbol(L):
    declared = _lib.header_symbols()
    assert len(declared) >= 15
    for name in declared:
        assert hasattr(L, name), name
    assert sorted(_lib.SIGNATURES) == declared


def test_error_strings(L):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert L.prox_error_string(code)
    assert L.prox_error_string(0) == b"ok"


def test_k_rule_matches_oracle(L):
    for n in (1, 7, 1024, 2816, 4096, 11008, 14336, 28672):
        for s in (0.0, 0.1, 0.3, 0.5, 0.6, 0.7, 0.8, 0.9, 0.95, 0.999999):
            assert L.prox_k_for(s, n) == O.k_for(s, n), (s, n)
    assert L.prox_k_for(1.0, 10) == -1
    assert L.prox_k_for(-0.1, 10) == -1
    assert L.prox_k_for(0.5, 0) == -1


def test_packed_bytes(L):
    d, F = 4096, 14336
    n = L.prox_packed_bytes(d, F, 128)
    payload = d * F + (d // 128) * F * 4 + F * 3 * d * 2
    assert payload <= n <= payload + 3 * 256
    assert L.prox_packed_bytes(4000, F, 128) == 0      # d not a multiple of 128
    assert L.prox_packed_bytes(d, F, 64) == 0          # group must be 128
    assert L.prox_packed_bytes(d, 100, 128) == 0       # d_ff not a multiple of 32
    assert L.prox_packed_bytes(32768, F, 128) == 0     # d_model above the limit


def _desc(d=1024, F=2816, base=FAKE, nbytes=None):
    p = _lib.prox_packed()
    p.d_model, p.d_ff, p.group = d, F, 128
    p.base = base
    p.bytes = nbytes if nbytes is not None else (1 << 40)
    return p


def test_forward_rejects_bad_arguments_before_launch(L):
    p = _desc()
    ref = ctypes.byref(p)
    fwd = L.prox_ffn_forward
    assert fwd(None, FAKE, 1, 0.5, 0.5, FAKE, None, FAKE, 1 << 30, None) == E_ARG
    assert fwd(ref, None, 1, 0.5, 0.5, FAKE, None, FAKE, 1 << 30, None) == E_ARG
    assert fwd(ref, FAKE, 0, 0.5, 0.5, FAKE, None, FAKE, 1 << 30, None) == E_ARG
    assert fwd(ref, FAKE, 1025, 0.5, 0.5, FAKE, None, FAKE, 1 << 30, None) == E_ARG
    assert fwd(ref, FAKE, 1, 1.0, 0.5, FAKE, None, FAKE, 1 << 30, None) == E_ARG
    assert fwd(ref, FAKE, 1, 0.5, -0.2, FAKE, None, FAKE, 1 << 30, None) == E_ARG
    assert fwd(ref, FAKE + 4, 1, 0.5, 0.5, FAKE, None, FAKE, 1 << 30, None) == E_ARG
    bad_shape = _desc(d=1000)
    assert fwd(ctypes.byref(bad_shape), FAKE, 1, 0.5, 0.5, FAKE, None, FAKE, 1 << 30, None) == E_ARG
    small = _desc(nbytes=1024)
    assert fwd(ctypes.byref(small), FAKE, 1, 0.5, 0.5, FAKE, None, FAKE, 1 << 30, None) == E_WS
    misaligned = _desc(base=FAKE + 16)
    assert fwd(ctypes.byref(misaligned), FAKE, 1, 0.5, 0.5, FAKE, None, FAKE, 1 << 30, None) == E_WS


def test_other_entry_points_reject_bad_arguments(L):
    p = _desc()
    ref = ctypes.byref(p)
    assert L.prox_build_mask(ref, FAKE, 1, 0.5, 0.5, None, FAKE, 1 << 30, None) == E_ARG
    assert L.prox_sparse_ffn(ref, FAKE, 1, FAKE, 0, FAKE, FAKE, 1 << 30, None) == E_ARG
    assert L.prox_sparse_ffn(ref, FAKE, 1, FAKE, 2817, FAKE, FAKE, 1 << 30, None) == E_ARG
    assert L.prox_dense_ffn(ref, None, 1, FAKE, FAKE, 1 << 30, None) == E_ARG
    assert L.prox_rmsnorm(None, FAKE, 1, 1024, 1e-6, None) == E_ARG
    assert L.prox_rmsnorm(FAKE, FAKE, 1, 1024, -1.0, None) == E_ARG
    out = _lib.prox_packed()
    assert L.prox_pack_weights(None, FAKE, FAKE, 1024, 2816, 128, FAKE, 1 << 30, None,
                               ctypes.byref(out)) == E_ARG
    assert L.prox_pack_weights(FAKE, FAKE, FAKE, 1024, 2816, 64, FAKE, 1 << 30, None,
                               ctypes.byref(out)) == E_ARG
    assert L.prox_pack_weights(FAKE, FAKE, FAKE, 1024, 2816, 128, FAKE, 1024, None,
                               ctypes.byref(out)) == E_WS
    assert L.prox_workspace_init(None, 4096, None) == E_ARG
    assert L.prox_workspace_init(FAKE + 8, 4096, None) == E_WS
    assert L.prox_debug_wait_timeout(None, 4096, 10, None) == E_ARG
    assert L.prox_debug_union(None, 1, 1, 32, FAKE, FAKE, FAKE, FAKE, 4096, None) == E_ARG
    assert L.prox_get_status(None, None) == E_ARG
