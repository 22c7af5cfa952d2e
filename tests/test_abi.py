"""CPU checks of the C ABI: the library builds, loads, exports every function
include/tp_api.h declares, and rejects bad arguments on the host with the
documented status codes before any CUDA call (so no GPU is needed)."""
import ctypes

import pytest

import sharded_gemm_gb300 as tp
from sharded_gemm_gb300 import build as tpbuild

FAKE = 0x10000  # a non-null, 16-byte aligned address that is never dereferenced


@pytest.fixture(scope="module")
def L():
    tpbuild.build()
    return tp.lib()


def _arr(n, v=FAKE):
    a = (ctypes.c_void_p * n)(*([v] * n))
    return ctypes.cast(a, ctypes.POINTER(ctypes.c_void_p)), a


def test_exports_every_declared_symbol(L):
    names = tp.declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(L, n), n


def test_launch_count_needs_no_gpu(L):
    n = L.tp_launch_count()
    assert n >= 0 and L.tp_launch_count() == n


def test_version(L):
    assert L.tp_version() >= 100


def test_all_to_sharded_not_divisible_message(L):
    w, k1 = _arr(2)
    y, k2 = _arr(2)
    rc = L.tp_all_to_sharded(2, FAKE, 4, 2, 2, w, 3, None, tp.TP_F32, y, 2, tp.TP_F32, None)
    assert rc == tp.TP_ERR_NOT_DIVISIBLE
    assert tp.tp_last_error() == "Cannot shard the output of size 3 across 2 devices."


def test_all_to_sharded_invalid_args(L):
    w, k1 = _arr(2)
    y, k2 = _arr(2)
    assert L.tp_all_to_sharded(0, FAKE, 4, 2, 2, w, 2, None, 0, y, 1, 0, None) == tp.TP_ERR_INVALID_ARG
    assert L.tp_all_to_sharded(2, None, 4, 2, 2, w, 2, None, 0, y, 1, 0, None) == tp.TP_ERR_INVALID_ARG
    assert L.tp_all_to_sharded(2, FAKE, 4, 2, 1, w, 2, None, 0, y, 1, 0, None) == tp.TP_ERR_INVALID_ARG
    assert L.tp_all_to_sharded(2, FAKE, 4, 2, 2, w, 2, None, 7, y, 1, 0, None) == tp.TP_ERR_INVALID_ARG
    assert L.tp_all_to_sharded(2, FAKE + 1, 4, 2, 2, w, 2, None, tp.TP_F32, y, 1, 0, None) == tp.TP_ERR_ALIGNMENT
    wn, k3 = _arr(2, None)
    assert L.tp_all_to_sharded(2, FAKE, 4, 2, 2, wn, 2, None, 0, y, 1, 0, None) == tp.TP_ERR_INVALID_ARG


def test_empty_batch_launches_nothing(L):
    w, k1 = _arr(2)
    y, k2 = _arr(2)
    assert L.tp_all_to_sharded(2, FAKE, 0, 2, 2, w, 2, None, tp.TP_BF16, y, 1, tp.TP_F32, None) == tp.TP_OK
    x, k3 = _arr(2)
    assert L.tp_sharded_to_all(2, x, 0, 4, 2, w, 3, None, tp.TP_BF16, FAKE, 3, tp.TP_F32, None) == tp.TP_OK


def test_sharded_to_all_not_divisible(L):
    x, k1 = _arr(4)
    w, k2 = _arr(4)
    rc = L.tp_sharded_to_all(4, x, 2, 10, 10, w, 3, None, tp.TP_BF16, FAKE, 3, tp.TP_F32, None)
    assert rc == tp.TP_ERR_NOT_DIVISIBLE


def test_mx_checks(L):
    a, k1 = _arr(4)
    assert L.tp_mx_quantize(FAKE, 4, 48, FAKE, FAKE, None) == tp.TP_ERR_NOT_DIVISIBLE
    assert L.tp_mx_quantize(None, 4, 64, FAKE, FAKE, None) == tp.TP_ERR_INVALID_ARG
    # column-parallel: O % N, K % 32
    assert L.tp_mx_all_to_sharded(4, FAKE, 2, 64, a, a, 10, None, a, 4, tp.TP_F32, None) == tp.TP_ERR_NOT_DIVISIBLE
    assert L.tp_mx_all_to_sharded(4, FAKE, 2, 48, a, a, 8, None, a, 4, tp.TP_F32, None) == tp.TP_ERR_NOT_DIVISIBLE
    # row-parallel: K % N, whole blocks per shard
    assert L.tp_mx_sharded_to_all(4, a, 2, 66, a, a, 8, None, FAKE, 8, tp.TP_F32, None) == tp.TP_ERR_NOT_DIVISIBLE
    assert L.tp_mx_sharded_to_all(4, a, 2, 64, a, a, 8, None, FAKE, 8, tp.TP_F32, None) == tp.TP_ERR_NOT_DIVISIBLE
    assert "whole blocks" in L.tp_last_error().decode()
    assert L.tp_mx_sharded_to_all(4, a, 0, 128, a, a, 8, None, FAKE, 8, tp.TP_F32, None) == tp.TP_OK


def test_backward_checks(L):
    a, k1 = _arr(4)
    # column-parallel dx: O % N, lddy < O/N
    assert L.tp_all_to_sharded_dx(4, a, 2, 10, 10, a, 8, tp.TP_BF16, FAKE, 8, tp.TP_F32, None) == \
        tp.TP_ERR_NOT_DIVISIBLE
    assert L.tp_all_to_sharded_dx(4, a, 2, 8, 1, a, 8, tp.TP_BF16, FAKE, 8, tp.TP_F32, None) == \
        tp.TP_ERR_INVALID_ARG
    # row-parallel dx: K % N
    assert L.tp_sharded_to_all_dx(4, FAKE, 2, 8, 8, a, 10, tp.TP_BF16, a, 8, tp.TP_F32, None) == \
        tp.TP_ERR_NOT_DIVISIBLE
    # weight grads: lddw < K, null shard
    assert L.tp_sharded_dw(4, a, 8, a, 8, 2, 8, 8, tp.TP_BF16, a, 4, tp.TP_F32, None) == tp.TP_ERR_INVALID_ARG
    an, k2 = _arr(4)
    k2[1] = None
    assert L.tp_sharded_dw(4, a, 8, an, 8, 2, 8, 8, tp.TP_BF16, a, 8, tp.TP_F32, None) == tp.TP_ERR_INVALID_ARG
    # bias grads: nout * nin above 64, ld < cols
    b, k3 = _arr(65)
    assert L.tp_bias_grad(5, 13, b, 2, 8, 8, tp.TP_BF16, b, None) == tp.TP_ERR_INVALID_ARG
    assert L.tp_bias_grad(1, 1, b, 2, 8, 4, tp.TP_BF16, b, None) == tp.TP_ERR_INVALID_ARG
    # SUMMA backward and linear: divisibility by q
    s16, k4 = _arr(16)
    for fn in (L.tp_summa_abt, L.tp_summa_atb):
        assert fn(4, s16, s16, s16, 10, 8, 8, tp.TP_BF16, None) == tp.TP_ERR_NOT_DIVISIBLE
    assert L.tp_summa_linear(4, s16, s16, None, s16, 8, 8, 10, tp.TP_BF16, None) == tp.TP_ERR_NOT_DIVISIBLE


def test_gated_checks(L):
    w, k1 = _arr(4)
    y, k2 = _arr(4)
    fn = L.tp_gated_all_to_sharded
    assert fn(4, FAKE, 2, 8, 8, w, w, 10, None, None, tp.TP_BF16, y, 3, tp.TP_BF16, None) == tp.TP_ERR_NOT_DIVISIBLE
    assert "output of size 10 across 4" in L.tp_last_error().decode()
    # ldh below F/N, ldx below K, a null up-projection shard, a null bias entry
    assert fn(4, FAKE, 2, 8, 8, w, w, 8, None, None, tp.TP_BF16, y, 1, tp.TP_BF16, None) == tp.TP_ERR_INVALID_ARG
    assert fn(4, FAKE, 2, 8, 4, w, w, 8, None, None, tp.TP_BF16, y, 2, tp.TP_BF16, None) == tp.TP_ERR_INVALID_ARG
    wn, k3 = _arr(4)
    k3[3] = None
    assert fn(4, FAKE, 2, 8, 8, w, wn, 8, None, None, tp.TP_BF16, y, 2, tp.TP_BF16, None) == tp.TP_ERR_INVALID_ARG
    assert fn(4, FAKE, 2, 8, 8, w, w, 8, wn, None, tp.TP_BF16, y, 2, tp.TP_BF16, None) == tp.TP_ERR_INVALID_ARG
    assert fn(4, FAKE, 0, 8, 8, w, w, 8, None, None, tp.TP_BF16, y, 2, tp.TP_BF16, None) == tp.TP_OK


def test_reduce_scatter_and_gather_checks(L):
    x, k1 = _arr(4)
    w, k2 = _arr(4)
    y, k3 = _arr(4)
    for fn in (L.tp_sharded_to_sharded, L.tp_gathered_to_sharded):
        # K % N and O % N are both required
        assert fn(4, x, 2, 10, 10, w, 8, None, tp.TP_BF16, y, 2, tp.TP_F32, None) == tp.TP_ERR_NOT_DIVISIBLE
        assert "input of size 10 across 4" in L.tp_last_error().decode()
        assert fn(4, x, 2, 8, 8, w, 6, None, tp.TP_BF16, y, 2, tp.TP_F32, None) == tp.TP_ERR_NOT_DIVISIBLE
        assert "output of size 6 across 4" in L.tp_last_error().decode()
        # ldy below O/N, ldx below K/N, null shard pointer, N*N above the part limit
        assert fn(4, x, 2, 8, 2, w, 8, None, tp.TP_BF16, y, 1, tp.TP_F32, None) == tp.TP_ERR_INVALID_ARG
        assert fn(4, x, 2, 8, 1, w, 8, None, tp.TP_BF16, y, 2, tp.TP_F32, None) == tp.TP_ERR_INVALID_ARG
        yn, k4 = _arr(4)
        k4[2] = None
        assert fn(4, x, 2, 8, 2, w, 8, None, tp.TP_BF16, yn, 2, tp.TP_F32, None) == tp.TP_ERR_INVALID_ARG
        x9, k5 = _arr(9)
        assert fn(9, x9, 2, 9, 1, x9, 9, None, tp.TP_BF16, x9, 1, tp.TP_F32, None) == tp.TP_ERR_UNSUPPORTED
        # T = 0 launches nothing and succeeds
        assert fn(4, x, 0, 8, 2, w, 8, None, tp.TP_BF16, y, 2, tp.TP_F32, None) == tp.TP_OK


def test_summa_checks(L):
    b, k = _arr(16)
    assert L.tp_summa(0, b, b, b, 8, 8, 8, tp.TP_BF16, None) == tp.TP_ERR_NOT_DIVISIBLE
    assert L.tp_summa(3, b, b, b, 8, 9, 9, tp.TP_BF16, None) == tp.TP_ERR_NOT_DIVISIBLE
    assert L.tp_summa(5, b, b, b, 10, 10, 10, tp.TP_BF16, None) == tp.TP_ERR_UNSUPPORTED
    assert L.tp_summa(2, None, b, b, 8, 8, 8, tp.TP_BF16, None) == tp.TP_ERR_INVALID_ARG


def test_shard_weight_checks(L):
    s, k = _arr(2)
    assert L.tp_shard_weight(FAKE, 10, 4, 2, 0, 3, 2, s, None) == tp.TP_ERR_NOT_DIVISIBLE
    assert tp.tp_last_error() == "Cannot shard the output of size 10 across 6 devices."
    assert L.tp_shard_weight(FAKE, 8, 4, 3, 0, 1, 2, s, None) == tp.TP_ERR_INVALID_ARG
    assert L.tp_shard_weight(FAKE, 8, 4, 2, 2, 1, 2, s, None) == tp.TP_ERR_INVALID_ARG
    assert L.tp_shard_weight(FAKE, 8, 4, 2, 0, 0, 2, s, None) == tp.TP_ERR_INVALID_ARG
    assert L.tp_shard_weight(FAKE, 8, 4, 2, 0, 1, 65, s, None) == tp.TP_ERR_INVALID_ARG
    assert L.tp_shard_weight(FAKE + 1, 8, 4, 2, 0, 1, 2, s, None) == tp.TP_ERR_ALIGNMENT


def test_q4_checks(L):
    a, k = _arr(8)
    assert L.tp_q4_quantize(FAKE, 4, 128, 32, FAKE, FAKE, FAKE, None) == tp.TP_ERR_UNSUPPORTED
    assert L.tp_q4_quantize(FAKE, 4, 100, 64, FAKE, FAKE, FAKE, None) == tp.TP_ERR_NOT_DIVISIBLE
    assert L.tp_q4_all_to_sharded(8, FAKE, 1, 128, a, a, a, 32, 64, None, a, 8, tp.TP_BF16, None) == tp.TP_ERR_UNSUPPORTED
    assert L.tp_q4_all_to_sharded(8, FAKE, 1, 128, a, a, a, 64, 60, None, a, 8, tp.TP_BF16, None) == tp.TP_ERR_NOT_DIVISIBLE
    # each shard must hold whole groups: K/N = 96 is not a multiple of 64
    assert L.tp_q4_sharded_to_all(8, a, 1, 768, a, a, a, 64, 16, None, FAKE, 16, tp.TP_F32, None) == tp.TP_ERR_NOT_DIVISIBLE


def test_policy_and_wait_limit_checks(L):
    assert L.tp_set_policy(7) == tp.TP_ERR_INVALID_ARG
    assert L.tp_set_policy(tp.TP_POLICY_AUTO) == tp.TP_OK
    assert L.tp_set_wait_limit_ns(10) == tp.TP_ERR_INVALID_ARG
    assert L.tp_set_wait_limit_ns(2_000_000_000) == tp.TP_OK
    assert L.tp_debug_wait_timeout(5, None) == tp.TP_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(tp, "_lib", None)
    monkeypatch.setattr(tp, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        tp.tp_version()
