"""The library's int8 converter (colibri_quantize_int8_block64, host code, no
GPU) against the oracle's quantiser: codes, scales and zero points must agree
bit for bit (a float decides each integer, and both sides decide it in double
precision from the float32 scale).  Also its argument checks."""

import ctypes

import numpy as np
import pytest
import torch

import oracle.quant as oq


@pytest.fixture(scope="module")
def sef():
    from sparse_expert_ffn_gb300 import build
    build.build()
    import sparse_expert_ffn_gb300
    return sparse_expert_ffn_gb300


def _cases():
    g = torch.Generator().manual_seed(4)
    w = torch.randn(256, 448, generator=g) * 0.05
    w[:64, :64] *= 40.0                       # an outlier block
    w[64:128, 64:128] = 0.0                   # a block of zeros
    w[128:192, :64] = w[128:192, :64].abs()   # all non-negative
    w[192:256, 64:128] = -w[192:256, 64:128].abs() - 0.3   # all negative, away from 0
    w[0:64, 128:192] = 0.25                   # constant block
    k = torch.arange(64 * 64, dtype=torch.float64).reshape(64, 64) % 255
    w[64:128, 192:256] = ((k - 127) / 100.0).float()   # on a 0.01 grid: many exact halves
    return w


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_converter_matches_the_oracle_bit_for_bit(sef, dtype):
    w = _cases().to(dtype)
    q, s, z = sef.quantize_int8_block64(w)
    q2, s2, z2 = oq.quantize_int8_block64(w.double().numpy())
    assert np.array_equal(q.numpy(), q2)
    assert np.array_equal(s.numpy(), s2)
    assert np.array_equal(z.numpy(), z2)


def test_converter_stack_and_threads(sef):
    # a matrix large enough to be split over host threads, as an expert stack
    g = torch.Generator().manual_seed(7)
    w = (torch.randn(2, 1024, 1408, generator=g) * 0.02).to(torch.bfloat16)
    q, s, z = sef.quantize_int8_block64(w)
    assert q.shape == (2, 1024, 1408) and s.shape == (2, 16, 22) and z.shape == (2, 16, 22)
    q2, s2, z2 = oq.quantize_experts(w.double().numpy())
    assert np.array_equal(q.numpy(), q2) and np.array_equal(s.numpy(), s2)
    assert np.array_equal(z.numpy(), z2)


def test_converter_rejects_bad_arguments(sef):
    w = torch.zeros(64, 128)
    q = torch.empty(64, 128, dtype=torch.int8)
    s = torch.empty(1, 2)
    z = torch.empty(1, 2, dtype=torch.int32)
    f = sef.colibri_quantize_int8_block64
    P = lambda t: t.data_ptr()  # noqa: E731
    assert f(P(w), sef.DTYPE_FP32, 64, 128, P(q), P(s), P(z)) == sef.OK
    assert f(P(w), sef.DTYPE_FP32, 64, 100, P(q), P(s), P(z)) == sef.ERR_INVALID_ARG
    assert f(P(w), sef.DTYPE_FP32, 0, 128, P(q), P(s), P(z)) == sef.ERR_INVALID_ARG
    assert f(None, sef.DTYPE_FP32, 64, 128, P(q), P(s), P(z)) == sef.ERR_INVALID_ARG
    assert f(P(w), 7, 64, 128, P(q), P(s), P(z)) == sef.ERR_INVALID_ARG
    w[3, 5] = float("nan")
    assert f(P(w), sef.DTYPE_FP32, 64, 128, P(q), P(s), P(z)) == sef.ERR_INVALID_ARG


def test_init_int8_rejects_bad_arguments(sef):
    cfg = sef.ColibriConfig(8, 2, 128, 256, 16, sef.DTYPE_FP32, 0, sef.EXEC_AUTO)
    h = ctypes.c_void_p(123)
    iw = sef.ColibriInt8Weights(None, None, None)
    # NULL int8 parts are rejected before any CUDA call, and *out is cleared
    st = sef.colibri_init_int8(ctypes.byref(cfg), ctypes.c_void_p(1), None, None, None, None, 1,
                               ctypes.byref(h))
    assert st == sef.ERR_INVALID_ARG and not h.value
    st = sef.colibri_init_int8(ctypes.byref(cfg), ctypes.c_void_p(1), None, ctypes.byref(iw),
                               ctypes.byref(iw), ctypes.byref(iw), 1, ctypes.byref(h))
    assert st == sef.ERR_INVALID_ARG and not h.value
