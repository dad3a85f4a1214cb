"""Pins of the oracle's int8 block quantiser (oracle/quant.py) against what
the format's definition fixes: worked blocks whose codes follow by hand, the
half-step error bound, nearest-code brute force, block independence, exact
round trips of on-grid weights and the zero block.  None of these re-types
the quantiser's formula."""

import numpy as np
import pytest

import oracle.quant as oq


def _block_from_codes(k):
    """A 64x64 block whose 4096 entries cycle through the integer list k."""
    k = np.asarray(k, dtype=np.float64)
    return np.resize(k, (64, 64))


def test_worked_block_symmetric_range():
    # w = (k - 127) / 100 for k = 0..254: lo = -1.27, hi = 1.27, so the step
    # is 2.54 / 254 = 0.01 and zero sits on code 0.
    k = np.arange(255)
    w = _block_from_codes((k - 127) / 100.0)
    q, s, z = oq.quantize_int8_block64(w)
    assert s.shape == (1, 1) and z.shape == (1, 1)
    assert s[0, 0] == np.float32(0.01)
    assert z[0, 0] == 0
    assert np.array_equal(q, _block_from_codes(k - 127).astype(np.int8))


def test_worked_block_positive_range():
    # w = k / 100 for k = 0..254: lo = 0, hi = 2.54, step 0.01; w = 0 maps to
    # code -127, so the zero point is -127 and code = k - 127.
    k = np.arange(255)
    w = _block_from_codes(k / 100.0)
    q, s, z = oq.quantize_int8_block64(w)
    assert s[0, 0] == np.float32(0.01)
    assert z[0, 0] == -127
    assert np.array_equal(q, _block_from_codes(k - 127).astype(np.int8))
    deq = oq.dequantize_int8_block64(q, s, z)
    assert np.max(np.abs(deq - w)) <= 0.5 * 0.01 * (1 + 1e-4)


def test_all_positive_block_keeps_zero_exact():
    # values in [1, 3.54]: the range is widened to [0, 3.54], zp stays within
    # [-127, 127] and the zero point dequantises to exactly 0
    w = _block_from_codes(1.0 + np.arange(255) / 100.0)
    q, s, z = oq.quantize_int8_block64(w)
    assert -127 <= z[0, 0] <= 127
    assert abs(float(s[0, 0]) - 3.54 / 254) <= 1e-6 * 3.54 / 254
    assert oq.dequantize_int8_block64(np.full((64, 64), z[0, 0], np.int8), s, z).max() == 0.0


@pytest.mark.parametrize("shape", [(64, 64), (128, 192), (192, 64)])
def test_half_step_error_bound_and_ranges(shape):
    rng = np.random.default_rng(11)
    w = rng.standard_normal(shape) * 0.02
    w[:64, :64] *= 50.0                      # one block with a much wider range
    q, s, z = oq.quantize_int8_block64(w)
    assert q.dtype == np.int8 and s.dtype == np.float32 and z.dtype == np.int32
    assert s.shape == (shape[0] // 64, shape[1] // 64)
    assert q.min() >= -127 and q.max() <= 127
    assert z.min() >= -127 and z.max() <= 127
    deq = oq.dequantize_int8_block64(q, s, z)
    # half a step; the float32 rounding of the step can move the clamped
    # extremes by up to 254 * 2**-24 of a step more
    bound = np.repeat(np.repeat(s.astype(np.float64), 64, 0), 64, 1) * 0.5 * (1 + 1e-4)
    assert np.all(np.abs(deq - w) <= bound)
    # every block's own extremes land within half a step
    for bi in range(s.shape[0]):
        for bj in range(s.shape[1]):
            blk = w[bi * 64:(bi + 1) * 64, bj * 64:(bj + 1) * 64]
            step = float(s[bi, bj])
            assert step <= (max(blk.max(), 0) - min(blk.min(), 0)) / 254 * (1 + 1e-6)
    # the wide block has the largest step, by about the factor it was widened
    if s.size > 1:
        assert s[0, 0] == s.max() and s[0, 0] > 20 * np.median(s[s != s[0, 0]])


def test_codes_are_the_nearest_grid_points_brute_force():
    rng = np.random.default_rng(3)
    w = rng.standard_normal((64, 64)) * 0.1 + 0.03
    q, s, z = oq.quantize_int8_block64(w)
    step, zp = float(s[0, 0]), int(z[0, 0])
    grid = (np.arange(-127, 128) - zp) * step            # every representable value
    best = np.abs(w.reshape(-1, 1) - grid.reshape(1, -1)).min(axis=1)
    got = np.abs(w - (q.astype(np.float64) - zp) * step).reshape(-1)
    assert np.allclose(got, best, rtol=0, atol=1e-15)


def test_blocks_are_quantised_independently():
    rng = np.random.default_rng(5)
    w = rng.standard_normal((128, 128))
    q0, s0, z0 = oq.quantize_int8_block64(w)
    w2 = w.copy()
    w2[70, 3] = 40.0                          # block (1, 0) only
    q1, s1, z1 = oq.quantize_int8_block64(w2)
    changed = (s0 != s1) | (z0 != z1)
    assert changed[1, 0] and changed.sum() == 1
    same = np.ones((128, 128), bool)
    same[64:128, 0:64] = False
    assert np.array_equal(q0[same], q1[same])


def test_on_grid_weights_round_trip_exactly():
    rng = np.random.default_rng(9)
    step = np.float32(0.0037)
    for zp in (-127, -40, 0, 55, 127):
        codes = rng.integers(-127, 128, size=(64, 64))
        codes[0, 0], codes[1, 1] = -127, 127      # the block spans the whole code range
        w = (codes - zp) * np.float64(step)
        q, s, z = oq.quantize_int8_block64(w)
        assert s[0, 0] == step and z[0, 0] == zp
        assert np.array_equal(q.astype(np.int64), codes)


def test_zero_block():
    q, s, z = oq.quantize_int8_block64(np.zeros((64, 128)))
    assert np.all(q == 0) and np.all(s == 1.0) and np.all(z == 0)
    assert np.all(oq.dequantize_int8_block64(q, s, z) == 0.0)


def test_rejects_ragged_shapes():
    with pytest.raises(ValueError):
        oq.quantize_int8_block64(np.zeros((64, 100)))
