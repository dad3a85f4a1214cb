"""Plant plausible mistakes in the oracle (on the CPU) and check a pin catches each.

If one of these passes, the pins are too weak to trust the oracle.
"""

import numpy as np
import pytest

import oracle
import oracle.moe as om
import oracle.quant as oq
import test_oracle_pins as pins
import test_oracle_quant as qpins


def _wrong_silu(z):                       # sign slip: z / (1 + e^z)
    return z / (1.0 + np.exp(z))


def _sigmoid_only(z):                     # dropped factor: sigmoid(z) instead of z*sigmoid(z)
    return 1.0 / (1.0 + np.exp(-z))


def _softmax_all_experts(l, idx):         # softmax over every expert, then pick the k
    e = np.exp(l - l.max(axis=1, keepdims=True))
    full = e / e.sum(axis=1, keepdims=True)
    return np.take_along_axis(full, idx.astype(np.int64), axis=1)


def _topk_high_index_ties(l, k):          # ties to the highest index
    T, E = l.shape
    out = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        row = np.where(np.isnan(l[t]), -np.inf, l[t])
        order = np.lexsort((-np.arange(E), -row))
        out[t] = order[:k]
    return out


def _topk_ascending(l, k):                # the k smallest
    return om.__dict__["_orig_topk"](-l, k)


def _combine_reversed(y_perm, g, inv, keep=None):    # gates applied to the wrong slot
    return om.__dict__["_orig_combine"](y_perm, g[:, ::-1].copy(), inv, keep)


def _dispatch_unstable(idx, E):           # pairs of one expert in decreasing r
    counts, offsets, perm, inv = om.__dict__["_orig_dispatch"](idx, E)
    perm = perm.copy()
    for e in range(E):
        perm[offsets[e]:offsets[e + 1]] = perm[offsets[e]:offsets[e + 1]][::-1]
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size)
    return counts, offsets, perm, inv


def _up_transposed(xs, wg, wu, wd, round_h=False):   # gate and up swapped
    h = om.silu(xs @ wu) * (xs @ wg)
    return h @ wd


def _capacity_last_C(idx, E, capacity=None):   # keeps the last C pairs of an expert
    keep = om.__dict__["_orig_capacity_keep"](idx[::-1], E, capacity)
    return keep[::-1].copy()


def _soft_uniform(l):                     # every expert weighted 1/E
    T, E = l.shape
    return np.tile(np.arange(E, dtype=np.int32), (T, 1)), np.full((T, E), 1.0 / E)


def _soft_top2_only(l):                   # softmax over the two largest, zeros elsewhere
    T, E = l.shape
    idx = np.tile(np.arange(E, dtype=np.int32), (T, 1))
    g = np.zeros((T, E))
    for t in range(T):
        top = np.argsort(-l[t])[:2]
        ex = np.exp(l[t, top] - l[t, top].max())
        g[t, top] = ex / ex.sum()
    return idx, g


def _rmsnorm_no_mean(h, gamma, eps):      # sum instead of mean
    return h / np.sqrt(np.sum(h * h, axis=1, keepdims=True) + eps) * gamma[None, :]


CASES = [
    ("silu", _wrong_silu, [pins.test_one_expert_k1_equals_dense_swiglu, pins.test_silu_values]),
    ("silu", _sigmoid_only, [pins.test_one_expert_k1_equals_dense_swiglu]),
    ("softmax_selected", _softmax_all_experts, [pins.test_softmax_k2_is_sigmoid_of_difference,
                                                pins.test_hand_worked_example]),
    ("topk_select", _topk_high_index_ties, [lambda: pins.test_topk_matches_brute_force(8, 2),
                                            pins.test_hand_worked_example]),
    ("topk_select", _topk_ascending, [pins.test_topk_tiny_config_all_pairs,
                                      pins.test_k1_any_E_equals_dense_ffn_of_argmax_expert]),
    ("combine", _combine_reversed, [pins.test_hand_worked_example,
                                    pins.test_layer_equals_tokenwise_sum]),
    ("dispatch", _dispatch_unstable, [lambda: pins.test_dispatch_invariants_and_brute_force(37, 8, 2)]),
    ("swiglu_expert", _up_transposed, [pins.test_one_expert_k1_equals_dense_swiglu,
                                       pins.test_hand_worked_example]),
    ("rmsnorm", _rmsnorm_no_mean, [pins.test_rmsnorm_closed_forms]),
    ("soft_route", _soft_uniform, [pins.test_soft_route_gates_are_the_full_softmax,
                                   pins.test_soft_layer_is_the_dense_mixture_of_all_experts]),
    ("soft_route", _soft_top2_only, [pins.test_soft_route_gates_are_the_full_softmax,
                                     pins.test_soft_layer_is_the_dense_mixture_of_all_experts]),
    ("capacity_keep", _capacity_last_C,
     [lambda: pins.test_capacity_keep_is_the_first_C_of_each_expert_segment(40, 8, 2, 3)]),
]


@pytest.mark.parametrize("name,bad,checks", CASES, ids=[f"{c[0]}-{c[1].__name__}" for c in CASES])
def test_planted_mistake_is_caught(monkeypatch, name, bad, checks):
    for orig in ("topk_select", "combine", "dispatch", "capacity_keep"):
        monkeypatch.setitem(om.__dict__, "_orig_" + orig.replace("_select", ""), getattr(om, orig))
    monkeypatch.setattr(om, name, bad)
    monkeypatch.setattr(oracle, name, bad)
    for check in checks:
        with pytest.raises(AssertionError):
            check()


# ---------------------------------------------------------------- int8 quantiser


def _quant_variant(levels=254, widen=True, per_matrix=False, rounding=np.rint):
    """A block quantiser with one plausible mistake switched on."""
    def quant(w):
        w = np.asarray(w, dtype=np.float64)
        R, C = w.shape
        if R % 64 or C % 64:
            raise ValueError("ragged")
        q = np.empty((R, C), np.int8)
        s = np.empty((R // 64, C // 64), np.float32)
        z = np.empty((R // 64, C // 64), np.int32)
        for bi in range(R // 64):
            for bj in range(C // 64):
                blk = w[bi * 64:(bi + 1) * 64, bj * 64:(bj + 1) * 64]
                src = w if per_matrix else blk
                lo, hi = float(src.min()), float(src.max())
                if widen:
                    lo, hi = min(lo, 0.0), max(hi, 0.0)
                s32 = np.float32(1.0) if hi == lo else np.float32((hi - lo) / levels)
                zz = 0 if hi == lo else int(rounding(-127 - lo / np.float64(s32)))
                q[bi * 64:(bi + 1) * 64, bj * 64:(bj + 1) * 64] = np.clip(
                    rounding(blk / np.float64(s32)) + zz, -127, 127).astype(np.int8)
                s[bi, bj], z[bi, bj] = s32, zz
        return q, s, z
    return quant


def _dequant_plus_zp(q, scale, zp):        # sign slip on the zero point
    return oq.__dict__["_orig_dequantize_int8_block64"](q, scale, -np.asarray(zp))


QUANT_CASES = [
    ("quantize_int8_block64", _quant_variant(levels=255), [qpins.test_worked_block_symmetric_range]),
    ("quantize_int8_block64", _quant_variant(per_matrix=True), [qpins.test_blocks_are_quantised_independently]),
    ("quantize_int8_block64", _quant_variant(widen=False), [qpins.test_all_positive_block_keeps_zero_exact]),
    ("quantize_int8_block64", _quant_variant(rounding=np.floor),
     [qpins.test_codes_are_the_nearest_grid_points_brute_force,
      lambda: qpins.test_half_step_error_bound_and_ranges((128, 192))]),
    ("dequantize_int8_block64", _dequant_plus_zp, [qpins.test_worked_block_positive_range]),
]


@pytest.mark.parametrize("name,bad,checks", QUANT_CASES,
                         ids=[f"{c[0]}-{i}" for i, c in enumerate(QUANT_CASES)])
def test_planted_quantiser_mistake_is_caught(monkeypatch, name, bad, checks):
    monkeypatch.setitem(oq.__dict__, "_orig_dequantize_int8_block64", oq.dequantize_int8_block64)
    monkeypatch.setattr(oq, name, bad)
    for check in checks:
        with pytest.raises(AssertionError):
            check()
