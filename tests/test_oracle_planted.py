"""Plant plausible mistakes in the oracle (on the CPU) and check a pin catches each.

If one of these passes, the pins are too weak to trust the oracle.
"""

import numpy as np
import pytest

import oracle
import oracle.moe as om
import test_oracle_pins as pins


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
