"""Pins of the CPU oracle against what the definitions and mathematics fix.

Nothing here re-types the oracle's formulas: each check comes from another
route (brute force over all subsets, pure-Python loops, closed forms,
invariants, a library routine for a special case, or a hand-worked example).
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _sigmoid(z):
    return 1.0 / (1.0 + math.exp(-z))


def _silu(z):
    return z * _sigmoid(z)


# ---------------------------------------------------------------- bfloat16


def test_bf16_roundtrip_matches_torch_on_fp32_values():
    g = torch.Generator().manual_seed(1)
    v = torch.randn(200000, generator=g) * torch.exp2(torch.randint(-140, 120, (200000,), generator=g).float())
    v = torch.cat([v, torch.tensor([0.0, -0.0, 1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 3.3895e38, -3.3895e38,
                                    2 ** -133, 2 ** -134, 3 * 2 ** -134, float("inf"), float("-inf")])])
    ref = v.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.f64_to_bf16_bits(v.double().numpy())
    assert np.array_equal(got, ref)
    back = oracle.bf16_bits_to_f64(ref)
    assert np.array_equal(back, v.to(torch.bfloat16).double().numpy(), equal_nan=True)


def test_bf16_known_patterns():
    bits = oracle.f64_to_bf16_bits(np.array([1.0, -2.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 0.5]))
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7 -> even (1.0); 1 + 3*2^-8 -> 1 + 2^-6
    assert bits.tolist() == [0x3F80, 0xC000, 0x3F80, 0x3F82, 0x3F00]


def test_bf16_direct_rounding_avoids_double_rounding():
    # 1 + 2^-8 + 2^-30 is above the bf16 tie: float32 would first round it to
    # the tie 1 + 2^-8 and then to 1.0; a single rounding gives 1 + 2^-7.
    assert oracle.f64_to_bf16_bits(np.array([1.0 + 2 ** -8 + 2 ** -30]))[0] == 0x3F81


# ---------------------------------------------------------------- top-k


def _brute_topk(row, k):
    """The k-subset S with every member beating every non-member, in order."""
    E = len(row)

    def beats(a, b):  # a ranks above b
        va, vb = row[a], row[b]
        if math.isnan(va) and math.isnan(vb):
            return a < b
        if math.isnan(va):
            return False
        if math.isnan(vb):
            return True
        return va > vb or (va == vb and a < b)

    for S in itertools.combinations(range(E), k):
        rest = [e for e in range(E) if e not in S]
        if all(beats(a, b) for a in S for b in rest):
            ordered = list(S)
            # insertion order by pairwise comparison (bubble)
            for i in range(k):
                for j in range(k - 1 - i):
                    if beats(ordered[j + 1], ordered[j]):
                        ordered[j], ordered[j + 1] = ordered[j + 1], ordered[j]
            return ordered
    raise AssertionError("no dominating subset")


@pytest.mark.parametrize("E,k", [(8, 2), (8, 1), (6, 4), (5, 5), (12, 3)])
def test_topk_matches_brute_force(E, k):
    rng = np.random.default_rng(E * 10 + k)
    l = rng.standard_normal((60, E))
    l[::7, 1] = l[::7, 3]                        # exact ties
    l[::11, :] = np.round(l[::11, :])            # many ties
    l[5, 2] = -np.inf
    l[6, 0] = np.nan
    l[9, :] = -np.inf
    idx = oracle.topk_select(l, k)
    for t in range(l.shape[0]):
        assert idx[t].tolist() == _brute_topk(l[t].tolist(), k), t


def test_topk_tiny_config_all_pairs():
    shape = synth.TINY
    x = oracle.to_f64(synth.tokens(shape, 16, 0))
    wr = oracle.to_f64(synth.router_weight(shape, 0))
    l = oracle.router_logits(x, wr)
    idx = oracle.topk_select(l, 2)
    for t in range(16):
        best = max(itertools.combinations(range(8), 2), key=lambda p: (l[t, p[0]] + l[t, p[1]], -p[0], -p[1]))
        assert sorted(idx[t].tolist()) == sorted(best)
        assert l[t, idx[t, 0]] >= l[t, idx[t, 1]]


def test_topk_masked_experts_never_selected_when_enough_live():
    E, k = 128, 4
    b = synth.router_offset(synth.DEEPSEEK_MASKED).double().numpy()
    rng = np.random.default_rng(3)
    l = rng.standard_normal((200, E)) + b[None, :]
    idx = oracle.topk_select(l, k)
    assert not np.any(idx % 4 == 3)


# ---------------------------------------------------------------- softmax


def test_softmax_k2_is_sigmoid_of_difference():
    rng = np.random.default_rng(0)
    l = rng.standard_normal((100, 8)) * 3
    idx = oracle.topk_select(l, 2)
    g = oracle.softmax_selected(l, idx)
    for t in range(100):
        a, b = l[t, idx[t, 0]], l[t, idx[t, 1]]
        assert g[t, 0] == pytest.approx(_sigmoid(a - b), rel=1e-15, abs=1e-15)
        assert g[t, 1] == pytest.approx(_sigmoid(b - a), rel=1e-14, abs=1e-15)


def test_softmax_invariants():
    rng = np.random.default_rng(1)
    l = rng.standard_normal((300, 16)) * 5
    for k in (1, 2, 4, 16):
        idx = oracle.topk_select(l, k)
        g = oracle.softmax_selected(l, idx)
        assert np.allclose(g.sum(axis=1), 1.0, atol=1e-15)
        assert np.all(np.diff(g, axis=1) <= 0)         # descending with the logits
        if k == 1:
            assert np.all(g == 1.0)
        if k == 16:                                      # full softmax
            e = np.exp(l - l.max(axis=1, keepdims=True))
            full = e / e.sum(axis=1, keepdims=True)
            assert np.allclose(np.sort(g, axis=1), np.sort(full, axis=1), rtol=1e-13)


def test_softmax_masked_entry_gets_zero_weight():
    l = np.array([[3.0, -np.inf, 1.0]])
    idx = oracle.topk_select(l, 3)
    g = oracle.softmax_selected(l, idx)
    assert idx[0].tolist() == [0, 2, 1]
    assert g[0, 2] == 0.0 and g[0, 0] == pytest.approx(_sigmoid(2.0), rel=1e-15)


# ---------------------------------------------------------------- dispatch


@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (37, 8, 2), (200, 64, 2), (129, 128, 4), (50, 3, 3)])
def test_dispatch_invariants_and_brute_force(T, E, k):
    rng = np.random.default_rng(T + E)
    l = rng.standard_normal((T, E))
    if E == 128:
        l[:, 3::4] = -np.inf
    idx = oracle.topk_select(l, k)
    counts, offsets, perm, inv = oracle.dispatch(idx, E)
    flat = idx.reshape(-1)
    assert counts.sum() == T * k
    assert np.array_equal(np.sort(perm), np.arange(T * k))            # bijection
    assert np.array_equal(inv[perm], np.arange(T * k))
    # brute force: sort (expert, r) pairs with Python's sort
    expected = [r for _, r in sorted((int(flat[r]), r) for r in range(T * k))]
    assert perm.tolist() == expected
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg) > 0)                                   # stable
        assert offsets[e + 1] - offsets[e] == counts[e]
    if E == 128:
        assert np.all(counts[3::4] == 0)


# ---------------------------------------------------------------- expert FFN


def _dense_swiglu_loops(x, wg, wu, wd):
    """Pure-Python triple loops: y[t,c] = sum_n silu(sum_i x wg) * (sum_i x wu) * wd[n,c]."""
    T, d = len(x), len(x[0])
    f = len(wg[0])
    y = [[0.0] * d for _ in range(T)]
    for t in range(T):
        h = []
        for n in range(f):
            g = sum(x[t][i] * wg[i][n] for i in range(d))
            u = sum(x[t][i] * wu[i][n] for i in range(d))
            h.append(_silu(g) * u)
        for c in range(d):
            y[t][c] = sum(h[n] * wd[n][c] for n in range(f))
    return y


def _small_layer(T=6, d=8, f=12, E=4, seed=5):
    shape = synth.LayerShape("t", d, f, E, 2, "fp32")
    p = synth.layer(shape, T, seed)
    return {k: (oracle.to_f64(v) if v is not None else None) for k, v in p.items()}


def test_one_expert_k1_equals_dense_swiglu():
    p = _small_layer(E=1)
    out = oracle.moe_layer(p["x"], p["w_router"], p["w_gate"], p["w_up"], p["w_down"], 1)
    ref = _dense_swiglu_loops(p["x"].tolist(), p["w_gate"][0].tolist(), p["w_up"][0].tolist(),
                              p["w_down"][0].tolist())
    assert np.allclose(out["y"], np.array(ref), rtol=1e-12, atol=1e-13)
    assert np.all(out["topk_w"] == 1.0)


def test_k1_any_E_equals_dense_ffn_of_argmax_expert():
    p = _small_layer(E=4)
    out = oracle.moe_layer(p["x"], p["w_router"], p["w_gate"], p["w_up"], p["w_down"], 1)
    for t in range(p["x"].shape[0]):
        e = int(np.argmax(p["x"][t] @ p["w_router"]))
        ref = _dense_swiglu_loops([p["x"][t].tolist()], p["w_gate"][e].tolist(), p["w_up"][e].tolist(),
                                  p["w_down"][e].tolist())
        assert np.allclose(out["y"][t], ref[0], rtol=1e-12, atol=1e-13)


def test_identical_experts_are_routing_invariant():
    p = _small_layer(E=5)
    for key in ("w_gate", "w_up", "w_down"):
        p[key] = np.repeat(p[key][:1], 5, axis=0)
    dense = _dense_swiglu_loops(p["x"].tolist(), p["w_gate"][0].tolist(), p["w_up"][0].tolist(),
                                p["w_down"][0].tolist())
    for k in (1, 2, 3, 5):
        for off in (None, np.array([0.0, 3.0, -1.0, 0.5, -np.inf])):
            out = oracle.moe_layer(p["x"], p["w_router"], p["w_gate"], p["w_up"], p["w_down"], k, off)
            assert np.allclose(out["y"], np.array(dense), rtol=1e-12, atol=1e-13)


def test_zero_down_projection_and_zero_input_give_zero():
    p = _small_layer()
    out = oracle.moe_layer(p["x"], p["w_router"], p["w_gate"], p["w_up"], np.zeros_like(p["w_down"]), 2)
    assert np.all(out["y"] == 0.0)
    out = oracle.moe_layer(np.zeros_like(p["x"]), p["w_router"], p["w_gate"], p["w_up"], p["w_down"], 2)
    assert np.all(out["y"] == 0.0)
    assert np.all(out["topk_idx"] == np.array([0, 1]))   # all logits 0: lowest indices


def test_silu_values():
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    assert oracle.silu(np.array([1.0]))[0] == pytest.approx(1.0 / (1.0 + math.e ** -1), rel=1e-15)
    assert oracle.silu(np.array([-1.0]))[0] == pytest.approx(-1.0 / (1.0 + math.e), rel=1e-15)
    assert oracle.silu(np.array([40.0]))[0] == pytest.approx(40.0, rel=1e-15)
    assert abs(oracle.silu(np.array([-40.0]))[0]) < 1e-15


def test_relabelling_experts_leaves_output_unchanged():
    p = _small_layer(E=4, T=9)
    out = oracle.moe_layer(p["x"], p["w_router"], p["w_gate"], p["w_up"], p["w_down"], 2)
    sig = np.array([2, 0, 3, 1])
    # expert new_e = old sig[new_e]: permute router columns and expert weights together
    out2 = oracle.moe_layer(p["x"], p["w_router"][:, sig], p["w_gate"][sig], p["w_up"][sig], p["w_down"][sig], 2)
    assert np.allclose(out["y"], out2["y"], rtol=1e-12, atol=1e-14)
    assert np.array_equal(sig[out2["topk_idx"]], out["topk_idx"])


def test_layer_equals_tokenwise_sum():
    p = _small_layer(E=4, T=11)
    out = oracle.moe_layer(p["x"], p["w_router"], p["w_gate"], p["w_up"], p["w_down"], 2)
    y = oracle.token_outputs(p["x"], out["topk_idx"], out["topk_w"],
                             lambda e: (p["w_gate"][e], p["w_up"][e], p["w_down"][e]))
    assert np.allclose(out["y"], y, rtol=1e-13, atol=1e-14)


def test_hand_worked_example():
    with open(os.path.join(GOLDEN, "worked_example.json")) as fh:
        ex = json.load(fh)
    x = np.array(ex["x"])
    out = oracle.moe_layer(x, np.array(ex["w_router"]), np.array(ex["w_gate"]), np.array(ex["w_up"]),
                           np.array(ex["w_down"]), 2)
    assert out["topk_idx"].tolist() == [[2, 1], [2, 0]]
    s1, s2 = _sigmoid(1.0), _sigmoid(2.0)
    assert out["topk_w"][0].tolist() == pytest.approx([s1, 1 - s1], rel=1e-15)
    assert out["topk_w"][1].tolist() == pytest.approx([s2, 1 - s2], rel=1e-15)
    h02 = _silu(1.0) * 2.0
    h01 = _silu(2.0) * 3.0
    y0 = [s1 * h02 + (1 - s1) * h01 * 0.5, -s1 * h02 + (1 - s1) * h01 * 2.0]
    h12 = _silu(2.0) * 2.0
    h10 = _silu(2.0) * 4.0
    y1 = [s2 * h12 + (1 - s2) * h10, -s2 * h12 + (1 - s2) * h10]
    assert out["y"].tolist()[0] == pytest.approx(y0, rel=1e-14)
    assert out["y"].tolist()[1] == pytest.approx(y1, rel=1e-14)
    assert out["counts"].tolist() == [1, 1, 2]
    assert out["perm"].tolist() == [3, 1, 0, 2]
    assert out["inv"].tolist() == [2, 1, 3, 0]


# ---------------------------------------------------------------- RMSNorm / stack


def test_rmsnorm_closed_forms():
    h = np.array([[3.0, 4.0], [1.0, 1.0]])
    u = oracle.rmsnorm(h, np.array([1.0, 2.0]), 0.0)
    # rms of (3,4) is sqrt(12.5)
    assert u[0].tolist() == pytest.approx([3 / math.sqrt(12.5), 8 / math.sqrt(12.5)], rel=1e-15)
    assert u[1].tolist() == pytest.approx([1.0, 2.0], rel=1e-15)
    # scale invariance (eps = 0)
    assert np.allclose(oracle.rmsnorm(h * 7.5, np.ones(2), 0.0), oracle.rmsnorm(h, np.ones(2), 0.0), rtol=1e-15)


def test_stack_layer_with_zero_down_is_identity():
    p = _small_layer(E=4, T=3)
    h = oracle.round_to_bf16(p["x"])
    out = oracle.stack_layer(h, np.ones(h.shape[1]), 1e-5, p["w_router"], p["w_gate"], p["w_up"],
                             np.zeros_like(p["w_down"]), 2)
    assert np.array_equal(out["h_out"], h)


# ---------------------------------------------------------------- near-tie helper


def test_near_tie_flags_exact_ties_only_when_close():
    x = np.array([[1.0, 0.0], [1.0, 0.0]])
    w = np.array([[1.0, 1.0 + 1e-9, 0.0], [0.0, 0.0, 0.0]])
    l = x @ w
    w2 = np.array([[1.0, 0.5, 0.0], [0.0, 0.0, 0.0]])
    assert oracle.near_tie_tokens(x, w, l, 1).tolist() == [True, True]
    assert oracle.near_tie_tokens(x, w2, x @ w2, 1).tolist() == [False, False]


# ---------------------------------------------------------------- capacity (hard)


@pytest.mark.parametrize("T,E,k,C", [(40, 8, 2, 3), (64, 4, 2, 20), (33, 16, 4, 1), (20, 8, 2, 0)])
def test_capacity_keep_is_the_first_C_of_each_expert_segment(T, E, k, C):
    rng = np.random.default_rng(T * C + E)
    l = rng.standard_normal((T, E))
    l[:, 0] += 2.0            # a hot expert that overflows
    idx = oracle.topk_select(l, k)
    keep = oracle.capacity_keep(idx, E, C)
    # second route: the dispatch permutation's segments, first C entries
    counts, offsets, perm, inv = oracle.dispatch(idx, E)
    expect = np.zeros(T * k, dtype=bool)
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        expect[seg[:C]] = True
    assert np.array_equal(keep.reshape(-1), expect)
    kept_per_expert = np.bincount(idx.reshape(-1)[keep.reshape(-1)], minlength=E)
    assert np.all(kept_per_expert == np.minimum(counts, C))


def test_capacity_limits_are_monotone_and_reach_no_limit():
    rng = np.random.default_rng(5)
    idx = oracle.topk_select(rng.standard_normal((50, 6)), 2)
    prev = oracle.capacity_keep(idx, 6, 0)
    assert not prev.any()
    for C in range(1, 60):
        cur = oracle.capacity_keep(idx, 6, C)
        assert np.all(prev <= cur)              # raising C never drops a kept pair
        prev = cur
    counts = np.bincount(idx.reshape(-1), minlength=6)
    assert oracle.capacity_keep(idx, 6, int(counts.max())).all()
    assert oracle.capacity_keep(idx, 6, None).all()


def test_layer_under_capacity_drops_exactly_the_rejected_pairs():
    p = _small_layer(E=4, T=12)
    base = oracle.moe_layer(p["x"], p["w_router"], p["w_gate"], p["w_up"], p["w_down"], 2)
    none = oracle.moe_layer(p["x"], p["w_router"], p["w_gate"], p["w_up"], p["w_down"], 2,
                            capacity=int(base["counts"].max()))
    assert np.array_equal(none["y"], base["y"])
    zero = oracle.moe_layer(p["x"], p["w_router"], p["w_gate"], p["w_up"], p["w_down"], 2, capacity=0)
    assert np.all(zero["y"] == 0.0)
    cap = oracle.moe_layer(p["x"], p["w_router"], p["w_gate"], p["w_up"], p["w_down"], 2, capacity=3)
    # token-wise: sum over the kept slots only, with the unchanged gates
    g = np.where(cap["keep"], cap["topk_w"], 0.0)
    y = oracle.token_outputs(p["x"], cap["topk_idx"], g,
                             lambda e: (p["w_gate"][e], p["w_up"][e], p["w_down"][e]))
    assert np.allclose(cap["y"], y, rtol=1e-13, atol=1e-14)
    assert not np.allclose(cap["y"], base["y"])


# ---------------------------------------------------------------- soft routing


def test_soft_route_gates_are_the_full_softmax():
    rng = np.random.default_rng(21)
    l = rng.standard_normal((6, 5)) * 3.0
    l[2, 4] = -np.inf
    idx, g = oracle.soft_route(l)
    assert idx.shape == (6, 5) and np.all(idx == np.arange(5))
    for t in range(6):
        # closed form per token, by pure-Python exponentials
        den = sum(math.exp(v) for v in l[t] if v != -np.inf)
        for e in range(5):
            want = 0.0 if l[t, e] == -np.inf else math.exp(l[t, e]) / den
            assert abs(g[t, e] - want) <= 1e-14
        # the ratio of two gates is the exponential of the logit difference
        assert abs(g[t, 0] / g[t, 1] - math.exp(l[t, 0] - l[t, 1])) <= 1e-12


def test_soft_layer_is_the_dense_mixture_of_all_experts():
    p = _small_layer(E=4)
    out = oracle.moe_layer(p["x"], p["w_router"], p["w_gate"], p["w_up"], p["w_down"], 4,
                           soft=True)
    assert np.all(out["counts"] == p["x"].shape[0])
    for t in range(p["x"].shape[0]):
        l = [sum(p["x"][t][i] * p["w_router"][i][e] for i in range(p["x"].shape[1]))
             for e in range(4)]
        m = max(l)
        w = [math.exp(v - m) for v in l]
        s = sum(w)
        ref = np.zeros(p["x"].shape[1])
        for e in range(4):
            y_e = _dense_swiglu_loops([p["x"][t].tolist()], p["w_gate"][e].tolist(),
                                      p["w_up"][e].tolist(), p["w_down"][e].tolist())[0]
            ref += (w[e] / s) * np.array(y_e)
        assert np.allclose(out["y"][t], ref, rtol=1e-12, atol=1e-13)


def test_soft_layer_with_one_live_expert_is_k1():
    p = _small_layer(E=4)
    off = np.array([-np.inf, 0.0, -np.inf, -np.inf])
    soft = oracle.moe_layer(p["x"], p["w_router"], p["w_gate"], p["w_up"], p["w_down"], 4, off,
                            soft=True)
    hard = oracle.moe_layer(p["x"], p["w_router"], p["w_gate"], p["w_up"], p["w_down"], 1, off)
    assert np.allclose(soft["y"], hard["y"], rtol=1e-13, atol=1e-14)
    assert np.all(soft["topk_w"][:, 1] == 1.0)


def test_soft_layer_rejects_partial_k():
    p = _small_layer(E=4)
    with pytest.raises(ValueError):
        oracle.moe_layer(p["x"], p["w_router"], p["w_gate"], p["w_up"], p["w_down"], 2, soft=True)
