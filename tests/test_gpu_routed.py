"""colibri_forward_routed: the layer with the caller's routing.

* Routing that the router would never produce: k = 3 experts per token drawn
  at random (a token may pick one expert twice) with gates that do not sum
  to 1.  Checked against the oracle's sum_j g_j FFN_{e_j}(x) at a
  decode size (weights-on-M GEMMs), a prefill size (CTA-pair tiles) and one
  above the one-CTA dispatch (three-launch dispatch); sampled tokens at
  the largest.
* Expert ids out of range: pass 1 of the dispatch reports them (colibri_check
  returns COLIBRI_ERR_CUDA, then the status is clear again), and the pair adds
  nothing; every other pair is unaffected."""

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import Y_RTOL, Case

pytestmark = pytest.mark.gpu

SHAPE = synth.LayerShape("routed", 512, 1024, 8, 2, "bf16")
# d_model 4096: gate/up as well as down run as weights-as-M CTA-pair GEMMs
WIDE = synth.LayerShape("routed_wide", 4096, 1024, 8, 2, "bf16")


def _routing(T, k, E, seed):
    g = torch.Generator().manual_seed(seed)
    idx = torch.randint(0, E, (T, k), generator=g, dtype=torch.int32)
    w = torch.rand((T, k), generator=g, dtype=torch.float32) + 0.05
    return idx, w


def _check(case, x64, y, idx, w, tokens, keep=None):
    tok = np.asarray(tokens)
    ref = oracle.token_outputs(x64[tok], idx[tok], w[tok].astype(np.float64), case.experts,
                               keep_rows=None if keep is None else keep[tok])
    got = oracle.to_f64(y[torch.as_tensor(tok, device=y.device)].cpu())
    err = np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30)
    assert err <= Y_RTOL["bf16"], f"max|err|/max|ref| = {err:.3e}"


@pytest.mark.parametrize("T", [5, 400, 7000])
def test_caller_routing_matches_the_oracle(lib, T):
    k = 3
    # the handle takes max_tokens * top_k pairs
    case = Case(SHAPE, seed=31, max_tokens=(T * k + SHAPE.top_k - 1) // SHAPE.top_k)
    try:
        x, x64 = case.tokens(T)
        idx, w = _routing(T, k, SHAPE.n_experts, 100 + T)
        y = case.layer.forward_routed(x, idx.to(case.dev), w.to(case.dev))
        torch.cuda.synchronize()
        assert case.layer.check() == 0
        tokens = np.arange(T) if T <= 400 else np.unique(np.concatenate(
            [np.arange(64), np.random.default_rng(T).integers(0, T, 192), [T - 1]]))
        _check(case, x64, y, idx.numpy(), w.numpy(), tokens)
        y2 = case.layer.forward_routed(x, idx.to(case.dev), w.to(case.dev))
        assert torch.equal(y, y2)
    finally:
        case.close()


@pytest.mark.parametrize("T", [40, 1100])
def test_out_of_range_ids_are_reported_and_add_nothing(lib, T):
    import sparse_expert_ffn_gb300 as sef
    k, E = 2, SHAPE.n_experts
    case = Case(SHAPE, seed=32, max_tokens=T)
    try:
        x, x64 = case.tokens(T)
        idx, w = _routing(T, k, E, 200 + T)
        bad = torch.zeros((T, k), dtype=torch.bool)
        bad[3, 1] = bad[T // 2, 0] = bad[T - 1, 1] = True
        idx_bad = idx.clone()
        idx_bad[3, 1], idx_bad[T // 2, 0], idx_bad[T - 1, 1] = E, -3, E + 100
        y = case.layer.forward_routed(x, idx_bad.to(case.dev), w.to(case.dev))
        torch.cuda.synchronize()
        assert case.layer.check() == sef.ERR_CUDA
        assert case.layer.check() == 0
        # the bad pairs' ids replaced by a valid one, kept out by the mask
        _check(case, x64, y, idx.numpy(), w.numpy(), np.arange(T), keep=~bad.numpy())
        # a valid call afterwards
        y2 = case.layer.forward_routed(x, idx.to(case.dev), w.to(case.dev))
        torch.cuda.synchronize()
        assert case.layer.check() == 0
        _check(case, x64, y2, idx.numpy(), w.numpy(), np.arange(T))
    finally:
        case.close()


def test_weights_as_m_token_boxes_of_every_width(lib):
    """Caller routing that gives each expert's last 256-row tile a different
    width (17, 49, ..., 241 rows: 32, 64, ..., 256 token columns), so the
    weights-as-M pair GEMMs load that tile's token rows through each of the
    eight box heights (16 .. 128 rows per CTA); experts 0, 3 and 6 also get
    a full tile first.  Every row against the oracle."""
    counts = [32 * j + 17 + (256 if j % 3 == 0 else 0) for j in range(8)]
    T = sum(counts)   # 1800 pairs: CTA-pair tiles (at least 128 per expert on average)
    case = Case(WIDE, seed=41, max_tokens=T)
    try:
        x, x64 = case.tokens(T)
        g = torch.Generator().manual_seed(7)
        idx = torch.repeat_interleave(torch.arange(8, dtype=torch.int32), torch.tensor(counts))
        idx = idx[torch.randperm(T, generator=g)].reshape(T, 1)
        w = torch.rand((T, 1), generator=g, dtype=torch.float32) + 0.05
        y = case.layer.forward_routed(x, idx.to(case.dev), w.to(case.dev))
        torch.cuda.synchronize()
        assert case.layer.check() == 0
        _check(case, x64, y, idx.numpy(), w.numpy(), np.arange(T))
    finally:
        case.close()
