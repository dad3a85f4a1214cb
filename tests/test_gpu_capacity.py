"""GPU parity of the hard expert capacity (colibri_set_capacity).

Reading of the pages (cf-1.com sections 2.3 and 4.2, zskr.cn section 2.2): an
expert accepts at most C (token, slot) pairs per batch, in token order then
slot order; the dropped pairs add nothing and the other gates are unchanged.
The oracle's capacity_keep applied to the GPU's own routing decides which
pairs are kept; routing itself (topk_idx, counts, perm) is unaffected."""

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import Case, check_output, check_routing

pytestmark = pytest.mark.gpu


def _run_capped(case, x, x64, capacity, executor, tokens=None):
    case.layer.set_capacity(capacity)
    try:
        y, r = case.run(x, executor)
    finally:
        case.layer.set_capacity(None)
    l, _ = check_routing(case, x64, r)
    err = check_output(case, x64, y, r, l, tokens, capacity=capacity)
    keep = oracle.capacity_keep(r["topk_idx"], case.shape.n_experts, capacity)
    return y, r, keep, err


def test_tiny_fp32_capacity(lib):
    c = Case(synth.TINY, seed=0, max_tokens=64)
    try:
        x, x64 = c.tokens(64)
        for C in (0, 1, 5, 12, 64):
            y, r, keep, _ = _run_capped(c, x, x64, C, "stream")
            assert keep.sum() == np.minimum(r["counts"], C).sum()
            if C == 0:
                assert torch.all(y == 0)
        y_free, _ = c.run(x, "stream")
        y_big, _, _, _ = _run_capped(c, x, x64, 128, "stream")
        assert torch.equal(y_free, y_big)          # a limit above every count changes nothing
    finally:
        c.close()


@pytest.mark.parametrize("T,C", [(512, 6), (512, 40), (2048, 64)])
def test_qwen_zipf_capacity_drops_the_hot_experts_overflow(lib, T, C):
    c = Case(synth.QWEN2, seed=0, max_tokens=2048)
    try:
        x, x64 = c.tokens(T)
        y, r, keep, _ = _run_capped(c, x, x64, C, "grouped")
        assert r["counts"][0] > C                  # Zipf: expert 0 overflows
        assert (~keep).any()
    finally:
        c.close()


@pytest.mark.parametrize("C", [400, 280])
def test_deepseek_capacity_multi_cta_dispatch_and_pairs(lib, C):
    """C = 400: every capped expert's kept rows end 144 rows into its second
    256-row pair tile; C = 280: 24 rows into it (a tile almost all padding)."""
    c = Case(synth.DEEPSEEK, seed=0, max_tokens=16384)
    try:
        x, x64 = c.tokens(16384)
        y, r, keep, _ = _run_capped(c, x, x64, C, "grouped")
        assert (r["counts"] > C).any() and (~keep).any()
        y2, _, _, _ = _run_capped(c, x, x64, C, "grouped", [0, 1])
        assert torch.equal(y, y2)                  # deterministic under capacity too
    finally:
        c.close()


def test_mixtral_capacity_weights_as_m_pairs(lib):
    """Mixtral-shaped T = 4096 (about 1024 pairs per expert) capped at 1000:
    the CTA-pair GEMMs with the weights as the MMA's M operand (gate/up too,
    at d_model 4096) see every capped expert's last tile end 232 rows in."""
    c = Case(synth.MIXTRAL, seed=0, max_tokens=4096)
    try:
        x, x64 = c.tokens(4096)
        y, r, keep, _ = _run_capped(c, x, x64, 1000, "grouped")
        assert (r["counts"] > 1000).any() and (~keep).any()
    finally:
        c.close()


def test_residual_layer_with_capacity_zero_is_identity(lib):
    shape = synth.LayerShape("cap_stack", 512, 1024, 8, 2, "bf16")
    c = Case(shape, seed=4, max_tokens=64)
    try:
        h = synth.tokens(shape, 64, 4, 0, c.dev)
        h0 = h.clone()
        gamma = torch.ones(shape.d_model, dtype=torch.bfloat16, device=c.dev)
        c.layer.set_capacity(0)
        c.layer.forward_stack_layer(h, gamma, 1e-5)
        torch.cuda.synchronize()
        assert c.layer.check() == 0
        assert torch.equal(h, h0)
    finally:
        c.close()
