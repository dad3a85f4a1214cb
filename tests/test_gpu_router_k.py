"""The tensor-core router (batches from 512 tokens) for k that fills its
top-k lists partly or to eight slots.

The router epilogue sorts each token's logits into a list of 1, 2, 4 or 8
slots, the shortest that holds k; k = 3 (a 4-slot list, one slot unused) and
k = 6 (the 8-slot list) run through both of its paths: 600 tokens (5 tiles,
K split into slices, the last slice's warp routes) and 5000 tokens (40
tiles, whole K).  Every token is checked against the oracle."""

import pytest
import torch

import synth
from parity import Case, check_output, check_routing

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("k", [3, 6])
def test_router_top_k_lists(lib, k):
    shape = synth.LayerShape(f"router_k{k}", 256, 256, 16, k, "bf16")
    c = Case(shape, seed=7, max_tokens=5000)
    try:
        for T in (600, 5000):
            x, x64 = c.tokens(T)
            y, r = c.run(x, "grouped")
            assert r["topk_idx"].shape == (T, k)
            l, near = check_routing(c, x64, r)
            assert near.sum() < T // 50
            check_output(c, x64, y, r, l)
            y2, _ = c.run(x, "grouped")
            assert torch.equal(y, y2)
    finally:
        c.close()
