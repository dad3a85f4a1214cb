"""GPU parity of the routing variants on the Mixtral-shaped layer: top-1,
top-4 and soft routing (top_k == E: every expert, softmax over all E logits,
m.nxbn.cn section 2.2), plus soft routing with 64 experts (Qwen2-shaped)."""

from dataclasses import replace

import numpy as np
import pytest
import torch

import synth
from parity import Case, check_output, check_routing

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", params=[1, 4, 8], ids=["top1", "top4", "soft"])
def mixtral_k(lib, request):
    c = Case(replace(synth.MIXTRAL, top_k=request.param), seed=0, max_tokens=1024)
    yield c
    c.close()


@pytest.mark.parametrize("T", [1, 16, 1024])
@pytest.mark.parametrize("executor", ["grouped", "stream"])
def test_mixtral_routing_variants(mixtral_k, T, executor):
    if executor == "stream" and T > 16:
        pytest.skip("the CUDA-core executor is for decode sizes")
    x, x64 = mixtral_k.tokens(T)
    y, r = mixtral_k.run(x, executor)
    l, _ = check_routing(mixtral_k, x64, r)
    if mixtral_k.shape.top_k == 8:
        assert np.all(r["counts"] == T)
    check_output(mixtral_k, x64, y, r, l)
    y2, _ = mixtral_k.run(x, executor)
    assert torch.equal(y, y2)


def test_qwen_soft_routing_64_experts(lib):
    c = Case(replace(synth.QWEN2, top_k=64), seed=3, max_tokens=64)
    try:
        for T in (1, 64):
            x, x64 = c.tokens(T)
            y, r = c.run(x)
            l, _ = check_routing(c, x64, r)
            assert np.all(r["counts"] == T)
            check_output(c, x64, y, r, l)
    finally:
        c.close()
