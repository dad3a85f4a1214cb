"""CTA-pair expert GEMMs (batches averaging at least 128 pairs per expert),
checked on every token.

Zipf-skewed routing over 8 experts gives ragged 256-row tiles of many
lengths (rows past an expert's count belong to the next expert or lie past
the end of the gathered buffer, where TMA reads zeros, and must not be
stored); d_ff = 384 gives an odd number of gate/up n-blocks (three blocks of
128 hidden units) and d_model = 512 two down n-blocks of 256."""

import pytest
import torch

import synth
from parity import Case, check_output, check_routing

pytestmark = pytest.mark.gpu

SHAPE = synth.LayerShape("pair_tiles", 512, 384, 8, 2, "bf16", bias="zipf")
T_MAX = 3000


@pytest.fixture(scope="module")
def case(lib):
    c = Case(SHAPE, seed=4, max_tokens=T_MAX)
    yield c
    c.close()


@pytest.mark.parametrize("T", [512, 777, 1500, T_MAX])
def test_every_token(case, T):
    x, x64 = case.tokens(T)
    y, r = case.run(x, "grouped")
    assert r["counts"].sum() == 2 * T and T * 2 >= 128 * SHAPE.n_experts
    l, _ = check_routing(case, x64, r)
    check_output(case, x64, y, r, l)
    y2, _ = case.run(x, "grouped")
    assert torch.equal(y, y2)
