"""GPU parity of the int8-weight layer (colibri_init_int8, weights converted
by colibri_quantize_int8_block64) on both executors (tcgen05 with shared-
memory dequantisation, and CUDA cores) against the oracle run on its own int8
quantisation of the same weights."""

import numpy as np
import pytest
import torch

import synth
from parity import Int8Case, check_output, check_routing

pytestmark = pytest.mark.gpu


def test_tiny_fp32_int8_ragged():
    c = Int8Case(synth.TINY, seed=0, max_tokens=64)
    try:
        for T in (1, 2, 17, 64):
            x, x64 = c.tokens(T)
            y, r = c.run(x)
            l, _ = check_routing(c, x64, r)
            check_output(c, x64, y, r, l)
    finally:
        c.close()


@pytest.fixture(scope="module")
def mixtral8(lib):
    c = Int8Case(synth.MIXTRAL, seed=0, max_tokens=1024)
    yield c
    c.close()


@pytest.mark.parametrize("T", [1, 2, 3, 4, 8, 16, 128])
@pytest.mark.parametrize("executor", ["grouped", "stream"])
def test_mixtral_int8_decode(mixtral8, T, executor):
    """grouped: TMA-fed int8 stages dequantised in shared memory for tcgen05
    (split-K with the last-slice fixup at these sizes); stream: CUDA cores
    (up to three tokens the int8 GEMV items: one, two or four token rows per
    pass, down projection in K slices; above, the per-row weight stream)."""
    x, x64 = mixtral8.tokens(T)
    y, r = mixtral8.run(x, executor)
    l, _ = check_routing(mixtral8, x64, r)
    check_output(mixtral8, x64, y, r, l)
    y2, _ = mixtral8.run(x, executor)
    assert torch.equal(y, y2)


def test_mixtral_int8_prefill_1024(mixtral8):
    x, x64 = mixtral8.tokens(1024)
    y, r = mixtral8.run(x, "grouped")
    l, _ = check_routing(mixtral8, x64, r)
    check_output(mixtral8, x64, y, r, l)


def test_tiny_fp32_int8_has_no_grouped_executor():
    import sparse_expert_ffn_gb300 as sef
    c = Int8Case(synth.TINY, seed=0, max_tokens=8)
    try:
        with pytest.raises(sef.ColibriError):
            c.layer.set_executor("grouped")
    finally:
        c.close()


def test_qwen_int8_zipf_with_capacity():
    c = Int8Case(synth.QWEN2, seed=1, max_tokens=64)
    try:
        x, x64 = c.tokens(64)
        y, r = c.run(x)
        l, _ = check_routing(c, x64, r)
        check_output(c, x64, y, r, l)
        c.layer.set_capacity(3)
        y, r = c.run(x)
        check_output(c, x64, y, r, l, capacity=3)
    finally:
        c.close()


def test_mixtral_int8_gemv_with_capacity(mixtral8):
    """Three tokens, every expert keeping one pair: the GEMV's tiles hold only
    the kept rows; dropped pairs add nothing in the combine."""
    x, x64 = mixtral8.tokens(3)
    y, r = mixtral8.run(x, "stream")
    l, _ = check_routing(mixtral8, x64, r)
    try:
        mixtral8.layer.set_capacity(1)
        y, r = mixtral8.run(x, "stream")
        check_output(mixtral8, x64, y, r, l, capacity=1)
    finally:
        mixtral8.layer.set_capacity(None)


def test_mixtral_int8_gemv_shared_experts_routed(mixtral8):
    """The caller's routing sends the three tokens to experts 3 and 5 only
    (the last token twice to 3): expert 3 gets four rows and expert 5 two,
    so the GEMV's four-row passes run with every row live and as a two-row
    pass; the output is the oracle's layer at that routing."""
    import oracle
    from parity import Y_RTOL
    x, x64 = mixtral8.tokens(3)
    idx = torch.tensor([[3, 5], [5, 3], [3, 3]], dtype=torch.int32, device=x.device)
    w = torch.tensor([[0.7, 0.3], [0.6, 0.4], [0.5, 0.5]], dtype=torch.float32, device=x.device)
    mixtral8.layer.set_executor("stream")
    y = mixtral8.layer.forward_routed(x, idx, w)
    torch.cuda.synchronize()
    assert mixtral8.layer.check() == 0
    y_ref = oracle.token_outputs(x64, idx.cpu().numpy(), w.double().cpu().numpy(), mixtral8.experts)
    y_gpu = oracle.to_f64(y.cpu())
    err = np.abs(y_gpu - y_ref).max() / np.abs(y_ref).max()
    assert err <= Y_RTOL["bf16"], f"max|err|/max|ref| = {err:.3e}"
    y2 = mixtral8.layer.forward_routed(x, idx, w)
    assert torch.equal(y, y2)
