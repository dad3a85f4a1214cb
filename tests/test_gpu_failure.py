"""Failure detection on the GPU without faulting it.

* An allocation failure injected on the host (COLIBRI_FAIL_ALLOC_AT=n fails
  init's n-th device allocation) must return COLIBRI_ERR_OOM, leave no handle
  and free everything init had allocated.
* The grouped GEMM's mbarrier waits are bounded.  A handle built with
  COLIBRI_TEST_STALL_TMA=1 has a TMA producer that never issues its copies (a
  flag that nothing sets), and COLIBRI_WAIT_LIMIT_NS=20000000 bounds every
  wait at 20 ms: the MMA warp's first wait on a full stage runs out, the kernel
  records a timeout in the handle's status word, every role stops, tensor
  memory is freed and the kernel returns.  colibri_check must report
  COLIBRI_ERR_TIMEOUT, and the context must stay usable: a normal handle used
  before and after computes the same result.
"""

import ctypes
import os

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

SHAPE = synth.LayerShape("failure_probe", 512, 1024, 8, 2, "bf16")


def _weights(dev):
    wr = synth.router_weight(SHAPE, 3, 0, dev)
    wg, wu, wd = synth.expert_weights(SHAPE, 3, 0, dev)
    return wr, wg, wu, wd


def test_injected_allocation_failure_rolls_back(lib, monkeypatch):
    sef = lib
    dev = torch.device("cuda", 0)
    ws = _weights(dev)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    # weights on the device: four device allocations (router, gate/up, down, workspace)
    for n in range(1, 5):
        monkeypatch.setenv("COLIBRI_FAIL_ALLOC_AT", str(n))
        with pytest.raises(sef.ColibriError) as ei:
            sef.MoELayer(*ws, SHAPE.top_k, max_tokens=256)
        assert ei.value.status == sef.ERR_OOM
    monkeypatch.delenv("COLIBRI_FAIL_ALLOC_AT")
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert abs(free1 - free0) < 64 << 20, "failed inits leaked device memory"
    layer = sef.MoELayer(*ws, SHAPE.top_k, max_tokens=256)
    layer.close()


# A d_model of 4096 puts gate/up on the weights-as-M pair kernel too (the
# narrower shape runs only its down projection that way).
WIDE = synth.LayerShape("failure_probe_wide", 4096, 1024, 8, 2, "bf16")


# 2 tokens split the gate/up GEMM over K (last-slice fixup), 256 tokens run
# the expert GEMMs on single CTAs, 1024 on CTA pairs (at least 128
# (token, slot) pairs per expert on average), with the weights as the MMA's
# M operand for the down projection, and for gate/up as well on WIDE.
@pytest.mark.parametrize("shape,T", [(SHAPE, 2), (SHAPE, 256), (SHAPE, 1024), (WIDE, 1024)],
                         ids=["split_k", "single_cta", "cta_pairs", "cta_pairs_wide"])
def test_bounded_wait_times_out_and_context_survives(lib, monkeypatch, shape, T):
    sef = lib
    dev = torch.device("cuda", 0)
    wr = synth.router_weight(shape, 3, 0, dev)
    ws = (wr, *synth.expert_weights(shape, 3, 0, dev))
    x = synth.tokens(shape, T, 3, 0, dev)

    ref_layer = sef.MoELayer(*ws, shape.top_k, max_tokens=T, executor="grouped")
    y_ref = ref_layer.forward(x)
    assert ref_layer.check() == sef.OK

    monkeypatch.setenv("COLIBRI_WAIT_LIMIT_NS", "20000000")
    monkeypatch.setenv("COLIBRI_TEST_STALL_TMA", "1")
    short = sef.MoELayer(*ws, shape.top_k, max_tokens=T, executor="grouped")
    monkeypatch.delenv("COLIBRI_WAIT_LIMIT_NS")
    monkeypatch.delenv("COLIBRI_TEST_STALL_TMA")
    short.forward(x)
    assert short.check() == sef.ERR_TIMEOUT
    # the status word is cleared by the check
    assert short.check() == sef.OK
    short.close()

    # the context is intact: the default-bound handle still gives its result
    y2 = ref_layer.forward(x)
    assert ref_layer.check() == sef.OK
    assert torch.equal(y_ref, y2)
    ref_layer.close()


def test_bounded_wait_times_out_on_the_int8_gemm(lib, monkeypatch):
    """The int8-weight GEMM's extra rings (A, codes, f16 B) and roles (A
    producer, converters) give up on a stalled producer the same way."""
    sef = lib
    dev = torch.device("cuda", 0)
    wr, wg, wu, wd = _weights(dev)
    parts = [tuple(t.to(dev) for t in sef.quantize_int8_block64(w)) for w in (wg, wu, wd)]
    x = synth.tokens(SHAPE, 8, 3, 0, dev)
    ref_layer = sef.MoELayer(wr, None, None, None, SHAPE.top_k, max_tokens=8, int8=parts)
    y_ref = ref_layer.forward(x)
    assert ref_layer.check() == sef.OK

    monkeypatch.setenv("COLIBRI_WAIT_LIMIT_NS", "20000000")
    monkeypatch.setenv("COLIBRI_TEST_STALL_TMA", "1")
    short = sef.MoELayer(wr, None, None, None, SHAPE.top_k, max_tokens=8, int8=parts)
    monkeypatch.delenv("COLIBRI_WAIT_LIMIT_NS")
    monkeypatch.delenv("COLIBRI_TEST_STALL_TMA")
    short.forward(x)
    assert short.check() == sef.ERR_TIMEOUT
    assert short.check() == sef.OK
    short.close()

    y2 = ref_layer.forward(x)
    assert ref_layer.check() == sef.OK
    assert torch.equal(y_ref, y2)
    ref_layer.close()


def test_bounded_wait_times_out_on_the_int8_gemv(lib, monkeypatch):
    """The CUDA-core int8 GEMV (one token, streaming executor): its consumer
    warps give up on a ring stage that never lands, the CTA winds down, and
    the status word reports the timeout."""
    sef = lib
    dev = torch.device("cuda", 0)
    wr, wg, wu, wd = _weights(dev)
    parts = [tuple(t.to(dev) for t in sef.quantize_int8_block64(w)) for w in (wg, wu, wd)]
    x = synth.tokens(SHAPE, 1, 3, 0, dev)
    ref_layer = sef.MoELayer(wr, None, None, None, SHAPE.top_k, max_tokens=1, int8=parts,
                             executor="stream")
    y_ref = ref_layer.forward(x)
    assert ref_layer.check() == sef.OK

    monkeypatch.setenv("COLIBRI_WAIT_LIMIT_NS", "20000000")
    monkeypatch.setenv("COLIBRI_TEST_STALL_TMA", "1")
    short = sef.MoELayer(wr, None, None, None, SHAPE.top_k, max_tokens=1, int8=parts,
                         executor="stream")
    monkeypatch.delenv("COLIBRI_WAIT_LIMIT_NS")
    monkeypatch.delenv("COLIBRI_TEST_STALL_TMA")
    short.forward(x)
    assert short.check() == sef.ERR_TIMEOUT
    assert short.check() == sef.OK
    short.close()

    y2 = ref_layer.forward(x)
    assert ref_layer.check() == sef.OK
    assert torch.equal(y_ref, y2)
    ref_layer.close()
