"""Layers at the edges of what the configuration accepts, every token checked
against the oracle.

* 256 experts (the most a handle takes) with top-8 (the most experts a token
  picks outside soft routing), on each router: one token (routing, dispatch
  and gather in one CTA), 40 tokens (CUDA-core router and dispatch kernels)
  and 600 tokens (tensor-core router: 256 logit columns per row).
* A bf16 layer whose d_model = 320 is a multiple of 64 but not of 256: the
  tensor-core GEMMs cannot tile it, so the auto executor streams the weights
  on CUDA cores.
* One expert with k = 1 (k equal to the expert count: the soft-routing
  path): every gate is exactly 1 and the layer is a dense SwiGLU FFN.
* Two experts with k = 1 at 700 tokens: the tensor-core router's 16-column
  logit tile holds two live columns.
* 65 536 tokens on the tiny fp32 shape (more token rows than a grid's y
  dimension holds: the combine strides over tokens), through colibri_forward
  and through colibri_combine_rows."""

import numpy as np
import pytest
import torch

import oracle
import sparse_expert_ffn_gb300 as sef
import synth
from parity import Y_RTOL, Case, check_output, check_routing

pytestmark = pytest.mark.gpu


def _check_all(case, Ts, executor="auto"):
    for T in Ts:
        x, x64 = case.tokens(T)
        y, r = case.run(x, executor)
        l, near = check_routing(case, x64, r)
        assert near.sum() <= max(1, T // 50)
        check_output(case, x64, y, r, l)
        y2, _ = case.run(x, executor)
        assert torch.equal(y, y2)


def test_256_experts_top8(lib):
    shape = synth.LayerShape("e256_k8", 256, 128, 256, 8, "bf16")
    c = Case(shape, seed=11, max_tokens=600)
    try:
        _check_all(c, (1, 40, 600))
    finally:
        c.close()


def test_bf16_layer_outside_the_tensor_core_tiling_streams(lib):
    shape = synth.LayerShape("d320", 320, 256, 8, 2, "bf16")
    c = Case(shape, seed=12, max_tokens=64)
    try:
        _check_all(c, (1, 7, 64))
        c.layer.set_executor("auto")
        with pytest.raises(sef.ColibriError):
            c.layer.set_executor("grouped")
    finally:
        c.close()


def test_single_expert_is_a_dense_ffn(lib):
    shape = synth.LayerShape("e1_k1", 256, 256, 1, 1, "bf16")
    c = Case(shape, seed=13, max_tokens=700)
    try:
        for T in (3, 700):
            x, x64 = c.tokens(T)
            y, r = c.run(x, "auto")
            assert (r["topk_idx"] == 0).all() and (r["topk_w"] == 1.0).all()
            l, _ = check_routing(c, x64, r)
            check_output(c, x64, y, r, l)
    finally:
        c.close()


def test_two_experts_top1_on_the_tensor_core_router(lib):
    shape = synth.LayerShape("e2_k1", 256, 256, 2, 1, "bf16")
    c = Case(shape, seed=14, max_tokens=700)
    try:
        _check_all(c, (700,))
    finally:
        c.close()


def test_65536_tokens_forward_and_combine_rows(lib):
    T = 65536
    c = Case(synth.TINY, seed=15, max_tokens=T)
    try:
        x, x64 = c.tokens(T)
        y, r = c.run(x, "auto")
        l, near = check_routing(c, x64, r)
        assert near.sum() <= 4
        check_output(c, x64, y, r, l)

        # colibri_combine_rows on rows in the expert order of the GPU's perm
        k, d = c.shape.top_k, c.shape.d_model
        dev = x.device
        rows = synth.normal((T * k, d), 3, 0, 99, device=dev).float()
        perm = torch.as_tensor(r["perm"].astype(np.int32), device=dev)
        gates = torch.as_tensor(r["topk_w"], device=dev)
        inv = torch.empty(T * k, dtype=torch.int32, device=dev)
        out = torch.empty(T, d, dtype=torch.float32, device=dev)
        st = sef.colibri_combine_rows(rows.data_ptr(), sef.DTYPE_FP32, gates.data_ptr(),
                                      perm.data_ptr(), T, k, d, sef.DTYPE_FP32, inv.data_ptr(),
                                      out.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert st == sef.OK
        torch.cuda.synchronize()
        _, _, _, inv_ref = oracle.dispatch(r["topk_idx"], c.shape.n_experts)
        ref = oracle.combine(rows.cpu().double().numpy(), r["topk_w"].astype(np.float64), inv_ref)
        err = np.abs(out.cpu().double().numpy() - ref).max() / np.abs(ref).max()
        assert err <= Y_RTOL["fp32"], err
    finally:
        c.close()
