"""Helpers for the GPU parity tests: build a layer from the seeded generator,
run it through the C ABI, and compare against the CPU oracle under the
routing near-tie rule.

Parity rules (all float tolerances are written here once):
* topk_idx must equal the oracle's on every token that is not a near-tie
  (oracle.near_tie_tokens); near-tie tokens may differ and are counted.
  With top_k == E (soft routing) it must equal 0..E-1 on every token.
* counts and perm must equal the oracle's dispatch of the GPU's own topk_idx
  (an integer function: always exact), and the oracle's own dispatch when no
  token is a near-tie.
* topk_w within GATE_ATOL + 1/2 max_j tau[t, j] of the softmax over the
  oracle's float64 logits at the GPU's selected experts.  tau is the logit
  error radius of the near-tie rule (the accuracy the routing contract grants
  float32 accumulation in any order); the softmax Jacobian bounds the induced
  gate error: |dg_i| <= 2 g_i (1 - g_i) max_j |dl_j| <= max_j |dl_j| / 2.
* y: max|y - y_ref| / max|y_ref| <= Y_RTOL[dtype], y_ref the oracle's
  sum_j g_j FFN_{e_j}(x) at the GPU's selected experts (identical to the plain
  oracle wherever routing agrees).
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

GATE_ATOL = 1e-6
NEAR_TIE_REL = 2.0 ** -20   # oracle.near_tie_tokens' default radius
Y_RTOL = {"fp32": 1e-4, "bf16": 2e-2}


class Experts:
    """Lazy float64 copies of one expert's (W_g, W_u, W_d) for the oracle."""

    def __init__(self, wg, wu, wd):
        self.wg, self.wu, self.wd = wg.cpu(), wu.cpu(), wd.cpu()
        self._cache = {}

    def __call__(self, e):
        if e not in self._cache:
            if len(self._cache) >= 2:
                self._cache.pop(next(iter(self._cache)))
            self._cache[e] = (oracle.to_f64(self.wg[e]), oracle.to_f64(self.wu[e]),
                              oracle.to_f64(self.wd[e]))
        return self._cache[e]


class Case:
    """One layer's weights on the GPU (one library handle) plus float64 CPU
    views for the oracle.  Token batches come from ``tokens(T)``: the first T
    rows of the seeded token stream, so a smaller T is a prefix of a larger."""

    def __init__(self, shape: synth.LayerShape, seed: int, max_tokens: int,
                 layer_idx: int = 0, executor: str = "auto", bias="recipe"):
        import sparse_expert_ffn_gb300 as sef
        self.dev = torch.device("cuda", 0)
        self.shape, self.seed, self.layer_idx = shape, seed, layer_idx
        wr = synth.router_weight(shape, seed, layer_idx, self.dev)
        wg, wu, wd = synth.expert_weights(shape, seed, layer_idx, self.dev)
        self.bias = synth.router_offset(shape) if isinstance(bias, str) else bias
        self.layer = sef.MoELayer(wr, wg, wu, wd, shape.top_k, router_bias=self.bias,
                                  max_tokens=max_tokens, executor=executor)
        self.wr64 = oracle.to_f64(wr)
        self.experts = Experts(wg, wu, wd)
        self.off64 = None if self.bias is None else self.bias.double().numpy()
        del wg, wu, wd
        torch.cuda.empty_cache()

    def tokens(self, T: int):
        x = synth.tokens(self.shape, T, self.seed, self.layer_idx, self.dev)
        return x, oracle.to_f64(x)

    def run(self, x, executor: str | None = None):
        if executor:
            self.layer.set_executor(executor)
        y = self.layer.forward(x)
        r = self.layer.routing()
        torch.cuda.synchronize()
        assert self.layer.check() == 0, "library reported a device-side failure"
        return y, {k: v.cpu().numpy() for k, v in r.items()}

    def close(self):
        self.layer.close()


class Int8Experts:
    """Per expert, the oracle's own int8 block quantisation of (W_g, W_u, W_d),
    dequantised to float64 (oracle/quant.py), computed on demand."""

    def __init__(self, wg, wu, wd):
        self.wg, self.wu, self.wd = wg.cpu(), wu.cpu(), wd.cpu()
        self._cache = {}

    def __call__(self, e):
        if e not in self._cache:
            if len(self._cache) >= 2:
                self._cache.pop(next(iter(self._cache)))
            mats = []
            for w in (self.wg[e], self.wu[e], self.wd[e]):
                q, s, z = oracle.quantize_int8_block64(oracle.to_f64(w))
                mats.append(oracle.dequantize_int8_block64(q, s, z))
            self._cache[e] = tuple(mats)
        return self._cache[e]


class Int8Case(Case):
    """A layer whose expert weights go through the library's int8 converter
    (colibri_quantize_int8_block64) and colibri_init_int8; the oracle side
    quantises the same float weights with its own quantiser."""

    def __init__(self, shape: synth.LayerShape, seed: int, max_tokens: int,
                 layer_idx: int = 0, bias="recipe"):
        import sparse_expert_ffn_gb300 as sef
        self.dev = torch.device("cuda", 0)
        self.shape, self.seed, self.layer_idx = shape, seed, layer_idx
        wr = synth.router_weight(shape, seed, layer_idx, self.dev)
        wg, wu, wd = synth.expert_weights(shape, seed, layer_idx, self.dev)
        self.bias = synth.router_offset(shape) if isinstance(bias, str) else bias
        parts = [tuple(t.to(self.dev) for t in sef.quantize_int8_block64(w)) for w in (wg, wu, wd)]
        self.layer = sef.MoELayer(wr, None, None, None, shape.top_k, router_bias=self.bias,
                                  max_tokens=max_tokens, int8=parts)
        self.wr64 = oracle.to_f64(wr)
        self.experts = Int8Experts(wg, wu, wd)
        self.off64 = None if self.bias is None else self.bias.double().numpy()
        del wg, wu, wd, parts
        torch.cuda.empty_cache()


def check_routing(case: Case, x64, r, allow_near_ties: bool = True):
    """Compare routing to the oracle; returns (logits64, near_tie mask)."""
    k, E = case.shape.top_k, case.shape.n_experts
    l = oracle.router_logits(x64, case.wr64, case.off64)
    if k == E:
        # soft routing: every expert in expert order, no selection to tie on
        ref_idx = oracle.soft_route(l)[0]
        near = np.zeros(l.shape[0], dtype=bool)
    else:
        ref_idx = oracle.topk_select(l, k)
        near = oracle.near_tie_tokens(x64, case.wr64, l, k)
    if not allow_near_ties:
        assert not near.any(), f"{int(near.sum())} near-tie tokens"
    gidx = r["topk_idx"]
    bad = np.nonzero((gidx != ref_idx).any(axis=1) & ~near)[0]
    assert bad.size == 0, f"topk_idx differs on {bad.size} non-near-tie tokens, e.g. t={bad[:5]}"
    # gates against the float64 softmax at the GPU's experts
    g_ref = oracle.softmax_selected(l, gidx)
    tau = NEAR_TIE_REL * (np.abs(x64) @ np.abs(case.wr64))
    tau_sel = np.take_along_axis(tau, gidx.astype(np.int64), axis=1).max(axis=1, keepdims=True)
    gerr = np.abs(r["topk_w"] - g_ref)
    bad = gerr > GATE_ATOL + 0.5 * tau_sel
    assert not bad.any(), f"gate error {gerr.max():.3e} (bound {GATE_ATOL} + tau/2)"
    # dispatch: exact function of the GPU's own topk_idx
    counts, offsets, perm, inv = oracle.dispatch(gidx, E)
    assert np.array_equal(r["counts"], counts), "counts differ"
    assert np.array_equal(r["perm"], perm), "perm differs"
    if not near.any():
        counts2, _, perm2, _ = oracle.dispatch(ref_idx, E)
        assert np.array_equal(r["counts"], counts2) and np.array_equal(r["perm"], perm2)
    return l, near


def check_output(case: Case, x64, y, r, l, tokens=None, capacity=None):
    """max|err|/max|ref| of y on `tokens` (all by default); returns the error.

    With a capacity, the pairs kept are the oracle's capacity_keep of the
    GPU's own topk_idx (an integer function of the routing, like dispatch)."""
    T = x64.shape[0]
    tok = np.arange(T) if tokens is None else np.asarray(tokens)
    gidx = r["topk_idx"][tok]
    g = oracle.softmax_selected(l[tok], gidx)
    keep = None
    if capacity is not None:
        keep = oracle.capacity_keep(r["topk_idx"], case.shape.n_experts, capacity)[tok]
    y_ref = oracle.token_outputs(x64[tok], gidx, g, case.experts, keep_rows=keep)
    y_gpu = oracle.to_f64(y[torch.as_tensor(tok, device=y.device)].cpu())
    if np.abs(y_ref).max() == 0.0:
        assert np.all(y_gpu == 0.0), "every pair dropped: y must be exactly 0"
        return 0.0
    err = np.abs(y_gpu - y_ref).max() / max(np.abs(y_ref).max(), 1e-30)
    tol = Y_RTOL[case.shape.dtype]
    assert err <= tol, f"max|err|/max|ref| = {err:.3e} > {tol}"
    return err


def stack_case_layers(n_layers: int, seed: int, max_tokens: int):
    """The decode stack's layers (Mixtral-shaped) as library handles, one per layer.

    Returns (layers, gamma) with gamma = ones [d] bf16 on the device.  Layer l
    draws its weights with layer index l of the seeded generator."""
    import sparse_expert_ffn_gb300 as sef
    shape = synth.MIXTRAL
    dev = torch.device("cuda", 0)
    layers = []
    for l in range(n_layers):
        wr = synth.router_weight(shape, seed, l, dev)
        wg, wu, wd = synth.expert_weights(shape, seed, l, dev)
        layers.append(sef.MoELayer(wr, wg, wu, wd, shape.top_k, max_tokens=max_tokens))
        del wr, wg, wu, wd
    torch.cuda.empty_cache()
    gamma = torch.ones(shape.d_model, dtype=torch.bfloat16, device=dev)
    return layers, gamma
