"""colibri_route_static: routing for callers that cannot allocate device memory.

Callers that may not call cudaMalloc (code running under CUDA-graph stream
capture, code inside a framework whose caching allocator owns the device
memory, or loops that cannot afford the implicit synchronisation of an
allocation) get the routing stage through this one entry point, which keeps
its intermediate data in a fixed device array inside the library instead of
allocating.  This test calls it through the C ABI twice in a row, with
different shapes and token counts so that leftovers of the first call would
show in the second, and checks each result against the handle-based path
(colibri_forward + colibri_get_routing on the same weights and tokens) within
the tolerances the parity tests use: the two paths compute the logits with
different kernels (different float32 summation orders), so expert ids must
agree on every token that is not a near-tie, gates within twice the parity
gate bound (each side is within one bound of the float64 softmax), and counts
and perm must agree bit for bit whenever the ids do.  Every result is also
checked against the CPU oracle under the parity rules of the other tests
(near-tie tokens excepted from the top-k comparison; counts and perm the
oracle's dispatch of the returned ids, bit for bit), including a batch at the
array's pair limit that takes the multi-CTA dispatch.  The file sorts last so
that a run stopping at the first failure has already run every other test.
"""

from types import SimpleNamespace

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import GATE_ATOL, NEAR_TIE_REL, check_routing

pytestmark = pytest.mark.gpu


def _routing_through_static_entry(sef, x, wr, bias, shape):
    T, k, E = x.shape[0], shape.top_k, shape.n_experts
    dev = x.device
    out = {
        "topk_idx": torch.full((T, k), -1, dtype=torch.int32, device=dev),
        "topk_w": torch.full((T, k), -1.0, dtype=torch.float32, device=dev),
        "counts": torch.full((E,), -1, dtype=torch.int32, device=dev),
        "perm": torch.full((T * k,), -1, dtype=torch.int32, device=dev),
    }
    st = sef.colibri_route_static(
        x.data_ptr(), wr.data_ptr(), None if bias is None else bias.data_ptr(), T,
        shape.d_model, E, k, sef.DTYPE_BF16 if x.dtype == torch.bfloat16 else sef.DTYPE_FP32,
        out["topk_idx"].data_ptr(), out["topk_w"].data_ptr(), out["counts"].data_ptr(),
        out["perm"].data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == sef.OK, sef.colibri_status_str(st)
    torch.cuda.synchronize()
    return out


def _check_against_oracle(x, wr, bias, shape, got):
    """The parity rules of the other GPU tests, applied to the static entry's output."""
    case = SimpleNamespace(shape=shape, wr64=oracle.to_f64(wr.cpu()),
                           off64=None if bias is None else bias.double().cpu().numpy())
    r = {k: v.cpu().numpy() for k, v in got.items()}
    assert int(r["counts"].sum()) == x.shape[0] * shape.top_k   # no failure reported (-1 counts)
    x64 = oracle.to_f64(x.cpu())
    _, near = check_routing(case, x64, r)
    tau = NEAR_TIE_REL * (np.abs(x64) @ np.abs(case.wr64))
    return near, tau


def test_route_static_matches_handle_path_on_two_calls_in_a_row(lib):
    sef = lib
    dev = torch.device("cuda", 0)
    cases = [(synth.QWEN2, 64, 0), (synth.DEEPSEEK_MASKED, 37, 1)]
    for shape, T, seed in cases:
        wr = synth.router_weight(shape, seed, 0, dev)
        wg, wu, wd = synth.expert_weights(shape, seed, 0, dev)
        b = synth.router_offset(shape)
        bias = None if b is None else b.to(dev)
        x = synth.tokens(shape, T, seed, 0, dev)

        got = _routing_through_static_entry(sef, x, wr, bias, shape)

        layer = sef.MoELayer(wr, wg, wu, wd, shape.top_k, router_bias=b, max_tokens=T)
        layer.forward(x)
        want = layer.routing()
        torch.cuda.synchronize()
        assert layer.check() == sef.OK
        layer.close()
        near, tau = _check_against_oracle(x, wr, bias, shape, got)
        g, w = ({k: v.cpu().numpy() for k, v in r.items()} for r in (got, want))
        same = (g["topk_idx"] == w["topk_idx"]).all(axis=1)
        assert (same | near).all(), f"{shape.name} T={T}: ids differ off near-ties"
        tau_sel = np.take_along_axis(tau, g["topk_idx"].astype(np.int64), axis=1).max(axis=1)
        bound = 2 * (GATE_ATOL + 0.5 * tau_sel)[:, None]
        assert (np.abs(g["topk_w"] - w["topk_w"])[same] <= bound[same]).all(), \
            f"{shape.name} T={T}: gates differ beyond the parity bound"
        if same.all():
            for key in ("counts", "perm"):
                assert np.array_equal(g[key], w[key]), f"{shape.name} T={T}: {key} differs"


def test_route_static_at_its_pair_limit_matches_oracle(lib):
    """131 072 (token, slot) pairs, the most the array holds: the router's
    many-token variant and the multi-CTA dispatch, then a small call that
    reuses the array."""
    sef = lib
    dev = torch.device("cuda", 0)
    for shape, T, seed in [(synth.QWEN2, 65536, 5), (synth.DEEPSEEK_MASKED, 300, 6)]:
        wr = synth.router_weight(shape, seed, 0, dev)
        b = synth.router_offset(shape)
        bias = None if b is None else b.to(dev)
        x = synth.tokens(shape, T, seed, 0, dev)
        got = _routing_through_static_entry(sef, x, wr, bias, shape)
        near, _ = _check_against_oracle(x, wr, bias, shape, got)
        assert near.sum() <= max(2, T // 5000)


def test_route_static_rejects_sizes_beyond_its_array(lib):
    sef = lib
    dev = torch.device("cuda", 0)
    buf = torch.zeros(16, dtype=torch.int32, device=dev)
    p = buf.data_ptr()
    s = torch.cuda.current_stream().cuda_stream
    # T * top_k above 131072 pairs
    assert sef.colibri_route_static(p, p, None, 65537, 128, 8, 2, sef.DTYPE_FP32,
                                    p, p, p, p, s) == sef.ERR_INVALID_ARG
    # d_model * n_experts above 1048576 elements
    assert sef.colibri_route_static(p, p, None, 1, 8192, 256, 2, sef.DTYPE_BF16,
                                    p, p, p, p, s) == sef.ERR_INVALID_ARG
