"""A forward is stream-ordered, never synchronises the host and never
allocates, so it can be captured into a CUDA graph: kernels launched with
programmatic stream serialization become graph dependencies, and the
per-call tensor map of x is captured by value.  The replayed graph must give
the eager forward's outputs bit for bit, at a decode size (fused routing,
decode GEMMs with split K) and at a prefill size (tensor-core router with
split K, dispatch, gather, CTA-pair GEMMs), and again after x is overwritten
in place between replays."""

import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T", [4, 1024])
def test_forward_replays_from_a_cuda_graph(lib, T):
    import sparse_expert_ffn_gb300 as sef
    shape = synth.LayerShape("graph", 512, 512, 8, 2, "bf16")
    dev = torch.device("cuda", 0)
    wr = synth.router_weight(shape, 3, 0, dev)
    wg, wu, wd = synth.expert_weights(shape, 3, 0, dev)
    layer = sef.MoELayer(wr, wg, wu, wd, shape.top_k, max_tokens=T)
    try:
        x = synth.tokens(shape, T, 3, 0, dev)
        x2 = -0.5 * x.flip(0)
        y_ref = layer.forward(x).clone()
        y2_ref = layer.forward(x2).clone()
        xs = x.clone()
        ys = torch.empty_like(x)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            layer.forward(xs, ys, stream=s)      # warm-up on the capture stream
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            layer.forward(xs, ys, stream=s)
        for src, ref in ((x, y_ref), (x2, y2_ref), (x, y_ref)):
            xs.copy_(src)
            g.replay()
            torch.cuda.synchronize()
            assert layer.check() == sef.OK
            assert torch.equal(ys, ref)
    finally:
        layer.close()
