"""The benchmark's algorithmic bytes and FLOPs (the numerators of every
roofline fraction it prints) against figures worked out by hand from the
metric's definition:

  bytes = active experts * 3*d*f*s + d*E*s (router) + 2*T*d*s (x in, y out)
          + T*k*8 (ids and gates)
  FLOPs = 2*T*d*E + 6*T*k*d*f

Expected values below are written out as the products they are, so that a
dropped term or a wrong factor in bench.algorithmic shows."""

import numpy as np
import pytest

import bench
import synth


def _counts(E, active):
    c = np.zeros(E, dtype=np.int64)
    c[:active] = 1
    return c


@pytest.mark.parametrize("shape,T,active,gb,tflop", [
    # Mixtral-shaped: 8 experts of 3 * 4096 * 14336 bf16 weights
    (synth.MIXTRAL, 4096, 8, 2.885, 2.886),
    (synth.MIXTRAL, 1, 2, 0.7047, 0.000705),
    (synth.MIXTRAL, 16, 8, 2.818, 0.01128),
    # DeepSeek-shaped: 128 experts of 3 * 2048 * 1408, k = 4; 96 live when masked
    (synth.DEEPSEEK, 16384, 128, 2.350, 1.143),
    (synth.DEEPSEEK, 16384, 96, 1.797, 1.143),
])
def test_layer_bytes_and_flops(shape, T, active, gb, tflop):
    a = bench.algorithmic(shape, T, _counts(shape.n_experts, active))
    assert a["active_experts"] == active
    assert a["bytes"] / 1e9 == pytest.approx(gb, rel=2e-3)
    assert a["flops"] / 1e12 == pytest.approx(tflop, rel=2e-3)


def test_terms_one_by_one():
    d, f, E, k, T, s = 4096, 14336, 8, 2, 4096, 2
    a = bench.algorithmic(synth.MIXTRAL, T, _counts(E, 8))
    assert a["bytes"] == 8 * 3 * d * f * s + d * E * s + 2 * T * d * s + T * k * 8
    assert a["flops"] == 2 * T * d * E + 6 * T * k * d * f
    # per GEMM: gate/up is two d x f products per pair, down one f x d
    assert a["up_flops"] == 2 * a["down_flops"] == 4 * T * k * d * f
    assert a["up_flops"] + a["down_flops"] + 2 * T * d * E == a["flops"]


def test_int8_weights_count_one_byte_plus_block_metadata():
    d, f = 4096, 14336
    a16 = bench.algorithmic(synth.MIXTRAL, 1, _counts(8, 2))
    a8 = bench.algorithmic(synth.MIXTRAL, 1, _counts(8, 2), weights="int8")
    per_matrix = d * f + 8 * (d // 64) * (f // 64)      # codes + (scale, zero point) per block
    assert a16["bytes"] - a8["bytes"] == 2 * 3 * (2 * d * f - per_matrix)


def test_inactive_experts_cost_no_weight_bytes():
    a0 = bench.algorithmic(synth.QWEN2, 64, _counts(64, 0))
    a1 = bench.algorithmic(synth.QWEN2, 64, _counts(64, 1))
    assert a1["bytes"] - a0["bytes"] == 3 * 2048 * 1408 * 2


def test_traffic_key_names_top_k_and_weight_format():
    from dataclasses import replace
    assert bench.traffic_key("mixtral", 4096, synth.MIXTRAL) == "mixtral_T4096"
    assert bench.traffic_key("mixtral", 4096, replace(synth.MIXTRAL, top_k=1)) == "mixtral_T4096_k1"
    assert bench.traffic_key("mixtral", 1, synth.MIXTRAL, "int8") == "mixtral_T1_int8"
    # a summary for another configuration is never matched
    assert bench.measured_traffic("grouped_gemm_tc<kGateUp>", "mixtral_T4096_k1") is None


def test_dominant_roofline_divides_per_launch():
    """Two calls of a layer, one gate/up launch each: the per-launch FLOPs are
    the per-call FLOPs, and the achieved rate is those over one launch's time."""
    a = bench.algorithmic(synth.MIXTRAL, 4096, _counts(8, 8))
    alg = dict(a, calls=2)
    for k in ("up_flops", "down_flops", "up_bytes", "down_bytes", "bytes", "flops"):
        alg[k] = a[k] * 2
    stages = {"expert_up": {"ms_total": 2.0, "launches": 2},     # 1 ms per launch
              "expert_down": {"ms_total": 1.2, "launches": 2}}
    pk = {"hbm_gbs": 6769.4, "bf16_tflops": 1858.5, "source": "measured"}
    roof = bench.dominant_roofline(stages, alg, lambda s: s, pk)
    assert roof["bound"] == "tensor" and roof["kernel"] == "expert_up"
    assert roof["algorithmic_per_launch"] == 4 * 4096 * 2 * 4096 * 14336
    assert roof["achieved"] == pytest.approx(4 * 4096 * 2 * 4096 * 14336 / 1e-3 / 1e12, rel=1e-3)
