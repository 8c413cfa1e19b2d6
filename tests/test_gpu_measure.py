"""The measurement hooks: sattn_measure_mma_rate reports the tcgen05.mma
rates of the forward's instruction shapes, and sattn_profile_events brackets
the attention kernel alone (inside the forward call's own time)."""
import pytest
import torch

import quantized_exact_attention_smoothing_gb300 as sattn
import synth
from helpers import to_device_bf16

pytestmark = pytest.mark.gpu


def test_mma_rates_are_dense_rates_and_fp8_doubles_fp16():
    f16 = sattn.measure_mma_rate("f16", 256, iters=1024)
    f8 = sattn.measure_mma_rate("f8", 144, iters=1024)
    # one M = 128 kind::f16 instruction moves 2 * 128 * 256 * 16 FLOP; the
    # dense rate is a few thousand FLOP per SM-clock
    assert 4000 < f16["flop_per_clk_sm"] < 20000
    assert 1.8 < f8["flop_per_clk_sm"] / f16["flop_per_clk_sm"] < 2.2
    assert f16["tflops"] > 0 and f8["tflops"] > f16["tflops"]


def test_mma_rate_rejects_bad_arguments():
    for kind, n in (("f16", 8), ("f8", 264), ("f16", 100)):
        with pytest.raises(sattn.SattnError):
            sattn.measure_mma_rate(kind, n)


def test_profile_events_bracket_the_attention_kernel():
    w = synth.workload("c2")
    q, k, v = synth.make_inputs(w)
    prep = sattn.prepare(to_device_bf16(q), to_device_bf16(k), to_device_bf16(v))
    out = sattn.forward(prep)
    s = torch.cuda.current_stream()
    e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    e[0].record(s)
    sattn.profile_events(e[1], e[2])
    try:
        sattn.forward(prep, out=out)
    finally:
        sattn.profile_events()
    e[3].record(s)
    torch.cuda.synchronize()
    kernel, call = e[1].elapsed_time(e[2]), e[0].elapsed_time(e[3])
    assert 0 < kernel <= call
    with pytest.raises(ValueError):
        sattn.profile_events(e[1], None)
