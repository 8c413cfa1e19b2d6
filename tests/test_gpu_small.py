"""GPU parity of the single-launch small-shape path (sattn_attention_small):
for one query tile of one head it must write the preparation's buffers with
the bytes sattn_prepare writes and the output sattn_prepare + sattn_forward
give, and match the oracle.  Shapes on both sides of Nkv = 256, where the
in-kernel preparation switches from staging the inputs in shared memory to
reading them from global memory."""
import numpy as np
import pytest
import torch

import quantized_exact_attention_smoothing_gb300 as sattn
import synth
from helpers import assert_close_output, bf16_bits, to_device_bf16

pytestmark = pytest.mark.gpu

BUFFERS = ("q_codes", "q_scales", "k_codes", "k_scales", "k_mean", "v_codes", "v_scales")


@pytest.mark.parametrize("Nq, Nkv, causal", [
    (128, 192, False), (128, 192, True), (100, 300, True), (1, 1, False), (128, 1024, False),
    (37, 700, False), (128, 129, True), (64, 64, True), (128, 256, False), (5, 257, True), (128, 33, False)])
def test_small_path_equals_two_calls_and_oracle(oracle_mod, Nq, Nkv, causal):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    w = synth.workload("c1", Nq=Nq, Nkv=Nkv, causal=causal)
    q, k, v = synth.make_inputs(w, seed=900 + Nkv)
    dq, dk, dv = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    out_s, buf_s = sattn.attention_small(dq, dk, dv, causal)
    prep = sattn.prepare(dq, dk, dv, causal)
    out_p = sattn.forward(prep)
    torch.cuda.synchronize()
    assert sattn.check_status(buf_s["forward_workspace"]) == 0
    for name in BUFFERS:
        a, b = buf_s[name].cpu().numpy(), prep[name].cpu().numpy()
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), f"{name} differs"
    assert torch.equal(out_s.view(torch.int16), out_p.view(torch.int16)), "output differs from the two calls"
    ref = oracle_mod.prepare(q, k, v)
    rb, _ = oracle_mod.forward(ref, Nq, Nkv, causal)
    assert_close_output(bf16_bits(out_s), rb, f"small path {Nq}x{Nkv}")


def test_small_path_repeats_on_the_same_buffers():
    w = synth.workload("c1")
    q, k, v = synth.make_inputs(w, seed=5)
    dq, dk, dv = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    out, buf = sattn.attention_small(dq, dk, dv)
    first = out.clone()
    q2, k2, v2 = synth.make_inputs(w, seed=6)
    dq.copy_(to_device_bf16(q2))
    dk.copy_(to_device_bf16(k2))
    dv.copy_(to_device_bf16(v2))
    out2, _ = sattn.attention_small(dq, dk, dv, buffers=buf, out=torch.empty_like(out),
                                    workspace=buf["forward_workspace"])
    ref = sattn.forward(sattn.prepare(dq, dk, dv))
    torch.cuda.synchronize()
    assert torch.equal(out2.view(torch.int16), ref.view(torch.int16))
    assert not torch.equal(out2.view(torch.int16), first.view(torch.int16))
