"""Failure detection on the GPU without a fault: a forward launch whose V tiles
are withheld (sattn_test_forward_withhold_v) ends through its bounded waits,
reports SATTN_ERR_TIMEOUT in the status block, and leaves the CUDA context
usable (the next forward matches the oracle)."""
import time

import numpy as np
import pytest
import torch

import quantized_exact_attention_smoothing_gb300 as sattn
import synth
from helpers import assert_close_output, bf16_bits, to_device_bf16

pytestmark = pytest.mark.gpu


def test_withheld_v_times_out_and_context_survives(oracle_mod):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    w = synth.workload("c2", Hq=4, Hkv=2, causal=True)
    q, k, v = synth.make_inputs(w)
    prep = sattn.prepare(to_device_bf16(q), to_device_bf16(k), to_device_bf16(v), w.causal)
    torch.cuda.synchronize()
    t0 = time.time()
    sattn.forward_withhold_v_for_test(prep)
    rc = sattn.check_status(prep["forward_workspace"])
    elapsed = time.time() - t0
    assert sattn.STATUS.get(rc) == "SATTN_ERR_TIMEOUT", rc
    assert 0.5 < elapsed < 30.0, elapsed            # the waits give up after about one second
    # the context still works: a normal launch on the same buffers is correct
    out = sattn.forward(prep)
    assert sattn.check_status(prep["forward_workspace"]) == 0
    ref = oracle_mod.prepare(q, k, v)
    rb, _ = oracle_mod.forward(ref, w.Nq, w.Nkv, w.causal)
    assert_close_output(bf16_bits(out), rb, "forward after a timed-out launch")
