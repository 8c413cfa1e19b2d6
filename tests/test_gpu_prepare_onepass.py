"""sattn_prepare_kv_onepass (the K/V preparation as one cooperative launch,
phases separated by grid barriers): byte-identical to sattn_prepare_kv on the
workloads and ragged shapes; its barriers' bounded waits report a timeout
through the prepare workspace and leave the context usable."""
import time

import numpy as np
import pytest
import torch

import quantized_exact_attention_smoothing_gb300 as sattn
import synth
from helpers import to_device_bf16

pytestmark = pytest.mark.gpu

KEYS = ("k_codes", "k_scales", "k_mean", "v_codes", "v_scales")


def _both(w, seed=None):
    q, k, v = synth.make_inputs(w, seed=seed)
    dk, dv = to_device_bf16(k), to_device_bf16(v)
    a = sattn.prepare_kv(dk, dv, w.Hq, w.Nq, w.causal)
    b = sattn.prepare_kv_onepass(dk, dv, w.Hq, w.Nq, w.causal)
    assert sattn.check_prepare_status(b) == 0
    return a, b


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c5"])
def test_onepass_equals_split_on_workloads(name):
    a, b = _both(synth.workload(name))
    for key in KEYS:
        assert torch.equal(a[key].view(torch.uint8), b[key].view(torch.uint8)), key


@pytest.mark.parametrize("shape", [(1, 2, 1, 33, 1, False), (2, 4, 2, 129, 4001, True), (1, 3, 3, 64, 32760, False)])
def test_onepass_equals_split_on_ragged_shapes(shape):
    B, Hq, Hkv, Nq, Nkv, causal = shape
    a, b = _both(synth.workload("c2", B=B, Hq=Hq, Hkv=Hkv, Nq=Nq, Nkv=Nkv, causal=causal), seed=77 + Nkv)
    for key in KEYS:
        assert torch.equal(a[key].view(torch.uint8), b[key].view(torch.uint8)), key


def test_onepass_barrier_timeout_reports_and_context_survives():
    w = synth.workload("c2", Hq=4, Hkv=2)
    q, k, v = synth.make_inputs(w)
    dk, dv = to_device_bf16(k), to_device_bf16(v)
    torch.cuda.synchronize()
    t0 = time.time()
    buf = sattn.prepare_kv_onepass(dk, dv, w.Hq, w.Nq, w.causal, _withhold_for_test=True)
    rc = sattn.check_prepare_status(buf)
    elapsed = time.time() - t0
    assert sattn.STATUS.get(rc) == "SATTN_ERR_TIMEOUT", rc
    assert 0.5 < elapsed < 30.0, elapsed   # the barrier gives up after about one second
    # the same buffers work again, and the next call is correct
    buf = sattn.prepare_kv_onepass(dk, dv, w.Hq, w.Nq, w.causal, buffers=buf)
    assert sattn.check_prepare_status(buf) == 0
    ref = sattn.prepare_kv(dk, dv, w.Hq, w.Nq, w.causal)
    for key in KEYS:
        assert torch.equal(ref[key].view(torch.uint8), buf[key].view(torch.uint8)), key
