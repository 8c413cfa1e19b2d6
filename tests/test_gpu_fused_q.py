"""GPU parity of the forward pass that quantises Q inside the kernel
(sattn_prepare_kv + sattn_forward_q_bf16).

Its Q codes and block scales are the preparation's, so its output must equal,
byte for byte, sattn_forward's on sattn_prepare's buffers; the K/V buffers of
sattn_prepare_kv must equal sattn_prepare's.  Together with the forward's
parity against the oracle (test_gpu_forward.py) this pins the fused path to
the oracle; one case is also compared with the oracle directly.
"""
import numpy as np
import pytest
import torch

import quantized_exact_attention_smoothing_gb300 as sattn
import synth
from helpers import assert_close_output, bf16_bits, to_device_bf16

pytestmark = pytest.mark.gpu

KV_NAMES = ("k_codes", "k_scales", "k_mean", "v_codes", "v_scales")


def _both(q, k, v, causal, sm_scale=0.0):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    dq, dk, dv = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    prep = sattn.prepare(dq, dk, dv, causal, sm_scale)
    ref = sattn.forward(prep)
    kv = sattn.prepare_kv(dk, dv, q.shape[1], q.shape[2], causal, sm_scale)
    got = sattn.forward_q_bf16(dq, kv)
    assert sattn.check_status(prep["forward_workspace"]) == 0
    assert sattn.check_status(kv["forward_workspace"]) == 0
    for n in KV_NAMES:
        assert torch.equal(kv[n], prep[n]), n
    return ref, got


def _assert_same(ref, got, what):
    if not torch.equal(ref.view(torch.int16), got.view(torch.int16)):
        diff = (ref.view(torch.int16) != got.view(torch.int16)).nonzero()
        raise AssertionError(f"{what}: {diff.shape[0]} output elements differ, first at {diff[0].tolist()}")


@pytest.mark.parametrize("shape", [
    (1, 1, 1, 128, 192, False), (1, 8, 8, 1024, 1024, False), (1, 2, 1, 100, 356, True),
    (1, 1, 1, 1, 300, True), (1, 2, 2, 260, 520, True), (1, 1, 1, 33, 129, False),
    (2, 16, 2, 160, 416, False), (1, 3, 3, 65, 4000, False), (2, 4, 1, 384, 384, True)])
def test_fused_q_equals_prepared_q(shape):
    B, Hq, Hkv, Nq, Nkv, causal = shape
    w = synth.workload("c1", B=B, Hq=Hq, Hkv=Hkv, Nq=Nq, Nkv=Nkv, causal=causal)
    q, k, v = synth.make_inputs(w, seed=4000 + Nq + 3 * Nkv + Hq)
    ref, got = _both(q, k, v, causal)
    _assert_same(ref, got, f"shape {shape}")


def test_fused_q_ties_zero_blocks_and_extremes():
    # exact rounding ties of the quantiser (amax 127 -> s = 1), an all-zero
    # 32-row block, a block of one huge value, and rows past Nq in the last tile
    q = np.random.default_rng(11).standard_normal((1, 2, 200, 128))
    q[0, 0, 0, :10] = [127.0, 2.5, 3.5, -2.5, -0.5, 0.5, 1.5, -1.5, 126.5, -126.5]
    q[0, 0, 1:32, :] = np.clip(np.round(q[0, 0, 1:32, :] * 30), -126, 126) + 0.5   # exact in BF16
    q[0, 0, 1:32, 0] = 127.0
    q[0, 0, 32:64, :] = 0.0
    q[0, 1, 64:96, :] *= 1e-3
    q[0, 1, 70, 5] = 3.0e4
    k = np.random.default_rng(12).standard_normal((1, 1, 300, 128)) + 2.0
    v = np.random.default_rng(13).standard_normal((1, 1, 300, 128))
    for causal in (False, True):
        ref, got = _both(synth.to_bf16_bits(q), synth.to_bf16_bits(k), synth.to_bf16_bits(v), causal)
        _assert_same(ref, got, f"ties causal={causal}")


def test_fused_q_explicit_scale():
    w = synth.workload("c1", B=1, Hq=2, Hkv=1, Nq=200, Nkv=300, causal=True)
    q, k, v = synth.make_inputs(w, seed=91)
    ref, got = _both(q, k, v, True, sm_scale=0.2)
    _assert_same(ref, got, "sm_scale 0.2")


def test_fused_q_against_oracle(oracle_mod):
    w = synth.workload("c2")
    q, k, v = synth.make_inputs(w)
    _, got = _both(q, k, v, w.causal)
    ref = oracle_mod.prepare(q, k, v)
    rb, _ = oracle_mod.forward(ref, w.Nq, w.Nkv, w.causal)
    assert_close_output(bf16_bits(got), rb, "c2 fused Q")


def test_fused_q_headline_size_and_repeatable():
    # the benchmark's workload (B4, Hq32/Hkv8, 8192 x 8192, causal) in the
    # launch configuration the benchmark times
    w = synth.workload("c5")
    q, k, v = synth.make_inputs(w)
    ref, got = _both(q, k, v, w.causal)
    _assert_same(ref, got, "c5")
    dq = to_device_bf16(q)
    kv = sattn.prepare_kv(to_device_bf16(k), to_device_bf16(v), w.Hq, w.Nq, w.causal)
    first = sattn.forward_q_bf16(dq, kv)
    for _ in range(2):
        again = sattn.forward_q_bf16(dq, kv)
        assert sattn.check_status(kv["forward_workspace"]) == 0
        _assert_same(first, again, "c5 repeat")
    _assert_same(ref, first, "c5 after prepare_kv")
