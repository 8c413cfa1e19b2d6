"""GPU parity of sattn_prepare: INT8 codes and scales, K mean, E4M3 V codes and
scales, bit for bit against the CPU oracle (same seeded inputs)."""
import numpy as np
import pytest
import torch

import quantized_exact_attention_smoothing_gb300 as sattn
import synth
from helpers import assert_prepare_bit_exact, to_device_bf16

pytestmark = pytest.mark.gpu


def _run(oracle_mod, q, k, v, causal=False):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    buf = sattn.prepare(to_device_bf16(q), to_device_bf16(k), to_device_bf16(v), causal)
    torch.cuda.synchronize()
    ref = oracle_mod.prepare(q, k, v)
    assert_prepare_bit_exact(buf, ref, k.shape[2])
    return buf, ref


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4", "c5"])
def test_prepare_bit_exact_on_workloads(oracle_mod, name):
    w = synth.workload(name)
    q, k, v = synth.make_inputs(w)
    _run(oracle_mod, q, k, v, w.causal)


@pytest.mark.parametrize("shape", [
    (1, 1, 1, 1, 1), (1, 2, 1, 31, 33), (1, 1, 1, 127, 129), (1, 1, 1, 129, 127),
    (2, 4, 2, 200, 200), (1, 3, 3, 65, 4000), (1, 1, 1, 5, 32760)])
def test_prepare_bit_exact_edge_shapes(oracle_mod, shape):
    B, Hq, Hkv, Nq, Nkv = shape
    w = synth.workload("c1", B=B, Hq=Hq, Hkv=Hkv, Nq=Nq, Nkv=Nkv)
    q, k, v = synth.make_inputs(w, seed=1000 + Nq + Nkv)
    _run(oracle_mod, q, k, v)


def test_prepare_zero_and_constant_inputs(oracle_mod):
    z = np.zeros((1, 2, 70, 128), dtype=np.uint16)
    _run(oracle_mod, z, z, z)
    rng = np.random.default_rng(7)
    const = synth.to_bf16_bits(np.broadcast_to(rng.standard_normal(128) * 3, (1, 2, 70, 128)))
    buf, _ = _run(oracle_mod, const, const, const)
    assert torch.all(buf["k_codes"] == 0)


def test_prepare_ties_and_extremes(oracle_mod):
    vals = np.array([127.0, 2.5, 3.5, -2.5, -0.5, 0.5, 1.5, -1.5, 126.5, -126.5])
    q = np.zeros((1, 1, 32, 128))
    q[0, 0, 0, :vals.size] = vals
    k = np.random.default_rng(3).standard_normal((1, 1, 32, 128)) * 1e3
    k[0, 0, 5, 7] = 3.0e38
    _run(oracle_mod, synth.to_bf16_bits(q), synth.to_bf16_bits(k), synth.to_bf16_bits(k * 1e-30))


def test_prepare_repeatable(oracle_mod):
    w = synth.workload("c2")
    q, k, v = synth.make_inputs(w)
    dq, dk, dv = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    a = sattn.prepare(dq, dk, dv)
    first = {n: a[n].clone() for n in ("q_codes", "k_codes", "v_codes", "k_mean")}
    for _ in range(3):
        sattn.prepare(dq, dk, dv, buffers=a)
    torch.cuda.synchronize()
    for n, t in first.items():
        assert torch.equal(t, a[n]), n


def test_int8_quantiser_exhaustive_over_bf16():
    # every positive finite BF16 amax and every BF16 x with |x| <= amax: the
    # division-free quantiser (including its exact tie decision) gives the
    # code of clamp(rint(fl(x / s))) with IEEE division, s = fl(amax / 127)
    bad, near, last = sattn.int8_quantiser_sweep_for_test()
    assert bad == 0, f"{bad} mismatches, last amax bits {last >> 16:#x} x bits {last & 0xffff:#x}"
    assert near > 100000   # the tie decision was exercised
