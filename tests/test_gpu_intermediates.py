"""GPU parity of the forward kernel's intermediates against the oracle, for the
first KV tile of query tile 0 of (batch 0, head 0): the raw QK accumulators,
the FP8 P bytes and the first PV partial.

A build with SATTN_DEBUG_DUMP (quantized_exact_attention_smoothing_gb300.build
.build_debug) makes the kernel write them to a buffer set with
sattn_debug_set_dump.  The accumulators must equal the oracle's exact int32
dot products.  P8 must equal the oracle's bytes, except that a value within
rounding distance of an E4M3 tie may take the neighbouring code (the kernel
forms exp2's argument with one FMA and uses ex2.approx).  The PV partial
must equal the oracle's, up to FP32 summation order and one E4M3 step of
weight at each key whose P8 byte differs.
"""
import ctypes

import numpy as np
import pytest
import torch

from quantized_exact_attention_smoothing_gb300 import _binding as bnd
from quantized_exact_attention_smoothing_gb300 import build as B
import synth
from helpers import to_device_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbg_lib():
    lib = ctypes.CDLL(B.build_debug())
    P, SP = ctypes.c_void_p, ctypes.POINTER(bnd.sattn_shape)
    lib.sattn_prepare.argtypes = [SP] + [P] * 12
    lib.sattn_forward.argtypes = [SP] + [P] * 9
    lib.sattn_debug_set_dump.argtypes = [P]
    return lib


def _run_dump(lib, q, k, v, causal):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    dq, dk, dv = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    Bn, Hq, Nq, _ = q.shape
    shape = bnd.make_shape(Bn, Hq, k.shape[1], Nq, k.shape[2], causal)
    buf = bnd.prepare_buffers(shape, dq.device)
    out = torch.empty((Bn, Hq, Nq, 128), dtype=torch.bfloat16, device="cuda")
    fws = torch.zeros(bnd.query_sizes(shape)["forward_workspace"] // 4, dtype=torch.int32, device="cuda")
    dump = torch.zeros(98304, dtype=torch.float32, device="cuda")
    s = bnd._stream(None)
    p = bnd._ptr
    assert lib.sattn_prepare(ctypes.byref(shape), p(dq), p(dk), p(dv), p(buf["q_codes"]), p(buf["q_scales"]),
                             p(buf["k_codes"]), p(buf["k_scales"]), p(buf["k_mean"]),
                             p(buf["v_codes"]), p(buf["v_scales"]), p(buf["workspace"]), s) == 0
    lib.sattn_debug_set_dump(ctypes.c_void_p(dump.data_ptr()))
    try:
        assert lib.sattn_forward(ctypes.byref(shape), p(buf["q_codes"]), p(buf["q_scales"]), p(buf["k_codes"]),
                                 p(buf["k_scales"]), p(buf["v_codes"]), p(buf["v_scales"]), p(out), p(fws), s) == 0
        torch.cuda.synchronize()
    finally:
        lib.sattn_debug_set_dump(None)
    assert int(fws[0]) == 0
    d = dump.cpu().numpy()
    s_acc = d[:32768].reshape(128, 256)
    p8 = d[32768:40960].view(np.uint32).reshape(128, 64).view(np.uint8).reshape(128, 256)
    part = d[40960:40960 + 128 * 144].reshape(128, 144)
    return s_acc, p8, part


@pytest.mark.parametrize("shape", [
    (1, 1, 1, 128, 192, False),    # c1: 192 kept keys of 256, every row
    (1, 1, 1, 128, 512, False),    # a full first tile
    (1, 2, 1, 256, 256, True),     # the causal diagonal runs through the tile
    (1, 1, 1, 100, 300, True)])    # ragged rows, bottom-right causal offset
def test_first_tile_intermediates_match_the_oracle(oracle_mod, dbg_lib, shape):
    Bn, Hq, Hkv, Nq, Nkv, causal = shape
    w = synth.workload("c1", B=Bn, Hq=Hq, Hkv=Hkv, Nq=Nq, Nkv=Nkv, causal=causal)
    q, k, v = synth.make_inputs(w, seed=500 + Nkv)
    s_acc, p8, part = _run_dump(dbg_lib, q, k, v, causal)
    ref = oracle_mod.prepare(q, k, v)
    acc_o, p8_o, _ = oracle_mod.first_tile(ref, Nq, Nkv, causal)
    rows, n = min(Nq, 128), min(Nkv, 256)

    # QK: exact integers, every key of the tile (pad keys read zero codes)
    assert np.array_equal(s_acc[:rows], acc_o[:rows].astype(np.float32))

    # P8: bytes equal but for rare one-code steps at E4M3 ties
    diff = p8[:rows].astype(np.int16) - p8_o[:rows].astype(np.int16)
    assert np.abs(diff).max() <= 1, "P8 differs by more than one code"
    assert np.count_nonzero(diff) <= max(2, rows * n // 1000), f"{np.count_nonzero(diff)} P8 codes differ"

    # PV: the oracle's partial of its own P8.  Where the P8 bytes agree the
    # sums agree up to FP32 summation order; each key whose byte differs by
    # one code moves a channel by at most one E4M3 step of the oracle's
    # weight (<= 1/8 of it, or 2^-9 below the normal range) times |v8|.
    _, _, part_o = oracle_mod.first_tile(ref, Nq, Nkv, causal)
    po = oracle_mod.e4m3_to_f32(p8_o[:rows].reshape(-1)).reshape(rows, 256).astype(np.float64)
    vv = np.zeros((256, 128))
    vv[:n] = oracle_mod.e4m3_to_f32(ref["v_codes"][0, 0, :n].reshape(-1)).reshape(n, 128)
    step = np.where(diff != 0, 0.125 * po + 2.0 ** -9, 0.0)
    bound = 4e-6 * (np.abs(po) @ np.abs(vv)) + step @ np.abs(vv) + 1e-30
    got = part[:rows, :128].astype(np.float64)
    assert np.all(np.abs(got - part_o[:rows, :128]) <= bound), "PV partial off beyond summation order and P8 steps"
    dsum = 4e-6 * po.sum(axis=1) + step.sum(axis=1)   # the ones row: sum of p8
    assert np.all(np.abs(part[:rows, 128].astype(np.float64) - part_o[:rows, 128]) <= dsum)
    assert not part[:rows, 129:].any()
