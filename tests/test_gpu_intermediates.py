"""GPU parity of the forward kernel's intermediates against the oracle
("Experiment Log" page, entry "Phase 2B Fixed Aligned Numerical Prototype":
QK, m, d, FP8 probability, rescale, PV, FP32 RO, reciprocal), for query tile 0
of (batch 0, head 0).

A build with SATTN_DEBUG_DUMP (quantized_exact_attention_smoothing_gb300.build
.build_debug) makes the kernel write them to a buffer set with
sattn_debug_set_dump: for KV tile 0 (256 keys) the raw QK accumulators, the FP8
P bytes and the PV partial; for KV tile 1 the running maximum, its rescale factor
alpha, d and RO after the outer update; at the end d and its reciprocal.

Exact: the accumulators (the int32 dot products), the P bytes, and the running
maximum.  Within FP32 rounding: the PV partial (tensor-core summation order),
alpha (hardware exp2, relative error below 2^-22), d and RO (the outer update
is one fused multiply-add per value) and the reciprocal, which must also be
the correctly rounded reciprocal of the kernel's own d.
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

TILE = 256
DBG_S, DBG_P8, DBG_PV, DBG_M1, DBG_A1, DBG_D1, DBG_RO1, DBG_DF, DBG_RCP = (
    0, 32768, 40960, 83000, 83128, 83256, 83384, 99768, 99896)
# debug builds read a test mode here: 1 (2) = one (two) P8 words of each row and
# tile are taken as undecided, so that the forward's exact fix-up runs on
# every tile: from the parked exponent arguments (one word) or by recomputing
# the blocks from the codes (two words)
DBG_MODE = 60012


@pytest.fixture(scope="module")
def dbg_lib():
    lib = ctypes.CDLL(B.build_debug())
    P, SP = ctypes.c_void_p, ctypes.POINTER(bnd.sattn_shape)
    lib.sattn_prepare.argtypes = [SP] + [P] * 12
    lib.sattn_forward.argtypes = [SP] + [P] * 9
    lib.sattn_debug_set_dump.argtypes = [P]
    return lib


def _run_dump(lib, q, k, v, causal, mode=0):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    dq, dk, dv = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    Bn, Hq, Nq, _ = q.shape
    shape = bnd.make_shape(Bn, Hq, k.shape[1], Nq, k.shape[2], causal)
    buf = bnd.prepare_buffers(shape, dq.device)
    out = torch.empty((Bn, Hq, Nq, 128), dtype=torch.bfloat16, device="cuda")
    fws = torch.zeros(bnd.query_sizes(shape)["forward_workspace"] // 4, dtype=torch.int32, device="cuda")
    dump = torch.zeros(102400, dtype=torch.float32, device="cuda")
    dump[DBG_MODE] = mode
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
    return dict(
        s=d[DBG_S:DBG_S + 128 * TILE].reshape(128, TILE),
        p8=d[DBG_P8:DBG_P8 + 128 * 64].view(np.uint32).reshape(128, 64).view(np.uint8).reshape(128, TILE),
        part=d[DBG_PV:DBG_PV + 128 * 144].reshape(128, 144),
        m1=d[DBG_M1:DBG_M1 + 128], a1=d[DBG_A1:DBG_A1 + 128], d1=d[DBG_D1:DBG_D1 + 128],
        ro1=d[DBG_RO1:DBG_RO1 + 128 * 128].reshape(128, 128),
        dfin=d[DBG_DF:DBG_DF + 128], rcp=d[DBG_RCP:DBG_RCP + 128],
        out=out.view(torch.int16).cpu().numpy())


SHAPES = [
    (1, 1, 1, 128, 192, False),    # c1: one tile, 192 kept keys of 256
    (1, 1, 1, 128, 700, False),    # three tiles, the last ragged
    (1, 2, 1, 256, 256, True),     # the causal diagonal runs through the only tile of query tile 0
    (1, 1, 1, 100, 300, True),     # ragged rows, bottom-right causal offset: rows below 56 keep no key of tile 1
    (1, 1, 1, 128, 512, False)]    # two full tiles


@pytest.mark.parametrize("shape", SHAPES)
def test_intermediates_match_the_oracle(oracle_mod, dbg_lib, shape):
    Bn, Hq, Hkv, Nq, Nkv, causal = shape
    w = synth.workload("c1", B=Bn, Hq=Hq, Hkv=Hkv, Nq=Nq, Nkv=Nkv, causal=causal)
    q, k, v = synth.make_inputs(w, seed=500 + Nkv)
    got = _run_dump(dbg_lib, q, k, v, causal)
    ref = oracle_mod.prepare(q, k, v)
    acc_o, p8_o, part_o = oracle_mod.first_tile(ref, Nq, Nkv, causal, tile=TILE)
    rows, n = min(Nq, 128), min(Nkv, TILE)

    # QK: exact integers, every key of the tile (pad keys read zero codes)
    assert np.array_equal(got["s"][:rows], acc_o[:rows].astype(np.float32))

    # FP8 P: the same bytes
    diff = np.count_nonzero(got["p8"][:rows] != p8_o[:rows])
    assert diff == 0, f"{diff} P8 bytes differ"

    # PV partial of tile 0: the same products, summed in the tensor core's FP32 order
    po = oracle_mod.e4m3_to_f32(p8_o[:rows].reshape(-1)).reshape(rows, TILE).astype(np.float64)
    vv = np.zeros((TILE, 128))
    vv[:n] = oracle_mod.e4m3_to_f32(ref["v_codes"][0, 0, :n].reshape(-1)).reshape(n, 128)
    bound = 4e-6 * (np.abs(po) @ np.abs(vv)) + 1e-30
    assert np.all(np.abs(got["part"][:rows, :128].astype(np.float64) - part_o[:rows, :128]) <= bound)
    assert np.all(np.abs(got["part"][:rows, 128].astype(np.float64) - part_o[:rows, 128]) <= 4e-6 * po.sum(axis=1))
    assert not got["part"][:rows, 129:].any()

    # the end of the recurrence: d and its reciprocal
    st_end = oracle_mod.tile_state(ref, Nq, Nkv, causal, which=0, tile=TILE)
    np.testing.assert_allclose(got["dfin"][:rows], st_end["d_final"][:rows], rtol=2e-5)
    rcp_own = (np.float32(1) / got["dfin"][:rows].astype(np.float32)).astype(np.float32)
    assert np.array_equal(got["rcp"][:rows], rcp_own), "reciprocal is not the correctly rounded 1/d"
    np.testing.assert_allclose(got["rcp"][:rows], st_end["rcp"][:rows], rtol=2e-5)

    # the fix-up paths forced on every tile give the same bytes, so every
    # intermediate and the output are identical
    for mode in (1, 2):
        forced = _run_dump(dbg_lib, q, k, v, causal, mode)
        for key in ("s", "p8", "part", "m1", "a1", "d1", "ro1", "dfin", "rcp", "out"):
            assert np.array_equal(forced[key], got[key]), f"mode {mode}: {key} differs"

    # tile 1 (where the item has one): running maximum, alpha, d and RO after the outer update
    if Nkv <= TILE or (causal and min(127, Nq - 1) + (Nkv - Nq) < TILE):
        return
    st = oracle_mod.tile_state(ref, Nq, Nkv, causal, which=1, tile=TILE)
    vis = st["visited"][:rows]
    assert vis.any()
    assert np.array_equal(got["m1"][:rows][vis], st["m"][:rows][vis].astype(np.float32))
    np.testing.assert_allclose(got["a1"][:rows][vis], st["alpha"][:rows][vis], rtol=1e-6, atol=1e-30)
    np.testing.assert_allclose(got["d1"][:rows][vis], st["d"][:rows][vis], rtol=2e-5)
    ro_ref = st["ro"][:rows][vis]
    scale = np.abs(ro_ref).max(axis=1, keepdims=True) + 1e-30
    assert np.all(np.abs(got["ro1"][:rows][vis].astype(np.float64) - ro_ref) <= 2e-5 * scale)
    # rows that keep no key of tile 1 pass it unchanged: alpha = 1, nothing added
    if (~vis).any():
        assert np.all(got["a1"][:rows][~vis] == 1.0)
        np.testing.assert_allclose(got["d1"][:rows][~vis], st["d_final"][:rows][~vis], rtol=2e-5)
