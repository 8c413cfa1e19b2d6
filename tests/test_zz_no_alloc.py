"""sattn_prepare_noalloc against sattn_prepare, through the C ABI.

The allocation-free entry point serves callers that cannot hand the library
a workspace: a host program whose device memory belongs to an allocator it
does not expose, or a caller that may not call cudaMalloc because it
synchronises the whole device.  It keeps its scratch in a fixed array inside
the library, shared by every call on the device, so this test makes two calls
in a row (a large shape, then a smaller one that finds the first call's
leftovers in the array) and checks each against the workspace entry point.
The file is named to be collected last.
"""
import numpy as np
import pytest
import torch

import quantized_exact_attention_smoothing_gb300 as sattn
import synth
from helpers import to_device_bf16

pytestmark = pytest.mark.gpu

NAMES = ("q_codes", "q_scales", "k_codes", "k_scales", "k_mean", "v_codes", "v_scales")


def _inputs(w):
    q, k, v = synth.make_inputs(w)
    return to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)


def test_noalloc_prepare_matches_workspace_prepare_two_calls_in_a_row():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    for w in (synth.workload("c5"), synth.workload("c3", B=1, Hq=4, Hkv=4)):
        dq, dk, dv = _inputs(w)
        ref = sattn.prepare(dq, dk, dv, w.causal)
        got = sattn.prepare_noalloc(dq, dk, dv, w.causal)
        torch.cuda.synchronize()
        for n in NAMES:
            # codes and scales are bit-exact, the tolerance every prepare test uses
            assert torch.equal(got[n].view(torch.uint8), ref[n].view(torch.uint8)), (w.name, n)
        # the forward pass gives the same output from either preparation
        a = sattn.forward(ref)
        b = sattn.forward(got)
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), w.name


def test_noalloc_scratch_limit_is_reported():
    z = torch.zeros(16, dtype=torch.uint8, device="cuda")
    q = torch.zeros((1, 1, 8, 128), dtype=torch.bfloat16, device="cuda")
    # B * Hkv * ceil(Nkv / 64) = 16 * 1024 > 8192: more scratch than the array holds
    shape = sattn.make_shape(1, 16, 16, 8, 65536)
    lib = sattn.load_library()
    import ctypes
    p = ctypes.c_void_p(z.data_ptr())
    rc = lib.sattn_prepare_noalloc(ctypes.byref(shape), ctypes.c_void_p(q.data_ptr()), p, p, p, p, p,
                                   p, p, p, p, None)
    assert rc == 6, rc
