"""Host-side checks of sattn_attention_small (no GPU): shapes other than one
query tile of one head with Nkv <= 1024 are refused before anything else."""
import ctypes

import pytest

import quantized_exact_attention_smoothing_gb300 as sattn


@pytest.mark.parametrize("B, Hq, Hkv, Nq, Nkv", [
    (2, 1, 1, 128, 192), (1, 2, 1, 128, 192), (1, 2, 2, 64, 64), (1, 1, 1, 129, 192), (1, 1, 1, 128, 1025)])
def test_small_path_refuses_other_shapes(B, Hq, Hkv, Nq, Nkv):
    lib = sattn.load_library()
    shape = sattn.make_shape(B, Hq, Hkv, Nq, Nkv, False)
    rc = lib.sattn_attention_small(ctypes.byref(shape), *([None] * 13))
    assert rc == 1   # SATTN_ERR_INVALID
    assert not sattn.small_shape_ok(B, Hq, Hkv, Nq, Nkv)


def test_small_shape_ok_accepts_the_single_head_case():
    assert sattn.small_shape_ok(1, 1, 1, 128, 192)
    assert sattn.small_shape_ok(1, 1, 1, 1, 1024)
