"""The C-ABI library builds, loads and exports every symbol include/sattn.h
declares; host-side argument checks answer without touching a GPU."""
import ctypes

import pytest

import quantized_exact_attention_smoothing_gb300 as sattn


@pytest.fixture(scope="module")
def lib():
    return sattn.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = sattn.declared_functions()
    assert set(names) >= {"sattn_query_sizes", "sattn_prepare", "sattn_forward",
                          "sattn_check_status", "sattn_attention_host", "sattn_status_string"}
    for n in names:
        assert hasattr(lib, n), n


def test_query_sizes_headline_shape():
    z = sattn.query_sizes(sattn.make_shape(4, 32, 8, 8192, 8192, True))
    assert z["q"] == 4 * 32 * 8192 * 128 * 2
    assert z["q_codes"] == 4 * 32 * 8192 * 128
    assert z["v_codes"] == 4 * 8 * 128 * 8192
    assert z["q_scales"] == 4 * 32 * 256 * 4
    # status block, then the FP16 copy of the K codes the tensor cores read
    assert z["forward_workspace"] == 256 + 4 * 8 * 8192 * 128 * 2
    assert "k_carrier" not in z
    assert all(v % 16 == 0 for v in z.values())


def test_query_sizes_ragged_padding():
    z = sattn.query_sizes(sattn.make_shape(1, 2, 1, 33, 129, False))
    assert z["q_codes"] == 2 * 64 * 128                    # 33 -> 64 (32-token blocks)
    assert z["k_codes"] == 160 * 128                       # 129 -> 160
    assert z["v_codes"] == 128 * 256                       # 129 -> 256 keys (128-key tiles)


@pytest.mark.parametrize("args", [
    (1, 3, 2, 8, 8, False),          # Hq % Hkv != 0
    (1, 1, 1, 0, 8, False),          # Nq < 1
    (1, 1, 1, 8, 0, False),          # Nkv < 1
    (1, 1, 1, 9, 8, True),           # causal with Nq > Nkv
    (0, 1, 1, 8, 8, False),          # B < 1
])
def test_invalid_shapes_rejected(args):
    with pytest.raises(sattn.SattnError) as e:
        sattn.query_sizes(sattn.make_shape(*args))
    assert e.value.code == 1


def test_head_dim_other_than_128_rejected(lib):
    s = sattn.make_shape(1, 1, 1, 8, 8)
    s.D = 64
    z = sattn.sattn_sizes()
    assert lib.sattn_query_sizes(ctypes.byref(s), ctypes.byref(z)) == 1


def test_null_and_misaligned_pointers_rejected_before_any_device_work(lib):
    s = sattn.make_shape(1, 1, 1, 8, 8)
    good = [ctypes.c_void_p(0x1000 * (i + 1)) for i in range(11)]
    args = list(good)
    args[3] = None
    assert lib.sattn_prepare(ctypes.byref(s), *args, None) == 1
    args = list(good)
    args[5] = ctypes.c_void_p(0x1008)
    assert lib.sattn_prepare(ctypes.byref(s), *args, None) == 2
    fwd = [ctypes.c_void_p(0x1000 * (i + 1)) for i in range(8)]
    fwd[6] = ctypes.c_void_p(0x2004)
    assert lib.sattn_forward(ctypes.byref(s), *fwd, None) == 2
    assert lib.sattn_check_status(None, None) == 1


def test_status_strings(lib):
    for code in range(6):
        assert lib.sattn_status_string(code)
    assert lib.sattn_status_string(99) == b"unknown status"


def test_kv_prepare_and_fused_forward_check_pointers_first(lib):
    s = sattn.make_shape(1, 1, 1, 8, 8)
    kv = [ctypes.c_void_p(0x1000 * (i + 1)) for i in range(8)]
    args = list(kv)
    args[2] = None                                   # k_codes
    assert lib.sattn_prepare_kv(ctypes.byref(s), *args, None) == 1
    args = list(kv)
    args[0] = ctypes.c_void_p(0x1001)                # k
    assert lib.sattn_prepare_kv(ctypes.byref(s), *args, None) == 2
    fwd = [ctypes.c_void_p(0x1000 * (i + 1)) for i in range(7)]
    args = list(fwd)
    args[0] = None                                   # q
    assert lib.sattn_forward_q_bf16(ctypes.byref(s), *args, None) == 1
    args = list(fwd)
    args[5] = ctypes.c_void_p(0x3008)                # out
    assert lib.sattn_forward_q_bf16(ctypes.byref(s), *args, None) == 2
    bad = sattn.make_shape(1, 3, 2, 8, 8)            # Hq % Hkv != 0
    assert lib.sattn_forward_q_bf16(ctypes.byref(bad), *fwd, None) == 1


def test_full_prepare_still_requires_q(lib):
    s = sattn.make_shape(1, 1, 1, 8, 8)
    args = [ctypes.c_void_p(0x1000 * (i + 1)) for i in range(11)]
    args[0] = None                                   # q
    assert lib.sattn_prepare(ctypes.byref(s), *args, None) == 1


def test_quantiser_sweep_hook_checks_arguments(lib):
    assert lib.sattn_test_int8_quantiser(0, 10, ctypes.c_void_p(0x1000), None) == 1
    assert lib.sattn_test_int8_quantiser(1, 0x7f81, ctypes.c_void_p(0x1000), None) == 1
    assert lib.sattn_test_int8_quantiser(5, 5, ctypes.c_void_p(0x1000), None) == 1
    assert lib.sattn_test_int8_quantiser(1, 10, None, None) == 1
    assert lib.sattn_test_int8_quantiser(1, 10, ctypes.c_void_p(0x1008), None) == 2


def test_graph_entry_points_check_arguments(lib):
    s = sattn.make_shape(1, 1, 1, 8, 8)
    bufs = [ctypes.c_void_p(0x1000 * (i + 1)) for i in range(13)]
    h = ctypes.c_void_p()
    assert lib.sattn_graph_create(ctypes.byref(s), *bufs, None) == 1          # no handle pointer
    args = list(bufs)
    args[11] = None                                                          # out
    assert lib.sattn_graph_create(ctypes.byref(s), *args, ctypes.byref(h)) == 1
    assert h.value is None
    args = list(bufs)
    args[0] = ctypes.c_void_p(0x1002)                                        # q misaligned
    assert lib.sattn_graph_create(ctypes.byref(s), *args, ctypes.byref(h)) == 2
    assert lib.sattn_graph_launch(None, None) == 1
    assert lib.sattn_graph_destroy(None) == 1


def test_binding_rejects_wrong_input_dtypes_and_shapes():
    # host tensors reach the shape checks of attention_host before any device work
    import torch
    q = torch.zeros((1, 2, 8, 128), dtype=torch.bfloat16)
    k = torch.zeros((1, 1, 8, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        sattn.attention_host(q.float(), k, k)
    with pytest.raises(ValueError):
        sattn.attention_host(q, k, torch.zeros((1, 1, 9, 128), dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        sattn.attention_host(torch.zeros((1, 3, 8, 128), dtype=torch.bfloat16), torch.zeros((1, 2, 8, 128), dtype=torch.bfloat16),
                             torch.zeros((1, 2, 8, 128), dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        sattn.attention_host(torch.zeros((1, 2, 8, 64), dtype=torch.bfloat16), k, k)


def _chunks(lib, shape, n_sm=152):
    bounds = (ctypes.c_int64 * 9)()
    n = ctypes.c_int()
    assert lib.sattn_test_host_chunks(ctypes.byref(shape), n_sm, bounds, ctypes.byref(n)) == 0
    b = list(bounds)[:n.value + 1]
    return [b[c + 1] - b[c] for c in range(n.value)], b


@pytest.mark.parametrize("dims, want", [
    ((4, 32, 8, 8192, 8192, True), [2, 3, 5, 6, 6, 5, 3, 2]),        # c5: ramp
    ((1, 16, 16, 32760, 32760, False), [2] * 8),                   # c4: ramp ends too small -> equal
    ((2, 32, 32, 4000, 4000, True), [10, 11, 11, 10, 11, 11]),     # c3: equal chunks of >= 10 heads
    ((1, 8, 8, 1024, 1024, False), [8]),                           # c2: too small to cut
    ((1, 1, 1, 128, 192, False), [1])])                            # c1
def test_host_chunk_plan(lib, dims, want):
    sizes, bounds = _chunks(lib, sattn.make_shape(*dims))
    assert sizes == want
    B, Hq, Hkv, Nq = dims[:4]
    units = B * Hkv
    assert bounds[0] == 0 and bounds[-1] == units and all(x > 0 for x in sizes)
    if len(sizes) > 1:   # every chunk holds at least two forward work items per SM
        items_per_unit = -(-Nq // 128) * (Hq // Hkv)
        assert min(sizes) * items_per_unit >= 2 * 152


def test_host_chunk_plan_properties_over_many_shapes(lib):
    rng = __import__("random").Random(3)
    for _ in range(300):
        Hkv = rng.choice([1, 2, 4, 8, 16, 32])
        g = rng.choice([1, 2, 4, 8])
        B, N = rng.randint(1, 6), rng.randint(1, 40000)
        for n_sm in (8, 152):
            sizes, bounds = _chunks(lib, sattn.make_shape(B, Hkv * g, Hkv, N, N, True), n_sm)
            assert 1 <= len(sizes) <= 8 and bounds[0] == 0 and bounds[-1] == B * Hkv
            assert all(x > 0 for x in sizes)
            if len(sizes) > 1:
                assert min(sizes) * (-(-N // 128) * g) >= 2 * n_sm

