"""Pins of the oracle's preparation stage: K smoothing, INT8 Q/K, FP8 V.

Each check follows from the definitions (per-block symmetric INT8 with
s = amax/127, per-channel E4M3 with s = amax/448, K minus its per-channel
mean over the sequence) without retyping the oracle's arithmetic: bounds,
constructed ties, exact special cases and the rounding error bound of the
summation.
"""
import numpy as np
import pytest

import synth

QBLK = 32
F32_EPS = 2.0 ** -24   # unit roundoff of FP32


def _bf(x):
    return synth.to_bf16_bits(np.asarray(x, dtype=np.float64))


def _f(bits):
    return synth.bf16_bits_to_f32(bits)


def _rand_inputs(rng, B, Hq, Hkv, Nq, Nkv, bias=2.0):
    q = _bf(rng.standard_normal((B, Hq, Nq, 128)))
    kk = rng.standard_normal((B, Hkv, Nkv, 128)) + bias * rng.standard_normal((B, Hkv, 1, 128))
    k = _bf(kk)
    v = _bf(rng.standard_normal((B, Hkv, Nkv, 128)))
    return q, k, v


def _check_int8_blocks(x, n, codes, scales):
    """Invariants of one head's per-block symmetric INT8 quantisation."""
    npad = codes.shape[0]
    assert npad % QBLK == 0 and npad >= n and npad - n < QBLK
    assert np.all(codes[n:] == 0)
    for b in range(npad // QBLK):
        blk = x[b * QBLK: min(n, (b + 1) * QBLK)].astype(np.float64)
        c = codes[b * QBLK: b * QBLK + blk.shape[0]].astype(np.float64)
        s = float(scales[b])
        amax = np.abs(blk).max()
        if amax == 0:
            assert s == 0 and np.all(c == 0)
            continue
        # the scale maps the block's largest magnitude to 127 (one FP32 rounding)
        assert abs(s * 127 - amax) <= amax * 2 * F32_EPS
        assert np.all(np.abs(c) <= 127)
        # the element of largest magnitude takes the extreme code
        idx = np.unravel_index(np.argmax(np.abs(blk)), blk.shape)
        assert c[idx] == np.sign(blk[idx]) * 127
        # round to nearest: reconstruction error at most half a step
        err = np.abs(blk - c * s)
        assert np.all(err <= 0.5 * s * (1 + 1e-5) + amax * 4 * F32_EPS)


@pytest.mark.parametrize("shape", [(1, 2, 2, 128, 192), (2, 4, 2, 37, 70), (1, 1, 1, 1, 1),
                                   (1, 2, 1, 95, 130)])
def test_int8_quantiser_invariants(oracle_mod, shape):
    B, Hq, Hkv, Nq, Nkv = shape
    rng = np.random.default_rng(10 + Nq)
    q, k, v = _rand_inputs(rng, *shape)
    p = oracle_mod.prepare(q, k, v)
    assert p["q_codes"].shape == (B, Hq, oracle_mod.pad32(Nq), 128)
    assert p["k_scales"].shape == (B, Hkv, oracle_mod.pad32(Nkv) // QBLK)
    for b in range(B):
        for h in range(Hq):
            _check_int8_blocks(_f(q[b, h]), Nq, p["q_codes"][b, h], p["q_scales"][b, h])
        for h in range(Hkv):
            ks = _f(k[b, h]) - p["k_mean"][b, h][None, :]      # FP32 subtraction
            _check_int8_blocks(ks, Nkv, p["k_codes"][b, h], p["k_scales"][b, h])


def test_int8_ties_round_to_even(oracle_mod):
    # amax 127 gives scale exactly 1.0, so codes are rint of the values themselves
    vals = np.array([127.0, 2.5, 3.5, -2.5, -0.5, 0.5, 1.5, -1.5, 126.5, -126.5, 0.25, 0.75])
    q = np.zeros((1, 1, 32, 128))
    q[0, 0, 0, : vals.size] = vals
    k = np.zeros((1, 1, 32, 128))
    p = oracle_mod.prepare(_bf(q), _bf(k), _bf(k))
    assert p["q_scales"][0, 0, 0] == np.float32(1.0)
    got = p["q_codes"][0, 0, 0, : vals.size].tolist()
    assert got == [127, 2, 4, -2, 0, 0, 2, -2, 126, -126, 0, 1]
    assert np.all(p["q_codes"][0, 0, 1:] == 0)


def test_zero_blocks_and_zero_channels(oracle_mod):
    q = np.zeros((1, 1, 64, 128))
    q[0, 0, 40, 3] = 1.0                 # block 1 is not zero, block 0 is
    z = np.zeros((1, 1, 50, 128))
    p = oracle_mod.prepare(_bf(q), _bf(z), _bf(z))
    assert p["q_scales"][0, 0].tolist()[0] == 0.0
    assert np.all(p["q_codes"][0, 0, :32] == 0)
    assert p["q_codes"][0, 0, 40, 3] == 127
    assert np.all(p["k_scales"] == 0) and np.all(p["k_codes"] == 0)
    assert np.all(p["v_scales"] == 0) and np.all(p["v_codes"] == 0)


@pytest.mark.parametrize("n", [1, 63, 64, 65, 4000])
def test_k_mean_of_constant_channels_is_exact(oracle_mod, n):
    rng = np.random.default_rng(n)
    consts = _f(_bf(rng.standard_normal(128) * 3))
    k = np.broadcast_to(consts, (1, 1, n, 128)).astype(np.float64)
    q = rng.standard_normal((1, 1, 8, 128))
    p = oracle_mod.prepare(_bf(q), _bf(k), _bf(k))
    assert np.array_equal(p["k_mean"][0, 0], consts)
    # smoothing removes the channel constants entirely
    assert np.all(p["k_codes"] == 0) and np.all(p["k_scales"] == 0)


@pytest.mark.parametrize("n", [31, 192, 4000, 32760])
def test_k_mean_within_summation_error_bound(oracle_mod, n):
    rng = np.random.default_rng(n)
    kk = rng.standard_normal((1, 1, n, 128)) * 2 + rng.standard_normal((1, 1, 1, 128)) * 3
    k = _bf(kk)
    p = oracle_mod.prepare(_bf(np.zeros((1, 1, 1, 128))), k, k)
    kf = _f(k[0, 0]).astype(np.float64)
    exact = kf.mean(axis=0)
    nchunks = (n + 63) // 64
    # chunked sequential FP32 sum: |error| <= (64 + nchunks) u sum|k|, plus the division
    bound = (64 + nchunks + 1) * F32_EPS * np.abs(kf).sum(axis=0) / n + F32_EPS * np.abs(exact)
    assert np.all(np.abs(p["k_mean"][0, 0] - exact) <= bound)


def test_smoothing_flag_and_zero_mean_after_smoothing(oracle_mod):
    rng = np.random.default_rng(5)
    q, k, v = _rand_inputs(rng, 1, 1, 1, 64, 256, bias=4.0)
    p0 = oracle_mod.prepare(q, k, v, smooth=False)
    p1 = oracle_mod.prepare(q, k, v, smooth=True)
    assert np.all(p0["k_mean"] == 0)
    # without smoothing the K codes quantise raw K (checked by the block invariants)
    _check_int8_blocks(_f(k[0, 0]), 256, p0["k_codes"][0, 0], p0["k_scales"][0, 0])
    # with smoothing the dequantised K has (nearly) zero channel means
    sk = np.repeat(p1["k_scales"][0, 0], QBLK)[:256, None]
    deq = p1["k_codes"][0, 0, :256] * sk
    assert np.abs(deq.mean(axis=0)).max() < 0.02
    # and the raw channel means are large, so the check is not vacuous
    assert np.abs(_f(k[0, 0]).mean(axis=0)).max() > 1.0


@pytest.mark.parametrize("n", [1, 33, 192, 1000])
def test_fp8_v_invariants(oracle_mod, n):
    rng = np.random.default_rng(100 + n)
    q, k, v = _rand_inputs(rng, 1, 2, 2, 8, n)
    v[0, 1, :, 5] = 0                                   # an all-zero channel
    p = oracle_mod.prepare(q, k, v)
    for h in range(2):
        vf = _f(v[0, h]).astype(np.float64)
        codes = p["v_codes"][0, h]
        sv = p["v_scales"][0, h].astype(np.float64)
        dec = oracle_mod.e4m3_to_f32(codes).astype(np.float64)
        amax = np.abs(vf).max(axis=0)
        for c in range(128):
            if amax[c] == 0:
                assert sv[c] == 0 and np.all(codes[:, c] == 0)
                continue
            assert abs(sv[c] * 448 - amax[c]) <= amax[c] * 2 * F32_EPS
            assert np.all(np.abs(dec[:, c]) <= 448)
            t = np.argmax(np.abs(vf[:, c]))
            assert codes[t, c] == (0x7E if vf[t, c] > 0 else 0xFE)
            # E4M3 round-to-nearest: relative error <= 2^-4 for normals,
            # absolute error <= 2^-10 (half the subnormal step) below 2^-6
            y = vf[:, c] / sv[c]
            err = np.abs(y - dec[:, c])
            assert np.all(err <= np.maximum(np.abs(y) * 2.0 ** -4, 2.0 ** -10) * (1 + 1e-5))


def test_prepare_rejects_bad_shapes(oracle_mod):
    z = np.zeros((1, 3, 8, 128), dtype=np.uint16)
    kv = np.zeros((1, 2, 8, 128), dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle_mod.prepare(z, kv, kv)            # Hq % Hkv != 0
