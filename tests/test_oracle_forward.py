"""Pins of the oracle's attention recurrence.

* The exact (FP64, quantisers bypassed) mode runs the same tiled skeleton as
  the quantised contract; it must equal brute-force softmax(Q K^T * scale) V
  computed with numpy (causal bottom-right mask, GQA, ragged lengths, any
  tile size), and K smoothing must not change it (shift invariance).
* The quantised mode: constant V reproduces V exactly, a dominant key selects
  its dequantised V row, the result does not depend on the tile size when the
  running max never changes, and it stays close to exact attention.
"""
import numpy as np
import pytest

import synth


def _bf(x):
    return synth.to_bf16_bits(np.asarray(x, dtype=np.float64))


def _f64(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def brute_attention(q, k, v, causal, scale=None):
    """softmax(q k^T * scale) v per head; causal keeps j <= i + (Nkv - Nq)."""
    B, Hq, Nq, D = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    out = np.empty_like(q)
    for b in range(B):
        for h in range(Hq):
            hk = h // (Hq // Hkv)
            s = q[b, h] @ k[b, hk].T * scale
            if causal:
                i = np.arange(Nq)[:, None]
                j = np.arange(Nkv)[None, :]
                s = np.where(j <= i + (Nkv - Nq), s, -np.inf)
            s = s - s.max(axis=1, keepdims=True)
            p = np.exp(s)
            out[b, h] = (p / p.sum(axis=1, keepdims=True)) @ v[b, hk]
    return out


CASES = [  # B, Hq, Hkv, Nq, Nkv, causal, tile
    (1, 1, 1, 128, 192, False, 128),
    (1, 2, 2, 37, 300, False, 64),
    (2, 4, 2, 70, 70, True, 32),
    (1, 4, 1, 50, 131, True, 128),      # causal with Nq < Nkv: bottom-right diagonal
    (1, 2, 1, 1, 1, False, 16),
    (1, 2, 2, 129, 129, True, 128),
    (1, 1, 1, 5, 5, True, 2),
]


@pytest.mark.parametrize("case", CASES)
def test_exact_mode_equals_brute_force_softmax(oracle_mod, case):
    B, Hq, Hkv, Nq, Nkv, causal, tile = case
    rng = np.random.default_rng(Nq * 7 + Nkv)
    q = rng.standard_normal((B, Hq, Nq, 128)) * 1.5
    k = rng.standard_normal((B, Hkv, Nkv, 128)) + 2.0 * rng.standard_normal((B, Hkv, 1, 128))
    v = rng.standard_normal((B, Hkv, Nkv, 128))
    got = oracle_mod.forward_exact(q, k, v, causal, smooth=False, tile=tile)
    ref = brute_attention(q, k, v, causal)
    assert np.abs(got - ref).max() <= 1e-12


@pytest.mark.parametrize("case", CASES[:4])
def test_exact_mode_shift_invariance_of_k_smoothing(oracle_mod, case):
    B, Hq, Hkv, Nq, Nkv, causal, tile = case
    rng = np.random.default_rng(3 + Nq)
    q = rng.standard_normal((B, Hq, Nq, 128))
    k = rng.standard_normal((B, Hkv, Nkv, 128)) + 3.0 * rng.standard_normal((B, Hkv, 1, 128))
    v = rng.standard_normal((B, Hkv, Nkv, 128))
    a = oracle_mod.forward_exact(q, k, v, causal, smooth=False, tile=tile)
    b = oracle_mod.forward_exact(q, k, v, causal, smooth=True, tile=tile)
    assert np.abs(a - b).max() <= 1e-12


def _quant(oracle_mod, q, k, v, causal, tile=128, smooth=True):
    p = oracle_mod.prepare(q, k, v, smooth=smooth)
    return p, oracle_mod.forward(p, q.shape[2], k.shape[2], causal, tile=tile)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_gives_that_constant_exactly(oracle_mod, causal):
    rng = np.random.default_rng(11)
    Nq, Nkv = 100, 300
    q = rng.standard_normal((1, 2, Nq, 128))
    k = rng.standard_normal((1, 1, Nkv, 128))
    # scores grow with the key index, so the running max rises in every tile
    # and every rescale factor alpha is below one
    q[..., 0] = 2.0
    k[..., 0] = np.linspace(-6, 6, Nkv)[None, None, :]
    v0 = _bf(rng.standard_normal(128))
    v = np.broadcast_to(synth.bf16_bits_to_f32(v0), (1, 1, Nkv, 128))
    for tile in (32, 64, 128):
        _, (ob, _) = _quant(oracle_mod, _bf(q), _bf(k), _bf(v), causal, tile)
        assert np.array_equal(ob, np.broadcast_to(v0, ob.shape)), tile


def test_dominant_key_selects_its_value_row(oracle_mod):
    rng = np.random.default_rng(12)
    Nq, Nkv, star = 40, 400, 263              # the dominant key sits in tile 2 of 4
    q = np.full((1, 1, Nq, 128), 4.0)
    k = rng.standard_normal((1, 1, Nkv, 128)) * 0.1
    k[0, 0, star] = 4.0
    v = rng.standard_normal((1, 1, Nkv, 128))
    p, (ob, of) = _quant(oracle_mod, _bf(q), _bf(k), _bf(v), False)
    row = oracle_mod.e4m3_to_f32(p["v_codes"][0, 0, star]).astype(np.float64) * p["v_scales"][0, 0]
    got = synth.bf16_bits_to_f32(ob[0, 0]).astype(np.float64)
    ulp = np.abs(row) * 2.0 ** -7
    assert np.all(np.abs(got - row[None, :]) <= ulp[None, :] + 1e-30)


def test_tile_size_invariance_when_running_max_is_fixed(oracle_mod):
    rng = np.random.default_rng(13)
    Nq, Nkv = 64, 512
    q = rng.standard_normal((1, 1, Nq, 128))
    k = rng.standard_normal((1, 1, Nkv, 128))
    v = rng.standard_normal((1, 1, Nkv, 128))
    q[..., 0] = 4.0
    k[0, 0, 0, 0] = 24.0          # key 0 (tile 0) holds every row's maximum score
    outs = []
    for tile in (16, 64, 128, 256):
        _, (_, of) = _quant(oracle_mod, _bf(q), _bf(k), _bf(v), False, tile)
        outs.append(of.astype(np.float64))
    for o in outs[1:]:
        # only the FP32 grouping of the PV sums differs between tilings
        assert np.abs(o - outs[0]).max() <= 1e-5 * np.abs(outs[0]).max()
    # the property is not vacuous: without a fixed maximum the tilings differ
    k2 = rng.standard_normal((1, 1, Nkv, 128))
    _, (_, a) = _quant(oracle_mod, _bf(q), _bf(k2), _bf(v), False, 16)
    _, (_, b) = _quant(oracle_mod, _bf(q), _bf(k2), _bf(v), False, 256)
    assert np.abs(a - b).max() > 1e-4


def _cos(a, b):
    a, b = a.ravel(), b.ravel()
    return float(a @ b / np.linalg.norm(a) / np.linalg.norm(b))


@pytest.mark.parametrize("case", CASES)
def test_quantised_mode_is_close_to_exact_attention(oracle_mod, case):
    B, Hq, Hkv, Nq, Nkv, causal, tile = case
    rng = np.random.default_rng(21 + Nq)
    q = _bf(rng.standard_normal((B, Hq, Nq, 128)))
    k = _bf(rng.standard_normal((B, Hkv, Nkv, 128)) + 2.0 * rng.standard_normal((B, Hkv, 1, 128)))
    v = _bf(rng.standard_normal((B, Hkv, Nkv, 128)))
    _, (_, of) = _quant(oracle_mod, q, k, v, causal, tile)
    ref = brute_attention(_f64(q), _f64(k), _f64(v), causal)
    for b in range(B):
        for h in range(Hq):
            for i in range(Nq):
                assert _cos(of[b, h, i], ref[b, h, i]) > 0.99, (b, h, i)
    assert _cos(of, ref) > 0.999


def test_smoothing_reduces_error_on_biased_k(oracle_mod):
    w = synth.workload("c1")
    q, k, v = synth.make_inputs(w)
    ref = brute_attention(_f64(q), _f64(k), _f64(v), False)
    _, (_, with_s) = _quant(oracle_mod, q, k, v, False, smooth=True)
    _, (_, without) = _quant(oracle_mod, q, k, v, False, smooth=False)
    assert np.abs(with_s - ref).max() < np.abs(without - ref).max()
    assert _cos(with_s, ref) > _cos(without, ref)


def test_single_key_returns_dequantised_value(oracle_mod):
    rng = np.random.default_rng(14)
    q = _bf(rng.standard_normal((1, 3, 7, 128)))
    k = _bf(rng.standard_normal((1, 1, 1, 128)))
    v = _bf(rng.standard_normal((1, 1, 1, 128)))
    p, (ob, _) = _quant(oracle_mod, q, k, v, False)
    row = oracle_mod.e4m3_to_f32(p["v_codes"][0, 0, 0]).astype(np.float64) * p["v_scales"][0, 0]
    got = synth.bf16_bits_to_f32(ob).astype(np.float64)
    assert np.all(np.abs(got - row) <= np.abs(row) * 2.0 ** -7 + 1e-30)


def test_row_subset_matches_full_forward(oracle_mod):
    w = synth.workload("c2", Hq=2, Hkv=2, Nq=300, Nkv=300, causal=True)
    q, k, v = synth.make_inputs(w)
    p = oracle_mod.prepare(q, k, v)
    full_b, full_f = oracle_mod.forward(p, w.Nq, w.Nkv, True)
    rows = np.array([0, 1, 299, 300, 457, 599])
    sb, sf = oracle_mod.forward(p, w.Nq, w.Nkv, True, rows=rows)
    assert np.array_equal(sb, full_b.reshape(-1, 128)[rows])
    assert np.array_equal(sf, full_f.reshape(-1, 128)[rows])


def test_forward_rejects_bad_shapes(oracle_mod):
    rng = np.random.default_rng(0)
    q = _bf(rng.standard_normal((1, 1, 9, 128)))
    k = _bf(rng.standard_normal((1, 1, 8, 128)))
    p = oracle_mod.prepare(q, k, k)
    with pytest.raises(ValueError):
        oracle_mod.forward(p, 9, 8, causal=True)       # causal needs Nq <= Nkv
    with pytest.raises(ValueError):
        oracle_mod.forward(p, 9, 8, causal=False, tile=0)


# --- first-tile intermediates (QK, m, FP8 P, PV of one tile) ----------------

@pytest.mark.parametrize("shape", [(1, 1, 1, 128, 192, False), (1, 2, 1, 100, 200, True),
                                   (2, 2, 2, 160, 256, True), (1, 1, 1, 128, 600, False)])
def test_first_tile_accumulators_are_exact_dot_products(oracle_mod, shape):
    B, Hq, Hkv, Nq, Nkv, causal = shape
    w = synth.workload("c1", B=B, Hq=Hq, Hkv=Hkv, Nq=Nq, Nkv=Nkv, causal=causal)
    q, k, v = synth.make_inputs(w, seed=300 + Nkv)
    prep = oracle_mod.prepare(q, k, v)
    b, h = B - 1, Hq - 1
    acc, p8, _ = oracle_mod.first_tile(prep, Nq, Nkv, causal, b=b, h=h)
    hk = h // (Hq // Hkv)
    n, rows = min(Nkv, 256), min(Nq, 128)
    ref = prep["q_codes"][b, h, :rows].astype(np.int64) @ prep["k_codes"][b, hk, :n].astype(np.int64).T
    assert np.array_equal(acc[:rows, :n], ref)
    assert not acc[:, n:].any() and not acc[rows:].any()
    # every row's largest kept weight is exp2(0) * 448 = 448 (byte 0x7e); masked keys carry 0
    last = np.arange(rows)[:, None] + (Nkv - Nq) if causal else np.full((rows, 1), Nkv - 1)
    kept = np.arange(256)[None, :] <= np.minimum(last, n - 1)
    assert np.all(p8[:rows].max(axis=1) == 0x7E)
    assert not p8[:rows][~kept].any()


@pytest.mark.parametrize("causal", [False, True])
def test_single_tile_intermediates_reproduce_the_forward(oracle_mod, causal):
    # with Nkv <= 256 the first tile is the whole recurrence: RO = partial,
    # d = its weight sum, out = bf16((RO * (1/d)) * s_v), equal to forward()
    w = synth.workload("c1", B=1, Hq=2, Hkv=1, Nq=200, Nkv=240, causal=causal)
    q, k, v = synth.make_inputs(w, seed=17)
    prep = oracle_mod.prepare(q, k, v)
    rb, _ = oracle_mod.forward(prep, w.Nq, w.Nkv, causal)
    for h in range(2):
        for q0 in (0, 128):
            _, _, part = oracle_mod.first_tile(prep, w.Nq, w.Nkv, causal, h=h, q0=q0)
            rows = min(128, w.Nq - q0)
            d = part[:rows, 128]
            r = (np.float32(1) / d).astype(np.float32)
            o = ((part[:rows, :128] * r[:, None]).astype(np.float32) * prep["v_scales"][0, 0][None, :]).astype(np.float32)
            got = oracle_mod.f32_to_bf16(o).reshape(rows, 128)
            assert np.array_equal(got, rb[0, h, q0:q0 + rows]), (h, q0)


# --- the state after a chosen tile (m, alpha, d, RO, reciprocal) -------------

def _scores(prep, b, h, hk, i, Nkv, c0):
    """fl(fl(acc * sig)) of every key for query row i, restated with numpy."""
    f32 = np.float32
    acc = prep["q_codes"][b, h, i].astype(np.int64) @ prep["k_codes"][b, hk, :Nkv].astype(np.int64).T
    sq = prep["q_scales"][b, h, i // 32]
    sk = prep["k_scales"][b, hk, np.arange(Nkv) // 32]
    sig = ((f32(sq) * sk).astype(f32) * f32(c0)).astype(f32)
    return (acc.astype(f32) * sig).astype(f32)


@pytest.mark.parametrize("causal", [False, True])
def test_tile_state_pins(oracle_mod, causal):
    w = synth.workload("c1", B=1, Hq=2, Hkv=1, Nq=130, Nkv=700, causal=causal)
    q, k, v = synth.make_inputs(w, seed=23)
    prep = oracle_mod.prepare(q, k, v)
    rb, rf = oracle_mod.forward(prep, w.Nq, w.Nkv, causal)
    c0 = np.float32(np.float32(1 / np.sqrt(128)) * np.float32(1.4426950408889634))
    T = 256
    ntiles = 3
    states = [oracle_mod.tile_state(prep, w.Nq, w.Nkv, causal, which=t, h=1) for t in range(ntiles)]
    for r in range(128):
        s2 = _scores(prep, 0, 1, 0, r, w.Nkv, c0)
        last = min(w.Nkv - 1, r + w.Nkv - w.Nq) if causal else w.Nkv - 1
        m_prev = -np.inf
        for t, st in enumerate(states):
            visited = T * t <= last
            assert bool(st["visited"][r]) == visited
            if not visited:
                continue
            # m: the maximum score over the kept keys of tiles 0 .. t
            m = np.float32(s2[:min(last, T * t + T - 1) + 1].max())
            assert st["m"][r] == m
            # alpha: exp2(m_prev - m), 0 on the first tile
            want = 0.0 if m_prev == -np.inf else float(oracle_mod.exp2_rn(np.float32(np.float32(m_prev) - m)).reshape(-1)[0])
            assert st["alpha"][r] == want
            m_prev = m
        # the final reciprocal is the correctly rounded 1 / d
        st = states[0]
        assert st["rcp"][r] == float(np.float32(1) / np.float32(st["d_final"][r]))
    # RO after the row's last tile, times the reciprocal and V scale, is the output
    for t, st in enumerate(states):
        rows = np.flatnonzero(st["visited"])
        for r in rows:
            last = min(w.Nkv - 1, r + w.Nkv - w.Nq) if causal else w.Nkv - 1
            if last // T != t:
                continue
            assert st["d"][r] == st["d_final"][r]
            o = ((st["ro"][r].astype(np.float32) * np.float32(st["rcp"][r])).astype(np.float32)
                 * prep["v_scales"][0, 0]).astype(np.float32)
            assert np.array_equal(o, rf[0, 1, r])


# --- the FP8 P step and its exp2 --------------------------------------------

def _exp2_rn_mp(x: float) -> np.float32:
    """2^x rounded to the nearest FP32 value, decided with 60-digit arithmetic."""
    import mpmath
    mpmath.mp.dps = 60
    e = mpmath.power(2, mpmath.mpf(float(x)))
    f = np.float32(float(e))
    cands = [f, np.nextafter(f, np.float32(np.inf)), np.nextafter(f, np.float32(-np.inf))]
    return min(cands, key=lambda c: abs(mpmath.mpf(float(c)) - e))


def _midpoint_dd(span=6):
    import torch
    codes = np.arange(0, 0x7f, dtype=np.uint8)
    vals = np.sort(torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64))
    mids = 0.5 * (vals[1:] + vals[:-1])
    base = np.log2(mids[mids > 0] / 448.0).astype(np.float32)
    offs = np.arange(-span, span + 1, dtype=np.int32)
    return (base.view(np.int32)[:, None] + offs[None, :]).view(np.float32).reshape(-1)


def test_exp2_rn_is_correctly_rounded_against_high_precision(oracle_mod):
    pytest.importorskip("mpmath")
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.uniform(-30, 0.5, 600).astype(np.float32), _midpoint_dd(2)])
    got = oracle_mod.exp2_rn(x)
    want = np.array([_exp2_rn_mp(v) for v in x], np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_p8_codes_against_an_independent_restatement(oracle_mod):
    # code = E4M3(fl(RN32(2^dd) * 448)), dd = fl(fl(acc * sig) - m); here the
    # exp2 comes from 60-digit arithmetic and the E4M3 rounding from torch's
    # converter, on scores placed within a few ulps of every rounding midpoint
    pytest.importorskip("mpmath")
    import torch
    dd = _midpoint_dd(3)
    p = np.array([_exp2_rn_mp(v) for v in dd], np.float32)
    y = (p * np.float32(448)).astype(np.float32)
    want = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle_mod.p8_codes(dd, np.float32(1), np.float32(0))
    assert np.array_equal(got, want)
    # the bytes do change at the midpoints: each band of placed scores holds two codes
    assert len(np.unique(got)) > 100


def test_p8_codes_basic_cases(oracle_mod):
    # the row maximum maps to 448 (0x7e); -inf scores (masked keys) to 0; far
    # below the maximum to 0; monotonic in the score
    assert oracle_mod.p8_codes(np.float32(5.0), np.float32(1), np.float32(5.0)) == 0x7E
    assert oracle_mod.p8_codes(np.float32(-np.inf), np.float32(1), np.float32(0)) == 0
    assert oracle_mod.p8_codes(np.float32(-30.0), np.float32(1), np.float32(0)) == 0
    dd = np.sort(np.random.default_rng(1).uniform(-20, 0, 5000).astype(np.float32))
    c = oracle_mod.p8_codes(dd, np.float32(1), np.float32(0)).astype(np.int32)
    assert np.all(np.diff(c) >= 0)
