"""The forward's FP8 P step against the oracle, byte for byte ("Experiment
Log" page, entry "Phase 1 State-Ownership Decision": exact FP8 score bytes).

The kernel takes each byte from ex2.approx with a bracket of +-2^-21 and
recomputes the keys the bracket cannot decide with a correctly rounded exp2
(float-float arithmetic).  Both halves are checked through the kernel's own
device functions (test hooks of the C ABI): the bytes of groups of 32 keys on
random scores, on scores placed within a few FP32 ulps of every E4M3 rounding
midpoint, on scores whose byte depends on the product acc * sig being
rounded before the maximum is subtracted, and on masked keys; and the exp2
over a dense sample of [-40, 0.5].
"""
import numpy as np
import pytest
import torch

import quantized_exact_attention_smoothing_gb300 as sattn

pytestmark = pytest.mark.gpu


def _midpoint_scores():
    """FP32 values of dd = s2 - m within +-40 ulps of log2(M / 448) for every
    E4M3 rounding midpoint M below 448 (the points where the byte changes)."""
    codes = np.arange(0, 0x7f, dtype=np.uint8)
    vals = np.array([float(x) for x in torch.from_numpy(codes).view(torch.float8_e4m3fn).float()])
    vals = np.sort(vals)
    mids = 0.5 * (vals[1:] + vals[:-1])
    mids = mids[mids > 0]
    base = np.log2(mids / 448.0).astype(np.float32)
    offs = np.arange(-40, 41, dtype=np.int32)
    bits = base.view(np.int32)[:, None] + np.where(base[:, None] < 0, -offs, offs)[None, :]
    return bits.astype(np.int32).view(np.float32).reshape(-1)


def _check(oracle_mod, acc, sig, m):
    G = acc.shape[0]
    got = sattn.p8_codes_for_test(torch.from_numpy(acc).cuda(), torch.from_numpy(sig).cuda(),
                                  torch.from_numpy(m).cuda()).cpu().numpy()
    ref = oracle_mod.p8_codes(acc, sig[:, None], m[:, None])
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{len(bad)} of {G * 32} bytes differ, first {bad[:3].tolist()}"


def test_p8_bytes_at_every_e4m3_midpoint(oracle_mod):
    # sig = 1 and m = 0 make dd = acc, so the scores sit exactly where placed
    dd = _midpoint_scores()
    pad = (-dd.size) % 32
    dd = np.concatenate([dd, np.zeros(pad, np.float32)]).reshape(-1, 32)
    G = dd.shape[0]
    _check(oracle_mod, dd, np.ones(G, np.float32), np.zeros(G, np.float32))
    # the same scores through a nontrivial scale and maximum: acc * sig - m
    rng = np.random.default_rng(3)
    sig = rng.uniform(1e-4, 3e-4, G).astype(np.float32)
    m = rng.uniform(-5, 5, G).astype(np.float32)
    acc = np.rint((dd + m[:, None]) / sig[:, None]).astype(np.float32)
    _check(oracle_mod, acc, sig, m)


def test_p8_bytes_random_scores_and_masks(oracle_mod):
    rng = np.random.default_rng(11)
    G = 1 << 15
    acc = np.rint(rng.standard_normal((G, 32)) * 15000).astype(np.float32)
    sig = rng.uniform(5e-5, 2e-4, G).astype(np.float32)
    m = ((acc.max(axis=1) * sig).astype(np.float32) + rng.uniform(0, 2, G).astype(np.float32)).astype(np.float32)
    acc[rng.random((G, 32)) < 0.05] = -np.inf     # masked keys carry byte 0
    _check(oracle_mod, acc, sig, m)


def test_p8_bytes_keep_both_roundings_of_the_score(oracle_mod):
    # dd = fl(fl(acc * sig) - m): a fused multiply-add (one rounding) moves dd
    # by up to an ulp of the product, which near an E4M3 rounding midpoint
    # changes the byte.  Keep the scores where it does.
    rng = np.random.default_rng(17)
    n = 1 << 22
    acc = rng.integers(-(1 << 21) + 1, 1 << 21, n).astype(np.float32)
    sig = rng.uniform(1e-4, 3e-4, n).astype(np.float32)
    s2 = (acc.astype(np.float64) * sig.astype(np.float64)).astype(np.float32)
    m = (s2.astype(np.float64) + rng.uniform(0, 14, n)).astype(np.float32)
    fused = (acc.astype(np.longdouble) * sig.astype(np.longdouble) - m.astype(np.longdouble)).astype(np.float32)
    two = oracle_mod.p8_codes(acc, sig, m)
    sel = two != oracle_mod.p8_codes(fused, np.float32(1), np.float32(0))
    assert sel.sum() >= 50, "too few scores that tell the two roundings apart"
    _check(oracle_mod, np.repeat(acc[sel][:, None], 32, axis=1), sig[sel], m[sel])


def test_exp2_is_correctly_rounded(oracle_mod):
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.uniform(-40, 0.5, 1 << 20).astype(np.float32),
        np.arange(-(1 << 20), 1 << 20, dtype=np.int64).astype(np.float32) * np.float32(2 ** -20),
        -np.float32(2.0) ** -np.arange(1, 40, dtype=np.float32)]).astype(np.float32)
    got = sattn.exp2_for_test(torch.from_numpy(x).cuda()).cpu().numpy()
    ref = oracle_mod.exp2_rn(x)
    bad = np.argwhere(got.view(np.uint32) != ref.view(np.uint32))
    assert bad.size == 0, f"{len(bad)} values differ, first x = {x[bad[:3, 0]].tolist()}"
