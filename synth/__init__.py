"""Seeded synthetic inputs for the quantized-attention workloads.

This module only draws random numbers and stores them in the BF16 input
format.  It holds no step of the attention method (no smoothing, no
quantisation, no softmax), so both the CPU oracle and the CUDA path can take
their inputs from it without sharing any of the method's arithmetic.

Generator (stated so that anyone can re-implement it):

* SplitMix64 finaliser ``mix(z)`` (Steele, Lea & Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014) applied to a counter:
  draw ``n`` of stream ``s`` under seed ``S`` is
  ``mix(key + (n + 1) * 0x9E3779B97F4A7C15)`` with
  ``key = mix(S * 0x9E3779B97F4A7C15 + s + 1)`` (all arithmetic mod 2**64).
* A pair of draws (2k, 2k+1) gives two standard normals by Box-Muller:
  ``u1 = ((z0 >> 11) + 1) * 2**-53`` in (0, 1], ``u2 = (z1 >> 11) * 2**-53``,
  ``r = sqrt(-2 ln u1)``, normals ``r cos(2 pi u2)`` and ``r sin(2 pi u2)``.
* Values are formed in FP64 and rounded once to BF16, round-to-nearest-even.

Workloads (the five shapes the attention is measured on; every tensor is
[B, H, N, 128], K carries a per-channel bias that is shared over tokens):

===  ===============================================================
c1   B1 H1, Nq128 x Nkv192, non-causal, K bias N(0, 2^2)
c2   B1 H8, Nq=Nkv=1024, non-causal, K bias N(0, 2^2)
c3   B2 H32, Nq=Nkv=4000 (ragged), causal, K bias N(0, 2^2) and four
     outlier channels per (b, kv head) scaled x20 (noise and bias)
c4   B1 H16, Nq=Nkv=32760 (ragged), non-causal, K bias N(0, 3^2)
c5   B4, Hq32 / Hkv8 (GQA), Nq=Nkv=8192, causal, K bias N(0, 2^2)
===  ===============================================================

Seed of workload ``cN`` is ``20261202 * 16 + N``; streams are Q=0, K=1, V=2,
K bias=3, outlier channel choice=4.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

__all__ = ["Workload", "WORKLOADS", "workload", "seed_of", "normals", "to_bf16_bits",
           "bf16_bits_to_f32", "make_inputs", "outlier_channels", "STREAM_Q", "STREAM_K",
           "STREAM_V", "STREAM_BIAS", "STREAM_OUTLIER"]

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

STREAM_Q, STREAM_K, STREAM_V, STREAM_BIAS, STREAM_OUTLIER = 0, 1, 2, 3, 4
_CHUNK = 1 << 22  # normals per generation chunk (bounds host memory)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nkv: int
    causal: bool
    bias_std: float
    outliers: int = 0          # outlier channels per (b, kv head)
    outlier_scale: float = 20.0
    D: int = 128

    @property
    def index(self) -> int:
        return int(self.name[1:])

    @property
    def literal_ops(self) -> float:
        """4 * B * Hq * Nq * Nkv * D: the metric's operation count."""
        return 4.0 * self.B * self.Hq * self.Nq * self.Nkv * self.D

    @property
    def unmasked_pairs(self) -> int:
        """Number of (query, key) pairs that the mask keeps, per (b, q head)."""
        if not self.causal:
            return self.Nq * self.Nkv
        off = self.Nkv - self.Nq
        # row i keeps keys 0 .. min(i + off, Nkv - 1)
        return sum(min(i + off, self.Nkv - 1) + 1 for i in range(self.Nq))

    @property
    def algorithmic_ops(self) -> float:
        """4 * D per unmasked (query, key) pair: the work a causal mask leaves."""
        return 4.0 * self.B * self.Hq * self.unmasked_pairs * self.D


WORKLOADS = {
    "c1": Workload("c1", 1, 1, 1, 128, 192, False, 2.0),
    "c2": Workload("c2", 1, 8, 8, 1024, 1024, False, 2.0),
    "c3": Workload("c3", 2, 32, 32, 4000, 4000, True, 2.0, outliers=4),
    "c4": Workload("c4", 1, 16, 16, 32760, 32760, False, 3.0),
    "c5": Workload("c5", 4, 32, 8, 8192, 8192, True, 2.0),
}


def workload(name: str, **overrides) -> Workload:
    """A named workload, optionally with fields replaced (e.g. fewer heads)."""
    w = WORKLOADS[name]
    return dataclasses.replace(w, **overrides) if overrides else w


def seed_of(w: Workload) -> int:
    return 20261202 * 16 + w.index


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _stream_key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        k = np.array([seed], dtype=np.uint64) * _GOLDEN + np.uint64(stream + 1)
        return _mix(k)[0]


def normals(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Standard normals number ``start`` .. ``start + count - 1`` of one stream (FP64)."""
    if count <= 0:
        return np.zeros(0, dtype=np.float64)
    key = _stream_key(seed, stream)
    p0 = start // 2
    p1 = (start + count + 1) // 2
    out = np.empty(2 * (p1 - p0), dtype=np.float64)
    with np.errstate(over="ignore"):
        for a in range(p0, p1, _CHUNK // 2):
            b = min(p1, a + _CHUNK // 2)
            pair = np.arange(a, b, dtype=np.uint64)
            z0 = _mix(key + (np.uint64(2) * pair + np.uint64(1)) * _GOLDEN)
            z1 = _mix(key + (np.uint64(2) * pair + np.uint64(2)) * _GOLDEN)
            u1 = ((z0 >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
            u2 = (z1 >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
            r = np.sqrt(-2.0 * np.log(u1))
            t = 2.0 * math.pi * u2
            seg = out[2 * (a - p0): 2 * (b - p0)]
            seg[0::2] = r * np.cos(t)
            seg[1::2] = r * np.sin(t)
    off = start - 2 * p0
    return out[off: off + count]


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """FP64 values -> BF16 bit patterns (uint16), one rounding, nearest-even."""
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)                       # x = m * 2**e, 0.5 <= |m| < 1
    e = np.maximum(e, -125)                  # BF16 subnormal quantum is 2**-133
    q = np.ldexp(np.rint(np.ldexp(x, 8 - e)), e - 8)   # keep 8 significant bits
    f = q.astype(np.float32)                 # exact: q has at most 8 significant bits
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def outlier_channels(w: Workload, seed: int | None = None) -> np.ndarray:
    """[B, Hkv, outliers] distinct channel indices chosen from the outlier stream."""
    seed = seed_of(w) if seed is None else seed
    if w.outliers == 0:
        return np.zeros((w.B, w.Hkv, 0), dtype=np.int64)
    key = _stream_key(seed, STREAM_OUTLIER)
    n = w.B * w.Hkv * w.D
    with np.errstate(over="ignore"):
        z = _mix(key + (np.arange(n, dtype=np.uint64) + np.uint64(1)) * _GOLDEN)
    z = z.reshape(w.B, w.Hkv, w.D)
    return np.argsort(z, axis=-1, kind="stable")[..., : w.outliers]


def _fill_bf16(dst: np.ndarray, seed: int, stream: int, scale_fn=None) -> None:
    """Fill a flat uint16 array with BF16 normals, chunk by chunk."""
    n = dst.size
    for a in range(0, n, _CHUNK):
        b = min(n, a + _CHUNK)
        x = normals(seed, stream, a, b - a)
        if scale_fn is not None:
            x = scale_fn(x, a, b)
        dst[a:b] = to_bf16_bits(x)


def make_inputs(w: Workload, seed: int | None = None, kv_heads: tuple[int, int] | None = None):
    """BF16 bit patterns (uint16) ``q [B,Hq,Nq,D]``, ``k, v [B,Hkv,Nkv,D]``.

    ``kv_heads=(h0, h1)`` restricts generation to KV heads h0..h1-1 and the
    query heads that read them (GQA groups), with values identical to the
    full tensors' slices; used to draw bounded samples of large workloads.
    """
    seed = seed_of(w) if seed is None else seed
    B, Hq, Hkv, Nq, Nkv, D = w.B, w.Hq, w.Hkv, w.Nq, w.Nkv, w.D
    g = Hq // Hkv
    h0, h1 = (0, Hkv) if kv_heads is None else kv_heads
    bias = normals(seed, STREAM_BIAS, 0, B * Hkv * D).reshape(B, Hkv, D) * w.bias_std
    outl = outlier_channels(w, seed)
    q = np.empty((B, (h1 - h0) * g, Nq, D), dtype=np.uint16)
    k = np.empty((B, h1 - h0, Nkv, D), dtype=np.uint16)
    v = np.empty((B, h1 - h0, Nkv, D), dtype=np.uint16)
    for b in range(B):
        for hk in range(h0, h1):
            for hq in range(hk * g, (hk + 1) * g):
                base = ((b * Hq + hq) * Nq) * D
                q[b, hq - h0 * g].reshape(-1)[:] = to_bf16_bits(normals(seed, STREAM_Q, base, Nq * D))
            base = ((b * Hkv + hk) * Nkv) * D
            kk = normals(seed, STREAM_K, base, Nkv * D).reshape(Nkv, D) + bias[b, hk][None, :]
            if w.outliers:
                kk[:, outl[b, hk]] *= w.outlier_scale
            k[b, hk - h0].reshape(-1)[:] = to_bf16_bits(kk.reshape(-1))
            v[b, hk - h0].reshape(-1)[:] = to_bf16_bits(normals(seed, STREAM_V, base, Nkv * D))
    return q, k, v
