"""CPU oracle of quantized exact attention with K smoothing (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU baseline use this package; the product path never imports it.
It shares no code with the CUDA library.  The arithmetic lives in
``sattn_oracle.c`` / ``attend_row.inc`` (plain C, compiled with gcc, OpenMP,
``-ffp-contract=off``); this module only builds it and marshals numpy arrays.

Functions follow the "Experiment Log" page (vortex_exact_attention), entries
"Phase 0 Import And Verification" (contract stages) and "Phase 1
State-Ownership Decision" (invariants); the readings taken where the page is
silent are stated in ``sattn_oracle.c``.

Parity status of each function (what pins it, see tests/test_oracle_*.py):
  bf16 / e4m3 codecs  pinned: torch's own converters, exhaustive tables
  prepare             pinned: quantiser invariants, constructed ties, exact
                      means, zero blocks, saturation
  forward_exact       pinned: brute-force FP64 softmax attention, shift
                      invariance of K smoothing
  forward             pinned: constant V, one-hot key, tile-size invariance,
                      accuracy against forward_exact, shares the pinned skeleton
  p8_codes            pinned: exhaustive E4M3 midpoints against exact rational
                      arithmetic, monotonicity, saturation, zeros
  tile_state          pinned: its last-tile state reproduces forward's output;
                      shares the per-row recurrence with forward
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HEAD_DIM = 128
QBLK = 32

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = [os.path.join(_HERE, "sattn_oracle.c"), os.path.join(_HERE, "attend_row.inc")]
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libsattn_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build/libsattn_oracle.so (gcc, OpenMP)."""
    newest = max(os.path.getmtime(p) for p in _SRC)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= newest:
        return _LIB_PATH
    os.makedirs(_OUT_DIR, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra", "-Wno-unused-parameter",
           _SRC[0], "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True, cwd=_HERE)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    i = ctypes.c_int
    lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f32.restype = ctypes.c_float
    lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
    lib.oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_f32.restype = ctypes.c_float
    lib.oracle_f32_to_e4m3.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_e4m3.restype = ctypes.c_uint8
    lib.oracle_prepare.argtypes = [i, i, i, i, i, i, P, P, P, P, P, P, P, P, P, P]
    lib.oracle_prepare.restype = i
    lib.oracle_forward.argtypes = [i, i, i, i, i, i, ctypes.c_float, i,
                                   P, P, P, P, P, P, P, P, i]
    lib.oracle_forward.restype = i
    lib.oracle_forward_rows.argtypes = [i, i, i, i, i, i, ctypes.c_float, i,
                                        P, P, P, P, P, P, ctypes.c_long, P, P, P, i]
    lib.oracle_forward_rows.restype = i
    lib.oracle_first_tile.argtypes = [i, i, i, i, i, i, ctypes.c_float, i, P, P, P, P, P, P, i, i, i, P, P, P]
    lib.oracle_first_tile.restype = i
    lib.oracle_forward_exact.argtypes = [i, i, i, i, i, i, ctypes.c_double, i,
                                         P, P, P, i, P]
    lib.oracle_forward_exact.restype = i
    lib.oracle_p8_codes.argtypes = [ctypes.c_long, P, P, P, P]
    lib.oracle_p8_codes.restype = i
    lib.oracle_exp2_rn.argtypes = [ctypes.c_long, P, P]
    lib.oracle_exp2_rn.restype = i
    lib.oracle_tile_state.argtypes = [i, i, i, i, i, i, ctypes.c_float, i, P, P, P, P, P, P, i, i, i, i, P, P]
    lib.oracle_tile_state.restype = i
    _lib = lib
    return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def pad32(n: int) -> int:
    return (n + QBLK - 1) // QBLK * QBLK


# --- storage formats ------------------------------------------------------

def f32_to_bf16(x) -> np.ndarray:
    lib = _load()
    x = np.asarray(x, dtype=np.float32)
    return np.array([lib.oracle_f32_to_bf16(float(v)) for v in x.reshape(-1)],
                    dtype=np.uint16).reshape(x.shape)


def bf16_to_f32(b) -> np.ndarray:
    lib = _load()
    b = np.asarray(b, dtype=np.uint16)
    return np.array([lib.oracle_bf16_to_f32(int(v)) for v in b.reshape(-1)],
                    dtype=np.float32).reshape(b.shape)


def f32_to_e4m3(x) -> np.ndarray:
    lib = _load()
    x = np.asarray(x, dtype=np.float32)
    return np.array([lib.oracle_f32_to_e4m3(float(v)) for v in x.reshape(-1)],
                    dtype=np.uint8).reshape(x.shape)


def e4m3_to_f32(c) -> np.ndarray:
    lib = _load()
    c = np.asarray(c, dtype=np.uint8)
    return np.array([lib.oracle_e4m3_to_f32(int(v)) for v in c.reshape(-1)],
                    dtype=np.float32).reshape(c.shape)


# --- preparation ------------------------------------------------------------

def prepare(q: np.ndarray, k: np.ndarray, v: np.ndarray, smooth: bool = True) -> dict:
    """BF16 bits q [B,Hq,Nq,128], k/v [B,Hkv,Nkv,128] -> codes and scales.

    Layouts: q_codes [B,Hq,Nq32,128] int8, q_scales [B,Hq,Nq32/32],
    k_codes [B,Hkv,Nkv32,128], k_scales [B,Hkv,Nkv32/32], k_mean [B,Hkv,128],
    v_codes [B,Hkv,Nkv,128] (token-major E4M3 bytes), v_scales [B,Hkv,128].
    """
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    B, Hq, Nq, D = q.shape
    _, Hkv, Nkv, _ = k.shape
    assert D == HEAD_DIM and k.shape == v.shape and k.shape[0] == B
    nq, nk = pad32(Nq), pad32(Nkv)
    out = dict(
        q_codes=np.empty((B, Hq, nq, D), np.int8), q_scales=np.empty((B, Hq, nq // QBLK), np.float32),
        k_codes=np.empty((B, Hkv, nk, D), np.int8), k_scales=np.empty((B, Hkv, nk // QBLK), np.float32),
        k_mean=np.empty((B, Hkv, D), np.float32),
        v_codes=np.empty((B, Hkv, Nkv, D), np.uint8), v_scales=np.empty((B, Hkv, D), np.float32))
    rc = lib.oracle_prepare(B, Hq, Hkv, Nq, Nkv, int(bool(smooth)), _ptr(q), _ptr(k), _ptr(v),
                            _ptr(out["q_codes"]), _ptr(out["q_scales"]), _ptr(out["k_codes"]),
                            _ptr(out["k_scales"]), _ptr(out["k_mean"]), _ptr(out["v_codes"]),
                            _ptr(out["v_scales"]))
    if rc != 0:
        raise ValueError("oracle_prepare: invalid shape")
    return out


# --- forward ----------------------------------------------------------------

def forward(prep: dict, Nq: int, Nkv: int, causal: bool, sm_scale: float = 0.0, tile: int = 256,
            rows: np.ndarray | None = None, nthreads: int = 0):
    """Quantised attention.  Returns (out_bf16_bits, out_f32).

    Without ``rows`` the outputs are [B,Hq,Nq,128]; with ``rows`` (flat
    indices (b*Hq + h)*Nq + i) they are [len(rows),128].
    """
    lib = _load()
    B, Hq = prep["q_codes"].shape[:2]
    Hkv = prep["k_codes"].shape[1]
    args = [_ptr(prep["q_codes"]), _ptr(prep["q_scales"]), _ptr(prep["k_codes"]),
            _ptr(prep["k_scales"]), _ptr(prep["v_codes"]), _ptr(prep["v_scales"])]
    if rows is None:
        ob = np.empty((B, Hq, Nq, HEAD_DIM), np.uint16)
        of = np.empty((B, Hq, Nq, HEAD_DIM), np.float32)
        rc = lib.oracle_forward(B, Hq, Hkv, Nq, Nkv, int(bool(causal)), float(sm_scale), tile,
                                *args, _ptr(ob), _ptr(of), nthreads)
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        ob = np.empty((rows.size, HEAD_DIM), np.uint16)
        of = np.empty((rows.size, HEAD_DIM), np.float32)
        rc = lib.oracle_forward_rows(B, Hq, Hkv, Nq, Nkv, int(bool(causal)), float(sm_scale), tile,
                                     *args, rows.size, _ptr(rows), _ptr(ob), _ptr(of), nthreads)
    if rc != 0:
        raise ValueError("oracle_forward: invalid shape or rows")
    return ob, of


def first_tile(prep: dict, Nq: int, Nkv: int, causal: bool, b: int = 0, h: int = 0, q0: int = 0,
               sm_scale: float = 0.0, tile: int = 256):
    """Intermediates of the first KV tile for query rows q0 .. q0 + 127 of
    (b, h): exact int32 QK accumulators [128, tile], P8 bytes [128, tile] and
    the tile's PV partial with its weight sum in column 128 [128, 129]."""
    lib = _load()
    B, Hq = prep["q_codes"].shape[:2]
    Hkv = prep["k_codes"].shape[1]
    acc = np.empty((128, tile), np.int32)
    p8 = np.empty((128, tile), np.uint8)
    part = np.empty((128, HEAD_DIM + 1), np.float32)
    rc = lib.oracle_first_tile(B, Hq, Hkv, Nq, Nkv, int(bool(causal)), float(sm_scale), tile,
                               _ptr(prep["q_codes"]), _ptr(prep["q_scales"]), _ptr(prep["k_codes"]),
                               _ptr(prep["k_scales"]), _ptr(prep["v_codes"]), _ptr(prep["v_scales"]),
                               b, h, q0, _ptr(acc), _ptr(p8), _ptr(part))
    if rc != 0:
        raise ValueError("oracle_first_tile: invalid shape or position")
    return acc, p8, part


def p8_codes(acc, sig, m) -> np.ndarray:
    """FP8 P bytes of elementwise (acc, sig, m): E4M3(fl(fl(exp2(fl(fl(acc * sig)
    - m))) * 448)) with a correctly rounded exp2 (the forward's P step)."""
    lib = _load()
    acc, sig, m = np.broadcast_arrays(np.asarray(acc, np.float32), np.asarray(sig, np.float32),
                                      np.asarray(m, np.float32))
    shape = acc.shape
    acc, sig, m = (np.ascontiguousarray(x.reshape(-1)) for x in (acc, sig, m))
    out = np.empty(acc.size, np.uint8)
    if lib.oracle_p8_codes(acc.size, _ptr(acc), _ptr(sig), _ptr(m), _ptr(out)) != 0:
        raise ValueError("oracle_p8_codes")
    return out.reshape(shape)


def exp2_rn(x) -> np.ndarray:
    """FP32 2^x, correctly rounded (the exp2 of the P step)."""
    lib = _load()
    x = np.ascontiguousarray(np.asarray(x, np.float32))
    out = np.empty_like(x)
    if lib.oracle_exp2_rn(x.size, _ptr(x), _ptr(out)) != 0:
        raise ValueError("oracle_exp2_rn")
    return out


def tile_state(prep: dict, Nq: int, Nkv: int, causal: bool, which: int, b: int = 0, h: int = 0, q0: int = 0,
               sm_scale: float = 0.0, tile: int = 256) -> dict:
    """Running state after KV tile ``which`` for query rows q0 .. q0 + 127 of
    (b, h): m, the tile's alpha, d and RO after it, the final d and 1/d, and
    whether each row visited that tile (arrays of 128 rows, RO [128, 128])."""
    lib = _load()
    B, Hq = prep["q_codes"].shape[:2]
    Hkv = prep["k_codes"].shape[1]
    st = np.zeros((128, 6), np.float64)
    ro = np.zeros((128, HEAD_DIM), np.float64)
    rc = lib.oracle_tile_state(B, Hq, Hkv, Nq, Nkv, int(bool(causal)), float(sm_scale), tile,
                               _ptr(prep["q_codes"]), _ptr(prep["q_scales"]), _ptr(prep["k_codes"]),
                               _ptr(prep["k_scales"]), _ptr(prep["v_codes"]), _ptr(prep["v_scales"]),
                               b, h, q0, which, _ptr(st), _ptr(ro))
    if rc != 0:
        raise ValueError("oracle_tile_state: invalid shape or position")
    return dict(m=st[:, 0], alpha=st[:, 1], d=st[:, 2], d_final=st[:, 3], rcp=st[:, 4],
                visited=st[:, 5] > 0, ro=ro)


def forward_exact(q: np.ndarray, k: np.ndarray, v: np.ndarray, causal: bool, smooth: bool,
                  sm_scale: float = 0.0, tile: int = 256) -> np.ndarray:
    """The same tiled recurrence in FP64 with every quantiser bypassed."""
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    B, Hq, Nq, D = q.shape
    _, Hkv, Nkv, _ = k.shape
    out = np.empty((B, Hq, Nq, D), np.float64)
    rc = lib.oracle_forward_exact(B, Hq, Hkv, Nq, Nkv, int(bool(causal)), float(sm_scale), tile,
                                  _ptr(q), _ptr(k), _ptr(v), int(bool(smooth)), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_forward_exact: invalid shape")
    return out
