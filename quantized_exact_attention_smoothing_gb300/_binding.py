"""ctypes binding of libsattn.so: the same entry points as include/sattn.h.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI.  PyTorch supplies device memory and streams.  There
is no CPU fallback; if the library cannot be built or loaded, or a tensor is
not on a CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

from . import build as _build

HEAD_DIM = 128
QBLOCK = 32
KV_TILE = 256      # keys per KV tile of the forward pass (part of the numerical contract)
V_PAD = 128        # V codes are padded to a multiple of 128 keys

_SIZE_FIELDS = ["q", "k", "v", "q_codes", "q_scales", "k_codes", "k_scales", "k_mean",
                "v_codes", "v_scales", "out", "prepare_workspace", "forward_workspace", "arena"]


class sattn_shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("Nq", ctypes.c_int32), ("Nkv", ctypes.c_int32), ("D", ctypes.c_int32),
                ("causal", ctypes.c_int32), ("sm_scale", ctypes.c_float)]


class sattn_sizes(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in _SIZE_FIELDS]


STATUS = {0: "SATTN_OK", 1: "SATTN_ERR_INVALID", 2: "SATTN_ERR_MISALIGNED", 3: "SATTN_ERR_DEVICE",
          4: "SATTN_ERR_LAUNCH", 5: "SATTN_ERR_TIMEOUT", 6: "SATTN_ERR_SCRATCH_LIMIT"}

# Scratch held by sattn_prepare_noalloc (a fixed array in the library's device memory).
NOALLOC_SCRATCH_BYTES = 8 << 20


class SattnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)} ({_lib_status_string(code)})")


_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load_library(build: bool = True):
    """Load libsattn.so, building it first (nvcc) when missing or stale."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build() if build else _build.LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"libsattn.so not found at {path}; build it with "
                           "quantized_exact_attention_smoothing_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    SP = ctypes.POINTER(sattn_shape)
    lib.sattn_query_sizes.argtypes = [SP, ctypes.POINTER(sattn_sizes)]
    lib.sattn_prepare.argtypes = [SP] + [P] * 12
    lib.sattn_forward.argtypes = [SP] + [P] * 9
    lib.sattn_test_forward_withhold_v.argtypes = [SP] + [P] * 9
    lib.sattn_prepare_noalloc.argtypes = [SP] + [P] * 11
    lib.sattn_prepare_kv.argtypes = [SP] + [P] * 9
    lib.sattn_prepare_kv_onepass.argtypes = [SP] + [P] * 9
    lib.sattn_test_prepare_kv_onepass_withhold.argtypes = [SP] + [P] * 9
    lib.sattn_check_prepare_status.argtypes = [SP, P, P]
    lib.sattn_forward_q_bf16.argtypes = [SP] + [P] * 8
    lib.sattn_check_status.argtypes = [P, P]
    lib.sattn_test_int8_quantiser.argtypes = [ctypes.c_uint32, ctypes.c_uint32, P, P]
    lib.sattn_test_p8_codes.argtypes = [ctypes.c_int, P, P, P, P, P]
    lib.sattn_test_exp2.argtypes = [ctypes.c_int, P, P, P]
    lib.sattn_profile_events.argtypes = [P, P]
    lib.sattn_attention_small.argtypes = [SP] + [P] * 13
    lib.sattn_measure_mma_rate.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]
    lib.sattn_graph_create.argtypes = [SP] + [P] * 13 + [ctypes.POINTER(ctypes.c_void_p)]
    lib.sattn_test_host_chunks.argtypes = [SP, ctypes.c_int, ctypes.POINTER(ctypes.c_int64),
                                           ctypes.POINTER(ctypes.c_int)]
    lib.sattn_graph_launch.argtypes = [P, P]
    lib.sattn_graph_destroy.argtypes = [P]
    lib.sattn_attention_host.argtypes = [SP, P, P, P, P, P, ctypes.c_size_t, P]
    lib.sattn_status_string.argtypes = [ctypes.c_int]
    lib.sattn_status_string.restype = ctypes.c_char_p
    for name in ("sattn_query_sizes", "sattn_prepare", "sattn_forward", "sattn_check_status",
                 "sattn_attention_host", "sattn_prepare_noalloc", "sattn_prepare_kv", "sattn_forward_q_bf16",
                 "sattn_test_int8_quantiser", "sattn_graph_create", "sattn_graph_launch", "sattn_graph_destroy",
                 "sattn_test_host_chunks", "sattn_test_p8_codes", "sattn_test_exp2", "sattn_profile_events",
                 "sattn_attention_small", "sattn_measure_mma_rate", "sattn_prepare_kv_onepass",
                 "sattn_test_prepare_kv_onepass_withhold", "sattn_check_prepare_status"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _lib_status_string(code: int) -> str:
    try:
        return load_library(build=False).sattn_status_string(code).decode()
    except Exception:  # the message is best effort; the code is in the exception
        return "?"


def declared_functions(header: str | None = None) -> list[str]:
    """Names of the functions include/sattn.h declares."""
    header = header or os.path.join(_build.ROOT, "include", "sattn.h")
    with open(header) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(sattn_\w+)\s*\(", text, re.M)))


def make_shape(B, Hq, Hkv, Nq, Nkv, causal=False, sm_scale=0.0) -> sattn_shape:
    return sattn_shape(B, Hq, Hkv, Nq, Nkv, HEAD_DIM, int(bool(causal)), float(sm_scale))


def query_sizes(shape: sattn_shape) -> dict:
    z = sattn_sizes()
    rc = load_library().sattn_query_sizes(ctypes.byref(shape), ctypes.byref(z))
    if rc != 0:
        raise SattnError(rc, "sattn_query_sizes")
    return {n: getattr(z, n) for n in _SIZE_FIELDS}


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need_cuda(*ts: torch.Tensor):
    for t in ts:
        if not t.is_cuda:
            raise ValueError("libsattn runs on CUDA tensors only (no CPU path)")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def _need_inputs(q: torch.Tensor | None, k: torch.Tensor, v: torch.Tensor):
    """BF16 [B, H, N, 128] inputs of one problem: q [B, Hq, Nq, 128] (if given),
    k and v [B, Hkv, Nkv, 128] with the same shape."""
    ts = (k, v) if q is None else (q, k, v)
    for t in ts:
        if t.dtype != torch.bfloat16 or t.dim() != 4 or t.shape[-1] != HEAD_DIM:
            raise ValueError("inputs must be BF16 tensors of shape [B, H, N, 128]")
    if k.shape != v.shape:
        raise ValueError("k and v must have the same shape")
    if q is not None and (q.shape[0] != k.shape[0] or q.shape[1] % k.shape[1] != 0):
        raise ValueError("q [B, Hq, Nq, 128] must share B with k, and Hq must be a multiple of Hkv")


def _empty(nbytes: int, device, dtype=torch.uint8) -> torch.Tensor:
    n = max(1, nbytes // torch.empty(0, dtype=dtype).element_size())
    return torch.empty(n, dtype=dtype, device=device)


def prepare_buffers(shape: sattn_shape, device, with_q: bool = True) -> dict:
    """Device buffers for sattn_prepare's outputs (without the Q codes and
    scales when with_q is false: sattn_prepare_kv), shaped as documented."""
    B, Hq, Hkv, Nq, Nkv = shape.B, shape.Hq, shape.Hkv, shape.Nq, shape.Nkv
    nq32 = -(-Nq // QBLOCK) * QBLOCK
    nk32 = -(-Nkv // QBLOCK) * QBLOCK
    nk128 = -(-Nkv // V_PAD) * V_PAD
    z = query_sizes(shape)
    buf = dict(
        k_codes=torch.empty((B, Hkv, nk32, HEAD_DIM), dtype=torch.int8, device=device),
        k_scales=torch.empty((B, Hkv, nk32 // QBLOCK), dtype=torch.float32, device=device),
        k_mean=torch.empty((B, Hkv, HEAD_DIM), dtype=torch.float32, device=device),
        v_codes=torch.empty((B, Hkv, HEAD_DIM, nk128), dtype=torch.uint8, device=device),
        v_scales=torch.empty((B, Hkv, HEAD_DIM), dtype=torch.float32, device=device),
        workspace=_empty(z["prepare_workspace"], device),
    )
    if with_q:
        buf["q_codes"] = torch.empty((B, Hq, nq32, HEAD_DIM), dtype=torch.int8, device=device)
        buf["q_scales"] = torch.empty((B, Hq, nq32 // QBLOCK), dtype=torch.float32, device=device)
    return buf


def prepare(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
            sm_scale: float = 0.0, buffers: dict | None = None, stream=None) -> dict:
    """sattn_prepare on BF16 device tensors q [B,Hq,Nq,128], k/v [B,Hkv,Nkv,128]."""
    _need_cuda(q, k, v)
    _need_inputs(q, k, v)
    B, Hq, Nq, _ = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    shape = make_shape(B, Hq, Hkv, Nq, Nkv, causal, sm_scale)
    buf = buffers if buffers is not None else prepare_buffers(shape, q.device)
    rc = load_library().sattn_prepare(
        ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(buf["q_codes"]), _ptr(buf["q_scales"]),
        _ptr(buf["k_codes"]), _ptr(buf["k_scales"]), _ptr(buf["k_mean"]),
        _ptr(buf["v_codes"]), _ptr(buf["v_scales"]), _ptr(buf["workspace"]), _stream(stream))
    if rc != 0:
        raise SattnError(rc, "sattn_prepare")
    buf["shape"] = shape
    return buf


def prepare_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
                    sm_scale: float = 0.0, buffers: dict | None = None, stream=None) -> dict:
    """sattn_prepare_noalloc: as prepare(), without a workspace.

    For callers that cannot give the library scratch memory (their device
    memory belongs to an allocator they do not expose, or they may not call
    cudaMalloc because it synchronises the device).  The library keeps the
    scratch in a fixed 8 MiB array of its own device memory, shared by every
    call on a device: calls that may overlap on the GPU race on it.  Shapes
    with B * Hkv * ceil(Nkv / 64) > 8192 raise SattnError
    (SATTN_ERR_SCRATCH_LIMIT).  The output buffers (``buffers``) are still
    the caller's; without them this wrapper allocates them with PyTorch.
    """
    _need_cuda(q, k, v)
    _need_inputs(q, k, v)
    B, Hq, Nq, _ = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    shape = make_shape(B, Hq, Hkv, Nq, Nkv, causal, sm_scale)
    buf = buffers if buffers is not None else prepare_buffers(shape, q.device)
    rc = load_library().sattn_prepare_noalloc(
        ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(buf["q_codes"]), _ptr(buf["q_scales"]),
        _ptr(buf["k_codes"]), _ptr(buf["k_scales"]), _ptr(buf["k_mean"]),
        _ptr(buf["v_codes"]), _ptr(buf["v_scales"]), _stream(stream))
    if rc != 0:
        raise SattnError(rc, "sattn_prepare_noalloc")
    buf["shape"] = shape
    return buf


def forward(prep: dict, out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
            stream=None) -> torch.Tensor:
    """sattn_forward on the buffers returned by prepare(); returns BF16 [B,Hq,Nq,128]."""
    shape = prep["shape"]
    dev = prep["q_codes"].device
    if out is None:
        out = torch.empty((shape.B, shape.Hq, shape.Nq, HEAD_DIM), dtype=torch.bfloat16, device=dev)
    if workspace is None:
        workspace = prep.get("forward_workspace")
        if workspace is None:
            workspace = _empty(query_sizes(shape)["forward_workspace"], dev)
            prep["forward_workspace"] = workspace
    _need_cuda(out, workspace)
    rc = load_library().sattn_forward(
        ctypes.byref(shape), _ptr(prep["q_codes"]), _ptr(prep["q_scales"]), _ptr(prep["k_codes"]),
        _ptr(prep["k_scales"]), _ptr(prep["v_codes"]), _ptr(prep["v_scales"]), _ptr(out),
        _ptr(workspace), _stream(stream))
    if rc != 0:
        raise SattnError(rc, "sattn_forward")
    return out


SMALL_MAX_NKV = 1024


def small_shape_ok(B: int, Hq: int, Hkv: int, Nq: int, Nkv: int) -> bool:
    """Whether sattn_attention_small takes this shape (one query tile of one head)."""
    return B == 1 and Hq == 1 and Hkv == 1 and Nq <= 128 and Nkv <= SMALL_MAX_NKV


def attention_small(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
                    sm_scale: float = 0.0, buffers: dict | None = None, out: torch.Tensor | None = None,
                    workspace: torch.Tensor | None = None, stream=None) -> tuple:
    """sattn_attention_small: preparation and attention in one launch for a
    single query tile of one head.  Returns (out, buffers); the buffers hold
    what prepare() would write."""
    _need_cuda(q, k, v)
    _need_inputs(q, k, v)
    B, Hq, Nq, _ = q.shape
    _, Hkv, Nkv, _ = k.shape
    shape = make_shape(B, Hq, Hkv, Nq, Nkv, causal, sm_scale)
    if buffers is None:
        buffers = prepare_buffers(shape, q.device)
    if out is None:
        out = torch.empty((B, Hq, Nq, HEAD_DIM), dtype=torch.bfloat16, device=q.device)
    if workspace is None:
        workspace = _empty(query_sizes(shape)["forward_workspace"], q.device)
    _need_cuda(out, workspace)
    rc = load_library().sattn_attention_small(
        ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(buffers["q_codes"]), _ptr(buffers["q_scales"]),
        _ptr(buffers["k_codes"]), _ptr(buffers["k_scales"]), _ptr(buffers["k_mean"]), _ptr(buffers["v_codes"]),
        _ptr(buffers["v_scales"]), _ptr(out), _ptr(workspace), _stream(stream))
    if rc != 0:
        raise SattnError(rc, "sattn_attention_small")
    buffers["forward_workspace"] = workspace
    return out, buffers


def prepare_kv_onepass(k: torch.Tensor, v: torch.Tensor, Hq: int, Nq: int, causal: bool = False,
                       sm_scale: float = 0.0, buffers: dict | None = None, stream=None,
                       _withhold_for_test: bool = False) -> dict:
    """sattn_prepare_kv_onepass: prepare_kv() as one cooperative kernel launch
    (statistics, per-head mean and V scales, quantisers, separated by grid
    barriers); the same bytes.  check_prepare_status() reads its status."""
    _need_cuda(k, v)
    _need_inputs(None, k, v)
    B, Hkv, Nkv, _ = k.shape
    shape = make_shape(B, Hq, Hkv, Nq, Nkv, causal, sm_scale)
    if buffers is None:
        buffers = prepare_buffers(shape, k.device, with_q=False)
    lib = load_library()
    fn = lib.sattn_test_prepare_kv_onepass_withhold if _withhold_for_test else lib.sattn_prepare_kv_onepass
    rc = fn(ctypes.byref(shape), _ptr(k), _ptr(v), _ptr(buffers["k_codes"]), _ptr(buffers["k_scales"]),
            _ptr(buffers["k_mean"]), _ptr(buffers["v_codes"]), _ptr(buffers["v_scales"]),
            _ptr(buffers["workspace"]), _stream(stream))
    if rc != 0:
        raise SattnError(rc, "sattn_prepare_kv_onepass")
    buffers["shape"] = shape
    return buffers


def check_prepare_status(buffers: dict, stream=None) -> int:
    """sattn_check_prepare_status on the buffers of prepare_kv_onepass()."""
    return load_library().sattn_check_prepare_status(ctypes.byref(buffers["shape"]), _ptr(buffers["workspace"]),
                                                     _stream(stream))


def prepare_kv(k: torch.Tensor, v: torch.Tensor, Hq: int, Nq: int, causal: bool = False,
               sm_scale: float = 0.0, buffers: dict | None = None, stream=None) -> dict:
    """sattn_prepare_kv: the K and V part of prepare(), for forward_q_bf16.

    The shape needs the query side too (Hq, Nq): it is checked here and
    kept with the buffers for the forward call.  The Q entries of the
    returned buffers are absent.
    """
    _need_cuda(k, v)
    _need_inputs(None, k, v)
    B, Hkv, Nkv, _ = k.shape
    shape = make_shape(B, Hq, Hkv, Nq, Nkv, causal, sm_scale)
    if buffers is None:
        buffers = prepare_buffers(shape, k.device, with_q=False)
    rc = load_library().sattn_prepare_kv(
        ctypes.byref(shape), _ptr(k), _ptr(v), _ptr(buffers["k_codes"]), _ptr(buffers["k_scales"]),
        _ptr(buffers["k_mean"]), _ptr(buffers["v_codes"]),
        _ptr(buffers["v_scales"]), _ptr(buffers["workspace"]), _stream(stream))
    if rc != 0:
        raise SattnError(rc, "sattn_prepare_kv")
    buffers["shape"] = shape
    return buffers


def forward_q_bf16(q: torch.Tensor, prep: dict, out: torch.Tensor | None = None,
                   workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """sattn_forward_q_bf16: the forward pass that quantises the BF16 Q itself,
    on the K/V buffers of prepare_kv() (or prepare()).  Same output bytes as
    forward() on prepare()'s codes."""
    shape = prep["shape"]
    _need_cuda(q)
    if tuple(q.shape) != (shape.B, shape.Hq, shape.Nq, HEAD_DIM) or q.dtype != torch.bfloat16:
        raise ValueError("q must be BF16 [B, Hq, Nq, 128] of the prepared shape")
    dev = q.device
    if out is None:
        out = torch.empty((shape.B, shape.Hq, shape.Nq, HEAD_DIM), dtype=torch.bfloat16, device=dev)
    if workspace is None:
        workspace = prep.get("forward_workspace")
        if workspace is None:
            workspace = _empty(query_sizes(shape)["forward_workspace"], dev)
            prep["forward_workspace"] = workspace
    _need_cuda(out, workspace)
    rc = load_library().sattn_forward_q_bf16(
        ctypes.byref(shape), _ptr(q), _ptr(prep["k_codes"]), _ptr(prep["k_scales"]), _ptr(prep["v_codes"]),
        _ptr(prep["v_scales"]), _ptr(out), _ptr(workspace), _stream(stream))
    if rc != 0:
        raise SattnError(rc, "sattn_forward_q_bf16")
    return out


def forward_withhold_v_for_test(prep: dict, out: torch.Tensor | None = None,
                                workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """sattn_test_forward_withhold_v: a forward launch that loads no V tile, so
    its bounded waits run out (about one second) and check_status() reports
    SATTN_ERR_TIMEOUT.  Test hook for failure detection; `out` is undefined."""
    shape = prep["shape"]
    dev = prep["q_codes"].device
    if out is None:
        out = torch.empty((shape.B, shape.Hq, shape.Nq, HEAD_DIM), dtype=torch.bfloat16, device=dev)
    if workspace is None:
        workspace = prep.get("forward_workspace")
        if workspace is None:
            workspace = _empty(query_sizes(shape)["forward_workspace"], dev)
            prep["forward_workspace"] = workspace
    _need_cuda(out, workspace)
    rc = load_library().sattn_test_forward_withhold_v(
        ctypes.byref(shape), _ptr(prep["q_codes"]), _ptr(prep["q_scales"]), _ptr(prep["k_codes"]),
        _ptr(prep["k_scales"]), _ptr(prep["v_codes"]), _ptr(prep["v_scales"]), _ptr(out),
        _ptr(workspace), _stream(stream))
    if rc != 0:
        raise SattnError(rc, "sattn_test_forward_withhold_v")
    return out


def int8_quantiser_sweep_for_test(amax_lo: int = 1, amax_hi: int = 0x7f80, device="cuda") -> tuple[int, int, int]:
    """sattn_test_int8_quantiser: (mismatches, tie decisions, last mismatch) of
    the INT8 quantiser against IEEE division over BF16 blocks (test hook)."""
    res = torch.zeros(4, dtype=torch.int64, device=device)
    rc = load_library().sattn_test_int8_quantiser(amax_lo, amax_hi, _ptr(res), _stream(None))
    if rc != 0:
        raise SattnError(rc, "sattn_test_int8_quantiser")
    bad, near, last = (int(v) for v in res[:3].cpu())
    return bad, near, last


def p8_codes_for_test(acc: torch.Tensor, sig: torch.Tensor, m: torch.Tensor) -> torch.Tensor:
    """sattn_test_p8_codes: the forward's FP8 P bytes for groups of 32 keys
    (acc [G, 32], sig [G], m [G], FP32 CUDA tensors); returns uint8 [G, 32]."""
    _need_cuda(acc, sig, m)
    G = acc.shape[0]
    if acc.dtype != torch.float32 or tuple(acc.shape) != (G, 32) or sig.shape != (G,) or m.shape != (G,):
        raise ValueError("acc [G, 32], sig [G], m [G] FP32")
    out = torch.empty((G, 32), dtype=torch.uint8, device=acc.device)
    rc = load_library().sattn_test_p8_codes(G, _ptr(acc), _ptr(sig), _ptr(m), _ptr(out), _stream(None))
    if rc != 0:
        raise SattnError(rc, "sattn_test_p8_codes")
    return out


def exp2_for_test(x: torch.Tensor) -> torch.Tensor:
    """sattn_test_exp2: the forward's correctly rounded 2^x (FP32 CUDA tensor)."""
    _need_cuda(x)
    if x.dtype != torch.float32:
        raise ValueError("x must be FP32")
    out = torch.empty_like(x)
    rc = load_library().sattn_test_exp2(x.numel(), _ptr(x), _ptr(out), _stream(None))
    if rc != 0:
        raise SattnError(rc, "sattn_test_exp2")
    return out


def measure_mma_rate(kind: str, n: int, iters: int = 4096) -> dict:
    """sattn_measure_mma_rate: tcgen05.mma throughput for kind "f16" (A and B
    in shared memory) or "f8" (E4M3, A in tensor memory), M = 128, N = n."""
    k = {"f16": 0, "f8": 1}[kind]
    f, t = ctypes.c_double(), ctypes.c_double()
    rc = load_library().sattn_measure_mma_rate(k, n, iters, ctypes.byref(f), ctypes.byref(t))
    if rc != 0:
        raise SattnError(rc, "sattn_measure_mma_rate")
    return {"kind": kind, "n": n, "flop_per_clk_sm": f.value, "tflops": t.value}


def profile_events(before=None, after=None) -> None:
    """sattn_profile_events: while set, each forward records the two
    torch.cuda.Event objects (created with enable_timing=True) just before and
    just after its attention kernel; call with no arguments to stop."""
    if (before is None) != (after is None):
        raise ValueError("give both events or neither")
    handles = []
    for ev in (before, after):
        if ev is None:
            handles.append(None)
            continue
        if ev.cuda_event == 0:   # torch creates the CUDA event at its first record
            ev.record()
        handles.append(ctypes.c_void_p(ev.cuda_event))
    rc = load_library().sattn_profile_events(*handles)
    if rc != 0:
        raise SattnError(rc, "sattn_profile_events")


class Graph:
    """sattn_graph_*: prepare + forward on fixed buffers recorded as one CUDA
    graph (the small-shape latency path).  q, k, v are the device tensors the
    graph reads: fill them in place and call launch() for each step.  The
    preparation buffers (``buffers``, as from prepare_buffers), ``out`` and
    ``workspace`` are allocated here unless given."""

    def __init__(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
                 sm_scale: float = 0.0, buffers: dict | None = None, out: torch.Tensor | None = None,
                 workspace: torch.Tensor | None = None):
        _need_cuda(q, k, v)
        _need_inputs(q, k, v)
        B, Hq, Nq, _ = q.shape
        shape = make_shape(B, Hq, k.shape[1], Nq, k.shape[2], causal, sm_scale)
        dev = q.device
        prep = buffers if buffers is not None else prepare_buffers(shape, dev)
        self.out = out if out is not None else torch.empty((B, Hq, Nq, HEAD_DIM), dtype=torch.bfloat16, device=dev)
        self.workspace = workspace if workspace is not None else _empty(query_sizes(shape)["forward_workspace"], dev)
        self.buffers = prep
        self._keep = (q, k, v)   # the graph holds their addresses
        self.shape = shape
        handle = ctypes.c_void_p()
        rc = load_library().sattn_graph_create(
            ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(prep["q_codes"]), _ptr(prep["q_scales"]),
            _ptr(prep["k_codes"]), _ptr(prep["k_scales"]), _ptr(prep["k_mean"]),
            _ptr(prep["v_codes"]), _ptr(prep["v_scales"]), _ptr(prep["workspace"]), _ptr(self.out),
            _ptr(self.workspace), ctypes.byref(handle))
        if rc != 0:
            raise SattnError(rc, "sattn_graph_create")
        self._handle = handle

    def launch(self, stream=None) -> torch.Tensor:
        rc = load_library().sattn_graph_launch(self._handle, _stream(stream))
        if rc != 0:
            raise SattnError(rc, "sattn_graph_launch")
        return self.out

    def close(self):
        if getattr(self, "_handle", None):
            torch.cuda.synchronize()
            load_library().sattn_graph_destroy(self._handle)
            self._handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # interpreter shutdown: the process releases the graph
            pass


def check_status(workspace: torch.Tensor, stream=None) -> int:
    """sattn_check_status: synchronises the stream, returns the status code."""
    return int(load_library().sattn_check_status(_ptr(workspace), _stream(stream)))


def attention(q, k, v, causal=False, sm_scale=0.0, stream=None) -> torch.Tensor:
    """prepare + forward on device tensors (the faster of the two paths on
    GB300; prepare_kv + forward_q_bf16 give the same bytes)."""
    return forward(prepare(q, k, v, causal, sm_scale, stream=stream), stream=stream)


def attention_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal=False, sm_scale=0.0,
                   out: torch.Tensor | None = None, arena: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    """sattn_attention_host: host BF16 tensors in, host BF16 tensor out.

    The copies, both passes and the copy back are enqueued on the stream; the
    result is valid after the stream is synchronised.  Pinned host tensors
    let the copies run asynchronously.
    """
    for t in (q, k, v):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("attention_host takes contiguous host tensors")
    _need_inputs(q, k, v)
    B, Hq, Nq, _ = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    shape = make_shape(B, Hq, Hkv, Nq, Nkv, causal, sm_scale)
    z = query_sizes(shape)
    if arena is None:
        arena = _empty(z["arena"], torch.device("cuda", torch.cuda.current_device()))
    if out is None:
        out = torch.empty((B, Hq, Nq, HEAD_DIM), dtype=torch.bfloat16, pin_memory=True)
    rc = load_library().sattn_attention_host(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                             _ptr(arena), ctypes.c_size_t(arena.numel() * arena.element_size()),
                                             _stream(stream))
    if rc != 0:
        raise SattnError(rc, "sattn_attention_host")
    return out
