"""Shared helpers of the GPU parity tests (marshalling and comparison only)."""
import numpy as np
import torch

import synth

# Output tolerance of the quantised attention against the oracle: the two
# sides share codes, scales and FP8 P bytes bit for bit; they differ only in
# the rescale factor alpha (hardware exp2, within 2^-22 relative), in the FP32
# summation order inside one tile's PV product and in the fused outer update.
TOL_MAXABS = 4e-3
TOL_COS = 0.99999


def to_device_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def as_f64(bits: np.ndarray) -> np.ndarray:
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def cosine(a: np.ndarray, b: np.ndarray) -> float:
    a, b = a.ravel(), b.ravel()
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    if na == 0 and nb == 0:
        return 1.0
    return float(a @ b / (na * nb))


def assert_close_output(gpu_bits: np.ndarray, ref_bits: np.ndarray, what="", tol_maxabs=TOL_MAXABS):
    g, r = as_f64(gpu_bits), as_f64(ref_bits)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    maxabs = float(np.abs(g - r).max()) if g.size else 0.0
    cos = cosine(g, r)
    assert maxabs <= tol_maxabs and cos >= TOL_COS, f"{what}: max-abs {maxabs:.3g}, cosine {cos:.8f}"
    return maxabs, cos


def assert_prepare_bit_exact(buf: dict, ref: dict, Nkv: int):
    """GPU prepare outputs against the oracle's, bit for bit."""
    for name in ("q_codes", "q_scales", "k_codes", "k_scales", "k_mean", "v_scales"):
        g = buf[name].cpu().numpy()
        r = ref[name]
        assert g.shape == r.shape, name
        same = g.view(np.uint8) == r.view(np.uint8)
        assert same.all(), f"{name}: {int((~same).sum())} bytes differ, first at {np.argwhere(~same)[:3].tolist()}"
    vc = buf["v_codes"].cpu().numpy()                   # [B,Hkv,128,Nkv128] channel-major
    tok = np.ascontiguousarray(vc.transpose(0, 1, 3, 2))
    assert np.all(tok[:, :, Nkv:] == 0), "v_codes pad keys must be 0"
    same = tok[:, :, :Nkv] == ref["v_codes"]
    assert same.all(), f"v_codes: {int((~same).sum())} differ, first at {np.argwhere(~same)[:3].tolist()}"
