"""Shared test helpers: the parity bar and host/device conversions."""
import numpy as np
import torch

# Attention parity bar: fp16 output vs the fp64 oracle. max |gpu - oracle| <= 2e-3, and
# max |gpu - oracle| / |oracle| <= 5e-3 over elements with |oracle| >= 0.4 (= 2e-3 / 5e-3,
# where the two bounds meet).
ATOL = 2e-3
RTOL = 5e-3
REL_FLOOR = ATOL / RTOL


def attn_errors(gpu_out: torch.Tensor, ref: np.ndarray):
    g = gpu_out.detach().float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(ref).all(), "oracle produced non-finite values"
    diff = np.abs(g - ref)
    max_abs = float(np.nanmax(diff)) if diff.size else 0.0
    if not np.isfinite(g).all():
        max_abs = float("inf")
    big = np.abs(ref) >= REL_FLOOR
    max_rel = float(np.max(diff[big] / np.abs(ref[big]))) if big.any() else 0.0
    return max_abs, max_rel


def assert_attn_close(gpu_out, ref, what=""):
    max_abs, max_rel = attn_errors(gpu_out, ref)
    assert max_abs <= ATOL and max_rel <= RTOL, f"{what}: max_abs={max_abs:.3g} max_rel={max_rel:.3g}"
    return max_abs, max_rel


def u16(t: torch.Tensor) -> np.ndarray:
    """fp16 tensor -> host uint16 bit patterns (NaN payloads preserved)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f16_host(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy()
