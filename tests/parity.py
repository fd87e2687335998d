"""Helpers for comparing the CUDA path (through the C ABI) with the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

from memory_bound_cnn_gb300 import wtconv as W

PARAMS = ("base_w", "base_bias", "base_scale", "wavelet_w", "wavelet_scale")
GRADS = ("d_base_w", "d_base_bias", "d_base_scale", "d_wavelet_w", "d_wavelet_scale")
# max |gpu - oracle| <= TOL * max |oracle|, per output tensor
TOL = {"f32": 1e-5, "bf16": 2e-2, "f16": 2e-2}


def to_device(inputs: dict, device="cuda") -> dict:
    return {k: v.to(device).contiguous() for k, v in inputs.items()}


def gpu_forward(d: dict) -> torch.Tensor:
    return W.wtconv_forward(d["x"], *[d[p] for p in PARAMS])


def gpu_backward(d: dict):
    return W.wtconv_backward(d["x"], d["dy"], *[d[p] for p in PARAMS])


def gpu_backward_split(d: dict):
    dx = W.wtconv_backward_input(d["dy"], *[d[p] for p in PARAMS])
    g = W.wtconv_backward_weights(d["x"], d["dy"], *[d[p] for p in PARAMS])
    return dx, g


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").double().numpy()


def max_rel_err(got, ref) -> float:
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    err = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    return err / scale if scale > 0 else err


def assert_close(name: str, got, ref, tol: float):
    r = max_rel_err(got, ref)
    assert np.all(np.isfinite(np.asarray(got))), f"{name}: non-finite values"
    assert r <= tol, f"{name}: max|gpu-oracle| / max|oracle| = {r:.3e} > {tol:.1e}"
    return r
