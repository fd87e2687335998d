"""Seeded synthetic inputs for the WTConv layer (x, parameters and upstream gradient).

This module draws random numbers and casts them to the activation dtype; it holds none of the
layer's arithmetic.  Both the CUDA path (through the binding) and the CPU oracle consume the very
same host tensors made here, so a parity check compares the two on identical inputs.

Distributions (WTConvNeXt-style layer settings; the second argument of N is the variance):
  x ~ N(0, 1); base_w and wavelet_w ~ N(0, 1/k^2) (variance; std 0.2 at k = 5);
  base_bias ~ N(0, 0.1) (variance); base_scale ~ U(0.5, 1.5); wavelet_scale ~ U(0.05, 0.2)
  per subband channel (4C per level); dy ~ N(0, 1).
Draw order is fixed: x, base_w, base_bias, base_scale, then for each level 1..L (wavelet_w,
wavelet_scale), then dy.  NumPy's PCG64 stream is used because it gives the same numbers on
x86 and Arm hosts; activations are drawn in fp32 and rounded to bf16 / fp16 with
round-to-nearest-even when the layer runs in that dtype.  Parameters stay fp32.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@dataclasses.dataclass(frozen=True)
class LayerShape:
    """One WTConv layer: input (B, C, H, W), L Haar levels, k x k depthwise kernels."""

    B: int
    C: int
    H: int
    W: int
    L: int
    k: int
    dtype: str = "f32"

    @property
    def numel(self) -> int:
        return self.B * self.C * self.H * self.W

    def as_dict(self) -> dict:
        return dataclasses.asdict(self)


# The paper's evaluation shapes, restated: a tiny case, ConvNeXt-T stage shapes (the
# WTConvNeXt-T setting), a high-resolution case with a deep pyramid, and four stacked layers.
WORKLOADS: dict[str, list[LayerShape]] = {
    "tiny_f32": [LayerShape(1, 4, 16, 16, 2, 5, "f32")],
    "stage1_f32": [LayerShape(64, 96, 56, 56, 3, 5, "f32")],
    "stage2_bf16": [LayerShape(64, 192, 28, 28, 2, 5, "bf16")],
    "hires_bf16": [LayerShape(16, 64, 256, 256, 5, 5, "bf16")],
    "four_layers_bf16": [
        LayerShape(128, 96, 64, 64, 4, 5, "bf16"),
        LayerShape(128, 192, 32, 32, 3, 5, "bf16"),
        LayerShape(128, 384, 16, 16, 2, 5, "bf16"),
        LayerShape(128, 768, 8, 8, 1, 5, "bf16"),
    ],
}
WORKLOAD_ORDER = ["tiny_f32", "stage1_f32", "stage2_bf16", "hires_bf16", "four_layers_bf16"]


def make_inputs(shape: LayerShape, seed: int = 0) -> dict[str, torch.Tensor]:
    """Return contiguous CPU tensors x, base_w, base_bias, base_scale, wavelet_w, wavelet_scale, dy.

    Layouts: x, dy (B, C, H, W) in the layer dtype; base_w (C, k, k), base_bias (C,),
    base_scale (C,), wavelet_w (L, 4C, k, k), wavelet_scale (L, 4C), all fp32.  Subband
    channel 4c+s holds subband s (0 LL, 1 LH, 2 HL, 3 HH) of input channel c.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    B, C, H, W, L, k = shape.B, shape.C, shape.H, shape.W, shape.L, shape.k
    f32 = np.float32
    w_std = f32(1.0 / k)
    x = rng.standard_normal((B, C, H, W), dtype=f32)
    base_w = rng.standard_normal((C, k, k), dtype=f32) * w_std
    base_bias = rng.standard_normal((C,), dtype=f32) * f32(math.sqrt(0.1))
    base_scale = rng.uniform(0.5, 1.5, size=(C,)).astype(f32)
    wavelet_w = np.empty((L, 4 * C, k, k), dtype=f32)
    wavelet_scale = np.empty((L, 4 * C), dtype=f32)
    for lvl in range(L):
        wavelet_w[lvl] = rng.standard_normal((4 * C, k, k), dtype=f32) * w_std
        wavelet_scale[lvl] = rng.uniform(0.05, 0.2, size=(4 * C,)).astype(f32)
    dy = rng.standard_normal((B, C, H, W), dtype=f32)
    act = DTYPES[shape.dtype]
    return {
        "x": torch.from_numpy(x).to(act).contiguous(),
        "base_w": torch.from_numpy(base_w),
        "base_bias": torch.from_numpy(base_bias),
        "base_scale": torch.from_numpy(base_scale),
        "wavelet_w": torch.from_numpy(wavelet_w),
        "wavelet_scale": torch.from_numpy(wavelet_scale),
        "dy": torch.from_numpy(dy).to(act).contiguous(),
    }


def workload_inputs(name: str) -> list[tuple[LayerShape, dict[str, torch.Tensor]]]:
    """Inputs for every layer of a named workload; stacked layers use seeds 0, 1, 2, ..."""
    return [(s, make_inputs(s, seed=i)) for i, s in enumerate(WORKLOADS[name])]
