"""The bench's PyTorch-op comparison arm computes the same layer as the oracle (CPU, fp64)."""
import numpy as np
import pytest
import torch

import oracle
from memory_bound_cnn_gb300.inputs import LayerShape, make_inputs

import bench

PARAMS = ("base_w", "base_bias", "base_scale", "wavelet_w", "wavelet_scale")


@pytest.mark.parametrize("shape", [LayerShape(2, 3, 16, 16, 2, 5, "f32"), LayerShape(1, 2, 8, 24, 3, 3, "f32")],
                         ids=["16x16_L2_k5", "8x24_L3_k3"])
def test_torch_cascade_matches_oracle(shape):
    inp = make_inputs(shape, seed=4)
    d = {k: v.double().clone().requires_grad_(k != "dy") for k, v in inp.items()}
    y = bench.torch_cascade(d["x"], *[d[p] for p in PARAMS])
    y.backward(d["dy"])
    y_ref = oracle.forward(inp["x"], inp)
    g_ref = oracle.backward(inp["x"], inp["dy"], inp)
    np.testing.assert_allclose(y.detach().numpy(), y_ref, rtol=0, atol=1e-10 * np.abs(y_ref).max())
    np.testing.assert_allclose(d["x"].grad.numpy(), g_ref["dx"], rtol=0, atol=1e-10 * np.abs(g_ref["dx"]).max())
    for p in PARAMS:
        ref = g_ref["d_" + p]
        np.testing.assert_allclose(d[p].grad.numpy(), ref, rtol=0, atol=1e-10 * np.abs(ref).max())
