"""CUDA path (through the C ABI) against the CPU oracle on the same seeded inputs.

Bar: max|gpu - oracle| <= 1e-5 max|oracle| for fp32 activations, <= 2e-2 max|oracle| for bf16 /
fp16, for every output tensor (y, dx and each parameter gradient)."""
import contextlib
import os

import numpy as np
import pytest
import torch

import oracle
from memory_bound_cnn_gb300 import wtconv as W
from memory_bound_cnn_gb300.inputs import WORKLOAD_ORDER, LayerShape, make_inputs, workload_inputs
from parity import GRADS, PARAMS, TOL, assert_close, gpu_backward, gpu_backward_split, gpu_forward, np64, to_device

pytestmark = pytest.mark.gpu


@contextlib.contextmanager
def env_path(var: str, path: str):
    """Set an environment variable for the calls inside (the library reads it at every call)."""
    old = os.environ.get(var)
    os.environ[var] = path
    try:
        yield
    finally:
        if old is None:
            del os.environ[var]
        else:
            os.environ[var] = old


def fwd_path(path: str):
    return env_path("WTCONV_FWD_PATH", path)


def check_layer(shape: LayerShape, inputs: dict, split: bool = True):
    """Forward, fused backward and (if `split`) the separate backward entry points against the
    oracle, on the default kernels and again with each other forward / input-gradient kernel set
    selected (batch-pair, whole-plane, tiled, fused whole-plane; where they apply)."""
    tol = TOL[shape.dtype]
    d = to_device(inputs)
    y_ref = oracle.forward(inputs["x"], inputs)
    g_ref = oracle.backward(inputs["x"], inputs["dy"], inputs)
    for path in ("default", "pair", "plane", "ptile", "tiles", "fused"):
        with fwd_path(path):
            y = gpu_forward(d)
            dx, g = gpu_backward(d)
            torch.cuda.synchronize()
        assert_close(f"y [{path}]", np64(y), y_ref, tol)
        assert_close(f"dx [{path}]", np64(dx), g_ref["dx"], tol)
        if path == "default":
            for n in GRADS:
                assert_close(n, np64(g[n]), g_ref[n], tol)
    if split:
        dx2, g2 = gpu_backward_split(d)
        torch.cuda.synchronize()
        assert_close("dx (backward_input)", np64(dx2), g_ref["dx"], tol)
        for n in GRADS:
            assert_close(n + " (backward_weights)", np64(g2[n]), g_ref[n], tol)
    # the weight gradient's other paths (where they apply): the tiled batch-pair kernel, the
    # batch-pair kernel, the fused
    # whole-plane kernel, the staged whole-plane kernel, tiled kernels and workspace pyramids
    for dpath in ("ptile", "pair", "fused", "plane", "tiles", "pyramid"):
        if dpath == "pyramid" and shape.numel > 20_000_000:
            continue  # the pyramid path already runs by default where planes are too large
        with env_path("WTCONV_DW_PATH", dpath):
            g3 = W.wtconv_backward_weights(d["x"], d["dy"], *[d[p] for p in PARAMS])
            torch.cuda.synchronize()
        for n in GRADS:
            assert_close(f"{n} [{dpath}]", np64(g3[n]), g_ref[n], tol)


@pytest.mark.parametrize("name", WORKLOAD_ORDER)
def test_workload_parity(name):
    """Every layer of every named workload, at full size."""
    for shape, inputs in workload_inputs(name):
        check_layer(shape, inputs, split=(shape.numel <= 20_000_000))


SWEEP = [
    # (B, C, H, W, L, k, dtype): ragged tiles, one-pixel deepest levels, non-square, packing
    (1, 1, 2, 2, 1, 3, "f32"),
    (1, 1, 4, 4, 2, 5, "f32"),
    (2, 3, 6, 10, 1, 5, "f32"),
    (3, 2, 8, 24, 3, 3, "f32"),
    (2, 5, 12, 20, 2, 7, "f32"),
    (4, 3, 32, 32, 5, 5, "f32"),
    (1, 2, 64, 32, 4, 7, "f32"),
    (5, 7, 16, 8, 3, 5, "bf16"),
    (3, 4, 40, 24, 3, 5, "bf16"),
    (2, 3, 28, 28, 2, 3, "f16"),
    (17, 3, 8, 8, 1, 5, "bf16"),
    (33, 2, 4, 4, 2, 5, "f32"),
    (2, 2, 96, 64, 5, 5, "bf16"),
    (2, 3, 6, 130, 1, 5, "f32"),     # rows of more than 32 eight-byte copy chunks
    (2, 2, 4, 98, 1, 3, "bf16"),
    # sides that are not multiples of 2^L: the planes run zero-padded and are cropped back
    (2, 3, 7, 9, 2, 3, "f32"),
    (1, 2, 13, 10, 3, 5, "bf16"),
    (3, 2, 5, 21, 1, 7, "f16"),
    (2, 2, 30, 45, 2, 5, "f32"),
    (2, 3, 57, 55, 3, 5, "f32"),
    (1, 2, 3, 3, 2, 5, "f32"),
    (1, 1, 1, 1, 1, 3, "f32"),       # a single pixel: every level pads
    (2, 2, 1, 37, 3, 5, "bf16"),     # one row, odd width
    # large fp32 planes on the planner's own choice (tiled kernels)
    (1, 2, 256, 256, 5, 5, "f32"),
    (1, 2, 128, 192, 4, 7, "f32"),
]


@pytest.mark.parametrize("case", SWEEP, ids=lambda c: "x".join(map(str, c)))
def test_shape_sweep(case):
    shape = LayerShape(*case)
    check_layer(shape, make_inputs(shape, seed=11))


@pytest.mark.parametrize("case", [(8, 16, 28, 28, 2, 5, "bf16"), (4, 8, 56, 56, 3, 5, "f32")],
                         ids=lambda c: "x".join(map(str, c)))
def test_backward_is_deterministic(case):
    shape = LayerShape(*case)
    d = to_device(make_inputs(shape, seed=3))
    dx1, g1 = gpu_backward(d)
    dx2, g2 = gpu_backward(d)
    torch.cuda.synchronize()
    assert torch.equal(dx1, dx2)
    for n in GRADS:
        assert torch.equal(g1[n], g2[n]), n


@pytest.mark.parametrize("case", [(6, 8, 64, 64, 4, 5, "bf16"), (3, 4, 96, 64, 5, 3, "f32")],
                         ids=lambda c: "x".join(map(str, c)))
def test_tiled_pair_weight_gradient_is_deterministic(case):
    """The tiled batch-pair weight gradient (three launches for L = 5) reduces in a fixed order."""
    shape = LayerShape(*case)
    d = to_device(make_inputs(shape, seed=4))
    with env_path("WTCONV_DW_PATH", "ptile"):
        g1 = W.wtconv_backward_weights(d["x"], d["dy"], *[d[p] for p in PARAMS])
        g2 = W.wtconv_backward_weights(d["x"], d["dy"], *[d[p] for p in PARAMS])
    torch.cuda.synchronize()
    for n in GRADS:
        assert torch.equal(g1[n], g2[n]), n


@pytest.mark.parametrize("case,launches", [((16, 64, 256, 256, 5, 5, "bf16"), 3), ((1, 2, 256, 256, 5, 5, "f32"), 3),
                                           ((2, 3, 128, 128, 4, 5, "bf16"), 2)],
                         ids=lambda c: "x".join(map(str, c)) if isinstance(c, tuple) else str(c))
def test_large_planes_run_the_tiled_pair_weight_gradient(case, launches):
    """Planes beyond the whole-plane kernels take the tiled batch-pair weight gradient by default:
    one launch per two Haar levels (the later ones on the low bands the previous launch writes),
    then the finalize; the launch count the library reports matches its kernel list."""
    B, C, H, Wd, L, k, dt = case
    code = {"f32": 0, "bf16": 1, "f16": 2}[dt]
    names = W.wtconv_plan_kernels(W.OP_BACKWARD_WEIGHTS, B, C, H, Wd, L, k, code)
    assert names == ["wtconv_ptile_dw_kernel", "wtconv_dw_finalize_kernel"], names
    assert W.wtconv_launch_count(W.OP_BACKWARD_WEIGHTS, B, C, H, Wd, L, k, code) == launches + 1
    shape = LayerShape(*case)
    if shape.numel <= 8_000_000:
        inputs = make_inputs(shape, seed=13)
        d = to_device(inputs)
        g = W.wtconv_backward_weights(d["x"], d["dy"], *[d[p] for p in PARAMS])
        torch.cuda.synchronize()
        g_ref = oracle.backward(inputs["x"], inputs["dy"], inputs)
        for n in GRADS:
            assert_close(n, np64(g[n]), g_ref[n], TOL[shape.dtype])


PTILE_FWD = [
    # (B, C, H, W, L, k, dtype): ragged last tile rows / columns, an odd batch (a half pair), L = 1
    # (no deeper levels), every kernel size and activation type
    (3, 2, 40, 200, 3, 5, "bf16"),
    (2, 3, 64, 96, 1, 3, "f32"),
    (5, 2, 48, 72, 2, 7, "f16"),
    (4, 2, 256, 256, 5, 5, "bf16"),
    (1, 3, 128, 64, 4, 7, "f32"),
]


@pytest.mark.parametrize("case", PTILE_FWD, ids=lambda c: "x".join(map(str, c)))
def test_tiled_pair_forward(case):
    """The tiled batch-pair shallow kernel (after the deep kernel where L >= 2), selected where it
    applies, against the oracle for the forward and the input gradient."""
    B, C, H, Wd, L, k, dt = case
    code = {"f32": 0, "bf16": 1, "f16": 2}[dt]
    with fwd_path("ptile"):
        names = W.wtconv_plan_kernels(W.OP_FORWARD, B, C, H, Wd, L, k, code)
        n = W.wtconv_launch_count(W.OP_FORWARD, B, C, H, Wd, L, k, code)
    want = (["wtconv_deep_kernel"] if L >= 2 else []) + ["wtconv_pshallow_kernel"]
    assert names == want, names
    assert n == len(want)
    shape = LayerShape(*case)
    inputs = make_inputs(shape, seed=17)
    d = to_device(inputs)
    tol = TOL[shape.dtype]
    with fwd_path("ptile"):
        y = gpu_forward(d)
        dx = W.wtconv_backward_input(d["dy"], *[d[p] for p in PARAMS])
    torch.cuda.synchronize()
    assert_close("y [ptile]", np64(y), oracle.forward(inputs["x"], inputs), tol)
    g_ref = oracle.backward(inputs["x"], inputs["dy"], inputs)
    assert_close("dx [ptile]", np64(dx), g_ref["dx"], tol)


@pytest.mark.parametrize("knobs", [{"WTCONV_PAIR_SPLIT": "0"}, {"WTCONV_PAIR_TMAP": "0"},
                                   {"WTCONV_PAIR_SPLIT": "0", "WTCONV_PAIR_TMAP": "0"}],
                         ids=lambda k: "+".join(f"{a}={b}" for a, b in k.items()))
@pytest.mark.parametrize("case", [(6, 8, 64, 64, 4, 5, "bf16"), (5, 6, 32, 32, 3, 3, "f16"), (3, 4, 56, 56, 3, 5, "f32"),
                                  (9, 8, 8, 8, 1, 7, "bf16"), (4, 6, 28, 28, 2, 5, "bf16")],
                         ids=lambda c: "x".join(map(str, c)))
def test_pair_kernels_without_level_split_or_tensor_copies(case, knobs):
    """The batch-pair kernels' other schedules against the oracle: every warp on every level
    (no last-warp split for levels >= 3) and one bulk copy per plane (no group tensor copy)."""
    shape = LayerShape(*case)
    inputs = make_inputs(shape, seed=21)
    d = to_device(inputs)
    tol = TOL[shape.dtype]
    with contextlib.ExitStack() as stack:
        for var, val in knobs.items():
            stack.enter_context(env_path(var, val))
        stack.enter_context(fwd_path("pair"))
        stack.enter_context(env_path("WTCONV_DW_PATH", "pair"))
        y = gpu_forward(d)
        dx, g = gpu_backward(d)
        torch.cuda.synchronize()
    y_ref = oracle.forward(inputs["x"], inputs)
    g_ref = oracle.backward(inputs["x"], inputs["dy"], inputs)
    assert_close("y", np64(y), y_ref, tol)
    assert_close("dx", np64(dx), g_ref["dx"], tol)
    for n in GRADS:
        assert_close(n, np64(g[n]), g_ref[n], tol)


def test_input_gradient_is_forward_with_rotated_kernels():
    """dx = forward(dy) with every kernel rotated 180 degrees and no bias (transpose identity)."""
    shape = LayerShape(2, 4, 32, 32, 3, 5, "f32")
    d = to_device(make_inputs(shape, seed=5))
    dx = W.wtconv_backward_input(d["dy"], *[d[p] for p in PARAMS])
    flipped = dict(d)
    flipped["base_w"] = torch.flip(d["base_w"], dims=(-2, -1)).contiguous()
    flipped["wavelet_w"] = torch.flip(d["wavelet_w"], dims=(-2, -1)).contiguous()
    flipped["base_bias"] = torch.zeros_like(d["base_bias"])
    y = W.wtconv_forward(d["dy"], *[flipped[p] for p in PARAMS])
    torch.cuda.synchronize()
    assert_close("dx vs rotated forward", np64(dx), np64(y), 1e-6)


@pytest.mark.parametrize("path", ["default", "pair", "plane", "ptile", "tiles", "fused"])
def test_outputs_stay_in_bounds_and_inputs_untouched(path):
    """Canary words around every output; inputs byte-identical after the calls."""
    shape = LayerShape(3, 5, 24, 16, 3, 5, "bf16")
    inputs = make_inputs(shape, seed=9)
    d = to_device(inputs)
    before = {k: v.clone() for k, v in d.items()}
    pad = 4096
    n = shape.numel
    ybuf = torch.full((n + 2 * pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    dxbuf = torch.full((n + 2 * pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    y = ybuf[pad:pad + n].view(shape.B, shape.C, shape.H, shape.W)
    dx = dxbuf[pad:pad + n].view(shape.B, shape.C, shape.H, shape.W)
    with fwd_path(path):
        W.wtconv_forward(d["x"], *[d[p] for p in PARAMS], y=y)
    gbufs = {}
    grads = {}
    for gname, p in zip(GRADS, PARAMS):
        m = d[p].numel()
        buf = torch.full((m + 2 * 64,), 7.0, device="cuda")
        gbufs[gname] = buf
        grads[gname] = buf[64:64 + m].view_as(d[p])
    with fwd_path(path):
        W.wtconv_backward(d["x"], d["dy"], *[d[p] for p in PARAMS], dx=dx, grads=grads)
    torch.cuda.synchronize()
    for buf in (ybuf, dxbuf):
        assert torch.all(buf[:pad] == 7.0) and torch.all(buf[pad + n:] == 7.0)
    for gname, buf in gbufs.items():
        assert torch.all(buf[:64] == 7.0) and torch.all(buf[-64:] == 7.0), gname
    for k in d:
        assert torch.equal(d[k], before[k]), k


def test_autograd_function_matches_oracle():
    shape = LayerShape(2, 3, 16, 16, 2, 5, "f32")
    inputs = make_inputs(shape, seed=2)
    d = to_device(inputs)
    leaves = {k: d[k].clone().requires_grad_(True) for k in ("x",) + PARAMS}
    y = W.WTConvFunction.apply(leaves["x"], *[leaves[p] for p in PARAMS])
    y.backward(d["dy"])
    g_ref = oracle.backward(inputs["x"], inputs["dy"], inputs)
    assert_close("autograd dx", np64(leaves["x"].grad), g_ref["dx"], 1e-5)
    for gname, p in zip(GRADS, PARAMS):
        assert_close("autograd " + gname, np64(leaves[p].grad), g_ref[gname], 1e-5)


def test_autograd_on_a_non_contiguous_input():
    """A transposed view as input: the forward and the backward read the same contiguous copy."""
    shape = LayerShape(2, 3, 16, 24, 2, 5, "f32")
    inputs = make_inputs(shape, seed=4)
    d = to_device(inputs)
    xt = d["x"].transpose(2, 3).contiguous().transpose(2, 3)  # same values, non-contiguous
    assert not xt.is_contiguous()
    leaves = {k: d[k].clone().requires_grad_(True) for k in PARAMS}
    xl = xt.clone().requires_grad_(True)
    y = W.WTConvFunction.apply(xl, *[leaves[p] for p in PARAMS])
    y.backward(d["dy"])
    g_ref = oracle.backward(inputs["x"], inputs["dy"], inputs)
    assert_close("autograd dx (non-contiguous x)", np64(xl.grad), g_ref["dx"], 1e-5)
    for gname, p in zip(GRADS, PARAMS):
        assert_close("autograd " + gname, np64(leaves[p].grad), g_ref[gname], 1e-5)


def test_invalid_call_raises_and_writes_nothing(monkeypatch):
    shape = LayerShape(2, 3, 16, 16, 2, 5, "f32")
    d = to_device(make_inputs(shape, seed=1))
    y = torch.full_like(d["x"], 3.0)
    # an even kernel size: consistent shapes, rejected by the library's validation
    even = dict(d, base_w=d["base_w"][:, :4, :4].contiguous(), wavelet_w=d["wavelet_w"][:, :, :4, :4].contiguous())
    with pytest.raises(W.WTConvError) as e:
        W.wtconv_forward(d["x"], *[even[p] for p in PARAMS], y=y)
    assert e.value.status == W.ERR_INVALID_ARG
    # a parameter shorter than the channel count: rejected by the binding before any call
    with pytest.raises(ValueError):
        W.wtconv_forward(d["x"], *[d[p] for p in PARAMS[:4]], d["wavelet_scale"][:, :4].contiguous(), y=y)
    y2 = torch.full_like(d["x"], 3.0)
    monkeypatch.setenv("WTCONV_INJECT_FAULT", "1")
    with pytest.raises(W.WTConvError) as e:
        W.wtconv_forward(d["x"], *[d[p] for p in PARAMS], y=y2)
    assert e.value.status == W.ERR_INJECTED
    torch.cuda.synchronize()
    assert torch.all(y == 3.0) and torch.all(y2 == 3.0)
