"""A training step of the layer captured in a CUDA graph and replayed.

The entry points only enqueue kernels on the caller's stream: after one eager call has planned
the shape (host-side), the forward and the fused backward can be captured with the caller's
buffers and workspace, and every replay gives the eager results bit for bit (the kernels are
deterministic).  The no-alloc weight-gradient entry point captures the same way with no
workspace at all."""
import pytest
import torch

from memory_bound_cnn_gb300 import inputs as I
from memory_bound_cnn_gb300 import wtconv as W
from parity import GRADS, PARAMS, to_device

SHAPES = [
    I.LayerShape(B=4, C=8, H=56, W=56, L=3, k=5, dtype="f32"),    # fused whole-plane kernels
    I.LayerShape(B=8, C=16, H=28, W=28, L=2, k=5, dtype="bf16"),  # staged whole-plane kernels
    I.LayerShape(B=2, C=4, H=30, W=45, L=2, k=3, dtype="f32"),    # padded planes (pad / crop kernels)
]


@pytest.mark.gpu
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s.dtype}_{s.H}x{s.W}_L{s.L}")
def test_step_replays_from_a_cuda_graph(shape):
    d = to_device(I.make_inputs(shape, seed=21))
    p = [d[n] for n in PARAMS]
    dims = (shape.B, shape.C, shape.H, shape.W, shape.L, shape.k, W.DTYPE_CODE[d["x"].dtype])
    ws_f = torch.empty(max(1, W.wtconv_workspace_size(W.OP_FORWARD, *dims)), dtype=torch.uint8, device="cuda")
    ws_b = torch.empty(max(1, W.wtconv_workspace_size(W.OP_BACKWARD, *dims)), dtype=torch.uint8, device="cuda")
    y = torch.empty_like(d["x"])
    dx = torch.empty_like(d["x"])
    grads = {g: torch.empty_like(d[q]) for g, q in zip(GRADS, PARAMS)}

    def step(stream=None):
        W.wtconv_forward(d["x"], *p, y=y, workspace=ws_f, stream=stream)
        W.wtconv_backward(d["x"], d["dy"], *p, dx=dx, grads=grads, workspace=ws_b, stream=stream)

    step()  # plans the shape
    torch.cuda.synchronize()
    ref = {"y": y.clone(), "dx": dx.clone(), **{g: grads[g].clone() for g in GRADS}}

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        step(stream=side)
    for t in [y, dx] + list(grads.values()):
        t.fill_(float("nan"))
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    got = {"y": y, "dx": dx, **grads}
    for name, want in ref.items():
        assert torch.equal(got[name], want), f"graph replay differs in {name}"


@pytest.mark.gpu
def test_noalloc_weight_gradient_replays_from_a_cuda_graph():
    shape = I.LayerShape(B=4, C=8, H=32, W=32, L=3, k=5, dtype="f32")
    d = to_device(I.make_inputs(shape, seed=22))
    p = [d[n] for n in PARAMS]
    out = {g: torch.empty_like(d[q]) for g, q in zip(GRADS, PARAMS)}
    W.wtconv_backward_weights_noalloc(d["x"], d["dy"], *p, out)  # plans the shape, finds the scratch
    torch.cuda.synchronize()
    ref = {g: out[g].clone() for g in GRADS}
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        W.wtconv_backward_weights_noalloc(d["x"], d["dy"], *p, out, stream=side)
    for t in out.values():
        t.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    for g in GRADS:
        assert torch.equal(out[g], ref[g]), f"graph replay differs in {g}"
