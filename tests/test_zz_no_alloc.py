"""wtconv_backward_weights_noalloc: the weight gradient on the library's fixed device scratch.

The file name sorts last so that the test also runs after every other GPU test in one process
(the scratch and its per-device address lookup then see a device the other tests have used);
it needs nothing from them and passes alone in a fresh process as well."""
import pytest
import torch

from memory_bound_cnn_gb300 import inputs as I
from memory_bound_cnn_gb300 import wtconv as W
from parity import GRADS, PARAMS, TOL, assert_close, np64, to_device

SHAPES = [
    I.LayerShape(B=4, C=16, H=32, W=32, L=3, k=5, dtype="f32"),
    I.LayerShape(B=8, C=32, H=28, W=28, L=2, k=5, dtype="bf16"),
    I.LayerShape(B=2, C=8, H=24, W=40, L=3, k=3, dtype="f16"),
]


def _grads_like(d):
    return {g: torch.full_like(d[p], float("nan")) for g, p in zip(GRADS, PARAMS)}


@pytest.mark.gpu
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s.dtype}_{s.H}x{s.W}_L{s.L}_k{s.k}")
def test_noalloc_matches_workspace_entry_point_twice(shape):
    d = to_device(I.make_inputs(shape, seed=11))
    ref = W.wtconv_backward_weights(d["x"], d["dy"], *[d[p] for p in PARAMS])
    torch.cuda.synchronize()
    for call in range(2):  # two calls in a row on the same scratch
        out = _grads_like(d)
        before = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
        W.wtconv_backward_weights_noalloc(d["x"], d["dy"], *[d[p] for p in PARAMS], out)
        after = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
        torch.cuda.synchronize()
        assert after == before, "the binding allocated device memory"
        for g in GRADS:
            assert_close(f"call {call} {g}", np64(out[g]), np64(ref[g]), TOL[shape.dtype])


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [
    I.LayerShape(B=1, C=4, H=256, W=256, L=2, k=5, dtype="bf16"),   # planes too large: pyramids needed
    I.LayerShape(B=2, C=8192, H=8, W=8, L=1, k=5, dtype="f32"),     # partials alone exceed the scratch
], ids=["large_planes", "many_channels"])
def test_noalloc_rejects_shapes_beyond_the_scratch(shape):
    d = to_device(I.make_inputs(shape, seed=12))
    out = _grads_like(d)
    with pytest.raises(W.WTConvError) as e:
        W.wtconv_backward_weights_noalloc(d["x"], d["dy"], *[d[p] for p in PARAMS], out)
    assert e.value.status == W.ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    for g in GRADS:  # nothing was launched: the outputs are untouched
        assert torch.isnan(out[g]).all()
