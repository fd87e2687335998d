"""After the GPU tests (this file sorts after the others, before the no-alloc file): no kernel's
bounded wait gave up.  The pipelined kernels hand tiles between warps through shared-memory
barriers whose waits are bounded; a wait that runs out raises a sticky device flag, which this
reads (and clears) through the C ABI."""
import pytest
import torch

from memory_bound_cnn_gb300 import inputs as I
from memory_bound_cnn_gb300 import wtconv as W
from parity import PARAMS, to_device


@pytest.mark.gpu
def test_no_bounded_wait_gave_up():
    # one more pipelined call of its own, so the check means something when run alone
    shape = I.LayerShape(B=3, C=4, H=40, W=72, L=3, k=5, dtype="f32")
    d = to_device(I.make_inputs(shape, seed=21))
    import os
    old = os.environ.get("WTCONV_FWD_PATH")
    os.environ["WTCONV_FWD_PATH"] = "tiles"
    try:
        W.wtconv_forward(d["x"], *[d[p] for p in PARAMS])
        W.wtconv_backward_input(d["dy"], *[d[p] for p in PARAMS])
    finally:
        if old is None:
            del os.environ["WTCONV_FWD_PATH"]
        else:
            os.environ["WTCONV_FWD_PATH"] = old
    torch.cuda.synchronize()
    assert W.wtconv_device_status() == W.OK


@pytest.mark.gpu
def test_a_wait_that_gives_up_is_reported_once():
    """The failure path without a fault: a kernel whose bounded wait is never completed raises
    the flag; the host reads it as ERR_DEVICE_TIMEOUT once, and the context stays usable."""
    assert W.wtconv_device_status() == W.OK
    W.wtconv_selftest_wait_timeout()
    assert W.wtconv_device_status() == W.ERR_DEVICE_TIMEOUT
    assert W.wtconv_device_status() == W.OK
    shape = I.LayerShape(B=1, C=2, H=16, W=16, L=2, k=3, dtype="f32")
    d = to_device(I.make_inputs(shape, seed=22))
    y = W.wtconv_forward(d["x"], *[d[p] for p in PARAMS])
    torch.cuda.synchronize()
    assert torch.isfinite(y).all()
