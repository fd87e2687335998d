"""The C-ABI library without a GPU: it loads, exports every entry point include/wtconv.h declares,
and rejects invalid arguments on the host before touching CUDA (no compute call is made)."""
import ctypes
import os
import re

import pytest

from memory_bound_cnn_gb300 import wtconv as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(wtconv_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol():
    lib = W.load()
    names = declared_functions()
    assert set(W.EXPORTED) <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_version_and_strerror():
    assert W.wtconv_version() >= 100
    for s in range(8):
        assert isinstance(W.wtconv_strerror(s), str) and W.wtconv_strerror(s)
    assert "unknown" in W.wtconv_strerror(99)


FAKE = ctypes.c_void_p(256)  # aligned, non-null; never dereferenced: validation fails first


def _fwd(lib, B=2, C=3, H=16, Wd=16, L=2, k=5, dt=0, x=FAKE, y=FAKE):
    return lib.wtconv_forward(B, C, H, Wd, L, k, dt, x, FAKE, FAKE, FAKE, FAKE, FAKE, y, None, 0, None)


@pytest.mark.parametrize("kw,status", [
    (dict(B=0), W.ERR_INVALID_ARG), (dict(C=-1), W.ERR_INVALID_ARG), (dict(L=0), W.ERR_INVALID_ARG),
    (dict(L=6), W.ERR_INVALID_ARG), (dict(k=4), W.ERR_INVALID_ARG), (dict(H=0), W.ERR_INVALID_ARG),
    (dict(Wd=-3), W.ERR_INVALID_ARG), (dict(H=1 << 16, Wd=(1 << 14) + 1, L=5), W.ERR_INVALID_ARG),
    (dict(x=None), W.ERR_INVALID_ARG), (dict(H=13, Wd=7, x=None), W.ERR_INVALID_ARG),
    (dict(y=ctypes.c_void_p(264)), W.ERR_INVALID_ARG), (dict(dt=7), W.ERR_UNSUPPORTED),
    (dict(k=9), W.ERR_UNSUPPORTED), (dict(k=1), W.ERR_UNSUPPORTED),
])
def test_forward_rejects_invalid_arguments(kw, status):
    assert _fwd(W.load(), **kw) == status


def test_backward_entry_points_reject_invalid_arguments():
    lib = W.load()
    shape = (2, 3, 16, 16, 2, 5, 0)
    p5 = [FAKE] * 5
    assert lib.wtconv_backward_input(*shape, *p5, None, FAKE, None, 0, None) == W.ERR_INVALID_ARG
    assert lib.wtconv_backward_weights(*shape, FAKE, None, *p5, *p5, None, 0, None) == W.ERR_INVALID_ARG
    assert lib.wtconv_backward(2, 3, 16, 16, 2, 6, 0, FAKE, FAKE, *p5, FAKE, *p5, None, 0, None) == W.ERR_INVALID_ARG
    assert lib.wtconv_backward(2, 3, 16, 16, 2, 5, 0, FAKE, FAKE, *p5, FAKE, FAKE, None, FAKE, FAKE, FAKE,
                               None, 0, None) == W.ERR_INVALID_ARG
    noalloc = lib.wtconv_backward_weights_noalloc
    assert noalloc(*shape, FAKE, None, *p5, *p5, None) == W.ERR_INVALID_ARG
    assert noalloc(2, 3, 12, 16, 3, 5, 0, FAKE, FAKE, *p5, *p5, None) == W.ERR_SCRATCH_LIMIT  # padded planes
    assert noalloc(2, 3, 12, 0, 3, 5, 0, FAKE, FAKE, *p5, *p5, None) == W.ERR_INVALID_ARG
    assert noalloc(2, 3, 16, 16, 2, 5, 0, FAKE, FAKE, *p5, FAKE, ctypes.c_void_p(258), FAKE, FAKE, FAKE,
                   None) == W.ERR_INVALID_ARG


def test_launch_count_of_invalid_shape_is_zero():
    assert W.wtconv_launch_count(W.OP_BACKWARD, 2, 3, 0, 16, 3, 5, 0) == 0
    assert W.wtconv_launch_count(W.OP_FORWARD, 2, 3, 16, 16, 2, 4, 0) == 0


def test_workspace_size_of_invalid_shape_is_zero():
    assert W.wtconv_workspace_size(W.OP_BACKWARD, 2, 3, 12, 16, 3, 5, 0) == 0
    assert W.wtconv_workspace_size(W.OP_FORWARD, 2, 3, 16, 16, 0, 5, 0) == 0


def test_forward_workspace_holds_the_deep_contribution():
    # levels >= 2 leave one fp32 value per level-1 position (B*C*(H/2)*(W/2)), rounded to 256 bytes
    n = 2 * 3 * 8 * 8 * 4
    assert W.wtconv_workspace_size(W.OP_FORWARD, 2, 3, 16, 16, 2, 5, 0) == (n + 255) // 256 * 256
    assert W.wtconv_workspace_size(W.OP_BACKWARD_INPUT, 2, 3, 16, 16, 2, 5, 1) == (n + 255) // 256 * 256
    assert W.wtconv_workspace_size(W.OP_FORWARD, 2, 3, 16, 16, 1, 5, 0) == 0


def test_fault_injection_returns_before_launch(monkeypatch):
    lib = W.load()
    monkeypatch.setenv("WTCONV_INJECT_FAULT", "1")
    assert _fwd(lib) == W.ERR_INJECTED
    p5 = [FAKE] * 5
    assert lib.wtconv_backward(2, 3, 16, 16, 2, 5, 0, FAKE, FAKE, *p5, FAKE, *p5, None, 0, None) == W.ERR_INJECTED
    assert lib.wtconv_backward_weights_noalloc(2, 3, 16, 16, 2, 5, 0, FAKE, FAKE, *p5, *p5, None) == W.ERR_INJECTED
    monkeypatch.setenv("WTCONV_INJECT_FAULT", "0")
    assert _fwd(lib, k=4) == W.ERR_INVALID_ARG


def test_binding_rejects_stream_or_workspace_on_another_device():
    """The binding makes the activations' device current for every call; an explicit stream or
    workspace on another device is rejected before the library is called."""
    import torch

    d0, d1 = torch.device("cuda", 0), torch.device("cuda", 1)

    class Stream:
        def __init__(self, device):
            self.device = device

    W.check_devices(d0)
    W.check_devices(d0, stream=Stream(d0))
    with pytest.raises(ValueError, match="stream"):
        W.check_devices(d0, stream=Stream(d1))
    with pytest.raises(ValueError, match="workspace"):
        W.check_devices(d0, workspace=torch.empty(16, dtype=torch.uint8))  # host memory
