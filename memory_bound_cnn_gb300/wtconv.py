"""Python binding of libwtconv.so (include/wtconv.h): argument marshalling only.

Every step of the layer runs in the library's CUDA kernels; this module checks tensors, passes
their device pointers and the current CUDA stream, and allocates the workspace from PyTorch's
caching allocator.  There is no CPU or PyTorch fallback: if the library cannot be loaded, every
call raises.

Functions carry the C names: ``wtconv_forward``, ``wtconv_backward_input``,
``wtconv_backward_weights``, ``wtconv_backward``, ``wtconv_backward_weights_noalloc``,
``wtconv_workspace_size``, ``wtconv_launch_count``, ``wtconv_plan_kernels``, ``wtconv_device_status``,
``wtconv_selftest_wait_timeout``, ``wtconv_fp32_fma_peak``, ``wtconv_strerror``, ``wtconv_version``.
``WTConvFunction`` wraps forward and the fused backward as a ``torch.autograd.Function``.

Every call runs with the activations' device current (the library plans, looks up its device
symbols and launches on the current device), and rejects a stream or workspace on another device.
"""
from __future__ import annotations

import contextlib
import ctypes
import os

import torch

from . import _build

F32, BF16, F16 = 0, 1, 2
OP_FORWARD, OP_BACKWARD_INPUT, OP_BACKWARD_WEIGHTS, OP_BACKWARD = 0, 1, 2, 3
(OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_INJECTED, ERR_SCRATCH_LIMIT,
 ERR_DEVICE_TIMEOUT) = range(8)
NOALLOC_SCRATCH_BYTES = 4 << 20  # WTCONV_NOALLOC_SCRATCH_BYTES
TORCH_DTYPE = {F32: torch.float32, BF16: torch.bfloat16, F16: torch.float16}
DTYPE_CODE = {v: k for k, v in TORCH_DTYPE.items()}

EXPORTED = ("wtconv_version", "wtconv_strerror", "wtconv_workspace_size", "wtconv_forward",
            "wtconv_backward_input", "wtconv_backward_weights", "wtconv_backward",
            "wtconv_backward_weights_noalloc", "wtconv_launch_count", "wtconv_device_status",
            "wtconv_plan_kernels", "wtconv_selftest_wait_timeout", "wtconv_fp32_fma_peak")

_lib = None


class WTConvError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {wtconv_strerror(status)} (status {status})")
        self.status = status


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libwtconv.so (building it first if it is missing or stale and nvcc exists)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if build_if_missing:
        try:
            path = _build.build()
        except OSError as e:  # no nvcc here: use what is built, if anything
            if not os.path.exists(path):
                raise RuntimeError(f"libwtconv.so is not built and cannot be built: {e}") from e
        # a compile error (RuntimeError) propagates: a stale library must not stand in for it
    lib = ctypes.CDLL(path)
    i, vp, sz, fp = ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p
    lib.wtconv_version.restype = i
    lib.wtconv_version.argtypes = []
    lib.wtconv_strerror.restype = ctypes.c_char_p
    lib.wtconv_strerror.argtypes = [i]
    lib.wtconv_workspace_size.restype = sz
    lib.wtconv_workspace_size.argtypes = [i] * 8
    lib.wtconv_plan_kernels.restype = ctypes.c_char_p
    lib.wtconv_plan_kernels.argtypes = [i] * 8
    lib.wtconv_device_status.restype = i
    lib.wtconv_device_status.argtypes = []
    lib.wtconv_selftest_wait_timeout.restype = i
    lib.wtconv_selftest_wait_timeout.argtypes = [ctypes.c_void_p]
    lib.wtconv_launch_count.restype = i
    lib.wtconv_launch_count.argtypes = [i] * 8
    lib.wtconv_fp32_fma_peak.restype = i
    lib.wtconv_fp32_fma_peak.argtypes = [i, ctypes.POINTER(ctypes.c_double)]
    shape = [i] * 7
    params = [fp] * 5
    lib.wtconv_forward.restype = i
    lib.wtconv_forward.argtypes = shape + [vp] + params + [vp, vp, sz, vp]
    lib.wtconv_backward_input.restype = i
    lib.wtconv_backward_input.argtypes = shape + params + [vp, vp, vp, sz, vp]
    lib.wtconv_backward_weights.restype = i
    lib.wtconv_backward_weights.argtypes = shape + [vp, vp] + params + [fp] * 5 + [vp, sz, vp]
    lib.wtconv_backward_weights_noalloc.restype = i
    lib.wtconv_backward_weights_noalloc.argtypes = shape + [vp, vp] + params + [fp] * 5 + [vp]
    lib.wtconv_backward.restype = i
    lib.wtconv_backward.argtypes = shape + [vp, vp] + params + [vp] + [fp] * 5 + [vp, sz, vp]
    _lib = lib
    return lib


def wtconv_version() -> int:
    return load().wtconv_version()


def wtconv_strerror(status: int) -> str:
    return load().wtconv_strerror(status).decode()


def wtconv_workspace_size(op: int, B: int, C: int, H: int, W: int, L: int, k: int, dtype: int) -> int:
    return load().wtconv_workspace_size(op, B, C, H, W, L, k, dtype)


def wtconv_plan_kernels(op: int, B: int, C: int, H: int, W: int, L: int, k: int, dtype: int) -> list[str]:
    """Kernels `op` launches for this shape, in launch order."""
    names = load().wtconv_plan_kernels(op, B, C, H, W, L, k, dtype).decode()
    return names.split("+") if names else []


def wtconv_device_status() -> int:
    """Synchronise the device; WTCONV_ERR_DEVICE_TIMEOUT if a kernel's bounded wait gave up."""
    return load().wtconv_device_status()


def wtconv_selftest_wait_timeout(stream=None) -> None:
    """Launch the diagnostic whose one bounded wait is never completed: the next
    wtconv_device_status() then returns ERR_DEVICE_TIMEOUT."""
    _raise(load().wtconv_selftest_wait_timeout(_stream(stream)), "wtconv_selftest_wait_timeout")


def wtconv_launch_count(op: int, B: int, C: int, H: int, W: int, L: int, k: int, dtype: int) -> int:
    return load().wtconv_launch_count(op, B, C, H, W, L, k, dtype)


def wtconv_fp32_fma_peak(iters: int = 20000, device=None) -> float:
    """Packed-FMA throughput of the device in TFLOP/s (synchronises it)."""
    out = ctypes.c_double(0.0)
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        _raise(load().wtconv_fp32_fma_peak(iters, ctypes.byref(out)), "wtconv_fp32_fma_peak")
    return out.value


# ------------------------------------------------------------------------------- marshalling

def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check_act(t: torch.Tensor, name: str):
    if not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
        raise ValueError(f"{name} must be a contiguous 4-D CUDA tensor")
    if t.dtype not in DTYPE_CODE:
        raise ValueError(f"{name} has unsupported dtype {t.dtype}")


def _check_param(t: torch.Tensor, name: str, device):
    if not t.is_cuda or not t.is_contiguous() or t.dtype != torch.float32 or t.device != device:
        raise ValueError(f"{name} must be a contiguous fp32 CUDA tensor on {device}")


def _shape(x: torch.Tensor, wavelet_w: torch.Tensor, base_w: torch.Tensor):
    B, C, H, W = x.shape
    return B, C, H, W, wavelet_w.shape[0], base_w.shape[-1], DTYPE_CODE[x.dtype]


def _workspace(op: int, shape, device, workspace: torch.Tensor | None):
    need = wtconv_workspace_size(op, *shape)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return workspace, nbytes


def _params(base_w, base_bias, base_scale, wavelet_w, wavelet_scale, act):
    """Checks every parameter against the activation's channel count (the library reads them
    through bare pointers, so a short tensor would be read past its end) and returns pointers."""
    device, C = act.device, act.shape[1]
    for t, n in ((base_w, "base_w"), (base_bias, "base_bias"), (base_scale, "base_scale"),
                 (wavelet_w, "wavelet_w"), (wavelet_scale, "wavelet_scale")):
        _check_param(t, n, device)
    k = base_w.shape[-1] if base_w.dim() == 3 else -1
    L = wavelet_w.shape[0] if wavelet_w.dim() == 4 else -1
    want = {"base_w": (C, k, k), "base_bias": (C,), "base_scale": (C,), "wavelet_w": (L, 4 * C, k, k),
            "wavelet_scale": (L, 4 * C)}
    for t, n in ((base_w, "base_w"), (base_bias, "base_bias"), (base_scale, "base_scale"),
                 (wavelet_w, "wavelet_w"), (wavelet_scale, "wavelet_scale")):
        if tuple(t.shape) != want[n]:
            raise ValueError(f"{n} has shape {tuple(t.shape)}, expected {want[n]} for {C} channels")
    return [_ptr(base_w), _ptr(base_bias), _ptr(base_scale), _ptr(wavelet_w), _ptr(wavelet_scale)]


def _check_out(t: torch.Tensor, name: str, like: torch.Tensor):
    _check_act(t, name)
    if t.shape != like.shape or t.dtype != like.dtype or t.device != like.device:
        raise ValueError(f"{name} must match the input's shape, dtype and device")


def _raise(status: int, where: str):
    if status != OK:
        raise WTConvError(status, where)


def check_devices(device: torch.device, stream=None, workspace: torch.Tensor | None = None):
    """Raise ValueError if an explicit stream or workspace lives on another device than `device`
    (the activations' device): the library would launch on one device with another's memory."""
    if stream is not None and getattr(stream, "device", device) != device:
        raise ValueError(f"stream is on {stream.device}, the tensors on {device}")
    if workspace is not None and workspace.device != device:
        raise ValueError(f"workspace is on {workspace.device}, the tensors on {device}")


@contextlib.contextmanager
def _on(device: torch.device, stream, workspace):
    """The activations' device made current for the call (checked against stream and workspace)."""
    check_devices(device, stream, workspace)
    with torch.cuda.device(device):
        yield


def wtconv_forward(x, base_w, base_bias, base_scale, wavelet_w, wavelet_scale, y=None, workspace=None,
                   stream=None) -> torch.Tensor:
    """y = WTConv(x); x (B, C, H, W) fp32 / bf16 / fp16 on CUDA, parameters fp32."""
    _check_act(x, "x")
    shape = _shape(x, wavelet_w, base_w)
    p = _params(base_w, base_bias, base_scale, wavelet_w, wavelet_scale, x)
    if y is None:
        y = torch.empty_like(x)
    _check_out(y, "y", x)
    with _on(x.device, stream, workspace):
        ws, nbytes = _workspace(OP_FORWARD, shape, x.device, workspace)
        rc = load().wtconv_forward(*shape, _ptr(x), *p, _ptr(y), _ptr(ws), nbytes, _stream(stream))
    _raise(rc, "wtconv_forward")
    return y


def wtconv_backward_input(dy, base_w, base_bias, base_scale, wavelet_w, wavelet_scale, dx=None,
                          workspace=None, stream=None) -> torch.Tensor:
    """dx = WTConv^T(dy) (the input gradient)."""
    _check_act(dy, "dy")
    shape = _shape(dy, wavelet_w, base_w)
    p = _params(base_w, base_bias, base_scale, wavelet_w, wavelet_scale, dy)
    if dx is None:
        dx = torch.empty_like(dy)
    _check_out(dx, "dx", dy)
    with _on(dy.device, stream, workspace):
        ws, nbytes = _workspace(OP_BACKWARD_INPUT, shape, dy.device, workspace)
        rc = load().wtconv_backward_input(*shape, *p, _ptr(dy), _ptr(dx), _ptr(ws), nbytes, _stream(stream))
    _raise(rc, "wtconv_backward_input")
    return dx


def _grad_buffers(base_w, base_bias, base_scale, wavelet_w, wavelet_scale, grads):
    if grads is None:
        grads = {
            "d_base_w": torch.empty_like(base_w), "d_base_bias": torch.empty_like(base_bias),
            "d_base_scale": torch.empty_like(base_scale), "d_wavelet_w": torch.empty_like(wavelet_w),
            "d_wavelet_scale": torch.empty_like(wavelet_scale),
        }
    order = ("d_base_w", "d_base_bias", "d_base_scale", "d_wavelet_w", "d_wavelet_scale")
    for n, like in zip(order, (base_w, base_bias, base_scale, wavelet_w, wavelet_scale)):
        _check_param(grads[n], n, base_w.device)
        if grads[n].shape != like.shape:
            raise ValueError(f"{n} has shape {tuple(grads[n].shape)}, expected {tuple(like.shape)}")
    return grads, [_ptr(grads[n]) for n in order]


def wtconv_backward_weights(x, dy, base_w, base_bias, base_scale, wavelet_w, wavelet_scale, grads=None,
                            workspace=None, stream=None) -> dict:
    """Every parameter gradient (dict d_base_w, d_base_bias, d_base_scale, d_wavelet_w, d_wavelet_scale)."""
    _check_act(x, "x")
    _check_act(dy, "dy")
    _check_out(dy, "dy", x)
    shape = _shape(x, wavelet_w, base_w)
    p = _params(base_w, base_bias, base_scale, wavelet_w, wavelet_scale, x)
    grads, gp = _grad_buffers(base_w, base_bias, base_scale, wavelet_w, wavelet_scale, grads)
    with _on(x.device, stream, workspace):
        ws, nbytes = _workspace(OP_BACKWARD_WEIGHTS, shape, x.device, workspace)
        rc = load().wtconv_backward_weights(*shape, _ptr(x), _ptr(dy), *p, *gp, _ptr(ws), nbytes,
                                            _stream(stream))
    _raise(rc, "wtconv_backward_weights")
    return grads


def wtconv_backward_weights_noalloc(x, dy, base_w, base_bias, base_scale, wavelet_w, wavelet_scale, grads,
                                    stream=None) -> dict:
    """wtconv_backward_weights on the library's fixed scratch: no workspace, no allocation.

    ``grads`` (the dict of gradient buffers) must be passed in, so this call allocates nothing
    either; calls that overlap in time race on the shared scratch."""
    if grads is None:
        raise ValueError("wtconv_backward_weights_noalloc needs preallocated gradient buffers")
    _check_act(x, "x")
    _check_act(dy, "dy")
    _check_out(dy, "dy", x)
    shape = _shape(x, wavelet_w, base_w)
    p = _params(base_w, base_bias, base_scale, wavelet_w, wavelet_scale, x)
    grads, gp = _grad_buffers(base_w, base_bias, base_scale, wavelet_w, wavelet_scale, grads)
    with _on(x.device, stream, None):
        rc = load().wtconv_backward_weights_noalloc(*shape, _ptr(x), _ptr(dy), *p, *gp, _stream(stream))
    _raise(rc, "wtconv_backward_weights_noalloc")
    return grads


def wtconv_backward(x, dy, base_w, base_bias, base_scale, wavelet_w, wavelet_scale, dx=None, grads=None,
                    workspace=None, stream=None) -> tuple[torch.Tensor, dict]:
    """Fused backward: (dx, parameter gradients) from one pass over x and dy."""
    _check_act(x, "x")
    _check_act(dy, "dy")
    shape = _shape(x, wavelet_w, base_w)
    p = _params(base_w, base_bias, base_scale, wavelet_w, wavelet_scale, x)
    if dx is None:
        dx = torch.empty_like(x)
    _check_out(dx, "dx", x)
    _check_out(dy, "dy", x)
    grads, gp = _grad_buffers(base_w, base_bias, base_scale, wavelet_w, wavelet_scale, grads)
    with _on(x.device, stream, workspace):
        ws, nbytes = _workspace(OP_BACKWARD, shape, x.device, workspace)
        rc = load().wtconv_backward(*shape, _ptr(x), _ptr(dy), *p, _ptr(dx), *gp, _ptr(ws), nbytes,
                                    _stream(stream))
    _raise(rc, "wtconv_backward")
    return dx, grads


class WTConvFunction(torch.autograd.Function):
    """Autograd wrapper: forward through wtconv_forward, backward through the fused wtconv_backward."""

    @staticmethod
    def forward(ctx, x, base_w, base_bias, base_scale, wavelet_w, wavelet_scale):
        xc = x.contiguous()  # the backward reads the same contiguous copy
        ctx.save_for_backward(xc, base_w, base_bias, base_scale, wavelet_w, wavelet_scale)
        return wtconv_forward(xc, base_w, base_bias, base_scale, wavelet_w, wavelet_scale)

    @staticmethod
    def backward(ctx, dy):
        x, base_w, base_bias, base_scale, wavelet_w, wavelet_scale = ctx.saved_tensors
        dx, g = wtconv_backward(x, dy.contiguous(), base_w, base_bias, base_scale, wavelet_w, wavelet_scale)
        return dx, g["d_base_w"], g["d_base_bias"], g["d_base_scale"], g["d_wavelet_w"], g["d_wavelet_scale"]
