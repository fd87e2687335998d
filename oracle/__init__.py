"""WTConv CPU oracle -- TEST INFRASTRUCTURE, not part of the product.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg may import this
package.  It wraps ``wtconv_oracle.c``: a plain fp64 restatement of the reference WTConv pipeline
(explicit Haar analysis per level, depthwise conv per subband, separate scale pass, sequential
inverse-Haar cascade, scaled base conv with bias) and its literal backward, written from the
paper "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware Reformulation"
(arXiv 2608.10805).  It shares no code with the CUDA library.

Parity status: the paper's pages print no worked example, so no function here is pinned to
printed numbers; each is pinned by the tests to mathematics (see tests/test_oracle_pins.py).

The shared library is compiled from source with the host C compiler on first use (or by
``build()``), into this directory.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "wtconv_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_dp = ctypes.POINTER(ctypes.c_double)


def compile_library(src: str, out: str) -> str:
    """Compile an oracle C source into a shared library (plain C11, no FMA contraction)."""
    tmp = out + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
           "-o", tmp, src]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/liboracle.so if it is missing or stale."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(SOURCE):
        compile_library(SOURCE, _LIB)
    return _LIB


def _f64(a) -> np.ndarray:
    """Any array-like (numpy, torch CPU tensor of any float dtype) -> C-contiguous float64."""
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def default_threads() -> int:
    if hasattr(os, "sched_getaffinity"):
        return max(1, len(os.sched_getaffinity(0)))
    return os.cpu_count() or 1


_PARAM_NAMES = ("base_w", "base_bias", "base_scale", "wavelet_w", "wavelet_scale")
GRAD_NAMES = ("dx", "d_base_w", "d_base_bias", "d_base_scale", "d_wavelet_w", "d_wavelet_scale")


class Oracle:
    """Handle on one compiled oracle library (the default one, or a test's variant)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i = ctypes.c_int
        lib.oracle_haar_analysis.argtypes = [_dp, i, i, _dp]
        lib.oracle_haar_synthesis.argtypes = [_dp, i, i, _dp]
        lib.oracle_dwconv.argtypes = [_dp, i, i, _dp, i, _dp]
        lib.oracle_forward.argtypes = [i] * 6 + [_dp] * 7 + [i]
        lib.oracle_forward.restype = i
        lib.oracle_backward.argtypes = [i] * 6 + [_dp] * 13 + [i]
        lib.oracle_backward.restype = i
        self.lib, self.path = lib, path

    def haar_analysis(self, plane) -> np.ndarray:
        """One Haar level of an (H, W) plane -> (4, H/2, W/2) subbands LL, LH, HL, HH."""
        x = _f64(plane)
        H, W = x.shape
        out = np.empty((4, H // 2, W // 2))
        self.lib.oracle_haar_analysis(_ptr(x), H, W, _ptr(out))
        return out

    def haar_synthesis(self, sub) -> np.ndarray:
        """Inverse of one Haar level: (4, h, w) -> (2h, 2w)."""
        s = _f64(sub)
        _, h, w = s.shape
        out = np.empty((2 * h, 2 * w))
        self.lib.oracle_haar_synthesis(_ptr(s), h, w, _ptr(out))
        return out

    def dwconv(self, plane, ker) -> np.ndarray:
        """k x k cross-correlation of an (H, W) plane, zero 'same' padding."""
        x, w = _f64(plane), _f64(ker)
        H, W = x.shape
        out = np.empty((H, W))
        self.lib.oracle_dwconv(_ptr(x), H, W, _ptr(w), w.shape[0], _ptr(out))
        return out

    def forward(self, x, params: dict, nthreads: int | None = None) -> np.ndarray:
        """WTConv forward of x (B, C, H, W) with the five parameter arrays in ``params``."""
        xd = _f64(x)
        B, C, H, W = xd.shape
        pw = [_f64(params[n]) for n in _PARAM_NAMES]
        L, k = pw[3].shape[0], pw[0].shape[-1]
        y = np.empty_like(xd)
        rc = self.lib.oracle_forward(B, C, H, W, L, k, _ptr(xd), *[_ptr(a) for a in pw],
                                     _ptr(y), nthreads or default_threads())
        if rc != 0:
            raise ValueError(f"oracle_forward failed with status {rc}")
        return y

    def backward(self, x, dy, params: dict, nthreads: int | None = None) -> dict:
        """dx and every parameter gradient (float64 arrays) for upstream gradient dy."""
        xd, dyd = _f64(x), _f64(dy)
        B, C, H, W = xd.shape
        pw = [_f64(params[n]) for n in _PARAM_NAMES]
        L, k = pw[3].shape[0], pw[0].shape[-1]
        g = {
            "dx": np.empty_like(xd),
            "d_base_w": np.empty((C, k, k)),
            "d_base_bias": np.empty((C,)),
            "d_base_scale": np.empty((C,)),
            "d_wavelet_w": np.empty((L, 4 * C, k, k)),
            "d_wavelet_scale": np.empty((L, 4 * C)),
        }
        rc = self.lib.oracle_backward(B, C, H, W, L, k, _ptr(xd), _ptr(dyd),
                                      *[_ptr(a) for a in pw], *[_ptr(g[n]) for n in GRAD_NAMES],
                                      nthreads or default_threads())
        if rc != 0:
            raise ValueError(f"oracle_backward failed with status {rc}")
        return g


_default: Oracle | None = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def haar_analysis(plane):
    return default().haar_analysis(plane)


def haar_synthesis(sub):
    return default().haar_synthesis(sub)


def dwconv(plane, ker):
    return default().dwconv(plane, ker)


def forward(x, params, nthreads=None):
    return default().forward(x, params, nthreads)


def backward(x, dy, params, nthreads=None):
    return default().backward(x, dy, params, nthreads)
