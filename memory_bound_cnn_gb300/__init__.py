"""GB300-native WTConv layer (forward + backward) behind a C ABI, with a thin Python binding.

The compute path is ``libwtconv.so`` (CUDA kernels for sm_103a, built in-tree by ``_build``);
``wtconv`` marshals PyTorch tensors into it.  ``inputs`` makes the seeded synthetic workloads.
"""
from . import inputs  # noqa: F401
from .wtconv import (  # noqa: F401
    WTConvError,
    WTConvFunction,
    wtconv_backward,
    wtconv_backward_input,
    wtconv_backward_weights,
    wtconv_forward,
    wtconv_strerror,
    wtconv_version,
    wtconv_workspace_size,
)
