"""Exact scaled-dot-product attention (forward and backward) for one NVIDIA
GB300, as hand-written sm_103a CUDA behind a C ABI (include/fa.h).

The Python surface is a thin ctypes binding: ``fwd``, ``bwd`` and helpers.
The library is built in-tree by ``exact_attention_78_gb300.build.build()``.
"""

from .binding import (  # noqa: F401
    FAError,
    bwd,
    bwd_workspace_size,
    exp2_probe,
    fwd,
    get_device_error,
    lib_path,
    load_library,
    status_string,
    wait_timeout_probe,
)
