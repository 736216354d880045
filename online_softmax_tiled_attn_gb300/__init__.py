"""Online-softmax tiled attention for GB300 (sm_103a): a C-ABI CUDA library and its binding.

``fa_fwd`` computes exact attention O = softmax(scale * Q K^T [causal]) V and its log-sum-exp,
tile by tile with the online softmax, on hand-written tcgen05/TMA kernels.  ``osm_softmax`` is
the standalone single-pass row softmax.  The CUDA library is loaded on first use; there is no
CPU fallback.
"""
from __future__ import annotations

__all__ = ["fa_fwd", "fa_fwd_splitkv", "osm_softmax", "lib"]


def __getattr__(name):
    if name in ("fa_fwd", "fa_fwd_splitkv", "osm_softmax", "lib", "FaError", "device_status"):
        from . import binding

        return getattr(binding, name)
    raise AttributeError(name)
