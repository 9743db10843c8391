"""GB300-native (sm_103a) paged Multi-head Latent Attention decode.

The compute path is the C-ABI library ``libmla.so`` built from ``csrc/``
(hand-written CUDA for sm_103a: tile scheduler, tcgen05/TMA split-KV decode
kernel, LSE combine).  ``api`` is a thin ctypes binding over it; importing the
package does not load the library, so the seeded input generators in
``workloads`` can be used on machines without a GPU.
"""
import importlib

__all__ = ["api", "workloads"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
