"""Paged LATENT (absorbed multi-head latent) attention for GB300 (sm_103a).

The operator runs in libpa_latent.so (C ABI in include/pa_latent.h): a write
phase (partial RoPE + paged scatter of new latent rows) and a read phase
(decode / chunked prefill attention over the paged latent cache).
``binding`` is the ctypes layer, ``api.PagedLatentAttention`` the operator
object, ``workloads`` the seeded synthetic inputs, ``build`` the nvcc build.
"""

__all__ = ["PagedLatentAttention"]


def __getattr__(name):
    if name == "PagedLatentAttention":
        from .api import PagedLatentAttention
        return PagedLatentAttention
    raise AttributeError(name)
