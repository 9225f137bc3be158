"""Absorbed Multi-Head Latent Attention (MLA) decode for GB300 (sm_103a).

The decode step reads only the compressed per-token cache (512 latent + 64 rotated
RoPE-key scalars, bf16, in 64-token pages) and never forms per-head K or V.  The
work runs in hand-written CUDA kernels behind the C ABI declared in
``include/mla_decode.h``; :mod:`.ops` is the thin ctypes binding over it.

Importing the package itself loads nothing native, so that the seeded input
generator (:mod:`.workloads`) and the byte/FLOP accounting (:mod:`.accounting`)
can be used on hosts without a GPU.  Importing :mod:`.ops` loads the shared
library and raises if it has not been built.
"""

__all__ = ["workloads", "accounting", "ops"]


def __getattr__(name):
    if name == "ops":
        import importlib
        return importlib.import_module(__name__ + ".ops")
    raise AttributeError(name)
