"""GGUF Q4_K / Q6_K x Q8 integer matmul for GB300 (sm_103a).

The compute path is the CUDA library ``libxq.so`` behind the C ABI in
``include/xq.h``; :mod:`gguf_quant_integer_gb300.xq` is its thin ctypes
binding (argument marshalling only). :mod:`gguf_quant_integer_gb300.synth`
draws the seeded synthetic inputs. Importing this package loads nothing: the
library is opened on first use, and a missing library is an error, never a
fallback.
"""

__all__ = ["xq", "synth", "build"]


def __getattr__(name):
    if name in ("xq", "synth", "build"):
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
