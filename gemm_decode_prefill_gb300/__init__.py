"""gemm_decode_prefill_gb300: low-bit weight-quantized GEMV/GEMM for LLM
inference on GB300 (sm_103a).

The compute lives in libqmv.so (CUDA kernels behind the C ABI in
include/qmv.h); ``qmv`` is its thin Python binding, imported lazily so that
``synth`` (seeded input generation) works without the built library.
"""
import importlib

__all__ = ["qmv", "synth", "build"]


def __getattr__(name):
    if name in ("qmv", "synth", "build"):
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
