"""GB300 (sm_103a) MoE expert-FFN layer: router top-k -> permutation by expert -> gate/up GEMMs
with fused SwiGLU -> down GEMM -> weighted sum, over MXFP4 expert weights.

The compute lives in ``libmoe_gb300.so`` (hand-written CUDA, C ABI in ``include/moe.h``);
``binding`` is the ctypes layer with the same entry-point names; ``layer`` builds a synthetic
device-resident layer; ``inputs`` holds the seeded input generators.
"""
__all__ = ["binding", "inputs", "layer"]


def __getattr__(name):
    import importlib
    if name in __all__:
        return importlib.import_module("." + name, __name__)
    raise AttributeError(name)
