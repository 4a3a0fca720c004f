"""GB300 (sm_103a) INT8 convrot linear: group-wise Hadamard-rotated int8 linear.

The layer is the one the page "INT8 Convrot Safetensors" (stable-diffusion.cpp
docs) defines: rotate activation rows group-wise by a normalized Kronecker
power of H4, quantize each row to int8 with one absmax scale, multiply by
identically rotated per-row-quantized int8 weights with exact integer
accumulation, and reconstruct Y = A * s_x * s_w + b.

Everything runs in libconvrot's CUDA kernels (C ABI in include/convrot.h);
``convrot`` is the ctypes binding, ``inputs`` the seeded synthetic workloads.
"""

from . import inputs  # noqa: F401

__all__ = ["inputs", "convrot"]


def __getattr__(name):
    if name == "convrot":
        import importlib

        return importlib.import_module(__name__ + ".convrot")
    raise AttributeError(name)
