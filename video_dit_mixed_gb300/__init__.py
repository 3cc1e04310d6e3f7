"""GB300-native hot path of 6Bit-Diffusion's dynamically quantized linear layer.

The compute lives in ``libsixbit.so`` (hand-written CUDA for sm_103a behind a
C ABI, see ``include/sixbit.h``); this package is a thin ctypes binding that
marshals torch tensors (device memory) and streams into those calls.  There is
no CPU fallback: if the library is missing, importing ``ops`` raises.
"""
__all__ = ["ops", "abi"]
