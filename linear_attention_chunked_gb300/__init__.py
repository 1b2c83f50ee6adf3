"""GB300-native (sm_103a) chunked KDA (Kimi Delta Attention) training kernels.

The compute lives in the CUDA library built from csrc/ (C ABI: include/kda.h); ``kda`` is its
ctypes binding, ``inputs`` the seeded workload generator, ``build`` the nvcc build step.
Import ``linear_attention_chunked_gb300.kda`` for the entry points.
"""
__all__ = ["kda", "inputs", "build"]
