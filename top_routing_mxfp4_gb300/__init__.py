"""GB300-native forward pass of a LatentMoE layer (top-16 of 896 experts,
SwiGLU experts on MXFP4 weights), as a C-ABI CUDA library for sm_103a.

`top_routing_mxfp4_gb300.lmoe` is the ctypes binding of liblmoe.so (see
include/lmoe.h); `top_routing_mxfp4_gb300.build` compiles it.  Neither is
imported here, so building does not need the library to exist yet.
"""
__all__ = ["build", "lmoe"]
