"""GB300 (sm_103a) CSA/HCA fused Compressor.

The gated-softmax pooling of the cuDNN-frontend "CSA Fused Compressor" page
as hand-written CUDA kernels behind a small C ABI (include/csa_compress.h);
this package holds the kernels (csrc/), their build and a thin Python binding.
"""
from .binding import (SEG_VIOLATIONS, CsaError, csa_check_segments, csa_compress_bwd,
                      csa_compress_bwd_noalloc_ptr, csa_compress_bwd_ptr, csa_compress_fwd,
                      csa_compress_fwd_ptr, load)
from .nvbuild import build

__all__ = ["SEG_VIOLATIONS", "CsaError", "build", "csa_check_segments", "csa_compress_bwd",
           "csa_compress_bwd_noalloc_ptr", "csa_compress_bwd_ptr", "csa_compress_fwd",
           "csa_compress_fwd_ptr", "load"]
