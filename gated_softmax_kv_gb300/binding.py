"""Python binding of the C ABI in include/csa_compress.h (argument marshalling only).

Every computation runs in libcsa_compress.so; this module checks tensor
dtypes/devices/shapes, derives the sizes the C calls want from tensor shapes,
and raises ``CsaError`` on a nonzero status. There is no CPU or eager
fallback: if the library is missing the call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import nvbuild as _build

LIB_PATH = _build.LIB

CSA_STATUS = {0: "CSA_OK", 1: "CSA_ERR_NULL", 2: "CSA_ERR_ALIGN", 3: "CSA_ERR_UNSUPPORTED",
              4: "CSA_ERR_RANGE", 5: "CSA_ERR_CUDA", 6: "CSA_ERR_SCRATCH"}

_lib = None


class CsaError(RuntimeError):
    def __init__(self, status: int, detail: str = ""):
        self.status = status
        name = CSA_STATUS.get(status, str(status))
        super().__init__(f"{name}: {detail}")


def load() -> ctypes.CDLL:
    """Load libcsa_compress.so (built by ``gated_softmax_kv_gb300.nvbuild.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build the CUDA library first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    common = [vp, vp, vp, vp, vp, i32, i64, i64, i32, i32, i32]
    lib.csa_compress_fwd.argtypes = common + [vp, vp]
    lib.csa_compress_fwd.restype = ctypes.c_int
    lib.csa_compress_bwd.argtypes = common + [vp, vp, vp, vp, vp]
    lib.csa_compress_bwd.restype = ctypes.c_int
    lib.csa_compress_fwd_exact.argtypes = common + [vp, vp]
    lib.csa_compress_fwd_exact.restype = ctypes.c_int
    lib.csa_compress_bwd_exact.argtypes = common + [vp, vp, vp, vp, vp]
    lib.csa_compress_bwd_exact.restype = ctypes.c_int
    lib.csa_compress_bwd_noalloc.argtypes = common + [vp, vp, vp, vp, vp]
    lib.csa_compress_bwd_noalloc.restype = ctypes.c_int
    lib.csa_check_segments.argtypes = [vp, vp, i32, i64, i64, i32, vp, vp]
    lib.csa_check_segments.restype = ctypes.c_int
    lib.csa_status_string.argtypes = [ctypes.c_int]
    lib.csa_status_string.restype = ctypes.c_char_p
    lib.csa_last_cuda_error.argtypes = []
    lib.csa_last_cuda_error.restype = i32
    _lib = lib
    return lib


def _raise(status: int):
    lib = load()
    detail = lib.csa_status_string(status).decode()
    if status == 5:
        detail += f" (cudaError {lib.csa_last_cuda_error()})"
    raise CsaError(status, detail)


# ------------------------------------------------------------- raw pointers


def csa_compress_fwd_ptr(kv: int, score: int, ape: int, cu_seqlens: int, cu_seqlens_comp: int,
                         num_seqs: int, total_tokens: int, capacity: int, ratio: int, coff: int,
                         head_dim: int, out: int, stream: int = 0, exact: bool = False) -> None:
    lib = load()
    fn = lib.csa_compress_fwd_exact if exact else lib.csa_compress_fwd
    st = fn(kv, score, ape, cu_seqlens, cu_seqlens_comp, num_seqs, total_tokens, capacity, ratio,
            coff, head_dim, out, stream)
    if st != 0:
        _raise(st)


def csa_compress_bwd_ptr(kv: int, score: int, ape: int, cu_seqlens: int, cu_seqlens_comp: int,
                         num_seqs: int, total_tokens: int, capacity: int, ratio: int, coff: int,
                         head_dim: int, grad_out: int, dkv: int, dscore: int, dape: int,
                         stream: int = 0, exact: bool = False) -> None:
    lib = load()
    fn = lib.csa_compress_bwd_exact if exact else lib.csa_compress_bwd
    st = fn(kv, score, ape, cu_seqlens, cu_seqlens_comp, num_seqs, total_tokens, capacity, ratio,
            coff, head_dim, grad_out, dkv, dscore, dape, stream)
    if st != 0:
        _raise(st)


# ------------------------------------------------------------- torch tensors


def _check_detail(t, name, dtype, dev, ndim):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor, got one on {t.device}")
    if t.get_device() != dev:
        raise ValueError(f"{name} is on {t.device}, expected cuda:{dev}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")
    raise ValueError(f"{name} is not a valid argument")


def _check(t, name, dtype, dev: int, ndim=None):
    """dtype, CUDA device index, contiguity and rank in one test (tensor
    attribute reads dominate the host cost of a call); the specific error is
    worked out only when the test fails."""
    try:
        ok = (t.dtype is dtype and t.get_device() == dev and t.is_contiguous()
              and (ndim is None or t.dim() == ndim))
    except AttributeError:
        ok = False
    if not ok:
        _check_detail(t, name, dtype, dev, ndim)


_raw_stream = None


def _stream_handle(stream, dev: int) -> int:
    """The CUDA stream to launch on: `stream`, else the current stream of the
    device (read as a raw handle where torch offers that, which avoids
    building a Stream object per call)."""
    global _raw_stream
    if stream is not None:
        return int(stream.cuda_stream)
    import torch
    if _raw_stream is None:
        _raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", False)
    if _raw_stream:
        return int(_raw_stream(dev))
    return int(torch.cuda.current_stream(dev).cuda_stream)


def _shapes(kv, score, ape, cu_seqlens, cu_seqlens_comp, ratio, coff, head_dim):
    import torch
    dev = kv.get_device() if isinstance(kv, torch.Tensor) else -1
    if dev < 0:  # also rejects CPU tensors: the kernels take device pointers
        _check_detail(kv, "kv", torch.bfloat16, 0, 2)
    _check(kv, "kv", torch.bfloat16, dev, 2)
    _check(score, "score", torch.bfloat16, dev, 2)
    _check(ape, "ape", torch.float32, dev, 2)
    _check(cu_seqlens, "cu_seqlens", torch.int32, dev, 1)
    _check(cu_seqlens_comp, "cu_seqlens_comp", torch.int32, dev, 1)
    ks = kv.shape
    if ks != score.shape or ks[1] != coff * head_dim:
        raise ValueError("kv and score must both be [total_tokens, coff*head_dim]")
    if ape.shape != (ratio, coff * head_dim):
        raise ValueError("ape must be [ratio, coff*head_dim]")
    n = cu_seqlens.shape[0]
    if cu_seqlens_comp.shape[0] != n or n < 2:
        raise ValueError("cu_seqlens and cu_seqlens_comp must both be [num_seqs + 1]")
    return dev, n - 1, ks[0]


def csa_compress_fwd(kv, score, ape, cu_seqlens, cu_seqlens_comp, capacity: int, ratio: int,
                     coff: int, head_dim: int, out=None, stream=None, exact: bool = False):
    """Forward on device tensors; returns out [capacity, head_dim] bf16.
    exact=True calls csa_compress_fwd_exact (windows of at most 8 slots)."""
    import torch
    dev, nseq, T = _shapes(kv, score, ape, cu_seqlens, cu_seqlens_comp, ratio, coff, head_dim)
    if out is None:
        out = torch.empty((capacity, head_dim), dtype=torch.bfloat16, device=dev)
    _check(out, "out", torch.bfloat16, dev, 2)
    if tuple(out.shape) != (capacity, head_dim):
        raise ValueError("out must be [capacity, head_dim]")
    csa_compress_fwd_ptr(kv.data_ptr(), score.data_ptr(), ape.data_ptr(), cu_seqlens.data_ptr(),
                         cu_seqlens_comp.data_ptr(), nseq, T, capacity, ratio, coff, head_dim,
                         out.data_ptr(), _stream_handle(stream, dev), exact)
    return out


def csa_compress_bwd(kv, score, ape, cu_seqlens, cu_seqlens_comp, capacity: int, ratio: int,
                     coff: int, head_dim: int, grad_out, dkv=None, dscore=None, dape=None,
                     stream=None, exact: bool = False):
    """Backward on device tensors; returns (dkv, dscore, dape). dkv/dscore may be
    uninitialised; dape is overwritten. exact=True calls csa_compress_bwd_exact
    (windows of at most 8 slots)."""
    import torch
    dev, nseq, T = _shapes(kv, score, ape, cu_seqlens, cu_seqlens_comp, ratio, coff, head_dim)
    _check(grad_out, "grad_out", torch.bfloat16, dev, 2)
    if tuple(grad_out.shape) != (capacity, head_dim):
        raise ValueError("grad_out must be [capacity, head_dim]")
    if dkv is None:
        dkv = torch.empty_like(kv)
    if dscore is None:
        dscore = torch.empty_like(score)
    if dape is None:
        dape = torch.empty_like(ape)
    _check(dkv, "dkv", torch.bfloat16, dev, 2)
    _check(dscore, "dscore", torch.bfloat16, dev, 2)
    _check(dape, "dape", torch.float32, dev, 2)
    if dkv.shape != kv.shape or dscore.shape != kv.shape or dape.shape != ape.shape:
        raise ValueError("gradient buffers must match kv / score / ape")
    csa_compress_bwd_ptr(kv.data_ptr(), score.data_ptr(), ape.data_ptr(), cu_seqlens.data_ptr(),
                         cu_seqlens_comp.data_ptr(), nseq, T, capacity, ratio, coff, head_dim,
                         grad_out.data_ptr(), dkv.data_ptr(), dscore.data_ptr(), dape.data_ptr(),
                         _stream_handle(stream, dev), exact)
    return dkv, dscore, dape


# ------------------------------------------------------------- no-allocation backward

NOALLOC_SCRATCH_FLOATS = 4 * 1024 * 1024


def csa_compress_bwd_noalloc_ptr(kv: int, score: int, ape: int, cu_seqlens: int,
                                 cu_seqlens_comp: int, num_seqs: int, total_tokens: int,
                                 capacity: int, ratio: int, coff: int, head_dim: int,
                                 grad_out: int, dkv: int, dscore: int, dape: int,
                                 stream: int = 0) -> None:
    """csa_compress_bwd_noalloc on raw device pointers: the backward for callers
    that cannot allocate device memory at call time. Its dape partials use the
    library's fixed 16 MiB device buffer, shared by every call (calls that
    overlap on the GPU race on it); raises CsaError(CSA_ERR_SCRATCH) when a
    problem needs more than that."""
    lib = load()
    fn = lib.csa_compress_bwd_noalloc
    st = fn(kv, score, ape, cu_seqlens, cu_seqlens_comp, num_seqs, total_tokens, capacity, ratio,
            coff, head_dim, grad_out, dkv, dscore, dape, stream)
    if st != 0:
        _raise(st)


# ------------------------------------------------------------- segment check

SEG_VIOLATIONS = {1: "cu_seqlens[0] or cu_seqlens_comp[0] is not 0",
                  2: "cu_seqlens decreases",
                  4: "cu_seqlens_comp does not step by floor(seqlen / ratio)",
                  8: "cu_seqlens[-1] > total_tokens",
                  16: "cu_seqlens_comp[-1] > capacity (rows past capacity get no output slot)"}


def csa_check_segments(cu_seqlens, cu_seqlens_comp, total_tokens: int, capacity: int, ratio: int,
                       stream=None) -> int:
    """The device-side preconditions of the segment arrays (csa_check_segments):
    returns the bitmask of violations, 0 when they all hold. Reads the result
    back, so it synchronises the stream: a debugging aid, not for the hot loop."""
    import torch
    dev = cu_seqlens.get_device() if isinstance(cu_seqlens, torch.Tensor) else -1
    if dev < 0:
        _check_detail(cu_seqlens, "cu_seqlens", torch.int32, 0, 1)
    _check(cu_seqlens, "cu_seqlens", torch.int32, dev, 1)
    _check(cu_seqlens_comp, "cu_seqlens_comp", torch.int32, dev, 1)
    n = cu_seqlens.shape[0]
    if cu_seqlens_comp.shape[0] != n or n < 2:
        raise ValueError("cu_seqlens and cu_seqlens_comp must both be [num_seqs + 1]")
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    with torch.cuda.stream(stream):
        word = torch.zeros(1, dtype=torch.int32, device=dev)  # zeroed in stream order
    st = load().csa_check_segments(cu_seqlens.data_ptr(), cu_seqlens_comp.data_ptr(), n - 1,
                                   total_tokens, capacity, ratio, word.data_ptr(),
                                   int(stream.cuda_stream))
    if st != 0:
        _raise(st)
    stream.synchronize()
    return int(word.cpu()[0])
