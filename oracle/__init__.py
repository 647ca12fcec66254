"""CPU oracle of the CSA/HCA fused Compressor -- TEST INFRASTRUCTURE ONLY.

A plain, slow C++ statement of the gated-softmax pooling defined on the
cuDNN-frontend "CSA Fused Compressor" page (sections "Semantics" and
"Numerics"), with an fp32 eager-order twin (O32) and an fp64 twin (O64).
Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package; the CUDA library never does.

``build()`` compiles ``csa_oracle.cpp`` with g++ (``-O2 -ffp-contract=off``,
OpenMP) into ``oracle/_build/libcsa_oracle.so``. Arrays are numpy: bf16 data
travels as ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa_oracle.cpp")
_HDR = os.path.join(_HERE, "csa_oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libcsa_oracle.so")

CXXFLAGS = ["-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
            "-fPIC", "-shared", "-Wall", "-Wextra"]

ERRORS = {0: "ok", 1: "bad argument", 2: "bad cu_seqlens", 3: "bad cu_seqlens_comp",
          4: "bad capacity"}

_lock = threading.Lock()
_lib = None


class OracleError(RuntimeError):
    def __init__(self, code: int):
        super().__init__(f"oracle rejected the inputs: {ERRORS.get(code, code)} (code {code})")
        self.code = code


def _stale() -> bool:
    if not os.path.exists(_LIB_PATH):
        return True
    t = os.path.getmtime(_LIB_PATH)
    return any(os.path.getmtime(p) > t for p in (_SRC, _HDR))


def build(force: bool = False) -> str:
    """Compile the oracle shared library (idempotent); returns its path."""
    with _lock:
        if force or _stale():
            os.makedirs(_OUT_DIR, exist_ok=True)
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            cmd = ["g++", *CXXFLAGS, _SRC, "-o", tmp]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    i32, i64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
    lib.oracle_exp_f32.argtypes = [ctypes.c_float]
    lib.oracle_exp_f32.restype = ctypes.c_float
    lib.oracle_exp_f32_n.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
    lib.oracle_exp_f32_n.restype = None
    lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
    lib.oracle_mul_add_f32.argtypes = [ctypes.c_float] * 3
    lib.oracle_mul_add_f32.restype = ctypes.c_float
    lib.oracle_row_map.argtypes = [vp, vp, i32, i64, i32, vp, vp, vp]
    lib.oracle_window_slot.argtypes = [i32, i32, i32, i64, i32, i32, i32, vp, vp, vp, vp]
    lib.oracle_window_slot.restype = None
    lib.oracle_validate.argtypes = [vp, vp, i32, i64, i64, i32, i32, i32]
    common = [vp, vp, vp, vp, vp, i32, i64, i64, i32, i32, i32]
    lib.oracle_fwd32.argtypes = common + [vp, vp, i32]
    lib.oracle_bwd32.argtypes = common + [vp, vp, vp, vp, i32]
    lib.oracle_fwd64.argtypes = common + [vp, i32]
    lib.oracle_bwd64.argtypes = common + [vp, vp, vp, vp, i32]
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


@dataclass
class Problem:
    """Segment structure and sizes of one Compressor call."""
    cu_seqlens: np.ndarray       # int32 [B+1]
    cu_seqlens_comp: np.ndarray  # int32 [B+1]
    total_tokens: int
    capacity: int
    ratio: int
    coff: int
    head_dim: int

    @property
    def num_seqs(self) -> int:
        return int(self.cu_seqlens.shape[0] - 1)

    @property
    def width(self) -> int:
        return self.coff * self.head_dim

    def _args(self):
        cu = np.ascontiguousarray(self.cu_seqlens, dtype=np.int32)
        cuc = np.ascontiguousarray(self.cu_seqlens_comp, dtype=np.int32)
        return cu, cuc, [_ptr(cu), _ptr(cuc), self.num_seqs, int(self.total_tokens),
                         int(self.capacity), int(self.ratio), int(self.coff),
                         int(self.head_dim)]


def _check(rc: int):
    if rc != 0:
        raise OracleError(rc)


def validate(p: Problem) -> int:
    lib = _load()
    cu, cuc, args = p._args()
    return lib.oracle_validate(*args)


def exp_f32(x: float) -> float:
    return _load().oracle_exp_f32(x)


def exp_f32_array(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty_like(x)
    _load().oracle_exp_f32_n(_ptr(x), _ptr(y), x.size)
    return y


def f32_to_bf16(x: float) -> int:
    return _load().oracle_f32_to_bf16(x)


def mul_add_f32(a: float, b: float, c: float) -> float:
    return _load().oracle_mul_add_f32(a, b, c)


def row_map(p: Problem, row: int):
    """(base_token, first_in_segment, padding) of one output row."""
    lib = _load()
    cu, cuc, _ = p._args()
    base = ctypes.c_int64()
    first = ctypes.c_int32()
    pad = ctypes.c_int32()
    _check(lib.oracle_row_map(_ptr(cu), _ptr(cuc), p.num_seqs, row, p.ratio,
                              ctypes.byref(base), ctypes.byref(first), ctypes.byref(pad)))
    return base.value, bool(first.value), bool(pad.value)


def window_slot(p: Problem, base: int, first: bool, j: int, k: int):
    """(token, col, ape_row, valid) of window slot k for output column j."""
    lib = _load()
    tok = ctypes.c_int64()
    col = ctypes.c_int32()
    arow = ctypes.c_int32()
    valid = ctypes.c_int32()
    lib.oracle_window_slot(p.ratio, p.coff, p.head_dim, base, int(first), j, k,
                           ctypes.byref(tok), ctypes.byref(col), ctypes.byref(arow),
                           ctypes.byref(valid))
    return tok.value, col.value, arow.value, bool(valid.value)


def fwd32(p: Problem, kv: np.ndarray, score: np.ndarray, ape: np.ndarray,
          nthreads: int = 0, want_f32: bool = False):
    """O32 forward: out [capacity, head_dim] as bf16 bits (and the fp32 pre-rounding values)."""
    lib = _load()
    cu, cuc, args = p._args()
    kv = np.ascontiguousarray(kv, dtype=np.uint16)
    score = np.ascontiguousarray(score, dtype=np.uint16)
    ape = np.ascontiguousarray(ape, dtype=np.float32)
    assert kv.shape == (p.total_tokens, p.width) and score.shape == kv.shape
    assert ape.shape == (p.ratio, p.width)
    out = np.empty((p.capacity, p.head_dim), dtype=np.uint16)
    out_f = np.empty((p.capacity, p.head_dim), dtype=np.float32) if want_f32 else None
    _check(lib.oracle_fwd32(_ptr(kv), _ptr(score), _ptr(ape), *args, _ptr(out),
                            _ptr(out_f) if want_f32 else None, nthreads))
    return (out, out_f) if want_f32 else out


def bwd32(p: Problem, kv, score, ape, grad_out, nthreads: int = 0):
    """O32 backward: (dkv, dscore) bf16 bits [T, coff*d] and dape fp32 [ratio, coff*d]."""
    lib = _load()
    cu, cuc, args = p._args()
    kv = np.ascontiguousarray(kv, dtype=np.uint16)
    score = np.ascontiguousarray(score, dtype=np.uint16)
    ape = np.ascontiguousarray(ape, dtype=np.float32)
    grad_out = np.ascontiguousarray(grad_out, dtype=np.uint16)
    assert grad_out.shape == (p.capacity, p.head_dim)
    dkv = np.empty((p.total_tokens, p.width), dtype=np.uint16)
    dscore = np.empty_like(dkv)
    dape = np.empty((p.ratio, p.width), dtype=np.float32)
    _check(lib.oracle_bwd32(_ptr(kv), _ptr(score), _ptr(ape), *args, _ptr(grad_out),
                            _ptr(dkv), _ptr(dscore), _ptr(dape), nthreads))
    return dkv, dscore, dape


def fwd64(p: Problem, kv, score, ape, nthreads: int = 0):
    """O64 forward on fp64 inputs: out [capacity, head_dim] float64."""
    lib = _load()
    cu, cuc, args = p._args()
    kv = np.ascontiguousarray(kv, dtype=np.float64)
    score = np.ascontiguousarray(score, dtype=np.float64)
    ape = np.ascontiguousarray(ape, dtype=np.float64)
    out = np.empty((p.capacity, p.head_dim), dtype=np.float64)
    _check(lib.oracle_fwd64(_ptr(kv), _ptr(score), _ptr(ape), *args, _ptr(out), nthreads))
    return out


def bwd64(p: Problem, kv, score, ape, grad_out, nthreads: int = 0):
    """O64 backward on fp64 inputs: (dkv, dscore, dape) float64."""
    lib = _load()
    cu, cuc, args = p._args()
    kv = np.ascontiguousarray(kv, dtype=np.float64)
    score = np.ascontiguousarray(score, dtype=np.float64)
    ape = np.ascontiguousarray(ape, dtype=np.float64)
    grad_out = np.ascontiguousarray(grad_out, dtype=np.float64)
    dkv = np.empty((p.total_tokens, p.width), dtype=np.float64)
    dscore = np.empty_like(dkv)
    dape = np.empty((p.ratio, p.width), dtype=np.float64)
    _check(lib.oracle_bwd64(_ptr(kv), _ptr(score), _ptr(ape), *args, _ptr(grad_out),
                            _ptr(dkv), _ptr(dscore), _ptr(dape), nthreads))
    return dkv, dscore, dape


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (plain bit placement, no rounding)."""
    return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
