"""Seeded synthetic inputs for the CSA fused Compressor.

This module is shared by the tests, the benchmark and the smoke check. It
holds random-number generation and the shapes of the workloads only -- none of
the Compressor's arithmetic.

Generator (documented so that any other implementation can reproduce it):
  * SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
    generators", OOPSLA 2014) used counter-style: draw i of stream s under
    seed S is mix64(key(S, s) + (i + 1) * 0x9E3779B97F4A7C15 mod 2^64), with
    key(S, s) = mix64((S + 1) * 0x9E3779B97F4A7C15 xor s * 0xD1B54A32D192ED03).
  * uniform in (0, 1): ((z >> 11) + 0.5) * 2^-53.
  * normal: Box-Muller on consecutive uniform pairs (u1, u2):
    sqrt(-2 ln u1) * cos(2 pi u2), sqrt(-2 ln u1) * sin(2 pi u2).
  * bf16 data: the fp64 normal times sigma, rounded to fp32, then to bf16 with
    round-to-nearest-even on the bit pattern.
  * uniform integers in [1, n]: 1 + floor(u * n).

Value distributions follow the page's gate distribution (cuDNN-frontend "CSA
Fused Compressor", section "Numerics", tolerance item 2): kv and grad_out
N(0, 1) bf16, score N(0, 1.5^2) bf16, ape N(0, 0.25^2) fp32.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_STREAM_MUL = 0xD1B54A32D192ED03
_MASK64 = (1 << 64) - 1

STREAM_KV, STREAM_SCORE, STREAM_APE, STREAM_GRAD, STREAM_LENS = 1, 2, 3, 4, 5

SIGMA_KV, SIGMA_SCORE, SIGMA_APE, SIGMA_GRAD = 1.0, 1.5, 0.25, 1.0

_CHUNK = 1 << 20


def _mix64_int(z: int) -> int:
    z &= _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, stream: int) -> int:
    return _mix64_int(((seed + 1) * 0x9E3779B97F4A7C15) ^ ((stream * _STREAM_MUL) & _MASK64))


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def raw_u64(key: int, start: int, count: int) -> np.ndarray:
    """Draws start .. start+count-1 of the stream with this key."""
    with np.errstate(over="ignore"):
        idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        return _mix64(np.uint64(key) + idx * _GAMMA)


def _uniform(key: int, start: int, count: int) -> np.ndarray:
    z = raw_u64(key, start, count)
    return ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def _normal_chunk(key: int, start: int, count: int) -> np.ndarray:
    # `start` and `count` are even: pair i uses draws (2i, 2i+1)
    u = _uniform(key, start, count)
    u1, u2 = u[0::2], u[1::2]
    rad = np.sqrt(-2.0 * np.log(u1))
    ang = (2.0 * np.pi) * u2
    out = np.empty(count, dtype=np.float64)
    out[0::2] = rad * np.cos(ang)
    out[1::2] = rad * np.sin(ang)
    return out


def _workers() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _fill_chunked(n: int, fn, dtype) -> np.ndarray:
    out = np.empty(n, dtype=dtype)
    starts = list(range(0, n, _CHUNK))

    def work(lo: int):
        hi = min(n, lo + _CHUNK)
        out[lo:hi] = fn(lo, hi - lo)

    if len(starts) <= 1:
        for lo in starts:
            work(lo)
    else:
        with ThreadPoolExecutor(_workers()) as ex:
            list(ex.map(work, starts))
    return out


def normal_f64(seed: int, stream: int, n: int, sigma: float = 1.0) -> np.ndarray:
    key = stream_key(seed, stream)
    npad = n + (n & 1)
    out = _fill_chunked(npad, lambda lo, c: _normal_chunk(key, lo, c + (c & 1))[:c] * sigma,
                        np.float64)
    return out[:n]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest-even on the bit pattern); finite inputs."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    with np.errstate(over="ignore"):
        return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def normal_bf16(seed: int, stream: int, n: int, sigma: float) -> np.ndarray:
    key = stream_key(seed, stream)

    def chunk(lo: int, c: int):
        v = _normal_chunk(key, lo, c + (c & 1))[:c] * sigma
        return f32_to_bf16_bits(v.astype(np.float32))

    return _fill_chunked(n, chunk, np.uint16)


def uniform_int(seed: int, stream: int, n: int, hi: int) -> np.ndarray:
    """n integers uniform in [1, hi]."""
    u = _uniform(stream_key(seed, stream), 0, n)
    return (1 + np.floor(u * hi)).astype(np.int64)


# --------------------------------------------------------------------------
# Cases


@dataclass
class Case:
    name: str
    ratio: int
    coff: int
    head_dim: int
    seqlens: np.ndarray               # int64 [B]
    total_tokens: int                 # rows of kv / score (>= cu_seqlens[-1])
    capacity: int                     # rows of out / grad_out
    seed: int = 0
    cu_seqlens: np.ndarray = field(init=False)
    cu_seqlens_comp: np.ndarray = field(init=False)
    kv: Optional[np.ndarray] = None       # uint16 bf16 bits [T, coff*d]
    score: Optional[np.ndarray] = None    # uint16 bf16 bits [T, coff*d]
    ape: Optional[np.ndarray] = None      # float32 [ratio, coff*d]
    grad_out: Optional[np.ndarray] = None # uint16 bf16 bits [capacity, d]

    def __post_init__(self):
        lens = np.asarray(self.seqlens, dtype=np.int64)
        self.seqlens = lens
        cu = np.zeros(len(lens) + 1, dtype=np.int64)
        cu[1:] = np.cumsum(lens)
        cuc = np.zeros(len(lens) + 1, dtype=np.int64)
        cuc[1:] = np.cumsum(lens // self.ratio)
        self.cu_seqlens = cu.astype(np.int32)
        self.cu_seqlens_comp = cuc.astype(np.int32)

    @property
    def num_seqs(self) -> int:
        return len(self.seqlens)

    @property
    def true_rows(self) -> int:
        return int(self.cu_seqlens_comp[-1])

    @property
    def width(self) -> int:
        return self.coff * self.head_dim

    def fill(self) -> "Case":
        t, w, r, d, s = self.total_tokens, self.width, self.ratio, self.head_dim, self.seed
        self.kv = normal_bf16(s, STREAM_KV, t * w, SIGMA_KV).reshape(t, w)
        self.score = normal_bf16(s, STREAM_SCORE, t * w, SIGMA_SCORE).reshape(t, w)
        self.ape = normal_f64(s, STREAM_APE, r * w, SIGMA_APE).astype(np.float32).reshape(r, w)
        self.grad_out = normal_bf16(s, STREAM_GRAD, self.capacity * d, SIGMA_GRAD).reshape(
            self.capacity, d)
        return self


def make_case(name: str, seqlens, ratio: int, coff: int, head_dim: int,
              pad_rows: int = 0, extra_tokens: int = 0, seed: int = 0,
              fill: bool = True) -> Case:
    """A case over the given segment lengths; `pad_rows` static-capacity rows
    beyond the true compressed rows and `extra_tokens` kv rows beyond the last
    segment (both never consumed by a true row)."""
    lens = np.asarray(seqlens, dtype=np.int64)
    true_rows = int(np.sum(lens // ratio))
    c = Case(name, ratio, coff, head_dim, lens, int(lens.sum()) + extra_tokens,
             true_rows + pad_rows, seed)
    return c.fill() if fill else c


def headline_seqlens(seed: int = 0, total: int = 262144, nseg: int = 64,
                     max_len: int = 8191) -> np.ndarray:
    """64 lengths U{1..8191} renormalised to `total` tokens: floor(L_i * total / sum L),
    at least 1, then the remainder added one token at a time to segments 0, 1, 2, ..."""
    raw = uniform_int(seed, STREAM_LENS, nseg, max_len)
    lens = np.maximum(1, (raw * total) // int(raw.sum()))
    rem = total - int(lens.sum())
    i = 0
    while rem != 0:
        step = 1 if rem > 0 else -1
        if step > 0 or lens[i % nseg] > 1:
            lens[i % nseg] += step
            rem -= step
        i += 1
    return lens


CONFIG_NAMES = ("tiny", "r4d512", "r2d128rag", "r128c1", "headline")


def config(name: str, seed: int = 0, fill: bool = True) -> Case:
    """The five workloads: a tiny case, three mid-size cases and the 256k-token headline."""
    if name == "tiny":
        # r=4, coff=2, d=64, lengths [37, 64, 19] (tails dropped), 4 padding rows
        return make_case(name, [37, 64, 19], 4, 2, 64, pad_rows=4, seed=seed, fill=fill)
    if name == "r4d512":
        return make_case(name, [4096] * 8, 4, 2, 512, seed=seed, fill=fill)
    if name == "r2d128rag":
        lens = uniform_int(seed, STREAM_LENS, 32, 4095)
        return make_case(name, lens, 2, 2, 128, seed=seed, fill=fill)
    if name == "r128c1":
        return make_case(name, [8192] * 16, 128, 1, 512, seed=seed, fill=fill)
    if name == "headline":
        return make_case(name, headline_seqlens(seed), 4, 2, 512, pad_rows=1024, seed=seed,
                         fill=fill)
    if name.startswith("pack-"):
        return pack(name, seed=seed, fill=fill)
    raise KeyError(name)


def pack(spec: str, seed: int = 0, fill: bool = True) -> Case:
    """A THD pack of equal segments, spelt `pack-r{ratio}c{coff}d{head_dim}-{n}x{len}`
    (e.g. `pack-r4c2d128-3x8192`): the segment counts and lengths at which the
    cuDNN-frontend "CSA Fused Compressor" page quotes its kernel times; no
    padding rows, the page's gate distribution."""
    import re
    m = re.fullmatch(r"pack-r(\d+)c([12])d(\d+)-(\d+)x(\d+)", spec)
    if m is None:
        raise KeyError(spec)
    r, coff, d, n, length = (int(x) for x in m.groups())
    return make_case(spec, [length] * n, r, coff, d, seed=seed, fill=fill)
