"""Counter-based seeded generator for the synthetic inputs.

This module draws random numbers only.  It holds none of the arithmetic of the
method under test (no summaries, scores, selection or attention): both the
CPU oracle side and the CUDA side take their inputs from here, so both see
bit-identical bf16 tensors.

Definition (every element is a pure function of ``(seed, tag, index)``):

* ``splitmix64`` is the published 64-bit finaliser of Steele, Lea and Flood
  ("Fast splittable pseudorandom number generators", OOPSLA 2014): add the
  golden-ratio increment, then two xor-shift-multiply rounds and a final
  xor-shift, all modulo 2**64.
* A stream base is ``splitmix64(splitmix64(seed) ^ tag)``; element ``i`` of the
  stream hashes ``base + i``.
* ``normal_bf16`` sums the four 16-bit fields of the hash (an Irwin-Hall sum of
  four discrete uniforms, mean 131070), centres it, scales it by the reciprocal
  of its exact standard deviation ``sqrt((65536**2 - 1) / 3)`` in fp32 and
  rounds to bf16 (round-to-nearest-even).  This is a unit-variance stand-in for
  N(0, 1) whose every step is integer-exact or a single IEEE fp32 rounding, so a
  CPU and a GPU evaluation agree bit for bit.

The implementation uses torch int64 tensors, so the same code runs on the CPU
and on a CUDA device.  int64 additions and multiplications wrap modulo 2**64
on both; logical right shifts are written as arithmetic shifts plus a mask.
"""
from __future__ import annotations

import torch

_M64 = (1 << 64) - 1


def _s64(x: int) -> int:
    """The int64 value with the same 64 bits as the unsigned integer ``x``."""
    x &= _M64
    return x - (1 << 64) if x >= (1 << 63) else x


_GOLDEN = 0x9E3779B97F4A7C15
_MIX1 = 0xBF58476D1CE4E5B9
_MIX2 = 0x94D049BB133111EB

# 1 / sqrt((65536**2 - 1) / 3), rounded to fp32
IH4_INV_STD = 2.6428997921303014e-05
IH4_MEAN = 131070


def splitmix64_int(x: int) -> int:
    """splitmix64 of one unsigned 64-bit Python integer (reference form)."""
    z = (x + _GOLDEN) & _M64
    z = ((z ^ (z >> 30)) * _MIX1) & _M64
    z = ((z ^ (z >> 27)) * _MIX2) & _M64
    return z ^ (z >> 31)


def _lsr(x: torch.Tensor, k: int) -> torch.Tensor:
    return (x >> k) & ((1 << (64 - k)) - 1)


def splitmix64(x: torch.Tensor) -> torch.Tensor:
    """splitmix64 applied elementwise to an int64 tensor (bits as unsigned)."""
    z = x + _s64(_GOLDEN)
    z = (z ^ _lsr(z, 30)) * _s64(_MIX1)
    z = (z ^ _lsr(z, 27)) * _s64(_MIX2)
    return z ^ _lsr(z, 31)


def stream_base(seed: int, tag: int) -> int:
    """64-bit base of the stream named by ``(seed, tag)``, as an int64 value."""
    return _s64(splitmix64_int(splitmix64_int(seed & _M64) ^ (tag & _M64)))


def hash64(seed: int, tag: int, index: torch.Tensor) -> torch.Tensor:
    """Raw 64-bit hashes (int64 bits) of the elements ``index`` of a stream."""
    return splitmix64(index.to(torch.int64) + stream_base(seed, tag))


def uniform_u32(seed: int, tag: int, index: torch.Tensor) -> torch.Tensor:
    """Uniform integers in [0, 2**32) (as int64) for the elements ``index``."""
    return _lsr(hash64(seed, tag, index), 32)


def normal_bf16(seed: int, tag: int, index: torch.Tensor) -> torch.Tensor:
    """Unit-variance Irwin-Hall(4) values rounded to bf16, one per index."""
    h = hash64(seed, tag, index)
    s = (h & 0xFFFF) + (_lsr(h, 16) & 0xFFFF) + (_lsr(h, 32) & 0xFFFF) + _lsr(h, 48)
    v = (s - IH4_MEAN).to(torch.float32) * torch.tensor(IH4_INV_STD, dtype=torch.float32)
    return v.to(torch.bfloat16)


def normal_f32(seed: int, tag: int, index: torch.Tensor) -> torch.Tensor:
    """The same Irwin-Hall(4) values as ``normal_bf16``, kept in fp32."""
    h = hash64(seed, tag, index)
    s = (h & 0xFFFF) + (_lsr(h, 16) & 0xFFFF) + (_lsr(h, 32) & 0xFFFF) + _lsr(h, 48)
    return (s - IH4_MEAN).to(torch.float32) * torch.tensor(IH4_INV_STD, dtype=torch.float32)


def random_subset(seed: int, tag: int, offset: int, n: int, k: int) -> torch.Tensor:
    """A uniformly random k-subset of range(n), sorted ascending (CPU int64).

    The subset is the k indices with the smallest (63-bit) hashes of the
    elements ``offset .. offset + n - 1`` of the stream; a stable sort makes
    the choice deterministic even in the (negligible) case of a tie.
    """
    if k > n:
        raise ValueError(f"subset of {k} from {n}")
    idx = torch.arange(offset, offset + n, dtype=torch.int64)
    order = torch.argsort(_lsr(hash64(seed, tag, idx), 1), stable=True)
    return torch.sort(order[:k]).values


def random_order(seed: int, tag: int, offset: int, n: int) -> torch.Tensor:
    """A uniformly random permutation of range(n) (CPU int64)."""
    idx = torch.arange(offset, offset + n, dtype=torch.int64)
    return torch.argsort(_lsr(hash64(seed, tag, idx), 1), stable=True)


def random_signs(seed: int, tag: int, index: torch.Tensor) -> torch.Tensor:
    """+1 / -1 (int64) for each index, each with probability 1/2."""
    return (_lsr(hash64(seed, tag, index), 63) * 2 - 1)
