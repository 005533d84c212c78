"""Counter-based random numbers for the synthetic verification workloads.

Philox4x32-10 (Salmon, Moraes, Dror & Shaw, "Parallel random numbers: as easy
as 1, 2, 3", SC 2011): a 128-bit counter and a 64-bit key go through ten rounds
of two 32x32->64 multiplies plus xors, with a Weyl sequence bumping the key
between rounds.  Written here with torch integer ops only, so the same seed,
stream and element index give the same 32-bit words on the CPU and on a GPU
(the multiplies are split into 16-bit limbs, so no int64 product overflows).

This module draws the inputs of the workloads; it holds none of the
verification arithmetic.
"""
from __future__ import annotations

import math

import torch

_MASK32 = 0xFFFFFFFF
_M0 = 0xD2511F53
_M1 = 0xCD9E8D57
_W0 = 0x9E3779B9
_W1 = 0xBB67AE85


def _mulhilo(a: torch.Tensor, m: int) -> tuple[torch.Tensor, torch.Tensor]:
    """hi and lo 32-bit words of a*m for a in [0, 2^32) (int64 tensor), m a 32-bit constant."""
    a1 = a >> 16
    a0 = a & 0xFFFF
    m1 = m >> 16
    m0 = m & 0xFFFF
    lo_part = a0 * m0                      # < 2^32
    mid = a1 * m0 + a0 * m1                # < 2^33
    hi_part = a1 * m1                      # < 2^32
    lo = lo_part + ((mid & 0xFFFF) << 16)  # < 2^33
    carry = lo >> 32
    lo = lo & _MASK32
    hi = (hi_part + (mid >> 16) + carry) & _MASK32
    return hi, lo


def philox4x32_10(c0, c1, c2, c3, k0: int, k1: int):
    """Ten Philox rounds on int64 tensors holding uint32 counter words."""
    for r in range(10):
        if r:
            k0 = (k0 + _W0) & _MASK32
            k1 = (k1 + _W1) & _MASK32
        hi0, lo0 = _mulhilo(c0, _M0)
        hi1, lo1 = _mulhilo(c2, _M1)
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return c0, c1, c2, c3


def random_words(n: int, seed: int, stream: int, device="cpu", offset: int = 0) -> torch.Tensor:
    """n uint32 words (as int64) of the stream (seed, stream), starting at word `offset`.

    Word w of a stream is lane (w % 4) of the Philox block whose counter is
    (w // 4, 0, 0, 0) under the key (seed, stream).
    """
    if n <= 0:
        return torch.zeros(0, dtype=torch.int64, device=device)
    first = offset // 4
    last = (offset + n - 1) // 4
    ctr = torch.arange(first, last + 1, dtype=torch.int64, device=device)
    c0 = ctr & _MASK32
    c1 = ctr >> 32
    zero = torch.zeros_like(c0)
    out = philox4x32_10(c0, c1, zero, zero, seed & _MASK32, stream & _MASK32)
    words = torch.stack(out, dim=1).reshape(-1)
    start = offset - first * 4
    return words[start:start + n]


_CHUNK = 1 << 24


def uniform_f32(shape, seed: int, stream: int, device="cpu") -> torch.Tensor:
    """float32 uniforms in [0, 1): the top 24 bits of each word times 2^-24 (exact)."""
    n = math.prod(shape)
    out = torch.empty(n, dtype=torch.float32, device=device)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        w = random_words(e - s, seed, stream, device, offset=s)
        out[s:e] = (w >> 8).to(torch.float32) * (2.0 ** -24)
    return out.reshape(shape)


def uniform_open_f64(shape, seed: int, stream: int, device="cpu", offset_words: int = 0) -> torch.Tensor:
    """float64 uniforms in (0, 1]: (top 24 bits + 1) * 2^-24, from consecutive words."""
    n = math.prod(shape)
    w = random_words(n, seed, stream, device, offset=offset_words)
    return (((w >> 8) + 1).to(torch.float64) * (2.0 ** -24)).reshape(shape)


def normal_f32(shape, seed: int, stream: int, device="cpu") -> torch.Tensor:
    """float32 standard normals by Box-Muller in float64: sqrt(-2 ln u1) cos(2 pi u2).

    Normal k uses words 2k and 2k+1 of the stream.
    """
    n = math.prod(shape)
    out = torch.empty(n, dtype=torch.float32, device=device)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        w = random_words(2 * (e - s), seed, stream, device, offset=2 * s)
        u1 = ((w[0::2] >> 8) + 1).to(torch.float64) * (2.0 ** -24)
        u2 = (w[1::2] >> 8).to(torch.float64) * (2.0 ** -24)
        out[s:e] = (torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)).to(torch.float32)
    return out.reshape(shape)


def gumbel_f32(shape, seed: int, stream: int, device="cpu") -> torch.Tensor:
    """float32 standard Gumbel noise -ln(-ln u), u in (0, 1) (computed in float64)."""
    n = math.prod(shape)
    out = torch.empty(n, dtype=torch.float32, device=device)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        w = random_words(e - s, seed, stream, device, offset=s)
        # (top 24 bits + 0.5) * 2^-24 lies strictly inside (0, 1)
        u = ((w >> 8).to(torch.float64) + 0.5) * (2.0 ** -24)
        out[s:e] = (-torch.log(-torch.log(u))).to(torch.float32)
    return out.reshape(shape)
