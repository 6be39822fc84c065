"""Counter-based random numbers for the synthetic workloads.

Philox-4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
as 1, 2, 3", SC'11, section 3): a 10-round bijection of a 128-bit counter under
a 64-bit key.  Written with int64 torch tensors so that the same integers come
out on the CPU and on a CUDA device.  Normals use the Box-Muller transform in
float64 and are rounded once to float32.

This module holds no arithmetic of the quantized GEMM; it only draws numbers.
"""
import math

import torch

_M0 = 0xD2511F53
_M1 = 0xCD9E8D57
_W0 = 0x9E3779B9
_W1 = 0xBB67AE85
_MASK = 0xFFFFFFFF


def _mulhilo(a, m):
    """(hi, lo) 32-bit halves of a * m for int64 tensors a < 2**32, int m < 2**32.

    The product is split on the 16-bit halves of m so no intermediate leaves int64.
    """
    p_lo = a * (m & 0xFFFF)
    p_hi = a * (m >> 16)
    lo = (p_lo + ((p_hi & 0xFFFF) << 16)) & _MASK
    hi = (p_hi + (p_lo >> 16)) >> 16
    return hi, lo


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Apply Philox-4x32-10 to counters (c0..c3) under key (k0, k1).

    All arguments are int64 tensors (or ints) holding values in [0, 2**32).
    Returns the four output words as int64 tensors.
    """
    for r in range(10):
        if r:
            k0 = (k0 + _W0) & _MASK
            k1 = (k1 + _W1) & _MASK
        hi0, lo0 = _mulhilo(c0, _M0)
        hi1, lo1 = _mulhilo(c2, _M1)
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return c0, c1, c2, c3


def random_u32(seed, stream, n_calls, offset=0, device="cpu"):
    """[n_calls, 4] int64 tensor of uint32 words.

    Call i uses counter (offset + i) split over words 0 and 1, the stream id in
    word 2 and 0 in word 3; the key is (low, high) 32 bits of the seed.
    """
    idx = torch.arange(n_calls, dtype=torch.int64, device=device) + int(offset)
    c0 = idx & _MASK
    c1 = idx >> 32
    c2 = torch.full_like(idx, int(stream) & _MASK)
    c3 = torch.zeros_like(idx)
    k0 = int(seed) & _MASK
    k1 = (int(seed) >> 32) & _MASK
    out = philox4x32_10(c0, c1, c2, c3, k0, k1)
    return torch.stack(out, dim=1)


def uniform(seed, stream, n, offset=0, device="cpu"):
    """n float64 uniforms in (0, 1): (u32 + 0.5) / 2**32, four per Philox call."""
    calls = (n + 3) // 4
    u = random_u32(seed, stream, calls, offset, device).reshape(-1)[:n]
    return (u.to(torch.float64) + 0.5) * (1.0 / 4294967296.0)


def normal(seed, stream, n, offset=0, device="cpu"):
    """n float32 standard normals; Box-Muller on word pairs (0,1) and (2,3) of each call.

    `offset` counts Philox calls, so element i of a tensor is always drawn by call
    offset + i // 4 whatever chunking the caller uses (n and offsets multiples of 4).
    """
    calls = (n + 3) // 4
    u = (random_u32(seed, stream, calls, offset, device).to(torch.float64) + 0.5) * (1.0 / 4294967296.0)
    r01 = torch.sqrt(-2.0 * torch.log(u[:, 0]))
    t01 = (2.0 * math.pi) * u[:, 1]
    r23 = torch.sqrt(-2.0 * torch.log(u[:, 2]))
    t23 = (2.0 * math.pi) * u[:, 3]
    z = torch.stack([r01 * torch.cos(t01), r01 * torch.sin(t01),
                     r23 * torch.cos(t23), r23 * torch.sin(t23)], dim=1)
    return z.reshape(-1)[:n].to(torch.float32)
