"""Quantization recipes that turn the synthetic fp32 draws into the GEMM's inputs.

These are the input recipes of the benchmark workloads (they encode; nothing
here decodes or multiplies).  Each rule is the plainest reading of the format's
public definition:

* grouped INT4: scale = absmax / 7 rounded to bf16, codes rint(w / scale)
  clamped to [-7, 7] (the value set of a zero-exponent e0m3 float);
* grouped UINT4 with zero point: scale = (max - min) / 15 in bf16, zero =
  clamp(rint(-min / scale), 0, 15), code = clamp(rint(w / scale) + zero, 0, 15);
* NVFP4: fp32 tensor scale g = amax / (6 * 448), e4m3 block-16 scale
  e4m3(amax_b / (6 g)) saturated at 448, e2m1 codes of x / (sb * g);
* MXFP4 (OCP Microscaling v1.0 section 6.3), weights and W4A4 activations:
  e8m0 block-32 scale 2**(floor(log2 amax_b) - 2), e2m1 codes of x / scale,
  saturating;
* FP8 per token: s_t = absmax_t / 448, e4m3(a / s_t) saturated;
* grouped INT8 (the e0m7 value set): scale = absmax / 127 in bf16, codes
  rint(w / scale) clamped to [-127, 127], one byte each;
* grouped UINT2 with zero point: scale = (max - min) / 3 in bf16, zero =
  clamp(rint(-min / scale), 0, 3), code = clamp(rint(w / scale) + zero, 0, 3),
  four codes per byte from the lowest bits up;
* grouped UINT1 / UINT3 with zero point (GPTQ style, bits b): the UINT2 rule
  with 2**b - 1 levels, codes as a little-endian bit string;
* MXINT4 (e8m0 block-32 scale): 2**(floor(log2 amax_b) - 2) (4 = 2**2 is the
  largest power of two of the integer range, as for MXFP4), codes rint(w /
  scale) clamped to [-7, 7];
* grouped FP8 E4M3 weights: scale = absmax / 448 in bf16, e4m3(w / scale);
* MXFP8 (OCP Microscaling v1.0 section 6.3): e8m0 block-32 scale
  2**(floor(log2 amax_b) - 8) (8 = E4M3's largest exponent), e4m3(x / scale).

Rounding is to nearest, ties to even, everywhere.  All functions take torch
tensors on any device and return tensors on the same device.  4-bit codes are
packed two per byte, low nibble = even k.
"""
import torch

E4M3_MAX = 448.0
E2M1_MAX = 6.0


def pack_nibbles(codes):
    """[..., K] uint8 codes in 0..15 -> [..., K/2] bytes, low nibble = even k."""
    c = codes.to(torch.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).contiguous()


def _rint(x):
    return torch.round(x)  # round half to even


def quant_int4_sym(w, group):
    """w fp32 [..., N, K] -> (packed codes uint8 [..., N, K/2], scales bf16 [..., N, K/group])."""
    *lead, n, k = w.shape
    wg = w.reshape(*lead, n, k // group, group)
    s = (wg.abs().amax(dim=-1) / 7.0).to(torch.bfloat16)
    sf = s.float().unsqueeze(-1)
    q = torch.where(sf > 0, _rint(wg / torch.where(sf > 0, sf, torch.ones_like(sf))), torch.zeros_like(wg))
    q = q.clamp(-7, 7).to(torch.int16)
    codes = (q & 0xF).to(torch.uint8).reshape(*lead, n, k)
    return pack_nibbles(codes), s.contiguous()


def quant_uint4_zp(w, group):
    """w fp32 [..., N, K] -> (packed codes, scales bf16 [..., N, K/g], zeros uint8 [..., N, K/g])."""
    *lead, n, k = w.shape
    wg = w.reshape(*lead, n, k // group, group)
    lo = wg.amin(dim=-1)
    hi = wg.amax(dim=-1)
    s = ((hi - lo) / 15.0).to(torch.bfloat16)
    sf = s.float()
    safe = torch.where(sf > 0, sf, torch.ones_like(sf))
    z = torch.where(sf > 0, _rint(-lo / safe), torch.zeros_like(sf)).clamp(0, 15)
    q = torch.where(sf.unsqueeze(-1) > 0, _rint(wg / safe.unsqueeze(-1)) + z.unsqueeze(-1), torch.zeros_like(wg))
    q = q.clamp(0, 15).to(torch.uint8).reshape(*lead, n, k)
    return pack_nibbles(q), s.contiguous(), z.to(torch.uint8).contiguous()


def e2m1_encode(v):
    """fp32 -> e2m1 code (uint8, 0..15): nearest on {0,.5,1,1.5,2,3,4,6}, ties to even, saturating.

    Zero magnitudes get code 0 (positive zero).
    """
    a = v.abs()
    # magnitude code m: thresholds between neighbours, tie goes to the even mantissa
    m = torch.zeros_like(a, dtype=torch.uint8)
    m = torch.where(a > 0.25, torch.full_like(m, 1), m)
    m = torch.where(a >= 0.75, torch.full_like(m, 2), m)
    m = torch.where(a > 1.25, torch.full_like(m, 3), m)
    m = torch.where(a >= 1.75, torch.full_like(m, 4), m)
    m = torch.where(a > 2.5, torch.full_like(m, 5), m)
    m = torch.where(a >= 3.5, torch.full_like(m, 6), m)
    m = torch.where(a > 5.0, torch.full_like(m, 7), m)
    sign = ((v < 0) & (m > 0)).to(torch.uint8) << 3
    return m | sign


def e4m3_encode(v):
    """fp32 -> e4m3fn byte, RNE, saturating at +-448."""
    return v.clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)


def _e4m3_value(b):
    return b.view(torch.float8_e4m3fn).to(torch.float32)


def quant_nvfp4(x, block=16, global_amax=None):
    """x fp32 [..., R, K] -> (packed e2m1 [..., R, K/2], ue4m3 scales [..., R, K/16], g fp32 scalar tensor).

    g is the per-tensor decode multiplier amax / (6 * 448); value = e2m1 * sb * g.
    """
    *lead, r, k = x.shape
    amax = x.abs().amax() if global_amax is None else global_amax
    g = (amax.to(torch.float32) / (E2M1_MAX * E4M3_MAX)).reshape(())
    xb = x.reshape(*lead, r, k // block, block)
    amax_b = xb.abs().amax(dim=-1)
    safe_g = torch.where(g > 0, g, torch.ones_like(g))
    sb = e4m3_encode(amax_b / (E2M1_MAX * safe_g))
    sbf = _e4m3_value(sb) * safe_g
    den = torch.where(sbf > 0, sbf, torch.ones_like(sbf)).unsqueeze(-1)
    q = e2m1_encode(xb / den)
    q = torch.where(sbf.unsqueeze(-1) > 0, q, torch.zeros_like(q)).reshape(*lead, r, k)
    return pack_nibbles(q), sb.contiguous(), g


def quant_mxfp4(w, block=32):
    """w fp32 [..., N, K] -> (packed e2m1 [..., N, K/2], e8m0 scales uint8 [..., N, K/32])."""
    *lead, n, k = w.shape
    wb = w.reshape(*lead, n, k // block, block)
    amax = wb.abs().amax(dim=-1)
    _, ex = torch.frexp(amax)  # amax = m * 2**ex, m in [0.5, 1): floor(log2 amax) = ex - 1
    e = (ex.to(torch.int32) - 1 - 2 + 127).clamp(0, 254)
    e = torch.where(amax > 0, e, torch.full_like(e, 127))
    scale = torch.ldexp(torch.ones_like(amax), (e - 127).to(torch.float32))
    q = e2m1_encode(wb / scale.unsqueeze(-1))
    q = torch.where(amax.unsqueeze(-1) > 0, q, torch.zeros_like(q)).reshape(*lead, n, k)
    return pack_nibbles(q), e.to(torch.uint8).contiguous()


def quant_e4m3_per_token(a):
    """a fp32 [T, K] -> (e4m3 bytes [T, K], per-token fp32 scale [T] = absmax / 448)."""
    s = a.abs().amax(dim=-1) / E4M3_MAX
    safe = torch.where(s > 0, s, torch.ones_like(s))
    q = e4m3_encode(a / safe.unsqueeze(-1))
    q = torch.where(s.unsqueeze(-1) > 0, q, torch.zeros_like(q))
    return q.contiguous(), s.to(torch.float32).contiguous()


def pack_crumbs(codes):
    """[..., K] uint8 codes in 0..3 -> [..., K/4] bytes; bits 2i, 2i + 1 of byte b hold k = 4b + i."""
    c = codes.to(torch.uint8)
    return (c[..., 0::4] | (c[..., 1::4] << 2) | (c[..., 2::4] << 4) | (c[..., 3::4] << 6)).contiguous()


def pack_bits(codes, bits):
    """[..., K] uint8 codes of `bits` bits -> [..., K * bits / 8] bytes: a little-endian bit string (bit j of code k
    is bit (k * bits + j) % 8 of byte (k * bits + j) // 8)."""
    c = codes.to(torch.int64)
    *lead, k = c.shape
    bit = ((c.unsqueeze(-1) >> torch.arange(bits, device=c.device)) & 1).reshape(*lead, k * bits // 8, 8)
    return (bit << torch.arange(8, device=c.device)).sum(dim=-1).to(torch.uint8).contiguous()


def quant_uint_zp(w, group, bits):
    """w fp32 [..., N, K] -> (bit-string codes [..., N, K*bits/8], scales bf16 [..., N, K/g], zeros uint8
    [..., N, K/g]); GPTQ-style unsigned codes with an integer zero point, 2**bits - 1 levels."""
    lv = float((1 << bits) - 1)
    *lead, n, k = w.shape
    wg = w.reshape(*lead, n, k // group, group)
    lo = wg.amin(dim=-1)
    hi = wg.amax(dim=-1)
    s = ((hi - lo) / lv).to(torch.bfloat16)
    sf = s.float()
    safe = torch.where(sf > 0, sf, torch.ones_like(sf))
    z = torch.where(sf > 0, _rint(-lo / safe), torch.zeros_like(sf)).clamp(0, lv)
    q = torch.where(sf.unsqueeze(-1) > 0, _rint(wg / safe.unsqueeze(-1)) + z.unsqueeze(-1), torch.zeros_like(wg))
    q = q.clamp(0, lv).to(torch.uint8).reshape(*lead, n, k)
    return pack_bits(q, bits), s.contiguous(), z.to(torch.uint8).contiguous()


def quant_int8_sym(w, group):
    """w fp32 [..., N, K] -> (int8 codes as bytes [..., N, K], scales bf16 [..., N, K/group])."""
    *lead, n, k = w.shape
    wg = w.reshape(*lead, n, k // group, group)
    s = (wg.abs().amax(dim=-1) / 127.0).to(torch.bfloat16)
    sf = s.float().unsqueeze(-1)
    q = torch.where(sf > 0, _rint(wg / torch.where(sf > 0, sf, torch.ones_like(sf))), torch.zeros_like(wg))
    q = q.clamp(-127, 127).to(torch.int16)
    return (q & 0xFF).to(torch.uint8).reshape(*lead, n, k).contiguous(), s.contiguous()


def quant_uint2_zp(w, group):
    """w fp32 [..., N, K] -> (packed 2-bit codes [..., N, K/4], scales bf16 [..., N, K/g], zeros uint8 [..., N, K/g])."""
    *lead, n, k = w.shape
    wg = w.reshape(*lead, n, k // group, group)
    lo = wg.amin(dim=-1)
    hi = wg.amax(dim=-1)
    s = ((hi - lo) / 3.0).to(torch.bfloat16)
    sf = s.float()
    safe = torch.where(sf > 0, sf, torch.ones_like(sf))
    z = torch.where(sf > 0, _rint(-lo / safe), torch.zeros_like(sf)).clamp(0, 3)
    q = torch.where(sf.unsqueeze(-1) > 0, _rint(wg / safe.unsqueeze(-1)) + z.unsqueeze(-1), torch.zeros_like(wg))
    q = q.clamp(0, 3).to(torch.uint8).reshape(*lead, n, k)
    return pack_crumbs(q), s.contiguous(), z.to(torch.uint8).contiguous()


def _e8m0_block_scale(amax, emax):
    """e8m0 byte and value of 2**(floor(log2 amax) - emax) per block (127, i.e. 1, for an all-zero block)."""
    _, ex = torch.frexp(amax)  # amax = m * 2**ex, m in [0.5, 1): floor(log2 amax) = ex - 1
    e = (ex.to(torch.int32) - 1 - emax + 127).clamp(0, 254)
    e = torch.where(amax > 0, e, torch.full_like(e, 127))
    return e, torch.ldexp(torch.ones_like(amax), (e - 127).to(torch.float32))


def quant_mxint4(w, block=32):
    """w fp32 [..., N, K] -> (packed int4 codes [..., N, K/2], e8m0 scales uint8 [..., N, K/32])."""
    *lead, n, k = w.shape
    wb = w.reshape(*lead, n, k // block, block)
    e, scale = _e8m0_block_scale(wb.abs().amax(dim=-1), 2)
    q = _rint(wb / scale.unsqueeze(-1)).clamp(-7, 7).to(torch.int16)
    codes = (q & 0xF).to(torch.uint8).reshape(*lead, n, k)
    return pack_nibbles(codes), e.to(torch.uint8).contiguous()


def quant_e4m3_grouped(w, group):
    """w fp32 [..., N, K] -> (e4m3 bytes [..., N, K], scales bf16 [..., N, K/group] = absmax / 448)."""
    *lead, n, k = w.shape
    wg = w.reshape(*lead, n, k // group, group)
    s = (wg.abs().amax(dim=-1) / E4M3_MAX).to(torch.bfloat16)
    sf = s.float().unsqueeze(-1)
    q = e4m3_encode(wg / torch.where(sf > 0, sf, torch.ones_like(sf)))
    q = torch.where(sf > 0, q, torch.zeros_like(q))
    return q.reshape(*lead, n, k).contiguous(), s.contiguous()


def quant_mxfp8(x, block=32):
    """x fp32 [..., R, K] -> (e4m3 bytes [..., R, K], e8m0 scales uint8 [..., R, K/32])."""
    *lead, r, k = x.shape
    xb = x.reshape(*lead, r, k // block, block)
    e, scale = _e8m0_block_scale(xb.abs().amax(dim=-1), 8)
    q = e4m3_encode(xb / scale.unsqueeze(-1)).reshape(*lead, r, k)
    return q.contiguous(), e.to(torch.uint8).contiguous()
