"""Plain CPU oracle of the fused-dequantization quantized GEMM (dense and MoE).

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module; the library never calls it, and it
shares no code with the CUDA path.

What it computes is the definition the Humming announcement gives for its
kernels: weights are decoded from their numeric format, scales and zero points
are applied ("Shared CUDA components across formats and architectures",
numeric-processing item), then a plain matrix product is taken and the output
stage applies scales and bias (same section, task-mapping item).  Repacking
preserves the quantization semantics ("A unified quantization representation").
The pages print no bit layouts, so each decoder follows the public definition of
its format, named at the function:

    Wdeq[n, k] = decode(codes, scales, zeros, global)  (exact, float64)
    Adeq[m, k] = decode(activation)                     (exact, float64)
    Y[m, n]    = sum_k Adeq[m, k] * Wdeq[n, k]          (float64 matmul)
    MoE row t*k+j = topk_w[t, j] * (Adeq[t] . Wdeq[ids[t, j]]),  + bias for dense

Conventions (the pages are silent on them): codes are two per byte with the low
nibble holding the even k; W is [N, K] ("out, in"); scale groups run along K.
"""
import numpy as np

# ---------------------------------------------------------------- scalar formats


def decode_int(code, bits, signed):
    """Integer code of `bits` bits -> value; signed codes are two's complement."""
    c = np.asarray(code).astype(np.int64) & ((1 << bits) - 1)
    if signed:
        c = np.where(c >= (1 << (bits - 1)), c - (1 << bits), c)
    return c.astype(np.float64)


def decode_e2m1(code):
    """OCP Microscaling v1.0, FP4 E2M1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit.

    Exponent field 0 is subnormal: 2**(1-1) * (m / 2).  No infinities or NaN.
    """
    c = np.asarray(code).astype(np.int64) & 0xF
    s = np.where(c & 0x8, -1.0, 1.0)
    e = (c >> 1) & 0x3
    m = (c & 0x1).astype(np.float64)
    mag = np.where(e == 0, m * 0.5, np.ldexp(1.0 + m * 0.5, (e - 1).astype(np.int32)))
    return s * mag


def decode_e4m3(byte):
    """OCP OFP8 E4M3 ("fn"): bias 7, S.1111.111 is NaN, no infinities, max 448.

    Exponent field 0 is subnormal: 2**-6 * (m / 8).
    """
    b = np.asarray(byte).astype(np.int64) & 0xFF
    s = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int32)))
    mag = np.where((e == 0xF) & ((b & 0x7) == 0x7), np.nan, mag)
    return s * mag


def decode_ue4m3(byte):
    """Unsigned use of E4M3 as a block scale: the sign bit must be 0 (else NaN)."""
    b = np.asarray(byte).astype(np.int64) & 0xFF
    return np.where(b & 0x80, np.nan, decode_e4m3(b))


def decode_e8m0(byte):
    """OCP Microscaling v1.0 E8M0 scale: 2**(e - 127); 0xFF is NaN."""
    b = np.asarray(byte).astype(np.int64) & 0xFF
    return np.where(b == 0xFF, np.nan, np.ldexp(1.0, (b - 127).astype(np.int32)))


def decode_bf16(bits):
    """bfloat16 bit pattern (uint16) -> value: the upper half of an IEEE binary32."""
    u = np.asarray(bits).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def unpack_nibbles(packed):
    """[..., K/2] bytes -> [..., K] 4-bit codes, low nibble = even k."""
    p = np.asarray(packed).astype(np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


# ---------------------------------------------------------------- tensor formats

WEIGHT_FORMATS = ("int4_sym", "uint4_zp", "nvfp4", "mxfp4")
ACT_FORMATS = ("bf16", "e4m3_tok", "nvfp4")
BLOCK = {"nvfp4": 16, "mxfp4": 32}


def dequant_weights(wfmt, codes, scales, zeros=None, gscale=None, group=128):
    """Decode one weight tensor [N, K] (or [E, N, K]) to float64.

    int4_sym : value = q * s, q two's complement in [-7, 7], s bf16 per (n, group)
    uint4_zp : value = (q - z) * s, q and z in [0, 15], s bf16 per (n, group)
    nvfp4    : value = e2m1(q) * ue4m3(sb) * g, sb per (n, 16 along K), g fp32 per tensor
    mxfp4    : value = e2m1(q) * e8m0(sb), sb per (n, 32 along K)
    """
    q = unpack_nibbles(codes)
    k = q.shape[-1]
    if wfmt == "int4_sym":
        s = decode_bf16(scales)
        return decode_int(q, 4, True) * np.repeat(s, group, axis=-1)[..., :k]
    if wfmt == "uint4_zp":
        s = decode_bf16(scales)
        z = np.asarray(zeros).astype(np.float64)
        zq = np.repeat(z, group, axis=-1)[..., :k]
        return (decode_int(q, 4, False) - zq) * np.repeat(s, group, axis=-1)[..., :k]
    if wfmt == "nvfp4":
        sb = np.repeat(decode_ue4m3(scales), BLOCK[wfmt], axis=-1)[..., :k]
        g = np.asarray(gscale, dtype=np.float64).reshape(-1)
        g = g.reshape((-1,) + (1,) * (q.ndim - 1)) if q.ndim == 3 else g[0]
        return decode_e2m1(q) * sb * g
    if wfmt == "mxfp4":
        sb = np.repeat(decode_e8m0(scales), BLOCK[wfmt], axis=-1)[..., :k]
        return decode_e2m1(q) * sb
    raise ValueError(wfmt)


def dequant_acts(afmt, data, scale=None, gscale=None):
    """Decode activations [M, K] to float64.

    bf16     : the bf16 values
    e4m3_tok : e4m3(a) * s_t, one fp32 scale per row (token)
    nvfp4    : e2m1(q) * ue4m3(sb) * g, sb per (row, 16 along K), g fp32 per tensor
    """
    if afmt == "bf16":
        return decode_bf16(data)
    if afmt == "e4m3_tok":
        s = np.asarray(scale, dtype=np.float64).reshape(-1, 1)
        return decode_e4m3(data) * s
    if afmt == "nvfp4":
        q = unpack_nibbles(data)
        sb = np.repeat(decode_ue4m3(scale), 16, axis=-1)[..., : q.shape[-1]]
        g = float(np.asarray(gscale, dtype=np.float64).reshape(-1)[0])
        return decode_e2m1(q) * sb * g
    raise ValueError(afmt)


# ---------------------------------------------------------------- the products


def gemm(adeq, wdeq, bias=None):
    """Dense output Y[M, N] = Adeq . Wdeq^T (+ bias[n]), float64."""
    y = np.asarray(adeq, dtype=np.float64) @ np.asarray(wdeq, dtype=np.float64).T
    if bias is not None:
        y = y + decode_bf16(bias).reshape(1, -1)
    return y


def moe_gemm(adeq, wdeq_of_expert, n_out, topk_ids, topk_weights=None, rows=None):
    """MoE output rows: row t*k + j = topk_w[t, j] * (Adeq[t] . Wdeq[ids[t, j]]^T), float64.

    `wdeq_of_expert(e)` returns expert e's decoded [N, K] weights, or None for an
    id that names no expert (such rows are undefined and come back as NaN).
    `rows` (flat indices t*k + j) restricts the rows computed; None computes all.
    """
    ids = np.asarray(topk_ids)
    T, k = ids.shape
    flat = np.arange(T * k) if rows is None else np.asarray(rows)
    y = np.full((len(flat), n_out), np.nan)
    cache = {}
    for i, r in enumerate(flat):
        t, j = divmod(int(r), k)
        e = int(ids[t, j])
        if e not in cache:
            cache[e] = wdeq_of_expert(e)
        w = cache[e]
        if w is None:
            continue
        v = np.asarray(adeq[t], dtype=np.float64) @ np.asarray(w, dtype=np.float64).T
        if topk_weights is not None:
            v = v * float(np.asarray(topk_weights)[t, j])
        y[i] = v
    return y
