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

It also quantizes bf16 activations to the FP8 (per-token scale) and NVFP4
operands of the W4A8 and W4A4 paths ("Selecting activation types"; section
"activation quantization" at the end), taking every decision in IEEE binary32.

Conventions (the pages are silent on them): 4-bit codes are two per byte with
the low nibble holding the even k, 2-bit codes four per byte from the lowest
bits up, 1- and 3-bit codes as a little-endian bit string, 8-bit codes one per
byte; W is [N, K] ("out, in"); scale groups run along K.
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


def unpack_crumbs(packed):
    """[..., K/4] bytes -> [..., K] 2-bit codes; bits 2i and 2i + 1 of a byte hold its k = 4b + i."""
    p = np.asarray(packed).astype(np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 4,), dtype=np.uint8)
    for i in range(4):
        out[..., i::4] = (p >> (2 * i)) & 0x3
    return out


def unpack_bits(packed, bits):
    """[..., K*bits/8] bytes -> [..., K] codes of `bits` bits from a little-endian bit string: code k occupies bits
    k*bits .. k*bits + bits - 1 of the row, bit j of the string being bit j % 8 of byte j // 8."""
    p = np.asarray(packed).astype(np.uint8)
    stream = np.unpackbits(p, axis=-1, bitorder="little")
    k = stream.shape[-1] // bits
    stream = stream[..., : k * bits].reshape(p.shape[:-1] + (k, bits)).astype(np.int64)
    weights = np.int64(1) << np.arange(bits, dtype=np.int64)
    return (stream * weights).sum(axis=-1).astype(np.uint8)


# ---------------------------------------------------------------- tensor formats

WEIGHT_FORMATS = ("int4_sym", "uint4_zp", "nvfp4", "mxfp4", "int8_sym", "uint2_zp", "mxint4", "e4m3", "uint1_zp",
                  "uint3_zp")
ACT_FORMATS = ("bf16", "e4m3_tok", "nvfp4", "mxfp8", "mxfp4")
BLOCK = {"nvfp4": 16, "mxfp4": 32, "mxint4": 32, "mxfp8": 32}


def dequant_weights(wfmt, codes, scales, zeros=None, gscale=None, group=128):
    """Decode one weight tensor [N, K] (or [E, N, K]) to float64.

    int4_sym : value = q * s, q two's complement in [-7, 7], s bf16 per (n, group)
    uint4_zp : value = (q - z) * s, q and z in [0, 15], s bf16 per (n, group)
    nvfp4    : value = e2m1(q) * ue4m3(sb) * g, sb per (n, 16 along K), g fp32 per tensor
    mxfp4    : value = e2m1(q) * e8m0(sb), sb per (n, 32 along K)
    int8_sym : value = q * s, q one byte, two's complement in [-127, 127] (the value set of the zero-exponent
               float e0m7, "Results: quantization support"), s bf16 per (n, group)
    uint2_zp : value = (q - z) * s, q and z in [0, 3], q four per byte (see unpack_crumbs), s bf16 per (n, group)
    mxint4   : value = q * e8m0(sb), q two's complement nibbles in [-7, 7], sb per (n, 32 along K)
    e4m3     : value = e4m3(q) * s, q one OCP OFP8 E4M3 byte, s bf16 per (n, group)
    uint1_zp : value = (q - z) * s, q and z in {0, 1}, q eight per byte (see unpack_bits), s bf16 per (n, group)
    uint3_zp : value = (q - z) * s, q and z in [0, 7], q a 3-bit little-endian bit string (see unpack_bits), s bf16
               per (n, group); the INT1 / INT3 widths of "Results: kernel microbenchmarks" read as the GPTQ-style
               unsigned codes with integer zero points that the GPTQ INT3 checkpoints of "vLLM integration" hold
    """
    if wfmt in ("uint1_zp", "uint3_zp"):
        bits = 1 if wfmt == "uint1_zp" else 3
        q = unpack_bits(codes, bits)
        k = q.shape[-1]
        s = np.repeat(decode_bf16(scales), group, axis=-1)[..., :k]
        zq = np.repeat(np.asarray(zeros).astype(np.float64), group, axis=-1)[..., :k]
        return (decode_int(q, bits, False) - zq) * s
    if wfmt in ("int8_sym", "e4m3"):
        q = np.asarray(codes).astype(np.uint8)
        k = q.shape[-1]
        s = np.repeat(decode_bf16(scales), group, axis=-1)[..., :k]
        return (decode_int(q, 8, True) if wfmt == "int8_sym" else decode_e4m3(q)) * s
    if wfmt == "uint2_zp":
        q = unpack_crumbs(codes)
        k = q.shape[-1]
        s = np.repeat(decode_bf16(scales), group, axis=-1)[..., :k]
        zq = np.repeat(np.asarray(zeros).astype(np.float64), group, axis=-1)[..., :k]
        return (decode_int(q, 2, False) - zq) * s
    q = unpack_nibbles(codes)
    k = q.shape[-1]
    if wfmt == "mxint4":
        sb = np.repeat(decode_e8m0(scales), BLOCK[wfmt], axis=-1)[..., :k]
        return decode_int(q, 4, True) * sb
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
    mxfp8    : e4m3(a) * e8m0(sb), sb per (row, 32 along K) (OCP Microscaling v1.0 MXFP8 E4M3)
    mxfp4    : e2m1(q) * e8m0(sb), q two per byte (low nibble = even k), sb per (row, 32 along K) (OCP
               Microscaling v1.0 MXFP4, the W4A4 operand of "W8A8 / W4A8 / W4A4")
    """
    if afmt == "bf16":
        return decode_bf16(data)
    if afmt == "mxfp4":
        q = unpack_nibbles(data)
        sb = np.repeat(decode_e8m0(scale), BLOCK[afmt], axis=-1)[..., : q.shape[-1]]
        return decode_e2m1(q) * sb
    if afmt == "mxfp8":
        q = np.asarray(data).astype(np.uint8)
        sb = np.repeat(decode_e8m0(scale), BLOCK[afmt], axis=-1)[..., : q.shape[-1]]
        return decode_e4m3(q) * sb
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


# ---------------------------------------------------------------- activation quantization
#
# The deployment picks the activation type of a quantized layer ("Selecting activation types"): token-wise FP8 for
# the W4A8 path ("End-to-end inference performance") and NVFP4 for W4A4 ("W8A8 / W4A8 / W4A4").  The pages give no
# recipe for the scales, so these follow the format definitions with the plainest scale choice: the largest magnitude
# of the scaled unit maps to the format's largest value.  Every step is one IEEE binary32 operation (float32 numpy),
# because the codes are integers decided by those float results: the device quantizer takes the same decisions in
# the same precision.

E4M3_MAX = np.float32(448.0)
E2M1_MAX = np.float32(6.0)


def _nearest_code(mag, values):
    """Index of the nearest entry of the ascending table `values` to each magnitude (float64 compare of exact float32
    inputs), ties to the even index: round to nearest even on the format's grid.  Magnitudes beyond the last entry
    saturate to it."""
    mag = np.asarray(mag, dtype=np.float64)
    hi = np.clip(np.searchsorted(values, mag, side="left"), 1, len(values) - 1)
    lo = hi - 1
    d_lo = mag - values[lo]
    d_hi = values[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    idx = np.where(pick_hi, hi, lo)
    return np.where(mag >= values[-1], len(values) - 1, idx)


_E4M3_POS = decode_e4m3(np.arange(0x7F))  # codes 0x00 .. 0x7E: 0 .. 448 ascending (0x7F is NaN)
_E2M1_POS = decode_e2m1(np.arange(8))  # 0, 0.5, 1, 1.5, 2, 3, 4, 6


def encode_e4m3(v):
    """float32 -> OCP OFP8 E4M3 byte: nearest value, ties to even, saturating at +-448.  The sign is kept, also on
    a zero result (IEEE conversion: -0 is 0x80)."""
    v = np.asarray(v, dtype=np.float32)
    m = _nearest_code(np.abs(v), _E4M3_POS).astype(np.uint8)
    return np.where(np.signbit(v), m | np.uint8(0x80), m).astype(np.uint8)


def encode_e2m1(v):
    """float32 -> OCP MX FP4 E2M1 code: nearest value, ties to even, saturating at +-6.  A zero result is +0 (code 0)
    whatever the sign, as the weight and activation recipes of the workloads encode it."""
    v = np.asarray(v, dtype=np.float32)
    m = _nearest_code(np.abs(v), _E2M1_POS).astype(np.uint8)
    return np.where(np.signbit(v) & (m > 0), m | np.uint8(0x8), m).astype(np.uint8)


def _bf16_to_f32(bits):
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32)


def quantize_act_e4m3_per_token(x_bits):
    """bf16 [M, K] (bit patterns) -> (e4m3 bytes [M, K], fp32 scale [M]).

    s_t = absmax_t / 448 (float32 division); code = e4m3(x / s_t); a row of zeros gets s_t = 0 and zero codes.
    Decoding gives x ~ code * s_t, the per-token activation the W4A8 GEMM consumes.
    """
    x = _bf16_to_f32(x_bits)
    amax = np.abs(x).max(axis=1) if x.shape[1] else np.zeros(x.shape[0], np.float32)
    s = (amax / E4M3_MAX).astype(np.float32)
    safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    q = encode_e4m3((x / safe[:, None]).astype(np.float32))
    q = np.where((s > 0)[:, None], q, np.uint8(0)).astype(np.uint8)
    return q, s


def quantize_act_nvfp4(x_bits, global_amax=None):
    """bf16 [M, K] (bit patterns), K a multiple of 16 -> (packed e2m1 [M, K/2], ue4m3 scales [M, K/16], g fp32).

    NVIDIA's NVFP4: e2m1 values, an e4m3 scale per 16 consecutive elements of a row and one fp32 tensor scale.
    g = amax / (6 * 448) with amax the tensor's largest magnitude (or a calibrated `global_amax`); per block
    sb = e4m3(amax_b / (6 * g)) (saturating), d = value(sb) * g, code = e2m1(x / d); d = 0 gives zero codes.
    Decoding gives x ~ e2m1 * value(sb) * g.
    """
    x = _bf16_to_f32(x_bits)
    M, K = x.shape
    if global_amax is None:
        amax = np.float32(np.abs(x).max()) if x.size else np.float32(0.0)
    else:
        amax = np.float32(global_amax)
    g = np.float32(amax / np.float32(E2M1_MAX * E4M3_MAX))
    xb = x.reshape(M, K // 16, 16)
    amax_b = np.abs(xb).max(axis=2).astype(np.float32)
    if g > 0:
        six_g = np.float32(E2M1_MAX * g)
        sb = encode_e4m3((amax_b / six_g).astype(np.float32))
        d = (decode_e4m3(sb).astype(np.float32) * g).astype(np.float32)
    else:
        sb = np.zeros_like(amax_b, dtype=np.uint8)
        d = np.zeros_like(amax_b, dtype=np.float32)
    safe = np.where(d > 0, d, np.float32(1.0)).astype(np.float32)
    q = encode_e2m1((xb / safe[:, :, None]).astype(np.float32))
    q = np.where((d > 0)[:, :, None], q, np.uint8(0)).reshape(M, K).astype(np.uint8)
    packed = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    return packed, sb.astype(np.uint8), g


# ---------------------------------------------------------------- MoE layer: Down GEMM with combine, gated activation
#
# A MoE layer's speed-up counts its Gate-up and its Down GEMM ("Results: kernel microbenchmarks").  Between them the
# gated activation joins the gate and up halves of each routed row; the Down GEMM takes the routed rows (row t*k + j
# goes to expert ids[t, j]) and the k results of a token are summed with their top-k weights into one row.


def moe_combine(adeq_rows, wdeq_of_expert, n_out, topk_ids, topk_weights=None, tokens=None):
    """out[t] = sum_j topk_w[t, j] * (Adeq_rows[t*k + j] . Wdeq[ids[t, j]]^T), float64.

    `wdeq_of_expert(e)` returns expert e's decoded [N, K] weights, or None for an id that names no expert (that
    routed row adds nothing).  `tokens` restricts the tokens computed; None computes all T.
    """
    ids = np.asarray(topk_ids)
    T, k = ids.shape
    toks = np.arange(T) if tokens is None else np.asarray(tokens)
    y = np.zeros((len(toks), n_out))
    cache = {}
    for i, t in enumerate(toks):
        for j in range(k):
            e = int(ids[t, j])
            if e not in cache:
                cache[e] = wdeq_of_expert(e)
            w = cache[e]
            if w is None:
                continue
            v = np.asarray(adeq_rows[int(t) * k + j], dtype=np.float64) @ np.asarray(w, dtype=np.float64).T
            if topk_weights is not None:
                v = v * float(np.asarray(topk_weights)[t, j])
            y[i] += v
    return y


def swiglu(x):
    """Gated activation of x = [gate | up] ([R, 2I]): silu(gate) * up with silu(g) = g / (1 + exp(-g)), float64."""
    x = np.asarray(x, dtype=np.float64)
    half = x.shape[1] // 2
    g, u = x[:, :half], x[:, half:]
    return g / (1.0 + np.exp(-g)) * u
