"""Checks that pin the CPU oracle to facts outside itself.

Each `pin_*` takes the oracle module (so a test can hand it a copy with a planted
mistake) and raises AssertionError on failure.  The facts come from:

* library decoders: torch.float8_e4m3fn, torch.float8_e5m2, torch.float8_e8m0fnu,
  torch.bfloat16 (independent implementations of the OCP / IEEE formats);
* a generic minifloat decoder written here and cross-checked against those library
  decoders, then applied to E2M1 (OCP Microscaling v1.0: 2 exponent bits, bias 1,
  1 mantissa bit, no inf/NaN), for which torch has no CPU decoder;
* the zero-exponent-float statement of the Humming announcement ("Results:
  quantization support"): INT8 without -128 and float8e0m7 both hold -127..127;
* exact integer arithmetic (integer operands, power-of-two scales) and
  brute-force Fraction sums on tiny shapes.
"""
import os
from fractions import Fraction

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------ independent decoders

def minifloat(code, ebits, mbits, bias, ieee_specials=False, fn_nan=False, signed=True):
    """Generic sign/exponent/mantissa decoder returning a Fraction (or 'nan'/'inf')."""
    code = int(code)
    s = (code >> (ebits + mbits)) & 1 if signed else 0
    e = (code >> mbits) & ((1 << ebits) - 1)
    m = code & ((1 << mbits) - 1)
    emax = (1 << ebits) - 1
    if ieee_specials and e == emax:
        return "nan" if m else ("-inf" if s else "inf")
    if fn_nan and e == emax and m == (1 << mbits) - 1:
        return "nan"
    if e == 0:
        mag = Fraction(m, 1 << mbits) * Fraction(2) ** (1 - bias)
    else:
        mag = (1 + Fraction(m, 1 << mbits)) * Fraction(2) ** (e - bias)
    return -mag if s else mag


def e2m1_table():
    return [minifloat(c, 2, 1, 1) for c in range(16)]


def int4_value(c, signed):
    v = np.array([(int(c) & 0xF) << 4], dtype=np.uint8).view(np.int8)[0]
    return int(v) >> 4 if signed else int(c) & 0xF


def e0m_value(code, mbits):
    """Zero-exponent float: sign bit above an mbits-bit integer magnitude."""
    s = (int(code) >> mbits) & 1
    m = int(code) & ((1 << mbits) - 1)
    return -m if s else m


def _same(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.array_equal(np.isnan(a), np.isnan(b)) and np.array_equal(a[~np.isnan(a)], b[~np.isnan(b)])


# ------------------------------------------------------------ pins on the decoders

def pin_minifloat_against_torch():
    """The generic decoder reproduces torch's e4m3fn and e5m2 tables exactly."""
    for dt, kw in ((torch.float8_e4m3fn, dict(ebits=4, mbits=3, bias=7, fn_nan=True)),
                   (torch.float8_e5m2, dict(ebits=5, mbits=2, bias=15, ieee_specials=True))):
        ref = torch.arange(256, dtype=torch.uint8).view(dt).double().numpy()
        mine = [minifloat(c, **kw) for c in range(256)]
        mine = np.array([float(x) for x in mine])
        assert _same(ref, mine), dt


def pin_e4m3(o):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    assert _same(o.decode_e4m3(np.arange(256)), ref)
    ue = o.decode_ue4m3(np.arange(256))
    assert _same(ue[:128], ref[:128]) and np.all(np.isnan(ue[128:]))


def pin_e8m0(o):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
    assert _same(o.decode_e8m0(np.arange(256)), ref)


def pin_e2m1(o):
    mine = np.array([float(x) for x in e2m1_table()])
    assert _same(o.decode_e2m1(np.arange(16)), mine)
    # closed-form facts of OCP E2M1: max 6, smallest positive 0.5, 8 magnitudes
    v = o.decode_e2m1(np.arange(16))
    assert v.max() == 6.0 and v[v > 0].min() == 0.5 and len(set(np.abs(v))) == 8


def pin_bf16(o):
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 16, size=4096, dtype=np.uint32).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]  # skip inf/NaN patterns
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    assert np.array_equal(o.decode_bf16(bits), ref)


def pin_int4(o):
    codes = np.arange(16)
    assert np.array_equal(o.decode_int(codes, 4, True), [int4_value(c, True) for c in codes])
    assert np.array_equal(o.decode_int(codes, 4, False), [int4_value(c, False) for c in codes])


def _golden_range(name):
    with open(os.path.join(GOLDEN, "e0m_value_sets.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                n, lo, hi = line.split()
                if n == name:
                    return int(lo), int(hi)
    raise KeyError(name)


def pin_e0m_equivalence(o):
    """Symmetric INT8 (no -128) and float8e0m7 share the value set -127..127; same at width 4."""
    lo, hi = _golden_range("int8_without_min")
    lo2, hi2 = _golden_range("float8e0m7")
    ints = set(o.decode_int(np.array([c for c in range(256) if c != 0x80]), 8, True).astype(int).tolist())
    e0m7 = {e0m_value(c, 7) for c in range(256)}
    assert ints == set(range(lo, hi + 1)) and e0m7 == set(range(lo2, hi2 + 1)) and ints == e0m7
    ints4 = set(o.decode_int(np.array([c for c in range(16) if c != 8]), 4, True).astype(int).tolist())
    assert ints4 == {e0m_value(c, 3) for c in range(16)} == set(range(-7, 8))


# ------------------------------------------------------------ pins on the products

def pack_nibbles_loop(q):
    """Independent packer: byte i holds k = 2i in the low nibble, k = 2i+1 in the high one."""
    q = np.asarray(q)
    out = np.zeros(q.shape[:-1] + (q.shape[-1] // 2,), dtype=np.uint8)
    for idx in np.ndindex(q.shape[:-1]):
        for i in range(q.shape[-1] // 2):
            out[idx + (i,)] = (int(q[idx + (2 * i,)]) & 0xF) | ((int(q[idx + (2 * i + 1,)]) & 0xF) << 4)
    return out


def bf16_pow2(j):
    return np.uint16((127 + j) << 7)


def pin_exact_int4(o, rng=None):
    """Integer codes, integer activations, power-of-two scales: the oracle equals integer math."""
    rng = rng or np.random.default_rng(1)
    N, K, M, G = 6, 64, 3, 16
    q = rng.integers(-7, 8, size=(N, K))
    a = rng.integers(-3, 4, size=(M, K))
    sj = rng.integers(-3, 3, size=(N, K // G))
    scales = np.vectorize(bf16_pow2)(sj).astype(np.uint16)
    w = o.dequant_weights("int4_sym", pack_nibbles_loop(q & 0xF), scales, group=G)
    y = o.gemm(o.decode_bf16(np.vectorize(lambda v: np.float32(v).view(np.uint32) >> 16)(a).astype(np.uint16)), w)
    ref = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            ref[m, n] = sum(int(a[m, k]) * int(q[n, k]) * 2.0 ** int(sj[n, k // G]) for k in range(K))
    assert np.array_equal(y, ref)
    # zero points
    qu = rng.integers(0, 16, size=(N, K))
    z = rng.integers(0, 16, size=(N, K // G))
    w = o.dequant_weights("uint4_zp", pack_nibbles_loop(qu), scales, zeros=z.astype(np.uint8), group=G)
    ref = np.array([[(qu[n, k] - z[n, k // G]) * 2.0 ** int(sj[n, k // G]) for k in range(K)] for n in range(N)])
    assert np.array_equal(w, ref)


def pin_exact_fp4(o, rng=None):
    """e2m1 codes with power-of-two block scales decode and multiply exactly (Fraction sums)."""
    rng = rng or np.random.default_rng(2)
    tab = e2m1_table()
    N, K, M = 4, 64, 2
    qw = rng.integers(0, 16, size=(N, K))
    qa = rng.integers(0, 16, size=(M, K))
    # NVFP4: ue4m3 power-of-two scales (byte (j + 7) << 3 is 2**j), global 2**-3
    jw = rng.integers(-4, 4, size=(N, K // 16))
    ja = rng.integers(-4, 4, size=(M, K // 16))
    sw = ((jw + 7) << 3).astype(np.uint8)
    sa = ((ja + 7) << 3).astype(np.uint8)
    w = o.dequant_weights("nvfp4", pack_nibbles_loop(qw), sw, gscale=np.array([0.125], np.float32))
    a = o.dequant_acts("nvfp4", pack_nibbles_loop(qa), sa, np.array([0.5], np.float32))
    y = o.gemm(a, w)
    for m in range(M):
        for n in range(N):
            ref = sum(tab[qa[m, k]] * Fraction(2) ** int(ja[m, k // 16]) * Fraction(1, 2)
                      * tab[qw[n, k]] * Fraction(2) ** int(jw[n, k // 16]) * Fraction(1, 8) for k in range(K))
            assert y[m, n] == float(ref)
    # MXFP4 weights: e8m0 scales, against e4m3 activations with a per-token power-of-two scale
    je = rng.integers(-6, 3, size=(N, K // 32))
    w = o.dequant_weights("mxfp4", pack_nibbles_loop(qw), (je + 127).astype(np.uint8))
    a8 = rng.integers(0, 256, size=(M, K)).astype(np.uint8)
    a8[(a8 & 0x7F) == 0x7F] = 0x38  # no NaN codes
    st = np.array([0.25, 2.0], dtype=np.float32)
    a = o.dequant_acts("e4m3_tok", a8, st)
    y = o.gemm(a, w)
    for m in range(M):
        for n in range(N):
            ref = sum(minifloat(a8[m, k], 4, 3, 7, fn_nan=True) * Fraction(float(st[m]))
                      * tab[qw[n, k]] * Fraction(2) ** int(je[n, k // 32]) for k in range(K))
            assert y[m, n] == float(ref)


def pin_library_special_case(o, rng=None):
    """Unit scales, zero zero-points, unit global scale: Y = A . decode(codes)^T by torch.matmul."""
    rng = rng or np.random.default_rng(3)
    N, K, M, G = 16, 128, 5, 32
    q = rng.integers(0, 16, size=(N, K))
    ones = np.full((N, K // G), 0x3F80, dtype=np.uint16)
    a = rng.standard_normal((M, K)).astype(np.float32)
    abits = (a.view(np.uint32) >> 16).astype(np.uint16)
    at = torch.from_numpy(abits.view(np.int16).copy()).view(torch.bfloat16).double()
    qt = torch.from_numpy(q.astype(np.int64))
    signed = torch.where(qt >= 8, qt - 16, qt).double()
    y = o.gemm(o.dequant_acts("bf16", abits), o.dequant_weights("int4_sym", pack_nibbles_loop(q), ones, group=G))
    assert np.allclose(y, (at @ signed.T).numpy(), rtol=1e-13, atol=1e-13)
    y = o.gemm(o.dequant_acts("bf16", abits),
               o.dequant_weights("uint4_zp", pack_nibbles_loop(q), ones, zeros=np.zeros((N, K // G), np.uint8), group=G))
    assert np.allclose(y, (at @ qt.double().T).numpy(), rtol=1e-13, atol=1e-13)
    # e4m3 activations with unit token scale against torch's e4m3 decoder
    a8 = rng.integers(0, 256, size=(M, K)).astype(np.uint8)
    a8[(a8 & 0x7F) == 0x7F] = 0
    a8t = torch.from_numpy(a8).view(torch.float8_e4m3fn).double()
    y = o.gemm(o.dequant_acts("e4m3_tok", a8, np.ones(M, np.float32)),
               o.dequant_weights("int4_sym", pack_nibbles_loop(q), ones, group=G))
    assert np.allclose(y, (a8t @ signed.T).numpy(), rtol=1e-13, atol=1e-12)


def pin_brute_force(o, rng=None):
    """M, N, K tiny: a pure-Python Fraction triple loop equals the oracle (bias and MoE included)."""
    rng = rng or np.random.default_rng(4)
    M, N, K, G = 3, 5, 32, 16
    q = rng.integers(0, 16, size=(N, K))
    z = rng.integers(0, 16, size=(N, K // G)).astype(np.uint8)
    s = (rng.standard_normal((N, K // G)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    a = (rng.standard_normal((M, K)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    bias = (rng.standard_normal(N).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)

    def bf(b):
        return Fraction(float(np.array([int(b) << 16], dtype=np.uint32).view(np.float32)[0]))

    y = o.gemm(o.dequant_acts("bf16", a), o.dequant_weights("uint4_zp", pack_nibbles_loop(q), s, zeros=z, group=G), bias)
    for m in range(M):
        for n in range(N):
            ref = sum(bf(a[m, k]) * (int(q[n, k]) - int(z[n, k // G])) * bf(s[n, k // G]) for k in range(K)) + bf(bias[n])
            assert abs(y[m, n] - float(ref)) <= 1e-12 * max(1.0, abs(float(ref)))
    # MoE: T=3 tokens, k=2 slots, E=3 experts of int4_sym weights
    E, T, k = 3, 3, 2
    qs = rng.integers(-7, 8, size=(E, N, K))
    ss = (rng.standard_normal((E, N, K // G)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    ids = np.array([[2, 0], [1, 2], [0, 1]])
    tw = rng.random((T, k)).astype(np.float32)
    wd = o.dequant_weights("int4_sym", pack_nibbles_loop(qs & 0xF), ss, group=G)
    ad = o.dequant_acts("bf16", a)
    ym = o.moe_gemm(ad, lambda e: wd[e], N, ids, tw)
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            for n in range(N):
                ref = Fraction(float(tw[t, j])) * sum(bf(a[t, kk]) * int(qs[e, n, kk]) * bf(ss[e, n, kk // G]) for kk in range(K))
                assert abs(ym[t * k + j, n] - float(ref)) <= 1e-12 * max(1.0, abs(float(ref)))


def pin_moe_reduces_to_dense(o, rng=None):
    rng = rng or np.random.default_rng(5)
    N, K, T, G = 8, 64, 4, 32
    q = rng.integers(-7, 8, size=(N, K))
    s = (rng.standard_normal((N, K // G)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    a = (rng.standard_normal((T, K)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    wd = o.dequant_weights("int4_sym", pack_nibbles_loop(q & 0xF), s, group=G)
    ad = o.dequant_acts("bf16", a)
    dense = o.gemm(ad, wd)
    moe = o.moe_gemm(ad, lambda e: wd, N, np.zeros((T, 1), np.int64), np.ones((T, 1), np.float32))
    assert np.array_equal(dense, moe)
    perm = rng.permutation(T)
    moe_p = o.moe_gemm(ad[perm], lambda e: wd, N, np.zeros((T, 1), np.int64))
    assert np.array_equal(moe_p, dense[perm])


def pack_crumbs_loop(q):
    """Independent packer of 2-bit codes: byte b holds k = 4b + i in bits 2i and 2i + 1."""
    q = np.asarray(q)
    out = np.zeros(q.shape[:-1] + (q.shape[-1] // 4,), dtype=np.uint8)
    for idx in np.ndindex(q.shape[:-1]):
        for b in range(q.shape[-1] // 4):
            v = 0
            for i in range(4):
                v |= (int(q[idx + (4 * b + i,)]) & 0x3) << (2 * i)
            out[idx + (b,)] = v
    return out


def pin_crumbs(o, rng=None):
    """2-bit code order: the oracle's unpacking inverts an independent loop packer, and a hand-made byte decodes as
    written (0b11_10_01_00 -> k = 0, 1, 2, 3 hold 0, 1, 2, 3)."""
    rng = rng or np.random.default_rng(11)
    q = rng.integers(0, 4, size=(3, 40))
    assert np.array_equal(o.unpack_crumbs(pack_crumbs_loop(q)), q)
    assert o.unpack_crumbs(np.array([0b11100100], np.uint8)).tolist() == [0, 1, 2, 3]


def pack_bits_loop(q, bits):
    """Independent packer of `bits`-bit codes into a little-endian bit string: bit j of code k goes to bit
    (k * bits + j) % 8 of byte (k * bits + j) // 8."""
    q = np.asarray(q)
    K = q.shape[-1]
    out = np.zeros(q.shape[:-1] + (K * bits // 8,), dtype=np.uint8)
    for idx in np.ndindex(q.shape[:-1]):
        for k in range(K):
            for j in range(bits):
                if (int(q[idx + (k,)]) >> j) & 1:
                    pos = k * bits + j
                    out[idx + (pos // 8,)] |= np.uint8(1 << (pos % 8))
    return out


def pin_bits(o, rng=None):
    """1- and 3-bit code order: the oracle's unpacking inverts an independent loop packer; hand-made bytes decode as
    written (0b10110001 -> k = 0..7 hold 1, 0, 0, 0, 1, 1, 0, 1; the 3-bit codes 5, 3, 6, 1, 0, 7, 2, 4 written by
    hand, lowest bit first, fill the bytes 0b10011101, 0b10000011, 0b10001011), and 2-bit codes agree with the
    crumb order."""
    rng = rng or np.random.default_rng(13)
    for bits in (1, 2, 3):
        q = rng.integers(0, 1 << bits, size=(3, 48))
        assert np.array_equal(o.unpack_bits(pack_bits_loop(q, bits), bits), q)
    assert o.unpack_bits(np.array([0b10110001], np.uint8), 1).tolist() == [1, 0, 0, 0, 1, 1, 0, 1]
    # codes 5, 3, 6, 1, 0, 7, 2, 4: bit string (LSB first) 101 110 011 100 000 111 010 001
    packed = np.array([0b10011101, 0b10000011, 0b10001011], np.uint8)
    assert o.unpack_bits(packed, 3).tolist() == [5, 3, 6, 1, 0, 7, 2, 4]
    q2 = rng.integers(0, 4, size=(2, 32))
    assert np.array_equal(o.unpack_bits(pack_crumbs_loop(q2), 2), o.unpack_crumbs(pack_crumbs_loop(q2)))


def _int_bf16(a):
    return np.vectorize(lambda v: np.float32(v).view(np.uint32) >> 16)(a).astype(np.uint16)


def pin_exact_more_formats(o, rng=None):
    """INT8 (e0m7 codes), UINT1 / UINT2 / UINT3 with zero points and MXINT4 with integer activations and power-of-two scales equal
    integer arithmetic; FP8 E4M3 weights equal torch's float8_e4m3fn decoder times a power-of-two scale; MXFP8
    activations equal the generic minifloat decoder times their e8m0 block scale (Fraction sums)."""
    rng = rng or np.random.default_rng(12)
    N, K, M, G = 5, 64, 3, 32
    a = rng.integers(-3, 4, size=(M, K))
    ad = o.dequant_acts("bf16", _int_bf16(a))
    sj = rng.integers(-3, 3, size=(N, K // G))
    scales = np.vectorize(bf16_pow2)(sj).astype(np.uint16)
    pw = 2.0 ** np.repeat(sj, G, axis=-1)

    def check(w, ref):
        assert np.array_equal(w, ref)
        y = o.gemm(ad, w)
        want = np.array([[sum(int(a[m, k]) * Fraction(ref[n, k]) for k in range(K)) for n in range(N)]
                         for m in range(M)], dtype=object)
        assert all(y[m, n] == float(want[m, n]) for m in range(M) for n in range(N))

    q8 = rng.integers(-127, 128, size=(N, K))
    check(o.dequant_weights("int8_sym", (q8 & 0xFF).astype(np.uint8), scales, group=G), q8 * pw)
    q2 = rng.integers(0, 4, size=(N, K))
    z2 = rng.integers(0, 4, size=(N, K // G))
    check(o.dequant_weights("uint2_zp", pack_crumbs_loop(q2), scales, zeros=z2.astype(np.uint8), group=G),
          (q2 - np.repeat(z2, G, axis=-1)) * pw)
    for bits, wf in ((1, "uint1_zp"), (3, "uint3_zp")):
        qb = rng.integers(0, 1 << bits, size=(N, K))
        zb = rng.integers(0, 1 << bits, size=(N, K // G))
        check(o.dequant_weights(wf, pack_bits_loop(qb, bits), scales, zeros=zb.astype(np.uint8), group=G),
              (qb - np.repeat(zb, G, axis=-1)) * pw)
    q4 = rng.integers(-7, 8, size=(N, K))
    je = rng.integers(-9, 5, size=(N, K // 32))
    check(o.dequant_weights("mxint4", pack_nibbles_loop(q4 & 0xF), (je + 127).astype(np.uint8)),
          q4 * 2.0 ** np.repeat(je, 32, axis=-1))
    b8 = rng.integers(0, 256, size=(N, K)).astype(np.uint8)
    b8[(b8 & 0x7F) == 0x7F] = 0x40  # no NaN codes
    ref = torch.from_numpy(b8.copy()).view(torch.float8_e4m3fn).double().numpy() * pw
    check(o.dequant_weights("e4m3", b8, scales, group=G), ref)
    # MXFP8 activations (e4m3 + e8m0 per 32) against int4 weights with unit scales
    a8 = rng.integers(0, 256, size=(M, K)).astype(np.uint8)
    a8[(a8 & 0x7F) == 0x7F] = 0x38
    ja = rng.integers(-5, 5, size=(M, K // 32))
    ax = o.dequant_acts("mxfp8", a8, (ja + 127).astype(np.uint8))
    qw = rng.integers(-7, 8, size=(N, K))
    w = o.dequant_weights("int4_sym", pack_nibbles_loop(qw & 0xF), np.full((N, K // G), 0x3F80, np.uint16), group=G)
    y = o.gemm(ax, w)
    for m in range(M):
        for n in range(N):
            ref = sum(minifloat(a8[m, k], 4, 3, 7, fn_nan=True) * Fraction(2) ** int(ja[m, k // 32]) * int(qw[n, k])
                      for k in range(K))
            assert y[m, n] == float(ref)
    # MXFP4 activations (e2m1 nibbles, low nibble = even k, + e8m0 per 32), same check with the E2M1 minifloat
    c4 = rng.integers(0, 16, size=(M, K))
    ax4 = o.dequant_acts("mxfp4", pack_nibbles_loop(c4), (ja + 127).astype(np.uint8))
    y4 = o.gemm(ax4, w)
    for m in range(M):
        for n in range(N):
            ref = sum(minifloat(c4[m, k], 2, 1, 1) * Fraction(2) ** int(ja[m, k // 32]) * int(qw[n, k])
                      for k in range(K))
            assert y4[m, n] == float(ref)


# ------------------------------------------------------------ pins on the activation quantizers

def _bf16_bits(x):
    """fp32 torch tensor -> bf16 bit patterns (numpy uint16), round to nearest even by torch."""
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _act_inputs(rng_seed, M, K):
    """bf16 activations with the awkward cases: a zero row, a single-spike row, tiny and huge values, ties."""
    g = torch.Generator().manual_seed(rng_seed)
    x = torch.randn(M, K, generator=g) * torch.exp2(torch.randint(-6, 7, (M, 1), generator=g).float())
    x[0] = 0.0
    if M > 1:
        x[1] = 0.0
        x[1, K // 3] = -3.0e4
    if M > 2:
        x[2] = torch.randn(K, generator=g) * 1e-30  # bf16 keeps these; their scales underflow
    return _bf16_bits(x)


def pin_encode_e4m3(o):
    """The saturating RNE e4m3 encoder is torch's float8_e4m3fn conversion of the input clamped to +-448, on random
    values, on every midpoint between neighbouring e4m3 values (exact ties) and one ulp either side of them."""
    vals = torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    mids = ((vals[:-1].astype(np.float64) + vals[1:]) / 2).astype(np.float32)
    rng = np.random.default_rng(7)
    rand = (rng.standard_normal(20000) * rng.choice([1e-3, 1.0, 30.0, 500.0], 20000)).astype(np.float32)
    v = np.concatenate([rand, mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9)),
                        np.array([0.0, 448.0, 460.0, 464.0, 480.0, 1e30, 2.0 ** -10, 3 * 2.0 ** -10], np.float32)])
    v = np.concatenate([v, -v]).astype(np.float32)
    ref = torch.from_numpy(np.clip(v, -448.0, 448.0)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(o.encode_e4m3(v), ref)


def pin_encode_e2m1(o):
    """Brute force over the 16 codes of the generic minifloat decoder: the nearest value, ties to the even code,
    +-6 saturation, and +0 for a zero result, on a grid that holds every tie and the points around it."""
    table = e2m1_table()
    grid = [Fraction(i, 16) for i in range(-128, 129)] + [Fraction(100), Fraction(-7)]
    v = np.array([float(x) for x in grid], np.float32)
    got = o.encode_e2m1(v)
    for x, c in zip(grid, got):
        best = None
        for code in range(8):  # magnitudes
            d = abs(abs(x) - table[code])
            key = (d, code % 2)  # nearest, then the even code
            if best is None or key < best[0]:
                best = (key, code)
        m = 7 if abs(x) >= 6 else best[1]
        want = m | (8 if (x < 0 and m > 0) else 0)
        assert int(c) == want, (x, int(c), want)


def pin_act_quant_e4m3(o):
    """Per-token FP8: the workloads' torch recipe gives the same bytes and scales; every non-zero row has an
    element at +-448; each element is within half an e4m3 step of x / s; zero rows have s = 0 and zero codes."""
    from workload import quant as WQ
    bits = _act_inputs(1, 9, 160)
    x = (bits.astype(np.uint32) << 16).view(np.float32)
    q, s = o.quantize_act_e4m3_per_token(bits)
    rq, rs = WQ.quant_e4m3_per_token(torch.from_numpy(x.copy()))
    assert np.array_equal(q, rq.numpy()) and np.array_equal(s.view(np.uint32), rs.numpy().view(np.uint32))
    dec = torch.from_numpy(q.copy()).view(torch.float8_e4m3fn).double().numpy()
    for m in range(x.shape[0]):
        if s[m] == 0:
            assert not x[m].any() and not q[m].any()
            continue
        assert np.abs(dec[m]).max() == 448.0
        y = x[m].astype(np.float64) / np.float64(s[m])
        assert np.all(np.abs(dec[m] - y) <= np.maximum(np.abs(y) * 2.0 ** -4, 2.0 ** -10) * (1 + 1e-6))


def pin_act_quant_nvfp4(o):
    """NVFP4: the workloads' torch recipe gives the same codes, block scales and tensor scale (also with a calibrated
    amax); g * 2688 is the amax; in each block whose scale is a normal unsaturated e4m3 the largest code is +-6."""
    from workload import quant as WQ
    bits = _act_inputs(2, 6, 96)
    x = (bits.astype(np.uint32) << 16).view(np.float32)
    for amax in (None, np.float32(np.abs(x).max() / 4)):
        q, sb, g = o.quantize_act_nvfp4(bits, global_amax=amax)
        ga = None if amax is None else torch.tensor(amax)
        rq, rsb, rg = WQ.quant_nvfp4(torch.from_numpy(x.copy()), global_amax=ga)
        assert np.array_equal(q, rq.numpy()) and np.array_equal(sb, rsb.numpy())
        assert np.float32(g).view(np.uint32) == rg.numpy().astype(np.float32).view(np.uint32)
    q, sb, g = o.quantize_act_nvfp4(bits)
    assert abs(float(g) * 2688.0 - float(np.abs(x).max())) <= 1e-6 * float(np.abs(x).max())
    codes = np.empty((q.shape[0], q.shape[1] * 2), np.uint8)
    codes[:, 0::2], codes[:, 1::2] = q & 0xF, q >> 4
    mag = np.array([float(v) for v in e2m1_table()])[codes & 7].reshape(q.shape[0], -1, 16)
    normal = (sb >= 8) & (sb < 0x7E)
    assert normal.any() and np.all(mag.max(axis=2)[normal] == 6.0)
    zero_rows = ~x.reshape(x.shape[0], -1).any(axis=1)
    assert not q[zero_rows].any() and not sb[zero_rows].any()


# ------------------------------------------------------------ pins on the MoE layer pieces

def pin_moe_combine(o, rng=None):
    """The combine equals an exact rational brute force on a tiny case (integer activations and weights, dyadic top-k
    weights), reduces to the routed-row product for k = 1, and does not depend on the order of a token's k slots."""
    rng = rng or np.random.default_rng(5)
    T, k, K, N, E = 3, 2, 4, 3, 3
    rows = rng.integers(-3, 4, size=(T * k, K)).astype(np.float64)
    W = rng.integers(-2, 3, size=(E, N, K)).astype(np.float64)
    ids = np.array([[0, 2], [1, 0], [2, 1]])
    tw = rng.integers(1, 8, size=(T, k)) / 8.0
    got = o.moe_combine(rows, lambda e: W[e], N, ids, tw)
    for t in range(T):
        for n in range(N):
            want = sum(Fraction(tw[t, j]) * sum(Fraction(rows[t * k + j, kk]) * Fraction(W[ids[t, j], n, kk])
                                                 for kk in range(K)) for j in range(k))
            assert Fraction(got[t, n]) == want
    one = o.moe_combine(rows, lambda e: W[e], N, ids.reshape(-1, 1))
    assert np.array_equal(one, np.stack([rows[i] @ W[ids.reshape(-1)[i]].T for i in range(T * k)]))
    perm = np.array([1, 0])
    rows_p = rows.reshape(T, k, K)[:, perm].reshape(T * k, K)
    assert np.array_equal(o.moe_combine(rows_p, lambda e: W[e], N, ids[:, perm], tw[:, perm]), got)


def pin_swiglu(o):
    """silu(gate) * up against torch's silu in float64, and the closed forms silu(0) = 0, silu(g) - silu(-g) = g."""
    g = torch.linspace(-30, 30, 241, dtype=torch.float64)
    u = torch.cos(g) * 3
    x = torch.cat([g.reshape(1, -1), u.reshape(1, -1)], dim=1).numpy()
    want = (torch.nn.functional.silu(g) * u).numpy()
    assert np.allclose(o.swiglu(x)[0], want, rtol=1e-14, atol=1e-300)
    ones = np.ones_like(g.numpy())
    sp = o.swiglu(np.concatenate([g.numpy(), ones])[None])[0]
    sm = o.swiglu(np.concatenate([-g.numpy(), ones])[None])[0]
    assert np.allclose(sp - sm, g.numpy(), rtol=1e-12, atol=1e-12)
    assert o.swiglu(np.array([[0.0, 5.0]]))[0, 0] == 0.0


ALL_PINS = [pin_e4m3, pin_e8m0, pin_e2m1, pin_bf16, pin_int4, pin_e0m_equivalence, pin_exact_int4,
            pin_exact_fp4, pin_crumbs, pin_bits, pin_exact_more_formats, pin_library_special_case, pin_brute_force, pin_moe_reduces_to_dense, pin_encode_e4m3,
            pin_encode_e2m1, pin_act_quant_e4m3, pin_act_quant_nvfp4, pin_moe_combine, pin_swiglu]
