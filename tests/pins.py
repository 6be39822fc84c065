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


ALL_PINS = [pin_e4m3, pin_e8m0, pin_e2m1, pin_bf16, pin_int4, pin_e0m_equivalence, pin_exact_int4,
            pin_exact_fp4, pin_library_special_case, pin_brute_force, pin_moe_reduces_to_dense]
