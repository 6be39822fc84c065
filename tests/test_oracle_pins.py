"""The CPU oracle against facts outside itself (no GPU)."""
import numpy as np
import pytest
import torch

import oracle
from tests import pins
from workload import quant


def test_generic_minifloat_matches_torch():
    pins.pin_minifloat_against_torch()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(oracle)


# ---------------------------------------------------------------- the input recipes

def test_int4_sym_codes_are_e0m3_and_round_trip():
    w = torch.randn(64, 256) * 0.02
    codes, s = quant.quant_int4_sym(w, 128)
    q = oracle.unpack_nibbles(codes.numpy())
    assert not np.any(q == 8)  # -8 is never produced: the code set is e0m3's
    deq = oracle.dequant_weights("int4_sym", codes.numpy(), s.view(torch.int16).numpy().view(np.uint16), group=128)
    sc = np.repeat(oracle.decode_bf16(s.view(torch.int16).numpy().view(np.uint16)), 128, axis=-1)
    assert np.all(np.abs(deq - w.double().numpy()) <= sc * 0.5 * (1 + 2 ** -7) + 1e-12)


def test_uint4_zp_round_trip():
    w = torch.randn(64, 256) * 0.02
    codes, s, z = quant.quant_uint4_zp(w, 128)
    sb = s.view(torch.int16).numpy().view(np.uint16)
    deq = oracle.dequant_weights("uint4_zp", codes.numpy(), sb, zeros=z.numpy(), group=128)
    sc = np.repeat(oracle.decode_bf16(sb), 128, axis=-1)
    assert np.all(np.abs(deq - w.double().numpy()) <= sc * 1.0 + 1e-12)
    assert np.mean(np.abs(deq - w.double().numpy()) <= sc * 0.5 * (1 + 2 ** -7)) > 0.99


def test_e2m1_encode_ties_to_even():
    v = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, -0.25, -5.0, 100.0])
    got = oracle.decode_e2m1(quant.e2m1_encode(v).numpy())
    assert np.array_equal(got, [0, 1, 1, 2, 2, 4, 4, 6, 0, -4, 6])


def test_nvfp4_round_trip():
    x = torch.randn(32, 256)
    codes, sb, g = quant.quant_nvfp4(x)
    deq = oracle.dequant_acts("nvfp4", codes.numpy(), sb.numpy(), g.reshape(1).numpy())
    unit = np.repeat(oracle.decode_ue4m3(sb.numpy()), 16, axis=-1) * float(g)
    # |x| / unit <= 6 within the scale's rounding; error at most one grid step (2 units at the top)
    assert np.all(np.abs(deq - x.double().numpy()) <= 2.0 * unit + 1e-9)


def test_mxfp4_round_trip():
    w = torch.randn(32, 256) * 0.02
    codes, e = quant.quant_mxfp4(w)
    deq = oracle.dequant_weights("mxfp4", codes.numpy(), e.numpy())
    unit = np.repeat(oracle.decode_e8m0(e.numpy()), 32, axis=-1)
    assert np.all(np.abs(deq - w.double().numpy()) <= 2.0 * unit)


def test_e4m3_per_token_round_trip():
    a = torch.randn(8, 512)
    q, s = quant.quant_e4m3_per_token(a)
    deq = oracle.dequant_acts("e4m3_tok", q.numpy(), s.numpy())
    rel = np.abs(deq - a.double().numpy()) / np.maximum(np.abs(a.double().numpy()), 2 ** -6 * s.numpy()[:, None])
    assert np.all(rel <= 2 ** -4 + 1e-9)
