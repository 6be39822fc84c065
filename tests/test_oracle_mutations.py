"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check that a pin catches each."""
import importlib.util
import os

import numpy as np
import pytest

from tests import pins

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "hq_oracle.py")


def _mutant(old, new):
    src = open(ORACLE_SRC).read()
    assert old in src, old
    spec = importlib.util.spec_from_loader("oracle_mutant", loader=None)
    mod = importlib.util.module_from_spec(spec)
    exec(compile(src.replace(old, new, 1), "oracle_mutant", "exec"), mod.__dict__)
    return mod


MUTATIONS = {
    "nibble_order_swapped": ("out[..., 0::2] = p & 0xF", "out[..., 0::2] = p >> 4\n    out[..., 1::2] = p & 0xF\n    return out\n    out[..., 0::2] = p & 0xF"),
    "zero_point_dropped": ("(decode_int(q, 4, False) - zq)", "(decode_int(q, 4, False))"),
    "zero_point_sign": ("(decode_int(q, 4, False) - zq)", "(decode_int(q, 4, False) + zq)"),
    "weight_transposed": ("@ np.asarray(wdeq, dtype=np.float64).T", "@ np.asarray(wdeq, dtype=np.float64).T[::-1]"),
    "e2m1_subnormal": ("m * 0.5, np.ldexp", "m * 0.75, np.ldexp"),
    "e2m1_bias": ("(e - 1).astype(np.int32)", "(e - 2).astype(np.int32)"),
    "e4m3_bias": ("(e - 7).astype(np.int32)", "(e - 8).astype(np.int32)"),
    "e4m3_subnormal": ("np.ldexp(m / 8.0, -6)", "np.ldexp(m / 8.0, -7)"),
    "e8m0_bias": ("(b - 127).astype(np.int32)", "(b - 128).astype(np.int32)"),
    "int4_unsigned_as_signed": ("c = np.where(c >= (1 << (bits - 1)), c - (1 << bits), c)", "c = np.where(c > (1 << (bits - 1)), c - (1 << bits), c)"),
    "nvfp4_global_dropped": ("return decode_e2m1(q) * sb * g\n    if wfmt", "return decode_e2m1(q) * sb\n    if wfmt"),
    "act_token_scale_dropped": ("return decode_e4m3(data) * s", "return decode_e4m3(data)"),
    "act_nvfp4_block": ("np.repeat(decode_ue4m3(scale), 16, axis=-1)", "np.repeat(decode_ue4m3(scale), 32, axis=-1)"),
    "group_index": ("np.repeat(s, group, axis=-1)[..., :k]\n    if wfmt == \"uint4_zp\"", "np.tile(s, group)[..., :k]\n    if wfmt == \"uint4_zp\""),
    "bias_dropped": ("y = y + decode_bf16(bias).reshape(1, -1)", "y = y"),
    "topk_weight_dropped": ("v = v * float(np.asarray(topk_weights)[t, j])", "v = v"),
    "moe_slot_order": ("t, j = divmod(int(r), k)", "j, t = divmod(int(r), T)"),
    "encode_ties_to_odd": ("(d_hi == d_lo) & (hi % 2 == 0)", "(d_hi == d_lo) & (hi % 2 == 1)"),
    "encode_ties_away": ("(d_hi == d_lo) & (hi % 2 == 0)", "(d_hi == d_lo)"),
    "e2m1_signed_zero": ("np.signbit(v) & (m > 0)", "np.signbit(v)"),
    "e4m3_sign_dropped": ("np.where(np.signbit(v), m | np.uint8(0x80), m)", "np.where(v < -1e30, m | np.uint8(0x80), m)"),
    "act_fp8_max": ("s = (amax / E4M3_MAX).astype(np.float32)", "s = (amax / np.float32(447.0)).astype(np.float32)"),
    "act_fp8_reciprocal": ("q = encode_e4m3((x / safe[:, None]).astype(np.float32))",
                           "q = encode_e4m3((x * (np.float32(1.0) / safe)[:, None]).astype(np.float32))"),
    "act_nvfp4_six": ("six_g = np.float32(E2M1_MAX * g)", "six_g = np.float32(np.float32(4.0) * g)"),
    "act_nvfp4_global": ("g = np.float32(amax / np.float32(E2M1_MAX * E4M3_MAX))",
                         "g = np.float32(amax / np.float32(E4M3_MAX))"),
    "act_nvfp4_block_scale_unrounded": ("d = (decode_e4m3(sb).astype(np.float32) * g).astype(np.float32)",
                                        "d = (amax_b / np.float32(6.0)).astype(np.float32)"),
    "combine_weight_dropped": ("                v = v * float(np.asarray(topk_weights)[t, j])\n            y[i] += v",
                               "                v = v\n            y[i] += v"),
    "combine_row_index": ("np.asarray(adeq_rows[int(t) * k + j]", "np.asarray(adeq_rows[j * T + int(t)]"),
    "combine_overwrites": ("            y[i] += v", "            y[i] = v"),
    "silu_sign": ("return g / (1.0 + np.exp(-g)) * u", "return g / (1.0 + np.exp(g)) * u"),
    "gate_up_swapped": ("g, u = x[:, :half], x[:, half:]", "u, g = x[:, :half], x[:, half:]"),
    "crumb_order_reversed": ("out[..., i::4] = (p >> (2 * i)) & 0x3", "out[..., i::4] = (p >> (6 - 2 * i)) & 0x3"),
    "int8_as_unsigned": ("(decode_int(q, 8, True) if wfmt", "(decode_int(q, 8, False) if wfmt"),
    "uint2_zero_point_dropped": ("return (decode_int(q, 2, False) - zq) * s", "return decode_int(q, 2, False) * s"),
    "mxint4_block_16": ("np.repeat(decode_e8m0(scales), BLOCK[wfmt], axis=-1)[..., :k]\n        return decode_int(q, 4, True)",
                        "np.repeat(decode_e8m0(scales), 16, axis=-1)[..., :k]\n        return decode_int(q, 4, True)"),
    "mxint4_unsigned": ("return decode_int(q, 4, True) * sb", "return decode_int(q, 4, False) * sb"),
    "e4m3_weight_scale_dropped": ("else decode_e4m3(q)) * s", "else decode_e4m3(q)) * (s if wfmt == 'int8_sym' else 1.0)"),
    "mxfp8_scale_dropped": ("return decode_e4m3(q) * sb", "return decode_e4m3(q)"),
    "bit_string_msb_first": ('stream = np.unpackbits(p, axis=-1, bitorder="little")', 'stream = np.unpackbits(p, axis=-1, bitorder="big")'),
    "bit_weights_reversed": ("weights = np.int64(1) << np.arange(bits, dtype=np.int64)",
                             "weights = np.int64(1) << np.arange(bits, dtype=np.int64)[::-1]"),
    "uint3_zero_point_dropped": ("return (decode_int(q, bits, False) - zq) * s", "return decode_int(q, bits, False) * s"),
    "uint3_as_signed": ("return (decode_int(q, bits, False) - zq) * s", "return (decode_int(q, bits, True) - zq) * s"),
    "act_mxfp4_scale_dropped": ("        return decode_e2m1(q) * sb\n    if afmt == \"mxfp8\"", "        return decode_e2m1(q)\n    if afmt == \"mxfp8\""),
    "act_nvfp4_nibbles": ("packed = (q[:, 0::2] | (q[:, 1::2] << 4))", "packed = (q[:, 1::2] | (q[:, 0::2] << 4))"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name):
    mod = _mutant(*MUTATIONS[name])
    caught = []
    for pin in pins.ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mod)
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"


def test_unmutated_copy_passes():
    mod = _mutant("import numpy as np", "import numpy as np")
    for pin in pins.ALL_PINS:
        pin(mod)
