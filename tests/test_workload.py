"""The seeded input generator: Philox known answers and the workload shapes (no GPU)."""
import torch

from workload import philox, configs


def _t(x):
    return torch.tensor([x], dtype=torch.int64)


def test_philox_known_answers():
    # Known-answer vectors of Philox-4x32-10 distributed with the Random123 library
    # (Salmon et al., SC'11): counter, key -> output.
    kat = [((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
           ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
           ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
            (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1))]
    for ctr, key, want in kat:
        got = philox.philox4x32_10(*[_t(c) for c in ctr], *key)
        assert tuple(int(g) for g in got) == want


def test_normal_is_chunk_invariant():
    full = philox.normal(7, 1, 4096)
    part = philox.normal(7, 1, 1024, offset=512)
    assert torch.equal(full[2048:3072], part)
    assert abs(float(full.mean())) < 0.1 and abs(float(full.std()) - 1) < 0.05


def test_routing_is_distinct_and_normalised():
    ids, w = configs.zipf_route(0, 64, 32, 8)
    for row in ids.tolist():
        assert len(set(row)) == 8 and all(0 <= e < 32 for e in row)
    assert torch.allclose(w.sum(1), torch.ones(64), atol=1e-6)
    # Zipf(1.1): expert 0 is the most popular
    counts = torch.bincount(ids.reshape(-1).long(), minlength=32)
    assert int(counts.argmax()) == 0


def test_dense_and_moe_shapes():
    d = configs.make_dense("w4a16_asym", 3, N=256, K=512)
    assert d["w"]["codes"].shape == (256, 256) and d["w"]["zeros"].shape == (256, 4)
    m = configs.make_moe("moe_mxfp4", 5, E=4, N=64, K=256)
    assert m["w"]["codes"].shape == (4, 64, 128) and m["w"]["scales"].shape == (4, 64, 8)
    assert m["a"]["data"].dtype == torch.uint8 and m["a"]["scale"].shape == (5,)


def test_bit_string_packer_matches_the_loop_packer():
    """The recipe's 1/2/3-bit packer writes the same bytes as the pins' independent loop packer."""
    import numpy as np

    from tests.pins import pack_bits_loop
    from workload import quant
    g = torch.Generator().manual_seed(3)
    for bits in (1, 2, 3):
        q = torch.randint(0, 1 << bits, (3, 64), generator=g, dtype=torch.uint8)
        assert np.array_equal(quant.pack_bits(q, bits).numpy(), pack_bits_loop(q.numpy(), bits))
    q2 = torch.randint(0, 4, (2, 32), generator=g, dtype=torch.uint8)
    assert torch.equal(quant.pack_bits(q2, 2), quant.pack_crumbs(q2))


def test_uint1_uint3_shapes_and_ranges():
    for wfmt, bits in (("uint1_zp", 1), ("uint3_zp", 3)):
        d = configs.make_dense(dict(kind="dense", wfmt=wfmt, afmt="bf16", G=128), 2, N=64, K=256)
        assert d["w"]["codes"].shape == (64, 256 * bits // 8)
        assert d["w"]["zeros"].shape == (64, 2) and int(d["w"]["zeros"].max()) < (1 << bits)
