"""Pins for the oracle's bf16 and FP8 E4M3 codecs.

The codecs are written from the format definitions (IEEE-754 binary32
truncated to bf16 with round-to-nearest-even; OCP FP8 E4M3FN).  They are pinned
here against PyTorch's own casts (an independent library implementation) and
against fixed points of the OCP specification.
"""
import numpy as np
import pytest
import torch


def _rand_f32_bits(rng, n):
    """Random finite fp32 values across the whole exponent range."""
    u = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    return f[np.isfinite(f)]


def test_bf16_encode_matches_torch_random(orc):
    rng = np.random.default_rng(11)
    x = _rand_f32_bits(rng, 1 << 20)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.bf16_encode(x)
    assert np.array_equal(got, want)


def test_bf16_encode_ties_and_neighbours(orc):
    rng = np.random.default_rng(12)
    hi = rng.integers(0, 0x7F7F, size=1 << 16, dtype=np.uint32)  # finite upper halves
    sign = rng.integers(0, 2, size=hi.size, dtype=np.uint32) << 31
    xs = []
    for low in (0x8000, 0x7FFF, 0x8001, 0x0000, 0xFFFF):
        xs.append(((hi << 16) | low | sign).astype(np.uint32).view(np.float32))
    x = np.concatenate(xs)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.bf16_encode(x), want)
    # ties go to the even pattern: 1 + 2^-8 sits halfway between 1 and 1 + 2^-7
    assert orc.bf16_encode(np.array([1.0 + 2.0**-8], np.float32))[0] == 0x3F80
    assert orc.bf16_encode(np.array([1.0 + 3 * 2.0**-8], np.float32))[0] == 0x3F82


def test_bf16_decode_matches_torch(orc):
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    want = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).float().numpy()
    got = orc.bf16_decode(h)
    fin = np.isfinite(want)
    assert np.array_equal(got[fin].view(np.uint32), want[fin].view(np.uint32))
    assert np.all(np.isnan(got[np.isnan(want)]))


def test_e4m3_decode_all_codes_match_torch(orc):
    codes = np.arange(256, dtype=np.uint32).astype(np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    got = orc.e4m3_decode(codes)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_e4m3_spec_points(orc):
    """Fixed points of the OCP FP8 E4M3 format (bias 7, no infinities)."""
    dec = orc.e4m3_decode(np.array([0x7E, 0x08, 0x01, 0x38, 0x00, 0x80, 0xFE], np.uint8))
    assert dec.tolist() == [448.0, 2.0**-6, 2.0**-9, 1.0, 0.0, 0.0, -448.0]
    assert np.isnan(orc.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()
    enc = orc.e4m3_encode(np.array([448.0, 2.0**-6, 2.0**-9, 1.0, -448.0], np.float32))
    assert enc.tolist() == [0x7E, 0x08, 0x01, 0x38, 0xFE]


def test_e4m3_roundtrip_fixed_point(orc):
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    v = orc.e4m3_decode(codes)
    again = orc.e4m3_decode(orc.e4m3_encode(v))
    assert np.array_equal(again, v)
    # encode(decode(c)) == c except that -0 and +0 stay distinct patterns
    assert np.array_equal(orc.e4m3_encode(v), codes)


def test_e4m3_encode_matches_torch_in_range(orc):
    rng = np.random.default_rng(13)
    x = np.concatenate([
        rng.uniform(-464, 464, 200000).astype(np.float32),
        (rng.standard_normal(200000) * 4).astype(np.float32),
        (rng.standard_normal(100000) * 2.0**-7).astype(np.float32),  # subnormal range
    ])
    # exact midpoints between neighbouring codes (ties) and their fp32 neighbours
    codes = np.array([c for c in range(127)], dtype=np.uint8)
    v = orc.e4m3_decode(codes).astype(np.float64)
    mids = ((v[:-1] + v[1:]) / 2).astype(np.float32)
    near = np.concatenate([mids, np.nextafter(mids, np.float32(0)),
                           np.nextafter(mids, np.float32(1e9))])
    x = np.concatenate([x, near, -near])
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = orc.e4m3_encode(x)
    assert np.array_equal(got, want)


def test_e4m3_saturates(orc):
    x = np.array([448.0, 449.0, 464.0, 465.0, 480.0, 1e6, np.inf, -1e6, -np.inf], np.float32)
    assert orc.e4m3_encode(x).tolist() == [0x7E] * 7 + [0xFE] * 2
    assert orc.e4m3_encode(np.array([np.nan], np.float32))[0] & 0x7F == 0x7F


@pytest.mark.parametrize("val,code", [(2.0**-10, 0x00), (3 * 2.0**-10, 0x02),
                                      (5 * 2.0**-10, 0x02), (1.0625, 0x38), (1.1875, 0x3A)])
def test_e4m3_ties_to_even(orc, val, code):
    assert orc.e4m3_encode(np.array([val], np.float32))[0] == code
