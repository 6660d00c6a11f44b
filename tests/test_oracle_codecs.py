"""Pins for the oracle's element and scale codecs (E2M1, E4M3, E8M0).

Each codec is checked against something other than itself: the format facts
the ResServe paper prints (App. B.2: largest magnitudes 6 and 448), the
library casts in ml_dtypes / torch, exhaustive round trips and every
rounding midpoint.
"""
import numpy as np
import pytest
import torch

from conftest import read_golden

E2M1_MAGS = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_format_facts_match_paper(oracle_mod):
    facts = {k: float(v[0]) for k, v in read_golden("format_facts.txt").items()}
    o = oracle_mod
    assert max(abs(o.e2m1_decode(c)) for c in range(16)) == facts["e2m1_max"]
    finite = [o.e4m3_decode(b) for b in range(256) if not np.isnan(o.e4m3_decode(b))]
    assert max(finite) == facts["e4m3_max"]
    assert o.block_size(o.NVFP4) == facts["nvfp4_block"]
    assert o.block_size(o.MXFP4) == facts["mxfp4_block"]
    assert facts["tensor_scale_divisor"] == facts["e2m1_max"] * facts["e4m3_max"]


def test_e2m1_decode_all_codes(oracle_mod):
    for c in range(16):
        mag = E2M1_MAGS[c & 7]
        v = oracle_mod.e2m1_decode(c)
        assert v == (-mag if c & 8 else mag)
        assert np.signbit(v) == bool(c & 8)


def test_e2m1_round_trip(oracle_mod):
    for c in range(16):
        assert oracle_mod.e2m1_encode(oracle_mod.e2m1_decode(c)) == c


@pytest.mark.parametrize("v,code", [
    (0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6),
    (np.nextafter(np.float32(0.25), np.float32(1)), 1),
    (np.nextafter(np.float32(0.75), np.float32(0)), 1),
    (np.nextafter(np.float32(1.25), np.float32(2)), 3),
    (np.nextafter(np.float32(1.75), np.float32(0)), 3),
    (np.nextafter(np.float32(2.5), np.float32(9)), 5),
    (np.nextafter(np.float32(3.5), np.float32(0)), 5),
    (np.nextafter(np.float32(5.0), np.float32(9)), 7),
    (6.5, 7), (100.0, 7), (3.0e38, 7), (0.0, 0), (-0.0, 8), (-0.1, 8), (-5.0, 14),
])
def test_e2m1_midpoints_and_saturation(oracle_mod, v, code):
    assert oracle_mod.e2m1_encode(float(np.float32(v))) == code


def test_e2m1_against_ml_dtypes(oracle_mod):
    mld = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(0)
    v = np.concatenate([
        rng.uniform(-6, 6, 200_000).astype(np.float32),
        np.arange(-6.0, 6.0001, 0.03125, dtype=np.float32),   # every quarter-step midpoint
    ])
    ours = oracle_mod.e2m1_encode_array(v)
    lib = v.astype(mld.float4_e2m1fn).view(np.uint8) & 0xF
    np.testing.assert_array_equal(ours, lib)


def test_e4m3_decode_against_torch(oracle_mod):
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = b.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([oracle_mod.e4m3_decode(i) for i in range(256)])
    nan = np.isnan(lib)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    np.testing.assert_array_equal(np.isnan(ours), nan)
    np.testing.assert_array_equal(ours[~nan], lib[~nan])


def test_e4m3_round_trip_all_finite(oracle_mod):
    for b in range(256):
        if b in (0x7F, 0xFF):
            continue
        assert oracle_mod.e4m3_encode(oracle_mod.e4m3_decode(b)) == b


def test_e4m3_ties_every_binade(oracle_mod):
    """Midpoint between consecutive codes rounds to the even code, including
    the subnormal range and the subnormal/normal boundary."""
    o = oracle_mod
    for c in range(0, 0x7E):
        lo, hi = o.e4m3_decode(c), o.e4m3_decode(c + 1)
        mid = np.float32((lo + hi) / 2)
        assert float(mid) == (lo + hi) / 2          # exact in fp32
        want = c if c % 2 == 0 else c + 1
        assert o.e4m3_encode(float(mid)) == want, (hex(c), float(mid))
        assert o.e4m3_encode(float(np.nextafter(mid, np.float32(0)))) == c
        assert o.e4m3_encode(float(np.nextafter(mid, np.float32(1e9)))) == c + 1


def test_e4m3_against_torch_cast(oracle_mod):
    rng = np.random.default_rng(1)
    v = np.concatenate([
        np.exp(rng.uniform(np.log(1e-4), np.log(460.0), 300_000)).astype(np.float32),
        rng.uniform(0, 2.0 ** -6, 50_000).astype(np.float32),   # subnormal range
    ])
    ours = oracle_mod.e4m3_encode_array(v)
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, lib)


def test_e4m3_saturates_never_nan(oracle_mod):
    for t in [448.0, 449.0, 463.9, 464.0, 500.0, 1e6, 3e38]:
        assert oracle_mod.e4m3_encode(t) == 0x7E
    assert oracle_mod.e4m3_decode(0x7E) == 448.0


def test_e8m0_decode_against_torch(oracle_mod):
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = b.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    ours = np.array([oracle_mod.e8m0_decode(i) for i in range(256)])
    assert np.isnan(lib[255]) and np.isnan(ours[255])
    np.testing.assert_array_equal(ours[:255], lib[:255])
