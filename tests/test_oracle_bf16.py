"""Pin of the oracle's bf16 decoding (every oracle value starts from it).

bfloat16 is the upper half of an IEEE-754 binary32: 1 sign bit, 8 exponent
bits (bias 127), 7 fraction bits.  ``bf16_to_f64`` is checked on all 65,536
bit patterns against torch's own bfloat16 -> float64 conversion and against
the format's definition evaluated field by field, with NaN patterns compared
as NaN."""
import math

import numpy as np
import torch

from oracle.dflash_oracle import bf16_to_f64


def _by_definition(bits: int) -> float:
    sign = -1.0 if bits >> 15 else 1.0
    exp = (bits >> 7) & 0xFF
    frac = bits & 0x7F
    if exp == 0xFF:
        return sign * math.inf if frac == 0 else math.nan
    if exp == 0:                       # subnormal: no implicit leading one
        return sign * math.ldexp(frac, -126 - 7)
    return sign * math.ldexp(128 + frac, exp - 127 - 7)


def test_bf16_to_f64_all_patterns_match_torch():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # the sign of zero survives
    assert np.signbit(got[0x8000]) and not np.signbit(got[0x0000])


def test_bf16_to_f64_matches_the_format_definition():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = bf16_to_f64(bits)
    ref = np.array([_by_definition(int(b)) for b in range(1 << 16)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_to_f64_worked_values():
    cases = {0x3F80: 1.0, 0xC000: -2.0, 0x3F00: 0.5, 0x4049: 3.140625, 0x0001: 2.0 ** -133,
             0x7F7F: (2 - 2.0 ** -7) * 2.0 ** 127, 0x7F80: math.inf, 0xFF80: -math.inf}
    for b, v in cases.items():
        assert bf16_to_f64(np.array([b], np.uint16))[0] == v, hex(b)


def test_round_bf16_matches_torch_and_round_trips():
    """float64 -> bf16 rounding of the oracle (used where float64 values are
    handed to a bf16 consumer): every bf16 value maps to itself, midpoints go
    to the even neighbour, and random float32 values round as torch rounds
    float32 to bfloat16."""
    from oracle.dflash_oracle import round_bf16
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = bf16_to_f64(bits)
    ok = ~np.isnan(vals)
    assert np.array_equal(round_bf16(vals[ok]), bits[ok])
    # midpoints between 1.0 (0x3F80) and its successor 0x3F81, and 0x3F81 / 0x3F82
    assert round_bf16(np.array([1.0 + 2.0 ** -8]))[0] == 0x3F80
    assert round_bf16(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 0x3F82
    rng = np.random.default_rng(9)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-30, 30, 200000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(round_bf16(x.astype(np.float64)), ref)
