"""Pins for the oracle's bf16 helpers, ``oracle.bf16_round`` and
``oracle.bf16_bits_to_f64``.

The GPU tests compare the library's bf16 output with the FP64 oracle rounded
to bf16 ("Hand-Writing Gemma 4 Flash-Decoding + an FP4 Matvec Bonus (Part 2)",
section "The test that catches what parity misses": an FP64 host reference
over the same bf16-rounded inputs). Both helpers sit on that checking path, so
each is pinned here against something other than itself:

  * bf16_bits_to_f64, on all 65,536 bit patterns, against torch's own
    bfloat16 -> float64 conversion;
  * bf16_round, on float32-exact inputs, against torch's float32 -> bfloat16
    conversion (one round-to-nearest-even step; torch converts float64 through
    float32, which rounds twice, so torch is used only where the float32 image
    is exact);
  * bf16_round, on general float64 inputs, against an exact rational
    definition of round-to-nearest-even written with Python's Fraction
    (the nearest multiple of the binade's quantum, ties to the even multiple,
    overflow to infinity at 2^128);
  * planted mistakes (ties to odd, truncation, the wrong overflow threshold, a
    wrong shift in the bit conversion) fail at least one of these checks.
"""

import inspect
import math
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle


# ----------------------------------------------------------------- references

def exact_bf16_bits(x: float) -> int:
    """Round a float64 to bf16 (8 significant bits, exponent range of
    float32, subnormals down to 2^-133) by exact rational arithmetic, ties to
    the even multiple; the result's bit pattern."""
    if math.isnan(x):
        return 0x7FC0
    sign = 0x8000 if math.copysign(1.0, x) < 0 else 0
    if math.isinf(x):
        return sign | 0x7F80
    ax = Fraction(abs(x))
    if ax == 0:
        return sign
    e = math.frexp(abs(x))[1] - 1          # 2^e <= |x| < 2^(e+1), exactly
    quantum = Fraction(2) ** (max(e, -126) - 7)
    n = ax / quantum
    k = n.numerator // n.denominator       # floor
    rem = n - k
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and k % 2 == 1):
        k += 1
    val = k * quantum
    if val >= Fraction(2) ** 128:
        return sign | 0x7F80
    f32 = struct.unpack("<I", struct.pack("<f", float(val)))[0]  # val is a bf16 value, exact in float32
    assert f32 & 0xFFFF == 0
    return sign | (f32 >> 16)


def torch_bf16_bits_from_f32(x32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------------ the checks

def _f32_exact_inputs(rng) -> np.ndarray:
    """float32 values: random bit patterns over every exponent (subnormals
    included), exact bf16 midpoints with odd and even lower neighbours, the
    neighbours of those midpoints, values at and around the overflow midpoint,
    signed zeros, infinities."""
    bits = rng.integers(0, 1 << 32, size=20000, dtype=np.uint64).astype(np.uint32)
    exp = (bits >> 23) & 0xFF
    bits = bits[exp != 0xFF]                                         # no NaN / inf here
    hi = rng.integers(0, 0x7F80, size=4000, dtype=np.uint32)         # finite bf16 magnitudes
    sgn = (rng.integers(0, 2, size=4000, dtype=np.uint32) << 31)
    mid = sgn | (hi << 16) | 0x8000                                  # exact ties, both parities
    around = np.concatenate([mid - 1, mid + 1])
    special = np.array([0x7F7F7FFF, 0x7F7F8000, 0x7F7F8001, 0x7F7FFFFF, 0xFF7F8000, 0xFF7F7FFF,
                        0x00000000, 0x80000000, 0x7F800000, 0xFF800000, 0x00000001, 0x00008000,
                        0x00018000, 0x80008000, 0x007FFFFF, 0x00800000, 0x3F808000, 0x3F818000],
                       dtype=np.uint32)
    allb = np.concatenate([bits, mid, around, special]).astype(np.uint32)
    return allb.view(np.float32)


def _f64_inputs(rng) -> np.ndarray:
    """float64 values that float32 cannot hold: random mantissas over every
    bf16 exponent (subnormal range included), and values one float64 step on
    either side of exact bf16 midpoints (where rounding through float32 first
    would round twice)."""
    e = rng.integers(-140, 128, size=3000)
    m = rng.random(3000) + 1.0
    s = np.where(rng.random(3000) < 0.5, -1.0, 1.0)
    rnd = s * np.ldexp(m, e)
    hi = rng.integers(1, 0x7F7F, size=1500, dtype=np.uint32)
    mid = ((hi << 16) | 0x8000).view(np.float32).astype(np.float64)
    near = np.concatenate([np.nextafter(mid, np.inf), np.nextafter(mid, -np.inf)])
    over = np.array([(2.0 - 2.0 ** -8) * 2.0 ** 127, np.nextafter((2.0 - 2.0 ** -8) * 2.0 ** 127, 0.0),
                     3.0e38, 3.5e38, 1e300, -1e300, 2.0 ** -134, 2.0 ** -133 * 1.5, 2.0 ** -134 * 1.0000001])
    return np.concatenate([rnd, near, -near, over])


def check_round(fn) -> list:
    """Failures of a bf16 rounding function against the two references."""
    rng = np.random.default_rng(2024)
    fails = []
    x32 = _f32_exact_inputs(rng)
    got = fn(x32.astype(np.float64))
    want = torch_bf16_bits_from_f32(x32)
    bad = got != want
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        fails.append(f"float32 input {x32[i]!r} (bits {x32.view(np.uint32)[i]:#010x}): "
                     f"got {int(got[i]):#06x}, torch {int(want[i]):#06x} ({int(bad.sum())} differ)")
    x64 = _f64_inputs(rng)
    got = fn(x64)
    want = np.array([exact_bf16_bits(float(v)) for v in x64], dtype=np.uint16)
    bad = got != want
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        fails.append(f"float64 input {x64[i]!r}: got {int(got[i]):#06x}, exact {int(want[i]):#06x} "
                     f"({int(bad.sum())} differ)")
    nan = fn(np.array([np.nan, -np.nan]))
    if not all(((int(b) & 0x7F80) == 0x7F80) and (int(b) & 0x7F) for b in nan):
        fails.append("NaN did not map to a bf16 NaN")
    return fails


def check_bits_to_f64(fn) -> list:
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = fn(bits)
    want = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    both_nan = np.isnan(got) & np.isnan(want)
    same = (got == want) & (np.signbit(got) == np.signbit(want))
    bad = ~(same | both_nan)
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        return [f"bits {i:#06x}: got {got[i]!r}, torch {want[i]!r} ({int(bad.sum())} differ)"]
    return []


def test_exact_reference_agrees_with_torch_where_torch_rounds_once():
    """The rational reference itself, on float32-exact inputs, equals torch."""
    rng = np.random.default_rng(7)
    x32 = _f32_exact_inputs(rng)[::7]
    want = torch_bf16_bits_from_f32(x32)
    got = np.array([exact_bf16_bits(float(v)) for v in x32.astype(np.float64)], dtype=np.uint16)
    assert (got == want).all()


def test_bf16_round_is_round_to_nearest_even():
    assert check_round(oracle.bf16_round) == []


def test_bf16_bits_to_f64_on_every_pattern():
    assert check_bits_to_f64(oracle.bf16_bits_to_f64) == []


def test_bf16_round_hand_values():
    # 1 + 2^-8 is the midpoint of 1 and 1 + 2^-7: ties to the even 1.0;
    # 1 + 3 * 2^-8 lies between 1 + 2^-7 (odd) and 1 + 2^-6: ties to 1 + 2^-6.
    cases = [(1.0, 0x3F80), (1.0 + 2.0 ** -8, 0x3F80), (1.0 + 3 * 2.0 ** -8, 0x3F82),
             (1.0 + 2.0 ** -8 + 2.0 ** -40, 0x3F81), (-2.0, 0xC000), (0.0, 0x0000), (-0.0, 0x8000),
             ((2.0 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F), ((2.0 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),
             (2.0 ** -133, 0x0001), (2.0 ** -134, 0x0000), (1.5 * 2.0 ** -133, 0x0002)]
    got = oracle.bf16_round(np.array([x for x, _ in cases]))
    assert [int(g) for g in got] == [b for _, b in cases]


# -------------------------------------------------------------- planted mistakes

def _mutant(fn, old: str, new: str):
    src = inspect.getsource(fn)
    assert src.count(old) == 1, f"mutation site not unique: {old!r}"
    ns = dict(oracle.__dict__)
    exec(compile(src.replace(old, new), f"<mutant of {fn.__name__}>", "exec"), ns)
    return ns[fn.__name__]


ROUND_MUTANTS = {
    # ties go to the candidate whose mantissa LSB is one
    "ties_to_odd": ("(((cands[i] >> 16) & 1) == 1) \\\n                & (((cands[j] >> 16) & 1) == 0)",
                    "(((cands[i] >> 16) & 1) == 0) \\\n                & (((cands[j] >> 16) & 1) == 1)"),
    # keep the upper 16 bits of the float32 image: truncation
    "truncation": ("bits = np.choose(best, cands)", "bits = cands[1]; best = np.ones_like(best)"),
    # overflow only from 2^128 on (the midpoint below it should already overflow)
    "overflow_threshold": ("over = np.abs(x) >= (2.0 - 2.0 ** -8) * 2.0 ** 127", "over = np.abs(x) >= 2.0 ** 128"),
    # round through float32 only (double rounding)
    "via_float32": ("errs = np.stack([np.abs(v - x) for v in vals])",
                    "errs = np.stack([np.abs(v - f.astype(np.float64)) for v in vals])"),
}


@pytest.mark.parametrize("name", sorted(ROUND_MUTANTS))
def test_round_pins_catch_planted_mistake(name):
    old, new = ROUND_MUTANTS[name]
    assert check_round(_mutant(oracle.bf16_round, old, new)) != []


def test_bits_pins_catch_planted_mistake():
    m = _mutant(oracle.bf16_bits_to_f64, "<< 16", "<< 15")
    assert check_bits_to_f64(m) != []
    m = _mutant(oracle.bf16_bits_to_f64, ".view(np.float32)", ".view(np.int32)")
    assert check_bits_to_f64(m) != []
