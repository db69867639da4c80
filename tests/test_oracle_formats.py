"""Pins for the oracle's number-format code (decoders and RNE rounding).

The oracle decodes fp16 / bf16 / e4m3 from the format definitions and rounds
FP64 results to fp16 / bf16 itself.  These tests pin it to things other than
itself: numpy's and torch's dtype casts over every bit pattern, and a
brute-force nearest-neighbour search over the complete table of representable
values (ties to the even bit pattern).
"""
import bisect
import math

import numpy as np
import pytest
import torch

import oracle


def _same(a: np.ndarray, b: np.ndarray) -> bool:
    nan_a, nan_b = np.isnan(a), np.isnan(b)
    return bool(np.array_equal(nan_a, nan_b) and np.array_equal(a[~nan_a], b[~nan_b]))


def test_decode_f16_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    assert _same(oracle.decode(bits, oracle.F16, orc), ref)


def test_decode_bf16_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert _same(oracle.decode(bits, oracle.BF16, orc), ref)


def test_decode_e4m3_all_patterns(orc):
    bits = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(bits).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.decode(bits, oracle.E4M3, orc)
    assert _same(got, ref)
    # format facts: largest finite 448, exactly two NaN encodings, no infinities
    assert np.nanmax(got) == 448.0 and np.isnan(got).sum() == 2 and not np.isinf(got).any()


def _table(fmt):
    """Sorted finite non-negative values of a 16-bit format with their bits (library decode)."""
    bits = np.arange(0, 0x8000, dtype=np.uint16)
    if fmt == oracle.F16:
        vals = bits.view(np.float16).astype(np.float64)
    else:
        vals = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    ok = np.isfinite(vals)
    order = np.argsort(vals[ok], kind="stable")
    return vals[ok][order], bits[ok][order]


def _nearest_even(x: float, vals, bits, inf_bits: int) -> int:
    """Brute force: nearest representable value by exact comparison, ties to even bits."""
    sign = 0x8000 if math.copysign(1.0, x) < 0 else 0
    a = abs(x)
    top = vals[-1]
    step = top - vals[-2]
    # the value one step past the largest finite one stands for infinity
    ext_vals = list(vals) + [top + step]
    ext_bits = list(bits) + [inf_bits]
    i = bisect.bisect_left(ext_vals, a)
    if i >= len(ext_vals):
        return sign | inf_bits
    if ext_vals[i] == a:
        return sign | int(ext_bits[i])
    lo, hi = i - 1, i
    dlo, dhi = a - ext_vals[lo], ext_vals[hi] - a
    if dlo < dhi:
        pick = lo
    elif dhi < dlo:
        pick = hi
    else:
        pick = lo if int(ext_bits[lo]) % 2 == 0 else hi
    return sign | int(ext_bits[pick])


def _probe_values(fmt, n_random=600, seed=7):
    rng = np.random.default_rng(seed)
    vals, _ = _table(fmt)
    xs = []
    # exact ties and near-ties between neighbours, across the whole range
    idx = rng.integers(0, len(vals) - 1, size=n_random)
    for i in idx:
        a, b = vals[i], vals[i + 1]
        mid = (a + b) / 2
        xs += [mid, np.nextafter(mid, -np.inf), np.nextafter(mid, np.inf), a, -mid]
    # random magnitudes including subnormal and overflow regions
    xs += list(rng.standard_normal(n_random) * np.exp2(rng.integers(-40, 140, n_random) if fmt == oracle.BF16 else rng.integers(-30, 18, n_random)))
    top, nxt = vals[-1], vals[-1] + (vals[-1] - vals[-2])
    xs += [top, (top + nxt) / 2, np.nextafter((top + nxt) / 2, 0), nxt, 0.0, -0.0]
    return [float(x) for x in xs if np.isfinite(x)]


@pytest.mark.parametrize("fmt", [oracle.F16, oracle.BF16])
def test_round_matches_bruteforce_nearest_even(orc, fmt):
    vals, bits = _table(fmt)
    inf_bits = 0x7C00 if fmt == oracle.F16 else 0x7F80
    xs = _probe_values(fmt)
    got = oracle.round_to(np.array(xs), fmt, orc)
    want = np.array([_nearest_even(x, vals, bits, inf_bits) for x in xs], dtype=np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(xs[i], hex(got[i]), hex(want[i])) for i in bad[:5]]


def test_round_f16_matches_numpy_single_step(orc):
    rng = np.random.default_rng(3)
    xs = rng.standard_normal(20000) * np.exp2(rng.integers(-28, 17, 20000))
    xs = np.concatenate([xs, [1 + 2**-11 + 2**-40, 65519.99, 65520.0, 6e-8, 3e-8]])
    with np.errstate(over="ignore"):
        want = xs.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.round_to(xs, oracle.F16, orc), want)


def test_round_bf16_matches_torch_on_float32_inputs(orc):
    # torch rounds float32 -> bf16 in one step, so float32-exact inputs are a valid pin
    rng = np.random.default_rng(4)
    with np.errstate(over="ignore"):
        xs = (rng.standard_normal(20000) * np.exp2(rng.integers(-130, 128, 20000))).astype(np.float32)
    xs = xs[np.isfinite(xs)]
    want = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.round_to(xs.astype(np.float64), oracle.BF16, orc), want)


def test_round_exact_ties_to_even(orc):
    # every midpoint between adjacent finite values: numpy (f16, from double) and torch
    # (bf16, from float32 -- midpoints of bf16 neighbours are exact in float32) round
    # ties to the even pattern in one step
    vals, _ = _table(oracle.F16)
    mids = (vals[:-1] + vals[1:]) / 2
    mids = np.concatenate([mids, -mids])
    assert np.array_equal(oracle.round_to(mids, oracle.F16, orc),
                          mids.astype(np.float16).view(np.uint16))
    vals, _ = _table(oracle.BF16)
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (vals[:-1] + vals[1:]) / 2)
    want = torch.from_numpy(mids).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.round_to(mids.astype(np.float64), oracle.BF16, orc), want)


def test_round_special_values(orc):
    f = oracle.round_to(np.array([np.inf, -np.inf, np.nan, 0.0, -0.0]), oracle.F16, orc)
    assert list(f[:2]) == [0x7C00, 0xFC00] and (f[2] & 0x7C00) == 0x7C00 and (f[2] & 0x3FF)
    assert list(f[3:]) == [0x0000, 0x8000]
    b = oracle.round_to(np.array([np.inf, -np.inf, np.nan]), oracle.BF16, orc)
    assert list(b[:2]) == [0x7F80, 0xFF80] and (b[2] & 0x7F80) == 0x7F80 and (b[2] & 0x7F)
