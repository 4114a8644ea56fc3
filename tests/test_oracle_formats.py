"""Pins of the oracle's number formats (bf16, e4m3, e2m1, the fp4 block round trip).

Each check compares the oracle with something other than itself: values worked by hand
from the pages' definitions (tests/golden), torch's own bf16 conversion, exact rational
arithmetic, or a second, differently built rounding routine (nearest-by-distance search).
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                yield line.split()


# ---- e2m1 -------------------------------------------------------------------------------

def test_e2m1_hand_worked_grid():
    for inp, code, val in _rows("e2m1_rne_grid.txt"):
        got = oracle.e2m1_from_f32(float(np.float32(inp)))
        assert got == int(code, 16), (inp, hex(got), code)
        v = oracle.e2m1_to_f64(got)
        assert v == float(val) and np.signbit(v) == np.signbit(float(val)), (inp, v, val)


E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1_by_search(q: float) -> int:
    """Second, independent e2m1 rounding: nearest grid point by distance, ties to the even code."""
    a = min(abs(q), 6.0)
    d = np.abs(E2M1_GRID - a)
    best = np.flatnonzero(d == d.min())
    code = int(best[0]) if len(best) == 1 else int([b for b in best if b % 2 == 0][0])
    return code | (8 if np.signbit(q) else 0)


def test_e2m1_against_search_on_dense_grid():
    qs = np.concatenate([np.linspace(-8, 8, 4001), E2M1_GRID, -E2M1_GRID,
                         (E2M1_GRID[1:] + E2M1_GRID[:-1]) / 2])
    for q in qs.astype(np.float32):
        assert oracle.e2m1_from_f32(float(q)) == e2m1_by_search(float(q)), q


# ---- e4m3 -------------------------------------------------------------------------------

def _all_e4m3_finite():
    vals = {}
    for b in range(256):
        v = oracle.e4m3_to_f64(b)
        if not np.isnan(v):
            vals[b] = v
    return vals


def test_e4m3_decode_table():
    vals = _all_e4m3_finite()
    assert len(vals) == 254  # 0x7F and 0xFF are NaN in the e4m3 "fn" format
    assert vals[0x7E] == 448.0 and vals[0x01] == 2.0 ** -9 and vals[0x08] == 2.0 ** -6 and vals[0x38] == 1.0
    assert sorted(v for b, v in vals.items() if b < 0x80) == [vals[b] for b in range(0x7F)]  # monotone


def test_e4m3_round_trip_and_nearest():
    vals = _all_e4m3_finite()
    pos = sorted(set(v for v in vals.values() if v >= 0))
    for b, v in vals.items():
        got = oracle.e4m3_from_f32(float(v))
        assert oracle.e4m3_to_f64(got) == v and (v != 0 or got == b)
    # midpoints between neighbours tie to the even mantissa; points just off a midpoint go to the nearer
    rng = np.random.default_rng(0)
    xs = list(rng.uniform(0, 460, 2000)) + list(rng.uniform(0, 0.05, 2000))
    xs += [(a + b) / 2 for a, b in zip(pos[:-1], pos[1:])]
    for x in np.array(xs, dtype=np.float32):
        x = float(x)
        got = oracle.e4m3_to_f64(oracle.e4m3_from_f32(x))
        d = [abs(p - x) for p in pos]
        m = min(d)
        cands = [p for p, dd in zip(pos, d) if dd == m]
        if x > 448:
            assert got == 448.0
        elif len(cands) == 1:
            assert got == cands[0], (x, got, cands)
        else:  # tie: even mantissa bit
            even = [p for p in cands if oracle.e4m3_from_f32(p) % 2 == 0]
            assert got == even[0], (x, got, cands)


def test_e4m3_scale_examples():
    for amax, bits, val in _rows("e4m3_scale_examples.txt"):
        blk = np.zeros(16, np.uint16)
        blk[3] = oracle.bf16_from_f32(float(amax))
        blk[7] = oracle.bf16_from_f32(-float(amax) / 2)
        _, scales, _ = oracle.fp4_e4m3(blk)
        assert scales[0] == int(bits, 16), (amax, hex(scales[0]), bits)
        assert oracle.e4m3_to_f64(int(scales[0])) == float(val)


# ---- bf16 -------------------------------------------------------------------------------

def test_bf16_from_f32_matches_torch():
    rng = np.random.default_rng(1)
    xs = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 20000),
                         np.array([0.0, -0.0, 1.0, 3.0e38, 1e-40, -1e-42, 65504.0], np.float32)]).astype(np.float32)
    # exact ties: float32 values with the low 16 bits = 0x8000
    ties = (rng.integers(0x00800000, 0x7F000000, 4000, dtype=np.int64) & ~0xFFFF | 0x8000).astype(np.uint32)
    xs = np.concatenate([xs, ties.view(np.float32)])
    ref = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_from_f32(float(x)) for x in xs], np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_from_f64_is_correctly_rounded():
    rng = np.random.default_rng(2)
    xs = rng.standard_normal(3000) * 10.0 ** rng.integers(-20, 20, 3000)
    for x in xs:
        h = oracle.bf16_from_f64(float(x))
        v = Fraction(oracle.bf16_to_f32(h))
        # neighbours of v in bf16
        lo = Fraction(oracle.bf16_to_f32(h - 1)) if (h & 0x7FFF) else None
        hi = Fraction(oracle.bf16_to_f32(h + 1))
        fx = Fraction(float(x))
        err = abs(v - fx)
        for nb in (lo, hi):
            if nb is not None:
                assert err <= abs(nb - fx), (x, h)


# ---- fp4 block --------------------------------------------------------------------------

def test_fp4_block_saturation_and_exact_dequant():
    # amax 6.375 -> scale e4m3(1.0625) = 1.0 (tie to even); 6.375 / 1 saturates to 6
    vals = [6.375, -3.0, 0.75, 0.25, 1.25, 5.0, -6.375, 0.0] + [0.5] * 8
    blk = np.array([oracle.bf16_from_f32(v) for v in vals], np.uint16)
    codes, scales, out = oracle.fp4_e4m3(blk)
    assert scales[0] == 0x38
    deq = [oracle.bf16_to_f32(int(h)) for h in out]
    assert deq[:8] == [6.0, -3.0, 1.0, 0.0, 1.0, 4.0, -6.0, 0.0]
    # nibble packing: element 2i in the low nibble
    assert codes[0] == (0x7 | (0xD << 4)) and codes[1] == (0x2 | (0x0 << 4))


def test_fp4_block_all_bf16_patterns_against_search():
    """Every finite bf16 pattern as the block's first value, with fixed companions: the
    oracle's codes must match a search-based e2m1 of x/scale, its scale the e4m3 of amax/6."""
    pats = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    f = (pats.astype(np.uint32) << 16).view(np.float32)
    pats = pats[np.isfinite(f)]
    companions = [np.float32(0.3), np.float32(-1.7)]
    blocks = np.zeros((pats.size, 16), np.uint16)
    blocks[:, 0] = pats
    for i in range(1, 16):
        blocks[:, i] = oracle.bf16_from_f32(float(companions[i % 2] * i))
    codes, scales, out = oracle.fp4_e4m3(blocks)
    codes = codes.reshape(-1, 8)
    out = out.reshape(-1, 16)
    rng = np.random.default_rng(3)
    idx = np.concatenate([rng.choice(pats.size, 3000, replace=False), np.arange(0, pats.size, 97)])
    for r in idx:
        vals = (blocks[r].astype(np.uint32) << 16).view(np.float32)
        amax = np.float32(np.max(np.abs(vals)))
        sq = np.float32(max(amax, np.float32(6 * 2.0 ** -9)) / np.float32(6.0))
        s_bits = int(scales[r])
        assert s_bits == oracle.e4m3_from_f32(float(sq))
        s = np.float32(oracle.e4m3_to_f64(s_bits))
        q = np.float32(vals[0] / s)
        c0 = int(codes[r, 0] & 0xF)
        assert c0 == e2m1_by_search(float(q)), (hex(blocks[r, 0]), float(q), c0)
        assert oracle.bf16_to_f32(int(out[r, 0])) == np.float32(E2M1_GRID[c0 & 7] * (1 - 2 * (c0 >> 3)) * s)


# ---- the indexer's fp4 block: power-of-two (e8m0) scales, block 32 ------------------------

def test_e8m0_scale_examples():
    for amax, byte, val in _rows("e8m0_scale_examples.txt"):
        blk = np.zeros(32, np.uint16)
        blk[5] = oracle.bf16_from_f32(float(amax))
        blk[30] = oracle.bf16_from_f32(-float(amax) / 3)
        _, scales, _ = oracle.fp4_e8m0(blk)
        assert scales[0] == int(byte), (amax, scales[0], byte)
        assert Fraction(2) ** (int(scales[0]) - 127) == Fraction(float(val))


def test_fp4_e8m0_blocks_against_exact_arithmetic():
    """Random blocks over 60 decades: the scale is the least power of two at or above the
    float32 quotient amax/6 (exact rationals), every code is the search-based e2m1 of
    value/scale, the dequantised value is code * scale, and codes pack two per byte."""
    rng = np.random.default_rng(4)
    nb = 3000
    mags = 10.0 ** rng.uniform(-30, 30, size=(nb, 1))
    vals = (rng.standard_normal((nb, 32)) * mags).astype(np.float32)
    vals[:20] = 0.0
    vals[20:40, 7] = 6.0 * 2.0 ** rng.integers(-20, 20, size=20)  # amax / 6 a power of two
    bits = np.stack([[oracle.bf16_from_f32(float(v)) for v in row] for row in vals]).astype(np.uint16)
    codes, scales, out = oracle.fp4_e8m0(bits)
    codes = codes.reshape(nb, 16)
    out = out.reshape(nb, 32)
    floor = Fraction(6) * Fraction(2) ** -126
    for r in range(nb):
        v = (bits[r].astype(np.uint32) << 16).view(np.float32)
        amax = max(Fraction(float(np.max(np.abs(v)))), floor)
        q = Fraction(float(np.float32(float(amax)) / np.float32(6.0)))  # the float32 quotient
        s = Fraction(2) ** (int(scales[r]) - 127)
        assert s >= q and s / 2 < q, (r, float(q), float(s))
        for i in range(32):
            c = int(codes[r, i // 2] >> (4 * (i % 2))) & 0xF
            assert c == e2m1_by_search(float(Fraction(float(v[i])) / s)), (r, i)
            want = Fraction(float(E2M1_GRID[c & 7])) * s * (-1 if c & 8 else 1)
            assert Fraction(float(oracle.bf16_to_f32(int(out[r, i])))) == want, (r, i)


def test_fp4_e8m0_exact_powers():
    # amax = 6 * 2^k: scale 2^k, the largest value maps to code 7 (6.0), half of it to 3.0
    for k in (-100, -3, 0, 5, 100):
        blk = np.zeros(32, np.uint16)
        blk[0] = oracle.bf16_from_f32(6.0 * 2.0 ** k)
        blk[1] = oracle.bf16_from_f32(-3.0 * 2.0 ** k)
        codes, scales, out = oracle.fp4_e8m0(blk)
        assert scales[0] == 127 + k
        assert codes[0] == (0x7 | (0xD << 4))
        assert oracle.bf16_to_f32(int(out[0])) == 6.0 * 2.0 ** k
