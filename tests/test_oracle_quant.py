"""Pins for the oracle's quantisation: scale rule, E2M1 rounding, packing, page
layout and the exact dequantise round-trip.  Each check compares the oracle with
something it does not contain: hand-worked encodings, an exact rational
derivation of the scale, an independent exponent-spacing RNE, the byte-size
invariant the pages print, and values that are already representable."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from sparse_attention_indexer_quant_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mxfp4_blocks.txt")


def _bf16_value(bits):
    u = np.array([int(bits) << 16], np.uint32)
    return float(u.view(np.float32)[0])


def _bits_of(x):
    """bf16 bits of a value that is exactly representable in bf16."""
    f = np.array([x], np.float32)
    u = int(f.view(np.uint32)[0])
    assert u & 0xFFFF == 0, f"{x} is not bf16-exact"
    return u >> 16


def _load_golden():
    cases = []
    with open(GOLDEN) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, vals, scale, data = [p.strip() for p in line.split("|")]
            bits = np.zeros(32, np.uint16)
            for tok in vals.split():
                i, v = tok.split(":", 1)
                if v.startswith("bf16:"):
                    bits[int(i)] = int(v[5:], 16)
                else:
                    bits[int(i)] = _bits_of(float(v))
            cases.append((name, bits, int(scale, 16), bytes.fromhex(data.replace(" ", ""))))
    return cases


GOLDEN_CASES = _load_golden()


@pytest.mark.parametrize("case", GOLDEN_CASES, ids=[c[0] for c in GOLDEN_CASES])
def test_golden_block(oracle, case):
    name, bits, scale, data = case
    # place the block in slot 1 of a 128-vector whose other blocks are zero
    vec = np.zeros(128, np.uint16)
    vec[32:64] = bits
    v, s = oracle.quant_vec128(vec)
    assert s[1] == scale, f"{name}: scale {s[1]:#x} != {scale:#x}"
    assert bytes(v[16:32]) == data, f"{name}: {bytes(v[16:32]).hex()} != {data.hex()}"
    assert s[0] == s[2] == s[3] == 0
    assert not v[:16].any() and not v[32:].any()


def test_golden_blocks_keep_block_order(oracle):
    """Four different blocks in one vector: scale bytes come out in block order
    and each block's 16 value bytes land at 16*block."""
    picks = [GOLDEN_CASES[i] for i in (0, 1, 2, 8)]
    vec = np.concatenate([c[1] for c in picks])
    v, s = oracle.quant_vec128(vec)
    assert list(s) == [c[2] for c in picks]
    assert bytes(v) == b"".join(c[3] for c in picks)


def _scale_closed_form(bits):
    """Scale byte from the fp32 bit fields of amax: amax = M*2^(E-127) with
    M in [1,2); 6*2^e = 1.5*2^(e+2), so e = E-129 when M <= 1.5 and E-128
    otherwise; byte = e + 127, clamped."""
    u = int(bits) << 16
    E = (u >> 23) & 0xFF
    m = u & 0x7FFFFF
    if (u & 0x7FFFFFFF) == 0:
        return 0
    byte = E - 2 + (1 if m > 0x400000 else 0)
    return min(max(byte, 0), 254)


def _scale_exact(value):
    """Scale byte with exact rational arithmetic: smallest e with amax <= 6*2^e."""
    a = Fraction(abs(value))
    if a == 0:
        return 0
    e = math.floor(math.log2(float(a) / 6.0)) - 2
    while a > 6 * Fraction(2) ** e:
        e += 1
    while a <= 6 * Fraction(2) ** (e - 1):
        e -= 1
    return min(max(e + 127, 0), 254)


def test_scale_all_positive_bf16(oracle):
    """Every positive finite bf16 as the block maximum: the oracle's scale byte
    equals the bit-field closed form; a sample also equals the exact rational
    derivation."""
    g = wl.rng(7)
    sample = set(g.choice(np.arange(1, 0x7F80), size=600, replace=False).tolist())
    block = np.zeros(32)
    for bits in range(1, 0x7F80):
        x = _bf16_value(bits)
        block[5] = x
        block[9] = -x * 0.5
        got = oracle.ue8m0_scale(block)
        assert got == _scale_closed_form(bits), hex(bits)
        if bits in sample:
            assert got == _scale_exact(x), hex(bits)


def _e2m1_by_spacing(y):
    """E2M1 code from the format's structure instead of a grid search: in
    [2^k, 2^(k+1)) (k >= 0) the step is 2^(k-1), below 1 it is 0.5; round
    y/step to nearest-even as an exact fraction; saturate above 6."""
    a = Fraction(abs(y))
    sign = 8 if math.copysign(1.0, y) < 0 else 0
    if a > 6:
        return sign | 7
    if a < 1:
        step = Fraction(1, 2)
    else:
        k = math.floor(math.log2(a))
        while Fraction(2) ** k > a:
            k -= 1
        while Fraction(2) ** (k + 1) <= a:
            k += 1
        step = Fraction(2) ** (k - 1)
    r = round(a / step) * step          # Fraction.__round__ is half-to-even
    grid = [Fraction(x) for x in (0, 0.5, 1, 1.5, 2, 3, 4, 6)]
    return sign | grid.index(r)


def test_e2m1_dense_grid(oracle):
    """All multiples of 1/64 in [-8, 8], both zeros and a few extremes."""
    ys = [i / 64.0 for i in range(-512, 513)] + [-0.0, 0.0, 6.0000001, 1e30, -1e30, 1e-30, -1e-30]
    for y in ys:
        assert oracle.e2m1_code(y) == _e2m1_by_spacing(y), y


def test_e2m1_random_bf16(oracle):
    g = wl.rng(11)
    bits = g.integers(0, 0x7F80, size=4000)
    for b in bits:
        for sgn in (1.0, -1.0):
            y = sgn * _bf16_value(int(b))
            y = y / 2.0 ** 120 if abs(y) > 1e30 else y
            assert oracle.e2m1_code(y) == _e2m1_by_spacing(y), y


def test_e2m1_values(oracle):
    assert [oracle.e2m1_value(c) for c in range(8)] == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert [oracle.e2m1_value(c | 8) for c in range(1, 8)] == [-0.5, -1, -1.5, -2, -3, -4, -6]


def test_round_trip_of_representable_values(oracle):
    """x = c * 2^e with c on the E2M1 grid and one |c| = 6 per block: the block
    scale is exactly 2^e, every code is exact, dequantise returns x."""
    g = wl.rng(3)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    for trial in range(200):
        x = np.empty(128)
        for b in range(4):
            e = int(g.integers(-60, 60))
            c = grid[g.integers(0, 8, size=32)] * np.where(g.random(32) < 0.5, -1, 1)
            c[g.integers(0, 32)] = 6.0 * (1 if g.random() < 0.5 else -1)
            x[32 * b:32 * b + 32] = c * 2.0 ** e
        bits = np.array([_bits_of(v) for v in x], np.uint16)
        v, s = oracle.quant_vec128(bits)
        back = oracle.dequant_vec128(v, s)
        assert np.array_equal(back, x)


def test_format_size_invariant(oracle):
    """128 bf16 -> 64 value + 4 scale = 68 bytes, against FP8's 128 + 4 = 132
    (vLLM PR #48558, "Benefit": 132 -> 68 B/token/head, ~1.94x); a page of 64
    tokens is 4352 bytes."""
    v, s = oracle.quant_vec128(np.zeros(128, np.uint16))
    assert v.nbytes + s.nbytes == 68
    assert 128 * 1 + 4 == 132
    assert abs(132 / 68 - 1.94) < 0.005
    cache = wl.poisoned_cache(2)
    assert cache.shape[1] == 64 * 68 == 4352


def test_insert_layout(oracle):
    """Token i at slot page*64 + off changes exactly value bytes
    [page*4352 + off*64, +64) and scale bytes [page*4352 + 4096 + off*4, +4);
    slot -1 writes nothing; out-of-range slots write nothing and are counted."""
    g = wl.rng(5)
    k = wl.normal_bf16(g, (5, 128))
    slots = np.array([3 * 64 + 17, -1, 0, 4 * 64 - 1, 4 * 64], np.int64)
    cache = wl.poisoned_cache(4)
    before = cache.copy()
    bad = oracle.quant_insert(k, slots, cache)
    assert bad == 1
    flat, flat0 = cache.reshape(-1), before.reshape(-1)
    changed = np.zeros(flat.size, bool)
    for i, slot in [(0, 3 * 64 + 17), (2, 0), (3, 4 * 64 - 1)]:
        page, off = divmod(slot, 64)
        v, s = oracle.quant_vec128(k[i])
        vo = page * 4352 + off * 64
        so = page * 4352 + 4096 + off * 4
        assert np.array_equal(flat[vo:vo + 64], v)
        assert np.array_equal(flat[so:so + 4], s)
        changed[vo:vo + 64] = True
        changed[so:so + 4] = True
    assert np.array_equal(flat[~changed], flat0[~changed])


def test_insert_respects_row_stride(oracle):
    """A K tensor with row stride > 128 (a view into a wider buffer) quantises
    only the first 128 columns of each row."""
    g = wl.rng(9)
    wide = wl.normal_bf16(g, (3, 192))
    cache_a = wl.poisoned_cache(1)
    cache_b = wl.poisoned_cache(1)
    slots = np.array([5, 6, 7], np.int64)
    oracle.quant_insert(wide, slots, cache_a)            # stride 192
    oracle.quant_insert(wide[:, :128].copy(), slots, cache_b)
    assert np.array_equal(cache_a, cache_b)


def test_quant_q_matches_vector_rule(oracle):
    g = wl.rng(13)
    q = wl.normal_bf16(g, (3, 4, 128))
    v, s = oracle.quant_q(q)
    assert v.shape == (12, 64) and s.shape == (12, 4)
    for r in range(12):
        v1, s1 = oracle.quant_vec128(q.reshape(12, 128)[r])
        assert np.array_equal(v[r], v1) and np.array_equal(s[r], s1)
