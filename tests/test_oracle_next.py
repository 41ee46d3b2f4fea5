"""Pins for the oracle's next steps: the fused q-RoPE + MXFP4 q-quant and the
K-pool compressed insert.  Each check compares the oracle with something it
does not contain: hand-worked rotations and pools, complex multiplication,
closed forms of the pooling (mean, one-hot, position-only weights), the mask
rule of the K-pool passage worked by hand on small batches, and special cases
that reduce to the already-pinned quantisation and insert."""
import math

import numpy as np
import pytest

from sparse_attention_indexer_quant_gb300 import workloads as wl


def _bf16_bits(x):
    return wl.bf16_bits(np.asarray(x, np.float32))


def _bf16_vals(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


def _table(num_pos, half, base=10000.0):
    """A rotary table: angle pos * base^(-i / half) for column i, fp32."""
    i = np.arange(half, dtype=np.float64)
    ang = np.arange(num_pos, dtype=np.float64)[:, None] * base ** (-i / max(half, 1))[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


# ---------------------------------------------------------------- RoPE + quant

def test_rope_identity_reduces_to_quant_q(oracle):
    q = wl.normal_bf16(wl.rng(11), (5, 4, 128))
    cs = np.ones((3, 32), np.float32)
    sn = np.zeros((3, 32), np.float32)
    v, s, r = oracle.rope_quant_q(q, [0, 1, 2, 1, 0], cs, sn, 64)
    v2, s2 = oracle.quant_q(q)
    assert np.array_equal(v, v2) and np.array_equal(s, s2)
    assert np.array_equal(r, _bf16_vals(q).reshape(-1, 128))


def test_rope_hand_worked_pairs(oracle):
    x = np.zeros(128, np.float32)
    x[0:4] = [1.0, 0.0, 3.0, 4.0]        # pairs (0, 1) and (2, 3)
    x[4:6] = [2.0, -1.0]                 # pair (4, 5)
    x[100] = 7.0                         # past rot_dim: unchanged
    q = _bf16_bits(x).reshape(1, 1, 128)
    cs = np.zeros((1, 32), np.float32)
    sn = np.zeros((1, 32), np.float32)
    cs[0, :3] = [0.0, -1.0, 0.0]         # pair 0: +90 degrees, pair 1: 180, pair 2: -90
    sn[0, :3] = [1.0, 0.0, -1.0]
    cs[0, 3:] = 1.0
    _, _, r = oracle.rope_quant_q(q, [0], cs, sn, 64)
    want = x.copy()
    want[0:2] = [0.0, 1.0]               # (1, 0) turned by 90 degrees
    want[2:4] = [-3.0, -4.0]             # (3, 4) turned by 180 degrees
    want[4:6] = [-1.0, -2.0]             # (2, -1) turned by -90 degrees
    assert np.array_equal(r[0], want)


def test_rope_matches_complex_multiplication(oracle):
    T, H = 6, 3
    q = wl.normal_bf16(wl.rng(12), (T, H, 128))
    cs, sn = _table(50, 64)
    pos = np.array([0, 7, 49, 3, 3, 20], np.int32)
    _, _, r = oracle.rope_quant_q(q, pos, cs, sn, 128)
    x = _bf16_vals(q).reshape(T, H, 128).astype(np.float64)
    z = (x[..., 0::2] + 1j * x[..., 1::2]) * (cs[pos] + 1j * sn[pos]).astype(np.complex128)[:, None, :]
    want = np.empty_like(x)
    want[..., 0::2], want[..., 1::2] = z.real, z.imag
    err = np.abs(r.reshape(T, H, 128) - want)
    # two fp32 roundings of products of magnitude <= |x| + |y|
    bound = 4 * 2.0 ** -24 * (np.abs(x[..., 0::2]) + np.abs(x[..., 1::2])).repeat(2, axis=-1)
    assert (err <= bound + 1e-30).all()


def test_rope_keeps_norms_and_scales_exactly(oracle):
    q = wl.normal_bf16(wl.rng(13), (1, 8, 128))
    cs, sn = _table(40, 64)
    _, _, r1 = oracle.rope_quant_q(q, [13], cs, sn, 128)
    x = _bf16_vals(q).reshape(8, 128).astype(np.float64)
    n0 = np.hypot(x[:, 0::2], x[:, 1::2])
    n1 = np.hypot(r1[:, 0::2].astype(np.float64), r1[:, 1::2].astype(np.float64))
    assert np.allclose(n0, n1, rtol=1e-6, atol=1e-30)
    # doubling the input doubles the rotated values exactly (power-of-two
    # scaling commutes with every fp32 rounding), and the quantised values
    # keep their codes with every scale byte one higher
    q2 = _bf16_bits(2.0 * _bf16_vals(q))
    v1, s1, _ = oracle.rope_quant_q(q, [13], cs, sn, 128)
    v2, s2, r2 = oracle.rope_quant_q(q2, [13], cs, sn, 128)
    assert np.array_equal(r2, 2.0 * r1)
    assert np.array_equal(v2, v1) and np.array_equal(s2.astype(int), s1.astype(int) + 1)


def test_quant_f32_matches_bf16_rule_and_hand_cases(oracle):
    # values that are bf16-exact quantise exactly as their bf16 bits do
    q = wl.normal_bf16(wl.rng(14), (40, 128))
    for row in q:
        v1, s1 = oracle.quant_vec128(row)
        v2, s2 = oracle.quant_vec128_f32(_bf16_vals(row))
        assert np.array_equal(v1, v2) and np.array_equal(s1, s2)
    # an fp32 value just above 6 (not a bf16 value) needs the next scale:
    # amax 6.0000005 -> 2^1 (byte 128); 6.0000005 / 2 = 3.00000024 -> code 5 (3.0)
    x = np.zeros(128, np.float32)
    x[0] = np.float32(6.0000005)
    x[1] = np.float32(-0.5)              # -0.25: halfway between 0 and 0.5 -> even code 0, sign kept
    x[2] = np.float32(-0.75)             # -0.375: nearer 0.5 -> code 1, sign kept
    v, s = oracle.quant_vec128_f32(x)
    assert s[0] == 128 and s[1] == 0
    assert v[0] == (0x5 | (0x8 << 4)) and (v[1] & 0xF) == 0x9


# ---------------------------------------------------------------- K-pool insert

def test_kpool_mask_rule_by_hand(oracle):
    """The passage's rule on small batches, worked by hand: rows p with a
    valid slot and p >= P - 1 are written at their slot; a valid slot at
    p < P - 1 belongs to a pool that began before the batch and is dropped;
    a batch shorter than one pool writes nothing."""
    P = 3
    k = wl.normal_bf16(wl.rng(15), (6, 128))
    gate = np.zeros((6, 128), np.float32)
    ape = np.zeros((P, 128), np.float32)
    slots = np.array([7, -1, 9, -1, -1, 11], np.int64)
    kc, mag = oracle.kpool_compress(k, gate, ape, slots, P)
    written = [p for p in range(6) if not np.isnan(kc[p, 0])]
    assert written == [2, 5]
    cache = wl.poisoned_cache(1)
    before = cache.copy()
    assert oracle.kpool_insert(kc.astype(np.float32), slots, P, cache) == 0
    # slot 7 (row 0) untouched; slots 9 and 11 written
    changed = {off for off in range(64) if not np.array_equal(cache[0, off * 64:off * 64 + 64],
                                                              before[0, off * 64:off * 64 + 64])}
    assert changed == {9, 11}
    short = np.array([0, 1], np.int64)
    kc2, _ = oracle.kpool_compress(k[:2], gate[:2], ape, short, P)
    assert np.isnan(kc2).all()
    cache2 = wl.poisoned_cache(1)
    oracle.kpool_insert(np.zeros((2, 128), np.float32), short, P, cache2)
    assert np.array_equal(cache2, wl.poisoned_cache(1))
    # out-of-range slots are skipped and counted
    bad = np.array([-1, -1, 64, -1, -1, 5], np.int64)
    kc3, _ = oracle.kpool_compress(k, gate, ape, bad, P)
    assert oracle.kpool_insert(kc3.astype(np.float32), bad, P, wl.poisoned_cache(1)) == 1


def test_kpool_uniform_gates_give_the_mean(oracle):
    P = 4
    k = wl.normal_bf16(wl.rng(16), (8, 128))
    slots = np.array([-1, -1, -1, 0, -1, -1, -1, 1], np.int64)
    kc, mag = oracle.kpool_compress(k, np.zeros((8, 128), np.float32),
                                    np.zeros((P, 128), np.float32), slots, P)
    x = _bf16_vals(k).astype(np.float64)
    assert np.allclose(kc[3], x[0:4].mean(axis=0), rtol=1e-15, atol=1e-300)
    assert np.allclose(kc[7], x[4:8].mean(axis=0), rtol=1e-15, atol=1e-300)
    assert np.allclose(mag[7], np.abs(x[4:8]).mean(axis=0), rtol=1e-15, atol=1e-300)


def test_kpool_one_hot_and_position_weights(oracle):
    P = 5
    k = wl.normal_bf16(wl.rng(17), (P, 128))
    x = _bf16_vals(k).astype(np.float64)
    slots = np.array([-1, -1, -1, -1, 3], np.int64)
    gate = np.zeros((P, 128), np.float32)
    gate[2, :] = 200.0                   # every other weight is e^-200 of it
    kc, _ = oracle.kpool_compress(k, gate, np.zeros((P, 128), np.float32), slots, P)
    assert np.allclose(kc[4], x[2], rtol=1e-80, atol=1e-300)
    # position-only weights: ape[j] = log(c_j) gives sum_j c_j k_j / sum_j c_j,
    # with the position index counted from the pool's first row
    c = np.array([1.0, 2.0, 4.0, 8.0, 16.0])
    ape = np.repeat(np.log(c).astype(np.float32)[:, None], 128, axis=1)
    kc, _ = oracle.kpool_compress(k, np.zeros((P, 128), np.float32), ape, slots, P)
    cw = np.exp(np.log(c).astype(np.float32).astype(np.float64))
    want = (cw[:, None] * x).sum(axis=0) / cw.sum()
    assert np.allclose(kc[4], want, rtol=1e-14, atol=1e-300)


def test_kpool_of_one_is_the_plain_insert(oracle):
    """With a pool of one token the softmax weight is 1: the pooled key is the
    key itself and the insert equals the plain quantise-and-insert."""
    n = 200
    k = wl.normal_bf16(wl.rng(18), (n, 128))
    g = wl.rng(19)
    slots = g.permutation(64 * 8)[:n].astype(np.int64)
    slots[g.choice(n, 30, replace=False)] = -1
    gate = g.standard_normal((n, 128)).astype(np.float32)
    ape = g.standard_normal((1, 128)).astype(np.float32)
    kc, _ = oracle.kpool_compress(k, gate, ape, slots, 1)
    ok = slots >= 0
    assert np.array_equal(kc[ok], _bf16_vals(k)[ok].astype(np.float64))
    c1 = wl.poisoned_cache(8)
    c2 = wl.poisoned_cache(8)
    oracle.kpool_insert(kc.astype(np.float32), slots, 1, c1)
    oracle.quant_insert(k, slots, c2)
    assert np.array_equal(c1, c2)


def test_kpool_equal_rows_and_magnitude(oracle):
    P = 6
    row = wl.normal_bf16(wl.rng(20), (1, 128))
    k = np.repeat(row, 10, axis=0)
    g = wl.rng(21)
    gate = (3 * g.standard_normal((10, 128))).astype(np.float32)
    ape = g.standard_normal((P, 128)).astype(np.float32)
    slots = np.arange(10, dtype=np.int64)
    kc, mag = oracle.kpool_compress(k, gate, ape, slots, P)
    x = _bf16_vals(row[0]).astype(np.float64)
    for p in range(P - 1, 10):
        assert np.allclose(kc[p], x, rtol=1e-14, atol=1e-300)
        assert np.allclose(mag[p], np.abs(x), rtol=1e-14, atol=1e-300)
    assert np.isnan(kc[:P - 1]).all()
