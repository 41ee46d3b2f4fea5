"""Pins for the oracle's logits, windows, gather and top-k.

The logits are checked on cases whose value is fixed by hand or by integer
arithmetic (all scales 2^0 with codes in {0, +-1}, one nonzero per block with
distinct block scales, one head per known dot product, all dots <= 0), by the
invariant that the paged path and the gathered contiguous path agree, and by
invariance under relocating cache pages.  Top-k is checked against Python's
sorted() on tiny rows."""
import math

import numpy as np
import pytest

from sparse_attention_indexer_quant_gb300 import workloads as wl

ONE, MINUS_ONE = 0x2, 0xA          # E2M1 codes of +1.0 and -1.0


def pack(codes):
    codes = np.asarray(codes, np.uint8).reshape(-1, 128)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def sign_codes(g, shape, p_zero=0.3):
    s = g.integers(0, 3, size=shape)            # 0 -> 0, 1 -> +1, 2 -> -1
    s[g.random(shape) < p_zero] = 0
    codes = np.where(s == 1, ONE, np.where(s == 2, MINUS_ONE, 0)).astype(np.uint8)
    vals = np.where(s == 1, 1, np.where(s == 2, -1, 0)).astype(np.int64)
    return codes, vals


def test_logits_integer_case(oracle):
    """Scales 127 (2^0) and codes in {0, +1, -1}: every dot product is an
    integer; the logit is sum_h w_h * max(dot_h, 0) and the magnitude is
    sum_h |w_h| * #(positions where both are nonzero)."""
    g = wl.rng(21)
    T, H, S = 3, 5, 40
    qc, qi = sign_codes(g, (T, H, 128))
    kc, ki = sign_codes(g, (S, 128))
    w = g.standard_normal((T, H)).astype(np.float32)
    qv, qs = pack(qc.reshape(-1, 128)), np.full((T * H, 4), 127, np.uint8)
    kv, ks = pack(kc), np.full((S, 4), 127, np.uint8)
    start = np.array([0, 7, 39], np.int32)
    end = np.array([40, 20, 40], np.int32)
    lg, mag = oracle.mqa_logits(qv, qs, H, kv, ks, w, start, end)
    for t in range(T):
        for s in range(S):
            if not (start[t] <= s < end[t]):
                assert math.isnan(lg[t, s])
                continue
            dots = qi[t] @ ki[s]                         # [H] integers
            both = (qi[t] != 0) & (ki[s] != 0)
            want = math.fsum(float(w[t, h]) * max(int(dots[h]), 0) for h in range(H))
            want_mag = math.fsum(abs(float(w[t, h])) * int(both[h].sum()) for h in range(H))
            assert lg[t, s] == pytest.approx(want, rel=1e-12, abs=1e-12)
            assert mag[t, s] == pytest.approx(want_mag, rel=1e-12)


def test_logits_block_scales(oracle):
    """One nonzero element per block with a different scale byte in every
    block of q and k: dot = sum_b v_q,b * v_k,b * 2^(sq_b-127) * 2^(sk_b-127).
    k also carries a nonzero at a position where q is zero, which must add
    nothing."""
    qcodes = np.zeros(128, np.uint8)
    kcodes = np.zeros(128, np.uint8)
    pos = [3, 40, 77, 126]
    qc = [0x7, 0x3, 0xC, 0x1]       # 6, 1.5, -2, 0.5
    kc = [0x5, 0xE, 0x6, 0x4]       # 3, -4, 4, 2
    for b in range(4):
        qcodes[pos[b]] = qc[b]
        kcodes[pos[b]] = kc[b]
    kcodes[10] = 0x7                # q is zero there
    qs = np.array([[127, 130, 120, 140]], np.uint8)
    ks = np.array([[125, 127, 131, 100]], np.uint8)
    vq = [6, 1.5, -2, 0.5]
    vk = [3, -4, 4, 2]
    dot = sum(vq[b] * vk[b] * 2.0 ** (int(qs[0, b]) - 127 + int(ks[0, b]) - 127) for b in range(4))
    adot = sum(abs(vq[b] * vk[b]) * 2.0 ** (int(qs[0, b]) - 127 + int(ks[0, b]) - 127)
               for b in range(4))
    w = np.array([[0.75]], np.float32)
    lg, mag = oracle.mqa_logits(pack(qcodes), qs, 1, pack(kcodes), ks, w,
                                np.array([0], np.int32), np.array([1], np.int32))
    assert dot != 0
    assert lg[0, 0] == 0.75 * max(dot, 0.0)
    assert mag[0, 0] == 0.75 * adot
    # flip the sign of q in the largest block: the ReLU now cuts the sum
    qcodes2 = qcodes.copy()
    qcodes2[pos[1]] ^= 0x8
    dot2 = dot - 2 * vq[1] * vk[1] * 2.0 ** (int(qs[0, 1]) - 127 + int(ks[0, 1]) - 127)
    lg2, _ = oracle.mqa_logits(pack(qcodes2), qs, 1, pack(kcodes), ks, w,
                               np.array([0], np.int32), np.array([1], np.int32))
    assert lg2[0, 0] == 0.75 * max(dot2, 0.0)


def test_logits_heads_and_weights(oracle):
    """Head h of q equals the first d_h positions of k (all +1): dot_h = d_h if
    positive, else the negated pattern gives -d_h.  logit = sum over heads
    with positive dot of w_h * d_h."""
    H = 8
    d = [5, 0, 17, 3, 64, 1, 9, 2]
    sgn = [1, 1, -1, 1, 1, -1, 1, -1]
    w = np.array([[0.5, -1.0, 2.0, -0.25, 0.125, 4.0, -3.0, 1.5]], np.float32)
    k = np.zeros(128, np.uint8)
    k[:64] = ONE
    q = np.zeros((H, 128), np.uint8)
    for h in range(H):
        q[h, :d[h]] = ONE if sgn[h] > 0 else MINUS_ONE
    lg, mag = oracle.mqa_logits(pack(q), np.full((H, 4), 127, np.uint8), H, pack(k),
                                np.full((1, 4), 127, np.uint8), w,
                                np.array([0], np.int32), np.array([1], np.int32))
    want = sum(float(w[0, h]) * d[h] for h in range(H) if sgn[h] > 0)
    assert lg[0, 0] == pytest.approx(want, rel=1e-15)
    assert mag[0, 0] == pytest.approx(sum(abs(float(w[0, h])) * d[h] for h in range(H)), rel=1e-15)


def test_logits_all_dots_nonpositive(oracle):
    """w >= 0, every k element >= 0 and every q element <= 0: every dot is
    <= 0, so every logit is exactly 0 while the magnitudes are not."""
    g = wl.rng(23)
    S, H = 16, 4
    kv, ks = oracle.quant_q(wl.normal_bf16(g, (S, 128)))
    qv, qs = oracle.quant_q(wl.normal_bf16(g, (H, 128)))
    kv = kv & np.uint8(0x77)          # clear both sign bits: all k >= 0
    qv = qv | np.uint8(0x88)          # set both sign bits: all q <= 0
    w = np.abs(g.standard_normal((1, H))).astype(np.float32)
    lg, mag = oracle.mqa_logits(qv, qs, H, kv, ks, w, np.array([0], np.int32),
                                np.array([S], np.int32))
    assert (lg[0] == 0.0).all()
    assert (mag[0] > 0.0).all()


def _small_decode(seed, lens, H, next_n):
    p = wl.make_decode("t", seed, lens, H, next_n)
    return p


def _insert_all(oracle, p):
    cache = wl.poisoned_cache(p.num_blocks)
    assert oracle.quant_insert(p.k, p.slots, cache) == 0
    return cache


def test_paged_equals_gathered_contiguous(oracle):
    """Paged decode logits through a shuffled block table equal the prefill
    logits on the gathered contiguous keys with the same windows."""
    p = _small_decode(31, [1, 130, 300, 64], H=4, next_n=2)
    cache = _insert_all(oracle, p)
    qv, qs = oracle.quant_q(p.q)
    ld = 320
    lg, mag = oracle.paged_mqa_logits(qv, qs, p.B, p.next_n, p.H, cache, p.block_table,
                                      p.context_lens, p.weights, ld)
    offs = np.concatenate([[0], np.cumsum(p.context_lens)]).astype(np.int64)
    kv, ks = oracle.gather_k(cache, p.block_table, p.context_lens, offs[:-1], int(offs[-1]))
    st, en = p.row_windows()
    b_of = np.repeat(np.arange(p.B), p.next_n)
    lg2, mag2 = oracle.mqa_logits(qv, qs, p.H, kv, ks, p.weights, (st + offs[b_of]).astype(np.int32),
                                  (en + offs[b_of]).astype(np.int32))
    for r in range(p.rows):
        b = b_of[r]
        n = en[r]
        assert np.array_equal(lg[r, :n], lg2[r, offs[b]:offs[b] + n])
        assert np.array_equal(mag[r, :n], mag2[r, offs[b]:offs[b] + n])
        assert np.isnan(lg[r, n:]).all()


def test_paged_windows(oracle):
    """Row (b, j) sees positions [0, L_b - next_n + j]."""
    p = _small_decode(37, [5, 70], H=2, next_n=2)
    cache = _insert_all(oracle, p)
    qv, qs = oracle.quant_q(p.q)
    lg, _ = oracle.paged_mqa_logits(qv, qs, p.B, 2, p.H, cache, p.block_table, p.context_lens,
                                    p.weights, 80)
    valid = ~np.isnan(lg)
    assert [int(valid[r].sum()) for r in range(4)] == [4, 5, 69, 70]
    assert all(valid[r, :int(valid[r].sum())].all() for r in range(4))


def test_page_relocation_invariance(oracle):
    """Moving every page to another block id (and rewriting the table to
    match) leaves the logits unchanged."""
    p = _small_decode(41, [200, 129], H=3, next_n=1)
    cache = _insert_all(oracle, p)
    qv, qs = oracle.quant_q(p.q)
    a, _ = oracle.paged_mqa_logits(qv, qs, p.B, 1, p.H, cache, p.block_table, p.context_lens,
                                   p.weights, 200)
    perm = wl.rng(2).permutation(p.num_blocks).astype(np.int32)
    cache2 = np.empty_like(cache)
    cache2[perm] = cache
    bt2 = np.where(p.block_table >= 0, perm[np.maximum(p.block_table, 0)], -1).astype(np.int32)
    b, _ = oracle.paged_mqa_logits(qv, qs, p.B, 1, p.H, cache2, bt2, p.context_lens, p.weights, 200)
    assert np.array_equal(a, b, equal_nan=True)


def test_gather_matches_direct_quant(oracle):
    p = _small_decode(43, [65, 3, 128], H=1, next_n=1)
    cache = _insert_all(oracle, p)
    offs = np.array([0, 65, 68], np.int64)
    kv, ks = oracle.gather_k(cache, p.block_table, p.context_lens, offs, 196)
    dv, ds = oracle.quant_q(p.k)
    assert np.array_equal(kv, dv) and np.array_equal(ks, ds)


@pytest.mark.parametrize("k", [1, 16, 2048])
def test_topk_brute_force(oracle, k):
    g = wl.rng(100 + k)
    lens = [0, 1, 5, k - 1, k, k + 1, 3 * k + 7]
    starts = [0, 3, 11, 0, 2, 5, 1]
    ld = max(s + n for s, n in zip(starts, lens)) + 4
    rows = len(lens)
    logits = np.full((rows, ld), np.nan)
    for r in range(rows):
        # few distinct values so that ties are common
        logits[r, starts[r]:starts[r] + lens[r]] = g.integers(-4, 5, size=lens[r]) * 0.5
    st = np.array(starts, np.int32)
    en = (st + np.array(lens)).astype(np.int32)
    out = oracle.topk_rows(logits, st, en, k)
    for r in range(rows):
        vals = logits[r, starts[r]:starts[r] + lens[r]]
        order = sorted(range(lens[r]), key=lambda i: (-vals[i], i))[:k]
        want = order + [-1] * (k - len(order))
        assert out[r].tolist() == want


def test_topk_uses_only_window(oracle):
    """Values outside [start, end) never enter, even when larger."""
    logits = np.array([[100.0, 1.0, 2.0, 3.0, 100.0]])
    out = oracle.topk_rows(logits, np.array([1], np.int32), np.array([4], np.int32), 2)
    assert out[0].tolist() == [2, 1]
