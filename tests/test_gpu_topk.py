"""GPU parity of top-k per row against the oracle through the C ABI: ragged
rows around k, rows with ties and all-equal rows, window offsets, k below
2048, and the prefill-shaped causal case."""
import numpy as np
import pytest
import torch

from sparse_attention_indexer_quant_gb300 import workloads as wl
from idx_testutil import check_topk, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def idx():
    from sparse_attention_indexer_quant_gb300 import binding
    binding.check_device(torch.cuda.current_device())
    return binding


def run(idx, logits32, starts, ends, k):
    out = idx.topk_rows(dev(logits32), dev(ends.astype(np.int32)), k,
                        row_start=dev(starts.astype(np.int32)))
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("k", [2048, 16, 1])
def test_topk_random_rows(idx, k):
    g = wl.rng(400 + k)
    lens = np.array([0, 1, 5, k - 1 if k > 1 else 0, k, k + 1, 2 * k + 3, 5000, 40000, 131072])
    starts = g.integers(0, 50, size=len(lens))
    ld = int((starts + lens).max()) + 7
    logits = np.full((len(lens), ld), np.nan, np.float32)
    for r, (s, n) in enumerate(zip(starts, lens)):
        logits[r, s:s + n] = g.standard_normal(n).astype(np.float32)
    out = run(idx, logits, starts, starts + lens, k)
    for r, (s, n) in enumerate(zip(starts, lens)):
        vals = logits[r, s:s + n].astype(np.float64)
        check_topk(out[r], vals, np.zeros_like(vals), int(n), k, f"row {r} len {n}")


def test_topk_ties(idx):
    """Few distinct values: the selected set must hold every index above the
    k-th value and fill the rest with indices equal to it."""
    g = wl.rng(410)
    k = 2048
    lens = np.array([3000, 10000, 70000])
    ld = int(lens.max())
    logits = np.full((3, ld), np.nan, np.float32)
    for r, n in enumerate(lens):
        logits[r, :n] = (g.integers(-3, 4, size=n) * 0.5).astype(np.float32)
    out = run(idx, logits, np.zeros(3, np.int64), lens, k)
    for r, n in enumerate(lens):
        vals = logits[r, :n].astype(np.float64)
        check_topk(out[r], vals, np.zeros_like(vals), int(n), k, f"ties row {r}")


def test_topk_all_equal_and_neg_inf(idx):
    k = 2048
    n = 20000
    logits = np.zeros((3, n), np.float32)
    logits[1, :] = -np.inf
    logits[1, 123] = 5.0
    logits[2, :] = 1.0
    logits[2, 5000:5010] = 2.0
    out = run(idx, logits, np.zeros(3, np.int64), np.full(3, n), k)
    for r in range(3):
        vals = logits[r].astype(np.float64)
        check_topk(out[r], vals, np.zeros_like(vals), n, k, f"row {r}")
    assert 123 in out[1].tolist()
    assert set(range(5000, 5010)) <= set(out[2].tolist())


def test_topk_causal_prefill_rows(idx):
    """Rows of a causal prefill: row t sees [0, t+1)."""
    g = wl.rng(420)
    T = 3000
    logits = g.standard_normal((T, T)).astype(np.float32)
    ends = np.arange(1, T + 1)
    out = run(idx, logits, np.zeros(T, np.int64), ends, 2048)
    for t in [0, 1, 2046, 2047, 2048, 2049, 2999]:
        vals = logits[t, :t + 1].astype(np.float64)
        check_topk(out[t], vals, np.zeros_like(vals), t + 1, 2048, f"t={t}")


@pytest.mark.parametrize("n,finite", [(20000, 1000), (9000, 100), (131072, 1500)])
def test_topk_rows_mostly_neg_inf(idx, n, finite):
    """Rows whose k-th largest value is -inf, long enough to be split over
    several CTAs, with unaligned window starts: every index must be distinct,
    inside the window, and cover all finite values."""
    g = wl.rng(430 + n)
    k = 2048
    rows = 3
    starts = np.array([0, 1, 3])
    ld = n + 8
    logits = np.full((rows, ld), np.nan, np.float32)
    for r in range(rows):
        row = np.full(n, -np.inf, np.float32)
        pos = g.choice(n, size=finite, replace=False)
        row[pos] = g.standard_normal(finite).astype(np.float32)
        logits[r, starts[r]:starts[r] + n] = row
    out = run(idx, logits, starts, starts + n, k)
    for r in range(rows):
        vals = logits[r, starts[r]:starts[r] + n].astype(np.float64)
        check_topk(out[r], vals, np.zeros_like(vals), n, k, f"row {r}")
        assert len(set(out[r].tolist())) == k
        if finite <= k:
            assert set(np.nonzero(np.isfinite(vals))[0].tolist()) <= set(out[r].tolist())


def test_topk_many_rows_long_tied_and_unaligned(idx):
    """More rows than SMs take the one-CTA-per-row kernel: long rows streamed
    in several rounds (aligned starts), long rows staged in several chunks
    (unaligned starts), rows whose boundary bin overflows the candidate list
    (few distinct values, all equal), rows whose k-th value is -inf."""
    g = wl.rng(440)
    k = 2048
    special = [(0, 20000, "rand"), (1, 70000, "rand"), (0, 30000, "ties"), (0, 10000, "equal"),
               (2, 20000, "neginf"), (0, 20000, "neginf"), (3, 4097, "rand"), (0, 8193, "rand"),
               (5, 2049, "rand"), (0, 0, "rand"), (0, 1, "rand"), (1, 9000, "ties3")]
    n_rows = 200
    starts = np.zeros(n_rows, np.int64)
    lens = g.integers(100, 3000, size=n_rows)
    for r, (s, n, _) in enumerate(special):
        starts[r], lens[r] = s, n
    ld = int((starts + lens).max()) + 12
    ld += (-ld) % 4
    logits = np.full((n_rows, ld), np.nan, np.float32)
    for r in range(n_rows):
        s, n = int(starts[r]), int(lens[r])
        kind = special[r][2] if r < len(special) else "rand"
        if kind == "rand":
            row = g.standard_normal(n).astype(np.float32)
        elif kind == "ties":
            row = (g.integers(-3, 4, size=n) * 0.5).astype(np.float32)
        elif kind == "ties3":
            row = g.choice(np.array([-1.0, 0.25, 2.0], np.float32), size=n)
        elif kind == "equal":
            row = np.full(n, 0.75, np.float32)
        else:
            row = np.full(n, -np.inf, np.float32)
            pos = g.choice(n, size=1000, replace=False)
            row[pos] = g.standard_normal(1000).astype(np.float32)
        logits[r, s:s + n] = row
    out = run(idx, logits, starts, starts + lens, k)
    for r in list(range(len(special))) + [50, 199]:
        s, n = int(starts[r]), int(lens[r])
        vals = logits[r, s:s + n].astype(np.float64)
        check_topk(out[r], vals, np.zeros_like(vals), n, k, f"row {r} len {n} start {s}")


def test_topk_many_rows_patterned_positions(idx):
    """Rows whose largest values sit in a regular pattern of positions (more
    rows than SMs, so the one-CTA-per-row kernel runs): large values only in
    the first 128 of every 2048 positions, small values only there, a rising
    row, one 2048-block holding the whole top k, and rows of 2 k to 3 k
    elements.  A select that estimated its threshold from a strided sample of
    the row would misjudge exactly these."""
    g = wl.rng(450)
    k = 2048
    n_rows = 200
    kinds = ["high", "low", "rising", "block", "short", "short2"] * 4
    lens = g.integers(2000, 40000, size=n_rows)
    ld = int(lens.max())
    ld += (-ld) % 4
    logits = np.full((n_rows, ld), np.nan, np.float32)
    for r in range(n_rows):
        kind = kinds[r] if r < len(kinds) else "rand"
        n = int(lens[r])
        if kind in ("short", "short2"):
            n = lens[r] = 2 * k + 50 if kind == "short" else 3 * k - 7
        row = g.standard_normal(n).astype(np.float32)
        seen = (np.arange(n) % 2048) < 128
        if kind == "high":
            row[seen] += 10.0
        elif kind == "low":
            row[seen] -= 10.0
        elif kind == "rising":
            row = np.arange(n, dtype=np.float32) / 7.0
        elif kind == "block":
            b = 2048 * int(g.integers(0, n // 2048))
            row[b:b + 2048] += 20.0
        logits[r, :n] = row
    out = run(idx, logits, np.zeros(n_rows, np.int64), lens, k)
    for r in list(range(len(kinds))) + [100, 199]:
        n = int(lens[r])
        vals = logits[r, :n].astype(np.float64)
        kind = kinds[r] if r < len(kinds) else "rand"
        check_topk(out[r], vals, np.zeros_like(vals), n, k, f"row {r} ({kind}) len {n}")
