"""GPU parity of the fused paged logits + top-k against the oracle through the
C ABI: windows around k and around the per-CTA chunk size, both head counts
and query-token counts, degenerate all-equal rows, and sampled rows of the
full-size decode workloads."""
import numpy as np
import pytest
import torch

from sparse_attention_indexer_quant_gb300 import workloads as wl
from idx_testutil import check_topk, dev, dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def idx():
    from sparse_attention_indexer_quant_gb300 import binding
    binding.check_device(torch.cuda.current_device())
    return binding


def run_fused(idx, p, k, cache=None, qv=None, qs=None, weights=None):
    if cache is None:
        cache = dev(wl.poisoned_cache(p.num_blocks))
        idx.quant_insert(dev_bf16(p.k), dev(p.slots), cache)
    if qv is None:
        qv, qs = idx.quant_q(dev_bf16(p.q))
    w = dev(p.weights if weights is None else weights)
    errs = idx.new_errors()
    out = idx.paged_logits_topk(qv, qs, w, cache, dev(p.block_table), dev(p.context_lens),
                                p.next_n, p.H, k, errors=errs)
    torch.cuda.synchronize()
    assert errs.cpu().tolist() == [0, 0]
    return out.cpu().numpy()


def oracle_rows(oracle, p, seqs, weights=None, qbits=None):
    """Oracle logits + magnitudes for the listed sequences, from their own
    bf16 keys and queries."""
    res = {}
    for b in seqs:
        lo, hi = int(p.tok_offsets[b]), int(p.tok_offsets[b + 1])
        L = hi - lo
        ocache = wl.poisoned_cache(p.num_blocks)
        oracle.quant_insert(p.k[lo:hi], p.slots[lo:hi], ocache)
        rows = slice(b * p.next_n, (b + 1) * p.next_n)
        q = p.q if qbits is None else qbits
        oqv, oqs = oracle.quant_q(q[rows])
        w = (p.weights if weights is None else weights)[rows]
        ol, om = oracle.paged_mqa_logits(oqv, oqs, 1, p.next_n, p.H, ocache, p.block_table[b:b + 1],
                                         np.array([L], np.int32), w, max(L, 1))
        res[b] = (ol, om, L)
    return res


LENS = [1, 2, 100, 2047, 2048, 2049, 4095, 4096, 4097, 8191, 8192, 8193, 20000]


@pytest.mark.parametrize("H,next_n", [(32, 1), (32, 2), (64, 1), (64, 2)])
def test_fused_parity(idx, oracle, H, next_n):
    p = wl.make_decode("t", 500 + H + next_n, LENS, H, next_n)
    k = 2048
    g = run_fused(idx, p, k)
    ref = oracle_rows(oracle, p, range(p.B))
    for b, (ol, om, L) in ref.items():
        for j in range(next_n):
            n = max(L - next_n + j + 1, 0)
            r = b * next_n + j
            check_topk(g[r], ol[j, :n], om[j, :n], n, k, f"seq {b} (L={L}) row {j}")


@pytest.mark.parametrize("k", [1, 64, 777])
def test_fused_small_k(idx, oracle, k):
    p = wl.make_decode("t", 520 + k, [5, 900, 9000], 32, 1)
    g = run_fused(idx, p, k)
    for b, (ol, om, L) in oracle_rows(oracle, p, range(p.B)).items():
        check_topk(g[b], ol[0, :L], om[0, :L], L, k, f"seq {b}")


def test_fused_all_equal_logits(idx, oracle):
    """Weights >= 0 and every query element <= 0 against keys >= 0 would need
    crafted bits; instead zero weights make every logit exactly 0, so any k
    distinct in-window indices are right."""
    p = wl.make_decode("t", 530, [10000, 3000], 32, 1)
    zeros = np.zeros_like(p.weights)
    g = run_fused(idx, p, 2048, weights=zeros)
    for b, L in enumerate(p.context_lens):
        sel = g[b, :2048]
        assert len(np.unique(sel)) == 2048 and sel.min() >= 0 and sel.max() < L


def test_fused_matches_unfused_path(idx, oracle):
    """Fused result and unfused logits + top_k_per_row both satisfy the oracle
    rule on the same inputs."""
    p = wl.make_decode("t", 540, [3000, 17000, 40000], 64, 2)
    cache = dev(wl.poisoned_cache(p.num_blocks))
    idx.quant_insert(dev_bf16(p.k), dev(p.slots), cache)
    qv, qs = idx.quant_q(dev_bf16(p.q))
    g = run_fused(idx, p, 2048, cache=cache, qv=qv, qs=qs)
    lg = idx.paged_mqa_logits(qv, qs, dev(p.weights), cache, dev(p.block_table),
                              dev(p.context_lens), 2, 64, clean=True)
    st, en = p.row_windows()
    u = idx.topk_rows(lg, dev(en), 2048, row_start=dev(st))
    torch.cuda.synchronize()
    u = u.cpu().numpy()
    for b, (ol, om, L) in oracle_rows(oracle, p, range(p.B)).items():
        for j in range(2):
            n = L - 2 + j + 1
            check_topk(g[b * 2 + j], ol[j, :n], om[j, :n], n, 2048, f"fused seq {b} row {j}")
            check_topk(u[b * 2 + j], ol[j, :n], om[j, :n], n, 2048, f"unfused seq {b} row {j}")


def test_fused_full_size_batched_decode_sampled(idx, oracle):
    p = wl.batched_decode()
    g = run_fused(idx, p, 2048)
    for b, (ol, om, L) in oracle_rows(oracle, p, [0, 17, 63]).items():
        check_topk(g[b], ol[0, :L], om[0, :L], L, 2048, f"seq {b}")


def test_fused_full_size_long_decode_sampled(idx, oracle):
    p = wl.long_decode()
    g = run_fused(idx, p, 2048)
    for b, (ol, om, L) in oracle_rows(oracle, p, [9]).items():
        for j in range(2):
            n = L - 2 + j + 1
            check_topk(g[b * 2 + j], ol[j, :n], om[j, :n], n, 2048, f"seq {b} row {j}")


def test_fused_workspace_too_small(idx):
    p = wl.make_decode("t", 550, [500], 32, 1)
    cache = dev(wl.poisoned_cache(p.num_blocks))
    qv, qs = idx.quant_q(dev_bf16(p.q))
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(idx.IdxError) as e:
        idx.paged_logits_topk(qv, qs, dev(p.weights), cache, dev(p.block_table),
                              dev(p.context_lens), 1, 32, 2048, workspace=ws)
    assert e.value.status == 3


def test_fused_more_sequences_than_the_length_cache(idx, oracle):
    """Past 1024 sequences the scoring pass hands out work items through its
    counter instead of equal tile shares: the same result rule holds."""
    rng = np.random.default_rng(914)
    lens = [int(x) for x in rng.integers(1, 1200, size=1030)]
    lens[0], lens[1029] = 4100, 2049
    p = wl.make_decode("t", 914, lens, 32, 1)
    g = run_fused(idx, p, 2048)
    for b, (ol, om, L) in oracle_rows(oracle, p, [0, 517, 1024, 1029]).items():
        check_topk(g[b], ol[0, :L], om[0, :L], L, 2048, f"seq {b}")


def test_fused_workspace_garbage_and_reuse(idx, oracle):
    """The workspace needs no initialisation and may be shared by calls of
    different shapes: the work-item counter starts from whatever the scratch
    holds (random bytes here, with a counter value close to carrying into its
    generation bits) and from the previous call's value."""
    probs = [wl.make_decode("a", 921, [4100, 9000, 300, 20000], 32, 1),
             wl.make_decode("b", 922, [8193, 50, 16000], 32, 2)]
    need = max(idx.paged_logits_topk_workspace_bytes(p.B, p.next_n, p.block_table.shape[1], 2048)
               for p in probs)
    ws = torch.randint(0, 256, (need,), dtype=torch.uint8, device="cuda")
    ws[:8] = torch.tensor(np.array([(0xABCDE12345 << 24) | 0xFFFFF0], np.uint64).view(np.uint8),
                          device="cuda")
    state = []
    for p in probs:
        cache = dev(wl.poisoned_cache(p.num_blocks))
        idx.quant_insert(dev_bf16(p.k), dev(p.slots), cache)
        qv, qs = idx.quant_q(dev_bf16(p.q))
        state.append((p, cache, qv, qs, oracle_rows(oracle, p, range(p.B))))
    for p, cache, qv, qs, ref in state + state[:1]:
        errs = idx.new_errors()
        out = idx.paged_logits_topk(qv, qs, dev(p.weights), cache, dev(p.block_table),
                                    dev(p.context_lens), p.next_n, p.H, 2048, workspace=ws,
                                    errors=errs)
        torch.cuda.synchronize()
        assert errs.cpu().tolist() == [0, 0]
        g = out.cpu().numpy()
        for b, (ol, om, L) in ref.items():
            for j in range(p.next_n):
                n = max(L - p.next_n + j + 1, 0)
                check_topk(g[b * p.next_n + j], ol[j, :n], om[j, :n], n, 2048,
                           f"{p.name} seq {b} row {j}")


def test_fused_more_sequences_than_ctas(idx, oracle):
    """With more sequences than persistent CTAs some sequences get no CTA's
    first work item and are reached only through the counter; zero-length and
    long sequences mixed."""
    rng = np.random.default_rng(931)
    lens = [int(x) for x in rng.integers(0, 3000, size=500)]
    for b, L in [(0, 0), (3, 20000), (455, 9000), (456, 12345), (457, 0), (499, 31000)]:
        lens[b] = L
    p = wl.make_decode("t", 931, lens, 32, 1)
    g = run_fused(idx, p, 2048)
    for b, (ol, om, L) in oracle_rows(oracle, p, [0, 1, 3, 200, 455, 456, 457, 498, 499]).items():
        check_topk(g[b], ol[0, :L], om[0, :L], L, 2048, f"seq {b}")


@pytest.mark.parametrize("B,next_n", [(100, 1), (48, 2)])
def test_fused_two_select_waves_longest_first(idx, oracle, B, next_n):
    """More query rows than half the SMs: the select runs two-CTA clusters in
    two waves, each cluster taking the sequences in order of decreasing length.
    Every row is checked, with equal lengths (the order breaks ties by index),
    empty rows and rows at k."""
    rng = np.random.default_rng(4242 + B)
    lens = [int(x) for x in rng.integers(0, 6000, size=B)]
    for b, L in [(0, 3000), (1, 3000), (2, 3000), (3, 3000), (4, 0), (5, 0), (6, 2048),
                 (7, 2050), (8, 9000), (9, 9000), (B - 1, 3000)]:
        lens[b] = L
    p = wl.make_decode("two_waves", 4242 + B, lens, 32, next_n)
    assert p.rows > 76 and p.block_table.shape[1] * 64 >= 8192
    g = run_fused(idx, p, 2048)
    for b, (ol, om, L) in oracle_rows(oracle, p, range(B)).items():
        for j in range(next_n):
            n = max(L - next_n + j + 1, 0)
            check_topk(g[b * next_n + j], ol[j, :n], om[j, :n], n, 2048,
                       f"seq {b} (L={L}) row {j}")
