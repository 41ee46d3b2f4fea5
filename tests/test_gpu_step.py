"""GPU parity, through the C ABI, of the two-launch decode step: the scoring
launch inserts the step's new keys and quantises its query heads before it
scores, then the select runs.  The whole cache is compared byte for byte with
the oracle's (the oracle inserts every key of every sequence), and the top-k
of every checked row against the oracle's logits under the tolerance rule;
the 8K single-sequence decode and the 64-sequence batched decode run at full
size, as do CUDA-graph replays of a captured step."""
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


def _setup(idx, p):
    """Device state before the step: the cache holds every key except the
    step's new ones (whose slots stay poisoned)."""
    new = p.new_token_rows()
    old = np.ones(p.total_tokens, bool)
    old[new] = False
    cache = dev(wl.poisoned_cache(p.num_blocks))
    rows = np.nonzero(old)[0]
    for lo in range(0, len(rows), 1 << 21):
        r = rows[lo:lo + (1 << 21)]
        idx.quant_insert(dev_bf16(p.k[r]), dev(p.slots[r]), cache)
    return cache, dev_bf16(p.k[new]), dev_bf16(p.q)


def _oracle(oracle, p, seqs=None):
    ocache = wl.poisoned_cache(p.num_blocks)
    for lo in range(0, p.total_tokens, 1 << 21):
        hi = min(p.total_tokens, lo + (1 << 21))
        oracle.quant_insert(p.k[lo:hi], p.slots[lo:hi], ocache)
    res = {}
    for b in (range(p.B) if seqs is None else seqs):
        L = int(p.context_lens[b])
        rows = slice(b * p.next_n, (b + 1) * p.next_n)
        oqv, oqs = oracle.quant_q(p.q[rows])
        ol, om = oracle.paged_mqa_logits(oqv, oqs, 1, p.next_n, p.H, ocache,
                                         p.block_table[b:b + 1], p.context_lens[b:b + 1],
                                         p.weights[rows], max(L, 1))
        res[b] = (ol, om, L)
    return ocache, res


def _check(p, g, res, k=2048):
    for b, (ol, om, L) in res.items():
        for j in range(p.next_n):
            n = max(L - p.next_n + j + 1, 0)
            check_topk(g[b * p.next_n + j], ol[j, :n], om[j, :n], n, k, f"seq {b} (L={L}) row {j}")


LENS = [1, 2, 100, 2047, 2048, 2049, 4097, 8193, 20000]


@pytest.mark.parametrize("H,next_n", [(32, 1), (32, 2), (64, 1), (64, 2)])
def test_step_parity(idx, oracle, H, next_n):
    p = wl.make_decode("t", 8000 + H + next_n, [max(L, next_n) for L in LENS], H, next_n)
    cache, k_new, q = _setup(idx, p)
    errs = idx.new_errors()
    out = idx.paged_decode_step(k_new, q, dev(p.weights), cache, dev(p.block_table),
                                dev(p.context_lens), next_n, H, 2048, errors=errs)
    torch.cuda.synchronize()
    assert errs.cpu().tolist() == [0, 0]
    ocache, res = _oracle(oracle, p)
    assert np.array_equal(cache.cpu().numpy(), ocache), "cache bytes differ from the oracle"
    _check(p, out.cpu().numpy(), res)


def test_step_single_sequence_8k(idx, oracle):
    p = wl.pr_ref()
    cache, k_new, q = _setup(idx, p)
    errs = idx.new_errors()
    out = idx.paged_decode_step(k_new, q, dev(p.weights), cache, dev(p.block_table),
                                dev(p.context_lens), 1, p.H, 2048, errors=errs)
    torch.cuda.synchronize()
    assert errs.cpu().tolist() == [0, 0]
    ocache, res = _oracle(oracle, p)
    assert np.array_equal(cache.cpu().numpy(), ocache)
    _check(p, out.cpu().numpy(), res)


def test_step_batched_decode_full_size(idx, oracle):
    p = wl.batched_decode()
    cache, k_new, q = _setup(idx, p)
    errs = idx.new_errors()
    out = idx.paged_decode_step(k_new, q, dev(p.weights), cache, dev(p.block_table),
                                dev(p.context_lens), 1, p.H, 2048, errors=errs)
    torch.cuda.synchronize()
    assert errs.cpu().tolist() == [0, 0]
    ocache, res = _oracle(oracle, p, [0, 17, 40, 63])
    assert np.array_equal(cache.cpu().numpy(), ocache)
    _check(p, out.cpu().numpy(), res)


def test_step_more_sequences_than_ctas(idx, oracle):
    rng = np.random.default_rng(8100)
    lens = [int(x) for x in rng.integers(1, 3000, size=700)]
    lens[5], lens[699] = 20000, 9000
    p = wl.make_decode("t", 8100, lens, 32, 1)
    cache, k_new, q = _setup(idx, p)
    errs = idx.new_errors()
    out = idx.paged_decode_step(k_new, q, dev(p.weights), cache, dev(p.block_table),
                                dev(p.context_lens), 1, 32, 2048, errors=errs)
    torch.cuda.synchronize()
    assert errs.cpu().tolist() == [0, 0]
    ocache, res = _oracle(oracle, p, [0, 5, 333, 698, 699])
    assert np.array_equal(cache.cpu().numpy(), ocache)
    _check(p, out.cpu().numpy(), res)


def test_step_graph_replays(idx, oracle):
    """A captured step replayed: every replay inserts the same keys again and
    gives the same top-k (the barrier and work counters start over)."""
    p = wl.make_decode("t", 8200, [5000, 12000, 300, 9000], 32, 2)
    cache, k_new, q = _setup(idx, p)
    w, bt, cl = dev(p.weights), dev(p.block_table), dev(p.context_lens)
    ws = torch.empty(idx.paged_decode_step_workspace_bytes(p.B, 2, 32, p.block_table.shape[1],
                                                           2048), dtype=torch.uint8, device="cuda")
    out = torch.empty((p.rows, 2048), dtype=torch.int32, device="cuda")
    run = lambda: idx.paged_decode_step(k_new, q, w, cache, bt, cl, 2, 32, 2048, workspace=ws,
                                        out=out)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    first = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    ocache, res = _oracle(oracle, p)
    for _ in range(3):
        out.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(cache.cpu().numpy(), ocache)
        _check(p, out.cpu().numpy(), res)
    _check(p, first.cpu().numpy(), res)


def test_step_bad_new_key_positions_are_counted(idx, oracle):
    """A sequence whose new token's page id lies outside the cache: that key is
    skipped and counted (and so is the page when the scoring reaches it); the
    other sequences are exact."""
    p = wl.make_decode("t", 8300, [3000, 5000, 700], 32, 1)
    bt = p.block_table.copy()
    L1 = int(p.context_lens[1])
    bt[1, (L1 - 1) // 64] = p.num_blocks + 5
    cache, k_new, q = _setup(idx, p)
    errs = idx.new_errors()
    out = idx.paged_decode_step(k_new, q, dev(p.weights), cache, dev(bt), dev(p.context_lens), 1,
                                32, 2048, errors=errs)
    torch.cuda.synchronize()
    assert errs.cpu().tolist()[0] >= 1 and errs.cpu().tolist()[1] == 0
    ocache, res = _oracle(oracle, p, [0, 2])
    got = cache.cpu().numpy()
    new_slot = int(p.slots[p.new_token_rows()[1]])
    page = new_slot // 64
    keep = np.ones(p.num_blocks, bool)
    keep[page] = False  # the page the step could not reach holds the poison where the key goes
    assert np.array_equal(got[keep], ocache[keep])
    _check(p, out.cpu().numpy(), res)
