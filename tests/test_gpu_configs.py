"""GPU parity, through the C ABI, on the workload configurations that the other
files do not run at full size:

  - the single-sequence 8K decode (one sequence of 8192 cached tokens, H = 32,
    next_n = 1): insert, q-quant, fused logits + top-k and the unfused logits,
    end to end, with the whole cache compared byte for byte;
  - the decode half of the mixed batch (128 sequences, contexts uniform in
    [1K, 128K], H = 32): the fused top-k and the unfused logits on sampled
    sequences, the shortest and the longest among them;
  - the insert batch of the mixed step: the 8 chunked prefills' 65536 new
    keys and the 128 decode sequences' new keys, with 5% padding rows at
    seeded positions, into a cache that already holds the prefills' cached
    prefixes, compared byte for byte over the whole cache.
"""
import numpy as np
import pytest
import torch

from sparse_attention_indexer_quant_gb300 import workloads as wl
from idx_testutil import check_logits, check_topk, dev, dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def idx():
    from sparse_attention_indexer_quant_gb300 import binding
    binding.check_device(torch.cuda.current_device())
    return binding


def test_single_sequence_decode_end_to_end(idx, oracle):
    p = wl.pr_ref()
    errs = idx.new_errors()
    cache = dev(wl.poisoned_cache(p.num_blocks))
    idx.quant_insert(dev_bf16(p.k), dev(p.slots), cache, errs)
    qv, qs = idx.quant_q(dev_bf16(p.q))
    w, bt, cl = dev(p.weights), dev(p.block_table), dev(p.context_lens)
    top = idx.paged_logits_topk(qv, qs, w, cache, bt, cl, 1, p.H, 2048, errors=errs)
    ld = p.block_table.shape[1] * 64 + 100
    lg = idx.paged_mqa_logits(qv, qs, w, cache, bt, cl, 1, p.H, ld=ld, clean=True, errors=errs)
    torch.cuda.synchronize()
    assert errs.cpu().tolist() == [0, 0]

    ocache = wl.poisoned_cache(p.num_blocks)
    oracle.quant_insert(p.k, p.slots, ocache)
    assert np.array_equal(cache.cpu().numpy(), ocache), "cache bytes differ from the oracle"
    oqv, oqs = oracle.quant_q(p.q)
    assert np.array_equal(qv.cpu().numpy(), oqv) and np.array_equal(qs.cpu().numpy(), oqs)
    L = int(p.context_lens[0])
    ol, om = oracle.paged_mqa_logits(oqv, oqs, 1, 1, p.H, ocache, p.block_table, p.context_lens,
                                     p.weights, L)
    g = lg.cpu().numpy()
    check_logits(g[0, :L], ol[0, :L], om[0, :L], "8K decode logits")
    assert np.isneginf(g[0, L:]).all()
    check_topk(top.cpu().numpy()[0], ol[0], om[0], L, 2048, "8K decode top-k")


def _oracle_sampled(oracle, p, seqs):
    """Oracle logits of the listed sequences of a decode problem, from one
    oracle cache holding just those sequences' keys."""
    ocache = wl.poisoned_cache(p.num_blocks)
    res = {}
    for b in seqs:
        lo, hi = int(p.tok_offsets[b]), int(p.tok_offsets[b + 1])
        oracle.quant_insert(p.k[lo:hi], p.slots[lo:hi], ocache)
    for b in seqs:
        L = int(p.context_lens[b])
        rows = slice(b * p.next_n, (b + 1) * p.next_n)
        oqv, oqs = oracle.quant_q(p.q[rows])
        ol, om = oracle.paged_mqa_logits(oqv, oqs, 1, p.next_n, p.H, ocache,
                                         p.block_table[b:b + 1], p.context_lens[b:b + 1],
                                         p.weights[rows], max(L, 1))
        res[b] = (ol, om, L)
    return res


def test_mixed_decode_half_full_size_sampled(idx, oracle):
    p = wl.mixed_decode_part()
    errs = idx.new_errors()
    cache = dev(wl.poisoned_cache(p.num_blocks))
    for lo in range(0, p.total_tokens, 1 << 21):  # bounded host->device chunks
        hi = min(p.total_tokens, lo + (1 << 21))
        idx.quant_insert(dev_bf16(p.k[lo:hi]), dev(p.slots[lo:hi]), cache, errs)
    qv, qs = idx.quant_q(dev_bf16(p.q))
    w, bt, cl = dev(p.weights), dev(p.block_table), dev(p.context_lens)
    top = idx.paged_logits_topk(qv, qs, w, cache, bt, cl, 1, p.H, 2048, errors=errs)
    lg = idx.paged_mqa_logits(qv, qs, w, cache, bt, cl, 1, p.H, clean=True, errors=errs)
    torch.cuda.synchronize()
    assert errs.cpu().tolist() == [0, 0]
    lens = p.context_lens.astype(np.int64)
    seqs = sorted({int(np.argmin(lens)), int(np.argmax(lens)), 5, 77})
    top = top.cpu().numpy()
    for b, (ol, om, L) in _oracle_sampled(oracle, p, seqs).items():
        check_topk(top[b], ol[0], om[0], L, 2048, f"mixed decode seq {b} (L={L}) top-k")
        g = lg[b].cpu().numpy()
        check_logits(g[:L], ol[0, :L], om[0, :L], f"mixed decode seq {b} (L={L}) logits")
        assert np.isneginf(g[L:]).all()


def test_mixed_insert_batch_with_padding_bit_exact(idx, oracle):
    ib = wl.mixed_insert_batch()
    n = len(ib.slots)
    assert ib.real_rows == 8 * 8192 + 128 and (ib.slots == -1).sum() == round(0.05 * ib.real_rows)
    errs = idx.new_errors()
    cache = dev(wl.poisoned_cache(ib.num_blocks))
    idx.quant_insert(dev_bf16(ib.pre_k), dev(ib.pre_slots), cache, errs)
    idx.quant_insert(dev_bf16(ib.k), dev(ib.slots), cache, errs)
    torch.cuda.synchronize()
    assert errs.cpu().tolist() == [0, 0]
    ocache = wl.poisoned_cache(ib.num_blocks)
    oracle.quant_insert(ib.pre_k, ib.pre_slots, ocache)
    oracle.quant_insert(ib.k, ib.slots, ocache)
    got = cache.cpu().numpy()
    same = got == ocache
    if not same.all():
        page = int(np.nonzero(~same.all(axis=1))[0][0])
        raise AssertionError(f"{int((~same).sum())} cache bytes differ over {n} rows; "
                             f"first differing page {page}")
