"""GPU parity of prefill logits (tcgen05 MXF4 path) and of the cache gather
against the oracle through the C ABI: causal and chunked windows, query counts
that are not a multiple of the per-CTA group, clean and unclean rows, the
paged-vs-gathered invariant, and sampled rows of the full-size prefills."""
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


def prepare(idx, oracle, p):
    """Paged insert of every token, gather into contiguous keys, q-quant; the
    oracle does the same from the bf16 inputs."""
    gcache = dev(wl.poisoned_cache(p.num_blocks))
    idx.quant_insert(dev_bf16(p.k), dev(p.slots), gcache)
    lens = (p.prefix_lens.astype(np.int64) + p.new_lens).astype(np.int32)
    offs = p.tok_offsets[:-1].astype(np.int64)
    total = int(p.tok_offsets[-1])
    errs = idx.new_errors()
    kv, ks = idx.gather_k(gcache, dev(p.block_table), dev(lens), dev(offs), total, errors=errs)
    qv, qs = idx.quant_q(dev_bf16(p.q))
    ocache = wl.poisoned_cache(p.num_blocks)
    oracle.quant_insert(p.k, p.slots, ocache)
    okv, oks = oracle.gather_k(ocache, p.block_table, lens, offs, total)
    oqv, oqs = oracle.quant_q(p.q)
    torch.cuda.synchronize()
    assert errs.cpu().tolist() == [0, 0]
    assert np.array_equal(kv.cpu().numpy(), okv) and np.array_equal(ks.cpu().numpy(), oks)
    return dict(kv=kv, ks=ks, qv=qv, qs=qs, okv=okv, oks=oks, oqv=oqv, oqs=oqs, cache=gcache,
                ocache=ocache)


@pytest.mark.parametrize("H", [32, 64])
@pytest.mark.parametrize("clean", [True, False])
def test_causal_prefill_parity(idx, oracle, H, clean):
    p = wl.make_prefill("t", 600 + H, [0], [701], H)
    d = prepare(idx, oracle, p)
    st, en = p.windows()
    S = int(p.tok_offsets[-1])
    ld = S + 5
    out = torch.full((p.T, ld), float("nan"), device="cuda")
    errs = idx.new_errors()
    idx.mqa_logits(d["qv"], d["qs"], dev(p.weights), d["kv"], d["ks"], dev(st), dev(en), H,
                   ld=ld, clean=clean, out=out, errors=errs)
    torch.cuda.synchronize()
    assert errs.cpu().tolist() == [0, 0]
    g = out.cpu().numpy()
    ol, om = oracle.mqa_logits(d["oqv"], d["oqs"], H, d["okv"], d["oks"], p.weights, st, en, ld)
    for t in range(p.T):
        check_logits(g[t, st[t]:en[t]], ol[t, st[t]:en[t]], om[t, st[t]:en[t]], f"t={t}")
        outside = np.r_[g[t, :st[t]], g[t, en[t]:S]]
        if clean:
            assert np.isneginf(outside).all(), f"t={t}"
        else:
            assert np.isnan(outside).all(), f"t={t}"
        assert np.isnan(g[t, S:]).all()


def test_chunked_prefill_windows(idx, oracle):
    """Three sequences with cached prefixes; the gathered buffer holds every
    sequence, each query sees only its own sequence's causal window."""
    p = wl.make_prefill("t", 610, [0, 100, 1000], [300, 50, 129], 32)
    d = prepare(idx, oracle, p)
    st, en = p.windows()
    S = int(p.tok_offsets[-1])
    out = idx.mqa_logits(d["qv"], d["qs"], dev(p.weights), d["kv"], d["ks"], dev(st), dev(en), 32,
                         clean=True)
    torch.cuda.synchronize()
    g = out.cpu().numpy()
    ol, om = oracle.mqa_logits(d["oqv"], d["oqs"], 32, d["okv"], d["oks"], p.weights, st, en, S)
    for t in range(p.T):
        check_logits(g[t, st[t]:en[t]], ol[t, st[t]:en[t]], om[t, st[t]:en[t]], f"t={t}")
        assert np.isneginf(np.r_[g[t, :st[t]], g[t, en[t]:]]).all()


def test_empty_and_clamped_windows(idx, oracle):
    p = wl.make_prefill("t", 620, [0], [20], 32)
    d = prepare(idx, oracle, p)
    S = 20
    st = np.zeros(20, np.int32)
    en = np.arange(1, 21, dtype=np.int32)
    en[3] = 0                     # empty window
    st[5], en[5] = 7, 7           # empty window
    en[6] = 50                    # past S: clamped and counted
    errs = idx.new_errors()
    out = idx.mqa_logits(d["qv"], d["qs"], dev(p.weights), d["kv"], d["ks"], dev(st), dev(en), 32,
                         clean=True, errors=errs)
    torch.cuda.synchronize()
    assert errs.cpu().tolist()[0] == 1
    g = out.cpu().numpy()
    assert np.isneginf(g[3]).all() and np.isneginf(g[5]).all()
    en_c = np.minimum(en, S)
    ol, om = oracle.mqa_logits(d["oqv"], d["oqs"], 32, d["okv"], d["oks"], p.weights, st, en_c, S)
    for t in [0, 6, 19]:
        check_logits(g[t, :en_c[t]], ol[t, :en_c[t]], om[t, :en_c[t]], f"t={t}")


def test_paged_decode_equals_gathered_prefill(idx, oracle):
    """The paged decode logits of a sequence's newest tokens equal the prefill
    logits of the same queries over the gathered keys (two GPU paths)."""
    p = wl.make_decode("t", 630, [513, 4000], 64, 2)
    cache = dev(wl.poisoned_cache(p.num_blocks))
    idx.quant_insert(dev_bf16(p.k), dev(p.slots), cache)
    qv, qs = idx.quant_q(dev_bf16(p.q))
    w = dev(p.weights)
    paged = idx.paged_mqa_logits(qv, qs, w, cache, dev(p.block_table), dev(p.context_lens), 2, 64,
                                 clean=True).cpu().numpy()
    offs = p.tok_offsets[:-1].astype(np.int64)
    kv, ks = idx.gather_k(cache, dev(p.block_table), dev(p.context_lens), dev(offs), p.total_tokens)
    st, en = p.row_windows()
    b_of = np.repeat(np.arange(p.B), 2)
    gst = (st + offs[b_of]).astype(np.int32)
    gen = (en + offs[b_of]).astype(np.int32)
    pre = idx.mqa_logits(qv, qs, w, kv, ks, dev(gst), dev(gen), 64).cpu().numpy()
    ocache = wl.poisoned_cache(p.num_blocks)
    oracle.quant_insert(p.k, p.slots, ocache)
    oqv, oqs = oracle.quant_q(p.q)
    ol, om = oracle.paged_mqa_logits(oqv, oqs, p.B, 2, 64, ocache, p.block_table, p.context_lens,
                                     p.weights, paged.shape[1])
    for r in range(p.rows):
        n = int(en[r])
        a = paged[r, :n].astype(np.float64)
        b = pre[r, gst[r]:gen[r]].astype(np.float64)
        assert (np.abs(a - b) <= 2e-5 * om[r, :n]).all(), f"row {r}"


def test_gather_bad_inputs(idx):
    p = wl.make_decode("t", 640, [100, 70], 32, 1)
    cache = dev(wl.poisoned_cache(p.num_blocks))
    bt = p.block_table.copy()
    bt[1, 0] = -3
    lens = p.context_lens.copy()
    errs = idx.new_errors()
    offs = np.array([0, 100], np.int64)
    idx.gather_k(cache, dev(bt), dev(lens), dev(offs), 150, errors=errs)   # row 1 overflows out_rows
    torch.cuda.synchronize()
    assert errs.cpu().tolist()[0] >= 2


def _sampled_prefill(idx, oracle, p, sample_rows):
    gcache = dev(wl.poisoned_cache(p.num_blocks))
    idx.quant_insert(dev_bf16(p.k), dev(p.slots), gcache)
    lens = (p.prefix_lens.astype(np.int64) + p.new_lens).astype(np.int32)
    offs = p.tok_offsets[:-1].astype(np.int64)
    S = int(p.tok_offsets[-1])
    kv, ks = idx.gather_k(gcache, dev(p.block_table), dev(lens), dev(offs), S)
    qv, qs = idx.quant_q(dev_bf16(p.q))
    st, en = p.windows()
    logits = idx.mqa_logits(qv, qs, dev(p.weights), kv, ks, dev(st), dev(en), p.H)
    top = idx.topk_rows(logits, dev(en), 2048, row_start=dev(st))
    torch.cuda.synchronize()
    rows = np.asarray(sample_rows)
    g = logits[torch.from_numpy(rows).cuda()].cpu().numpy()
    gt = top.cpu().numpy()[rows]
    del logits
    # oracle: its own keys (all of them) and the sampled queries only
    ocache = wl.poisoned_cache(p.num_blocks)
    oracle.quant_insert(p.k, p.slots, ocache)
    okv, oks = oracle.gather_k(ocache, p.block_table, lens, offs, S)
    oqv, oqs = oracle.quant_q(p.q[rows])
    ol, om = oracle.mqa_logits(oqv, oqs, p.H, okv, oks, p.weights[rows], st[rows], en[rows], S)
    for i, t in enumerate(rows):
        a, b = st[t], en[t]
        check_logits(g[i, a:b], ol[i, a:b], om[i, a:b], f"t={t}")
        check_topk(gt[i], ol[i, a:b], om[i, a:b], int(b - a), 2048, f"topk t={t}")


def test_full_size_causal_prefill_sampled(idx, oracle):
    p = wl.prefill()
    _sampled_prefill(idx, oracle, p, [0, 1, 7, 2047, 2048, 2049, 16385, 32767])


def test_full_size_mixed_prefill_sampled(idx, oracle):
    """Chunked prefill of the mixed batch, one call per sequence over that
    sequence's gathered keys (as a serving step would issue it)."""
    p = wl.mixed_prefill_part()
    gcache = dev(wl.poisoned_cache(p.num_blocks))
    idx.quant_insert(dev_bf16(p.k), dev(p.slots), gcache)
    lens = (p.prefix_lens.astype(np.int64) + p.new_lens).astype(np.int32)
    offs = p.tok_offsets[:-1].astype(np.int64)
    S = int(p.tok_offsets[-1])
    kv, ks = idx.gather_k(gcache, dev(p.block_table), dev(lens), dev(offs), S)
    qv, qs = idx.quant_q(dev_bf16(p.q))
    ocache = wl.poisoned_cache(p.num_blocks)
    oracle.quant_insert(p.k, p.slots, ocache)
    q_off = np.concatenate([[0], np.cumsum(p.new_lens)]).astype(np.int64)
    H = p.H
    for b in [int(np.argmax(p.prefix_lens)), int(np.argmin(p.prefix_lens))]:
        L = int(lens[b])
        P = int(p.prefix_lens[b])
        T = int(p.new_lens[b])
        st = np.zeros(T, np.int32)
        en = (P + np.arange(T) + 1).astype(np.int32)
        qa, qb = int(q_off[b]), int(q_off[b + 1])
        kvb = kv[offs[b]:offs[b] + L]
        ksb = ks[offs[b]:offs[b] + L]
        logits = idx.mqa_logits(qv[qa * H:qb * H], qs[qa * H:qb * H], dev(p.weights[qa:qb]), kvb,
                                ksb, dev(st), dev(en), H)
        top = idx.topk_rows(logits, dev(en), 2048)
        torch.cuda.synchronize()
        rows = np.array([0, 1, T // 2, T - 1])
        g = logits.cpu().numpy()[rows]
        gt = top.cpu().numpy()[rows]
        okv, oks = oracle.gather_k(ocache, p.block_table[b:b + 1], lens[b:b + 1],
                                   np.array([0], np.int64), L)
        oqv, oqs = oracle.quant_q(p.q[qa + rows])
        ol, om = oracle.mqa_logits(oqv, oqs, H, okv, oks, p.weights[qa + rows], st[rows],
                                   en[rows], L)
        for i, t in enumerate(rows):
            n = int(en[t])
            check_logits(g[i, :n], ol[i, :n], om[i, :n], f"seq {b} t={t}")
            check_topk(gt[i], ol[i, :n], om[i, :n], n, 2048, f"seq {b} topk t={t}")
