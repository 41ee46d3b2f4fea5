"""CUDA-graph capture of every entry point: each call is captured once and
replayed, and a replay's output equals an eager call's on the same inputs (the
entries allocate nothing and never synchronise, so a captured call reads its
buffers afresh on every replay).  The fused decode call is replayed with new
query values before each replay, which also checks that its work-item counter
starts over on every replay of the same captured launch."""
import numpy as np
import pytest
import torch

from sparse_attention_indexer_quant_gb300 import workloads as wl
from idx_testutil import dev, dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def idx():
    from sparse_attention_indexer_quant_gb300 import binding
    binding.check_device(torch.cuda.current_device())
    return binding


def capture(fn):
    """fn run once on a side stream (per-device setup), then captured."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def same_sets(a: torch.Tensor, b: torch.Tensor):
    a = np.sort(a.cpu().numpy(), axis=1)
    b = np.sort(b.cpu().numpy(), axis=1)
    np.testing.assert_array_equal(a, b)


def test_graph_fused_decode_replays(idx):
    p = wl.make_decode("g", 951, [4100, 9000, 20000, 300, 2049], 32, 1)
    cache = dev(wl.poisoned_cache(p.num_blocks))
    idx.quant_insert(dev_bf16(p.k), dev(p.slots), cache)
    qv, qs = idx.quant_q(dev_bf16(p.q))
    w, bt, cl = dev(p.weights), dev(p.block_table), dev(p.context_lens)
    ws = idx.new_paged_topk_workspace(p.B, 1, p.block_table.shape[1], 2048)
    out = torch.empty((p.rows, 2048), dtype=torch.int32, device="cuda")
    g = capture(lambda: idx.paged_logits_topk(qv, qs, w, cache, bt, cl, 1, 32, 2048,
                                              workspace=ws, out=out))
    rng = np.random.default_rng(952)
    for r in range(3):
        q = wl.normal_bf16(rng, p.q.shape)
        nv, ns = idx.quant_q(dev_bf16(q))
        qv.copy_(nv)
        qs.copy_(ns)
        g.replay()
        ref = idx.paged_logits_topk(qv, qs, w, cache, bt, cl, 1, 32, 2048)
        torch.cuda.synchronize()
        same_sets(out, ref)


def test_graph_other_entries(idx):
    p = wl.make_decode("g", 953, [3000, 700, 12000], 64, 2)
    k, slots = dev_bf16(p.k), dev(p.slots)
    # insert and q-quant
    cache_g = dev(wl.poisoned_cache(p.num_blocks))
    cache_e = cache_g.clone()
    g = capture(lambda: idx.quant_insert(k, slots, cache_g))
    cache_g.copy_(cache_e)
    g.replay()
    idx.quant_insert(k, slots, cache_e)
    q = dev_bf16(p.q)
    qv = torch.empty((p.rows * p.H, 64), dtype=torch.uint8, device="cuda")
    qs = torch.empty((p.rows * p.H, 4), dtype=torch.uint8, device="cuda")
    g2 = capture(lambda: idx.quant_q(q, out_vals=qv, out_scales=qs))
    qv.zero_()
    g2.replay()
    ev, es = idx.quant_q(q)
    torch.cuda.synchronize()
    assert torch.equal(cache_g, cache_e) and torch.equal(qv, ev) and torch.equal(qs, es)
    # paged logits (clean rows) and the rows' top-k
    w, bt, cl = dev(p.weights), dev(p.block_table), dev(p.context_lens)
    ld = p.block_table.shape[1] * 64
    lg = torch.empty((p.rows, ld), dtype=torch.float32, device="cuda")
    g3 = capture(lambda: idx.paged_mqa_logits(qv, qs, w, cache_e, bt, cl, 2, 64, ld=ld,
                                              clean=True, out=lg))
    lg.zero_()
    g3.replay()
    lref = idx.paged_mqa_logits(qv, qs, w, cache_e, bt, cl, 2, 64, ld=ld, clean=True)
    torch.cuda.synchronize()
    assert torch.equal(lg, lref)
    st, en = p.row_windows()
    st_d, en_d = dev(st), dev(en)
    tk = torch.empty((p.rows, 2048), dtype=torch.int32, device="cuda")
    g4 = capture(lambda: idx.topk_rows(lg, en_d, 2048, row_start=st_d, out=tk))
    tk.zero_()
    g4.replay()
    tref = idx.topk_rows(lg, en_d, 2048, row_start=st_d)
    torch.cuda.synchronize()
    same_sets(tk, tref)
    # gather and prefill logits over the gathered keys of sequence 2
    lens = p.context_lens.astype(np.int32)
    offs = np.zeros(p.B, np.int64)
    offs[1:] = np.cumsum(lens[:-1])
    S = int(lens.sum())
    lens_d, offs_d = dev(lens), dev(offs)
    holder = {}
    g5 = capture(lambda: holder.__setitem__("kv", idx.gather_k(cache_e, bt, lens_d, offs_d, S)))
    g5.replay()
    kv_g, ks_g = holder["kv"]
    kv_e, ks_e = idx.gather_k(cache_e, bt, lens_d, offs_d, S)
    torch.cuda.synchronize()
    assert torch.equal(kv_g, kv_e) and torch.equal(ks_g, ks_e)
    T = 64
    qp = dev_bf16(wl.normal_bf16(np.random.default_rng(954), (T, 64, 128)))
    pqv, pqs = idx.quant_q(qp)
    pw = dev(wl.head_weights(np.random.default_rng(955), T, 64))
    end = (np.arange(T, dtype=np.int32) + int(offs[2]) + int(lens[2]) - T + 1)
    start = np.full(T, int(offs[2]), np.int32)
    st2, en2 = dev(start), dev(end)
    pl = torch.empty((T, S), dtype=torch.float32, device="cuda")
    g6 = capture(lambda: idx.mqa_logits(pqv, pqs, pw, kv_e, ks_e, st2, en2, 64, clean=True,
                                        out=pl))
    pl.zero_()
    g6.replay()
    pref = idx.mqa_logits(pqv, pqs, pw, kv_e, ks_e, st2, en2, 64, clean=True)
    torch.cuda.synchronize()
    assert torch.equal(pl, pref)
