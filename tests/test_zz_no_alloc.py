"""The no-allocation variant of the fused decode entry (callers that cannot
allocate device memory pass only inputs and outputs; the scratch is the
library's built-in array).  Through the C ABI, two calls in a row must agree
with idx_paged_logits_topk on the same inputs, under the top-k tolerance rule
the other tests use; a batch larger than the built-in scratch is refused.

This file is collected last so that a failure here leaves every other test
already run."""
import ctypes

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


def _call_noalloc(idx, d, p, k, out):
    lib = idx.lib
    st = lib.idx_paged_logits_topk_noalloc(
        ctypes.c_void_p(d["qv"].data_ptr()), ctypes.c_void_p(d["qs"].data_ptr()), p.B, p.next_n,
        p.H, ctypes.c_void_p(d["cache"].data_ptr()), p.num_blocks, 64,
        ctypes.c_void_p(d["bt"].data_ptr()), p.block_table.shape[1],
        ctypes.c_void_p(d["cl"].data_ptr()), ctypes.c_void_p(d["w"].data_ptr()), k,
        ctypes.c_void_p(out.data_ptr()), None,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def test_noalloc_matches_workspace_entry(idx, oracle):
    p = wl.make_decode("t", 900, [300, 2047, 2049, 9000, 20000, 5], 64, 2)
    k = 2048
    cache = dev(wl.poisoned_cache(p.num_blocks))
    idx.quant_insert(dev_bf16(p.k), dev(p.slots), cache)
    qv, qs = idx.quant_q(dev_bf16(p.q))
    d = dict(cache=cache, qv=qv, qs=qs, w=dev(p.weights), bt=dev(p.block_table),
             cl=dev(p.context_lens))
    ref = idx.paged_logits_topk(qv, qs, d["w"], cache, d["bt"], d["cl"], p.next_n, p.H, k)
    torch.cuda.synchronize()
    ref = ref.cpu().numpy()
    ocache = wl.poisoned_cache(p.num_blocks)
    oracle.quant_insert(p.k, p.slots, ocache)
    oqv, oqs = oracle.quant_q(p.q)
    ld = p.block_table.shape[1] * 64
    ol, om = oracle.paged_mqa_logits(oqv, oqs, p.B, p.next_n, p.H, ocache, p.block_table,
                                     p.context_lens, p.weights, ld)
    st, en = p.row_windows()
    for call in range(2):
        out = torch.full((p.rows, k), -7, dtype=torch.int32, device="cuda")
        assert _call_noalloc(idx, d, p, k, out) == 0
        torch.cuda.synchronize()
        g = out.cpu().numpy()
        for r in range(p.rows):
            n = int(en[r])
            check_topk(g[r], ol[r, :n], om[r, :n], n, k, f"call {call} row {r}")
            # against the workspace entry: same set up to values tied within tolerance
            m = min(n, k)
            diff = set(g[r, :m].tolist()) ^ set(ref[r, :m].tolist())
            if diff:
                order = np.lexsort((np.arange(n), -ol[r, :n]))
                vk = ol[r, order[k - 1]]
                tol = 1e-5 * om[r, :n]
                for i in diff:
                    assert abs(ol[r, i] - vk) <= tol[i] + tol[order[k - 1]], (call, r, i)
            assert (g[r, m:] == -1).all() and (ref[r, m:] == -1).all()


def test_noalloc_refuses_batches_above_its_scratch(idx):
    p = wl.make_decode("t", 901, [100], 32, 1, max_blocks=4096)
    cache = dev(wl.poisoned_cache(p.num_blocks))
    qv, qs = idx.quant_q(dev_bf16(p.q))
    d = dict(cache=cache, qv=qv, qs=qs, w=dev(p.weights), bt=dev(p.block_table),
             cl=dev(p.context_lens))
    big = wl.DecodeProblem(**{**p.__dict__, "B": 64})
    bt = np.tile(p.block_table, (64, 1))
    d["bt"], d["cl"] = dev(bt), dev(np.tile(p.context_lens, 64))
    d["qv"], d["qs"] = qv.repeat(64, 1), qs.repeat(64, 1)
    d["w"] = dev(np.tile(p.weights, (64, 1)))
    assert idx.paged_logits_topk_workspace_bytes(64, 1, 4096, 2048) > (32 << 20)
    out = torch.empty((64, 2048), dtype=torch.int32, device="cuda")
    big.block_table = bt
    assert _call_noalloc(idx, d, big, 2048, out) == 1


def test_noalloc_through_the_binding(idx, oracle):
    """The Python binding of the entry, on a batch at both head counts' MMA
    widths of the decode core (H = 32, next_n = 1 and 2), with the refusal
    raised as an IdxError carrying the library's detail."""
    for seed, next_n in ((910, 1), (911, 2)):
        p = wl.make_decode("t", seed, [64, 2048, 2049, 7000], 32, next_n)
        cache = dev(wl.poisoned_cache(p.num_blocks))
        idx.quant_insert(dev_bf16(p.k), dev(p.slots), cache)
        qv, qs = idx.quant_q(dev_bf16(p.q))
        errs = idx.new_errors()
        got = idx.paged_logits_topk_noalloc(qv, qs, dev(p.weights), cache, dev(p.block_table),
                                            dev(p.context_lens), next_n, 32, 2048, errors=errs)
        torch.cuda.synchronize()
        assert errs.cpu().tolist() == [0, 0]
        ocache = wl.poisoned_cache(p.num_blocks)
        oracle.quant_insert(p.k, p.slots, ocache)
        oqv, oqs = oracle.quant_q(p.q)
        ol, om = oracle.paged_mqa_logits(oqv, oqs, p.B, next_n, 32, ocache, p.block_table,
                                         p.context_lens, p.weights, p.block_table.shape[1] * 64)
        st, en = p.row_windows()
        g = got.cpu().numpy()
        for r in range(p.rows):
            n = int(en[r])
            check_topk(g[r], ol[r, :n], om[r, :n], n, 2048, f"next_n {next_n} row {r}")
    p = wl.make_decode("t", 912, [100], 32, 1, max_blocks=4096)
    bt = dev(np.tile(p.block_table, (64, 1)))
    cache = dev(wl.poisoned_cache(p.num_blocks))
    qv, qs = idx.quant_q(dev_bf16(np.tile(p.q, (64, 1, 1))))
    with pytest.raises(idx.IdxError) as e:
        idx.paged_logits_topk_noalloc(qv, qs, dev(np.tile(p.weights, (64, 1))), cache, bt,
                                      dev(np.tile(p.context_lens, 64)), 1, 32, 2048)
    assert e.value.status == 1 and e.value.detail  # invalid argument, with the reason
