"""GPU parity of the paged decode logits (tcgen05 MXF4 path) against the
oracle, through the C ABI: ragged contexts spanning several tiles with partial
tails, both head counts and both query-token counts, clean and unclean rows,
and sampled rows of the full-size decode workloads."""
import numpy as np
import pytest
import torch

from sparse_attention_indexer_quant_gb300 import workloads as wl
from idx_testutil import check_logits, dev, dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def idx():
    from sparse_attention_indexer_quant_gb300 import binding
    binding.check_device(torch.cuda.current_device())
    return binding


def upload(idx, oracle, p):
    """Insert on the GPU (and separately in the oracle) and quantise q."""
    gcache = dev(wl.poisoned_cache(p.num_blocks))
    idx.quant_insert(dev_bf16(p.k), dev(p.slots), gcache)
    qv, qs = idx.quant_q(dev_bf16(p.q))
    ocache = wl.poisoned_cache(p.num_blocks)
    oracle.quant_insert(p.k, p.slots, ocache)
    oqv, oqs = oracle.quant_q(p.q)
    return dict(cache=gcache, qv=qv, qs=qs, w=dev(p.weights), bt=dev(p.block_table),
                cl=dev(p.context_lens), ocache=ocache, oqv=oqv, oqs=oqs)


LENS = [1, 2, 63, 64, 65, 127, 128, 129, 700, 2500, 4097]


@pytest.mark.parametrize("H,next_n", [(32, 1), (32, 2), (64, 1), (64, 2)])
@pytest.mark.parametrize("clean", [True, False])
def test_paged_logits_parity(idx, oracle, H, next_n, clean):
    p = wl.make_decode("t", 300 + H + next_n, LENS, H, next_n)
    d = upload(idx, oracle, p)
    ld = p.block_table.shape[1] * 64 + 8
    out = torch.full((p.rows, ld), float("nan"), device="cuda")
    errs = idx.new_errors()
    idx.paged_mqa_logits(d["qv"], d["qs"], d["w"], d["cache"], d["bt"], d["cl"], next_n, H,
                         ld=ld, clean=clean, out=out, errors=errs)
    torch.cuda.synchronize()
    assert errs.cpu().tolist() == [0, 0]
    g = out.cpu().numpy()
    ol, om = oracle.paged_mqa_logits(d["oqv"], d["oqs"], p.B, next_n, H, d["ocache"],
                                     p.block_table, p.context_lens, p.weights, ld)
    st, en = p.row_windows()
    for r in range(p.rows):
        n = int(en[r])
        check_logits(g[r, :n], ol[r, :n], om[r, :n], f"row {r} len {n}")
        tail = g[r, n:]
        if clean:
            assert np.isneginf(tail).all(), f"row {r}: clean tail not -inf"
        else:
            assert np.isnan(tail).all(), f"row {r}: unclean tail was written"


def test_paged_logits_bad_inputs_are_counted(idx, oracle):
    """An out-of-range page id and an over-long context are skipped and
    counted; the kernel does not fault and the other rows stay correct."""
    p = wl.make_decode("t", 311, [300, 200, 100], 32, 1)
    d = upload(idx, oracle, p)
    bt = p.block_table.copy()
    bt[0, 1] = p.num_blocks + 5          # bad page id in row 0
    cl = p.context_lens.copy()
    cl[1] = bt.shape[1] * 64 + 1         # longer than the block table
    ld = bt.shape[1] * 64
    errs = idx.new_errors()
    out = idx.paged_mqa_logits(d["qv"], d["qs"], d["w"], d["cache"], dev(bt), dev(cl), 1, 32,
                               ld=ld, clean=True, errors=errs)
    torch.cuda.synchronize()
    e = errs.cpu().tolist()
    assert e[0] >= 2 and e[1] == 0
    ol, om = oracle.paged_mqa_logits(d["oqv"], d["oqs"], p.B, 1, 32, d["ocache"], p.block_table,
                                     p.context_lens, p.weights, ld)
    check_logits(out.cpu().numpy()[2, :100], ol[2, :100], om[2, :100], "row 2")


def _sampled_full_size(idx, oracle, p, rows_to_check, ld=None):
    """GPU logits for the whole batch; the oracle recomputes the sampled
    sequences from their own bf16 keys (its own quantisation), so no oracle
    input comes from the GPU."""
    gcache = dev(wl.poisoned_cache(p.num_blocks))
    idx.quant_insert(dev_bf16(p.k), dev(p.slots), gcache)
    qv, qs = idx.quant_q(dev_bf16(p.q))
    ld = ld or p.block_table.shape[1] * 64
    out = idx.paged_mqa_logits(qv, qs, dev(p.weights), gcache, dev(p.block_table),
                               dev(p.context_lens), p.next_n, p.H, ld=ld, clean=True)
    torch.cuda.synchronize()
    g = out.cpu().numpy()
    for b in rows_to_check:
        lo, hi = int(p.tok_offsets[b]), int(p.tok_offsets[b + 1])
        L = hi - lo
        sub_bt = p.block_table[b:b + 1]
        ocache = wl.poisoned_cache(p.num_blocks)
        oracle.quant_insert(p.k[lo:hi], p.slots[lo:hi], ocache)
        rows = slice(b * p.next_n, (b + 1) * p.next_n)
        oqv, oqs = oracle.quant_q(p.q[rows])
        ol, om = oracle.paged_mqa_logits(oqv, oqs, 1, p.next_n, p.H, ocache, sub_bt,
                                         np.array([L], np.int32), p.weights[rows], ld)
        for j in range(p.next_n):
            n = L - p.next_n + j + 1
            r = b * p.next_n + j
            check_logits(g[r, :n], ol[j, :n], om[j, :n], f"seq {b} row {j}")
            assert np.isneginf(g[r, n:]).all()


def test_full_size_batched_decode_sampled(idx, oracle):
    p = wl.batched_decode()
    _sampled_full_size(idx, oracle, p, [0, 31, 63])


def test_full_size_long_decode_sampled(idx, oracle):
    p = wl.long_decode()
    _sampled_full_size(idx, oracle, p, [5])
