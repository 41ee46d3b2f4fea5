"""GPU parity, through the C ABI, of the prefill logits + top-k without a logits
tensor (idx_mqa_logits_topk) against the oracle's logits and ranking: causal
and chunked windows at both head counts, rows shorter and longer than k,
empty windows, rows whose every position is a candidate (all logits equal,
and logits rising with the position), and sampled rows of the full-size
32768-token causal prefill."""
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


def _prefill_inputs(idx, p):
    S = int(p.tok_offsets[-1])
    cache = dev(wl.poisoned_cache(p.num_blocks))
    idx.quant_insert(dev_bf16(p.k), dev(p.slots), cache)
    kv, ks = idx.gather_k(cache, dev(p.block_table),
                          dev((p.prefix_lens + p.new_lens).astype(np.int32)),
                          dev(p.tok_offsets[:-1].astype(np.int64)), S)
    qv, qs = idx.quant_q(dev_bf16(p.q))
    return S, kv, ks, qv, qs


def _oracle_rows(oracle, p, qv, qs, kv, ks, rows, weights=None):
    st, en = p.windows()
    w = p.weights if weights is None else weights
    qv_h = qv.cpu().numpy().reshape(p.T, p.H, 64)[rows].reshape(-1, 64)
    qs_h = qs.cpu().numpy().reshape(p.T, p.H, 4)[rows].reshape(-1, 4)
    lg, mag = oracle.mqa_logits(qv_h, qs_h, p.H, kv.cpu().numpy(), ks.cpu().numpy(), w[rows],
                                st[rows], en[rows])
    return st, en, lg, mag


def _check_rows(p, got, rows, st, en, lg, mag, k):
    for i, r in enumerate(rows):
        a, b = int(st[r]), int(en[r])
        check_topk(got[r], lg[i, a:b], mag[i, a:b], b - a, k, f"row {r} (len {b - a})")


@pytest.mark.parametrize("T,H", [(3000, 32), (2500, 64), (130, 32)])
def test_prefill_topk_causal(idx, oracle, T, H):
    p = wl.make_prefill("t", 9000 + T, [0], [T], H)
    S, kv, ks, qv, qs = _prefill_inputs(idx, p)
    st, en = p.windows()
    errs = idx.new_errors()
    out = idx.mqa_logits_topk(qv, qs, dev(p.weights), kv, ks, dev(st), dev(en), H, 2048,
                              errors=errs)
    torch.cuda.synchronize()
    assert errs.cpu().tolist() == [0, 0]
    rows = np.arange(T)
    _, _, lg, mag = _oracle_rows(oracle, p, qv, qs, kv, ks, rows)
    _check_rows(p, out.cpu().numpy(), rows, st, en, lg, mag, 2048)


def test_prefill_topk_chunked_and_small_k(idx, oracle):
    p = wl.make_prefill("t", 9100, [3000, 0, 777], [1500, 900, 2100], 32)
    S, kv, ks, qv, qs = _prefill_inputs(idx, p)
    st, en = p.windows()
    rows = np.arange(p.T)
    _, _, lg, mag = _oracle_rows(oracle, p, qv, qs, kv, ks, rows)
    for k in (2048, 100, 1):
        out = idx.mqa_logits_topk(qv, qs, dev(p.weights), kv, ks, dev(st), dev(en), 32, k)
        torch.cuda.synchronize()
        _check_rows(p, out.cpu().numpy(), rows, st, en, lg, mag, k)


def test_prefill_topk_matches_unfused(idx, oracle):
    """Both routes satisfy the oracle's rule on the same rows."""
    p = wl.make_prefill("t", 9200, [0], [4500], 32)
    S, kv, ks, qv, qs = _prefill_inputs(idx, p)
    st, en = p.windows()
    st_d, en_d = dev(st), dev(en)
    fused = idx.mqa_logits_topk(qv, qs, dev(p.weights), kv, ks, st_d, en_d, 32, 2048)
    lgt = idx.mqa_logits(qv, qs, dev(p.weights), kv, ks, st_d, en_d, 32)
    unfused = idx.topk_rows(lgt, en_d, 2048, row_start=st_d)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 2046, 2047, 2048, 3000, 4499])
    _, _, lg, mag = _oracle_rows(oracle, p, qv, qs, kv, ks, rows)
    _check_rows(p, fused.cpu().numpy(), rows, st, en, lg, mag, 2048)
    _check_rows(p, unfused.cpu().numpy(), rows, st, en, lg, mag, 2048)


def test_prefill_topk_every_position_a_candidate(idx, oracle):
    """All logits equal (zero weights): every position reaches the threshold,
    so every list holds the whole window; any k distinct positions are right."""
    p = wl.make_prefill("t", 9300, [0], [5000], 32)
    S, kv, ks, qv, qs = _prefill_inputs(idx, p)
    st, en = p.windows()
    out = idx.mqa_logits_topk(qv, qs, dev(np.zeros_like(p.weights)), kv, ks, dev(st), dev(en), 32,
                              2048)
    torch.cuda.synchronize()
    g = out.cpu().numpy()
    for r in (0, 10, 2047, 2048, 2049, 4999):
        n = int(en[r] - st[r])
        m = min(n, 2048)
        sel = g[r, :m]
        assert (g[r, m:] == -1).all() and len(np.unique(sel)) == m
        assert sel.min() >= 0 and sel.max() < n


def test_prefill_topk_rising_logits(idx, oracle):
    """Keys whose logits rise with the position (one nonzero dimension whose
    value grows along the sequence, all weights positive): every position
    is admitted when it arrives, and the k largest are the last k."""
    T = 4096
    g = wl.rng(9400)
    kx = np.zeros((T, 128), np.float32)
    kx[:, 0] = 1.0 + np.arange(T, dtype=np.float32) / 64.0
    qx = np.zeros((T, 32, 128), np.float32)
    qx[:, :, 0] = 1.0
    p = wl.make_prefill("t", 9400, [0], [T], 32)
    p.k = wl.bf16_bits(kx)
    p.q = wl.bf16_bits(qx)
    p.weights = np.abs(p.weights) + 0.01
    S, kv, ks, qv, qs = _prefill_inputs(idx, p)
    st, en = p.windows()
    out = idx.mqa_logits_topk(qv, qs, dev(p.weights), kv, ks, dev(st), dev(en), 32, 2048)
    torch.cuda.synchronize()
    rows = np.array([100, 2047, 2048, 3000, 4095])
    _, _, lg, mag = _oracle_rows(oracle, p, qv, qs, kv, ks, rows)
    _check_rows(p, out.cpu().numpy(), rows, st, en, lg, mag, 2048)
    del g


def test_prefill_topk_empty_windows(idx):
    p = wl.make_prefill("t", 9500, [0], [600], 32)
    S, kv, ks, qv, qs = _prefill_inputs(idx, p)
    st = np.zeros(p.T, np.int32)
    en = np.zeros(p.T, np.int32)
    en[5] = 3
    out = idx.mqa_logits_topk(qv, qs, dev(p.weights), kv, ks, dev(st), dev(en), 32, 64)
    torch.cuda.synchronize()
    g = out.cpu().numpy()
    assert (g[np.arange(p.T) != 5] == -1).all()
    assert sorted(g[5, :3].tolist()) == [0, 1, 2] and (g[5, 3:] == -1).all()


def test_prefill_topk_full_size_sampled(idx, oracle):
    p = wl.prefill()
    S, kv, ks, qv, qs = _prefill_inputs(idx, p)
    st, en = p.windows()
    errs = idx.new_errors()
    out = idx.mqa_logits_topk(qv, qs, dev(p.weights), kv, ks, dev(st), dev(en), 32, 2048,
                              errors=errs)
    torch.cuda.synchronize()
    assert errs.cpu().tolist() == [0, 0]
    rows = np.array([0, 2046, 2047, 2048, 9999, 20000, 32766, 32767])
    _, _, lg, mag = _oracle_rows(oracle, p, qv, qs, kv, ks, rows)
    _check_rows(p, out.cpu().numpy(), rows, st, en, lg, mag, 2048)
