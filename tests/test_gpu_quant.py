"""GPU parity of MXFP4 key insert and query quantisation: bit-exact against
the oracle, through the C ABI."""
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


def _insert_both(idx, oracle, k_bits, slots, num_blocks, k_dev=None):
    ocache = wl.poisoned_cache(num_blocks)
    bad = oracle.quant_insert(k_bits, slots, ocache)
    gcache = dev(wl.poisoned_cache(num_blocks))
    errs = idx.new_errors()
    idx.quant_insert(k_dev if k_dev is not None else dev_bf16(k_bits), dev(slots), gcache, errs)
    torch.cuda.synchronize()
    return gcache.cpu().numpy(), ocache, errs.cpu().numpy(), bad


@pytest.mark.parametrize("n,num_blocks", [(1000, 20), (70000, 1300)])
def test_insert_random_bit_exact(idx, oracle, n, num_blocks):
    """Padding (-1), out-of-range and negative slots among valid ones, below
    and above the size where a thread group takes four vectors."""
    g = wl.rng(201)
    k = wl.normal_bf16(g, (n, 128), wl.outlier_channels(g))
    slots = g.permutation(num_blocks * 64)[:n].astype(np.int64)
    slots[g.choice(n, 50, replace=False)] = -1
    slots[7] = num_blocks * 64          # out of range: skipped and counted
    slots[8] = -5                       # negative, not padding: skipped and counted
    gc, oc, errs, bad = _insert_both(idx, oracle, k, slots, num_blocks)
    assert bad == 2 and errs.tolist() == [2, 0]
    assert np.array_equal(gc, oc)


def test_insert_every_bf16_pattern(idx, oracle):
    """Every finite bf16 bit pattern appears as a key element, in blocks of
    mixed magnitude."""
    pats = np.array([p for p in range(1 << 16) if (p & 0x7F80) != 0x7F80], np.uint16)
    g = wl.rng(202)
    pats = pats[g.permutation(len(pats))]
    pad = (-len(pats)) % 128
    pats = np.concatenate([pats, np.zeros(pad, np.uint16)]).reshape(-1, 128)
    n = pats.shape[0]
    num_blocks = (n + 63) // 64
    slots = np.arange(n, dtype=np.int64)
    gc, oc, errs, _ = _insert_both(idx, oracle, pats, slots, num_blocks)
    assert errs.tolist() == [0, 0]
    assert np.array_equal(gc, oc)


def test_insert_special_blocks(idx, oracle):
    """Zeros, negative zeros, subnormals, exact ties and huge values."""
    rows = []
    def f2b(x):
        return wl.bf16_bits(np.asarray(x, np.float32))
    rows.append(np.zeros(128, np.uint16))
    rows.append(np.full(128, 0x8000, np.uint16))                       # all -0
    rows.append(np.array([1, 0x8001] * 64, np.uint16))                 # subnormals
    ties = f2b([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25] * 4)
    ties[31] = f2b([6.0])[0]
    rows.append(np.tile(ties, 4))
    rows.append(f2b(np.concatenate([np.full(32, 2.0 ** 100), np.full(32, -3e38),
                                    np.full(32, 1.5), np.full(32, 1.5078125)])))
    rows.append(f2b(np.linspace(-7, 7, 128)))
    k = np.stack(rows).astype(np.uint16)
    slots = np.arange(len(rows), dtype=np.int64) * 3
    gc, oc, errs, _ = _insert_both(idx, oracle, k, slots, 1)
    assert np.array_equal(gc, oc)


def test_insert_strided_rows(idx, oracle):
    g = wl.rng(203)
    wide = wl.normal_bf16(g, (300, 192))
    slots = g.permutation(5 * 64)[:300].astype(np.int64)
    kd = dev_bf16(wide)[:, :128]            # a view with row stride 192
    assert kd.stride(0) == 192
    gc, oc, errs, _ = _insert_both(idx, oracle, wide, slots, 5, k_dev=kd)
    assert np.array_equal(gc, oc)


def test_insert_empty_is_noop(idx):
    cache = dev(wl.poisoned_cache(2))
    before = cache.clone()
    idx.quant_insert(torch.empty((0, 128), dtype=torch.bfloat16, device="cuda"),
                     torch.empty(0, dtype=torch.int64, device="cuda"), cache)
    torch.cuda.synchronize()
    assert torch.equal(cache, before)


@pytest.mark.parametrize("rows", [1, 3 * 32, 64 * 2 * 64 + 5, 65536, 65536 * 2 + 77])
def test_quant_q_bit_exact(idx, oracle, rows):
    g = wl.rng(204 + rows)
    q = wl.normal_bf16(g, (rows, 128), wl.outlier_channels(g))
    qv, qs = idx.quant_q(dev_bf16(q))
    ov, os_ = oracle.quant_q(q)
    assert np.array_equal(qv.cpu().numpy(), ov)
    assert np.array_equal(qs.cpu().numpy(), os_)


def test_insert_full_size_batched_decode(idx, oracle):
    """The 64-sequence decode workload at full size: every cache byte equals
    the oracle's (the oracle quantises all 1.3M keys)."""
    p = wl.batched_decode()
    gc, oc, errs, bad = _insert_both(idx, oracle, p.k, p.slots, p.num_blocks)
    assert bad == 0 and errs.tolist() == [0, 0]
    assert np.array_equal(gc, oc)
