"""GPU parity, through the C ABI, of the fused q-RoPE + MXFP4 q-quant and the
K-pool compressed insert against the oracle.

The rotary result is an fp32 computation whose rounding decides the codes;
kernel and oracle state the same fp32 operations, so the quantised bytes are
compared bit for bit.  The K-pool pooling (a softmax over the pool) is
compared within a tolerance, and the cache bytes are compared bit for bit
against the oracle's write step applied to the kernel's own pooled fp32
vectors (both sides take the quantisation decision on the same fp32 values),
over the whole cache, with the pool-granular mask rule checked row by row."""
import numpy as np
import pytest
import torch

from sparse_attention_indexer_quant_gb300 import workloads as wl
from idx_testutil import dev, dev_bf16

pytestmark = pytest.mark.gpu

# pooled-vector tolerance, relative to sum_j w_j |k_j| per dimension: the fp32
# softmax (gate + position term rounded once, exp, a sum of at most 128
# terms, one division) stays far inside it
POOL_RTOL = 1e-5


@pytest.fixture(scope="module")
def idx():
    from sparse_attention_indexer_quant_gb300 import binding
    binding.check_device(torch.cuda.current_device())
    return binding


def _table(num_pos, half, base=10000.0):
    i = np.arange(half, dtype=np.float64)
    ang = np.arange(num_pos, dtype=np.float64)[:, None] * base ** (-i / max(half, 1))[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


@pytest.mark.parametrize("T,H,rot_dim", [(1, 32, 64), (37, 32, 64), (300, 64, 128), (5, 32, 0),
                                         (2048, 32, 64), (129, 64, 2)])
def test_rope_quant_q_bit_exact(idx, oracle, T, H, rot_dim):
    g = wl.rng(7000 + T + rot_dim)
    q = wl.normal_bf16(g, (T, H, 128), outliers=wl.outlier_channels(g))
    num_pos = 4096
    cs, sn = _table(num_pos, rot_dim // 2)
    pos = g.integers(0, num_pos, size=T).astype(np.int32)
    errs = idx.new_errors()
    v, s = idx.rope_quant_q(dev_bf16(q), dev(pos), dev(cs) if rot_dim else None,
                            dev(sn) if rot_dim else None, rot_dim, errors=errs)
    torch.cuda.synchronize()
    assert errs.cpu().tolist() == [0, 0]
    ov, osc, _ = oracle.rope_quant_q(q, pos, cs, sn, rot_dim)
    assert np.array_equal(v.cpu().numpy(), ov), "value bytes differ"
    assert np.array_equal(s.cpu().numpy(), osc), "scale bytes differ"


def test_rope_quant_q_identity_table_equals_quant_q(idx):
    q = wl.normal_bf16(wl.rng(7100), (64, 32, 128))
    cs = np.ones((3, 32), np.float32)
    sn = np.zeros((3, 32), np.float32)
    pos = np.arange(64, dtype=np.int32) % 3
    v1, s1 = idx.rope_quant_q(dev_bf16(q), dev(pos), dev(cs), dev(sn), 64)
    v2, s2 = idx.quant_q(dev_bf16(q))
    torch.cuda.synchronize()
    assert torch.equal(v1, v2) and torch.equal(s1, s2)


def test_rope_quant_q_positions_off_the_table_are_skipped(idx, oracle):
    T, H = 10, 32
    q = wl.normal_bf16(wl.rng(7200), (T, H, 128))
    cs, sn = _table(50, 32)
    pos = np.array([0, 49, 50, -1, 3, 7, 100, 2, 2, 1], np.int32)
    errs = idx.new_errors()
    vals = torch.full((T * H, 64), 0x5A, dtype=torch.uint8, device="cuda")
    scl = torch.full((T * H, 4), 0x5A, dtype=torch.uint8, device="cuda")
    idx.rope_quant_q(dev_bf16(q), dev(pos), dev(cs), dev(sn), 64, out_vals=vals, out_scales=scl,
                     errors=errs)
    torch.cuda.synchronize()
    assert errs.cpu().tolist() == [3, 0]
    ok = (pos >= 0) & (pos < 50)
    ov, osc, _ = oracle.rope_quant_q(q[ok], pos[ok], cs, sn, 64)
    v = vals.cpu().numpy().reshape(T, H, 64)
    s = scl.cpu().numpy().reshape(T, H, 4)
    assert np.array_equal(v[ok].reshape(-1, 64), ov) and np.array_equal(s[ok].reshape(-1, 4), osc)
    assert (v[~ok] == 0x5A).all() and (s[~ok] == 0x5A).all()


def test_rope_quant_q_groups_straddling_tokens(idx, oracle):
    """At 65536 rows and more a 16-thread group quantises four consecutive
    head rows; with H = 6 a group's rows can belong to two tokens, each with
    its own table row.  Some positions lie off the table: those tokens'
    rows stay untouched and each such token is counted once."""
    T, H = 11003, 6
    g = wl.rng(7150)
    q = wl.normal_bf16(g, (T, H, 128))
    num_pos = 20000
    cs, sn = _table(num_pos, 32)
    pos = g.integers(0, num_pos, size=T).astype(np.int32)
    bad = g.choice(T, 37, replace=False)
    pos[bad[:20]] = num_pos + g.integers(0, 100, size=20)
    pos[bad[20:]] = -1 - g.integers(0, 100, size=17)
    errs = idx.new_errors()
    vals = torch.full((T * H, 64), 0x5A, dtype=torch.uint8, device="cuda")
    scl = torch.full((T * H, 4), 0x5A, dtype=torch.uint8, device="cuda")
    idx.rope_quant_q(dev_bf16(q), dev(pos), dev(cs), dev(sn), 64, out_vals=vals, out_scales=scl,
                     errors=errs)
    torch.cuda.synchronize()
    assert errs.cpu().tolist() == [37, 0]
    ok = (pos >= 0) & (pos < num_pos)
    ov, osc, _ = oracle.rope_quant_q(q[ok], pos[ok], cs, sn, 64)
    v = vals.cpu().numpy().reshape(T, H, 64)
    sc = scl.cpu().numpy().reshape(T, H, 4)
    assert np.array_equal(v[ok].reshape(-1, 64), ov) and np.array_equal(sc[ok].reshape(-1, 4), osc)
    assert (v[~ok] == 0x5A).all() and (sc[~ok] == 0x5A).all()


def _pool_batch(seed, n, P, pad_front=0, frac_bad=0.0, num_blocks=64):
    """A prefill-like batch: rows in token order, the last row of every
    complete pool (counted from row pad_front) has a distinct slot, the other
    rows -1; optionally some slots past the cache."""
    g = wl.rng(seed)
    k = wl.normal_bf16(g, (n, 128))
    gate = (2.0 * g.standard_normal((n, 128))).astype(np.float32)
    ape = g.standard_normal((P, 128)).astype(np.float32)
    slots = np.full(n, -1, np.int64)
    ends = np.arange(pad_front + P - 1, n, P)
    free = g.permutation(num_blocks * 64)
    slots[ends] = free[:len(ends)]
    if pad_front:  # a completion inside the leading partial pool: dropped
        slots[min(pad_front - 1, n - 1)] = free[len(ends)]
    if frac_bad:
        bad = g.choice(ends, max(1, int(frac_bad * len(ends))), replace=False)
        slots[bad] = num_blocks * 64 + g.integers(0, 1000, size=len(bad))
    return k, gate, ape, slots


@pytest.mark.parametrize("n,P,pad_front", [(1000, 4, 0), (4096, 16, 0), (777, 64, 3),
                                           (130, 128, 0), (333, 1, 0), (3, 4, 0), (4, 4, 0),
                                           (4099, 2, 1), (3001, 3, 2)])
def test_kpool_insert_parity(idx, oracle, n, P, pad_front):
    k, gate, ape, slots = _pool_batch(7300 + n + P, n, P, pad_front)
    cache = dev(wl.poisoned_cache(64))
    pooled = torch.full((n, 128), float("nan"), dtype=torch.float32, device="cuda")
    errs = idx.new_errors()
    idx.kpool_insert(dev_bf16(k), dev(gate), dev(ape), dev(slots), cache, pooled=pooled,
                     errors=errs)
    torch.cuda.synchronize()
    assert errs.cpu().tolist() == [0, 0]
    kc, mag = oracle.kpool_compress(k, gate, ape, slots, P)
    got = pooled.cpu().numpy()
    written = ~np.isnan(kc[:, 0])
    # exactly the rows the mask rule writes carry a pooled vector
    assert np.array_equal(~np.isnan(got[:, 0]), written)
    err = np.abs(got[written].astype(np.float64) - kc[written])
    assert (err <= POOL_RTOL * mag[written] + 1e-30).all(), float((err / mag[written]).max())
    ocache = wl.poisoned_cache(64)
    assert oracle.kpool_insert(got, slots, P, ocache) == 0
    assert np.array_equal(cache.cpu().numpy(), ocache), "cache bytes differ"


def test_kpool_insert_bad_slots_counted_and_skipped(idx, oracle):
    n, P = 2000, 8
    k, gate, ape, slots = _pool_batch(7400, n, P, frac_bad=0.1)
    cache = dev(wl.poisoned_cache(64))
    errs = idx.new_errors()
    idx.kpool_insert(dev_bf16(k), dev(gate), dev(ape), dev(slots), cache, errors=errs)
    torch.cuda.synchronize()
    n_bad = int((slots >= 64 * 64).sum())
    assert errs.cpu().tolist() == [n_bad, 0]
    pooled = torch.zeros((n, 128), dtype=torch.float32, device="cuda")
    cache2 = dev(wl.poisoned_cache(64))
    idx.kpool_insert(dev_bf16(k), dev(gate), dev(ape), dev(slots), cache2, pooled=pooled)
    torch.cuda.synchronize()
    assert torch.equal(cache, cache2)
    ocache = wl.poisoned_cache(64)
    assert oracle.kpool_insert(pooled.cpu().numpy(), slots, P, ocache) == n_bad
    assert np.array_equal(cache.cpu().numpy(), ocache)


def test_kpool_of_one_equals_quant_insert(idx):
    n = 5000
    g = wl.rng(7500)
    k = wl.normal_bf16(g, (n, 128))
    slots = g.permutation(64 * 100)[:n].astype(np.int64)
    slots[g.choice(n, 500, replace=False)] = -1
    c1 = dev(wl.poisoned_cache(100))
    c2 = dev(wl.poisoned_cache(100))
    idx.kpool_insert(dev_bf16(k), dev(g.standard_normal((n, 128)).astype(np.float32)),
                     dev(np.zeros((1, 128), np.float32)), dev(slots), c1)
    idx.quant_insert(dev_bf16(k), dev(slots), c2)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)
