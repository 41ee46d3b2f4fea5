"""Seeded synthetic inputs for the indexer path.

This module only draws and lays out inputs: random bf16 keys and queries,
weights, context lengths, shuffled block tables, slot mappings and poisoned
cache buffers.  It holds none of the method's arithmetic (no quantisation, no
logits, no selection), so both the CUDA path and the CPU oracle can take their
inputs from it.

Shapes follow the workloads that the pages describe: 32 or 64 index heads,
head_dim 128, page size 64, contexts of 8K-131K tokens and top-k 2048
(vLLM PR #48558, sections "Benefit" and "Notes"; vLLM API docs for
``sparse_indexer``, ``SparseAttnIndexerKpool.__init__`` topk_tokens).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

HEAD_DIM = 128
PAGE_SIZE = 64
VAL_BYTES = 64
SCALE_BYTES = 4
TOKEN_BYTES = VAL_BYTES + SCALE_BYTES
TOPK = 2048
VALUE_POISON = 0xA5
SCALE_POISON = 0xFF


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to the nearest bf16 (ties to even) and return the 16-bit
    patterns as uint16.  Inputs must be finite."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def outlier_channels(g: np.random.Generator, frac: float = 0.01) -> np.ndarray:
    """ceil(frac * 128) seeded channel indices (the same set for K and q)."""
    n = int(math.ceil(frac * HEAD_DIM))
    return np.sort(g.choice(HEAD_DIM, size=n, replace=False))


def normal_bf16(g: np.random.Generator, shape, outliers=None, gain: float = 8.0,
                chunk: int = 1 << 22) -> np.ndarray:
    """N(0,1) draws rounded to bf16 (uint16 bit patterns); the listed channels
    of the last axis are multiplied by ``gain`` before rounding."""
    shape = tuple(int(s) for s in shape)
    total = int(np.prod(shape)) if shape else 1
    out = np.empty(total, np.uint16)
    for lo in range(0, total, chunk):
        hi = min(total, lo + chunk)
        x = g.standard_normal(hi - lo, dtype=np.float32)
        if outliers is not None and len(outliers):
            x = x.reshape(-1, shape[-1])
            x[:, outliers] *= np.float32(gain)
            x = x.reshape(-1)
        out[lo:hi] = bf16_bits(x)
    return out.reshape(shape)


def head_weights(g: np.random.Generator, rows: int, H: int) -> np.ndarray:
    """Per-row, per-head gate weights ~ N(0,1)/sqrt(H), fp32 [rows, H]."""
    return (g.standard_normal((rows, H), dtype=np.float32) / np.float32(math.sqrt(H))).astype(
        np.float32)


def poisoned_cache(num_blocks: int, page_size: int = PAGE_SIZE) -> np.ndarray:
    """A paged cache [num_blocks, page_size*68] filled with poison: 0xA5 in the
    value area and 0xFF (a NaN E8M0 scale) in the scale area of every page."""
    c = np.empty((num_blocks, page_size * TOKEN_BYTES), np.uint8)
    c[:, :page_size * VAL_BYTES] = VALUE_POISON
    c[:, page_size * VAL_BYTES:] = SCALE_POISON
    return c


def shuffled_block_table(g: np.random.Generator, context_lens, page_size: int = PAGE_SIZE,
                         pool_factor: float = 1.25, max_blocks: int | None = None):
    """Block table for sequences of the given lengths, drawn from a page pool
    of ceil(pool_factor * pages needed) pages taken in a seeded permuted order,
    so no table is contiguous.  Unused entries are -1.

    Returns (block_table int32 [B, max_blocks], num_blocks)."""
    lens = np.asarray(context_lens, np.int64)
    pages = (lens + page_size - 1) // page_size
    need = int(pages.sum())
    num_blocks = max(1, int(math.ceil(pool_factor * max(need, 1))))
    if max_blocks is None:
        max_blocks = max(1, int(pages.max()) if len(pages) else 1)
    perm = g.permutation(num_blocks).astype(np.int32)
    bt = np.full((len(lens), max_blocks), -1, np.int32)
    pos = 0
    for b, p in enumerate(pages):
        bt[b, :p] = perm[pos:pos + p]
        pos += int(p)
    return bt, num_blocks


def slots_of(block_table: np.ndarray, b: int, positions, page_size: int = PAGE_SIZE) -> np.ndarray:
    """Cache slot (page id * page_size + offset) of token positions of sequence b."""
    pos = np.asarray(positions, np.int64)
    return block_table[b, pos // page_size].astype(np.int64) * page_size + pos % page_size


@dataclasses.dataclass
class DecodeProblem:
    """A batch of decode sequences with their cached keys.

    Sequence b holds context_lens[b] tokens (the next_n newest included), whose
    bf16 keys are rows [tok_offsets[b], tok_offsets[b] + context_lens[b]) of
    ``k``; ``slots`` gives each row's cache slot.  Query row r = b*next_n + j."""
    name: str
    B: int
    next_n: int
    H: int
    page_size: int
    context_lens: np.ndarray      # int32 [B]
    block_table: np.ndarray       # int32 [B, max_blocks]
    num_blocks: int
    k: np.ndarray                 # uint16 bf16 bits [total_tokens, 128]
    tok_offsets: np.ndarray       # int64 [B+1]
    slots: np.ndarray             # int64 [total_tokens]
    q: np.ndarray                 # uint16 bf16 bits [B*next_n, H, 128]
    weights: np.ndarray           # fp32 [B*next_n, H]
    topk: int = TOPK

    @property
    def rows(self) -> int:
        return self.B * self.next_n

    @property
    def total_tokens(self) -> int:
        return int(self.tok_offsets[-1])

    def new_token_rows(self) -> np.ndarray:
        """Rows of ``k`` holding each sequence's next_n newest tokens (those a
        decode step inserts)."""
        idx = []
        for b in range(self.B):
            hi = int(self.tok_offsets[b + 1])
            lo = max(int(self.tok_offsets[b]), hi - self.next_n)
            idx.extend(range(lo, hi))
        return np.asarray(idx, np.int64)

    def row_windows(self):
        """(start, end) per query row: row (b, j) sees [0, L_b - next_n + j + 1)."""
        L = self.context_lens.astype(np.int64)
        j = np.arange(self.next_n)
        end = (L[:, None] - self.next_n + j[None, :] + 1).reshape(-1)
        end = np.maximum(end, 0).astype(np.int32)
        return np.zeros_like(end), end


def make_decode(name: str, seed: int, context_lens, H: int, next_n: int,
                outliers: bool = False, page_size: int = PAGE_SIZE,
                max_blocks: int | None = None, topk: int = TOPK) -> DecodeProblem:
    g = rng(seed)
    lens = np.asarray(context_lens, np.int32)
    B = len(lens)
    oc = outlier_channels(g) if outliers else None
    bt, num_blocks = shuffled_block_table(g, lens, page_size, max_blocks=max_blocks)
    offs = np.zeros(B + 1, np.int64)
    offs[1:] = np.cumsum(lens.astype(np.int64))
    k = normal_bf16(g, (int(offs[-1]), HEAD_DIM), oc)
    slots = np.empty(int(offs[-1]), np.int64)
    for b in range(B):
        slots[offs[b]:offs[b + 1]] = slots_of(bt, b, np.arange(lens[b]), page_size)
    q = normal_bf16(g, (B * next_n, H, HEAD_DIM), oc)
    w = head_weights(g, B * next_n, H)
    return DecodeProblem(name, B, next_n, H, page_size, lens, bt, num_blocks, k, offs, slots,
                         q, w, topk)


# The five workloads.  Each function takes the sizes as arguments so tests can
# build scaled-down instances of the same recipe.

def pr_ref(seed: int = 1001, L: int = 8192, H: int = 32) -> DecodeProblem:
    """One sequence of L tokens, one decode query, H index heads."""
    return make_decode("pr_ref", seed, [L], H, 1)


def batched_decode(seed: int = 1002, B: int = 64, lo: int = 8192, hi: int = 32768,
                   H: int = 32) -> DecodeProblem:
    """B sequences with context lengths uniform in [lo, hi], 1% outlier
    channels x8 in K and q, next_n = 1."""
    g = rng(seed + 7919)
    lens = g.integers(lo, hi + 1, size=B)
    return make_decode("batched_decode", seed, lens, H, 1, outliers=True)


def long_decode(seed: int = 1003, B: int = 16, L: int = 131072, H: int = 64,
                next_n: int = 2) -> DecodeProblem:
    """B sequences of L tokens each, H = 64 index heads, two query tokens per
    sequence."""
    return make_decode("long_decode", seed, [L] * B, H, next_n)


@dataclasses.dataclass
class PrefillProblem:
    """Chunked prefill: sequence b has a cached prefix of prefix_lens[b] tokens
    and adds new_lens[b] tokens; query rows are the new tokens, in sequence
    order.  ``k`` holds every token of every sequence (prefix first)."""
    name: str
    H: int
    page_size: int
    prefix_lens: np.ndarray       # int32 [B]
    new_lens: np.ndarray          # int32 [B]
    block_table: np.ndarray
    num_blocks: int
    k: np.ndarray                 # uint16 [total_tokens, 128]
    tok_offsets: np.ndarray       # int64 [B+1]
    slots: np.ndarray             # int64 [total_tokens]
    q: np.ndarray                 # uint16 [T, H, 128]
    weights: np.ndarray           # fp32 [T, H]
    topk: int = TOPK

    @property
    def B(self) -> int:
        return len(self.prefix_lens)

    @property
    def T(self) -> int:
        return int(self.new_lens.sum())

    def windows(self):
        """Key window of each query row in the contiguous gathered key buffer,
        where sequence b's tokens occupy [tok_offsets[b], tok_offsets[b+1]):
        new token t of sequence b sees [tok_offsets[b], tok_offsets[b] +
        prefix_lens[b] + t + 1) (causal)."""
        st, en = [], []
        for b in range(self.B):
            base = int(self.tok_offsets[b])
            P = int(self.prefix_lens[b])
            t = np.arange(int(self.new_lens[b]))
            st.append(np.full(len(t), base, np.int64))
            en.append(base + P + t + 1)
        return (np.concatenate(st).astype(np.int32), np.concatenate(en).astype(np.int32))


def make_prefill(name: str, seed: int, prefix_lens, new_lens, H: int,
                 page_size: int = PAGE_SIZE, topk: int = TOPK,
                 with_queries: bool = True) -> PrefillProblem:
    g = rng(seed)
    P = np.asarray(prefix_lens, np.int32)
    N = np.asarray(new_lens, np.int32)
    lens = P.astype(np.int64) + N
    bt, num_blocks = shuffled_block_table(g, lens, page_size)
    offs = np.zeros(len(P) + 1, np.int64)
    offs[1:] = np.cumsum(lens)
    k = normal_bf16(g, (int(offs[-1]), HEAD_DIM))
    slots = np.empty(int(offs[-1]), np.int64)
    for b in range(len(P)):
        slots[offs[b]:offs[b + 1]] = slots_of(bt, b, np.arange(lens[b]), page_size)
    T = int(N.sum())
    # the queries are drawn after the keys, so leaving them out (an insert
    # needs only the keys) changes nothing else
    if with_queries:
        q = normal_bf16(g, (T, H, HEAD_DIM))
        w = head_weights(g, T, H)
    else:
        q = np.zeros((0, H, HEAD_DIM), np.uint16)
        w = np.zeros((0, H), np.float32)
    return PrefillProblem(name, H, page_size, P, N, bt, num_blocks, k, offs, slots, q, w, topk)


def prefill(seed: int = 1004, T: int = 32768, H: int = 32) -> PrefillProblem:
    """One sequence of T new tokens, no cached prefix: the causal T x T case."""
    return make_prefill("prefill", seed, [0], [T], H)


def mixed_prefill_part(seed: int = 1005, B: int = 8, new: int = 8192, max_prefix: int = 65536,
                       H: int = 32, with_queries: bool = True) -> PrefillProblem:
    """The chunked-prefill half of the mixed batch: B sequences with prefixes
    uniform in [0, max_prefix], each adding ``new`` tokens."""
    g = rng(seed + 104729)
    P = g.integers(0, max_prefix + 1, size=B)
    return make_prefill("mixed_prefill", seed, P, [new] * B, H, with_queries=with_queries)


def mixed_decode_part(seed: int = 1006, B: int = 128, lo: int = 1024, hi: int = 131072,
                      H: int = 32) -> DecodeProblem:
    """The decode half of the mixed batch: B sequences with contexts uniform in
    [lo, hi], next_n = 1."""
    g = rng(seed + 15485863)
    lens = g.integers(lo, hi + 1, size=B)
    return make_decode("mixed_decode", seed, lens, H, 1)


def with_padding(g: np.random.Generator, slots: np.ndarray, frac: float = 0.05):
    """Insert round(frac * n) extra -1 (padding) rows at seeded positions.
    Returns (padded slots, index of each original row in the padded batch)."""
    n = len(slots)
    n_pad = int(round(frac * n))
    total = n + n_pad
    pad_pos = np.sort(g.choice(total, size=n_pad, replace=False))
    is_pad = np.zeros(total, bool)
    is_pad[pad_pos] = True
    out = np.full(total, -1, np.int64)
    real_pos = np.nonzero(~is_pad)[0]
    out[real_pos] = slots
    return out, real_pos


@dataclasses.dataclass
class InsertBatch:
    """One insert batch into a paged cache, with the keys the cache must
    already hold (``pre_k`` at ``pre_slots``).  ``slots`` holds -1 for the
    padding rows; their keys are drawn like the others but never written."""
    name: str
    num_blocks: int
    pre_k: np.ndarray             # uint16 [n_pre, 128]
    pre_slots: np.ndarray         # int64 [n_pre]
    k: np.ndarray                 # uint16 [n, 128]
    slots: np.ndarray             # int64 [n]

    @property
    def real_rows(self) -> int:
        return int((self.slots >= 0).sum())


def mixed_insert_batch(seed: int = 1007, frac_pad: float = 0.05, prefill_seed: int = 1005,
                       decode_seed: int = 1006, B_prefill: int = 8, new: int = 8192,
                       max_prefix: int = 65536, B_decode: int = 128, lo: int = 1024,
                       hi: int = 131072) -> InsertBatch:
    """The insert batch of the mixed chunked-prefill + decode step: the new
    tokens of the chunked prefills (each sequence's ``new`` tokens after its
    cached prefix) and one new token per decode sequence (at the end of its
    context), plus round(frac_pad * n) padding rows (slot -1) at seeded
    positions.  Both halves share one cache: the prefill half's pages first,
    then the decode half's (the same page pools and block tables as
    ``mixed_prefill_part`` and ``mixed_decode_part``).  The prefills' cached
    prefixes are the keys the cache holds before the batch.  The decode
    tokens' keys are fresh N(0,1) rows: the decode contexts themselves are
    not needed for an insert."""
    pp = mixed_prefill_part(seed=prefill_seed, B=B_prefill, new=new, max_prefix=max_prefix,
                            with_queries=False)
    gl = rng(decode_seed + 15485863)
    lens = gl.integers(lo, hi + 1, size=B_decode)
    dbt, d_blocks = shuffled_block_table(rng(decode_seed), lens)
    pre_rows, new_rows = [], []
    for b in range(pp.B):
        base, P = int(pp.tok_offsets[b]), int(pp.prefix_lens[b])
        pre_rows.append(np.arange(base, base + P))
        new_rows.append(np.arange(base + P, int(pp.tok_offsets[b + 1])))
    pre_rows = np.concatenate(pre_rows)
    new_rows = np.concatenate(new_rows)
    d_slots = np.array([slots_of(dbt, b, [int(lens[b]) - 1])[0] for b in range(B_decode)],
                       np.int64) + pp.num_blocks * PAGE_SIZE
    g = rng(seed)
    d_k = normal_bf16(g, (B_decode, HEAD_DIM))
    real_slots = np.concatenate([pp.slots[new_rows], d_slots])
    real_k = np.concatenate([pp.k[new_rows], d_k])
    slots, real_pos = with_padding(g, real_slots, frac_pad)
    k = normal_bf16(g, (len(slots), HEAD_DIM))
    k[real_pos] = real_k
    return InsertBatch("mixed_insert", pp.num_blocks + d_blocks, pp.k[pre_rows],
                       pp.slots[pre_rows], k, slots)
