"""Runs one step of the path alone on seeded synthetic inputs, a few times,
for a profiler to capture (ncu -k on the step's kernel) and prints its median
CUDA-event time.  Cases:

    prefill T     causal single-sequence prefill of T tokens, H = 32:
                  mqa_logits, then topk_rows (k = 2048) on its logits
    decode        the batched decode workload: the fused paged logits + top-k
    quant T       q-quant of a T-token prefill's query heads (H = 32), then
                  the insert of its T keys into a paged cache

Usage: python -m sparse_attention_indexer_quant_gb300.profile_case prefill 8192
"""
import sys

import numpy as np
import torch

from sparse_attention_indexer_quant_gb300 import binding as idx
from sparse_attention_indexer_quant_gb300 import workloads as wl


def _bf16(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def _time(fn, flush, reps):
    ts = []
    for _ in range(reps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b))
    return sorted(ts)[len(ts) // 2]


def main(argv):
    dev = torch.device("cuda")
    idx.check_device(torch.cuda.current_device())
    buf = torch.empty(64 << 20, dtype=torch.int32, device=dev)  # 256 MiB, twice L2
    sink = torch.empty((), dtype=torch.int64, device=dev)

    def flush():
        buf.fill_(1)
        torch.sum(buf, 0, dtype=torch.int64, out=sink)

    reps = 5
    if argv and argv[0] == "prefill":
        T = int(argv[1]) if len(argv) > 1 else 8192
        p = wl.prefill(T=T)
        S = int(p.tok_offsets[-1])
        cache = torch.from_numpy(wl.poisoned_cache(p.num_blocks)).to(dev)
        idx.quant_insert(_bf16(p.k, dev), torch.from_numpy(p.slots).to(dev), cache)
        kv, ks = idx.gather_k(cache, torch.from_numpy(p.block_table).to(dev),
                              torch.from_numpy(p.new_lens.astype(np.int32)).to(dev),
                              torch.zeros(1, dtype=torch.int64, device=dev), S)
        qv, qs = idx.quant_q(_bf16(p.q, dev))
        w = torch.from_numpy(p.weights).to(dev)
        st, en = p.windows()
        st_d, en_d = torch.from_numpy(st).to(dev), torch.from_numpy(en).to(dev)
        logits = torch.empty((p.T, S), dtype=torch.float32, device=dev)
        out = torch.empty((p.T, 2048), dtype=torch.int32, device=dev)
        ms = _time(lambda: idx.mqa_logits(qv, qs, w, kv, ks, st_d, en_d, p.H, out=logits),
                   flush, reps)
        print(f"prefill T={T}: mqa_logits {ms:.3f} ms")
        ms = _time(lambda: idx.topk_rows(logits, en_d, 2048, row_start=st_d, out=out), flush, reps)
        print(f"prefill T={T}: topk_rows {ms:.3f} ms")
    elif argv and argv[0] == "decode":
        p = wl.batched_decode()
        cache = torch.from_numpy(wl.poisoned_cache(p.num_blocks)).to(dev)
        idx.quant_insert(_bf16(p.k, dev), torch.from_numpy(p.slots).to(dev), cache)
        qv, qs = idx.quant_q(_bf16(p.q, dev))
        w = torch.from_numpy(p.weights).to(dev)
        bt = torch.from_numpy(p.block_table).to(dev)
        cl = torch.from_numpy(p.context_lens).to(dev)
        ws = idx.new_paged_topk_workspace(p.B, p.next_n, p.block_table.shape[1], 2048, dev)
        out = torch.empty((p.rows, 2048), dtype=torch.int32, device=dev)
        ms = _time(lambda: idx.paged_logits_topk(qv, qs, w, cache, bt, cl, p.next_n, p.H, 2048,
                                                 workspace=ws, out=out), flush, reps)
        print(f"batched decode: paged_logits_topk {ms * 1e3:.1f} us")
    elif argv and argv[0] == "quant":
        T = int(argv[1]) if len(argv) > 1 else 32768
        p = wl.prefill(T=T)
        q = _bf16(p.q, dev)
        qv, qs = idx.quant_q(q)
        ms = _time(lambda: idx.quant_q(q, out_vals=qv, out_scales=qs), flush, reps)
        print(f"prefill T={T}: quant_q of {T * p.H} rows {ms * 1e3:.1f} us")
        cache = torch.from_numpy(wl.poisoned_cache(p.num_blocks)).to(dev)
        k = _bf16(p.k, dev)
        slots = torch.from_numpy(p.slots).to(dev)
        ms = _time(lambda: idx.quant_insert(k, slots, cache), flush, reps)
        print(f"prefill T={T}: quant_insert of {k.shape[0]} keys {ms * 1e3:.1f} us")
    else:
        print(__doc__)
        return 2
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))
