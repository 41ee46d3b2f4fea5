"""Helpers shared by the GPU parity tests: device transfer of seeded inputs and
the comparison rules.

Comparison rules (the tolerance the indexer's logits are held to):
  - cache bytes, quantised q, gathered keys: bit-exact;
  - logits: |gpu - oracle| <= 1e-5 * sum_h |w_h| * sum_d |q^_hd * k^_d| per
    element (the oracle returns that magnitude beside each logit);
  - top-k: no duplicates, every index in range, -1 exactly in the slots past
    the window length, and every index in the symmetric difference between the
    GPU set and the oracle set lies within the tolerance of the oracle's k-th
    value (several answers are right when values tie within the tolerance).
"""
import numpy as np
import torch

LOGIT_RTOL = 1e-5


def dev_bf16(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def check_logits(gpu_row: np.ndarray, ref_row: np.ndarray, mag_row: np.ndarray, what=""):
    g = gpu_row.astype(np.float64)
    err = np.abs(g - ref_row)
    tol = LOGIT_RTOL * mag_row
    bad = ~(err <= tol)
    if bad.any():
        i = int(np.nonzero(bad)[0][0])
        raise AssertionError(f"{what}: {int(bad.sum())} logits out of tolerance; first at col {i}: "
                             f"gpu {g[i]!r} oracle {ref_row[i]!r} tol {tol[i]!r}")


def check_topk(gpu_idx: np.ndarray, ref_logits: np.ndarray, mag: np.ndarray, n_valid: int, k: int,
               what=""):
    """gpu_idx: [k] int32 (positions relative to the window start); ref_logits,
    mag: oracle fp64 values over the window [0, n_valid)."""
    g = gpu_idx.astype(np.int64)
    m = min(k, n_valid)
    assert (g[m:] == -1).all(), f"{what}: expected -1 past slot {m}"
    sel = g[:m]
    assert ((sel >= 0) & (sel < n_valid)).all(), f"{what}: index out of range"
    assert len(np.unique(sel)) == m, f"{what}: duplicate indices"
    if n_valid <= k:
        return
    order = np.lexsort((np.arange(n_valid), -ref_logits[:n_valid]))
    ref_set = set(order[:k].tolist())
    vk = ref_logits[order[k - 1]]
    tol = LOGIT_RTOL * mag
    diff = set(sel.tolist()) ^ ref_set
    for i in diff:
        if ref_logits[i] == vk:
            continue
        if abs(ref_logits[i] - vk) > tol[i] + tol[order[k - 1]]:
            raise AssertionError(f"{what}: index {i} (logit {ref_logits[i]!r}) differs from the "
                                 f"oracle set beyond tolerance (k-th value {vk!r})")
