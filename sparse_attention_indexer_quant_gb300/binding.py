"""Thin PyTorch binding of libidx (include/idx.h).

Every function checks tensor dtypes, devices and shapes, then passes raw
device pointers and the current CUDA stream to the C entry point of the same
name.  All arithmetic happens in the library's kernels; if the library is
missing the import fails loudly (there is no fallback).
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libidx.so")

IDX_OK = 0
STATUS_NAMES = {0: "IDX_OK", 1: "IDX_ERR_INVALID_ARG", 2: "IDX_ERR_UNSUPPORTED_DEVICE",
                3: "IDX_ERR_WORKSPACE_TOO_SMALL", 4: "IDX_ERR_CUDA"}
HEAD_DIM = 128
PAGE_SIZE = 64
PAGE_BYTES = PAGE_SIZE * 68

# Every symbol include/idx.h declares, with (restype, argtypes).
_P = ctypes.c_void_p
_I64, _I32, _SZ = ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
SIGNATURES = {
    "idx_version": (ctypes.c_int, []),
    "idx_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "idx_last_error_detail": (ctypes.c_char_p, []),
    "idx_arch_supported": (ctypes.c_int, [ctypes.c_int, ctypes.c_int]),
    "idx_check_device": (ctypes.c_int, [ctypes.c_int]),
    "idx_quant_insert": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _I64, _I32, _P, _P]),
    "idx_quant_q": (ctypes.c_int, [_P, _I64, _P, _P, _P]),
    "idx_paged_mqa_logits": (ctypes.c_int, [_P, _P, _I32, _I32, _I32, _P, _I64, _I32, _P, _I32,
                                            _P, _P, _P, _I64, ctypes.c_int, _P, _P]),
    "idx_mqa_logits": (ctypes.c_int, [_P, _P, _I64, _I32, _P, _P, _I64, _P, _P, _P, _P, _I64,
                                      ctypes.c_int, _P, _P]),
    "idx_topk_rows": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _I32, _P, _P]),
    "idx_paged_logits_topk_workspace_bytes": (_SZ, [_I32, _I32, _I32, _I32, _I32]),
    "idx_paged_logits_topk": (ctypes.c_int, [_P, _P, _I32, _I32, _I32, _P, _I64, _I32, _P, _I32,
                                             _P, _P, _I32, _P, _P, _SZ, _P, _P]),
    "idx_gather_k": (ctypes.c_int, [_P, _I64, _I32, _P, _I32, _P, _P, _I32, _P, _P, _I64, _P,
                                    _P]),
    "idx_paged_logits_topk_noalloc": (ctypes.c_int, [_P, _P, _I32, _I32, _I32, _P, _I64, _I32, _P,
                                                     _I32, _P, _P, _I32, _P, _P, _P]),
    "idx_paged_decode_step_workspace_bytes": (_SZ, [_I32, _I32, _I32, _I32, _I32, _I32]),
    "idx_paged_decode_step": (ctypes.c_int, [_P, _P, _I32, _I32, _I32, _P, _I64, _I32, _P, _I32,
                                             _P, _P, _I32, _P, _P, _SZ, _P, _P]),
    "idx_mqa_logits_topk_workspace_bytes": (_SZ, [_I64, _I64, _I32]),
    "idx_mqa_logits_topk": (ctypes.c_int, [_P, _P, _I64, _I32, _P, _P, _I64, _P, _P, _P, _I32, _P,
                                           _P, _SZ, _P, _P]),
    "idx_rope_quant_q": (ctypes.c_int, [_P, _I64, _I32, _P, _P, _P, _I32, _I32, _P, _P, _P, _P]),
    "idx_kpool_insert": (ctypes.c_int, [_P, _P, _P, _P, _I64, _I32, _P, _I64, _I32, _P, _P, _P]),
    "idx_copy_async": (ctypes.c_int, [_P, _P, _SZ, _P]),
}


class IdxError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str):
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)}: {detail}")
        self.status = status
        self.detail = detail


def load_library(path: str = LIB_PATH):
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: the CUDA library must be built first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = load_library()


def _check(fn: str, status: int):
    if status != IDX_OK:
        raise IdxError(fn, status, lib.idx_last_error_detail().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, dtype, name, contiguous=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def new_errors(device=None) -> torch.Tensor:
    """A zeroed idx_device_errors struct: int32 [bad_inputs, timeouts]."""
    return torch.zeros(2, dtype=torch.int32, device=device or "cuda")


def arch_supported(major: int, minor: int) -> bool:
    return lib.idx_arch_supported(major, minor) == IDX_OK


def check_device(device: int = 0) -> None:
    _check("idx_check_device", lib.idx_check_device(device))


def new_cache(num_blocks: int, device=None) -> torch.Tensor:
    return torch.zeros((num_blocks, PAGE_BYTES), dtype=torch.uint8, device=device or "cuda")


def quant_insert(k: torch.Tensor, slot_mapping: torch.Tensor, kcache: torch.Tensor,
                 errors: torch.Tensor | None = None, stream=None) -> None:
    """Quantise k ([N, >=128] bf16, row-major, rows may be strided) to MXFP4 and
    scatter into kcache ([num_blocks, 4352] uint8) at slot_mapping ([N] int64)."""
    _need(k, torch.bfloat16, "k", contiguous=False)
    _need(slot_mapping, torch.int64, "slot_mapping")
    _need(kcache, torch.uint8, "kcache")
    if k.dim() != 2 or k.stride(1) != 1 or k.shape[1] < HEAD_DIM:
        raise ValueError("k must be [N, >=128] with unit stride in the last dim")
    n = k.shape[0]
    if slot_mapping.numel() != n:
        raise ValueError("slot_mapping must have one entry per row of k")
    if kcache.dim() != 2 or kcache.shape[1] != PAGE_BYTES:
        raise ValueError("kcache must be [num_blocks, 4352]")
    stride = k.stride(0) if n > 1 else max(k.stride(0), HEAD_DIM)
    _check("idx_quant_insert", lib.idx_quant_insert(
        _ptr(k), n, stride, _ptr(slot_mapping), _ptr(kcache), kcache.shape[0], PAGE_SIZE,
        _ptr(errors), _stream(stream)))


def quant_q(q: torch.Tensor, out_vals=None, out_scales=None, stream=None):
    """q [..., 128] bf16 -> (vals [rows, 64] uint8, scales [rows, 4] uint8)."""
    _need(q, torch.bfloat16, "q")
    if q.shape[-1] != HEAD_DIM:
        raise ValueError("q must end in 128")
    rows = q.numel() // HEAD_DIM
    vals = out_vals if out_vals is not None else torch.empty((rows, 64), dtype=torch.uint8,
                                                             device=q.device)
    scales = out_scales if out_scales is not None else torch.empty((rows, 4), dtype=torch.uint8,
                                                                   device=q.device)
    _check("idx_quant_q", lib.idx_quant_q(_ptr(q), rows, _ptr(vals), _ptr(scales),
                                          _stream(stream)))
    return vals, scales


def rope_quant_q(q: torch.Tensor, positions: torch.Tensor, cos: torch.Tensor | None,
                 sin: torch.Tensor | None, rot_dim: int, out_vals=None, out_scales=None,
                 errors=None, stream=None):
    """Rotary embedding of q ([T, H, 128] bf16) by table rows positions ([T]
    int32) of cos/sin ([num_pos, rot_dim/2] fp32), fused with the MXFP4
    quantisation: (vals [T*H, 64] uint8, scales [T*H, 4] uint8)."""
    _need(q, torch.bfloat16, "q")
    _need(positions, torch.int32, "positions")
    if q.dim() != 3 or q.shape[2] != HEAD_DIM:
        raise ValueError("q must be [T, H, 128]")
    T, H = q.shape[0], q.shape[1]
    if positions.numel() != T:
        raise ValueError("positions must have one entry per token")
    num_pos = 0
    if rot_dim > 0:
        _need(cos, torch.float32, "cos")
        _need(sin, torch.float32, "sin")
        if cos.shape != sin.shape or cos.dim() != 2 or cos.shape[1] != rot_dim // 2:
            raise ValueError("cos/sin must be [num_pos, rot_dim / 2]")
        num_pos = cos.shape[0]
    rows = T * H
    vals = out_vals if out_vals is not None else torch.empty((rows, 64), dtype=torch.uint8,
                                                             device=q.device)
    scales = out_scales if out_scales is not None else torch.empty((rows, 4), dtype=torch.uint8,
                                                                   device=q.device)
    _check("idx_rope_quant_q", lib.idx_rope_quant_q(
        _ptr(q), T, H, _ptr(positions), _ptr(cos) if rot_dim > 0 else None,
        _ptr(sin) if rot_dim > 0 else None, num_pos, rot_dim, _ptr(vals), _ptr(scales),
        _ptr(errors), _stream(stream)))
    return vals, scales


def kpool_insert(k: torch.Tensor, gate: torch.Tensor, ape: torch.Tensor,
                 slot_mapping: torch.Tensor, kcache: torch.Tensor, pooled=None, errors=None,
                 stream=None) -> None:
    """K-pool compressed insert: pools of kpool = ape.shape[0] keys of k
    ([n, 128] bf16) weighted by a softmax of gate ([n, 128] fp32) plus ape
    ([kpool, 128] fp32), written as MXFP4 keys at the pool-granular
    slot_mapping ([n] int64) of kcache; pooled ([n, 128] fp32, optional)
    receives the pooled vectors of the written rows."""
    _need(k, torch.bfloat16, "k")
    _need(gate, torch.float32, "gate")
    _need(ape, torch.float32, "ape")
    _need(slot_mapping, torch.int64, "slot_mapping")
    _need(kcache, torch.uint8, "kcache")
    n = k.shape[0]
    if k.dim() != 2 or k.shape[1] != HEAD_DIM or gate.shape != k.shape:
        raise ValueError("k and gate must be [n, 128]")
    if ape.dim() != 2 or ape.shape[1] != HEAD_DIM or slot_mapping.numel() != n:
        raise ValueError("ape must be [kpool, 128] and slot_mapping [n]")
    if pooled is not None:
        _need(pooled, torch.float32, "pooled")
        if pooled.shape != k.shape:
            raise ValueError("pooled must be [n, 128]")
    _check("idx_kpool_insert", lib.idx_kpool_insert(
        _ptr(k), _ptr(gate), _ptr(ape), _ptr(slot_mapping), n, ape.shape[0], _ptr(kcache),
        kcache.shape[0], PAGE_SIZE, _ptr(pooled), _ptr(errors), _stream(stream)))


def _paged_common(q_vals, q_scales, weights, kcache, block_table, context_lens, next_n, H):
    _need(q_vals, torch.uint8, "q_vals")
    _need(q_scales, torch.uint8, "q_scales")
    _need(weights, torch.float32, "weights")
    _need(kcache, torch.uint8, "kcache")
    _need(block_table, torch.int32, "block_table")
    _need(context_lens, torch.int32, "context_lens")
    B = context_lens.numel()
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [B, max_blocks]")
    if weights.numel() != B * next_n * H or q_vals.numel() != B * next_n * H * 64:
        raise ValueError("q/weights do not match B * next_n * H")
    return B, block_table.shape[1]


def paged_mqa_logits(q_vals, q_scales, weights, kcache, block_table, context_lens, next_n: int,
                     H: int, ld: int | None = None, clean: bool = False, out=None, errors=None,
                     stream=None):
    B, max_blocks = _paged_common(q_vals, q_scales, weights, kcache, block_table, context_lens,
                                  next_n, H)
    if ld is None:
        ld = max_blocks * PAGE_SIZE
    logits = out if out is not None else torch.empty((B * next_n, ld), dtype=torch.float32,
                                                     device=q_vals.device)
    _check("idx_paged_mqa_logits", lib.idx_paged_mqa_logits(
        _ptr(q_vals), _ptr(q_scales), B, next_n, H, _ptr(kcache), kcache.shape[0], PAGE_SIZE,
        _ptr(block_table), max_blocks, _ptr(context_lens), _ptr(weights), _ptr(logits), ld,
        1 if clean else 0, _ptr(errors), _stream(stream)))
    return logits


def paged_logits_topk_workspace_bytes(B: int, next_n: int, max_blocks: int, k: int) -> int:
    return int(lib.idx_paged_logits_topk_workspace_bytes(B, next_n, max_blocks, PAGE_SIZE, k))


def new_paged_topk_workspace(B: int, next_n: int, max_blocks: int, k: int, device=None):
    n = paged_logits_topk_workspace_bytes(B, next_n, max_blocks, k)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device or "cuda")


def paged_logits_topk(q_vals, q_scales, weights, kcache, block_table, context_lens, next_n: int,
                      H: int, k: int = 2048, workspace=None, out=None, errors=None, stream=None):
    B, max_blocks = _paged_common(q_vals, q_scales, weights, kcache, block_table, context_lens,
                                  next_n, H)
    if workspace is None:
        workspace = new_paged_topk_workspace(B, next_n, max_blocks, k, q_vals.device)
    _need(workspace, torch.uint8, "workspace")
    idx = out if out is not None else torch.empty((B * next_n, k), dtype=torch.int32,
                                                  device=q_vals.device)
    _check("idx_paged_logits_topk", lib.idx_paged_logits_topk(
        _ptr(q_vals), _ptr(q_scales), B, next_n, H, _ptr(kcache), kcache.shape[0], PAGE_SIZE,
        _ptr(block_table), max_blocks, _ptr(context_lens), _ptr(weights), k, _ptr(idx),
        _ptr(workspace), workspace.numel(), _ptr(errors), _stream(stream)))
    return idx


def paged_logits_topk_noalloc(q_vals, q_scales, weights, kcache, block_table, context_lens,
                              next_n: int, H: int, k: int = 2048, out=None, errors=None,
                              stream=None):
    """idx_paged_logits_topk_noalloc: the fused decode path with the library's
    built-in 32 MiB scratch instead of a caller workspace (for callers that
    cannot allocate device memory)."""
    B, max_blocks = _paged_common(q_vals, q_scales, weights, kcache, block_table, context_lens,
                                  next_n, H)
    idx = out if out is not None else torch.empty((B * next_n, k), dtype=torch.int32,
                                                  device=q_vals.device)
    _check("idx_paged_logits_topk_noalloc", lib.idx_paged_logits_topk_noalloc(
        _ptr(q_vals), _ptr(q_scales), B, next_n, H, _ptr(kcache), kcache.shape[0], PAGE_SIZE,
        _ptr(block_table), max_blocks, _ptr(context_lens), _ptr(weights), k, _ptr(idx),
        _ptr(errors), _stream(stream)))
    return idx


def paged_decode_step_workspace_bytes(B: int, next_n: int, H: int, max_blocks: int,
                                      k: int) -> int:
    return int(lib.idx_paged_decode_step_workspace_bytes(B, next_n, H, max_blocks, PAGE_SIZE, k))


def paged_decode_step(k_new, q, weights, kcache, block_table, context_lens, next_n: int, H: int,
                      k: int = 2048, workspace=None, out=None, errors=None, stream=None):
    """One decode step: insert the step's new keys (k_new [B*next_n, 128] bf16,
    at positions L_b - next_n + j through the block table), quantise its query
    heads (q [B*next_n, H, 128] bf16) and return the top-k of every row
    ([B*next_n, k] int32), in two launches."""
    _need(k_new, torch.bfloat16, "k_new")
    _need(q, torch.bfloat16, "q")
    _need(weights, torch.float32, "weights")
    _need(kcache, torch.uint8, "kcache")
    _need(block_table, torch.int32, "block_table")
    _need(context_lens, torch.int32, "context_lens")
    B = context_lens.numel()
    max_blocks = block_table.shape[1]
    if k_new.numel() != B * next_n * HEAD_DIM or q.numel() != B * next_n * H * HEAD_DIM:
        raise ValueError("k_new / q do not match B * next_n (* H) rows of 128")
    if weights.numel() != B * next_n * H:
        raise ValueError("weights must be [B * next_n, H]")
    if workspace is None:
        n = paged_decode_step_workspace_bytes(B, next_n, H, max_blocks, k)
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)
    _need(workspace, torch.uint8, "workspace")
    idx = out if out is not None else torch.empty((B * next_n, k), dtype=torch.int32,
                                                  device=q.device)
    _check("idx_paged_decode_step", lib.idx_paged_decode_step(
        _ptr(k_new), _ptr(q), B, next_n, H, _ptr(kcache), kcache.shape[0], PAGE_SIZE,
        _ptr(block_table), max_blocks, _ptr(context_lens), _ptr(weights), k, _ptr(idx),
        _ptr(workspace), workspace.numel(), _ptr(errors), _stream(stream)))
    return idx


def mqa_logits(q_vals, q_scales, weights, k_vals, k_scales, row_start, row_end, H: int,
               ld: int | None = None, clean: bool = False, out=None, errors=None, stream=None):
    _need(q_vals, torch.uint8, "q_vals")
    _need(q_scales, torch.uint8, "q_scales")
    _need(k_vals, torch.uint8, "k_vals")
    _need(k_scales, torch.uint8, "k_scales")
    _need(weights, torch.float32, "weights")
    _need(row_start, torch.int32, "row_start")
    _need(row_end, torch.int32, "row_end")
    T = row_end.numel()
    S = k_vals.numel() // 64
    if ld is None:
        ld = S
    logits = out if out is not None else torch.empty((T, ld), dtype=torch.float32,
                                                     device=q_vals.device)
    _check("idx_mqa_logits", lib.idx_mqa_logits(
        _ptr(q_vals), _ptr(q_scales), T, H, _ptr(k_vals), _ptr(k_scales), S, _ptr(weights),
        _ptr(row_start), _ptr(row_end), _ptr(logits), ld, 1 if clean else 0, _ptr(errors),
        _stream(stream)))
    return logits


def mqa_logits_topk_workspace_bytes(T: int, S: int, k: int) -> int:
    return int(lib.idx_mqa_logits_topk_workspace_bytes(T, S, k))


def mqa_logits_topk(q_vals, q_scales, weights, k_vals, k_scales, row_start, row_end, H: int,
                    k: int = 2048, workspace=None, out=None, errors=None, stream=None):
    """Prefill logits + top-k of every row without a logits tensor:
    [T, k] int32 positions relative to row_start (-1 padded)."""
    _need(q_vals, torch.uint8, "q_vals")
    _need(q_scales, torch.uint8, "q_scales")
    _need(k_vals, torch.uint8, "k_vals")
    _need(k_scales, torch.uint8, "k_scales")
    _need(weights, torch.float32, "weights")
    _need(row_start, torch.int32, "row_start")
    _need(row_end, torch.int32, "row_end")
    T = row_end.numel()
    S = k_vals.numel() // 64
    if workspace is None:
        workspace = torch.empty(max(mqa_logits_topk_workspace_bytes(T, S, k), 256),
                                dtype=torch.uint8, device=q_vals.device)
    _need(workspace, torch.uint8, "workspace")
    idx = out if out is not None else torch.empty((T, k), dtype=torch.int32, device=q_vals.device)
    _check("idx_mqa_logits_topk", lib.idx_mqa_logits_topk(
        _ptr(q_vals), _ptr(q_scales), T, H, _ptr(k_vals), _ptr(k_scales), S, _ptr(weights),
        _ptr(row_start), _ptr(row_end), k, _ptr(idx), _ptr(workspace), workspace.numel(),
        _ptr(errors), _stream(stream)))
    return idx


def topk_rows(logits, row_end, k: int = 2048, row_start=None, out=None, stream=None):
    _need(logits, torch.float32, "logits", contiguous=False)
    _need(row_end, torch.int32, "row_end")
    if row_start is not None:
        _need(row_start, torch.int32, "row_start")
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be 2-D with unit column stride")
    rows = logits.shape[0]
    idx = out if out is not None else torch.empty((rows, k), dtype=torch.int32,
                                                  device=logits.device)
    _check("idx_topk_rows", lib.idx_topk_rows(_ptr(logits), rows, logits.stride(0),
                                              _ptr(row_start), _ptr(row_end), k, _ptr(idx),
                                              _stream(stream)))
    return idx


def gather_k(kcache, block_table, seq_lens, out_offsets, out_rows: int, errors=None,
             stream=None):
    _need(kcache, torch.uint8, "kcache")
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(out_offsets, torch.int64, "out_offsets")
    B = seq_lens.numel()
    vals = torch.empty((out_rows, 64), dtype=torch.uint8, device=kcache.device)
    scales = torch.empty((out_rows, 4), dtype=torch.uint8, device=kcache.device)
    _check("idx_gather_k", lib.idx_gather_k(
        _ptr(kcache), kcache.shape[0], PAGE_SIZE, _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), _ptr(out_offsets), B, _ptr(vals), _ptr(scales), out_rows,
        _ptr(errors), _stream(stream)))
    return vals, scales


def copy_async(dst: torch.Tensor, src: torch.Tensor, stream=None) -> None:
    """Copy src into dst (both contiguous, the same number of bytes; each a CUDA
    tensor of the current device or a pinned CPU tensor) with the GPU's SMs,
    enqueued on `stream`."""
    for t, name in ((dst, "dst"), (src, "src")):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if not (t.is_cuda or t.is_pinned()):
            raise ValueError(f"{name} must be a CUDA tensor or a pinned CPU tensor")
    n = dst.numel() * dst.element_size()
    if src.numel() * src.element_size() != n:
        raise ValueError("dst and src must hold the same number of bytes")
    _check("idx_copy_async", lib.idx_copy_async(_ptr(dst), _ptr(src), n, _stream(stream)))
