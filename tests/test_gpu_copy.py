"""idx_copy_async: SM-driven copies between pinned host memory and the device
(the decode step's per-step transfers), checked byte for byte."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def idx():
    from sparse_attention_indexer_quant_gb300 import binding
    return binding


SIZES = [1, 15, 16, 17, 4095, 4096, 679936, (1 << 20) + 3]


def _pinned_bytes(n, seed):
    g = np.random.default_rng(seed)
    t = torch.from_numpy(g.integers(0, 256, size=n, dtype=np.uint8)).pin_memory()
    assert t.is_pinned()
    return t


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("offset", [0, 3])
def test_host_to_device_and_back(idx, n, offset):
    src = _pinned_bytes(n + 16, n)[offset:offset + n]
    dev = torch.empty(n + 16, dtype=torch.uint8, device="cuda")[offset:offset + n]
    idx.copy_async(dev, src)
    back = torch.empty(n + 16, dtype=torch.uint8).pin_memory()[offset:offset + n]
    back.zero_()
    idx.copy_async(back, dev)
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu(), src)
    assert torch.equal(back, src)


def test_device_to_device_and_stream_order(idx):
    n = 1 << 16
    a = torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda")
    b = torch.empty_like(a)
    idx.copy_async(b, a)
    a.add_(1)                        # later work in the stream sees the copy done
    c = torch.empty_like(a)
    idx.copy_async(c, a)
    torch.cuda.synchronize()
    assert torch.equal(c, b + 1)


def test_zero_bytes_is_a_no_op(idx):
    e = torch.empty(0, dtype=torch.uint8, device="cuda")
    idx.copy_async(e, e)


def test_refuses_pageable_host_memory(idx):
    """Pageable memory is refused before anything is enqueued."""
    src = np.zeros(4096, np.uint8)
    dev = torch.empty(4096, dtype=torch.uint8, device="cuda")
    st = idx.lib.idx_copy_async(ctypes.c_void_p(dev.data_ptr()),
                                ctypes.c_void_p(src.ctypes.data), 4096,
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert idx.STATUS_NAMES[st] == "IDX_ERR_INVALID_ARG"
    with pytest.raises(ValueError):
        idx.copy_async(dev, torch.zeros(4096, dtype=torch.uint8))
