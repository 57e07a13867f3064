"""dsa_indexer_topk_noalloc: the fused indexer + top-k for callers that cannot
allocate device memory (their allocator belongs to a host framework, they are
plug-ins handed only input and output buffers, or cudaMalloc is not allowed on
their latency-critical path because it may synchronise the device).  Its
scratch is the library's fixed device array instead of a workspace.

Checked through the C ABI against dsa_indexer_topk (the workspace entry
point), bit for bit as every top-k test here is, on two calls in a row with
different shapes so that anything left in the shared array by the first call
would show in the second.  This file is collected last so that a run which
stops at the first failure has run every other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_util import DEV, cu_from_lengths, dev, dev_bf16, rand_bf16_bits
from sparse_attention_gemm_gb300 import ops
from sparse_attention_gemm_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__

    __graft_entry__.build()
    ops.device_status(clear=True)
    yield
    torch.cuda.synchronize()
    assert ops.device_status(clear=True) == 0


def _inputs(seed, lengths, Hi, d, kind):
    rng = np.random.default_rng(seed)
    cu = cu_from_lengths(lengths)
    T = int(cu[-1])
    if kind == "int":
        qi = W.f32_to_bf16_bits(rng.integers(-4, 5, size=(T, Hi, d)).astype(np.float32))
        ki = W.f32_to_bf16_bits(rng.integers(-4, 5, size=(T, d)).astype(np.float32))
        w = rng.integers(1, 5, size=(T, Hi)).astype(np.float32)
    else:
        qi = rand_bf16_bits(rng, (T, Hi, d))
        ki = rand_bf16_bits(rng, (T, d))
        w = (rng.random((T, Hi), dtype=np.float32) / np.float32(8)).astype(np.float32)
    return (dev_bf16(qi), dev_bf16(ki), dev(w), dev(cu)), T, int(max(lengths))


def _noalloc(a, T, Hi, d, k, s_max):
    qi, ki, w, cu = a
    idx = torch.full((T, k), 7, dtype=torch.int32, device=DEV)
    tl = torch.full((T,), 7, dtype=torch.int32, device=DEV)
    rc = ops.lib().dsa_indexer_topk_noalloc(ops._p(qi), ops._p(ki), ops._p(w), ops._p(cu), cu.numel() - 1, T, Hi, d,
                                           k, s_max, ops._p(idx), ops._p(tl), ops._stream())
    assert rc == ops.DSA_OK, ops.lib().dsa_last_error()
    return idx, tl


def test_noalloc_equals_workspace_entry_point_on_two_calls_in_a_row():
    cases = [
        (1, [2048], 64, 128, 512, "normal"),
        (2, [700, 1, 300, 129], 32, 128, 256, "int"),
    ]
    for seed, lengths, Hi, d, k, kind in cases:
        a, T, s_max = _inputs(seed, lengths, Hi, d, kind)
        got_idx, got_tl = _noalloc(a, T, Hi, d, k, s_max)
        ref_idx, ref_tl = ops.indexer_topk(*a, k, s_max)
        torch.cuda.synchronize()
        assert torch.equal(got_idx, ref_idx), f"case {seed}: ids differ"
        assert torch.equal(got_tl, ref_tl), f"case {seed}: lengths differ"


def test_noalloc_rejects_shapes_beyond_its_scratch():
    fake = ctypes.c_void_p(4096)  # validation fails before anything is dereferenced
    rc = ops.lib().dsa_indexer_topk_noalloc(fake, fake, fake, fake, 1, 4096, 64, 128, 2048, 4096, fake, None, None)
    assert rc == ops.DSA_ERR_WORKSPACE
    assert b"fixed array" in ops.lib().dsa_last_error()
