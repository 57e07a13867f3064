"""Failure detection on the GPU without a fault: every bounded wait of the
tcgen05 / TMA kernels is made to give up at once (dsa_set_wait_limit_ns(1)),
so each kernel takes its abort path (the roles agree to stop, drain their own
copies and MMAs, free TMEM and return).  The test checks that each call
returns, that the status word reports the timeout and no failed drain, that
the device is still usable, and that the next normal call is bit-identical to
one made before the aborts.  Nothing here traps, faults or hangs: every input
is valid, only the waiting limit is shortened."""
import math

import numpy as np
import pytest
import torch

from gpu_util import DEV, cu_from_lengths, dev, dev_bf16, rand_bf16_bits
from sparse_attention_gemm_gb300 import ops

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__

    __graft_entry__.build()
    ops.set_wait_limit_ns(0)
    ops.device_status(clear=True)
    yield
    ops.set_wait_limit_ns(0)
    torch.cuda.synchronize()
    ops.device_status(clear=True)


def _inputs(T=2048, Hi=64, d=128, H=64, K=256, seed=5):
    """One document of T tokens: indexer and attention inputs, several units
    per persistent CTA so that CTAs abort in the middle of their work."""
    rng = np.random.default_rng(seed)
    cu = cu_from_lengths([T])
    return {
        "T": T, "H": H, "K": K, "cu": dev(cu),
        "qi": dev_bf16(rand_bf16_bits(rng, (T, Hi, d))),
        "ki": dev_bf16(rand_bf16_bits(rng, (T, d))),
        "w": dev((rng.random((T, Hi), dtype=np.float32) / np.float32(8.0))),
        "q": dev_bf16(rand_bf16_bits(rng, (T, H, 576), 0.1)),
        "kv": dev_bf16(rand_bf16_bits(rng, (T, 576), 0.1)),
        "sink": dev(rng.standard_normal(H).astype(np.float32)),
        "dout": dev_bf16(rand_bf16_bits(rng, (T, H, 512), 0.1)),
        "scale": 1.0 / math.sqrt(576.0),
    }


def _calls(x):
    """The library calls whose kernels wait on mbarriers, each returning its
    outputs; every call gets a fresh zero-filled workspace so that an aborted
    stage leaves well-formed (if meaningless) data for the next stage."""
    T, K = x["T"], x["K"]
    Hi, d = x["qi"].shape[1], x["qi"].shape[2]

    def dense():
        return [ops.indexer_scores(x["qi"], x["ki"], x["w"], x["cu"], T)]

    def fused():
        ws = torch.zeros(ops.indexer_topk_workspace_size(T, Hi, d, K, T), dtype=torch.uint8, device=DEV)
        return list(ops.indexer_topk(x["qi"], x["ki"], x["w"], x["cu"], K, T, workspace=ws))

    def attn_inputs():
        idx, tl = ops.indexer_topk(x["qi"], x["ki"], x["w"], x["cu"], K, T)
        return idx, tl

    def attention(idx, tl):
        r = ops.sparse_attn_fwd(x["q"], x["kv"], idx, x["scale"], topk_length=tl, sink=x["sink"], want_lse_kv=True)
        return [r["out"], r["lse"], r["lse_kv"]]

    def backward(idx, tl, fwd, deterministic=True):
        ws = torch.zeros(ops.sparse_attn_bwd_workspace_size(T, T, x["H"], K, deterministic), dtype=torch.uint8,
                         device=DEV)
        r = ops.sparse_attn_bwd(x["q"], x["kv"], fwd[0], x["dout"], fwd[2], idx, x["scale"], topk_length=tl,
                                sink=x["sink"], workspace=ws, deterministic=deterministic)
        return [r["dq"], r["dkv"], r["d_sink"]]

    return dense, fused, attn_inputs, attention, backward


def _same(a, b):
    return all(torch.equal(u.view(torch.uint8) if u.dtype == torch.bfloat16 else u,
                           v.view(torch.uint8) if v.dtype == torch.bfloat16 else v) for u, v in zip(a, b))


def test_forced_wait_timeout_aborts_every_kernel_cleanly():
    x = _inputs()
    dense, fused, attn_inputs, attention, backward = _calls(x)

    # reference results with the default limit
    ref_dense = dense()
    ref_fused = fused()
    idx, tl = attn_inputs()
    ref_attn = attention(idx, tl)
    ref_bwd = backward(idx, tl, ref_attn)
    torch.cuda.synchronize()
    assert ops.device_status(clear=True) == 0

    # every wait that is not already satisfied gives up at once
    ops.set_wait_limit_ns(1)
    try:
        for name, fn in (("dense indexer", dense), ("fused indexer + top-k", fused),
                         ("sparse attention", lambda: attention(idx, tl)),
                         ("attention backward", lambda: backward(idx, tl, ref_attn)),
                         ("attention backward, atomic dkv", lambda: backward(idx, tl, ref_attn, False))):
            fn()
            torch.cuda.synchronize()  # the kernels returned: the context is usable
            st = ops.device_status(clear=True)
            assert st & ops.DSA_STATUS_WAIT_TIMEOUT, f"{name}: no wait gave up (status {st:#x})"
            assert not st & ops.DSA_STATUS_DRAIN_TIMEOUT, f"{name}: a CTA could not drain its own work"
    finally:
        ops.set_wait_limit_ns(0)
    ops.device_status(clear=True)

    # the same calls, after the aborts, give the same bits as before them
    assert _same(dense(), ref_dense)
    assert _same(fused(), ref_fused)
    idx2, tl2 = attn_inputs()
    assert torch.equal(idx2, idx) and torch.equal(tl2, tl)
    again = attention(idx, tl)
    assert _same(again, ref_attn)
    assert _same(backward(idx, tl, ref_attn), ref_bwd)
    # the atomic variant: dq and d_sink are the deterministic variant's bits
    at = backward(idx, tl, ref_attn, False)
    assert _same([at[0], at[2]], [ref_bwd[0], ref_bwd[2]])
    torch.cuda.synchronize()
    assert ops.device_status(clear=True) == 0


def test_wait_limit_default_restored_runs_exact_twice():
    """After the hook is reset, repeated calls stay exact (no leftover state
    from the control block)."""
    x = _inputs(T=512, K=64, seed=9)
    dense, fused, attn_inputs, attention, _ = _calls(x)
    ops.set_wait_limit_ns(0)
    a = fused()
    b = fused()
    assert _same(a, b)
    idx, tl = attn_inputs()
    assert _same(attention(idx, tl), attention(idx, tl))
    torch.cuda.synchronize()
    assert ops.device_status(clear=True) == 0
