"""Helpers shared by the GPU parity tests: moving workload bits to the device,
widening them for the oracle, and the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

from sparse_attention_gemm_gb300 import workloads as W

DEV = torch.device("cuda:0")

# Tolerances stated for the DSA forward path: attention out max-abs <= 1e-2 and
# lse <= 1e-3 (abs) for bf16 inputs; indexer scores <= 1e-4 relative (with a
# floor of 1e-6 times the absolute-value sum of the terms, for scores that
# cancel); top-k indices bit-exact.
OUT_ABS = 1e-2
LSE_ABS = 1e-3
SCORE_REL = 1e-4
SCORE_FLOOR = 1e-6
# Derived (not stated): the Frobenius-relative error of out.  P is rounded to
# bf16 (2^-9 relative) before the value product and out is rounded to bf16
# (2^-9), so 1e-2 leaves a 2.5x margin; it catches systematic errors that the
# loose absolute bound would miss on small outputs.
OUT_FRO_REL = 1e-2
# Derived (not stated): the top-k softmax runs in fp32 with CUDA's expf/logf
# (a few ulp each) over at most 2048 terms, so its lse is off by a few fp32
# ulp of its magnitude plus ~1e-6 from the sum, and each probability by the
# same relative amount; 1e-4 relative leaves a wide margin.
TOPK_SOFTMAX_REL = 1e-4


# Derived (not stated): the backward rounds P and scale*dS to bf16 (2^-9
# relative) before the tensor-core products and dq to bf16 on output; the
# sums are fp32.  Normwise the error is a few 2^-9 of the result, so 1e-2
# Frobenius-relative per output leaves a margin, and no element may be off by
# more than 2e-2 of the output's largest magnitude.  d_sink involves no bf16
# rounding beyond the inputs: 1e-3 of the sum of its terms' magnitudes.
BWD_FRO_REL = 1e-2
BWD_MAX_REL = 2e-2


def assert_bwd_close(got, ref, name):
    g = got.float().cpu().numpy().astype(np.float64) if hasattr(got, "cpu") else np.asarray(got, np.float64)
    assert np.all(np.isfinite(g)), f"{name}: non-finite values"
    scale = max(np.max(np.abs(ref)), 1e-30)
    err = np.abs(g - ref)
    assert err.max() <= BWD_MAX_REL * scale, f"{name}: max err {err.max():.3g} vs max |ref| {scale:.3g}"
    fro = np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30)
    assert fro <= BWD_FRO_REL, f"{name}: Frobenius-relative err {fro:.3g}"


def assert_topk_softmax_close(sm, lse, ref_sm, ref_lse):
    sm = sm.cpu().numpy().astype(np.float64) if sm is not None else None
    lse = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isneginf(lse), ~fin), "lse: -inf rows differ"
    if fin.any():
        e = np.abs(lse[fin] - ref_lse[fin]) / np.maximum(1.0, np.abs(ref_lse[fin]))
        assert e.max() <= TOPK_SOFTMAX_REL, f"lse rel err {e.max():.3g}"
    if sm is not None:
        bad = np.abs(sm - ref_sm) > TOPK_SOFTMAX_REL * ref_sm + 1e-7
        assert not bad.any(), f"{bad.sum()} probabilities out of tolerance"


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def f64(bits: np.ndarray) -> np.ndarray:
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def rand_bf16_bits(rng, shape, sigma=1.0) -> np.ndarray:
    return W.f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(sigma))


def cu_from_lengths(lengths) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


def assert_scores_close(got: np.ndarray, ref: np.ndarray, mag: np.ndarray, mask: np.ndarray):
    g, r, a = got[mask].astype(np.float64), ref[mask], mag[mask]
    bad = np.abs(g - r) > SCORE_REL * np.abs(r) + SCORE_FLOOR * a
    assert not bad.any(), f"{bad.sum()} scores out of tolerance; worst |g-r| {np.max(np.abs(g - r)):.3g}"


def assert_attention_close(got: dict, ref: dict, hv=None):
    out = got["out"].float().cpu().numpy().astype(np.float64)
    rout = ref["out"]
    if hv is not None:
        out, rout = out[:, :hv], rout[:, :hv]
    err = np.abs(out - rout)
    assert np.all(np.isfinite(out)), "non-finite output"
    assert err.max() <= OUT_ABS, f"out max abs err {err.max():.3g}"
    nrm = np.linalg.norm(rout)
    if nrm > 0:
        fro = np.linalg.norm(out - rout) / nrm
        assert fro <= OUT_FRO_REL, f"out relative Frobenius err {fro:.3g}"
    for key, tol in (("lse", LSE_ABS), ("lse_kv", LSE_ABS), ("max_logits", LSE_ABS), ("lse_indexer", LSE_ABS)):
        if key in got:
            g = got[key].cpu().numpy().astype(np.float64)
            r = ref[key]
            if hv is not None:
                g, r = g[:, :hv], r[:, :hv]
            same_inf = (np.isinf(g) & np.isinf(r) & (np.sign(g) == np.sign(r)))
            fin = np.isfinite(r)
            assert np.array_equal(np.isinf(g), np.isinf(r)) and np.all(same_inf | fin), f"{key}: infinity mismatch"
            if fin.any():
                e = np.abs(g[fin] - r[fin]).max()
                assert e <= tol, f"{key} max abs err {e:.3g}"
