"""Thin Python binding of libdsa.so (include/dsa.h), same entry-point names.

Argument marshalling only: tensors are checked for device, dtype and
contiguity, outputs are allocated with torch (device memory is the caller's
business on the C side), and every call goes straight to the C ABI on the
current torch stream.  Every step of the path runs in the library's CUDA
kernels; there is no fallback.  If the library is missing, the first call
raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# DSA_LIB_PATH selects another build of this library (the range-checked one
# under _build_checked/, for its tests); by default the optimised build.
LIB_PATH = os.environ.get("DSA_LIB_PATH") or os.path.join(_HERE, "_build", "libdsa.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "dsa.h")

DSA_OK = 0
DSA_ERR_VALUE = 1
DSA_ERR_UNSUPPORTED = 2
DSA_ERR_CUDA = 3
DSA_ERR_WORKSPACE = 4
DSA_STATUS_WAIT_TIMEOUT = 0x1
DSA_STATUS_CAND_OVERFLOW = 0x2
DSA_STATUS_DRAIN_TIMEOUT = 0x4
DSA_STATUS_CHECK_FAILED = 0x8
MAX_TOPK = 2048

_lock = threading.Lock()
_lib = None

P = ctypes.c_void_p
I = ctypes.c_int
I64 = ctypes.c_int64
F = ctypes.c_float
SZ = ctypes.c_size_t

_SIGNATURES = {
    "dsa_last_error": ([], ctypes.c_char_p),
    "dsa_device_status": ([P, I], I),
    "dsa_set_wait_limit_ns": ([ctypes.c_uint64], I),
    "dsa_thd_metadata": ([P, I, I, P, P, P], I),
    "dsa_indexer_scores": ([P, P, P, P, I, I, I, I, I, P, I64, P], I),
    "dsa_topk": ([P, I64, P, P, I, I, P, P, P, P], I),
    "dsa_compact_sort_indices": ([P, I, I, I64, P, P, P], I),
    "dsa_indexer_topk_workspace_size": ([I, I, I, I, I], SZ),
    "dsa_indexer_topk": ([P, P, P, P, I, I, I, I, I, I, P, P, P, SZ, P], I),
    "dsa_indexer_topk_ex": ([P, P, P, P, I, I, I, I, I, I, P, P, P, P, P, P, SZ, P], I),
    "dsa_topk_softmax": ([P, P, I, I, P, P, P], I),
    "dsa_forward_host": ([P, I, I, I, I, I, I, I, I, I, F, I, P, P], I),
    "dsa_indexer_topk_noalloc": ([P, P, P, P, I, I, I, I, I, I, P, P, P], I),
    "dsa_indexer_candidates": ([P, P, P, P, I, I, I, I, I, I, P, SZ, P], I),
    "dsa_select_candidates": ([P, I, I, I, I, I, I, P, SZ, P, P, P], I),
    "dsa_sparse_attn_fwd": ([P, P, P, P, P, P, I, I, I, I, I, I, F, P, P, P, P, P], I),
    "dsa_sparse_attn_fwd_ex": ([P, P, P, P, P, P, I, I, I, I, I, I, F, P, P, P, P, I, P, P], I),
    "dsa_pack_routes": ([P, I, I, I, P, P], I),
    "dsa_thd_metadata_ratio": ([P, P, P, I, I, I, P, P, P], I),
    "dsa_indexer_scores_ratio": ([P, P, P, P, P, P, I, I, I, I, I, I, I, P, I64, P], I),
    "dsa_indexer_topk_ratio": ([P, P, P, P, P, P, I, I, I, I, I, I, I, I, P, P, P, P, P, P, SZ, P], I),
    "dsa_indexer_scores_fp8": ([P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, I64, P], I),
    "dsa_indexer_topk_fp8": ([P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, P, P, P, P, P, P, SZ, P], I),
    "dsa_indexer_scores_mxfp8": ([P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, I64, P], I),
    "dsa_indexer_topk_mxfp8": ([P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, P, P, P, P, P, P, SZ, P], I),
    "dsa_sparse_attn_bwd_workspace_size": ([I, I, I, I], SZ),
    "dsa_sparse_attn_bwd": ([P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, P, P, P, P, SZ, P], I),
    "dsa_sparse_attn_bwd_workspace_size_ex": ([I, I, I, I, I], SZ),
    "dsa_sparse_attn_bwd_ex": ([P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, P, P, P, I, P, SZ, P], I),
}


class DsaError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed ({code}): {msg}")
        self.code = code


def header_functions() -> list[str]:
    """Names of the functions that include/dsa.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(dsa_\w+)\s*\(", text, re.M)))


def lib() -> ctypes.CDLL:
    """The loaded libdsa.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libdsa.so is not built ({LIB_PATH}); run __graft_entry__.build()")
            L = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in _SIGNATURES.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = res
            _lib = L
    return _lib


def _check(fn: str, rc: int) -> None:
    if rc != DSA_OK:
        msg = lib().dsa_last_error().decode(errors="replace")
        if rc in (DSA_ERR_VALUE, DSA_ERR_WORKSPACE):
            raise ValueError(f"{fn}: {msg}")
        raise DsaError(fn, rc, msg)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _need(t, name, dtype, dim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dimensions, got {t.dim()}")
    return t


def device_status(clear: bool = True) -> int:
    v = ctypes.c_uint32(0)
    _check("dsa_device_status", lib().dsa_device_status(ctypes.byref(v), 1 if clear else 0))
    return int(v.value)


def set_wait_limit_ns(limit_ns: int) -> None:
    """Bounded-wait limit of the kernels launched afterwards on the current
    device (0: the library default).  Failure-detection hook; synchronises."""
    _check("dsa_set_wait_limit_ns", lib().dsa_set_wait_limit_ns(int(limit_ns)))


def thd_metadata(cu_seqlens: torch.Tensor, T: int):
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    start = torch.empty(T, dtype=torch.int32, device=cu_seqlens.device)
    length = torch.empty(T, dtype=torch.int32, device=cu_seqlens.device)
    _check("dsa_thd_metadata", lib().dsa_thd_metadata(_p(cu_seqlens), cu_seqlens.numel() - 1, T, _p(start),
                                                      _p(length), _stream()))
    return start, length


def thd_metadata_ratio(cu_seqlens_q, cu_seqlens_k, q_causal_offsets, ratio: int, T: int):
    """start, len [T] of the ratio-causal compressed-key mask."""
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    if q_causal_offsets is not None:
        _need(q_causal_offsets, "q_causal_offsets", torch.int32, 1)
    start = torch.empty(T, dtype=torch.int32, device=cu_seqlens_q.device)
    length = torch.empty(T, dtype=torch.int32, device=cu_seqlens_q.device)
    _check("dsa_thd_metadata_ratio",
           lib().dsa_thd_metadata_ratio(_p(cu_seqlens_q), _p(cu_seqlens_k), _p(q_causal_offsets),
                                        cu_seqlens_q.numel() - 1, T, int(ratio), _p(start), _p(length), _stream()))
    return start, length


def _ratio_inputs(qi, ki, w, cu_seqlens_q, cu_seqlens_k, q_causal_offsets):
    _need(qi, "qi", torch.bfloat16, 3)
    _need(ki, "ki", torch.bfloat16, 2)
    _need(w, "w", torch.float32, 2)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    if q_causal_offsets is not None:
        _need(q_causal_offsets, "q_causal_offsets", torch.int32, 1)
    if cu_seqlens_k.numel() != cu_seqlens_q.numel():
        raise ValueError("cu_seqlens_q and cu_seqlens_k must have the same length")
    return qi.shape[0], ki.shape[0], qi.shape[1], qi.shape[2]


def indexer_scores_ratio(qi, ki, w, cu_seqlens_q, cu_seqlens_k, q_causal_offsets, ratio: int, s_max: int,
                         ld: int | None = None, out=None):
    """Dense compressed-key indexer scores fp32 [Tq, ld] under the ratio-causal mask."""
    Tq, Tk, Hi, d = _ratio_inputs(qi, ki, w, cu_seqlens_q, cu_seqlens_k, q_causal_offsets)
    ld = ld or (s_max + 3) // 4 * 4
    if out is None:
        out = torch.empty((Tq, ld), dtype=torch.float32, device=qi.device)
    _check("dsa_indexer_scores_ratio",
           lib().dsa_indexer_scores_ratio(_p(qi), _p(ki), _p(w), _p(cu_seqlens_q), _p(cu_seqlens_k),
                                          _p(q_causal_offsets), cu_seqlens_q.numel() - 1, Tq, Tk, Hi, d, int(ratio),
                                          s_max, _p(out), ld, _stream()))
    return out


def indexer_topk_ratio(qi, ki, w, cu_seqlens_q, cu_seqlens_k, q_causal_offsets, ratio: int, k: int, s_max: int,
                       want_logits: bool = False, want_softmax: bool = False, want_lse: bool = False, workspace=None):
    """Combined compressed-key indexer + top-k: dict(idx [Tq, k] ascending
    global key rows, topk_length[, logits][, softmax][, lse])."""
    Tq, Tk, Hi, d = _ratio_inputs(qi, ki, w, cu_seqlens_q, cu_seqlens_k, q_causal_offsets)
    dev = qi.device
    if workspace is None:
        workspace = torch.empty(indexer_topk_workspace_size(Tq, Hi, d, k, s_max), dtype=torch.uint8, device=dev)
    want_logits = want_logits or want_softmax or want_lse
    idx = torch.empty((Tq, k), dtype=torch.int32, device=dev)
    tl = torch.empty(Tq, dtype=torch.int32, device=dev)
    logits = torch.empty((Tq, k), dtype=torch.float32, device=dev) if want_logits else None
    sm = torch.empty((Tq, k), dtype=torch.float32, device=dev) if want_softmax else None
    lse = torch.empty(Tq, dtype=torch.float32, device=dev) if want_lse else None
    _check("dsa_indexer_topk_ratio",
           lib().dsa_indexer_topk_ratio(_p(qi), _p(ki), _p(w), _p(cu_seqlens_q), _p(cu_seqlens_k),
                                        _p(q_causal_offsets), cu_seqlens_q.numel() - 1, Tq, Tk, Hi, d, int(ratio), k,
                                        s_max, _p(idx), _p(tl), _p(logits), _p(sm), _p(lse), _p(workspace),
                                        workspace.numel() * workspace.element_size(), _stream()))
    res = {"idx": idx, "topk_length": tl}
    for name, t in (("logits", logits), ("softmax", sm), ("lse", lse)):
        if t is not None:
            res[name] = t
    return res


def _fp8_inputs(qi8, ki8, q_scale, k_scale, w, cu_seqlens_q, cu_seqlens_k, q_causal_offsets):
    _need(qi8, "qi8", torch.uint8, 3)
    _need(ki8, "ki8", torch.uint8, 2)
    _need(q_scale, "q_scale", torch.float32, 2)
    _need(k_scale, "k_scale", torch.float32, 1)
    _need(w, "w", torch.float32, 2)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    if q_causal_offsets is not None:
        _need(q_causal_offsets, "q_causal_offsets", torch.int32, 1)
    return qi8.shape[0], ki8.shape[0], qi8.shape[1], qi8.shape[2]


def indexer_scores_fp8(qi8, ki8, q_scale, k_scale, w, cu_seqlens_q, cu_seqlens_k, q_causal_offsets, ratio: int,
                       s_max: int, ld: int | None = None, out=None):
    """Dense indexer scores fp32 [Tq, ld] from E4M3 qi8 / ki8 (uint8 codes) and fp32 descales."""
    Tq, Tk, Hi, d = _fp8_inputs(qi8, ki8, q_scale, k_scale, w, cu_seqlens_q, cu_seqlens_k, q_causal_offsets)
    ld = ld or (s_max + 3) // 4 * 4
    if out is None:
        out = torch.empty((Tq, ld), dtype=torch.float32, device=qi8.device)
    _check("dsa_indexer_scores_fp8",
           lib().dsa_indexer_scores_fp8(_p(qi8), _p(ki8), _p(q_scale), _p(k_scale), _p(w), _p(cu_seqlens_q),
                                        _p(cu_seqlens_k), _p(q_causal_offsets), cu_seqlens_q.numel() - 1, Tq, Tk, Hi,
                                        d, int(ratio), s_max, _p(out), ld, _stream()))
    return out


def indexer_topk_fp8(qi8, ki8, q_scale, k_scale, w, cu_seqlens_q, cu_seqlens_k, q_causal_offsets, ratio: int, k: int,
                     s_max: int, want_logits: bool = False, want_softmax: bool = False, want_lse: bool = False,
                     workspace=None, idx=None, topk_length=None):
    """Combined indexer + top-k on E4M3 inputs: dict(idx, topk_length[, logits][, softmax][, lse])."""
    Tq, Tk, Hi, d = _fp8_inputs(qi8, ki8, q_scale, k_scale, w, cu_seqlens_q, cu_seqlens_k, q_causal_offsets)
    dev = qi8.device
    if workspace is None:
        workspace = torch.empty(indexer_topk_workspace_size(Tq, Hi, d, k, s_max), dtype=torch.uint8, device=dev)
    want_logits = want_logits or want_softmax or want_lse
    idx = torch.empty((Tq, k), dtype=torch.int32, device=dev) if idx is None else idx
    tl = torch.empty(Tq, dtype=torch.int32, device=dev) if topk_length is None else topk_length
    logits = torch.empty((Tq, k), dtype=torch.float32, device=dev) if want_logits else None
    sm = torch.empty((Tq, k), dtype=torch.float32, device=dev) if want_softmax else None
    lse = torch.empty(Tq, dtype=torch.float32, device=dev) if want_lse else None
    _check("dsa_indexer_topk_fp8",
           lib().dsa_indexer_topk_fp8(_p(qi8), _p(ki8), _p(q_scale), _p(k_scale), _p(w), _p(cu_seqlens_q),
                                      _p(cu_seqlens_k), _p(q_causal_offsets), cu_seqlens_q.numel() - 1, Tq, Tk, Hi, d,
                                      int(ratio), k, s_max, _p(idx), _p(tl), _p(logits), _p(sm), _p(lse),
                                      _p(workspace), workspace.numel() * workspace.element_size(), _stream()))
    res = {"idx": idx, "topk_length": tl}
    for name, t in (("logits", logits), ("softmax", sm), ("lse", lse)):
        if t is not None:
            res[name] = t
    return res


def _mxfp8_inputs(qi8, ki8, q_sf, k_sf, w, cu_seqlens_q, cu_seqlens_k, q_causal_offsets):
    _need(qi8, "qi8", torch.uint8, 3)
    _need(ki8, "ki8", torch.uint8, 2)
    _need(q_sf, "q_sf", torch.uint8, 3)
    _need(k_sf, "k_sf", torch.uint8, 2)
    _need(w, "w", torch.float32, 2)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    if q_causal_offsets is not None:
        _need(q_causal_offsets, "q_causal_offsets", torch.int32, 1)
    if q_sf.shape != (qi8.shape[0], qi8.shape[1], qi8.shape[2] // 32) or k_sf.shape != (ki8.shape[0], ki8.shape[1] // 32):
        raise ValueError("q_sf / k_sf must hold one scale byte per 32 elements of qi8 / ki8")
    return qi8.shape[0], ki8.shape[0], qi8.shape[1], qi8.shape[2]


def indexer_scores_mxfp8(qi8, ki8, q_sf, k_sf, w, cu_seqlens_q, cu_seqlens_k, q_causal_offsets, ratio: int,
                         s_max: int, ld: int | None = None, out=None):
    """Dense indexer scores fp32 [Tq, ld] from E4M3 qi8 / ki8 with E8M0 block scales q_sf / k_sf (uint8)."""
    Tq, Tk, Hi, d = _mxfp8_inputs(qi8, ki8, q_sf, k_sf, w, cu_seqlens_q, cu_seqlens_k, q_causal_offsets)
    ld = ld or (s_max + 3) // 4 * 4
    if out is None:
        out = torch.empty((Tq, ld), dtype=torch.float32, device=qi8.device)
    _check("dsa_indexer_scores_mxfp8",
           lib().dsa_indexer_scores_mxfp8(_p(qi8), _p(ki8), _p(q_sf), _p(k_sf), _p(w), _p(cu_seqlens_q),
                                          _p(cu_seqlens_k), _p(q_causal_offsets), cu_seqlens_q.numel() - 1, Tq, Tk,
                                          Hi, d, int(ratio), s_max, _p(out), ld, _stream()))
    return out


def indexer_topk_mxfp8(qi8, ki8, q_sf, k_sf, w, cu_seqlens_q, cu_seqlens_k, q_causal_offsets, ratio: int, k: int,
                       s_max: int, want_logits: bool = False, want_softmax: bool = False, want_lse: bool = False,
                       workspace=None, idx=None, topk_length=None):
    """Combined indexer + top-k on MXFP8 inputs: dict(idx, topk_length[, logits][, softmax][, lse])."""
    Tq, Tk, Hi, d = _mxfp8_inputs(qi8, ki8, q_sf, k_sf, w, cu_seqlens_q, cu_seqlens_k, q_causal_offsets)
    dev = qi8.device
    if workspace is None:
        workspace = torch.empty(indexer_topk_workspace_size(Tq, Hi, d, k, s_max), dtype=torch.uint8, device=dev)
    want_logits = want_logits or want_softmax or want_lse
    idx = torch.empty((Tq, k), dtype=torch.int32, device=dev) if idx is None else idx
    tl = torch.empty(Tq, dtype=torch.int32, device=dev) if topk_length is None else topk_length
    logits = torch.empty((Tq, k), dtype=torch.float32, device=dev) if want_logits else None
    sm = torch.empty((Tq, k), dtype=torch.float32, device=dev) if want_softmax else None
    lse = torch.empty(Tq, dtype=torch.float32, device=dev) if want_lse else None
    _check("dsa_indexer_topk_mxfp8",
           lib().dsa_indexer_topk_mxfp8(_p(qi8), _p(ki8), _p(q_sf), _p(k_sf), _p(w), _p(cu_seqlens_q),
                                        _p(cu_seqlens_k), _p(q_causal_offsets), cu_seqlens_q.numel() - 1, Tq, Tk, Hi,
                                        d, int(ratio), k, s_max, _p(idx), _p(tl), _p(logits), _p(sm), _p(lse),
                                        _p(workspace), workspace.numel() * workspace.element_size(), _stream()))
    res = {"idx": idx, "topk_length": tl}
    for name, t in (("logits", logits), ("softmax", sm), ("lse", lse)):
        if t is not None:
            res[name] = t
    return res


def indexer_scores(qi, ki, w, cu_seqlens, s_max: int, ld: int | None = None, out=None):
    """Dense indexer scores fp32 [T, ld] (columns >= s_max untouched)."""
    _need(qi, "qi", torch.bfloat16, 3)
    _need(ki, "ki", torch.bfloat16, 2)
    _need(w, "w", torch.float32, 2)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    T, Hi, d = qi.shape
    ld = ld or (s_max + 3) // 4 * 4
    if out is None:
        out = torch.empty((T, ld), dtype=torch.float32, device=qi.device)
    _check("dsa_indexer_scores", lib().dsa_indexer_scores(_p(qi), _p(ki), _p(w), _p(cu_seqlens), cu_seqlens.numel() - 1,
                                                          T, Hi, d, s_max, _p(out), ld, _stream()))
    return out


def topk(scores, lengths, k: int, row_start=None, want_vals: bool = False, idx=None, topk_length=None):
    _need(scores, "scores", torch.float32, 2)
    _need(lengths, "lengths", torch.int32, 1)
    if row_start is not None:
        _need(row_start, "row_start", torch.int32, 1)
    T, ld = scores.shape
    dev = scores.device
    idx = torch.empty((T, k), dtype=torch.int32, device=dev) if idx is None else idx
    topk_length = torch.empty(T, dtype=torch.int32, device=dev) if topk_length is None else topk_length
    vals = torch.empty((T, k), dtype=torch.float32, device=dev) if want_vals else None
    _check("dsa_topk", lib().dsa_topk(_p(scores), ld, _p(lengths), _p(row_start), T, k, _p(idx), _p(topk_length),
                                      _p(vals), _stream()))
    return idx, topk_length, vals


def compact_sort_indices(indices, key_count: int, out=None):
    _need(indices, "indices", torch.int32, 2)
    T, K = indices.shape
    out = torch.empty_like(indices) if out is None else out
    lengths = torch.empty(T, dtype=torch.int32, device=indices.device)
    _check("dsa_compact_sort_indices", lib().dsa_compact_sort_indices(_p(indices), T, K, int(key_count), _p(out),
                                                                      _p(lengths), _stream()))
    return out, lengths


def indexer_topk_workspace_size(T: int, Hi: int, d: int, k: int, s_max: int) -> int:
    return int(lib().dsa_indexer_topk_workspace_size(T, Hi, d, k, s_max))


def indexer_topk(qi, ki, w, cu_seqlens, k: int, s_max: int, workspace=None, idx=None, topk_length=None):
    """Fused indexer + top-k: (idx [T, k] ascending global ids, topk_length [T])."""
    _need(qi, "qi", torch.bfloat16, 3)
    _need(ki, "ki", torch.bfloat16, 2)
    _need(w, "w", torch.float32, 2)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    T, Hi, d = qi.shape
    dev = qi.device
    nbytes = indexer_topk_workspace_size(T, Hi, d, k, s_max)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev) if idx is None else idx
    topk_length = torch.empty(T, dtype=torch.int32, device=dev) if topk_length is None else topk_length
    _check("dsa_indexer_topk", lib().dsa_indexer_topk(_p(qi), _p(ki), _p(w), _p(cu_seqlens), cu_seqlens.numel() - 1,
                                                      T, Hi, d, k, s_max, _p(idx), _p(topk_length), _p(workspace),
                                                      workspace.numel() * workspace.element_size(), _stream()))
    return idx, topk_length


def indexer_topk_ex(qi, ki, w, cu_seqlens, k: int, s_max: int, want_softmax: bool = True, want_lse: bool = True,
                    workspace=None):
    """Fused indexer + top-k with its aligned logits, and optionally their
    softmax and lse: dict(idx, topk_length, logits[, softmax][, lse])."""
    _need(qi, "qi", torch.bfloat16, 3)
    _need(ki, "ki", torch.bfloat16, 2)
    _need(w, "w", torch.float32, 2)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    T, Hi, d = qi.shape
    dev = qi.device
    if workspace is None:
        workspace = torch.empty(indexer_topk_workspace_size(T, Hi, d, k, s_max), dtype=torch.uint8, device=dev)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    tl = torch.empty(T, dtype=torch.int32, device=dev)
    logits = torch.empty((T, k), dtype=torch.float32, device=dev)
    sm = torch.empty((T, k), dtype=torch.float32, device=dev) if want_softmax else None
    lse = torch.empty(T, dtype=torch.float32, device=dev) if want_lse else None
    _check("dsa_indexer_topk_ex",
           lib().dsa_indexer_topk_ex(_p(qi), _p(ki), _p(w), _p(cu_seqlens), cu_seqlens.numel() - 1, T, Hi, d, k, s_max,
                                     _p(idx), _p(tl), _p(logits), _p(sm), _p(lse), _p(workspace),
                                     workspace.numel() * workspace.element_size(), _stream()))
    res = {"idx": idx, "topk_length": tl, "logits": logits}
    if sm is not None:
        res["softmax"] = sm
    if lse is not None:
        res["lse"] = lse
    return res


def topk_softmax(logits, idx, want_softmax: bool = True, want_lse: bool = True):
    """Softmax and lse of top-k logits over the slots with a valid id: (softmax or None, lse or None)."""
    _need(logits, "logits", torch.float32, 2)
    _need(idx, "idx", torch.int32, 2)
    T, k = logits.shape
    sm = torch.empty_like(logits) if want_softmax else None
    lse = torch.empty(T, dtype=torch.float32, device=logits.device) if want_lse else None
    _check("dsa_topk_softmax", lib().dsa_topk_softmax(_p(logits), _p(idx), T, k, _p(sm), _p(lse), _stream()))
    return sm, lse


class ForwardBuffers(ctypes.Structure):
    """dsa_forward_buffers (include/dsa.h), field for field."""
    _fields_ = [(name, ctypes.c_void_p) for name in (
        "qi", "ki", "w", "cu_seqlens", "q", "kv", "sink", "qi_d", "ki_d", "w_d", "cu_seqlens_d", "q_d", "kv_d",
        "sink_d", "idx_d", "topk_length_d", "out_d", "lse_d", "workspace")] + [("ws_bytes", ctypes.c_size_t)] + [
        (name, ctypes.c_void_p) for name in ("idx", "topk_length", "out", "lse")]


def forward_host(host: dict, dev: dict, res_dev: dict, res_host: dict, workspace, n_docs: int, k: int, s_max: int,
                 scale: float, chunks: int = 4, copy_stream=None):
    """One forward step from host buffers through dsa_forward_host.

    host: qi, ki, w, cu_seqlens, q, kv, sink (page-locked CPU tensors; sink may
    be None); dev: device tensors of the same shapes; res_dev / res_host: idx,
    topk_length, out, lse on the device / in page-locked host memory.  Enqueues
    on the current stream and `copy_stream` and returns at once."""
    T, Hi, d = host["qi"].shape
    _, H, Dqk = host["q"].shape
    Dv = res_dev["out"].shape[2]
    if copy_stream is None:
        copy_stream = torch.cuda.Stream(device=dev["qi"].device)
    b = ForwardBuffers()
    for name in ("qi", "ki", "w", "cu_seqlens", "q", "kv", "sink"):
        setattr(b, name, None if host.get(name) is None else host[name].data_ptr())
        setattr(b, name + "_d", None if dev.get(name) is None else dev[name].data_ptr())
    for name in ("idx", "topk_length", "out", "lse"):
        setattr(b, name + "_d", res_dev[name].data_ptr())
        setattr(b, name, res_host[name].data_ptr())
    b.workspace = workspace.data_ptr()
    b.ws_bytes = workspace.numel() * workspace.element_size()
    _check("dsa_forward_host", lib().dsa_forward_host(ctypes.byref(b), n_docs, T, Hi, d, k, s_max, H, Dqk, Dv,
                                                      float(scale), chunks, _stream(),
                                                      ctypes.c_void_p(copy_stream.cuda_stream)))
    return copy_stream


def indexer_candidates(qi, ki, w, cu_seqlens, k: int, s_max: int, workspace=None):
    """Stage 1 of indexer_topk: fills and returns the candidate workspace."""
    _need(qi, "qi", torch.bfloat16, 3)
    _need(ki, "ki", torch.bfloat16, 2)
    _need(w, "w", torch.float32, 2)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    T, Hi, d = qi.shape
    if workspace is None:
        workspace = torch.empty(indexer_topk_workspace_size(T, Hi, d, k, s_max), dtype=torch.uint8, device=qi.device)
    _check("dsa_indexer_candidates",
           lib().dsa_indexer_candidates(_p(qi), _p(ki), _p(w), _p(cu_seqlens), cu_seqlens.numel() - 1, T, Hi, d, k,
                                        s_max, _p(workspace), workspace.numel() * workspace.element_size(),
                                        _stream()))
    return workspace


def select_candidates(cu_seqlens, T: int, Hi: int, d: int, k: int, s_max: int, workspace, idx=None,
                      topk_length=None):
    """Stage 2 of indexer_topk over a workspace filled by indexer_candidates."""
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    _need(workspace, "workspace", torch.uint8, 1)
    dev = workspace.device
    idx = torch.empty((T, k), dtype=torch.int32, device=dev) if idx is None else idx
    topk_length = torch.empty(T, dtype=torch.int32, device=dev) if topk_length is None else topk_length
    _check("dsa_select_candidates",
           lib().dsa_select_candidates(_p(cu_seqlens), cu_seqlens.numel() - 1, T, Hi, d, k, s_max, _p(workspace),
                                       workspace.numel(), _p(idx), _p(topk_length), _stream()))
    return idx, topk_length


def indexer_topk_noalloc(qi, ki, w, cu_seqlens, k: int, s_max: int, idx=None, topk_length=None):
    """indexer_topk with the library's fixed scratch array (no workspace)."""
    _need(qi, "qi", torch.bfloat16, 3)
    _need(ki, "ki", torch.bfloat16, 2)
    _need(w, "w", torch.float32, 2)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    T, Hi, d = qi.shape
    dev = qi.device
    idx = torch.empty((T, k), dtype=torch.int32, device=dev) if idx is None else idx
    topk_length = torch.empty(T, dtype=torch.int32, device=dev) if topk_length is None else topk_length
    _check("dsa_indexer_topk_noalloc",
           lib().dsa_indexer_topk_noalloc(_p(qi), _p(ki), _p(w), _p(cu_seqlens), cu_seqlens.numel() - 1, T, Hi, d,
                                          k, s_max, _p(idx), _p(topk_length), _stream()))
    return idx, topk_length


def sparse_attn_fwd(q, kv, idx, scale: float, topk_length=None, sink=None, v=None, want_lse_kv: bool = False,
                    want_max_logits: bool = False, out=None, lse=None, indexer_topk: int = 0):
    """Sparse MQA attention forward; returns dict(out, lse[, lse_kv][, max_logits][, lse_indexer]).
    indexer_topk > 0 adds lse_indexer (dsa_sparse_attn_fwd_ex)."""
    _need(q, "q", torch.bfloat16, 3)
    _need(kv, "kv", torch.bfloat16, 2)
    _need(idx, "idx", torch.int32, 2)
    if topk_length is not None:
        _need(topk_length, "topk_length", torch.int32, 1)
    if sink is not None:
        _need(sink, "sink", torch.float32, 1)
    if v is not None:
        _need(v, "v", torch.bfloat16, 2)
    T, H, Dqk = q.shape
    Tkv = kv.shape[0]
    Dv = v.shape[1] if v is not None else 512
    K = idx.shape[1]
    dev = q.device
    out = torch.empty((T, H, Dv), dtype=torch.bfloat16, device=dev) if out is None else out
    lse = torch.empty((T, H), dtype=torch.float32, device=dev) if lse is None else lse
    lse_kv = torch.empty((T, H), dtype=torch.float32, device=dev) if want_lse_kv else None
    ml = torch.empty((T, H), dtype=torch.float32, device=dev) if want_max_logits else None
    if indexer_topk:
        li = torch.empty((T, H), dtype=torch.float32, device=dev)
        _check("dsa_sparse_attn_fwd_ex",
               lib().dsa_sparse_attn_fwd_ex(_p(q), _p(kv), _p(v), _p(idx), _p(topk_length), _p(sink), T, Tkv, H, Dqk,
                                            Dv, K, float(scale), _p(out), _p(lse), _p(lse_kv), _p(ml),
                                            int(indexer_topk), _p(li), _stream()))
    else:
        li = None
        _check("dsa_sparse_attn_fwd",
               lib().dsa_sparse_attn_fwd(_p(q), _p(kv), _p(v), _p(idx), _p(topk_length), _p(sink), T, Tkv, H, Dqk,
                                         Dv, K, float(scale), _p(out), _p(lse), _p(lse_kv), _p(ml), _stream()))
    res = {"out": out, "lse": lse}
    if li is not None:
        res["lse_indexer"] = li
    if lse_kv is not None:
        res["lse_kv"] = lse_kv
    if ml is not None:
        res["max_logits"] = ml
    return res


def pack_routes(routes):
    _need(routes, "routes", torch.int32, 3)
    B, S, W = routes.shape
    Wp = (W + 3) // 4 * 4
    out = torch.empty((B * S, Wp), dtype=torch.int32, device=routes.device)
    _check("dsa_pack_routes", lib().dsa_pack_routes(_p(routes), B, S, W, _p(out), _stream()))
    return out


def sparse_attn_bwd_workspace_size(T: int, Tkv: int, H: int, K: int, deterministic: bool = True) -> int:
    return int(lib().dsa_sparse_attn_bwd_workspace_size_ex(T, Tkv, H, K, 1 if deterministic else 0))


def sparse_attn_bwd(q, kv, out, dout, lse_kv, idx, scale: float, topk_length=None, sink=None, workspace=None,
                    deterministic: bool = True):
    """Sparse attention backward (latent K = V): dict(dq bf16 [T, H, 576],
    dkv fp32 [Tkv, 576], d_sink fp32 [H] or None).  deterministic=False
    accumulates dkv with fp32 atomics (not bitwise reproducible)."""
    _need(q, "q", torch.bfloat16, 3)
    _need(kv, "kv", torch.bfloat16, 2)
    _need(out, "out", torch.bfloat16, 3)
    _need(dout, "dout", torch.bfloat16, 3)
    _need(lse_kv, "lse_kv", torch.float32, 2)
    _need(idx, "idx", torch.int32, 2)
    if topk_length is not None:
        _need(topk_length, "topk_length", torch.int32, 1)
    if sink is not None:
        _need(sink, "sink", torch.float32, 1)
    T, H, Dqk = q.shape
    Tkv = kv.shape[0]
    Dv = out.shape[2]
    K = idx.shape[1]
    dev = q.device
    if workspace is None:
        workspace = torch.empty(sparse_attn_bwd_workspace_size(T, Tkv, H, K, deterministic), dtype=torch.uint8,
                                device=dev)
    dq = torch.empty((T, H, Dqk), dtype=torch.bfloat16, device=dev)
    dkv = torch.empty((Tkv, Dqk), dtype=torch.float32, device=dev)
    d_sink = torch.empty(H, dtype=torch.float32, device=dev) if sink is not None else None
    _check("dsa_sparse_attn_bwd_ex",
           lib().dsa_sparse_attn_bwd_ex(_p(q), _p(kv), _p(out), _p(dout), _p(lse_kv), _p(sink), _p(idx),
                                        _p(topk_length), T, Tkv, H, Dqk, Dv, K, float(scale), _p(dq), _p(dkv),
                                        _p(d_sink), 1 if deterministic else 0, _p(workspace),
                                        workspace.numel() * workspace.element_size(), _stream()))
    return {"dq": dq, "dkv": dkv, "d_sink": d_sink}
