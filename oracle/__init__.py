"""fp64 CPU oracle for the DSA forward path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product path (``sparse_attention_gemm_gb300``) never imports it and shares no
code with it.  The arithmetic lives in ``dsa_oracle.c`` (plain C, fp64); this
module compiles it with gcc and marshals numpy arrays to it.

Sources are cited per function in ``dsa_oracle.c``: the NeMo AutoModel API
reference pages (``glm_moe_dsa.kernels.cudnn_dsa``,
``common.cudnn_sparse_attention``, ``qwen3_8_flash_next.cudnn_qsa``) and the
cuDNN Frontend "DeepSeek Sparse Attention (DSA)" page.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile dsa_oracle.c into oracle/_build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)  # no OpenMP available
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # DSA_ORACLE_LIB lets the mutation tests load a deliberately broken copy.
            lib = ctypes.CDLL(os.environ.get("DSA_ORACLE_LIB") or build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            L = ctypes.c_int64
            D = ctypes.c_double
            lib.oracle_num_threads.restype = I
            lib.oracle_set_num_threads.argtypes = [I]
            lib.oracle_set_num_threads.restype = I
            lib.oracle_thd_metadata.argtypes = [P, I, I, P, P]
            lib.oracle_thd_metadata.restype = I
            lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_value.restype = D
            lib.oracle_fp8_dequant.argtypes = [P, P, L, I, P]
            lib.oracle_fp8_dequant.restype = None
            lib.oracle_e8m0_value.argtypes = [ctypes.c_uint8]
            lib.oracle_e8m0_value.restype = D
            lib.oracle_mxfp8_dequant.argtypes = [P, P, L, I, P]
            lib.oracle_mxfp8_dequant.restype = None
            lib.oracle_ratio_metadata.argtypes = [P, P, P, I, I, I, I, P, P]
            lib.oracle_ratio_metadata.restype = I
            lib.oracle_indexer_scores.argtypes = [P, P, P, P, P, I, I, I, I, P, P]
            lib.oracle_indexer_scores.restype = None
            lib.oracle_topk.argtypes = [P, L, P, P, I, I, P, P]
            lib.oracle_topk.restype = I
            lib.oracle_topk_softmax.argtypes = [P, L, P, P, P, I, I, P, P, P]
            lib.oracle_topk_softmax.restype = None
            lib.oracle_compact_sort.argtypes = [P, I, I, L, P, P]
            lib.oracle_compact_sort.restype = None
            lib.oracle_pack_routes.argtypes = [P, I, I, I, P]
            lib.oracle_pack_routes.restype = None
            lib.oracle_sparse_attn.argtypes = [P, P, L, P, P, P, P, I, I, I, I, I, I, D, P, P, P, P, I, P]
            lib.oracle_sparse_attn.restype = None
            lib.oracle_sparse_attn_bwd.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, D, P, P, P]
            lib.oracle_sparse_attn_bwd.restype = None
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> int:
    """Threads of the oracle's row loops from now on; returns the previous count."""
    return int(_load().oracle_set_num_threads(int(n)))


def thd_metadata(cu_seqlens, T: int):
    """start[t], len[t] for every token (see dsa_oracle.c)."""
    cu = _i32(cu_seqlens)
    start = np.empty(T, np.int32)
    length = np.empty(T, np.int32)
    rc = _load().oracle_thd_metadata(_ptr(cu), cu.size - 1, T, _ptr(start), _ptr(length))
    if rc != 0:
        raise ValueError("cu_seqlens is not a valid prefix array over [0, T)")
    return start, length


def ratio_metadata(cu_q, cu_k, q_causal_offsets, ratio: int, Tq: int, Tk: int):
    """start[t], len[t] of the ratio-causal compressed-key mask (cuDNN DSA
    page, section 3: k_local < clamp((q_causal_offsets[b] + q_local + 1) //
    ratio, 0, seqlen_k_b)); keys of segment b start at cu_k[b]."""
    cq, ck = _i32(cu_q), _i32(cu_k)
    off = None if q_causal_offsets is None else _i32(q_causal_offsets)
    if cq.size != ck.size or (off is not None and off.size != cq.size - 1):
        raise ValueError("cu_q, cu_k and q_causal_offsets disagree on the number of segments")
    start = np.empty(Tq, np.int32)
    length = np.empty(Tq, np.int32)
    rc = _load().oracle_ratio_metadata(_ptr(cq), _ptr(ck), _ptr(off), cq.size - 1, Tq, Tk, int(ratio), _ptr(start),
                                       _ptr(length))
    if rc != 0:
        raise ValueError("cu_q / cu_k are not valid prefix arrays over [0, Tq) / [0, Tk), or ratio < 1")
    return start, length


def e4m3_value(code: int) -> float:
    """The value of one E4M3 code (see dsa_oracle.c)."""
    return float(_load().oracle_e4m3_value(int(code) & 0xFF))


def fp8_dequant(codes, scales):
    """fp64 codes[..., len] decoded from E4M3 and multiplied by one fp32 descale
    per row: scales has the shape of codes without its last axis."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    s = np.ascontiguousarray(scales, dtype=np.float32)
    if c.shape[:-1] != s.shape:
        raise ValueError("one descale per row of codes")
    out = np.empty(c.shape, np.float64)
    rows = int(np.prod(c.shape[:-1]))
    _load().oracle_fp8_dequant(_ptr(c), _ptr(s), rows, int(c.shape[-1]), _ptr(out))
    return out


def e8m0_value(code: int) -> float:
    """The value of one E8M0 scale byte (see dsa_oracle.c)."""
    return float(_load().oracle_e8m0_value(int(code) & 0xFF))


def mxfp8_dequant(codes, scales):
    """fp64 codes[..., len] decoded from E4M3, each block of 32 consecutive
    elements multiplied by its E8M0 scale: scales has the shape of codes with
    the last axis len / 32 (uint8 biased exponents)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    s = np.ascontiguousarray(scales, dtype=np.uint8)
    if c.shape[-1] % 32 != 0 or s.shape != c.shape[:-1] + (c.shape[-1] // 32,):
        raise ValueError("one E8M0 scale per 32 elements of each row of codes")
    out = np.empty(c.shape, np.float64)
    rows = int(np.prod(c.shape[:-1]))
    _load().oracle_mxfp8_dequant(_ptr(c), _ptr(s), rows, int(c.shape[-1]), _ptr(out))
    return out


def indexer_scores(qi_rows, ki, w_rows, start_rows, len_rows, s_max: int, want_abs: bool = False):
    """scores [n, s_max] (fp64, -inf beyond len) and optionally abs_scale."""
    qi_rows, ki, w_rows = _f64(qi_rows), _f64(ki), _f64(w_rows)
    n, Hi, d = qi_rows.shape
    start_rows, len_rows = _i32(start_rows), _i32(len_rows)
    out = np.empty((n, s_max), np.float64)
    mag = np.empty((n, s_max), np.float64) if want_abs else None
    _load().oracle_indexer_scores(_ptr(qi_rows), _ptr(ki), _ptr(w_rows), _ptr(start_rows),
                                  _ptr(len_rows), n, Hi, d, s_max, _ptr(out), _ptr(mag))
    return (out, mag) if want_abs else out


def topk(scores, len_rows, k: int, start_rows=None):
    """(idx [n, k] int32 ascending with -1 suffix, topk_len [n])."""
    scores = _f64(scores)
    n, ld = scores.shape
    len_rows = _i32(len_rows)
    start_rows = None if start_rows is None else _i32(start_rows)
    idx = np.empty((n, k), np.int32)
    tl = np.empty(n, np.int32)
    rc = _load().oracle_topk(_ptr(scores), ld, _ptr(len_rows), _ptr(start_rows), n, k, _ptr(idx), _ptr(tl))
    if rc != 0:
        raise MemoryError("oracle_topk: allocation failed")
    return idx, tl


def topk_softmax(scores, idx, topk_len, start_rows=None):
    """(logits [n, k], softmax [n, k], lse [n]) of the selected slots, cuDNN
    DSA page section 4: logits aligned with idx (-inf in padded slots), their
    softmax over the row's selected slots (0 elsewhere) and its log-sum-exp
    (-inf for a row with no slot)."""
    scores = _f64(scores)
    n, ld = scores.shape
    idx = _i32(idx)
    k = idx.shape[1]
    tl = _i32(topk_len)
    st = None if start_rows is None else _i32(start_rows)
    logits = np.empty((n, k), np.float64)
    sm = np.empty((n, k), np.float64)
    lse = np.empty(n, np.float64)
    _load().oracle_topk_softmax(_ptr(scores), ld, _ptr(idx), _ptr(st), _ptr(tl), n, k, _ptr(logits), _ptr(sm),
                                _ptr(lse))
    return logits, sm, lse


def compact_sort(indices, key_count: int):
    ind = _i32(indices)
    T, K = ind.shape
    out = np.empty_like(ind)
    lengths = np.empty(T, np.int32)
    _load().oracle_compact_sort(_ptr(ind), T, K, int(key_count), _ptr(out), _ptr(lengths))
    return out, lengths


def pack_routes(routes):
    r = _i32(routes)
    B, S, W = r.shape
    Wp = (W + 3) // 4 * 4
    out = np.empty((B * S, Wp), np.int32)
    _load().oracle_pack_routes(_ptr(r), B, S, W, _ptr(out))
    return out


def sparse_attn(q_rows, kv, idx_rows, scale: float, topk_length=None, sink=None, v=None, dqk=None, dv=None,
                indexer_topk: int = 0):
    """Returns dict(out [n,H,Dv], lse, lse_kv, max_logits) in fp64, plus
    lse_indexer [n,H] when indexer_topk > 0 (the LSE of the logits of the
    first indexer_topk slots, cuDNN DSA page section 1).

    kv is [Tkv, kv_ld]; QK uses its first ``dqk`` columns (default: q's last
    dim); V is ``v`` when given, else the first ``dv`` columns of kv.
    """
    q_rows, kv = _f64(q_rows), _f64(kv)
    n, H, Dqk = q_rows.shape
    if dqk is not None and dqk != Dqk:
        raise ValueError("q's last dimension must equal dqk")
    Tkv, kv_ld = kv.shape
    vv = None if v is None else _f64(v)
    Dv = dv if dv is not None else (vv.shape[1] if vv is not None else min(512, Dqk))
    idx_rows = _i32(idx_rows)
    K = idx_rows.shape[1]
    tl = None if topk_length is None else _i32(topk_length)
    sk = None if sink is None else _f64(sink)
    out = np.empty((n, H, Dv), np.float64)
    lse = np.empty((n, H), np.float64)
    lse_kv = np.empty((n, H), np.float64)
    ml = np.empty((n, H), np.float64)
    li = np.empty((n, H), np.float64) if indexer_topk > 0 else None
    _load().oracle_sparse_attn(_ptr(q_rows), _ptr(kv), kv_ld, _ptr(vv), _ptr(idx_rows), _ptr(tl), _ptr(sk),
                               n, Tkv, H, Dqk, Dv, K, float(scale), _ptr(out), _ptr(lse), _ptr(lse_kv), _ptr(ml),
                               int(indexer_topk), _ptr(li))
    res = {"out": out, "lse": lse, "lse_kv": lse_kv, "max_logits": ml}
    if li is not None:
        res["lse_indexer"] = li
    return res


def sparse_attn_bwd(q_rows, kv, idx_rows, scale: float, out_rows, dout_rows, lse_kv_rows, topk_length=None,
                    sink=None, dv=None):
    """(dq [n, H, Dqk], dkv [Tkv, Dqk], d_sink [H]) in fp64 (cuDNN DSA page,
    section 2; formulas in dsa_oracle.c).  kv is the latent K = V tensor;
    out / lse_kv are the forward's outputs for these rows."""
    q = _f64(q_rows)
    kvf = _f64(kv)
    n, H, Dqk = q.shape
    Tkv = kvf.shape[0]
    if kvf.shape[1] != Dqk:
        raise ValueError("kv rows must hold the Dqk query dims")
    o = _f64(out_rows)
    Dv = o.shape[2] if dv is None else dv
    idx = _i32(idx_rows)
    K = idx.shape[1]
    tl = None if topk_length is None else _i32(topk_length)
    sk = None if sink is None else _f64(sink)
    dq = np.empty((n, H, Dqk), np.float64)
    dkv = np.zeros((Tkv, Dqk), np.float64)
    dsink = np.zeros(H, np.float64)
    _load().oracle_sparse_attn_bwd(_ptr(q), _ptr(kvf), _ptr(idx), _ptr(tl), _ptr(sk), _ptr(o), _ptr(_f64(dout_rows)),
                                   _ptr(_f64(lse_kv_rows)), n, Tkv, H, Dqk, Dv, K, float(scale), _ptr(dq), _ptr(dkv),
                                   _ptr(dsink))
    return dq, dkv, dsink
