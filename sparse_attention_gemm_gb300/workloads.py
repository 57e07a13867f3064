"""Seeded synthetic inputs for the DSA forward path.

This module only draws random numbers and rounds them to the storage types
the kernels read (bf16 bit patterns, fp32, int32).  It holds none of the
method's arithmetic, so both the CUDA path and the CPU oracle consume the
very same bits from here.

Recipe (every draw is reproducible and addressable by row):

* Each tensor field has a fixed field id.  Rows along the token axis are
  drawn in chunks of ``CHUNK_ROWS``; chunk ``c`` of field ``f`` under
  workload seed ``s`` uses ``numpy.random.Generator(PCG64(SeedSequence([s,
  f, c])))``.  Any subset of rows can therefore be regenerated without
  drawing the whole tensor (the oracle does this for sampled rows of the
  long-context workload), and chunks are drawn on several threads.
* Normal fields: ``standard_normal(float32) * float32(sigma)`` rounded to
  bf16 with round-to-nearest-even (the harness conversion for fp32 inputs).
* Integer fields (tiny workload): ``integers(lo, hi + 1)`` stored exactly as
  bf16 (indexer q/k) or fp32 (head weights).
* Head weights of the bf16 workloads: ``uniform(0, 1, float32) / 8`` (fp32).
* Sink: ``standard_normal(float64)`` rounded to fp32.
* Document lengths (THD workload): integers uniform in [512, 4096]
  (inclusive) drawn until the total reaches T; the last one is truncated so
  that the total is exactly T.
* Block routes (GQA workload): for token position p of a batch row (one
  document per row), the complete 4-token blocks before p's own block are
  ``0 .. p//4 - 1``; ``min(63, p//4)`` of them are drawn uniformly without
  replacement and written in ascending block order as groups of 4 ids, then
  p's own block as a causal tail ``4*(p//4) .. p`` padded with -1, then
  groups of -1 up to the route width.  Row b uses its own generator
  ``SeedSequence([s, FIELD_ROUTES, b])`` and draws tokens in order.
* Compressed-key indexer workloads: query segments as above; segment b's
  causal offset (the global position of its first query, as for a later
  chunk of a longer document) is 0 or uniform in [1, 16384], each with
  probability 1/2, from ``SeedSequence([s, FIELD_OFFSETS, 0])``; the segment
  holds ``ceil((offset + queries) / ratio)`` compressed key rows (every block
  of ``ratio`` tokens up to its last query, the last one possibly partial).
  Indexer q/k/w as for the bf16 workloads, ki with that many rows.
* MXFP8 indexer inputs (any workload): the bf16 qi / ki values, quantized per
  block of 32 consecutive elements of a row (OCP MX recipe): the block's
  E8M0 scale byte is floor(log2(max |x|)) - 8 + 127 (E4M3's largest power of
  two is 2^8), clamped to [0, 254] (127 for an all-zero block), and the codes
  are E4M3 of x / 2^(byte - 127) clipped to [-448, 448], rounded to nearest
  even (torch's float8_e4m3fn conversion).
* FP8 indexer inputs (any workload): the bf16 qi / ki values, quantized per
  row (a (token, head) row of qi, a key row of ki): descale =
  float32(max |x| / 448) (1 for an all-zero row), code = E4M3 of x / descale
  clipped to [-448, 448], rounded to nearest even (torch's float8_e4m3fn
  conversion).
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
import os

import numpy as np

CHUNK_ROWS = 1024

FIELD_Q = 1
FIELD_KV = 2
FIELD_V = 3
FIELD_SINK = 4
FIELD_QI = 5
FIELD_KI = 6
FIELD_W = 7
FIELD_DOCS = 8
FIELD_ROUTES = 9
FIELD_OFFSETS = 10


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 exactly."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(seed: int, fid: int, chunk: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, fid, chunk])))


_POOL = None


def _pool() -> ThreadPoolExecutor:
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=max(1, min(32, os.cpu_count() or 1)))
    return _POOL


@dataclass
class Workload:
    """One synthetic DSA forward workload (shapes, seeds, generators)."""

    name: str
    seed: int
    T: int
    H: int
    Dqk: int
    Dv: int
    K: int
    scale: float
    Hi: int = 0
    d: int = 0
    cu_seqlens: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int32))
    has_sink: bool = True
    separate_v: bool = False
    qkv_kind: str = "normal"          # "normal": bf16 N(0,1)*sigma_qkv
    sigma_qkv: float = 0.1
    indexer_kind: str = "normal"      # "normal" | "int" | "none"
    sigma_index: float = 1.0
    w_kind: str = "uniform8"          # "uniform8" | "int"
    fused: bool = False
    B: int = 0                        # GQA route workload: batch rows
    S: int = 0                        # GQA route workload: sequence length
    W: int = 0                        # GQA route workload: route width
    ratio: int = 1                    # compressed-key indexer: tokens per key
    cu_k: np.ndarray | None = None    # compressed-key indexer: key segment bounds
    q_offsets: np.ndarray | None = None  # compressed-key indexer: causal offset per segment

    # ---- derived sizes -------------------------------------------------
    @property
    def n_docs(self) -> int:
        return int(self.cu_seqlens.size - 1)

    @property
    def s_max(self) -> int:
        """Longest key segment (a row never sees more keys than its segment holds)."""
        cu = self.cu_seqlens if self.cu_k is None else self.cu_k
        return int(np.max(np.diff(cu)))

    @property
    def Tk(self) -> int:
        """Indexer key rows."""
        return self.T if self.cu_k is None else int(self.cu_k[-1])

    # ---- chunked generation ----------------------------------------------
    def _rows(self, fid: int, n_total: int, row_elems: int, make, rows=None, dtype=np.uint16):
        """Generate rows (all, or the given subset) of a [n_total, row_elems] field."""
        if rows is None:
            out = np.empty((n_total, row_elems), dtype)
            nchunks = (n_total + CHUNK_ROWS - 1) // CHUNK_ROWS

            def work(c):
                r0 = c * CHUNK_ROWS
                r1 = min(n_total, r0 + CHUNK_ROWS)
                out[r0:r1] = make(_rng(self.seed, fid, c), (r1 - r0, row_elems))

            list(_pool().map(work, range(nchunks)))
            return out
        rows = np.asarray(rows, dtype=np.int64)
        out = np.empty((rows.size, row_elems), dtype)
        for c in np.unique(rows // CHUNK_ROWS):
            r0 = int(c) * CHUNK_ROWS
            r1 = min(n_total, r0 + CHUNK_ROWS)
            blk = make(_rng(self.seed, fid, int(c)), (r1 - r0, row_elems))
            sel = np.nonzero(rows // CHUNK_ROWS == c)[0]
            out[sel] = blk[rows[sel] - r0]
        return out

    def _normal_bf16(self, sigma):
        s = np.float32(sigma)

        def make(rng, shape):
            return f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * s)

        return make

    @staticmethod
    def _int_bf16(lo, hi):
        def make(rng, shape):
            return f32_to_bf16_bits(rng.integers(lo, hi + 1, size=shape).astype(np.float32))

        return make

    def q_bits(self, rows=None) -> np.ndarray:
        """Query, bf16 bits [n, H, Dqk]."""
        n = self.T
        a = self._rows(FIELD_Q, n, self.H * self.Dqk, self._normal_bf16(self.sigma_qkv), rows)
        return a.reshape(-1, self.H, self.Dqk)

    def kv_bits(self) -> np.ndarray:
        """Shared latent K/V (or K alone when V is separate), bf16 bits [T, Dqk]."""
        return self._rows(FIELD_KV, self.T, self.Dqk, self._normal_bf16(self.sigma_qkv))

    def v_bits(self) -> np.ndarray | None:
        """Separate value tensor, bf16 bits [T, Dv] (GQA route workload only)."""
        if not self.separate_v:
            return None
        return self._rows(FIELD_V, self.T, self.Dv, self._normal_bf16(self.sigma_qkv))

    def sink(self) -> np.ndarray | None:
        """Per-head attention sink logits, fp32 [H] (None: no sink)."""
        if not self.has_sink:
            return None
        return _rng(self.seed, FIELD_SINK, 0).standard_normal(self.H).astype(np.float32)

    def qi_bits(self, rows=None) -> np.ndarray:
        """Indexer query, bf16 bits [n, Hi, d]."""
        if self.indexer_kind == "int":
            make = self._int_bf16(-4, 4)
        else:
            make = self._normal_bf16(self.sigma_index)
        a = self._rows(FIELD_QI, self.T, self.Hi * self.d, make, rows)
        return a.reshape(-1, self.Hi, self.d)

    def ki_bits(self) -> np.ndarray:
        """Indexer key, bf16 bits [Tk, d]."""
        make = self._int_bf16(-4, 4) if self.indexer_kind == "int" else self._normal_bf16(self.sigma_index)
        return self._rows(FIELD_KI, self.Tk, self.d, make)

    @staticmethod
    def _to_fp8(bits: np.ndarray):
        """(E4M3 codes, fp32 descale per row) of bf16 bits [..., n]."""
        import torch

        x = bf16_bits_to_f32(bits)
        amax = np.max(np.abs(x), axis=-1)
        scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
        y = np.clip(x / scale[..., None], -448.0, 448.0).astype(np.float32)
        codes = torch.from_numpy(np.ascontiguousarray(y)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        return codes, scale

    @staticmethod
    def _to_mxfp8(bits: np.ndarray):
        """(E4M3 codes, E8M0 scale bytes per 32 elements) of bf16 bits [..., n]."""
        import torch

        x = bf16_bits_to_f32(bits)
        blk = x.reshape(x.shape[:-1] + (x.shape[-1] // 32, 32))
        amax = np.max(np.abs(blk), axis=-1)
        with np.errstate(divide="ignore"):
            e = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 8, 0).astype(np.int32)
        byte = np.clip(e + 127, 0, 254)
        y = np.clip(blk / np.ldexp(np.float32(1.0), byte - 127)[..., None], -448.0, 448.0).astype(np.float32)
        codes = torch.from_numpy(np.ascontiguousarray(y)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        return codes.reshape(x.shape), byte.astype(np.uint8)

    def qi_mxfp8(self, rows=None):
        """Indexer query as E4M3 codes [n, Hi, d] (uint8) and E8M0 block scales [n, Hi, d/32] (uint8)."""
        return self._to_mxfp8(self.qi_bits(rows))

    def ki_mxfp8(self):
        """Indexer key as E4M3 codes [Tk, d] (uint8) and E8M0 block scales [Tk, d/32] (uint8)."""
        return self._to_mxfp8(self.ki_bits())

    def qi_fp8(self, rows=None):
        """Indexer query as E4M3 codes [n, Hi, d] (uint8) and descales [n, Hi] (fp32)."""
        return self._to_fp8(self.qi_bits(rows))

    def ki_fp8(self):
        """Indexer key as E4M3 codes [Tk, d] (uint8) and descales [Tk] (fp32)."""
        return self._to_fp8(self.ki_bits())

    def w(self, rows=None) -> np.ndarray:
        """Pre-scaled indexer head weights, fp32 [n, Hi]."""
        if self.w_kind == "int":
            def make(rng, shape):
                return rng.integers(1, 5, size=shape).astype(np.float32)
        else:
            def make(rng, shape):
                return rng.random(shape, dtype=np.float32) / np.float32(8.0)
        return self._rows(FIELD_W, self.T, self.Hi, make, rows, dtype=np.float32)

    def routes(self) -> np.ndarray:
        """Batch-local block routes, int32 [B, S, W] (GQA route workload)."""
        groups = self.W // 4
        out = np.full((self.B, self.S, self.W), -1, np.int32)
        for b in range(self.B):
            rng = _rng(self.seed, FIELD_ROUTES, b)
            for p in range(self.S):
                nb = p // 4
                take = min(groups - 1, nb)
                blocks = np.sort(rng.choice(nb, size=take, replace=False)) if take > 0 else np.zeros(0, np.int64)
                ids = (blocks[:, None] * 4 + np.arange(4)[None, :]).reshape(-1)
                tail = np.arange(4 * nb, p + 1)
                row = np.concatenate([ids, tail]).astype(np.int32)
                out[b, p, : row.size] = row
        return out


def _doc_lengths(seed: int, T: int, lo: int, hi: int) -> np.ndarray:
    rng = _rng(seed, FIELD_DOCS, 0)
    lens = []
    total = 0
    while total < T:
        n = int(rng.integers(lo, hi + 1))
        n = min(n, T - total)
        lens.append(n)
        total += n
    return np.array(lens, np.int32)


def _cu(lens) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


def tiny() -> Workload:
    """T=256, one document, H=64, integer indexer (Hi=8, d=64), top-k 64, seed 0."""
    return Workload(name="tiny_T256_H64_k64", seed=0, T=256, H=64, Dqk=576, Dv=512, K=64,
                    scale=1.0 / math.sqrt(576.0), Hi=8, d=64, cu_seqlens=_cu([256]),
                    indexer_kind="int", w_kind="int")


def single_doc_4k() -> Workload:
    """T=4096, one document, H=64, Hi=64, d=128, top-k 2048, seed 1."""
    return Workload(name="single_doc_T4096_H64_k2048", seed=1, T=4096, H=64, Dqk=576, Dv=512, K=2048,
                    scale=1.0 / math.sqrt(576.0), Hi=64, d=128, cu_seqlens=_cu([4096]))


def thd_16k() -> Workload:
    """T=16384 packed documents (lengths U[512,4096]), H=128, top-k 512, seed 2."""
    return Workload(name="thd_T16384_H128_k512", seed=2, T=16384, H=128, Dqk=576, Dv=512, K=512,
                    scale=1.0 / math.sqrt(576.0), Hi=64, d=128,
                    cu_seqlens=_cu(_doc_lengths(2, 16384, 512, 4096)), sigma_index=0.1)


def long_64k() -> Workload:
    """T=65536, one document, H=64, Hi=64, d=128, top-k 2048, fused indexer+top-k, seed 3."""
    return Workload(name="long_T65536_H64_k2048", seed=3, T=65536, H=64, Dqk=576, Dv=512, K=2048,
                    scale=1.0 / math.sqrt(576.0), Hi=64, d=128, cu_seqlens=_cu([65536]), fused=True)


def gqa_routes() -> Workload:
    """B=8 x S=4096 block-routed sparse GQA: q [32768,12,256], k/v [32768,256], scale 1/16, seed 4."""
    B, S = 8, 4096
    return Workload(name="gqa_routes_B8_S4096_Hq12_W256", seed=4, T=B * S, H=12, Dqk=256, Dv=256, K=256,
                    scale=1.0 / 16.0, cu_seqlens=_cu([S] * B), has_sink=False, separate_v=True,
                    indexer_kind="none", B=B, S=S, W=256)


def _compressed(name: str, seed: int, lens, ratio: int, K: int, offsets=None) -> Workload:
    lens = np.asarray(lens, np.int64)
    if offsets is None:
        rng = _rng(seed, FIELD_OFFSETS, 0)
        offsets = np.where(rng.random(lens.size) < 0.5, 0, rng.integers(1, 16385, size=lens.size))
    offsets = np.asarray(offsets, np.int64)
    nk = (offsets + lens + ratio - 1) // ratio
    return Workload(name=name, seed=seed, T=int(lens.sum()), H=64, Dqk=576, Dv=512, K=K,
                    scale=1.0 / math.sqrt(576.0), Hi=64, d=128, cu_seqlens=_cu(lens), fused=True, ratio=ratio,
                    cu_k=_cu(nk), q_offsets=offsets.astype(np.int32))


def compressed_thd_8k() -> Workload:
    """Compressed-key indexer: T=8192 packed query segments (lengths U[512,4096]),
    causal offsets 0 or U[1,16384], ratio 4, Hi=64, d=128, top-k 512, seed 6."""
    return _compressed("compressed_thd_T8192_r4_k512", 6, _doc_lengths(6, 8192, 512, 4096), 4, 512)


def compressed_64k() -> Workload:
    """Compressed-key indexer: T=65536 queries in one segment, offset 0, ratio 4
    (16384 keys), Hi=64, d=128, top-k 2048, seed 7."""
    return _compressed("compressed_T65536_r4_k2048", 7, [65536], 4, 2048, offsets=[0])


ALL = {1: tiny, 2: single_doc_4k, 3: thd_16k, 4: long_64k, 5: gqa_routes, 6: compressed_thd_8k, 7: compressed_64k}
