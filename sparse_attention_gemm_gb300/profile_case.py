"""One small, self-contained invocation of one stage of the DSA forward path,
for profiling a single kernel launch (ncu ``-k <kernel> -s 1 -c 1``).

    python -m sparse_attention_gemm_gb300.profile_case CASE [--T N] [--k K]

Every case runs its call twice (the first launch warms up; profile the second)
on a single document of T tokens shaped like the long-context workload
(H = 64 heads, indexer Hi = 64, d = 128, latent 576/512, top-k k), with
seeded device-side draws: qi, ki ~ N(0, 1), head weights U(0, 1) / 8, q, kv
~ N(0, 1) * 0.1 in bf16, sink N(0, 1).  At the default T = 16384 every case
holds a few GB on the device and its inputs exceed the 129 MB L2.

Cases (kernel to select with -k in parentheses):
  indexer_dense   dsa_indexer_scores, scores [T, T] fp32       (indexer_kernel)
  indexer_fused   stage 1 of dsa_indexer_topk                   (indexer_kernel)
  indexer_mxfp8   dsa_indexer_scores_mxfp8 on E4M3 codes with E8M0 scales per 32
                  elements (drawn codes and scales), scores [T, T] fp32
                                                                (indexer_kernel)
  select          stage 2 of dsa_indexer_topk                   (fused_select_multi_kernel)
  topk            dsa_topk on the dense causal scores           (topk_stream_kernel)
  attention       dsa_sparse_attn_fwd on the fused top-k ids    (sparse_attn_kernel)
  gqa             dsa_sparse_attn_fwd, block-routed GQA, B = 8 x S = T / 8 packed
                  tokens, Hq = 12, D = 256, routes as the GQA workload draws them
                                                                (sparse_attn_kernel)
  backward        dsa_sparse_attn_bwd on the fused top-k ids, dout ~ N(0, 1) * 0.1
                  (bwd_prep_kernel, bwd_dq_kernel, bwd_dkv_kernel, bwd_reduce_*);
                  with --atomic the variant whose dkv goes through fp32 atomics
"""
from __future__ import annotations

import argparse
import math
import sys

import numpy as np
import torch

CASES = ("indexer_dense", "indexer_fused", "indexer_mxfp8", "select", "topk", "attention", "gqa", "backward")


def _bf16(shape, sigma, g, dev):
    return (torch.randn(shape, generator=g, device=dev, dtype=torch.float32) * sigma).to(torch.bfloat16)


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=CASES)
    ap.add_argument("--T", type=int, default=16384)
    ap.add_argument("--k", type=int, default=2048)
    ap.add_argument("--atomic", action="store_true", help="backward: dkv by fp32 atomics")
    args = ap.parse_args(argv)

    import os

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from sparse_attention_gemm_gb300 import build, ops

    build.build()
    dev = torch.device("cuda:0")
    T, K, H, Hi, d = args.T, args.k, 64, 64, 128
    g = torch.Generator(device=dev)
    g.manual_seed(1234)
    cu = torch.tensor([0, T], dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def twice(fn):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()

    if args.case == "gqa":
        from sparse_attention_gemm_gb300 import workloads as W

        B, S, Hq, D = 8, T // 8, 12, 256
        wl = W.gqa_routes()
        wl.B, wl.S, wl.T = B, S, B * S
        routes = torch.from_numpy(wl.routes()).to(dev)
        idx = ops.pack_routes(routes)
        q = _bf16((B * S, Hq, D), 0.1, g, dev)
        k = _bf16((B * S, D), 0.1, g, dev)
        v = _bf16((B * S, D), 0.1, g, dev)
        twice(lambda: ops.sparse_attn_fwd(q, k, idx, 1.0 / 16.0, v=v))
        print(f"gqa: B={B} S={S} Hq={Hq} D={D} width={idx.shape[1]}")
        return 0

    if args.case == "indexer_mxfp8":
        # E4M3 codes of N(0,1) draws with scale bytes around 2^-2 (no NaN codes)
        q8 = torch.randn((T, Hi, d), generator=g, device=dev).to(torch.float8_e4m3fn).view(torch.uint8)
        k8 = torch.randn((T, d), generator=g, device=dev).to(torch.float8_e4m3fn).view(torch.uint8)
        qs = torch.randint(123, 128, (T, Hi, d // 32), generator=g, device=dev, dtype=torch.int32).to(torch.uint8)
        ks = torch.randint(123, 128, (T, d // 32), generator=g, device=dev, dtype=torch.int32).to(torch.uint8)
        w = torch.rand((T, Hi), generator=g, device=dev, dtype=torch.float32) / 8.0
        scores = torch.empty((T, T), dtype=torch.float32, device=dev)
        twice(lambda: ops.indexer_scores_mxfp8(q8, k8, qs, ks, w, cu, cu, None, 1, T, out=scores))
        print(f"{args.case}: T={T} status={ops.device_status(clear=True):#x}")
        return 0
    qi = _bf16((T, Hi, d), 1.0, g, dev)
    ki = _bf16((T, d), 1.0, g, dev)
    w = torch.rand((T, Hi), generator=g, device=dev, dtype=torch.float32) / 8.0
    if args.case in ("indexer_dense", "topk"):
        scores = torch.empty((T, T), dtype=torch.float32, device=dev)
        if args.case == "indexer_dense":
            twice(lambda: ops.indexer_scores(qi, ki, w, cu, T, out=scores))
        else:
            ops.indexer_scores(qi, ki, w, cu, T, out=scores)
            start, length = ops.thd_metadata(cu, T)
            twice(lambda: ops.topk(scores, length, K, row_start=start))
        print(f"{args.case}: T={T} k={K}")
        return 0
    ws = torch.empty(ops.indexer_topk_workspace_size(T, Hi, d, K, T), dtype=torch.uint8, device=dev)
    if args.case == "indexer_fused":
        twice(lambda: ops.indexer_candidates(qi, ki, w, cu, K, T, workspace=ws))
    elif args.case == "select":
        ops.indexer_candidates(qi, ki, w, cu, K, T, workspace=ws)
        twice(lambda: ops.select_candidates(cu, T, Hi, d, K, T, ws))
    else:  # attention, backward
        idx, tl = ops.indexer_topk(qi, ki, w, cu, K, T, workspace=ws)
        del ws, qi, ki, w
        q = _bf16((T, H, 576), 0.1, g, dev)
        kv = _bf16((T, 576), 0.1, g, dev)
        sink = torch.randn(H, generator=g, device=dev, dtype=torch.float32)
        scale = 1.0 / math.sqrt(576.0)
        if args.case == "attention":
            twice(lambda: ops.sparse_attn_fwd(q, kv, idx, scale, topk_length=tl, sink=sink))
        else:
            fwd = ops.sparse_attn_fwd(q, kv, idx, scale, topk_length=tl, sink=sink, want_lse_kv=True)
            dout = _bf16((T, H, 512), 0.1, g, dev)
            det = not args.atomic
            bws = torch.empty(ops.sparse_attn_bwd_workspace_size(T, T, H, K, det), dtype=torch.uint8, device=dev)
            twice(lambda: ops.sparse_attn_bwd(q, kv, fwd["out"], dout, fwd["lse_kv"], idx, scale, topk_length=tl,
                                              sink=sink, workspace=bws, deterministic=det))
    status = ops.device_status(clear=True)
    print(f"{args.case}: T={T} k={K} status={status:#x}")
    return 1 if status else 0


if __name__ == "__main__":
    sys.exit(main())
