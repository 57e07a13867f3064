"""GPU parity of every hot-path step against the fp64 oracle, through the C ABI
(ops.* marshals straight into libdsa.so).  Sizes span several tiles and a
ragged tail while the oracle still finishes in seconds; edge cases cover
empty/ragged inputs, ties, invalid ids and the padded-head paths."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import (DEV, assert_attention_close, assert_bwd_close, assert_scores_close, assert_topk_softmax_close,
                      cu_from_lengths, dev, dev_bf16, f64, rand_bf16_bits)
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
    assert ops.device_status(clear=True) == 0, "a kernel raised a device status flag"


# ------------------------------------------------------------------ metadata
@pytest.mark.parametrize("lengths", [[256], [1], [3, 1, 7, 1, 12], W.thd_16k().cu_seqlens[1:] - W.thd_16k().cu_seqlens[:-1]])
def test_thd_metadata(lengths):
    cu = cu_from_lengths(lengths)
    T = int(cu[-1])
    s, l = ops.thd_metadata(dev(cu), T)
    rs, rl = oracle.thd_metadata(cu, T)
    assert np.array_equal(s.cpu().numpy(), rs) and np.array_equal(l.cpu().numpy(), rl)


# -------------------------------------------------------------- route packing
def test_pack_routes_gqa_workload():
    r = W.gqa_routes().routes()
    got = ops.pack_routes(dev(r)).cpu().numpy()
    assert np.array_equal(got, oracle.pack_routes(r))


@pytest.mark.parametrize("W_", [1, 3, 4, 6, 257])
def test_pack_routes_ragged_width(W_):
    rng = np.random.default_rng(W_)
    r = rng.integers(-3, 40, size=(3, 37, W_)).astype(np.int32)
    assert np.array_equal(ops.pack_routes(dev(r)).cpu().numpy(), oracle.pack_routes(r))


# ---------------------------------------------------------------- compact/sort
@pytest.mark.parametrize("K", [1, 7, 64, 512, 2052, 16384])
def test_compact_sort(K):
    rng = np.random.default_rng(K)
    T, kc = 37, 3000
    ind = rng.integers(-50, kc + 50, size=(T, K)).astype(np.int32)
    ind[3] = -1
    ind[4] = 5  # all duplicates
    out, lengths = ops.compact_sort_indices(dev(ind), kc)
    ro, rl = oracle.compact_sort(ind, kc)
    assert np.array_equal(out.cpu().numpy(), ro) and np.array_equal(lengths.cpu().numpy(), rl)
    # in place (out aliases in)
    t = dev(ind)
    ops.compact_sort_indices(t, kc, out=t)
    assert np.array_equal(t.cpu().numpy(), ro)


# -------------------------------------------------------------------- indexer
def _indexer_inputs(rng, lengths, Hi, d, kind="normal"):
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
    return cu, T, qi, ki, w


def _oracle_scores(cu, T, qi, ki, w, s_max):
    start, length = oracle.thd_metadata(cu, T)
    sc, mag = oracle.indexer_scores(f64(qi), f64(ki), w, start, length, s_max, want_abs=True)
    return start, length, sc, mag


def test_indexer_integer_inputs_exact():
    wl = W.tiny()
    qi, ki, w = wl.qi_bits(), wl.ki_bits(), wl.w()
    got = ops.indexer_scores(dev_bf16(qi), dev_bf16(ki), dev(w), dev(wl.cu_seqlens), wl.s_max).cpu().numpy()
    _, length, sc, _ = _oracle_scores(wl.cu_seqlens, wl.T, qi, ki, w, wl.s_max)
    fin = np.isfinite(sc)
    assert np.array_equal(got[:, : wl.s_max][fin].astype(np.float64), sc[fin])
    assert np.all(np.isneginf(got[:, : wl.s_max][~fin]))


@pytest.mark.parametrize("Hi,d", [(64, 128), (32, 128), (16, 64), (8, 64), (64, 64), (8, 128)])
@pytest.mark.parametrize("lengths", [[700], [129, 1, 300, 257]])
def test_indexer_bf16_tolerance(Hi, d, lengths):
    rng = np.random.default_rng(Hi * 1000 + d + len(lengths))
    cu, T, qi, ki, w = _indexer_inputs(rng, lengths, Hi, d)
    s_max = int(max(lengths))
    got = ops.indexer_scores(dev_bf16(qi), dev_bf16(ki), dev(w), dev(cu), s_max).cpu().numpy()[:, :s_max]
    _, length, sc, mag = _oracle_scores(cu, T, qi, ki, w, s_max)
    fin = np.isfinite(sc)
    assert_scores_close(got, sc, mag, fin)
    assert np.all(np.isneginf(got[~fin]))


# ------------------------------------------------- compressed-key (ratio) indexer
# (query lengths, key lengths, offsets or None, ratio, s_max or None = longest key segment)
RATIO_CASES = {
    "one_segment_r4": ([700], [175], None, 4, None),
    "segments_offsets_r4": ([300, 1, 513, 129], [200, 3, 300, 40], [500, 10, 683, 0], 4, None),
    "clamped_rows_r2": ([600], [100], [150], 2, None),
    "empty_key_segment": ([40, 300], [0, 90], [0, 60], 4, None),
    "negative_offset_r3": ([400, 250], [130, 120], [-20, 100], 3, None),
    "rows_cut_at_s_max_r4": ([1024], [300], [100], 4, 200),
    "ratio_one": ([129, 1, 300], [129, 1, 300], None, 1, None),
}


def _ratio_inputs(name):
    lq, lk, off, ratio, s_max = RATIO_CASES[name]
    rng = np.random.default_rng(sum(lq) * 7 + ratio)
    cq, ck = cu_from_lengths(lq), cu_from_lengths(lk)
    Tq, Tk = int(cq[-1]), int(ck[-1])
    qi = rand_bf16_bits(rng, (Tq, 64, 128))
    ki = rand_bf16_bits(rng, (max(Tk, 1), 128))
    w = (rng.random((Tq, 64), dtype=np.float32) / np.float32(8)).astype(np.float32)
    off = None if off is None else np.asarray(off, np.int32)
    s_max = s_max or int(max(max(lk), 1))
    return cq, ck, off, ratio, s_max, Tq, Tk, qi, ki, w


def _ratio_dev(cq, ck, off, qi, ki, w):
    return (dev_bf16(qi), dev_bf16(ki), dev(w), dev(cq), dev(ck), None if off is None else dev(off))


@pytest.mark.parametrize("name", sorted(RATIO_CASES))
def test_ratio_metadata(name):
    cq, ck, off, ratio, _, Tq, Tk, *_ = _ratio_inputs(name)
    s, l = ops.thd_metadata_ratio(dev(cq), dev(ck), None if off is None else dev(off), ratio, Tq)
    rs, rl = oracle.ratio_metadata(cq, ck, off, ratio, Tq, max(Tk, 0))
    assert np.array_equal(s.cpu().numpy(), rs) and np.array_equal(l.cpu().numpy(), rl)


@pytest.mark.parametrize("name", sorted(RATIO_CASES))
def test_ratio_indexer_scores(name):
    """Dense compressed-key scores against the oracle under its ratio-causal
    mask (rows cut at s_max), -inf elsewhere."""
    cq, ck, off, ratio, s_max, Tq, Tk, qi, ki, w = _ratio_inputs(name)
    if Tk == 0:
        pytest.skip("no keys")
    a = _ratio_dev(cq, ck, off, qi, ki, w)
    got = ops.indexer_scores_ratio(*a, ratio, s_max).cpu().numpy()[:, :s_max]
    start, length = oracle.ratio_metadata(cq, ck, off, ratio, Tq, Tk)
    length = np.minimum(length, s_max)
    sc, mag = oracle.indexer_scores(f64(qi), f64(ki), w, start, length, s_max, want_abs=True)
    fin = np.isfinite(sc)
    assert_scores_close(got, sc, mag, fin)
    assert np.all(np.isneginf(got[~fin]))


@pytest.mark.parametrize("name", sorted(RATIO_CASES))
@pytest.mark.parametrize("k", [1, 64, 256])
def test_ratio_fused_topk_equals_dense_then_topk(name, k):
    """The combined compressed-key call equals dense scores + dsa_topk with
    global ids, bit for bit, and the oracle's top-k of those scores."""
    cq, ck, off, ratio, s_max, Tq, Tk, qi, ki, w = _ratio_inputs(name)
    if Tk == 0:
        pytest.skip("no keys")
    a = _ratio_dev(cq, ck, off, qi, ki, w)
    res = ops.indexer_topk_ratio(*a, ratio, k, s_max, want_logits=True, want_softmax=True, want_lse=True)
    sc = ops.indexer_scores_ratio(*a, ratio, s_max)
    start, length = oracle.ratio_metadata(cq, ck, off, ratio, Tq, Tk)
    length = np.minimum(length, s_max).astype(np.int32)
    di, dt, _ = ops.topk(sc, dev(length), k, row_start=dev(start))
    assert torch.equal(res["idx"], di) and torch.equal(res["topk_length"], dt)
    scn = sc.cpu().numpy().astype(np.float64)
    ri, rt = oracle.topk(scn, length, k, start_rows=start)
    assert np.array_equal(res["idx"].cpu().numpy(), ri)
    rl, rs, re = oracle.topk_softmax(scn, ri, rt, start_rows=start)
    assert np.array_equal(res["logits"].cpu().numpy().astype(np.float64), rl)
    assert_topk_softmax_close(res["softmax"], res["lse"], rs, re)


def test_ratio_one_equals_plain_entry_points():
    """ratio 1, no offsets, keys stored like the queries: the compressed-key
    calls give the plain calls' results bit for bit."""
    rng = np.random.default_rng(21)
    cu, T, qi, ki, w = _indexer_inputs(rng, [129, 1, 300, 2049], 64, 128)
    s_max = 2049
    a = (dev_bf16(qi), dev_bf16(ki), dev(w), dev(cu))
    plain = ops.indexer_scores(*a, s_max)
    ratio = ops.indexer_scores_ratio(*a[:3], dev(cu), dev(cu), None, 1, s_max)
    assert torch.equal(plain[:, :s_max], ratio[:, :s_max])  # columns past s_max are not written
    idx, tl = ops.indexer_topk(*a, 512, s_max)
    res = ops.indexer_topk_ratio(*a[:3], dev(cu), dev(cu), None, 1, 512, s_max)
    assert torch.equal(res["idx"], idx) and torch.equal(res["topk_length"], tl)


# ------------------------------------------------------------- fp8 indexer inputs
FP8_CASES = {
    "plain_one_doc": ([700], None, None, 1, 64),
    "plain_thd": ([129, 1, 300, 257], None, None, 1, 32),
    "compressed_offsets_r4": ([300, 1, 513, 129], [200, 3, 300, 40], [500, 10, 683, 0], 4, 64),
}


def _fp8_inputs(name):
    lq, lk, off, ratio, Hi = FP8_CASES[name]
    lk = lq if lk is None else lk
    rng = np.random.default_rng(sum(lq) * 11 + Hi)
    cq, ck = cu_from_lengths(lq), cu_from_lengths(lk)
    Tq, Tk = int(cq[-1]), int(ck[-1])
    q8, qs = W.Workload._to_fp8(rand_bf16_bits(rng, (Tq, Hi, 128)))
    k8, ks = W.Workload._to_fp8(rand_bf16_bits(rng, (Tk, 128)))
    w = (rng.random((Tq, Hi), dtype=np.float32) / np.float32(8)).astype(np.float32)
    off = None if off is None else np.asarray(off, np.int32)
    return cq, ck, off, ratio, int(max(lk)), Tq, Tk, q8, qs, k8, ks, w


def _fp8_dev(cq, ck, off, q8, qs, k8, ks, w):
    return (dev(q8), dev(k8), dev(qs), dev(ks), dev(w), dev(cq), dev(ck), None if off is None else dev(off))


@pytest.mark.parametrize("name", sorted(FP8_CASES))
def test_fp8_indexer_scores(name):
    """E4M3 inputs with fp32 descales against the oracle's dequantized scores."""
    cq, ck, off, ratio, s_max, Tq, Tk, q8, qs, k8, ks, w = _fp8_inputs(name)
    got = ops.indexer_scores_fp8(*_fp8_dev(cq, ck, off, q8, qs, k8, ks, w), ratio, s_max).cpu().numpy()[:, :s_max]
    start, length = oracle.ratio_metadata(cq, ck, off, ratio, Tq, Tk)
    sc, mag = oracle.indexer_scores(oracle.fp8_dequant(q8, qs), oracle.fp8_dequant(k8, ks), w, start, length, s_max,
                                    want_abs=True)
    fin = np.isfinite(sc)
    assert_scores_close(got, sc, mag, fin)
    assert np.all(np.isneginf(got[~fin]))


@pytest.mark.parametrize("name", sorted(FP8_CASES))
@pytest.mark.parametrize("k", [1, 64, 512])
def test_fp8_fused_topk_equals_dense_then_topk(name, k):
    cq, ck, off, ratio, s_max, Tq, Tk, q8, qs, k8, ks, w = _fp8_inputs(name)
    a = _fp8_dev(cq, ck, off, q8, qs, k8, ks, w)
    res = ops.indexer_topk_fp8(*a, ratio, k, s_max, want_logits=True)
    sc = ops.indexer_scores_fp8(*a, ratio, s_max)
    start, length = oracle.ratio_metadata(cq, ck, off, ratio, Tq, Tk)
    di, dt, _ = ops.topk(sc, dev(length), k, row_start=dev(start))
    assert torch.equal(res["idx"], di) and torch.equal(res["topk_length"], dt)
    scn = sc.cpu().numpy().astype(np.float64)
    ri, rt = oracle.topk(scn, length, k, start_rows=start)
    assert np.array_equal(res["idx"].cpu().numpy(), ri)
    rl, _, _ = oracle.topk_softmax(scn, ri, rt, start_rows=start)
    assert np.array_equal(res["logits"].cpu().numpy().astype(np.float64), rl)


# ---------------------------------------------------------- mxfp8 indexer inputs
def _mx_inputs(name, jitter=True):
    """MXFP8 inputs of an FP8_CASES geometry: E4M3 codes with per-32-element
    E8M0 scales (the workload quantiser), then each scale byte moved by a
    random -3..3 and the codes kept, so that every block of every row carries
    its own power of two and a scale applied to the wrong block, row or
    operand changes the scores."""
    lq, lk, off, ratio, Hi = FP8_CASES[name]
    lk = lq if lk is None else lk
    rng = np.random.default_rng(sum(lq) * 13 + Hi)
    cq, ck = cu_from_lengths(lq), cu_from_lengths(lk)
    Tq, Tk = int(cq[-1]), int(ck[-1])
    q8, qs = W.Workload._to_mxfp8(rand_bf16_bits(rng, (Tq, Hi, 128)))
    k8, ks = W.Workload._to_mxfp8(rand_bf16_bits(rng, (Tk, 128)))
    if jitter:
        qs = np.clip(qs.astype(np.int32) + rng.integers(-3, 4, size=qs.shape), 1, 254).astype(np.uint8)
        ks = np.clip(ks.astype(np.int32) + rng.integers(-3, 4, size=ks.shape), 1, 254).astype(np.uint8)
    w = (rng.random((Tq, Hi), dtype=np.float32) / np.float32(8)).astype(np.float32)
    off = None if off is None else np.asarray(off, np.int32)
    return cq, ck, off, ratio, int(max(lk)), Tq, Tk, q8, qs, k8, ks, w


@pytest.mark.parametrize("name", sorted(FP8_CASES))
def test_mxfp8_indexer_scores(name):
    """E4M3 inputs with E8M0 block scales against the oracle's dequantized scores."""
    cq, ck, off, ratio, s_max, Tq, Tk, q8, qs, k8, ks, w = _mx_inputs(name)
    got = ops.indexer_scores_mxfp8(*_fp8_dev(cq, ck, off, q8, qs, k8, ks, w), ratio, s_max).cpu().numpy()[:, :s_max]
    start, length = oracle.ratio_metadata(cq, ck, off, ratio, Tq, Tk)
    sc, mag = oracle.indexer_scores(oracle.mxfp8_dequant(q8, qs), oracle.mxfp8_dequant(k8, ks), w, start, length,
                                    s_max, want_abs=True)
    fin = np.isfinite(sc)
    assert_scores_close(got, sc, mag, fin)
    assert np.all(np.isneginf(got[~fin]))


def test_mxfp8_integer_scores_exact():
    """Codes of integers in [-3, 3], power-of-two scales 2^-1 .. 2^1 per block
    and weights 1 or 2: a dot product is a multiple of 2^-2 below 128 * 9 * 4,
    the score below 64 * 2 times that, so every product and partial sum has
    at most 22 significant bits and is exact in fp32: the GPU scores equal the
    oracle's bit for bit, whatever the summation order."""
    rng = np.random.default_rng(77)
    T, Hi = 300, 64
    enc = np.vectorize(_e4m3_code_int)
    q8 = enc(rng.integers(-3, 4, size=(T, Hi, 128))).astype(np.uint8)
    k8 = enc(rng.integers(-3, 4, size=(T, 128))).astype(np.uint8)
    qs = rng.integers(126, 129, size=(T, Hi, 4)).astype(np.uint8)
    ks = rng.integers(126, 129, size=(T, 4)).astype(np.uint8)
    w = rng.integers(1, 3, size=(T, Hi)).astype(np.float32)
    cu = cu_from_lengths([T])
    got = ops.indexer_scores_mxfp8(dev(q8), dev(k8), dev(qs), dev(ks), dev(w), dev(cu), dev(cu), None, 1,
                                   T).cpu().numpy()
    start, length = oracle.thd_metadata(cu, T)
    ref = oracle.indexer_scores(oracle.mxfp8_dequant(q8, qs), oracle.mxfp8_dequant(k8, ks), w.astype(np.float64),
                                start, length, T)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin].astype(np.float64), ref[fin])


def _e4m3_code_int(v):
    v = int(v)
    if v == 0:
        return 0
    a = abs(v)
    e = a.bit_length() - 1
    return (0x80 if v < 0 else 0) | ((e + 7) << 3) | (((a << 3) >> e) & 7)


@pytest.mark.parametrize("name", sorted(FP8_CASES))
@pytest.mark.parametrize("k", [1, 64, 512])
def test_mxfp8_fused_topk_equals_dense_then_topk(name, k):
    cq, ck, off, ratio, s_max, Tq, Tk, q8, qs, k8, ks, w = _mx_inputs(name)
    a = _fp8_dev(cq, ck, off, q8, qs, k8, ks, w)
    res = ops.indexer_topk_mxfp8(*a, ratio, k, s_max, want_logits=True)
    sc = ops.indexer_scores_mxfp8(*a, ratio, s_max)
    start, length = oracle.ratio_metadata(cq, ck, off, ratio, Tq, Tk)
    di, dt, _ = ops.topk(sc, dev(length), k, row_start=dev(start))
    assert torch.equal(res["idx"], di) and torch.equal(res["topk_length"], dt)
    scn = sc.cpu().numpy().astype(np.float64)
    ri, rt = oracle.topk(scn, length, k, start_rows=start)
    assert np.array_equal(res["idx"].cpu().numpy(), ri)
    rl, _, _ = oracle.topk_softmax(scn, ri, rt, start_rows=start)
    assert np.array_equal(res["logits"].cpu().numpy().astype(np.float64), rl)


# ---------------------------------------------------------------------- top-k
def test_topk_on_gpu_scores_is_exact():
    rng = np.random.default_rng(5)
    cu, T, qi, ki, w = _indexer_inputs(rng, [1500, 37, 900], 64, 128)
    s_max = 1500
    sc = ops.indexer_scores(dev_bf16(qi), dev_bf16(ki), dev(w), dev(cu), s_max)
    start, length = oracle.thd_metadata(cu, T)
    for k in (1, 64, 512, 2048):
        idx, tl, vals = ops.topk(sc, dev(length), k, row_start=dev(start), want_vals=True)
        scn = sc.cpu().numpy().astype(np.float64)
        ri, rt = oracle.topk(scn, length, k, start_rows=start)
        assert np.array_equal(idx.cpu().numpy(), ri), k
        assert np.array_equal(tl.cpu().numpy(), rt)
        v = vals.cpu().numpy()
        for t in (0, 5, T - 1):
            n = rt[t]
            assert np.array_equal(v[t, :n], scn[t, ri[t, :n] - start[t]].astype(np.float32))
            assert np.all(np.isneginf(v[t, n:]))


def test_topk_softmax_of_dense_topk():
    """dsa_topk's values are the selected scores; dsa_topk_softmax over them
    against the oracle's softmax and lse of the same selection."""
    rng = np.random.default_rng(6)
    cu, T, qi, ki, w = _indexer_inputs(rng, [1500, 37, 900], 64, 128)
    sc = ops.indexer_scores(dev_bf16(qi), dev_bf16(ki), dev(w), dev(cu), 1500)
    start, length = oracle.thd_metadata(cu, T)
    scn = sc.cpu().numpy().astype(np.float64)
    for k in (1, 64, 2048):
        idx, tl, vals = ops.topk(sc, dev(length), k, row_start=dev(start), want_vals=True)
        sm, lse = ops.topk_softmax(vals, idx)
        rl, rs, re = oracle.topk_softmax(scn, idx.cpu().numpy(), tl.cpu().numpy(), start_rows=start)
        assert np.array_equal(vals.cpu().numpy().astype(np.float64), rl), k
        assert_topk_softmax_close(sm, lse, rs, re)


@pytest.mark.parametrize("lengths,k", [([3000], 512), ([300, 2100, 40, 1500], 1024), ([4096], 2048),
                                       ([256], 64)])
def test_fused_topk_logits_softmax(lengths, k):
    """The fused call's logits are the dense scores of the selected keys, bit
    for bit (-inf on padding); its softmax and lse match the oracle's."""
    rng = np.random.default_rng(sum(lengths) + k)
    cu, T, qi, ki, w = _indexer_inputs(rng, lengths, 64, 128)
    s_max = int(max(lengths))
    a = (dev_bf16(qi), dev_bf16(ki), dev(w), dev(cu))
    ext = ops.indexer_topk_ex(*a, k, s_max)
    idx, tl = ops.indexer_topk(*a, k, s_max)
    assert torch.equal(ext["idx"], idx) and torch.equal(ext["topk_length"], tl)
    sc = ops.indexer_scores(*a, s_max).cpu().numpy().astype(np.float64)
    start, _ = oracle.thd_metadata(cu, T)
    rl, rs, re = oracle.topk_softmax(sc, idx.cpu().numpy(), tl.cpu().numpy(), start_rows=start)
    assert np.array_equal(ext["logits"].cpu().numpy().astype(np.float64), rl)
    assert_topk_softmax_close(ext["softmax"], ext["lse"], rs, re)


@pytest.mark.parametrize("case", ["all_equal", "three_values", "two_values_long", "normal", "neg_zero", "lengths"])
def test_topk_ties_and_edges(case):
    rng = np.random.default_rng(7)
    T, ld = 24, 20000
    if case == "all_equal":
        sc = np.full((T, ld), 1.5, np.float32)
    elif case == "three_values":
        sc = rng.integers(0, 3, size=(T, ld)).astype(np.float32)
    elif case == "two_values_long":
        sc = (rng.random((T, ld)) < 0.02).astype(np.float32)  # ~400 ones, the rest tie at 0
    elif case == "neg_zero":
        sc = np.where(rng.random((T, ld)) < 0.5, np.float32(-0.0), np.float32(0.0)).astype(np.float32)
        sc[:, ::97] = 1.0
    else:
        sc = rng.standard_normal((T, ld)).astype(np.float32)
    lengths = np.full(T, ld, np.int32)
    if case == "lengths":
        lengths = rng.integers(0, ld + 1, size=T).astype(np.int32)
        lengths[:4] = [0, 1, 2047, 2048]
    for k in (1, 100, 2048):
        idx, tl, _ = ops.topk(dev(sc), dev(lengths), k)
        ri, rt = oracle.topk(sc.astype(np.float64), lengths, k)
        assert np.array_equal(idx.cpu().numpy(), ri), (case, k)
        assert np.array_equal(tl.cpu().numpy(), rt)


def _sampled_columns(n):
    """Columns that the streaming top-k samples in a row of n > 4096 columns:
    512 runs of 8 adjacent columns, run j starting at floor(j*n/512) rounded
    down to a multiple of 4 (the kernel's sampling rule, restated here so the
    test can plant values that the sample sees or misses)."""
    starts = (np.arange(512, dtype=np.int64) * n // 512) & ~3
    return np.unique((starts[:, None] + np.arange(8)[None, :]).ravel())


@pytest.mark.parametrize("case", ["normal_long", "rising", "falling", "sample_misses_the_top",
                                  "sample_overestimates", "sample_sees_only_ties", "short_rows"])
def test_topk_streaming_paths(case):
    """Rows up to 65536 columns take the sampled single-pass kernel; these
    cases drive its run sample, its whole-row sample, and both ways the sample
    can misjudge a row (too few candidates, too many), each of which must
    fall back to the exact passes with the same result."""
    rng = np.random.default_rng(11)
    T, ld = 12, 65536
    sc = rng.standard_normal((T, ld)).astype(np.float32)
    lengths = np.full(T, ld, np.int32)
    lengths[1:6] = [65535, 40000, 4097, 9001, 30000]
    if case == "rising":
        sc = np.sort(sc, axis=1)
    elif case == "falling":
        sc = -np.sort(sc, axis=1)
    elif case == "sample_misses_the_top":
        # every sampled column is 0 and most others are 1: the sample sees
        # only the bottom, tau0 admits the whole row and the buffer overflows
        sc = (1.0 + 0.01 * rng.standard_normal((T, ld))).astype(np.float32)
        for t in range(T):
            sc[t, _sampled_columns(int(lengths[t]))] = 0.0
    elif case == "sample_overestimates":
        # 300 sampled columns hold the row's largest values: tau0 lands above
        # the k-th key, so fewer than k keys pass
        sc = rng.random((T, ld)).astype(np.float32)
        for t in range(T):
            cols = _sampled_columns(int(lengths[t]))
            sc[t, rng.choice(cols, 300, replace=False)] = 10.0 + rng.random(300).astype(np.float32)
    elif case == "sample_sees_only_ties":
        sc = np.zeros((T, ld), np.float32)
        sc[:, ::101] = 2.0
    elif case == "short_rows":
        lengths = rng.integers(2049, 4097, size=T).astype(np.int32)
        lengths[:3] = [2049, 4096, 4095]
    for k in (2048, 777, 64):
        idx, tl, vals = ops.topk(dev(sc), dev(lengths), k, want_vals=True)
        ri, rt = oracle.topk(sc.astype(np.float64), lengths, k)
        assert np.array_equal(idx.cpu().numpy(), ri), (case, k)
        assert np.array_equal(tl.cpu().numpy(), rt)
        v = vals.cpu().numpy()
        for t in (0, 3, T - 1):
            n = rt[t]
            assert np.array_equal(v[t, :n], sc[t, ri[t, :n]])


def test_topk_streaming_unaligned_output():
    """k not a multiple of 4 and an id buffer that is not 16-byte aligned:
    the staged ids are stored one by one."""
    rng = np.random.default_rng(12)
    sc = rng.standard_normal((5, 8192)).astype(np.float32)
    lengths = np.array([8192, 8000, 3000, 2050, 7], np.int32)
    buf = torch.full((5 * 2046 + 1,), -7, dtype=torch.int32, device=DEV)
    out = buf[1:].view(5, 2046)
    idx, tl, _ = ops.topk(dev(sc), dev(lengths), 2046, idx=out)
    ri, rt = oracle.topk(sc.astype(np.float64), lengths, 2046)
    assert np.array_equal(idx.cpu().numpy(), ri) and np.array_equal(tl.cpu().numpy(), rt)
    assert int(buf[0]) == -7


def test_topk_unaligned_rows_use_scalar_path():
    rng = np.random.default_rng(8)
    sc = rng.integers(0, 50, size=(9, 3001)).astype(np.float32)
    lengths = np.array([3001, 3000, 2999, 5, 0, 1, 3001, 2048, 2049], np.int32)
    idx, tl, _ = ops.topk(dev(sc), dev(lengths), 2048)
    ri, rt = oracle.topk(sc.astype(np.float64), lengths, 2048)
    assert np.array_equal(idx.cpu().numpy(), ri) and np.array_equal(tl.cpu().numpy(), rt)


# ------------------------------------------------------- fused indexer + top-k
@pytest.mark.parametrize("lengths,Hi,d,k,kind", [
    ([256], 8, 64, 64, "int"),
    ([3000], 64, 128, 512, "normal"),
    ([4096], 64, 128, 2048, "normal"),
    ([700, 1, 1300, 129], 64, 128, 256, "normal"),
    ([999, 513], 32, 128, 300, "int"),
])
def test_fused_indexer_topk_equals_unfused(lengths, Hi, d, k, kind):
    rng = np.random.default_rng(sum(lengths) + k)
    cu, T, qi, ki, w = _indexer_inputs(rng, lengths, Hi, d, kind)
    s_max = int(max(lengths))
    a = (dev_bf16(qi), dev_bf16(ki), dev(w), dev(cu))
    idx, tl = ops.indexer_topk(*a, k, s_max)
    sc = ops.indexer_scores(*a, s_max)
    start, length = oracle.thd_metadata(cu, T)
    ui, ut, _ = ops.topk(sc, dev(length), k, row_start=dev(start))
    assert np.array_equal(idx.cpu().numpy(), ui.cpu().numpy())
    assert np.array_equal(tl.cpu().numpy(), ut.cpu().numpy())
    # and the unfused result is the oracle's top-k of the GPU's own scores
    ri, _ = oracle.topk(sc.cpu().numpy()[:, :s_max].astype(np.float64), length, k, start_rows=start)
    assert np.array_equal(ui.cpu().numpy(), ri)
    if kind == "int":  # exact scores: the oracle's own top-k matches too
        _, _, osc, _ = _oracle_scores(cu, T, qi, ki, w, s_max)
        oi, _ = oracle.topk(osc, length, k, start_rows=start)
        assert np.array_equal(idx.cpu().numpy(), oi)


@pytest.mark.parametrize("lengths,Hi,k,kind", [([3000], 64, 512, "normal"), ([700, 1, 300, 2049], 16, 256, "int")])
def test_stage_calls_equal_the_fused_call(lengths, Hi, k, kind):
    rng = np.random.default_rng(sum(lengths) + 7)
    cu, T, qi, ki, w = _indexer_inputs(rng, lengths, Hi, 128, kind)
    s_max = int(max(lengths))
    a = (dev_bf16(qi), dev_bf16(ki), dev(w), dev(cu))
    idx, tl = ops.indexer_topk(*a, k, s_max)
    ws = ops.indexer_candidates(*a, k, s_max)
    si, stl = ops.select_candidates(a[3], T, Hi, 128, k, s_max, ws)
    assert torch.equal(idx, si) and torch.equal(tl, stl)


def _ordered_scores_inputs(T, pattern, Hi=8, d=64):
    """Integer inputs whose exact scores follow a pattern along the key axis:
    score[j] = 256 * a[j] + b[j] from one head (q = (256, 1, 0, ...) against
    k[j] = (a[j], b[j], 0, ...)), exact in bf16 and in fp32 accumulation."""
    j = np.arange(T)
    if pattern == "rising":
        a, b = j >> 8, j & 255
    elif pattern == "falling":
        a, b = 255 - (j >> 8), 255 - (j & 255)
    elif pattern == "equal":
        a, b = np.zeros(T, np.int64), np.zeros(T, np.int64)
    elif pattern == "plateaus":  # rising steps of 1024 equal keys
        a, b = j >> 10, np.zeros(T, np.int64)
    else:
        raise ValueError(pattern)
    qi = np.zeros((T, Hi, d), np.float32)
    qi[:, 0, 0], qi[:, 0, 1] = 256.0, 1.0
    ki = np.zeros((T, d), np.float32)
    ki[:, 0], ki[:, 1] = a, b
    w = np.zeros((T, Hi), np.float32)
    w[:, 0] = 1.0
    return W.f32_to_bf16_bits(qi), W.f32_to_bf16_bits(ki), w, (256 * a + b).astype(np.float64)


@pytest.mark.parametrize("pattern", ["rising", "falling", "equal", "plateaus"])
@pytest.mark.parametrize("k", [2048, 64])
def test_fused_topk_exact_when_every_key_beats_the_running_threshold(pattern, k):
    """Rows of 32768 keys whose scores rise along the row emit every key as a
    candidate (each beats the k-th largest seen so far), far more than a row's
    candidate segments hold; equal scores and plateaus do the same through
    ties.  The fused call must still give the exact top-k, with no status flag."""
    T = 32768
    qi, ki, w, sc = _ordered_scores_inputs(T, pattern)
    cu = np.array([0, T], np.int32)
    a = (dev_bf16(qi), dev_bf16(ki), dev(w), dev(cu))
    ops.device_status(clear=True)
    idx, tl = ops.indexer_topk(*a, k, T)
    torch.cuda.synchronize()
    assert ops.device_status(clear=True) == 0
    got = idx.cpu().numpy()
    # the same result as the unfused path on every row
    dsc = ops.indexer_scores(*a, T)
    start, length = oracle.thd_metadata(cu, T)
    ui, ut, _ = ops.topk(dsc, dev(length), k, row_start=dev(start))
    assert np.array_equal(got, ui.cpu().numpy())
    assert np.array_equal(tl.cpu().numpy(), ut.cpu().numpy())
    del dsc
    # closed forms: rising -> the last k keys; falling or equal -> the first k
    t = np.arange(T)
    long_rows = t + 1 > k
    if pattern == "rising":
        want = (t[long_rows, None] - k + 1) + np.arange(k)[None, :]
        assert np.array_equal(got[long_rows], want)
    elif pattern in ("falling", "equal"):
        assert np.array_equal(got[long_rows], np.broadcast_to(np.arange(k), (long_rows.sum(), k)))
    # and the oracle's top-k of the exact scores on sampled rows
    rows = np.array([k - 1, k, 16383, 16384, 20000, 30001, T - 1])
    ref = np.full((rows.size, T), -np.inf)
    for i, r in enumerate(rows):
        ref[i, :r + 1] = sc[:r + 1]
    oi, _ = oracle.topk(ref, (rows + 1).astype(np.int32), k)
    assert np.array_equal(got[rows], oi)


def _long_rising_inputs(T, Hi=8, d=64):
    """Integer inputs whose scores are 2^21 + j along the key axis, strictly
    rising within one narrow band (2^21 .. 2^21 + T, under 4% wide), exact in
    bf16 and in fp32 accumulation: q = (2^21, 65536, 256, 1) against
    k[j] = (1, c, a, b) with j = 65536 c + 256 a + b."""
    j = np.arange(T)
    qi = np.zeros((T, Hi, d), np.float32)
    qi[:, 0, :4] = (2.0 ** 21, 65536.0, 256.0, 1.0)
    ki = np.zeros((T, d), np.float32)
    ki[:, 0], ki[:, 1], ki[:, 2], ki[:, 3] = 1.0, j >> 16, (j >> 8) & 255, j & 255
    w = np.zeros((T, Hi), np.float32)
    w[:, 0] = 1.0
    return W.f32_to_bf16_bits(qi), W.f32_to_bf16_bits(ki), w


@pytest.mark.parametrize("k", [1, 16])
def test_fused_topk_long_rising_rows_in_one_narrow_band(k):
    """Rows of up to 70001 keys whose scores rise inside a band a few percent
    wide: every key beats the running threshold, so more than 65535 keys of a
    row land in the same histogram bin.  The threshold must stay a lower bound
    of the k-th key (a bin count that wrapped into its neighbour would push it
    above the row's maximum); the top-k are the last k keys of each row."""
    T = 70001
    qi, ki, w = _long_rising_inputs(T)
    cu = np.array([0, T], np.int32)
    a = (dev_bf16(qi), dev_bf16(ki), dev(w), dev(cu))
    ops.device_status(clear=True)
    idx, tl = ops.indexer_topk(*a, k, T)
    torch.cuda.synchronize()
    assert ops.device_status(clear=True) == 0
    got = idx.cpu().numpy()
    t = np.arange(T)
    long_rows = t + 1 > k
    want = (t[long_rows, None] - k + 1) + np.arange(k)[None, :]
    assert np.array_equal(got[long_rows], want)
    assert np.array_equal(tl.cpu().numpy(), np.minimum(t + 1, k))


def test_fused_topk_rows_longer_than_65536_columns():
    """Rows past 65536 columns take the other stage-2 selection (its column
    bitmap has no 16-bit limit); the result must still equal the unfused path."""
    rng = np.random.default_rng(70001)
    T, Hi, d, k = 70001, 8, 64, 256
    qi = rand_bf16_bits(rng, (T, Hi, d))
    ki = rand_bf16_bits(rng, (T, d))
    w = (rng.random((T, Hi), dtype=np.float32) / np.float32(8)).astype(np.float32)
    cu = np.array([0, T], np.int32)
    a = (dev_bf16(qi), dev_bf16(ki), dev(w), dev(cu))
    idx, tl = ops.indexer_topk(*a, k, T)
    sc = ops.indexer_scores(*a, T)
    start, length = oracle.thd_metadata(cu, T)
    ui, ut, _ = ops.topk(sc, dev(length), k, row_start=dev(start))
    del sc
    assert torch.equal(idx, ui)
    assert torch.equal(tl, ut)


# ------------------------------------------------------------------ attention
def _attn_case(rng, T, H, Tkv, K, Dqk=576, Dv=512, sigma=0.1, qmul=1.0, sink_scale=1.0, sink=True, sep_v=False):
    q = rand_bf16_bits(rng, (T, H, Dqk), sigma * qmul)
    kv = rand_bf16_bits(rng, (Tkv, Dqk), sigma)
    v = rand_bf16_bits(rng, (Tkv, Dv), sigma) if sep_v else None
    sk = (rng.standard_normal(H) * sink_scale).astype(np.float32) if sink else None
    return q, kv, v, sk


def _run_attn(q, kv, v, idx, tl, sk, scale, want=True):
    return ops.sparse_attn_fwd(dev_bf16(q), dev_bf16(kv), dev(idx), scale,
                               topk_length=None if tl is None else dev(tl),
                               sink=None if sk is None else dev(sk), v=None if v is None else dev_bf16(v),
                               want_lse_kv=want, want_max_logits=want)


def _ref_attn(q, kv, v, idx, tl, sk, scale, Dv=512):
    return oracle.sparse_attn(f64(q), f64(kv), idx, scale, topk_length=tl, sink=sk,
                              v=None if v is None else f64(v), dv=Dv)


def test_attention_tiny_workload():
    wl = W.tiny()
    start, length = oracle.thd_metadata(wl.cu_seqlens, wl.T)
    sc = oracle.indexer_scores(f64(wl.qi_bits()), f64(wl.ki_bits()), wl.w(), start, length, wl.s_max)
    idx, tl = oracle.topk(sc, length, wl.K, start_rows=start)
    q, kv, sk = wl.q_bits(), wl.kv_bits(), wl.sink()
    got = _run_attn(q, kv, None, idx, tl, sk, wl.scale)
    assert_attention_close(got, _ref_attn(q, kv, None, idx, tl, sk, wl.scale))


@pytest.mark.parametrize("qmul", [1.0, 30.0])
def test_attention_all_keys_selected(qmul):
    # every causal key selected (K >= len): sparse attention = dense causal attention with sink
    rng = np.random.default_rng(int(qmul))
    T, H = 300, 64
    K = 384
    q, kv, _, sk = _attn_case(rng, T, H, T, K, qmul=qmul, sink_scale=3.0)
    idx = np.full((T, K), -1, np.int32)
    for t in range(T):
        idx[t, : t + 1] = np.arange(t + 1)
    tl = np.minimum(np.arange(T) + 1, K).astype(np.int32)
    scale = 1 / 24
    got = _run_attn(q, kv, None, idx, tl, sk, scale)
    assert_attention_close(got, _ref_attn(q, kv, None, idx, tl, sk, scale))


def test_attention_slot_edge_cases():
    rng = np.random.default_rng(3)
    T, H, Tkv, K = 96, 64, 500, 300
    q, kv, _, sk = _attn_case(rng, T, H, Tkv, K, qmul=10.0, sink_scale=5.0)
    idx = rng.integers(0, Tkv, size=(T, K)).astype(np.int32)
    idx[:, 5] = -1                    # invalid inside the prefix
    idx[:, 6] = Tkv + 3               # out of range
    idx[:, 7] = idx[:, 8]             # duplicate slot
    idx[10] = -1                      # row with no valid id
    tl = rng.integers(0, K + 1, size=T).astype(np.int32)
    tl[:6] = [0, 1, 127, 128, 129, K]
    tl[6] = K + 50                    # clamped to K
    tl[7] = -3                        # clamped to 0
    scale = 0.05
    got = _run_attn(q, kv, None, idx, tl, sk, scale)
    assert_attention_close(got, _ref_attn(q, kv, None, idx, tl, sk, scale))
    # without lengths every slot is considered; no sink
    got = _run_attn(q, kv, None, idx, None, None, scale)
    assert_attention_close(got, _ref_attn(q, kv, None, idx, None, None, scale))


@pytest.mark.parametrize("H,P,sep_v", [(64, 64, False), (64, 128, False), (128, 256, False), (12, 192, False),
                                       (12, 256, True)])
def test_attention_lse_indexer(H, P, sep_v):
    """lse_indexer over the first P slots: prefixes with invalid ids, rows
    shorter than the prefix, an empty row and a prefix of invalid ids only."""
    rng = np.random.default_rng(20 + P + H)
    T, Tkv, K = 80, 600, 320
    Dqk, Dv = (256, 256) if sep_v else (576, 512)
    q, kv, v, sk = _attn_case(rng, T, H, Tkv, K, Dqk=Dqk, Dv=Dv, qmul=8.0, sink=not sep_v, sep_v=sep_v)
    idx = rng.integers(0, Tkv, size=(T, K)).astype(np.int32)
    idx[:, 3] = -1
    idx[:, 70] = Tkv + 1
    idx[9] = -1
    idx[11, :P] = -1
    tl = rng.integers(0, K + 1, size=T).astype(np.int32)
    tl[:5] = [0, 1, P - 1, P, P + 1]
    scale = 1 / math.sqrt(Dqk)
    got = ops.sparse_attn_fwd(dev_bf16(q), dev_bf16(kv), dev(idx), scale, topk_length=dev(tl),
                              sink=None if sk is None else dev(sk), v=None if v is None else dev_bf16(v),
                              want_lse_kv=True, want_max_logits=True, indexer_topk=P)
    ref = oracle.sparse_attn(f64(q), f64(kv), idx, scale, topk_length=tl, sink=sk,
                             v=None if v is None else f64(v), dv=Dv, indexer_topk=P)
    assert_attention_close(got, ref, hv=H)


def test_attention_short_units_repeatable():
    """Many units of one or two tiles (65..128 slots), where the epilogue of a
    unit follows its last tile closely: ten launches give the same bits, and
    sampled rows match the oracle.  (The epilogue once waited on the per-tile
    value-product barrier by parity, which could pass while the unit's
    previous tile was still being accumulated.)"""
    rng = np.random.default_rng(44)
    T, H, Tkv, K = 4096, 128, 4096, 128
    q, kv, _, sk = _attn_case(rng, T, H, Tkv, K)
    idx = rng.integers(0, Tkv, size=(T, K)).astype(np.int32)
    tl = rng.integers(65, K + 1, size=T).astype(np.int32)
    tl[::7] = rng.integers(1, 65, size=tl[::7].size)
    scale = 1 / 24
    qd, kvd, idd, tld, skd = dev_bf16(q), dev_bf16(kv), dev(idx), dev(tl), dev(sk)
    first = None
    for _ in range(10):
        r = ops.sparse_attn_fwd(qd, kvd, idd, scale, topk_length=tld, sink=skd)
        o = r["out"].view(torch.int16)
        if first is None:
            first = (o.clone(), r["lse"].clone())
        else:
            assert torch.equal(o, first[0]) and torch.equal(r["lse"], first[1])
    rows = np.unique(np.concatenate([np.arange(8), rng.choice(T, 56, replace=False)]))
    got = {"out": first[0].view(torch.bfloat16)[rows], "lse": first[1][rows]}
    assert_attention_close(got, _ref_attn(q[rows], kv, None, idx[rows], tl[rows], sk, scale))


@pytest.mark.parametrize("H", [1, 12, 64, 100, 128])
def test_attention_head_counts(H):
    rng = np.random.default_rng(H)
    T, Tkv, K = 70, 400, 200
    q, kv, _, sk = _attn_case(rng, T, H, Tkv, K, qmul=5.0)
    idx = rng.integers(-1, Tkv, size=(T, K)).astype(np.int32)
    got = _run_attn(q, kv, None, idx, None, sk, 0.07)
    assert_attention_close(got, _ref_attn(q, kv, None, idx, None, sk, 0.07))


def test_attention_dqk512():
    rng = np.random.default_rng(11)
    T, H, Tkv, K = 64, 64, 300, 256
    q, kv, _, sk = _attn_case(rng, T, H, Tkv, K, Dqk=512)
    idx = rng.integers(0, Tkv, size=(T, K)).astype(np.int32)
    tl = rng.integers(1, K + 1, size=T).astype(np.int32)
    got = _run_attn(q, kv, None, idx, tl, sk, 1 / math.sqrt(512))
    assert_attention_close(got, _ref_attn(q, kv, None, idx, tl, sk, 1 / math.sqrt(512)))


def test_attention_separate_v_gqa_shape():
    rng = np.random.default_rng(12)
    T, H, Tkv, K = 200, 12, 200, 260
    q, kv, v, _ = _attn_case(rng, T, H, Tkv, K, Dqk=256, Dv=256, sink=False, sep_v=True, qmul=4.0)
    routes = rng.integers(-1, Tkv, size=(T, K)).astype(np.int32)
    got = _run_attn(q, kv, v, routes, None, None, 1 / 16)
    assert_attention_close(got, _ref_attn(q, kv, v, routes, None, None, 1 / 16, Dv=256))


def test_attention_empty_inputs():
    rng = np.random.default_rng(13)
    T, H, Tkv = 5, 64, 10
    q, kv, _, sk = _attn_case(rng, T, H, Tkv, 0)
    got = _run_attn(q, kv, None, np.zeros((T, 0), np.int32), None, sk, 0.1)
    ref = _ref_attn(q, kv, None, np.zeros((T, 0), np.int32), None, sk, 0.1)
    assert_attention_close(got, ref)


# ----------------------------------------------------------- attention backward
def _bwd_inputs(T, Tkv, H, K, seed, sink=True, lengths="mixed"):
    """Inputs of the backward, out / lse_kv from the oracle forward (rounded to
    the storage types the GPU reads; the oracle backward sees the same values)."""
    rng = np.random.default_rng(seed)
    q = rand_bf16_bits(rng, (T, H, 576), 0.1)
    kv = rand_bf16_bits(rng, (Tkv, 576), 0.1)
    dout = rand_bf16_bits(rng, (T, H, 512), 1.0)
    idx = rng.integers(-3, Tkv + 3, size=(T, K)).astype(np.int32)
    idx[0, 1] = idx[0, 0]                 # duplicates inside a tile
    if K > 70:
        idx[1, 70] = idx[1, 3]            # and across tiles
    if lengths == "mixed":
        tl = rng.integers(0, K + 1, size=T).astype(np.int32)
        fixed = [K, 0, 1, min(K, 65)][:T]
        tl[: len(fixed)] = fixed
    else:
        tl = np.full(T, K, np.int32)
    sk = rng.standard_normal(H).astype(np.float32) if sink else None
    scale = 1.0 / math.sqrt(576.0)
    f = oracle.sparse_attn(f64(q), f64(kv), idx, scale, topk_length=tl, sink=sk, dv=512)
    out_bits = W.f32_to_bf16_bits(f["out"].astype(np.float32))
    lse_kv = f["lse_kv"].astype(np.float32)
    return q, kv, dout, idx, tl, sk, scale, out_bits, lse_kv


@pytest.mark.parametrize("deterministic", [True, False])
@pytest.mark.parametrize("T,Tkv,H,K,sink", [(40, 300, 64, 256, True), (9, 100, 12, 100, True),
                                            (6, 500, 128, 130, False), (3, 64, 64, 64, True)])
def test_attention_bwd_against_oracle(T, Tkv, H, K, sink, deterministic):
    q, kv, dout, idx, tl, sk, scale, out_bits, lse_kv = _bwd_inputs(T, Tkv, H, K, T * 7 + H, sink)
    res = ops.sparse_attn_bwd(dev_bf16(q), dev_bf16(kv), dev_bf16(out_bits), dev_bf16(dout), dev(lse_kv), dev(idx),
                              scale, topk_length=dev(tl), sink=None if sk is None else dev(sk),
                              deterministic=deterministic)
    dq, dkv, ds = oracle.sparse_attn_bwd(f64(q), f64(kv), idx, scale, f64(out_bits), f64(dout),
                                         lse_kv.astype(np.float64), topk_length=tl, sink=sk)
    assert_bwd_close(res["dq"], dq, "dq")
    assert_bwd_close(res["dkv"], dkv, "dkv")
    if sk is not None:
        g = res["d_sink"].cpu().numpy().astype(np.float64)
        assert np.all(np.abs(g - ds) <= 1e-3 * np.maximum(np.abs(ds), 1e-3) + 1e-5), (g, ds)


def test_attention_bwd_is_deterministic():
    q, kv, dout, idx, tl, sk, scale, out_bits, lse_kv = _bwd_inputs(64, 200, 64, 192, 5, True, lengths="full")
    a = (dev_bf16(q), dev_bf16(kv), dev_bf16(out_bits), dev_bf16(dout), dev(lse_kv), dev(idx), scale)
    r1 = ops.sparse_attn_bwd(*a, topk_length=dev(tl), sink=dev(sk))
    r2 = ops.sparse_attn_bwd(*a, topk_length=dev(tl), sink=dev(sk))
    for key in ("dq", "dkv", "d_sink"):
        assert torch.equal(r1[key].view(torch.int32) if r1[key].dtype == torch.float32 else r1[key].view(torch.int16),
                           r2[key].view(torch.int32) if r2[key].dtype == torch.float32 else r2[key].view(torch.int16)), key


def test_attention_bwd_atomic_variant_matches_the_deterministic_one():
    """The atomic variant differs from the deterministic one only in the
    order of dkv's fp32 additions: dq and d_sink are bitwise equal, and dkv
    (including the slots with repeated ids) agrees with it to the tolerance
    both are held to against the oracle, while differing in its last bits."""
    q, kv, dout, idx, tl, sk, scale, out_bits, lse_kv = _bwd_inputs(64, 200, 64, 192, 9, True, lengths="full")
    a = (dev_bf16(q), dev_bf16(kv), dev_bf16(out_bits), dev_bf16(dout), dev(lse_kv), dev(idx), scale)
    r1 = ops.sparse_attn_bwd(*a, topk_length=dev(tl), sink=dev(sk))
    r2 = ops.sparse_attn_bwd(*a, topk_length=dev(tl), sink=dev(sk), deterministic=False)
    assert torch.equal(r1["dq"].view(torch.int16), r2["dq"].view(torch.int16))
    assert torch.equal(r1["d_sink"].view(torch.int32), r2["d_sink"].view(torch.int32))
    d1 = r1["dkv"].cpu().numpy().astype(np.float64)
    assert np.count_nonzero(d1) > 0
    assert_bwd_close(r2["dkv"], d1, "dkv (atomic against deterministic)")


def test_attention_bwd_all_rows_empty():
    q, kv, dout, idx, tl, sk, scale, out_bits, lse_kv = _bwd_inputs(5, 80, 64, 64, 6, True)
    tl[:] = 0
    lse_kv[:] = np.inf
    res = ops.sparse_attn_bwd(dev_bf16(q), dev_bf16(kv), dev_bf16(out_bits), dev_bf16(dout), dev(lse_kv), dev(idx),
                              scale, topk_length=dev(tl), sink=dev(sk))
    assert torch.all(res["dq"].float() == 0) and torch.all(res["dkv"] == 0) and torch.all(res["d_sink"] == 0)
