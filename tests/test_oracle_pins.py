"""Pins for the fp64 CPU oracle (runs without a GPU).

Each test ties the oracle to something other than itself: hand-derived
fixtures under tests/golden (each citing the passage it follows), brute force
over all subsets on tiny inputs, closed forms, special cases that reduce to
numpy/scipy routines, and invariants.  The cases are chosen so that a dropped
term, a wrong sign, a wrong index or a transposed operand in the oracle fails
at least one of them (tests/test_oracle_mutants.py plants such mistakes and
checks that they are caught).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- metadata
def test_metadata_golden():
    g = _gold("thd_metadata.json")
    start, length = oracle.thd_metadata(np.array(g["cu_seqlens"]), g["T"])
    assert start.tolist() == g["start"]
    assert length.tolist() == g["len"]


@pytest.mark.parametrize("cu,T", [([1, 4], 4), ([0, 3, 2], 3), ([0, 3], 4)])
def test_metadata_rejects_invalid(cu, T):
    with pytest.raises(ValueError):
        oracle.thd_metadata(np.array(cu), T)


# ----------------------------------------------------------------- indexer
def test_ratio_metadata_golden():
    g = _gold("ratio_metadata.json")
    for c in g["cases"]:
        s, l = oracle.ratio_metadata(np.array(c["cu_q"]), np.array(c["cu_k"]),
                                     None if c["q_causal_offsets"] is None else np.array(c["q_causal_offsets"]),
                                     c["ratio"], c["Tq"], c["Tk"])
        assert s.tolist() == c["start"] and l.tolist() == c["len"]


def test_ratio_metadata_ratio_one_is_thd_metadata():
    """ratio 1, zero offsets and keys stored like the queries: the plain
    causal THD metadata."""
    rng = np.random.default_rng(11)
    for _ in range(20):
        lens = rng.integers(0, 40, size=rng.integers(1, 6))
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        T = int(cu[-1])
        if T == 0:
            continue
        assert [a.tolist() for a in oracle.ratio_metadata(cu, cu, None, 1, T, T)] == \
            [a.tolist() for a in oracle.thd_metadata(cu, T)]


def test_ratio_metadata_brute_force():
    """Key j of segment b is visible to local row q iff every token it
    compresses, (j+1)*ratio - 1 at the latest, is at or before the query's
    global position offset + q, and j is one of the segment's keys."""
    rng = np.random.default_rng(12)
    for _ in range(40):
        nb = int(rng.integers(1, 5))
        ratio = int(rng.integers(1, 6))
        lq = rng.integers(0, 30, size=nb)
        off = rng.integers(-3, 40, size=nb)
        lk = np.array([max(0, int((o + q) // ratio) + int(rng.integers(-3, 3))) for o, q in zip(off, lq)])
        cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
        ck = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
        Tq, Tk = int(cq[-1]), int(ck[-1])
        s, l = oracle.ratio_metadata(cq, ck, off.astype(np.int32), ratio, Tq, Tk)
        for b in range(nb):
            for q in range(int(lq[b])):
                t = int(cq[b]) + q
                vis = [j for j in range(int(lk[b])) if (j + 1) * ratio - 1 <= int(off[b]) + q]
                assert vis == list(range(len(vis))), "the visible keys form a prefix"
                assert l[t] == len(vis) and s[t] == ck[b], (b, q, ratio, int(off[b]))


@pytest.mark.parametrize("cu_q,cu_k,ratio,Tq,Tk", [([0, 4], [0, 2], 0, 4, 2), ([0, 4], [1, 2], 2, 4, 2),
                                                     ([0, 3, 2], [0, 1, 2], 2, 2, 2), ([0, 4], [0, 3], 2, 4, 2)])
def test_ratio_metadata_rejects_invalid(cu_q, cu_k, ratio, Tq, Tk):
    with pytest.raises(ValueError):
        oracle.ratio_metadata(np.array(cu_q), np.array(cu_k), None, ratio, Tq, Tk)


def test_e4m3_golden_values():
    g = _gold("e4m3.json")
    for code, v in g["values"].items():
        got = oracle.e4m3_value(int(code))
        assert got == v and np.signbit(got) == np.signbit(v), (code, got, v)
    for code in g["nan"]:
        assert np.isnan(oracle.e4m3_value(code))


def test_e4m3_all_codes_match_torch_float8():
    """Every one of the 256 codes against torch's float8_e4m3fn decoding (a
    library implementation of the same format)."""
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.fp8_dequant(codes[None, :], np.ones(1, np.float32))[0]
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin]) and np.array_equal(np.signbit(got[fin]), np.signbit(ref[fin]))


def _e4m3_code_of_int(v):
    """E4M3 code of a small integer |v| <= 15 (exact): written out from the format."""
    if v == 0:
        return 0
    s = 0x80 if v < 0 else 0
    a = abs(v)
    e = a.bit_length() - 1            # a = 2^e * (1 + m/8)
    m = ((a << 3) >> e) & 7
    return s | ((e + 7) << 3) | m


def test_fp8_scores_reduce_to_integer_bf16_case():
    """Codes of small integers with descales 1 are the integer inputs of the
    exact bf16 case: the fp8 path's scores equal that case's scores exactly."""
    rng = np.random.default_rng(31)
    T, Hi, d = 9, 4, 16
    qi = rng.integers(-4, 5, size=(T, Hi, d))
    ki = rng.integers(-4, 5, size=(T, d))
    w = rng.integers(1, 5, size=(T, Hi)).astype(np.float64)
    enc = np.vectorize(_e4m3_code_of_int)
    q8, k8 = enc(qi).astype(np.uint8), enc(ki).astype(np.uint8)
    start, length = oracle.thd_metadata(np.array([0, 4, 9], np.int32), T)
    ref = oracle.indexer_scores(qi.astype(np.float64), ki.astype(np.float64), w, start, length, 5)
    got = oracle.indexer_scores(oracle.fp8_dequant(q8, np.ones((T, Hi), np.float32)),
                                oracle.fp8_dequant(k8, np.ones(T, np.float32)), w, start, length, 5)
    assert np.array_equal(got, ref)


def test_fp8_descales_scale_rows_and_columns():
    """score is positively homogeneous in each descale: doubling q_scale of
    every head of row t doubles row t; doubling k_scale of key s doubles
    column s - start of every row that sees it."""
    rng = np.random.default_rng(32)
    T, Hi, d = 12, 4, 32
    q8 = rng.integers(0, 256, size=(T, Hi, d)).astype(np.uint8)
    q8[(q8 & 0x7F) == 0x7F] = 0x38  # no NaN codes
    k8 = rng.integers(0, 256, size=(T, d)).astype(np.uint8)
    k8[(k8 & 0x7F) == 0x7F] = 0x38
    qs = rng.uniform(0.5, 2.0, size=(T, Hi)).astype(np.float32)
    ks = rng.uniform(0.5, 2.0, size=T).astype(np.float32)
    w = rng.random((T, Hi))
    start, length = oracle.thd_metadata(np.array([0, T], np.int32), T)
    base = oracle.indexer_scores(oracle.fp8_dequant(q8, qs), oracle.fp8_dequant(k8, ks), w, start, length, T)
    qs2 = qs.copy(); qs2[5] *= 2
    r = oracle.indexer_scores(oracle.fp8_dequant(q8, qs2), oracle.fp8_dequant(k8, ks), w, start, length, T)
    fin = np.isfinite(base)
    assert np.allclose(r[5][fin[5]], 2 * base[5][fin[5]], rtol=1e-12)
    assert np.array_equal(np.delete(r, 5, 0), np.delete(base, 5, 0))
    ks2 = ks.copy(); ks2[3] *= 2
    r = oracle.indexer_scores(oracle.fp8_dequant(q8, qs), oracle.fp8_dequant(k8, ks2), w, start, length, T)
    assert np.allclose(r[3:, 3], 2 * base[3:, 3], rtol=1e-12)
    assert np.array_equal(np.delete(r, 3, 1), np.delete(base, 3, 1))


def test_e8m0_golden_values():
    g = _gold("e8m0.json")
    for code, v in g["values"].items():
        assert oracle.e8m0_value(int(code)) == v, code
    for code in g["nan"]:
        assert np.isnan(oracle.e8m0_value(code))


def test_mxfp8_unit_scales_reduce_to_e4m3():
    """With every E8M0 scale 127 (the power 1) the block-scaled decoding is
    the plain E4M3 decoding of the per-row-descale path with descale 1."""
    rng = np.random.default_rng(41)
    codes = rng.integers(0, 256, size=(6, 128)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38
    got = oracle.mxfp8_dequant(codes, np.full((6, 4), 127, np.uint8))
    ref = oracle.fp8_dequant(codes, np.ones(6, np.float32))
    assert np.array_equal(got, ref)


def test_mxfp8_block_scaled_score_closed_form():
    """One query head and one key of 128 elements, every code 1.0 (0x38),
    scales 2^b on the query's block b: the score is 32 * (1 + 2 + 4 + 8) =
    480.  With the key's scales 2^(3-b) every block contributes 32 * 8: 1024.
    A block of -1.0 codes (0xB8) subtracts its share, and a negative total is
    cut by the ReLU."""
    q = np.full((1, 1, 128), 0x38, np.uint8)
    k = np.full((1, 128), 0x38, np.uint8)
    w = np.ones((1, 1))
    st, ln = np.zeros(1, np.int32), np.ones(1, np.int32)
    qs = np.array([[[127, 128, 129, 130]]], np.uint8)

    def score(qc, qsc, kc, ksc):
        return oracle.indexer_scores(oracle.mxfp8_dequant(qc, qsc), oracle.mxfp8_dequant(kc, ksc), w, st, ln, 1)[0, 0]

    assert score(q, qs, k, np.full((1, 4), 127, np.uint8)) == 480.0
    assert score(q, qs, k, np.array([[130, 129, 128, 127]], np.uint8)) == 1024.0
    qn = q.copy()
    qn[0, 0, 64:96] = 0xB8  # block 2 (scale 4) negated: 32 * (1 + 2 - 4 + 8)
    assert score(qn, qs, k, np.full((1, 4), 127, np.uint8)) == 224.0
    qn[0, 0, 96:128] = 0xB8  # blocks 2 and 3 negated: 32 * (1 + 2 - 4 - 8) < 0
    assert score(qn, qs, k, np.full((1, 4), 127, np.uint8)) == 0.0


def test_mxfp8_scale_moves_only_its_block():
    """Raising one scale byte of one row by 1 doubles exactly the 32 elements
    of that block of that row; every other element is unchanged."""
    rng = np.random.default_rng(42)
    codes = rng.integers(0, 256, size=(5, 3, 64)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38
    sc = rng.integers(110, 140, size=(5, 3, 2)).astype(np.uint8)
    base = oracle.mxfp8_dequant(codes, sc)
    sc2 = sc.copy()
    sc2[3, 1, 1] += 1
    r = oracle.mxfp8_dequant(codes, sc2)
    assert np.array_equal(r[3, 1, 32:], 2 * base[3, 1, 32:])
    mask = np.ones(base.shape, bool)
    mask[3, 1, 32:] = False
    assert np.array_equal(r[mask], base[mask])


def _rand_bf16_like(rng, shape, lo=-4, hi=4):
    return rng.integers(lo, hi + 1, size=shape).astype(np.float64)


def test_indexer_single_head_is_relu_matmul():
    # Hi = 1, w = 1: score[t, j] = max(0, qi[t] . ki[start + j]) -- a plain matmul.
    rng = np.random.default_rng(11)
    T, d = 13, 7
    qi = rng.standard_normal((T, 1, d))
    ki = rng.standard_normal((T, d))
    w = np.ones((T, 1))
    start, length = oracle.thd_metadata(np.array([0, T]), T)
    got = oracle.indexer_scores(qi, ki, w, start, length, T)
    ref = np.maximum(qi[:, 0, :] @ ki.T, 0.0)
    for t in range(T):
        np.testing.assert_allclose(got[t, : t + 1], ref[t, : t + 1], rtol=1e-13, atol=1e-13)
        assert np.all(np.isneginf(got[t, t + 1:]))


def test_indexer_one_hot_weights_select_the_head():
    # w = e_h picks head h alone; distinct data per head catches a head/dim mix-up.
    rng = np.random.default_rng(12)
    T, Hi, d = 9, 3, 5
    qi = rng.standard_normal((T, Hi, d))
    ki = rng.standard_normal((T, d))
    start, length = oracle.thd_metadata(np.array([0, T]), T)
    for h in range(Hi):
        w = np.zeros((T, Hi))
        w[:, h] = 2.5
        got = oracle.indexer_scores(qi, ki, w, start, length, T)
        ref = 2.5 * np.maximum(qi[:, h, :] @ ki.T, 0.0)
        for t in range(T):
            np.testing.assert_allclose(got[t, : t + 1], ref[t, : t + 1], rtol=1e-13, atol=1e-13)


def test_indexer_linear_in_weights_and_sign():
    rng = np.random.default_rng(13)
    T, Hi, d = 8, 4, 6
    qi = rng.standard_normal((T, Hi, d))
    ki = rng.standard_normal((T, d))
    start, length = oracle.thd_metadata(np.array([0, T]), T)
    w1 = rng.random((T, Hi))
    w2 = rng.random((T, Hi))
    s1 = oracle.indexer_scores(qi, ki, w1, start, length, T)
    s2 = oracle.indexer_scores(qi, ki, w2, start, length, T)
    s12 = oracle.indexer_scores(qi, ki, w1 + w2, start, length, T)
    sneg = oracle.indexer_scores(qi, ki, -w1, start, length, T)
    for t in range(T):
        np.testing.assert_allclose(s12[t, : t + 1], s1[t, : t + 1] + s2[t, : t + 1], rtol=1e-12)
        np.testing.assert_allclose(sneg[t, : t + 1], -s1[t, : t + 1], rtol=1e-14)
        assert np.all(s1[t, : t + 1] >= 0.0)


def test_indexer_document_isolation_and_mask():
    # THD: a token sees exactly the keys from its document start to itself.
    rng = np.random.default_rng(14)
    cu = np.array([0, 4, 5, 11])
    T, Hi, d = 11, 2, 3
    qi = _rand_bf16_like(rng, (T, Hi, d))
    ki = _rand_bf16_like(rng, (T, d))
    w = _rand_bf16_like(rng, (T, Hi), 1, 4)
    start, length = oracle.thd_metadata(cu, T)
    s_max = int(np.max(np.diff(cu)))
    base = oracle.indexer_scores(qi, ki, w, start, length, s_max)
    # finite exactly on j < len, -inf beyond
    for t in range(T):
        assert np.all(np.isfinite(base[t, : length[t]]))
        assert np.all(np.isneginf(base[t, length[t]:]))
    # scramble the keys of every other document: row t is unchanged
    for b in range(len(cu) - 1):
        ki2 = ki.copy()
        others = [r for r in range(T) if not (cu[b] <= r < cu[b + 1])]
        ki2[others] = _rand_bf16_like(rng, (len(others), d))
        s2 = oracle.indexer_scores(qi, ki2, w, start, length, s_max)
        rows = slice(cu[b], cu[b + 1])
        np.testing.assert_array_equal(s2[rows], base[rows])
    # the diagonal (key == query) is included: brute-force one entry by hand
    t = 7
    j = length[t] - 1
    assert start[t] + j == t
    hand = sum(w[t, h] * max(0.0, float(np.dot(qi[t, h], ki[t]))) for h in range(Hi))
    assert base[t, j] == hand


def test_indexer_integer_inputs_are_exact_and_bounded():
    # The tiny workload's integer inputs give integer scores below 2^24 (exact in fp32).
    rng = np.random.default_rng(15)
    T, Hi, d = 32, 8, 64
    qi = _rand_bf16_like(rng, (T, Hi, d))
    ki = _rand_bf16_like(rng, (T, d))
    w = _rand_bf16_like(rng, (T, Hi), 1, 4)
    start, length = oracle.thd_metadata(np.array([0, T]), T)
    s, a = oracle.indexer_scores(qi, ki, w, start, length, T, want_abs=True)
    fin = np.isfinite(s)
    assert np.all(s[fin] == np.round(s[fin]))
    assert np.all(np.abs(s[fin]) <= a[fin])
    assert np.max(a[fin]) < 2 ** 24


# -------------------------------------------------------------------- top-k
def test_topk_golden_ties():
    g = _gold("topk_ties.json")
    for c in g["k_cases"]:
        idx, tl = oracle.topk(np.array([c["scores"]], float), np.array([c["len"]]), c["k"],
                              start_rows=np.array([c["start"]]))
        assert idx[0].tolist() == c["idx"]
        assert tl[0] == c["topk_length"]


def _brute_topk(scores, k):
    """The unique subset whose every member beats every non-member under
    (score descending, index ascending), found by enumerating all subsets."""
    n = len(scores)
    m = min(k, n)

    def beats(a, b):
        return scores[a] > scores[b] or (scores[a] == scores[b] and a < b)

    found = []
    for sub in itertools.combinations(range(n), m):
        rest = [j for j in range(n) if j not in sub]
        if all(beats(a, b) for a in sub for b in rest):
            found.append(sorted(sub))
    assert len(found) == 1
    return found[0]


def test_topk_brute_force_small_with_ties():
    rng = np.random.default_rng(21)
    for trial in range(300):
        n = int(rng.integers(0, 10))
        k = int(rng.integers(1, 6))
        ld = 10
        row = np.full(ld, -np.inf)
        row[:n] = rng.integers(-2, 3, size=n)  # heavy ties
        start = int(rng.integers(0, 100))
        idx, tl = oracle.topk(row[None], np.array([n]), k, start_rows=np.array([start]))
        want = [start + j for j in _brute_topk(list(row[:n]), k)] if n else []
        assert idx[0, : len(want)].tolist() == want, (trial, row, k)
        assert np.all(idx[0, len(want):] == -1)
        assert tl[0] == len(want)


def test_topk_distinct_scores_match_argsort():
    rng = np.random.default_rng(22)
    n, k = 500, 37
    row = rng.permutation(n).astype(float) * 0.5 - 100
    idx, tl = oracle.topk(row[None], np.array([n]), k)
    want = np.sort(np.argsort(-row, kind="stable")[:k])
    np.testing.assert_array_equal(idx[0], want)
    assert tl[0] == k


def test_topk_all_equal_takes_lowest_indices():
    n, k = 50, 8
    idx, _ = oracle.topk(np.zeros((1, n)), np.array([n]), k, start_rows=np.array([1000]))
    assert idx[0].tolist() == list(range(1000, 1008))


def test_topk_invariants_random():
    rng = np.random.default_rng(23)
    T, ld, k = 40, 300, 64
    lens = rng.integers(0, ld + 1, size=T)
    sc = rng.integers(0, 40, size=(T, ld)).astype(float)
    starts = rng.integers(0, 5000, size=T)
    idx, tl = oracle.topk(sc, lens, k, start_rows=starts)
    for t in range(T):
        n = min(k, lens[t])
        assert tl[t] == n
        sel = idx[t, :n] - starts[t]
        assert np.all(np.diff(sel) > 0) and np.all(idx[t, n:] == -1)
        assert np.all((sel >= 0) & (sel < lens[t]))
        rest = np.setdiff1d(np.arange(lens[t]), sel)
        if rest.size and n:
            # every selected score >= every unselected one; at equality the
            # selected index is the smaller one
            minsel = sc[t, sel].min()
            assert np.all(sc[t, rest] <= minsel)
            tied = rest[sc[t, rest] == minsel]
            assert np.all(tied > sel[sc[t, sel] == minsel].max())


# ----------------------------------------------------------- compact / sort
def test_compact_sort_golden():
    g = _gold("compact_sort.json")
    out, lengths = oracle.compact_sort(np.array(g["in"]), g["key_count"])
    assert out.tolist() == g["out"]
    assert lengths.tolist() == g["lengths"]


def test_compact_sort_matches_numpy_sort():
    rng = np.random.default_rng(31)
    T, K, kc = 50, 33, 40
    ind = rng.integers(-5, 50, size=(T, K)).astype(np.int32)
    out, lengths = oracle.compact_sort(ind, kc)
    for t in range(T):
        v = np.sort(ind[t][(ind[t] >= 0) & (ind[t] < kc)])
        assert lengths[t] == v.size
        np.testing.assert_array_equal(out[t, : v.size], v)
        assert np.all(out[t, v.size:] == -1)


# ----------------------------------------------------------- route packing
def test_pack_routes_golden():
    g = _gold("pack_routes.json")
    out = oracle.pack_routes(np.array(g["routes"]))
    assert out.tolist() == g["packed"]


def test_pack_routes_invariants():
    rng = np.random.default_rng(41)
    B, S, W = 3, 17, 10
    r = rng.integers(-3, S + 3, size=(B, S, W)).astype(np.int32)
    out = oracle.pack_routes(r)
    assert out.shape == (B * S, 12)
    assert np.all(out[:, W:] == -1)
    valid = (r >= 0) & (r < S)
    assert np.array_equal(out[:, :W] >= 0, valid.reshape(B * S, W))
    b_of_row = np.repeat(np.arange(B), S)
    ok = out[:, :W] >= 0
    assert np.all((out[:, :W][ok] // S) == np.broadcast_to(b_of_row[:, None], (B * S, W))[ok])
    assert np.all((out[:, :W][ok] % S) == r.reshape(B * S, W)[ok])


# --------------------------------------------------------------- attention
def test_attention_golden_hand_example():
    g = _gold("attention_hand.json")
    res = oracle.sparse_attn(np.array(g["q"]), np.array(g["kv"]), np.array(g["idx"]), math.log(3) / 2,
                             sink=np.array(g["sink"]), dv=1)
    np.testing.assert_allclose(res["out"], np.array(g["out"]), rtol=1e-14)
    assert res["lse"][0, 0] == pytest.approx(math.log(g["lse_ln"]), rel=1e-14)
    assert res["lse_kv"][0, 0] == pytest.approx(math.log(g["lse_kv_ln"]), rel=1e-14)
    assert res["max_logits"][0, 0] == pytest.approx(math.log(g["max_logits_ln"]), rel=1e-14)


def _dense_causal_with_sink(q, kv, sink, scale, dv, t):
    """Dense causal attention for row t with the sink as an extra logit whose
    value vector is zero, through scipy's softmax/logsumexp."""
    logits = scale * q[t] @ kv[: t + 1].T                  # [H, t+1]
    full = np.concatenate([logits, sink[:, None]], axis=1)  # sink as one more column
    p = softmax(full, axis=1)
    out = p[:, :-1] @ kv[: t + 1, :dv]
    return out, logsumexp(full, axis=1), logsumexp(logits, axis=1), logits.max(axis=1), p


@pytest.mark.parametrize("qscale", [1.0, 30.0])
def test_attention_all_selected_equals_dense(qscale):
    rng = np.random.default_rng(51)
    T, H, Dqk, Dv = 12, 3, 10, 6
    q = rng.standard_normal((T, H, Dqk)) * qscale
    kv = rng.standard_normal((T, Dqk))
    sink = rng.standard_normal(H) * 3
    K = T
    idx = np.full((T, K), -1, np.int32)
    for t in range(T):
        idx[t, : t + 1] = rng.permutation(t + 1)  # every causal key, in any slot order
    res = oracle.sparse_attn(q, kv, idx, 0.37, sink=sink, dv=Dv)
    for t in range(T):
        out, lse, lse_kv, ml, p = _dense_causal_with_sink(q, kv, sink, 0.37, Dv, t)
        np.testing.assert_allclose(res["out"][t], out, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(res["lse"][t], lse, rtol=1e-12)
        np.testing.assert_allclose(res["lse_kv"][t], lse_kv, rtol=1e-12)
        np.testing.assert_allclose(res["max_logits"][t], ml, rtol=1e-12)
        np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=1e-12)


def test_attention_single_key_no_sink():
    rng = np.random.default_rng(52)
    q = rng.standard_normal((1, 2, 8))
    kv = rng.standard_normal((5, 8))
    res = oracle.sparse_attn(q, kv, np.array([[3, -1, -1]]), 0.5, dv=4)
    np.testing.assert_allclose(res["out"][0], np.broadcast_to(kv[3, :4], (2, 4)), rtol=1e-14)
    np.testing.assert_allclose(res["lse"][0], 0.5 * q[0] @ kv[3], rtol=1e-13)


def test_attention_identical_keys_closed_form():
    # n copies of one key: out = V * n e^s / (n e^s + e^sink).
    rng = np.random.default_rng(53)
    q = rng.standard_normal((1, 4, 6))
    kv = rng.standard_normal((3, 6))
    sink = rng.standard_normal(4)
    n = 5
    res = oracle.sparse_attn(q, kv, np.array([[1] * n + [-1]]), 0.8, sink=sink, dv=6)
    s = 0.8 * q[0] @ kv[1]
    frac = n * np.exp(s) / (n * np.exp(s) + np.exp(sink))
    np.testing.assert_allclose(res["out"][0], frac[:, None] * kv[1][None, :], rtol=1e-12)
    np.testing.assert_allclose(res["lse"][0], np.log(n * np.exp(s) + np.exp(sink)), rtol=1e-12)


def test_attention_slot_semantics():
    rng = np.random.default_rng(54)
    T, H, D, Tkv, K = 6, 2, 8, 20, 7
    q = rng.standard_normal((T, H, D))
    kv = rng.standard_normal((Tkv, D))
    sink = rng.standard_normal(H)
    idx = rng.integers(0, Tkv, size=(T, K)).astype(np.int32)
    base = oracle.sparse_attn(q, kv, idx, 0.3, sink=sink, dv=5)
    # slot order is irrelevant
    perm = oracle.sparse_attn(q, kv, idx[:, rng.permutation(K)], 0.3, sink=sink, dv=5)
    np.testing.assert_allclose(perm["out"], base["out"], rtol=1e-12)
    # invalid and out-of-range slots are absent slots
    bad = np.concatenate([idx, np.array([[-1, Tkv, Tkv + 5, -7]] * T, np.int32)], axis=1)
    withbad = oracle.sparse_attn(q, kv, bad, 0.3, sink=sink, dv=5)
    np.testing.assert_allclose(withbad["out"], base["out"], rtol=1e-13)
    np.testing.assert_allclose(withbad["lse"], base["lse"], rtol=1e-13)
    # topk_length truncation equals -1 padding; lengths clamp to [0, K]
    lens = np.array([0, 3, 7, 9, -2, 5], np.int32)
    trunc = oracle.sparse_attn(q, kv, idx, 0.3, sink=sink, dv=5, topk_length=lens)
    pad = idx.copy()
    for t in range(T):
        pad[t, max(0, min(K, lens[t])):] = -1
    padded = oracle.sparse_attn(q, kv, pad, 0.3, sink=sink, dv=5)
    np.testing.assert_allclose(trunc["out"], padded["out"], rtol=1e-13)
    np.testing.assert_allclose(trunc["lse"], padded["lse"], rtol=1e-13)
    # lse (with sink) = logaddexp(lse_kv, sink) on non-empty rows
    np.testing.assert_allclose(base["lse"], np.logaddexp(base["lse_kv"], sink[None, :]), rtol=1e-12)


def test_attention_empty_rows():
    q = np.ones((2, 3, 4))
    kv = np.ones((4, 4))
    sink = np.array([0.5, -1.0, 2.0])
    res = oracle.sparse_attn(q, kv, np.full((2, 3), -1, np.int32), 1.0, sink=sink, dv=2)
    assert np.all(res["out"] == 0.0)
    assert np.all(np.isposinf(res["lse_kv"])) and np.all(np.isneginf(res["max_logits"]))
    np.testing.assert_array_equal(res["lse"], np.broadcast_to(sink, (2, 3)))
    nos = oracle.sparse_attn(q, kv, np.full((2, 3), -1, np.int32), 1.0, dv=2)
    assert np.all(np.isneginf(nos["lse"]))


def test_attention_separate_v_equals_latent_layout():
    # With V separate: pad q with zeros in front of kv' = [v | k]; V' = first Dv columns.
    rng = np.random.default_rng(55)
    T, H, Dk, Dv, Tkv, K = 5, 3, 6, 4, 9, 5
    q = rng.standard_normal((T, H, Dk))
    k = rng.standard_normal((Tkv, Dk))
    v = rng.standard_normal((Tkv, Dv))
    idx = rng.integers(-1, Tkv, size=(T, K)).astype(np.int32)
    a = oracle.sparse_attn(q, k, idx, 0.6, v=v)
    q2 = np.concatenate([np.zeros((T, H, Dv)), q], axis=2)
    kv2 = np.concatenate([v, k], axis=1)
    b = oracle.sparse_attn(q2, kv2, idx, 0.6, dv=Dv)
    np.testing.assert_allclose(a["out"], b["out"], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(a["lse"], b["lse"], rtol=1e-12)


# ---------------------------------------------------- attention: lse_indexer
def test_lse_indexer_golden_hand_example():
    g = _gold("attention_hand.json")
    for P, ln_arg in g["lse_indexer_ln"].items():
        res = oracle.sparse_attn(np.array(g["q"]), np.array(g["kv"]), np.array(g["idx"]), math.log(3) / 2,
                                 sink=np.array(g["sink"]), dv=1, indexer_topk=int(P))
        assert res["lse_indexer"][0, 0] == pytest.approx(math.log(ln_arg), rel=1e-14), P


def test_lse_indexer_prefix_and_suffix_make_lse_kv():
    """The prefix LSE and the LSE of the remaining slots combine to the
    KV-only LSE of the whole row; a full prefix is that LSE itself; the prefix
    LSE grows with the prefix."""
    rng = np.random.default_rng(56)
    T, H, D, Tkv, K = 7, 3, 9, 40, 16
    q = rng.standard_normal((T, H, D)) * 2
    kv = rng.standard_normal((Tkv, D))
    sink = rng.standard_normal(H)
    idx = rng.integers(-2, Tkv + 2, size=(T, K)).astype(np.int32)  # some invalid ids
    idx[:, 0] = rng.integers(0, Tkv, size=T)                        # every row has a valid slot
    full = oracle.sparse_attn(q, kv, idx, 0.4, sink=sink, dv=4, indexer_topk=K)
    np.testing.assert_allclose(full["lse_indexer"], full["lse_kv"], rtol=1e-13)
    prev = None
    for P in (1, 5, 8, 13):
        pre = oracle.sparse_attn(q, kv, idx, 0.4, sink=sink, dv=4, indexer_topk=P)["lse_indexer"]
        suf_idx = idx.copy()
        suf_idx[:, :P] = -1
        suf = oracle.sparse_attn(q, kv, suf_idx, 0.4, sink=sink, dv=4)["lse_kv"]
        both = np.logaddexp(pre, np.where(np.isinf(suf), -np.inf, suf))
        np.testing.assert_allclose(both, full["lse_kv"], rtol=1e-12)
        if prev is not None:
            assert np.all(pre >= prev - 1e-12)
        prev = pre


def test_lse_indexer_empty_and_truncated():
    rng = np.random.default_rng(57)
    q = rng.standard_normal((3, 2, 5))
    kv = rng.standard_normal((6, 5))
    idx = np.array([[-1, -1, -1, -1], [-1, 2, 3, 4], [1, 2, 3, 4]], np.int32)
    res = oracle.sparse_attn(q, kv, idx, 1.0, dv=3, indexer_topk=1)
    assert np.all(np.isposinf(res["lse_indexer"][:2]))   # empty row; prefix of invalid ids only
    assert np.all(np.isfinite(res["lse_indexer"][2]))
    # topk_length shorter than the prefix: the prefix covers every valid slot
    tl = np.array([0, 2, 3], np.int32)
    r2 = oracle.sparse_attn(q, kv, idx, 1.0, dv=3, topk_length=tl, indexer_topk=4)
    np.testing.assert_allclose(r2["lse_indexer"][1:], r2["lse_kv"][1:], rtol=1e-13)
    assert np.all(np.isposinf(r2["lse_indexer"][0]))


# ------------------------------------------------- top-k logits and softmax
def _ln(v):
    return {"ln2": math.log(2), "ln3": math.log(3), "ln7": math.log(7)}.get(v, v)


def test_topk_softmax_golden():
    g = _gold("topk_softmax.json")
    sc = np.array([[_ln(v) for v in row] for row in g["scores"]], np.float64)
    idx, tl = oracle.topk(sc, np.array(g["length"], np.int32), g["k"], start_rows=np.array(g["start"], np.int32))
    assert idx.tolist() == g["idx"]
    logits, sm, lse = oracle.topk_softmax(sc, idx, tl, start_rows=np.array(g["start"], np.int32))
    for r in range(3):
        for j in range(2):
            want = g["logits_ln"][r][j]
            if want is None:
                assert np.isneginf(logits[r, j])
            else:
                assert logits[r, j] == pytest.approx(math.log(want), rel=1e-15)
            assert sm[r, j] == pytest.approx(g["softmax"][r][j], rel=1e-14, abs=1e-300)
        if g["lse_ln"][r] is None:
            assert np.isneginf(lse[r])
        else:
            assert lse[r] == pytest.approx(math.log(g["lse_ln"][r]), rel=1e-14)


def test_topk_softmax_invariants():
    rng = np.random.default_rng(58)
    T, ld, k = 40, 300, 64
    sc = rng.standard_normal((T, ld)) * 3
    lengths = rng.integers(0, ld + 1, size=T).astype(np.int32)
    lengths[:3] = [0, 1, k]
    idx, tl = oracle.topk(sc, lengths, k)
    logits, sm, lse = oracle.topk_softmax(sc, idx, tl)
    for t in range(T):
        n = tl[t]
        assert np.all(np.isneginf(logits[t, n:])) and np.all(sm[t, n:] == 0.0)
        if n == 0:
            assert np.isneginf(lse[t])
            continue
        assert sm[t, :n].sum() == pytest.approx(1.0, rel=1e-12)
        # the selected logits are the top-n scores of the row, aligned with the ids
        np.testing.assert_array_equal(logits[t, :n], sc[t, idx[t, :n]])
        assert logits[t, :n].min() >= np.sort(sc[t, : lengths[t]])[::-1][n - 1]
        # probability ratios are exponentials of logit differences
        np.testing.assert_allclose(sm[t, 1:n] / sm[t, 0], np.exp(logits[t, 1:n] - logits[t, 0]), rtol=1e-12)
        assert lse[t] >= logits[t, :n].max()
    # shifting every score shifts the lse and leaves the softmax alone
    l2, s2, e2 = oracle.topk_softmax(sc + 2.5, idx, tl)
    np.testing.assert_allclose(s2, sm, rtol=1e-12, atol=1e-300)
    fin = np.isfinite(lse)
    np.testing.assert_allclose(e2[fin], lse[fin] + 2.5, rtol=1e-13)



# ------------------------------------------------------- attention backward
def _bwd_case(rng, n=3, H=3, Dqk=12, Dv=8, Tkv=10, K=7):
    q = rng.standard_normal((n, H, Dqk))
    kv = rng.standard_normal((Tkv, Dqk))
    idx = rng.integers(-2, Tkv + 2, size=(n, K)).astype(np.int32)
    idx[0, :3] = [4, 4, 7]            # a duplicate pair
    tl = np.array([K, 4, 0][:n], np.int32)  # a truncated row and an empty one
    sink = rng.standard_normal(H)
    dout = rng.standard_normal((n, H, Dv))
    return q, kv, idx, tl, sink, dout


def _loss(q, kv, idx, tl, sink, dout, scale, Dv):
    f = oracle.sparse_attn(q, kv, idx, scale, topk_length=tl, sink=sink, dv=Dv)
    return float(np.sum(f["out"] * dout))


def test_attn_bwd_matches_finite_differences():
    """Every gradient against central differences of sum(dout * out) through
    the (separately pinned) forward oracle, in fp64."""
    rng = np.random.default_rng(41)
    q, kv, idx, tl, sink, dout = _bwd_case(rng)
    scale, Dv, eps = 0.37, dout.shape[2], 1e-6
    f = oracle.sparse_attn(q, kv, idx, scale, topk_length=tl, sink=sink, dv=Dv)
    dq, dkv, ds = oracle.sparse_attn_bwd(q, kv, idx, scale, f["out"], dout, f["lse_kv"], topk_length=tl, sink=sink)
    for name, x, g in (("q", q, dq), ("kv", kv, dkv), ("sink", sink, ds)):
        num = np.zeros_like(x)
        for i in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[i] += eps
            xm[i] -= eps
            args = {"q": q, "kv": kv, "sink": sink}
            lp = _loss(**{**args, name: xp}, idx=idx, tl=tl, dout=dout, scale=scale, Dv=Dv)
            lm = _loss(**{**args, name: xm}, idx=idx, tl=tl, dout=dout, scale=scale, Dv=Dv)
            num[i] = (lp - lm) / (2 * eps)
        assert np.allclose(g, num, rtol=1e-6, atol=1e-8), (name, np.max(np.abs(g - num)))


def test_attn_bwd_single_key_closed_form():
    """One valid key, no sink: P = 1 and out = v, so delta = dP and dS = 0:
    dq = 0 and the key row receives exactly dout on its value dims."""
    rng = np.random.default_rng(42)
    H, Dqk, Dv = 2, 6, 4
    q = rng.standard_normal((1, H, Dqk))
    kv = rng.standard_normal((5, Dqk))
    idx = np.array([[3, -1]], np.int32)
    dout = rng.standard_normal((1, H, Dv))
    f = oracle.sparse_attn(q, kv, idx, 0.5, dv=Dv)
    dq, dkv, ds = oracle.sparse_attn_bwd(q, kv, idx, 0.5, f["out"], dout, f["lse_kv"])
    assert np.allclose(dq, 0.0, atol=1e-14)
    want = np.zeros_like(kv)
    want[3, :Dv] = dout[0].sum(axis=0)
    assert np.allclose(dkv, want, atol=1e-14) and np.all(ds == 0.0)


def test_attn_bwd_empty_row_contributes_nothing():
    rng = np.random.default_rng(43)
    q, kv, idx, tl, sink, dout = _bwd_case(rng)
    tl = np.zeros_like(tl)
    f = oracle.sparse_attn(q, kv, idx, 0.3, topk_length=tl, sink=sink, dv=dout.shape[2])
    dq, dkv, ds = oracle.sparse_attn_bwd(q, kv, idx, 0.3, f["out"], dout, f["lse_kv"], topk_length=tl, sink=sink)
    assert np.all(dq == 0.0) and np.all(dkv == 0.0) and np.all(ds == 0.0)
