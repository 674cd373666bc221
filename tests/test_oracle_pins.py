"""Pins for the oracle: values the pages print, closed forms, invariants and
independent brute force.  CPU only (no GPU, no CUDA library).

Each test pins the oracle to something other than itself, so that a dropped
term, a wrong sign or index, or a transposed operand in oracle/ fails here.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import MaskSpec
from tests.conftest import letter_matrix, nums, read_golden
import workloads

# ---------------------------------------------------------------------------
# Online softmax and the merge law ("Pallas Kernels and Splash Attention",
# §5.1, exercises 7 and 8).
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("fixture", ["online_softmax_example.txt", "exercise7_online_softmax.txt"])
def test_online_softmax_worked_examples(fixture):
    g = read_golden(fixture)
    x = nums(g["x"])
    dec = int(g["decimals"])
    trace, sm = oracle.online_softmax_trace(x, int(g["block"]))
    assert [round(m, dec) for m, _ in trace] == nums(g["trace_m"])
    assert [round(l, dec) for _, l in trace] == nums(g["trace_l"])
    # the online result is the direct two-pass softmax
    np.testing.assert_allclose(sm, oracle.safe_softmax(x), rtol=0, atol=1e-15)
    if "softmax" in g:
        assert [round(p, dec) for p in sm] == nums(g["softmax"])


def test_merge_law_equals_full_row():
    rng = np.random.default_rng(7)
    for trial in range(50):
        n = int(rng.integers(2, 300))
        s = rng.normal(scale=3.0, size=n)
        v = rng.normal(size=(n, 16))
        cut = int(rng.integers(1, n))
        m1, l1, o1 = oracle.partial_state(s[:cut], v[:cut])
        m2, l2, o2 = oracle.partial_state(s[cut:], v[cut:])
        m, l, o = oracle.merge(m1, l1, o1, m2, l2, o2)
        full = oracle.safe_softmax(s) @ v
        np.testing.assert_allclose(o, full, rtol=1e-13, atol=1e-14)
        assert m == pytest.approx(np.max(s), abs=0)
        assert l == pytest.approx(np.sum(np.exp(s - np.max(s))), rel=1e-14)


def test_merge_is_order_independent_over_many_segments():
    rng = np.random.default_rng(11)
    s = rng.normal(scale=4.0, size=1000)
    v = rng.normal(size=(1000, 8))
    cuts = np.sort(rng.choice(np.arange(1, 1000), size=9, replace=False))
    segs = np.split(np.arange(1000), cuts)
    states = [oracle.partial_state(s[i], v[i]) for i in segs]
    full = oracle.safe_softmax(s) @ v
    for order in (list(range(len(states))), list(reversed(range(len(states))))):
        m, l, o = states[order[0]]
        o = o / l
        for t in order[1:]:
            m2, l2, o2 = states[t]
            m, l, o = oracle.merge(m, l, o * l, m2, l2, o2)
        np.testing.assert_allclose(o, full, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# Max Logit Estimate ("Pallas Kernels and Splash Attention" §5.4, exercise 10).
# ---------------------------------------------------------------------------


def test_mle_exp_limits_are_the_printed_ones_and_numpys():
    g = read_golden("exercise10_mle_safe_range.txt")
    over, sub = oracle.exp_limits(np.float32)
    assert over == pytest.approx(float(g["overflow_limit"]), abs=0.05)
    assert sub == pytest.approx(float(g["subnormal_limit"]), abs=0.05)
    # brute force on float32 exp itself: finite just below, inf just above;
    # normal just above the subnormal bound, subnormal just below it
    with np.errstate(over="ignore", under="ignore"):
        assert np.isfinite(np.exp(np.float32(over - 0.01)))
        assert np.isinf(np.exp(np.float32(over + 0.01)))
        tiny = np.finfo(np.float32).tiny
        assert np.exp(np.float32(sub + 0.01)) >= tiny
        assert 0 < np.exp(np.float32(sub - 0.01)) < tiny


def test_mle_safe_range_matches_exercise10():
    g = read_golden("exercise10_mle_safe_range.txt")
    lo, hi = oracle.mle_safe_range(float(g["score_max"]), float(g["row_max_floor"]), np.float32)
    tol = float(g["tolerance"])
    assert lo == pytest.approx(float(g["c_low"]), abs=tol)
    assert hi == pytest.approx(float(g["c_high"]), abs=tol)


def test_mle_constant_cancels_inside_the_range_and_fails_outside():
    # scores spanning the exercise's [-30, 40]: one row reaching 40, one whose
    # maximum is -30
    rng = np.random.default_rng(10)
    top = np.concatenate([[40.0], rng.uniform(-30, 40, size=255)])
    low = np.concatenate([[-30.0], rng.uniform(-60, -30, size=255)])
    lo, hi = oracle.mle_safe_range(40.0, -30.0, np.float32, n_terms=256)
    for c in np.linspace(lo + 0.5, hi - 0.5, 9):
        for row in (top, low):
            w, l, lse = oracle.mle_softmax(row, c, np.float32)
            assert np.all(np.isfinite(w)) and l > 0
            # terms far below the row's maximum may flush; they weigh < 1e-6
            np.testing.assert_allclose(w, oracle.safe_softmax(row), rtol=2e-4, atol=1e-6)
            m = np.max(row)
            assert float(lse) == pytest.approx(m + np.log(np.sum(np.exp(row - m))), abs=2e-4)
    # in float64 any moderate constant gives the same weights (c cancels)
    for c in (-200.0, 0.0, 40.0, 300.0):
        w, _, _ = oracle.mle_softmax(top, c, np.float64)
        np.testing.assert_allclose(w, oracle.safe_softmax(top), rtol=1e-12, atol=0)
    # below the range the top row overflows; far above it the low row's
    # exponentials all underflow to zero
    w, l, _ = oracle.mle_softmax(top, lo - 2.0 - np.log(256), np.float32)
    assert not np.all(np.isfinite(w))
    # the sum's own bound: 256 equal maxima overflow the sum (not the terms)
    # just below c = 40 - ln(FLT_MAX) + ln(256), and not just above it
    flat = np.full(256, 40.0)
    w, l, _ = oracle.mle_softmax(flat, lo - 0.05, np.float32)
    assert np.isinf(l) and np.all(w == 0)
    w, l, _ = oracle.mle_softmax(flat, lo + 0.05, np.float32)
    assert np.isfinite(l)
    np.testing.assert_allclose(w, 1 / 256, rtol=1e-6)
    w, l, _ = oracle.mle_softmax(low, hi + 20.0, np.float32)
    assert l == 0 and not np.any(np.isfinite(w))


def test_mle_softcap_constant_is_always_safe():
    # with scores cap * tanh(.) in (-cap, cap) and c = cap, exp(s - c) <= 1
    # never overflows, and a row keeps normal exponentials while 2 cap < 87
    for cap in (10.0, 30.0, 43.0):
        s = cap * np.tanh(np.random.default_rng(int(cap)).normal(scale=5.0, size=512) / 1.0)
        s[0] = -cap * (1 - 1e-7)
        lo, hi = oracle.mle_safe_range(cap, -cap, np.float32)
        assert lo < cap < hi
        w, l, _ = oracle.mle_softmax(s, cap, np.float32)
        np.testing.assert_allclose(w, oracle.safe_softmax(s), rtol=2e-4, atol=1e-6)


# ---------------------------------------------------------------------------
# MaskInfo: the pages' worked examples (§6.1, §6.2, §6.6, exercises 11, 12).
# ---------------------------------------------------------------------------


def test_maskinfo_worked_example_causal_1024x2048():
    g = read_golden("maskinfo_causal_4096_1024x2048.txt")
    L = int(g["L"])
    mi = oracle.mask_info(MaskSpec(causal=True), L, L, int(g["bq"]), int(g["bk"]))
    assert mi.block_mask.reshape(-1).tolist() == nums(g["block_mask"], int)
    assert mi.active_rows.tolist() == nums(g["active_rows"], int)
    assert mi.active_cols.tolist() == nums(g["active_cols"], int)
    assert mi.mask_next.tolist() == nums(g["mask_next"], int)
    assert mi.bounds_start.tolist() == nums(g["bounds_start"], int)
    assert mi.bounds_end.tolist() == nums(g["bounds_end"], int)
    assert mi.num_partial == int(g["num_partial"])
    assert mi.num_patterns == int(g["num_patterns"])
    # the two patterns are the q - kv offset 0 triangle and the offset 1024 one
    p0, p1 = mi.partial_mask_blocks
    i = np.arange(1024)[:, None]
    j = np.arange(2048)[None, :]
    np.testing.assert_array_equal(p0, (j <= i).astype(np.uint8))
    np.testing.assert_array_equal(p1, (j <= i + 1024).astype(np.uint8))


def test_exercise11_causal_1024():
    g = read_golden("exercise11_causal_4096_1024.txt")
    L = int(g["L"])
    mi = oracle.mask_info(MaskSpec(causal=True), L, L, int(g["bq"]), int(g["bk"]))
    assert mi.num_active == int(g["num_active"])
    assert int(np.count_nonzero(mi.block_mask == 2)) == int(g["num_full"])
    assert mi.num_partial == int(g["num_partial"])
    assert mi.num_patterns == int(g["num_patterns"])


def test_exercise12_documents():
    g = read_golden("exercise12_documents_1000_2000_1096.txt")
    lens = nums(g["doc_lengths"], int)
    seg = workloads.segment_ids_from_lengths([lens]).numpy()
    L = seg.shape[1]
    mi = oracle.mask_info(MaskSpec(causal=False, q_segment_ids=seg, kv_segment_ids=seg), L, L,
                          int(g["bq"]), int(g["bk"]))
    assert mi.block_mask[0].tolist() == letter_matrix(g["matrix"])
    assert int(np.count_nonzero(mi.block_mask == 0)) == int(g["num_empty"])
    assert int(np.count_nonzero(mi.block_mask == 2)) == int(g["num_full"])
    assert int(np.count_nonzero(mi.block_mask == 1)) == int(g["num_partial"])


def test_picture_causal_8():
    g = read_golden("picture_causal_8_2x2.txt")
    L = int(g["L"])
    mi = oracle.mask_info(MaskSpec(causal=True), L, L, int(g["bq"]), int(g["bk"]))
    assert mi.block_mask[0].tolist() == letter_matrix(g["matrix"])


def test_pattern_counts_16384():
    g = read_golden("pattern_counts_16384_1024.txt")
    L, bq, bk = int(g["L"]), int(g["bq"]), int(g["bk"])
    assert oracle.mask_info(MaskSpec(causal=True), L, L, bq, bk).num_patterns == int(g["causal_patterns"])
    wl = int(g["local_window_left"])
    mi = oracle.mask_info(MaskSpec(causal=True, window_left=wl, window_right=0), L, L, bq, bk)
    assert mi.num_patterns == int(g["local_patterns"])
    # a symmetric local band of the same block-aligned width also has two
    sym = oracle.mask_info(MaskSpec(causal=False, window_left=wl, window_right=wl), L, L, bq, bk)
    assert sym.num_patterns == int(g["local_patterns"])


# ---------------------------------------------------------------------------
# Closed forms for causal, windowed and document masks.
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("L,b", [(256, 64), (1024, 128), (4096, 128), (512, 16)])
def test_causal_closed_form_square_blocks(L, b):
    n = L // b
    mi = oracle.mask_info(MaskSpec(causal=True), L, L, b, b)
    assert mi.num_active == n * (n + 1) // 2
    assert mi.num_partial == n
    assert mi.num_patterns == 1
    assert mi.allowed_pairs == L * (L + 1) // 2


@pytest.mark.parametrize("L,bq,bk", [(1024, 64, 128), (1024, 128, 64), (768, 32, 96), (4096, 1024, 2048),
                                     (4096, 256, 128)])
def test_causal_closed_form_rectangular_blocks(L, bq, bk):
    nq, nk = L // bq, L // bk
    mi = oracle.mask_info(MaskSpec(causal=True), L, L, bq, bk)
    for i in range(nq):
        active = min(nk, ((i + 1) * bq - 1) // bk + 1)
        full = min(nk, (i * bq + 1) // bk)
        row = mi.block_mask[0, i]
        assert int(np.count_nonzero(row)) == active
        assert int(np.count_nonzero(row == 2)) == full
    assert mi.allowed_pairs == L * (L + 1) // 2


def test_causal_tall_blocks_two_patterns():
    # bq = 2 bk, causal: row i holds 2i + 2 active blocks, of which the last
    # two are partial -- block 2i (the upper half on the diagonal, the lower
    # half full) and block 2i + 1 (the upper half empty, the lower half on
    # the diagonal) -- and every row repeats the same two patterns
    L, bq, bk = 4096, 256, 128
    mi = oracle.mask_info(MaskSpec(causal=True), L, L, bq, bk)
    n = L // bq
    assert mi.num_active == sum(2 * i + 2 for i in range(n)) == 272
    assert mi.num_partial == 2 * n and mi.num_patterns == 2
    tri = np.tril(np.ones((bk, bk), dtype=np.uint8))
    np.testing.assert_array_equal(mi.partial_mask_blocks[0], np.vstack([tri, np.ones((bk, bk), np.uint8)]))
    np.testing.assert_array_equal(mi.partial_mask_blocks[1], np.vstack([np.zeros((bk, bk), np.uint8), tri]))
    assert list(mi.mask_next[:2]) == [0, 1] and list(mi.mask_next[2:6]) == [-1, -1, 0, 1]


@pytest.mark.parametrize("L,b,w", [(4096, 128, 8), (8192, 128, 8), (2048, 64, 5), (65536, 1024, 4)])
def test_causal_window_closed_form(L, b, w):
    n, W = L // b, w * b
    mi = oracle.mask_info(MaskSpec(causal=True, window_left=W - 1, window_right=0), L, L, b, b)
    assert mi.num_active == w * (w + 1) // 2 + (n - w) * (w + 1)
    assert mi.num_partial == w + 2 * (n - w)
    assert mi.num_patterns == 2
    assert mi.allowed_pairs == W * (W + 1) // 2 + (L - W) * W


def test_local_window_causal_workload_counts():
    """The local-window workload (L = 65536, 128 x 128 blocks, 4096 keys):
    A = 32*33/2 + 480*33 = 16368 active blocks, 992 partial, 2 patterns."""
    w = workloads.workload(5)
    mi = oracle.mask_info(MaskSpec(causal=True, window_left=w.window_left, window_right=w.window_right),
                          w.L, w.L, w.bq, w.bk)
    assert (mi.num_active, mi.num_partial, mi.num_patterns) == (16368, 992, 2)


def test_document_causal_useful_pairs():
    lens = workloads.document_lengths(8192, 99, mean=700, lo=64, hi=3000)[0]
    seg = workloads.segment_ids_from_lengths([lens]).numpy()
    L = seg.shape[1]
    mi = oracle.mask_info(MaskSpec(causal=True, q_segment_ids=seg, kv_segment_ids=seg), L, L, 128, 128)
    assert mi.allowed_pairs == sum(n * (n + 1) // 2 for n in lens)


def test_window_wider_than_sequence_is_causal():
    L = 512
    a = oracle.mask_info(MaskSpec(causal=True), L, L, 64, 64)
    b = oracle.mask_info(MaskSpec(causal=True, window_left=10 * L, window_right=10 * L), L, L, 64, 64)
    for f in ("block_mask", "row_ptr", "active_cols", "mask_next", "partial_mask_blocks"):
        np.testing.assert_array_equal(getattr(a, f), getattr(b, f))


# ---------------------------------------------------------------------------
# Independent brute force on tiny sizes: a dense boolean mask built with numpy
# broadcasting, then every MaskInfo array derived from it directly.
# ---------------------------------------------------------------------------


def dense_mask(spec, Lq, Lk):
    i = np.arange(Lq)[:, None]
    j = np.arange(Lk)[None, :]
    m = np.ones((Lq, Lk), dtype=bool)
    if spec.causal:
        m &= j <= i
    if spec.window_left >= 0:
        m &= (i - j) <= spec.window_left
    if spec.window_right >= 0:
        m &= (j - i) <= spec.window_right
    if spec.q_segment_ids is None:
        return m[None]
    qs = np.atleast_2d(spec.q_segment_ids)
    ks = np.atleast_2d(spec.kv_segment_ids if spec.kv_segment_ids is not None else spec.q_segment_ids)
    return m[None] & (qs[:, :, None] == ks[:, None, :])


def brute_maskinfo(spec, Lq, Lk, bq, bk):
    dm = dense_mask(spec, Lq, Lk)
    nbm, nq, nk = dm.shape[0], -(-Lq // bq), -(-Lk // bk)
    # ragged lengths: pad the dense mask to whole blocks with masked entries
    dm = np.pad(dm, ((0, 0), (0, nq * bq - Lq), (0, nk * bk - Lk)))
    blocks = dm.reshape(nbm, nq, bq, nk, bk).transpose(0, 1, 3, 2, 4)
    cnt = blocks.sum(axis=(3, 4))
    cls = np.where(cnt == 0, 0, np.where(cnt == bq * bk, 2, 1)).astype(np.int8)
    rows, cols, nxt, bs, be, pats, ptr = [], [], [], [], [], [], [0]
    for bm in range(nbm):
        for r in range(nq):
            act = [c for c in range(nk) if cls[bm, r, c]]
            for t, c in enumerate(act):
                rows.append(r)
                cols.append(c)
                bs.append(int(t == 0))
                be.append(int(t == len(act) - 1))
                if cls[bm, r, c] == 1:
                    p = blocks[bm, r, c].astype(np.uint8)
                    idx = next((u for u, q in enumerate(pats) if np.array_equal(q, p)), None)
                    if idx is None:
                        pats.append(p)
                        idx = len(pats) - 1
                    nxt.append(idx)
                else:
                    nxt.append(-1)
            ptr.append(len(rows))
    return dict(block_mask=cls, row_ptr=ptr, active_rows=rows, active_cols=cols, mask_next=nxt,
                bounds_start=bs, bounds_end=be, patterns=pats, allowed=int(dm.sum()))


def tiny_specs():
    rng = np.random.default_rng(2024)
    specs = []
    for L in (16, 32, 48, 64):
        for causal in (False, True):
            for wl, wr in ((-1, -1), (0, 0), (3, -1), (-1, 5), (7, 2), (20, 20)):
                specs.append((L, MaskSpec(causal=causal, window_left=wl, window_right=wr)))
        for sorted_ids in (True, False):
            seg = workloads.random_segment_ids(2, L, int(rng.integers(1 << 30)), 4, sorted_ids).numpy()
            specs.append((L, MaskSpec(causal=True, q_segment_ids=seg, kv_segment_ids=seg)))
            specs.append((L, MaskSpec(causal=False, window_left=5, window_right=3, q_segment_ids=seg,
                                      kv_segment_ids=seg)))
            kv = workloads.random_segment_ids(2, L, int(rng.integers(1 << 30)), 4, sorted_ids).numpy()
            specs.append((L, MaskSpec(causal=False, q_segment_ids=seg, kv_segment_ids=kv)))
    return specs


@pytest.mark.parametrize("L,spec", tiny_specs())
@pytest.mark.parametrize("bq,bk", [(4, 4), (8, 8), (16, 16), (8, 16), (16, 4), (5, 7), (16, 12)])
def test_maskinfo_matches_dense_brute_force(L, spec, bq, bk):
    check_against_brute_force(spec, L, L, bq, bk)


def ragged_specs():
    rng = np.random.default_rng(77)
    out = []
    for Lq, Lk in ((30, 30), (37, 37), (45, 29), (21, 50)):
        for causal in (False, True):
            for wl, wr in ((-1, -1), (3, -1), (7, 2)):
                out.append((Lq, Lk, MaskSpec(causal=causal, window_left=wl, window_right=wr)))
        qs = workloads.random_segment_ids(2, Lq, int(rng.integers(1 << 30)), 3, True).numpy()
        ks = workloads.random_segment_ids(2, Lk, int(rng.integers(1 << 30)), 3, True).numpy()
        out.append((Lq, Lk, MaskSpec(causal=True, q_segment_ids=qs, kv_segment_ids=ks)))
    return out


@pytest.mark.parametrize("Lq,Lk,spec", ragged_specs())
@pytest.mark.parametrize("bq,bk", [(8, 8), (16, 16), (8, 16)])
def test_ragged_maskinfo_matches_dense_brute_force(Lq, Lk, spec, bq, bk):
    check_against_brute_force(spec, Lq, Lk, bq, bk)


def test_ragged_grid_worked_example():
    g = read_golden("ragged_1000_256.txt")
    L, b = int(g["L"]), int(g["block"])
    mi = oracle.mask_info(MaskSpec(), L, L, b, b)
    computed = mi.num_active * b * b
    assert computed == int(g["computed_elements"])
    assert mi.allowed_pairs == L * L
    assert round(100 * mi.allowed_pairs / computed, 1) == float(g["useful_percent"])
    # the 7 blocks on the ragged edge are partial (padding masked); the last
    # row's, the last column's and the corner's patterns are the three
    assert mi.num_partial == 7 and mi.num_patterns == 3
    assert int(np.count_nonzero(mi.block_mask == 2)) == 9


def check_against_brute_force(spec, Lq, Lk, bq, bk):
    mi = oracle.mask_info(spec, Lq, Lk, bq, bk)
    ref = brute_maskinfo(spec, Lq, Lk, bq, bk)
    np.testing.assert_array_equal(mi.block_mask, ref["block_mask"])
    assert mi.row_ptr.tolist() == ref["row_ptr"]
    assert mi.active_rows.tolist() == ref["active_rows"]
    assert mi.active_cols.tolist() == ref["active_cols"]
    assert mi.mask_next.tolist() == ref["mask_next"]
    assert mi.bounds_start.tolist() == ref["bounds_start"]
    assert mi.bounds_end.tolist() == ref["bounds_end"]
    assert mi.num_patterns == len(ref["patterns"])
    for u, p in enumerate(ref["patterns"]):
        np.testing.assert_array_equal(mi.partial_mask_blocks[u], p)
    assert mi.allowed_pairs == ref["allowed"]


# ---------------------------------------------------------------------------
# Attention: reductions to textbook routines and closed forms.
# ---------------------------------------------------------------------------


def bf16(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def as_f64(t):
    return t.to(torch.float64).numpy()


def rand_qkv(B, Hq, Hkv, L, dqk, dv, seed):
    return (workloads.normal_bf16((B, Hq, L, dqk), seed), workloads.normal_bf16((B, Hkv, L, dqk), seed + 1),
            workloads.normal_bf16((B, Hkv, L, dv), seed + 2))


def textbook_attention(q, k, v, allowed, scale, cap=0.0):
    """softmax(scale*QK^T (capped), masked) V with dense numpy matrix algebra."""
    s = scale * (q @ k.T)
    if cap > 0:
        s = cap * np.tanh(s / cap)
    s = np.where(allowed, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    return (e / l) @ v, (m + np.log(l))[:, 0]


@pytest.mark.parametrize("causal,cap", [(False, 0.0), (True, 0.0), (True, 5.0), (False, 2.0)])
def test_attention_matches_textbook_dense(causal, cap):
    B, Hq, Hkv, L, d, dv = 2, 4, 2, 96, 32, 24
    q, k, v = rand_qkv(B, Hq, Hkv, L, d, dv, 500)
    scale = 0.3
    spec = MaskSpec(causal=causal)
    O, lse = oracle.attention(q, k, v, spec, scale, cap)
    allowed = dense_mask(spec, L, L)[0]
    for b in range(B):
        for h in range(Hq):
            kvh = h // (Hq // Hkv)
            Oref, lref = textbook_attention(as_f64(q[b, h]), as_f64(k[b, kvh]), as_f64(v[b, kvh]),
                                            allowed, scale, cap)
            np.testing.assert_allclose(O[b, h], Oref, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(lse[b, h], lref, rtol=1e-12, atol=1e-12)


def test_single_allowed_key_gives_that_value():
    # causal: query 0 sees only key 0; window 0 both sides: every query sees only itself
    q, k, v = rand_qkv(1, 2, 2, 64, 16, 8, 900)
    scale = 0.25
    O, lse = oracle.attention(q, k, v, MaskSpec(causal=False, window_left=0, window_right=0), scale)
    qf, kf, vf = as_f64(q), as_f64(k), as_f64(v)
    np.testing.assert_allclose(O, vf, rtol=0, atol=0)
    np.testing.assert_allclose(lse, scale * np.einsum("bhld,bhld->bhl", qf, kf), rtol=1e-14)


def test_zero_query_gives_mean_of_allowed_values():
    B, H, L, d, dv = 1, 2, 80, 16, 8
    q = torch.zeros(B, H, L, d, dtype=torch.bfloat16)
    _, k, v = rand_qkv(B, H, H, L, d, dv, 77)
    wl = 9
    O, lse = oracle.attention(q, k, v, MaskSpec(causal=True, window_left=wl), 1.0)
    vf = as_f64(v)
    for i in range(L):
        lo = max(0, i - wl)
        np.testing.assert_allclose(O[0, :, i], vf[0, :, lo:i + 1].mean(axis=1), rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(lse[0, :, i], math.log(i + 1 - lo), rtol=1e-14)


def test_document_causal_equals_per_document_causal():
    L = 160
    lens = [37, 64, 59]
    seg = workloads.segment_ids_from_lengths([lens]).numpy()
    q, k, v = rand_qkv(1, 2, 1, L, 16, 16, 31)
    scale = 0.25
    O, lse = oracle.attention(q, k, v, MaskSpec(causal=True, q_segment_ids=seg, kv_segment_ids=seg), scale)
    s = 0
    for n in lens:
        Od, ld = oracle.attention(q[:, :, s:s + n], k[:, :, s:s + n], v[:, :, s:s + n],
                                  MaskSpec(causal=True), scale)
        np.testing.assert_allclose(O[:, :, s:s + n], Od, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(lse[:, :, s:s + n], ld, rtol=1e-13, atol=1e-14)
        s += n


def test_gqa_equals_mha_with_repeated_kv():
    B, Hq, Hkv, L, d, dv = 1, 6, 2, 48, 16, 8
    q, k, v = rand_qkv(B, Hq, Hkv, L, d, dv, 3)
    G = Hq // Hkv
    O1, l1 = oracle.attention(q, k, v, MaskSpec(causal=True), 0.5)
    O2, l2 = oracle.attention(q, k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1),
                              MaskSpec(causal=True), 0.5)
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(l1, l2)


def test_huge_cap_equals_no_cap_and_cap_bounds_scores():
    q, k, v = rand_qkv(1, 2, 2, 64, 32, 16, 12)
    O0, l0 = oracle.attention(q, k, v, MaskSpec(causal=True), 0.5)
    O1, l1 = oracle.attention(q, k, v, MaskSpec(causal=True), 0.5, softcap=1e9)
    np.testing.assert_allclose(O1, O0, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(l1, l0, rtol=1e-9, atol=1e-12)
    cap = 1.5
    _, l2 = oracle.attention(q * 8, k, v, MaskSpec(causal=True), 0.5, softcap=cap)
    n = np.arange(1, 65)
    assert np.all(l2[0] < cap + np.log(n)[None, :])
    assert np.all(l2[0] > -cap + np.log(n)[None, :])


def test_lse_normalises_the_weights_and_merges_across_key_splits():
    """exp(s - LSE) sums to one over a row, and splitting every row's keys in
    two (segment IDs select each half) then merging the halves with the
    pages' two-segment rule reproduces the full result."""
    L, d, dv = 128, 16, 8
    q, k, v = rand_qkv(1, 1, 1, L, d, dv, 41)
    scale = 0.4
    O, lse = oracle.attention(q, k, v, MaskSpec(causal=False), scale)
    qf, kf = as_f64(q)[0, 0], as_f64(k)[0, 0]
    s = scale * qf @ kf.T
    np.testing.assert_allclose(np.exp(s - lse[0, 0][:, None]).sum(axis=1), 1.0, rtol=1e-13)
    for cut in (1, 50, 127):
        kseg = (np.arange(L) >= cut).astype(np.int32)[None]
        halves = []
        for part in (0, 1):
            qseg = np.full((1, L), part, dtype=np.int32)
            halves.append(oracle.attention(q, k, v, MaskSpec(q_segment_ids=qseg, kv_segment_ids=kseg), scale))
        (O1, l1), (O2, l2) = halves
        # each half's state as (m, l, o) = (LSE, 1, O): exp(LSE) is its sum
        for i in range(L):
            m, lsum, o = oracle.merge(l1[0, 0, i], 1.0, O1[0, 0, i], l2[0, 0, i], 1.0, O2[0, 0, i])
            np.testing.assert_allclose(o, O[0, 0, i], rtol=1e-12, atol=1e-13)
            assert m + math.log(lsum) == pytest.approx(lse[0, 0, i], rel=1e-13)


def test_fully_masked_rows_give_zero_and_minus_infinity():
    L = 32
    qseg = np.zeros((1, L), dtype=np.int32)
    qseg[0, 10:20] = 5                      # queries 10..19 have no key of segment 5
    kseg = np.zeros((1, L), dtype=np.int32)
    q, k, v = rand_qkv(1, 1, 1, L, 8, 8, 5)
    O, lse = oracle.attention(q, k, v, MaskSpec(causal=True, q_segment_ids=qseg, kv_segment_ids=kseg), 1.0)
    assert np.all(O[0, 0, 10:20] == 0)
    assert np.all(np.isneginf(lse[0, 0, 10:20]))
    assert np.all(np.isfinite(lse[0, 0, :10]))


def test_sampled_rows_equal_full_computation():
    q, k, v = rand_qkv(2, 4, 2, 64, 16, 16, 8)
    spec = MaskSpec(causal=True, window_left=20)
    O, lse = oracle.attention(q, k, v, spec, 0.25)
    rows = np.array([0, 5, 63, 64 * 3 + 7, 64 * 7 + 63, 64 * 5])
    Os, ls = oracle.attention(q, k, v, spec, 0.25, rows=rows)
    np.testing.assert_array_equal(Os, O.reshape(-1, 16)[rows])
    np.testing.assert_array_equal(ls, lse.reshape(-1)[rows])
