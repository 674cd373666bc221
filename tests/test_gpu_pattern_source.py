"""Partial-block masks computed in the kernel from positions and segment IDs
("Pallas Kernels and Splash Attention" §6.6) against the stored patterns: the
two sources give the same element masks, so every output of the forward (one
pass, split-KV, Max Logit Estimate, host buffers) must be identical bit for
bit, and equal to the f64 oracle within tolerance."""
import math

import pytest
import torch

import oracle
import workloads
from tests.parity import compare_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bsf():
    from block_sparse_flash_gb300 import build as b
    b.build()
    import block_sparse_flash_gb300 as m
    return m


CASES = [
    # label, B, Hq, Hkv, Lq, Lk, d, blk, softcap, causal, wl, wr
    ("causal GQA", 2, 4, 2, 1024, 1024, 128, 128, 0.0, True, -1, -1),
    ("window 4096-style + causal + cap", 1, 4, 2, 2048, 2048, 128, 128, 30.0, True, 511, 0),
    ("two-sided window, blocks 64", 1, 2, 2, 1024, 1024, 64, 64, 0.0, False, 100, 37),
    ("ragged causal 1000", 1, 2, 1, 1000, 1000, 128, 128, 0.0, True, -1, -1),
    ("ragged no mask 777 x 1300", 1, 2, 2, 777, 1300, 128, 128, 20.0, False, -1, -1),
    ("d192/128 window", 1, 2, 2, 640, 640, 192, 128, 0.0, True, 130, 0),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_positions_equal_stored_patterns(bsf, case):
    label, B, Hq, Hkv, Lq, Lk, d, blk, cap, causal, wl, wr = case
    dv = 128 if d == 192 else d
    seed = 29 * CASES.index(case)
    q = workloads.normal_bf16((B, Hq, Lq, d), seed + 1).cuda()
    k = workloads.normal_bf16((B, Hkv, Lk, d), seed + 2).cuda()
    v = workloads.normal_bf16((B, Hkv, Lk, dv), seed + 3).cuda()
    mi = bsf.build_mask_info(bsf.MaskSpec(causal, wl, wr, None, None), Lq, Lk, blk, blk)
    scale = 1.0 / math.sqrt(d)
    runs = {}
    for source in ("stored", "positions"):
        mi.set_pattern_source(source)
        runs[source] = (bsf.attention_fwd(q, k, v, mi, scale, cap),
                        bsf.attention_fwd(q, k, v, mi, scale, cap, num_splits=3),
                        bsf.attention_fwd(q, k, v, mi, scale, cap, max_logit=cap if cap > 0 else 8.0))
    torch.cuda.synchronize()
    assert bsf.last_device_error() == 0, label
    for (a_out, a_lse), (b_out, b_lse) in zip(runs["stored"], runs["positions"]):
        assert torch.equal(a_out, b_out) and torch.equal(a_lse, b_lse), label
    O, L = oracle.attention(q.cpu(), k.cpu(), v.cpu(), oracle.MaskSpec(causal, wl, wr), scale, cap)
    out, lse = runs["positions"][0]
    compare_rows(out.float().cpu().numpy().reshape(-1, dv), lse.cpu().numpy().reshape(-1),
                 O.reshape(-1, dv), L.reshape(-1), label)
    mi.close()


SEG_CASES = [
    # label, B, Hq, Hkv, L, d, bq, bk, softcap, causal, wl, wr, max_id, sorted, B_mask
    ("documents + causal GQA", 2, 4, 2, 2048, 128, 128, 128, 0.0, True, -1, -1, 6, True, 2),
    ("documents, no band, blocks 64", 1, 2, 2, 1024, 64, 64, 64, 0.0, False, -1, -1, 9, True, 1),
    ("non-monotone IDs + causal + cap", 1, 4, 4, 1024, 128, 128, 128, 30.0, True, -1, -1, 3, False, 1),
    ("many short documents + window", 2, 2, 1, 1536, 128, 128, 128, 0.0, True, 200, 0, 40, True, 2),
    ("ragged 1000, documents + causal", 1, 2, 1, 1000, 128, 128, 128, 0.0, True, -1, -1, 5, True, 1),
    ("256-row q-blocks, documents + causal", 1, 2, 2, 1024, 128, 256, 128, 0.0, True, -1, -1, 4, True, 1),
    ("d192/128, documents", 1, 2, 2, 768, 192, 128, 128, 0.0, True, -1, -1, 5, True, 1),
]


@pytest.mark.parametrize("case", SEG_CASES, ids=[c[0] for c in SEG_CASES])
def test_positions_with_segment_ids_equal_stored_patterns(bsf, case):
    """Masks with segment IDs: the kernel forms partial blocks' masks from the
    positions and the segment arrays ("Pallas Kernels and Splash Attention"
    §6.4, §6.6); the outputs equal those from the stored patterns bit for bit
    (one pass, split-KV, Max Logit Estimate, host buffers), and the oracle
    within tolerance.  Non-monotone and short-document IDs put several
    segments in one warp's rows (the key-by-key path)."""
    label, B, Hq, Hkv, L, d, bq, bk, cap, causal, wl, wr, max_id, srt, bm = case
    dv = 128 if d == 192 else d
    seed = 31 * SEG_CASES.index(case) + 7
    q = workloads.normal_bf16((B, Hq, L, d), seed + 1).cuda()
    k = workloads.normal_bf16((B, Hkv, L, d), seed + 2).cuda()
    v = workloads.normal_bf16((B, Hkv, L, dv), seed + 3).cuda()
    seg = workloads.random_segment_ids(bm, L, seed, max_id, srt).cuda()
    mi = bsf.build_mask_info(bsf.MaskSpec(causal, wl, wr, seg, seg), L, L, bq, bk)
    assert mi.counts()["num_partial"] > 0, label
    scale = 1.0 / math.sqrt(d)
    runs = {}
    for source in ("stored", "positions"):
        mi.set_pattern_source(source)
        runs[source] = (bsf.attention_fwd(q, k, v, mi, scale, cap, seg, seg),
                        bsf.attention_fwd(q, k, v, mi, scale, cap, seg, None, num_splits=3),
                        bsf.attention_fwd(q, k, v, mi, scale, cap, seg, seg, max_logit=cap if cap > 0 else 8.0),
                        bsf.attention_fwd_host(q.cpu(), k.cpu(), v.cpu(), mi, scale, cap,
                                               q_segment_ids=seg, kv_segment_ids=seg))
    torch.cuda.synchronize()
    assert bsf.last_device_error() == 0, label
    for (a_out, a_lse), (b_out, b_lse) in zip(runs["stored"], runs["positions"]):
        assert torch.equal(a_out, b_out) and torch.equal(a_lse, b_lse), label
    seg_c = seg.cpu().numpy()  # one row serves every batch row (B_mask = 1), as in the library
    O, Lse = oracle.attention(q.cpu(), k.cpu(), v.cpu(), oracle.MaskSpec(causal, wl, wr, seg_c, seg_c), scale, cap)
    out, lse = runs["positions"][0]
    compare_rows(out.float().cpu().numpy().reshape(-1, dv), lse.cpu().numpy().reshape(-1),
                 O.reshape(-1, dv), Lse.reshape(-1), label)
    mi.close()


def test_positions_with_segment_ids_need_the_arrays(bsf):
    """A table with segment IDs whose pattern source is positions needs the
    segment arrays in the forward call: without them the call is refused
    before any launch."""
    seg = workloads.random_segment_ids(1, 512, 5, 3, True).cuda()
    mi = bsf.build_mask_info(bsf.MaskSpec(True, -1, -1, seg, seg), 512, 512, 128, 128)
    mi.set_pattern_source("positions")
    q = workloads.normal_bf16((1, 2, 512, 128), 1).cuda()
    k = workloads.normal_bf16((1, 2, 512, 128), 2).cuda()
    with pytest.raises(bsf.SplashError):
        bsf.attention_fwd(q, k, k, mi, 0.1, 0.0)
    mi.set_pattern_source("stored")
    bsf.attention_fwd(q, k, k, mi, 0.1, 0.0)
    torch.cuda.synchronize()
    assert bsf.last_device_error() == 0
    mi.close()


RECT_CASES = [
    # label, B_mask, Hq, Hkv, Lq, Lk, d, blk, causal, wl, wr
    ("700 x 1300, own q / kv IDs, no band", 1, 2, 1, 700, 1300, 128, 128, False, -1, -1),
    ("1300 x 700, own q / kv IDs, two-sided window, batch 2", 2, 2, 2, 1300, 700, 64, 64, False, 150, 90),
]


@pytest.mark.parametrize("case", RECT_CASES, ids=[c[0] for c in RECT_CASES])
def test_positions_with_different_q_and_kv_segment_ids(bsf, case):
    """Lq != Lk with query and key segment arrays of their own (the key IDs
    indexed by key position, the query IDs by query position): masks from
    positions and segment IDs equal the stored patterns bit for bit, and the
    oracle within tolerance."""
    label, bm, Hq, Hkv, Lq, Lk, d, blk, causal, wl, wr = case
    seed = 53 * RECT_CASES.index(case) + 11
    q = workloads.normal_bf16((bm, Hq, Lq, d), seed + 1).cuda()
    k = workloads.normal_bf16((bm, Hkv, Lk, d), seed + 2).cuda()
    v = workloads.normal_bf16((bm, Hkv, Lk, d), seed + 3).cuda()
    sq = workloads.random_segment_ids(bm, Lq, seed + 4, 4, True).cuda()
    skv = workloads.random_segment_ids(bm, Lk, seed + 5, 4, True).cuda()
    mi = bsf.build_mask_info(bsf.MaskSpec(causal, wl, wr, sq, skv), Lq, Lk, blk, blk)
    scale = 1.0 / math.sqrt(d)
    runs = {}
    for source in ("stored", "positions"):
        mi.set_pattern_source(source)
        runs[source] = bsf.attention_fwd(q, k, v, mi, scale, 0.0, sq, skv)
    torch.cuda.synchronize()
    assert bsf.last_device_error() == 0, label
    assert torch.equal(runs["stored"][0], runs["positions"][0]), label
    assert torch.equal(runs["stored"][1], runs["positions"][1]), label
    O, Lse = oracle.attention(q.cpu(), k.cpu(), v.cpu(),
                              oracle.MaskSpec(causal, wl, wr, sq.cpu().numpy(), skv.cpu().numpy()), scale, 0.0)
    out, lse = runs["positions"]
    compare_rows(out.float().cpu().numpy().reshape(-1, d), lse.cpu().numpy().reshape(-1),
                 O.reshape(-1, d), Lse.reshape(-1), label)
    mi.close()
