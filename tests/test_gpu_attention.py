"""Attention forward on the GPU vs the f64 oracle: every row on small shapes
(several tiles, all kernel variants, edge cases), sampled rows on the five
workloads at full size."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import MARGINS, compare_rows, gather_rows, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bsf():
    from block_sparse_flash_gb300 import build as b
    b.build()
    import block_sparse_flash_gb300 as m
    return m


def run_case(bsf, B, Hq, Hkv, Lq, Lk, dqk, dv, blk, causal=True, wl=-1, wr=-1, seg_q=None, seg_kv=None,
             softcap=0.0, q_gain=1.0, seed=0, rows=None, label=""):
    q = workloads.normal_bf16((B, Hq, Lq, dqk), seed + 1)
    if q_gain != 1.0:
        q = (q.float() * q_gain).to(torch.bfloat16)
    k = workloads.normal_bf16((B, Hkv, Lk, dqk), seed + 2)
    v = workloads.normal_bf16((B, Hkv, Lk, dv), seed + 3)
    scale = 1.0 / math.sqrt(dqk)
    sq = seg_q.cuda() if seg_q is not None else None
    skv = seg_kv.cuda() if seg_kv is not None else None
    mi = bsf.build_mask_info(bsf.MaskSpec(causal, wl, wr, sq, skv), Lq, Lk, blk, blk)
    out, lse = bsf.attention_fwd(q.cuda(), k.cuda(), v.cuda(), mi, scale, softcap)
    torch.cuda.synchronize()
    assert bsf.last_device_error() == 0, f"{label}: device error"
    ospec = oracle.MaskSpec(causal, wl, wr, seg_q.numpy() if seg_q is not None else None,
                            (seg_kv if seg_kv is not None else seg_q).numpy() if seg_q is not None else None)
    if rows is None:
        O, L = oracle.attention(q, k, v, ospec, scale, softcap)
        got = compare_rows(out.float().cpu().numpy().reshape(-1, dv), lse.cpu().numpy().reshape(-1),
                           O.reshape(-1, dv), L.reshape(-1), label)
    else:
        O, L = oracle.attention(q, k, v, ospec, scale, softcap, rows=rows)
        o, l = gather_rows(out, lse, rows)
        got = compare_rows(o, l, O, L, label)
    mi.close()
    return got


SMALL = [
    # label, B, Hq, Hkv, Lq, Lk, dqk, dv, blk, kwargs
    ("tiny causal MHA d64 b64", 1, 2, 2, 256, 256, 64, 64, 64, {}),
    ("causal GQA d128", 2, 4, 2, 512, 512, 128, 128, 128, {}),
    ("odd heads G=3 causal window", 1, 3, 1, 512, 512, 128, 128, 128, dict(wl=100)),
    ("MHA pairs d192/128", 2, 2, 2, 384, 384, 192, 128, 128, {}),
    ("MHA pairs d128, odd heads", 1, 3, 3, 512, 512, 128, 128, 128, dict(wl=200)),
    ("GQA G=3 pairs straddle groups", 1, 6, 2, 512, 512, 128, 128, 128, {}),
    ("d64 blocks 128", 1, 4, 4, 512, 512, 64, 64, 128, {}),
    ("d128 blocks 64", 1, 4, 2, 512, 512, 128, 128, 64, {}),
    ("no mask", 1, 2, 1, 256, 256, 128, 128, 128, dict(causal=False)),
    ("bidirectional window", 1, 2, 2, 640, 640, 128, 128, 128, dict(causal=False, wl=70, wr=130)),
    ("softcap 30 large logits", 1, 4, 2, 512, 512, 128, 128, 128, dict(softcap=30.0, q_gain=6.0)),
    ("softcap + window", 1, 2, 1, 768, 768, 128, 128, 128, dict(softcap=20.0, wl=255, q_gain=3.0)),
    ("softcap small logits (series path)", 2, 4, 2, 512, 512, 128, 128, 128, dict(softcap=50.0)),
    ("softcap mixed rows", 1, 2, 2, 512, 512, 64, 64, 64, dict(softcap=8.0, q_gain=1.5)),
    ("Lq < Lk causal", 1, 2, 2, 256, 512, 128, 128, 128, {}),
    ("huge logits (reference jumps)", 1, 4, 2, 1024, 1024, 128, 128, 128, dict(q_gain=40.0)),
    ("huge logits soft-capped", 1, 2, 2, 512, 512, 64, 64, 64, dict(q_gain=40.0, softcap=100.0)),
    ("long row many blocks", 1, 2, 2, 2048, 2048, 128, 128, 128, dict(q_gain=2.0)),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_shapes_every_row(bsf, case):
    label, B, Hq, Hkv, Lq, Lk, dqk, dv, blk, kw = case
    run_case(bsf, B, Hq, Hkv, Lq, Lk, dqk, dv, blk, label=label, seed=10 * SMALL.index(case), **kw)


def test_segments_per_batch_with_fully_masked_rows(bsf):
    # non-monotone ids + causal: some queries find no key of their segment
    seg = workloads.random_segment_ids(2, 512, 77, 5, False)
    run_case(bsf, 2, 4, 2, 512, 512, 128, 128, 128, seg_q=seg, seg_kv=seg, label="segments B=2")


def test_documents_causal_gqa(bsf):
    lens = workloads.document_lengths(2048, 9, mean=300, lo=64, hi=1000)
    seg = workloads.segment_ids_from_lengths(lens)
    run_case(bsf, 1, 4, 2, 2048, 2048, 128, 128, 128, seg_q=seg, seg_kv=seg, label="documents")


def test_everything_masked(bsf):
    q = torch.zeros(1, 256, dtype=torch.int32)
    kv = torch.ones(1, 256, dtype=torch.int32)
    run_case(bsf, 1, 2, 2, 256, 256, 64, 64, 64, seg_q=q, seg_kv=kv, label="all masked")


def test_outputs_are_written_in_place(bsf):
    q = workloads.normal_bf16((1, 2, 256, 64), 1).cuda()
    k = workloads.normal_bf16((1, 2, 256, 64), 2).cuda()
    v = workloads.normal_bf16((1, 2, 256, 64), 3).cuda()
    mi = bsf.build_mask_info(bsf.MaskSpec(True), 256, 256, 64, 64)
    out = torch.full((1, 2, 256, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((1, 2, 256), 7.0, dtype=torch.float32, device="cuda")
    o2, l2 = bsf.attention_fwd(q, k, v, mi, 0.125, out=out, lse=lse)
    assert o2.data_ptr() == out.data_ptr() and l2.data_ptr() == lse.data_ptr()
    assert not torch.any(out == 7.0) and not torch.any(lse == 7.0)
    mi.close()


def test_device_wait_timeout_is_reported(bsf):
    # a wait on an mbarrier that nothing arrives on gives up after ~5 ms
    assert bsf.debug_wait_selftest(5_000_000) == 5
    assert bsf.last_device_error() == 0  # the word was cleared


def full_size_rows(w, seed):
    """Rows compared at full size: every row of the first and the last query
    head in every batch row (on the document workload also of the middle
    head, so that every q-block row's document-edge partial blocks are seen
    for three heads), three whole q-blocks, and 256 seeded random rows.  The
    tiny workload is compared on every row."""
    if w.index == 1:
        return np.arange(w.B * w.Hq * w.q_len, dtype=np.int64)
    nq = w.q_len // w.bq  # whole blocks in all five workloads
    heads = (0, w.Hq // 2, w.Hq - 1) if w.documents else (0, w.Hq - 1)
    extra = [(0, 0, 0), (w.B - 1, w.Hq - 1, nq - 1), (0, w.Hq // 2, nq // 2)]
    extra += [(b, h, r) for b in range(w.B) for h in heads for r in range(nq)]
    return sample_rows(w.B, w.Hq, w.q_len, w.bq, 256, seed, extra)


@pytest.mark.parametrize("index", [1, 2, 3, 4, 5])
def test_workloads_sampled_rows(bsf, index):
    w = workloads.workload(index)
    inp = workloads.make_inputs(w)
    seg = inp.segment_ids
    mi = bsf.build_mask_info(bsf.MaskSpec(w.causal, w.window_left, w.window_right,
                                          seg.cuda() if seg is not None else None,
                                          seg.cuda() if seg is not None else None), w.L, w.L, w.bq, w.bk)
    out, lse = bsf.attention_fwd(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), mi, w.scale, w.softcap)
    torch.cuda.synchronize()
    assert bsf.last_device_error() == 0
    rows = full_size_rows(w, 1000 + index)
    ospec = oracle.MaskSpec(w.causal, w.window_left, w.window_right,
                            seg.numpy() if seg is not None else None, seg.numpy() if seg is not None else None)
    O, L = oracle.attention(inp.q, inp.k, inp.v, ospec, w.scale, w.softcap, rows=rows)
    o, l = gather_rows(out, lse, rows)
    got = compare_rows(o, l, O, L, w.name)
    MARGINS[f"workload {index} ({w.name})"] = dict(got, rows=len(rows))
    # properties at every row: finite (self is always allowed in these masks)
    assert torch.isfinite(lse).all()
    assert torch.isfinite(out.float()).all()
    mi.close()
