"""256-row query blocks (bq = 256, bk = 128) on the GPU.

The MaskInfo of a 256 x 128 grid must equal the oracle's bit for bit (the
pages' own worked example, "Pallas Kernels and Splash Attention" §6.2,
already has bq != bk).  The forward then computes each q-block as two
128-row tiles of one head that share every K / V tile; blocks of the row's
active list that are masked for one half are computed for it and contribute
nothing.  Every row must match the f64 oracle, for stored patterns and masks
from positions, one-pass / split-KV / Max Logit Estimate, ragged lengths
(including a last block whose lower half is all padding), and nothing may be
written past the output tensors."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import compare_rows
from tests.test_gpu_mask_info import assert_same, gpu_and_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bsf():
    from block_sparse_flash_gb300 import build as b
    b.build()
    import block_sparse_flash_gb300 as m
    return m


MASKS = [
    # label, Lq, Lk, causal, wl, wr, segments (0 none, 1 shared documents, 2 per-batch different)
    ("causal 4096", 4096, 4096, True, -1, -1, 0),
    ("causal 1000 (ragged)", 1000, 1000, True, -1, -1, 0),
    ("window 300 + causal 1500", 1500, 1500, True, 299, 0, 0),
    ("two-sided window 700 x 900", 700, 900, False, 100, 250, 0),
    ("documents + causal 2048", 2048, 2048, True, -1, -1, 1),
    ("different q / kv segments 1100 x 1300", 1100, 1300, False, -1, -1, 2),
    ("one short row, 100", 100, 100, True, -1, -1, 0),
]


@pytest.mark.parametrize("case", MASKS, ids=[c[0] for c in MASKS])
def test_tall_mask_info_bit_exact(bsf, case):
    label, Lq, Lk, causal, wl, wr, segs = case
    seg_q = seg_kv = None
    if segs == 1:
        seg_q = seg_kv = workloads.random_segment_ids(2, Lq, 5, 6, True)
    elif segs == 2:
        seg_q = workloads.random_segment_ids(2, Lq, 6, 3, True)
        seg_kv = workloads.random_segment_ids(2, Lk, 7, 3, True)
    got, ref = gpu_and_oracle(bsf, causal, wl, wr, seg_q, seg_kv, Lq, Lk, 256, 128)
    assert_same(got, ref, label)


FWD = [
    # label, B, Hq, Hkv, Lq, Lk, dqk, dv, softcap, q_gain, mask kwargs
    ("causal MHA d192/128", 1, 4, 4, 1024, 1024, 192, 128, 0.0, 1.0, dict(causal=True)),
    ("causal GQA d128, batch 2", 2, 4, 2, 768, 768, 128, 128, 0.0, 1.0, dict(causal=True)),
    ("no mask d64, 640 x 1000", 1, 2, 1, 640, 1000, 64, 64, 0.0, 1.0, dict(causal=False)),
    ("window 300 + causal + cap 20", 1, 2, 2, 1280, 1280, 128, 128, 20.0, 3.0, dict(causal=True, wl=299)),
    ("documents + causal, batch 2", 2, 2, 2, 1024, 1024, 128, 128, 0.0, 1.0, dict(causal=True, docs=True)),
    ("ragged 1000, lower half partly padding", 1, 2, 2, 1000, 1000, 192, 128, 0.0, 1.0, dict(causal=True)),
    ("ragged 300, lower half all padding", 1, 3, 3, 300, 300, 128, 128, 0.0, 1.0, dict(causal=True)),
    ("a single short block, 100", 1, 2, 2, 100, 100, 64, 64, 0.0, 1.0, dict(causal=True)),
    ("huge logits (reference jumps)", 1, 2, 2, 768, 768, 128, 128, 0.0, 40.0, dict(causal=True)),
    ("window 500 + causal + cap 30, d192 GQA", 1, 4, 2, 1536, 1536, 192, 128, 30.0, 2.0, dict(causal=True, wl=499)),
    ("documents, d192/128 MHA", 1, 3, 3, 1280, 1280, 192, 128, 0.0, 1.0, dict(causal=True, docs=True)),
    ("no mask d192, 384 x 2000 (many blocks per row)", 1, 2, 2, 384, 2000, 192, 128, 0.0, 1.0, dict(causal=False)),
]


def make(bsf, B, Hq, Hkv, Lq, Lk, dqk, dv, q_gain, causal=True, wl=-1, wr=-1, docs=False, seed=0):
    q = workloads.normal_bf16((B, Hq, Lq, dqk), seed + 1)
    if q_gain != 1.0:
        q = (q.float() * q_gain).to(torch.bfloat16)
    k = workloads.normal_bf16((B, Hkv, Lk, dqk), seed + 2)
    v = workloads.normal_bf16((B, Hkv, Lk, dv), seed + 3)
    seg = workloads.random_segment_ids(B, Lq, seed + 4, 4, True) if docs else None
    segd = seg.cuda() if seg is not None else None
    mi = bsf.build_mask_info(bsf.MaskSpec(causal, wl, wr, segd, segd), Lq, Lk, 256, 128)
    assert mi.shape()["bq"] == 256
    ospec = oracle.MaskSpec(causal, wl, wr, seg.numpy() if seg is not None else None,
                            seg.numpy() if seg is not None else None)
    return q, k, v, mi, ospec


def guarded(shape, dtype, fill):
    n = int(np.prod(shape))
    buf = torch.full((n + 4096,), fill, dtype=dtype, device="cuda")
    return buf, buf[:n].view(shape)


@pytest.mark.parametrize("case", FWD, ids=[c[0] for c in FWD])
def test_tall_forward_matches_the_oracle(bsf, case):
    label, B, Hq, Hkv, Lq, Lk, dqk, dv, cap, gain, kw = case
    q, k, v, mi, ospec = make(bsf, B, Hq, Hkv, Lq, Lk, dqk, dv, gain, seed=31 * FWD.index(case), **kw)
    scale = 1.0 / math.sqrt(dqk)
    O, L = oracle.attention(q, k, v, ospec, scale, cap)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    obuf, out = guarded((B, Hq, Lq, dv), torch.bfloat16, 7.0)
    lbuf, lse = guarded((B, Hq, Lq), torch.float32, 7.0)
    bsf.attention_fwd(qd, kd, vd, mi, scale, cap, out=out, lse=lse)
    torch.cuda.synchronize()
    assert bsf.last_device_error() == 0, f"{label}: device error"
    assert torch.all(obuf[out.numel():] == 7.0) and torch.all(lbuf[lse.numel():] == 7.0), f"{label}: wrote past"
    compare_rows(out.float().cpu().numpy().reshape(-1, dv), lse.cpu().numpy().reshape(-1),
                 O.reshape(-1, dv), L.reshape(-1), label)
    # the same table, split-KV and the Max Logit Estimate
    out2, lse2 = bsf.attention_fwd(qd, kd, vd, mi, scale, cap, num_splits=3)
    results = [(out2, lse2, "split-KV")]
    if gain == 1.0:
        out3, lse3 = bsf.attention_fwd(qd, kd, vd, mi, scale, cap, max_logit=cap if cap > 0 else 8.0)
        results.append((out3, lse3, "MLE"))
    torch.cuda.synchronize()
    assert bsf.last_device_error() == 0, f"{label}: device error"
    for o_, l_, what in results:
        compare_rows(o_.float().cpu().numpy().reshape(-1, dv), l_.cpu().numpy().reshape(-1),
                     O.reshape(-1, dv), L.reshape(-1), f"{label}, {what}")
    mi.close()


@pytest.mark.parametrize("case", [c for c in FWD if not c[10].get("docs")][:6],
                         ids=[c[0] for c in FWD if not c[10].get("docs")][:6])
def test_tall_masks_from_positions_equal_stored(bsf, case):
    # the band part of the mask computed in the kernel from positions gives
    # the same bits as the stored patterns ("Pallas Kernels and Splash
    # Attention" §6.6): identical outputs, bit for bit
    label, B, Hq, Hkv, Lq, Lk, dqk, dv, cap, gain, kw = case
    q, k, v, mi, _ = make(bsf, B, Hq, Hkv, Lq, Lk, dqk, dv, gain, seed=77, **kw)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    scale = 1.0 / math.sqrt(dqk)
    a = bsf.attention_fwd(qd, kd, vd, mi, scale, cap)
    mi.set_pattern_source("positions")
    b = bsf.attention_fwd(qd, kd, vd, mi, scale, cap)
    torch.cuda.synchronize()
    assert bsf.last_device_error() == 0, label
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]), label
    mi.close()


def test_tall_equals_square_blocks(bsf):
    # the table's block shape changes the work split, not the result: the
    # 256-row and the 128-row tables give the same rows up to the fp32
    # summation order (both within the oracle tolerance; here compared to
    # each other at the bf16 output's resolution)
    B, Hq, Hkv, L, d = 1, 4, 4, 1024, 128
    q = workloads.normal_bf16((B, Hq, L, d), 1).cuda()
    k = workloads.normal_bf16((B, Hkv, L, d), 2).cuda()
    v = workloads.normal_bf16((B, Hkv, L, d), 3).cuda()
    outs = []
    for bq in (128, 256):
        mi = bsf.build_mask_info(bsf.MaskSpec(True), L, L, bq, 128)
        outs.append(bsf.attention_fwd(q, k, v, mi, d ** -0.5))
        mi.close()
    torch.cuda.synchronize()
    assert (outs[0][0].float() - outs[1][0].float()).abs().max().item() <= 1.6e-2
    assert (outs[0][1] - outs[1][1]).abs().max().item() <= 1e-4


def test_tall_rejected_with_64_key_blocks(bsf):
    q = workloads.normal_bf16((1, 2, 512, 64), 1).cuda()
    mi = bsf.build_mask_info(bsf.MaskSpec(True), 512, 512, 256, 64)
    with pytest.raises(bsf.SplashError):
        bsf.attention_fwd(q, q, q, mi, 0.125)
    mi.close()


GROUPED = [
    # label, B, Hq, Hkv, L, dqk, dv, bq: all heads' K / V exceeds 64 MB and the
    # rows span the keys, so the items are ordered by head groups, the last
    # group smaller than the others
    ("40 heads MHA d192, 256-row blocks", 1, 40, 40, 4096, 192, 128, 256),
    ("68 heads GQA (G=2) d128, head pairs", 1, 68, 34, 4096, 128, 128, 128),
]


@pytest.mark.parametrize("case", GROUPED, ids=[c[0] for c in GROUPED])
def test_head_grouped_order_sampled_rows(bsf, case):
    from tests.parity import gather_rows, sample_rows
    label, B, Hq, Hkv, L, dqk, dv, bq = case
    q = workloads.normal_bf16((B, Hq, L, dqk), 71)
    k = workloads.normal_bf16((B, Hkv, L, dqk), 72)
    v = workloads.normal_bf16((B, Hkv, L, dv), 73)
    assert B * Hkv * L * (dqk + dv) * 2 > 64 << 20
    mi = bsf.build_mask_info(bsf.MaskSpec(True), L, L, bq, 128)
    scale = 1.0 / math.sqrt(dqk)
    out, lse = bsf.attention_fwd(q.cuda(), k.cuda(), v.cuda(), mi, scale)
    torch.cuda.synchronize()
    assert bsf.last_device_error() == 0, label
    nq = L // bq
    # whole blocks of the first head, the last head (last, smaller group) and
    # a head in between, plus random rows
    extra = [(0, 0, nq - 1), (0, Hq - 1, 0), (0, Hq - 1, nq - 1), (0, Hq // 2, nq // 2)]
    rows = sample_rows(B, Hq, L, bq, 256, 4242, extra)
    O, Lref = oracle.attention(q, k, v, oracle.MaskSpec(True), scale, 0.0, rows=rows)
    o, l = gather_rows(out, lse, rows)
    compare_rows(o, l, O, Lref, label)
    assert torch.isfinite(lse).all() and torch.isfinite(out.float()).all()
    mi.close()
