"""Partial-block masks computed from positions in the kernel ("Pallas Kernels
and Splash Attention" §6.6) against the stored patterns: for masks without
segment IDs the two sources give the same element masks, so every output of
the forward (one pass, split-KV, Max Logit Estimate) must be identical bit
for bit, and equal to the f64 oracle within tolerance."""
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


def test_positions_need_a_mask_without_segment_ids(bsf):
    seg = workloads.random_segment_ids(1, 512, 5, 3, True).cuda()
    mi = bsf.build_mask_info(bsf.MaskSpec(True, -1, -1, seg, seg), 512, 512, 128, 128)
    with pytest.raises(bsf.SplashError):
        mi.set_pattern_source("positions")
    mi.set_pattern_source("stored")
    mi.close()
