"""A MaskInfo rebuild and the forward captured into a CUDA graph.

The build queues its kernels without a host wait whenever the pattern buffer
can be sized from a bound (every shape here), so after a first build has
allocated the table, rebuild + attention can be captured and replayed: the
replay must give the eager results bit for bit.  Covers the three build
paths: the single-CTA band build, the one-launch build for a larger band
table, and the one-launch build with segment IDs (cooperative launch)."""
import math

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bsf():
    from block_sparse_flash_gb300 import build as b
    b.build()
    import block_sparse_flash_gb300 as m
    return m


CASES = [
    # label, B, Hq, Hkv, L, blk, causal, wl, docs
    ("small band table (single-CTA build)", 1, 4, 2, 2048, 128, True, -1, False),
    ("larger band table (one-launch build)", 1, 2, 1, 65536, 128, True, 4095, False),
    ("documents (one-launch build, segment IDs)", 1, 4, 2, 8192, 128, True, -1, True),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_rebuild_and_forward_replay_equal_eager(bsf, case):
    label, B, Hq, Hkv, L, blk, causal, wl, docs = case
    d = 128
    seed = 41 * CASES.index(case)
    q = workloads.normal_bf16((B, Hq, L, d), seed + 1).cuda()
    k = workloads.normal_bf16((B, Hkv, L, d), seed + 2).cuda()
    v = workloads.normal_bf16((B, Hkv, L, d), seed + 3).cuda()
    seg = None
    if docs:
        lens = workloads.document_lengths(L, seed + 4, mean=700, lo=64, hi=3000, batch_rows=B)
        seg = workloads.segment_ids_from_lengths(lens).cuda()
    spec = bsf.MaskSpec(causal, wl, 0 if wl >= 0 else -1, seg, seg)
    scale = 1.0 / math.sqrt(d)
    mi = bsf.build_mask_info(spec, L, L, blk, blk)  # allocates the table
    out_e, lse_e = bsf.attention_fwd(q, k, v, mi, scale)
    torch.cuda.synchronize()
    out = torch.empty_like(out_e)
    lse = torch.empty_like(lse_e)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm the rebuild on the capture stream
        mi.rebuild(spec, L, L, blk, blk)
        bsf.attention_fwd(q, k, v, mi, scale, out=out, lse=lse)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        mi.rebuild(spec, L, L, blk, blk)
        bsf.attention_fwd(q, k, v, mi, scale, out=out, lse=lse)
    out.zero_()
    lse.zero_()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert bsf.last_device_error() == 0, label
    assert torch.equal(out, out_e) and torch.equal(lse, lse_e), label
    eager_counts = mi.counts()
    assert eager_counts["num_active"] > 0
    del g
    mi.close()
