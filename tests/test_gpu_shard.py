"""The (batch, KV head) split of one workload across ranks, emulated on one
GPU: the ranks' shares run one after the other (no rank waits on another),
each writing its slice of the caller's out / lse through the views that
shard_views gives.  Every (batch, head, q-block) item is computed the same
way whichever launch takes it, so the assembled output equals the unsplit
forward bit for bit."""
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
    # label, B, Hq, Hkv, L, dqk, dv, bq, bk, mask kwargs, documents
    ("causal GQA", 2, 8, 2, 1024, 128, 128, 128, 128, dict(causal=True), False),
    ("documents + causal, batch 2", 2, 6, 3, 1536, 128, 128, 128, 128, dict(causal=True), True),
    ("window + soft cap, MHA odd heads", 1, 5, 5, 1024, 64, 64, 64, 64,
     dict(causal=True, window_left=300), False),
    ("wide-head MHA, 256-row q-blocks", 1, 4, 4, 1024, 192, 128, 256, 128, dict(causal=True), False),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_head_shards_equal_the_whole_forward(bsf, case):
    label, B, Hq, Hkv, L, dqk, dv, bq, bk, mk, docs = case
    q = workloads.normal_bf16((B, Hq, L, dqk), 71).cuda()
    k = workloads.normal_bf16((B, Hkv, L, dqk), 72).cuda()
    v = workloads.normal_bf16((B, Hkv, L, dv), 73).cuda()
    seg = None
    if docs:
        seg = workloads.segment_ids_from_lengths(
            workloads.document_lengths(L, 74, mean=300, lo=64, hi=800, batch_rows=B)).cuda()
    softcap = 20.0 if "cap" in label else 0.0
    scale = 1.0 / math.sqrt(dqk)
    mi = bsf.build_mask_info(bsf.MaskSpec(q_segment_ids=seg, kv_segment_ids=seg, **mk), L, L, bq, bk)
    out, lse = bsf.attention_fwd(q, k, v, mi, scale, softcap)
    mi.close()
    for world in (2, 3):
        out2 = torch.full_like(out, float("nan"))
        lse2 = torch.full_like(lse, float("nan"))
        for rank in range(world):
            b0, b1 = bsf.shard_items(B, Hkv, world, rank)
            if b1 == b0:
                continue
            sv = bsf.shard_views(q, k, v, b0, b1, out=out2, lse=lse2, segment_ids=seg)
            s = sv.get("segment_ids")
            mr = bsf.build_mask_info(bsf.MaskSpec(q_segment_ids=s, kv_segment_ids=s, **mk), L, L, bq, bk)
            bsf.attention_fwd(sv["q"], sv["k"], sv["v"], mr, scale, softcap, out=sv["out"], lse=sv["lse"])
            mr.close()
        torch.cuda.synchronize()
        assert bsf.last_device_error() == 0
        assert torch.equal(out2, out), f"{label}: world {world} out differs"
        assert torch.equal(lse2, lse), f"{label}: world {world} lse differs"
