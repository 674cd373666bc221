"""The forward for host tensors (copies in, attention, copies out, pipelined
in chunks on library streams) must give exactly the device forward's output:
every (batch, head, q-block) item is computed independently, so chunking the
heads changes nothing."""
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
    # label, B, Hq, Hkv, Lq, Lk, dqk, dv, blk, softcap, causal, wl, docs, pinned
    ("GQA causal, batch 2, pinned", 2, 16, 4, 1024, 1024, 128, 128, 128, 0.0, True, -1, False, True),
    ("MHA window + cap, pageable", 1, 6, 6, 768, 768, 64, 64, 64, 30.0, True, 200, False, False),
    ("documents, batch 2 (one chunk)", 2, 4, 2, 640, 640, 128, 128, 128, 0.0, True, -1, True, True),
    ("ragged 1000 x 1300, d192", 1, 4, 2, 1000, 1300, 192, 128, 128, 0.0, False, -1, False, True),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_host_pipeline_equals_device_forward(bsf, case):
    label, B, Hq, Hkv, Lq, Lk, dqk, dv, blk, cap, causal, wl, docs, pinned = case
    seed = 37 * CASES.index(case)
    q = workloads.normal_bf16((B, Hq, Lq, dqk), seed + 1)
    k = workloads.normal_bf16((B, Hkv, Lk, dqk), seed + 2)
    v = workloads.normal_bf16((B, Hkv, Lk, dv), seed + 3)
    seg = workloads.random_segment_ids(B, Lq, seed + 4, 4, True).cuda() if docs else None
    mi = bsf.build_mask_info(bsf.MaskSpec(causal, wl, -1, seg, seg), Lq, Lk, blk, blk)
    scale = 1.0 / math.sqrt(dqk)
    out_d, lse_d = bsf.attention_fwd(q.cuda(), k.cuda(), v.cuda(), mi, scale, cap)
    qh, kh, vh = (t.pin_memory() for t in (q, k, v)) if pinned else (q, k, v)
    out_h, lse_h = bsf.attention_fwd_host(qh, kh, vh, mi, scale, cap)
    torch.cuda.synchronize()
    assert bsf.last_device_error() == 0, label
    assert torch.equal(out_h, out_d.cpu()) and torch.equal(lse_h, lse_d.cpu()), label
    # twice in a row on the same stream (the library's events are reused)
    out_h2, lse_h2 = bsf.attention_fwd_host(qh, kh, vh, mi, scale, cap)
    torch.cuda.synchronize()
    assert torch.equal(out_h2, out_h) and torch.equal(lse_h2, lse_h), label
    mi.close()


def test_host_pipeline_rejects_device_tensors(bsf):
    q = workloads.normal_bf16((1, 2, 256, 64), 1).cuda()
    mi = bsf.build_mask_info(bsf.MaskSpec(True, -1, -1, None, None), 256, 256, 64, 64)
    with pytest.raises(ValueError):
        bsf.attention_fwd_host(q, q, q, mi, 0.125)
    mi.close()
