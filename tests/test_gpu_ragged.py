"""Ragged lengths on the GPU: Lq / Lk not multiples of the block.

The grid is padded to whole blocks and the padding is masked ("Pallas
Kernels and Splash Attention" §2.3).  The GPU MaskInfo must equal the
oracle's padded-grid table bit for bit; the forward (one pass, split-KV and
the Max Logit Estimate) and the backward must match the f64 oracle on every
real row and must not write past their output tensors."""
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


def mask_cases():
    rng = np.random.default_rng(4321)
    cases = []
    for n in range(24):
        Lq = int(rng.integers(65, 1500))
        Lk = Lq if rng.integers(2) else int(rng.integers(65, 1500))
        bq = int(rng.choice([64, 128]))
        bk = int(rng.choice([64, 128]))
        causal = bool(rng.integers(2))
        wl = int(rng.choice([-1, 0, 63, 100, 300]))
        wr = int(rng.choice([-1, 0, 64, 200]))
        kind = int(rng.integers(3)) if Lq == Lk else int(rng.integers(2)) * 2  # 1 needs Lq == Lk
        cases.append((n, Lq, Lk, bq, bk, causal, wl, wr, kind, int(rng.integers(1 << 30))))
    # the worked example's grid, and lengths one short of / one past a block
    cases += [(100, 1000, 1000, 128, 128, False, -1, -1, 0, 1), (101, 1023, 1023, 128, 128, True, -1, -1, 0, 2),
              (102, 1025, 1025, 64, 64, True, 200, 0, 0, 3), (103, 1025, 4097, 128, 128, False, -1, -1, 2, 4)]
    return cases


@pytest.mark.parametrize("n,Lq,Lk,bq,bk,causal,wl,wr,kind,seed", mask_cases())
def test_ragged_mask_info_bit_exact(bsf, n, Lq, Lk, bq, bk, causal, wl, wr, kind, seed):
    seg_q = seg_kv = None
    if kind == 1:
        seg_q = seg_kv = workloads.random_segment_ids(1, Lq, seed, 5, True)
    elif kind == 2:
        seg_q = workloads.random_segment_ids(2, Lq, seed, 3, True)
        seg_kv = workloads.random_segment_ids(2, Lk, seed + 1, 3, True)
    got, ref = gpu_and_oracle(bsf, causal, wl, wr, seg_q, seg_kv, Lq, Lk, bq, bk)
    assert_same(got, ref, f"ragged case {n}")


ATTN = [
    # label, B, Hq, Hkv, Lq, Lk, dqk, dv, blk, softcap, mask kwargs
    ("causal, 1000 x 1000, GQA", 1, 4, 2, 1000, 1000, 128, 128, 128, 0.0, dict(causal=True)),
    ("no mask, 777 x 1300, softcap", 2, 2, 1, 777, 1300, 128, 128, 128, 30.0, dict(causal=False)),
    ("window + causal, 1090, blocks 64", 1, 2, 2, 1090, 1090, 64, 64, 64, 0.0, dict(causal=True, wl=200)),
    ("documents, 900, batch 2", 2, 2, 2, 900, 900, 128, 128, 128, 0.0, dict(causal=True, docs=True)),
    ("d192/128 MHA, 650 x 700", 1, 2, 2, 650, 700, 192, 128, 128, 0.0, dict(causal=False)),
    ("one real row past a block, 129", 1, 2, 1, 129, 129, 128, 128, 128, 0.0, dict(causal=True)),
    ("a single query against 4096 keys (decode)", 2, 4, 1, 1, 4096, 128, 128, 128, 0.0, dict(causal=False)),
    ("keys shorter than a block, 300 x 50", 1, 2, 2, 300, 50, 64, 64, 64, 10.0, dict(causal=False)),
    ("a single query, causal (sees key 0 only)", 1, 2, 2, 1, 777, 128, 128, 128, 0.0, dict(causal=True)),
]


def make(bsf, B, Hq, Hkv, Lq, Lk, dqk, dv, blk, causal=True, wl=-1, wr=-1, docs=False, seed=0):
    q = workloads.normal_bf16((B, Hq, Lq, dqk), seed + 1)
    k = workloads.normal_bf16((B, Hkv, Lk, dqk), seed + 2)
    v = workloads.normal_bf16((B, Hkv, Lk, dv), seed + 3)
    seg = workloads.random_segment_ids(B, Lq, seed + 4, 4, True) if docs else None
    segd = seg.cuda() if seg is not None else None
    mi = bsf.build_mask_info(bsf.MaskSpec(causal, wl, wr, segd, segd), Lq, Lk, blk, blk)
    ospec = oracle.MaskSpec(causal, wl, wr, seg.numpy() if seg is not None else None,
                            seg.numpy() if seg is not None else None)
    return q, k, v, mi, ospec


def guarded(shape, dtype, fill):
    """A view of `shape` at the start of a larger buffer whose tail holds a
    sentinel: a write past the tensor changes the tail."""
    n = int(np.prod(shape))
    buf = torch.full((n + 4096,), fill, dtype=dtype, device="cuda")
    return buf, buf[:n].view(shape)


@pytest.mark.parametrize("case", ATTN, ids=[c[0] for c in ATTN])
def test_ragged_forward_matches_the_oracle(bsf, case):
    label, B, Hq, Hkv, Lq, Lk, dqk, dv, blk, cap, kw = case
    q, k, v, mi, ospec = make(bsf, B, Hq, Hkv, Lq, Lk, dqk, dv, blk, seed=17 * ATTN.index(case), **kw)
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
    # split-KV over the same ragged table
    out2, lse2 = bsf.attention_fwd(qd, kd, vd, mi, scale, cap, num_splits=3)
    # the Max Logit Estimate (with a cap, c = cap; else a constant above the scores)
    out3, lse3 = bsf.attention_fwd(qd, kd, vd, mi, scale, cap, max_logit=cap if cap > 0 else 8.0)
    torch.cuda.synchronize()
    assert bsf.last_device_error() == 0, f"{label}: device error"
    for o_, l_, what in ((out2, lse2, "split-KV"), (out3, lse3, "MLE")):
        compare_rows(o_.float().cpu().numpy().reshape(-1, dv), l_.cpu().numpy().reshape(-1),
                     O.reshape(-1, dv), L.reshape(-1), f"{label}, {what}")
    mi.close()


RAGGED_BWD = [
    # label, B, Hq, Hkv, Lq, Lk, d, softcap, mask kwargs
    ("causal GQA 1000", 1, 4, 2, 1000, 1000, 128, 0.0, dict(causal=True)),
    ("no mask 700 x 900, cap, batch 2", 2, 2, 1, 700, 900, 64, 20.0, dict(causal=False)),
    ("window + causal 1090", 1, 2, 2, 1090, 1090, 128, 0.0, dict(causal=True, wl=300)),
]


@pytest.mark.parametrize("case", RAGGED_BWD, ids=[c[0] for c in RAGGED_BWD])
def test_ragged_backward_matches_the_oracle(bsf, case):
    from tests.test_gpu_backward import compare_grad, d_term_allowance
    label, B, Hq, Hkv, Lq, Lk, d, cap, kw = case
    q, k, v, mi, ospec = make(bsf, B, Hq, Hkv, Lq, Lk, d, d, 128, seed=23 * RAGGED_BWD.index(case), **kw)
    g = workloads.normal_bf16((B, Hq, Lq, d), 500 + RAGGED_BWD.index(case))
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd, gd = q.cuda(), k.cuda(), v.cuda(), g.cuda()
    out, lse = bsf.attention_fwd(qd, kd, vd, mi, scale, cap)
    # guard tails after dk / dv: padding keys must never be stored
    kbuf, dk = guarded(tuple(k.shape), torch.bfloat16, 7.0)
    vbuf, dv = guarded(tuple(v.shape), torch.bfloat16, 7.0)
    dq, dk, dv = bsf.attention_bwd(qd, kd, vd, out, lse, gd, mi, scale, cap, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert bsf.last_device_error() == 0, label
    assert torch.all(kbuf[dk.numel():] == 7.0) and torch.all(vbuf[dv.numel():] == 7.0), f"{label}: wrote past"
    ref = oracle.attention_bwd(q, k, v, g, ospec, scale, cap)
    extra = d_term_allowance(q, k, v, g, ospec, scale, cap)
    compare_grad(dq, ref["dq"], f"{label}: dq", extra)
    compare_grad(dk, ref["dk"], f"{label}: dk")
    compare_grad(dv, ref["dv"], f"{label}: dv")
    mi.close()
