"""Split-KV forward + LSE merge on the GPU.

The merged result must match the f64 oracle exactly as the one-pass forward
does (every row, several splits per row, splits beyond a row's block count),
one split must reproduce the one-pass forward bit for bit, and the merge
kernel alone must match the oracle's two-segment merge folded over splits."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle.softmax_ref import merge as oracle_merge
from tests.parity import compare_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bsf():
    from block_sparse_flash_gb300 import build as b
    b.build()
    import block_sparse_flash_gb300 as m
    return m


CASES = [
    # label, B, Hq, Hkv, Lq, Lk, dqk, dv, blk, splits, kwargs
    ("few queries, long keys, GQA", 1, 4, 2, 256, 4096, 128, 128, 128, (2, 3, 7), dict(causal=False)),
    ("causal, empty splits on early rows", 1, 2, 2, 1024, 1024, 64, 64, 64, (4, 16), {}),
    ("window + causal + softcap", 1, 4, 2, 2048, 2048, 128, 128, 128, (3,), dict(wl=700, softcap=30.0)),
    ("document mask, batch of 2", 2, 2, 1, 1024, 1024, 128, 128, 128, (2, 5), dict(docs=True)),
    ("MHA pairs d192/128", 1, 2, 2, 512, 1536, 192, 128, 128, (4,), dict(causal=False)),
    ("odd heads, blocks 64", 1, 3, 1, 512, 2048, 128, 128, 64, (6,), dict(causal=False, wl=900, wr=300)),
]


def make(bsf, B, Hq, Hkv, Lq, Lk, dqk, dv, blk, causal=True, wl=-1, wr=-1, softcap=0.0, docs=False, seed=0):
    q = workloads.normal_bf16((B, Hq, Lq, dqk), seed + 1)
    k = workloads.normal_bf16((B, Hkv, Lk, dqk), seed + 2)
    v = workloads.normal_bf16((B, Hkv, Lk, dv), seed + 3)
    seg = workloads.random_segment_ids(B, Lq, seed + 4, 5, True) if docs else None
    segd = seg.cuda() if seg is not None else None
    mi = bsf.build_mask_info(bsf.MaskSpec(causal, wl, wr, segd, segd), Lq, Lk, blk, blk)
    ospec = oracle.MaskSpec(causal, wl, wr, seg.numpy() if seg is not None else None,
                            seg.numpy() if seg is not None else None)
    return q, k, v, mi, ospec


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_split_then_merge_matches_the_oracle(bsf, case):
    label, B, Hq, Hkv, Lq, Lk, dqk, dv, blk, splits, kw = case
    softcap = kw.get("softcap", 0.0)
    q, k, v, mi, ospec = make(bsf, B, Hq, Hkv, Lq, Lk, dqk, dv, blk, seed=7 * CASES.index(case), **kw)
    scale = 1.0 / math.sqrt(dqk)
    O, L = oracle.attention(q, k, v, ospec, scale, softcap)
    for S in splits:
        out, lse = bsf.attention_fwd(q.cuda(), k.cuda(), v.cuda(), mi, scale, softcap, num_splits=S)
        torch.cuda.synchronize()
        assert bsf.last_device_error() == 0, f"{label}: device error"
        compare_rows(out.float().cpu().numpy().reshape(-1, dv), lse.cpu().numpy().reshape(-1),
                     O.reshape(-1, dv), L.reshape(-1), f"{label}, {S} splits")
    mi.close()


def test_one_split_is_the_one_pass_forward(bsf):
    q, k, v, mi, _ = make(bsf, 1, 4, 2, 1024, 1024, 128, 128, 128, wl=300, softcap=20.0, seed=3)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out1, lse1 = bsf.attention_fwd(qd, kd, vd, mi, 128 ** -0.5, 20.0)
    o_part, lse_part = bsf.attention_fwd_split(qd, kd, vd, mi, 128 ** -0.5, 20.0, 1)
    out2, lse2 = bsf.attention_merge(o_part, lse_part)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2)
    assert torch.equal(lse1, lse2)
    mi.close()


def test_partials_are_normalised_per_split(bsf):
    # each split's o_part is its own softmax average: merging any subset of
    # the splits with the merge kernel equals the oracle merge of that subset
    q, k, v, mi, _ = make(bsf, 1, 2, 2, 256, 2048, 64, 64, 64, causal=False, seed=5)
    o_part, lse_part = bsf.attention_fwd_split(q.cuda(), k.cuda(), v.cuda(), mi, 0.125, 0.0, 4)
    torch.cuda.synchronize()
    op, lp = o_part.cpu().numpy().astype(np.float64), lse_part.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(lp))  # 32 kv-blocks per row: every split has keys
    for subset in ([0, 1], [1, 2, 3], [0, 3]):
        out, lse = bsf.attention_merge(o_part[subset].contiguous(), lse_part[subset].contiguous())
        ref_o, ref_l = fold(op[subset].reshape(len(subset), -1, 64), lp[subset].reshape(len(subset), -1))
        np.testing.assert_allclose(out.float().cpu().numpy().reshape(-1, 64), ref_o, atol=1e-2, rtol=1e-2)
        np.testing.assert_allclose(lse.cpu().numpy().reshape(-1), ref_l, atol=1e-5, rtol=1e-6)
    mi.close()


def fold(o_part, lse_part):
    """Oracle merge (two segments at a time) of normalised partials: segment
    state (m, l, unnormalised o) = (lse_s, 1, o_s)."""
    S, R, dv = o_part.shape
    out = np.zeros((R, dv))
    lse = np.full(R, -np.inf)
    for r in range(R):
        state = None
        for s in range(S):
            if not np.isfinite(lse_part[s, r]):
                continue
            seg = (lse_part[s, r], 1.0, o_part[s, r])
            if state is None:
                state = seg
            else:
                m, l, o = oracle_merge(*state, *seg)
                state = (m, l, o * l)
        if state is not None:
            out[r] = state[2] / state[1]
            lse[r] = state[0] + np.log(state[1])
    return out, lse


@pytest.mark.parametrize("dv", [64, 128])
def test_merge_kernel_alone(bsf, dv):
    rng = np.random.default_rng(dv)
    S, R = 5, 777
    o_part = rng.standard_normal((S, R, dv)).astype(np.float32)
    lse_part = (rng.standard_normal((S, R)) * 8).astype(np.float32)
    lse_part[rng.random((S, R)) < 0.3] = -np.inf       # empty splits
    lse_part[:, :3] = -np.inf                           # rows with no keys at all
    o_part[~np.isfinite(lse_part)] = 0.0
    out, lse = bsf.attention_merge(torch.from_numpy(o_part).cuda(), torch.from_numpy(lse_part).cuda())
    torch.cuda.synchronize()
    ref_o, ref_l = fold(o_part.astype(np.float64), lse_part.astype(np.float64))
    got_o, got_l = out.float().cpu().numpy(), lse.cpu().numpy()
    assert np.all(got_o[:3] == 0) and np.all(np.isneginf(got_l[:3]))
    np.testing.assert_allclose(got_o, ref_o, atol=2e-2, rtol=1e-2)
    np.testing.assert_allclose(got_l[3:], ref_l[3:], atol=1e-4, rtol=1e-6)


def test_invalid_split_arguments(bsf):
    q, k, v, mi, _ = make(bsf, 1, 2, 2, 256, 256, 64, 64, 64, seed=1)
    with pytest.raises(bsf.SplashError):
        bsf.attention_fwd_split(q.cuda(), k.cuda(), v.cuda(), mi, 0.125, 0.0, 0)
    with pytest.raises(bsf.SplashError):
        bsf.attention_fwd_split(q.cuda(), k.cuda(), v.cuda(), mi, 0.125, 0.0, 1000)
    mi.close()
