"""Max Logit Estimate forward on the GPU ("Pallas Kernels and Splash
Attention" §5.4): the softmax reference fixed at a constant c.

Inside the safe range c cancels, so the result must match the f64 oracle of
the plain definition to the same tolerances as the plain forward.  With a
soft cap, c = cap is always safe.  A constant far below the scores exercises
the kernel's overflow guard (the result must still match); one far above a
row's scores makes the row underflow, which gives the documented fully
masked output."""
import math

import numpy as np
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
    # label, B, Hq, Hkv, L, dqk, dv, blk, scale multiplier, softcap, c, mask kwargs
    ("softcap 30, c = cap, window + causal", 1, 4, 2, 2048, 128, 128, 128, 1.0, 30.0, 30.0, dict(wl=700)),
    ("softcap 50, c = cap, tiny MHA", 1, 2, 2, 256, 64, 64, 64, 1.0, 50.0, 50.0, {}),
    ("softcap 20, c = cap, sharp scores, GQA", 1, 8, 2, 1024, 128, 128, 128, 4.0, 20.0, 20.0, {}),
    ("no cap, c = 8, dense causal", 2, 4, 1, 1024, 128, 128, 128, 1.0, 0.0, 8.0, {}),
    ("no cap, c = 0, documents", 2, 2, 2, 1024, 128, 128, 128, 1.0, 0.0, 0.0, dict(docs=True)),
    ("no cap, d192/128 MHA, c = 5", 1, 2, 2, 512, 192, 128, 128, 1.0, 0.0, 5.0, dict(causal=False)),
    # scores up to ~40 against c = -20: blocks overflow the fixed reference
    # and take the guard's recompute
    ("guard: c far below the scores", 1, 4, 2, 1024, 128, 128, 128, 8.0, 0.0, -20.0, {}),
]


def make(bsf, B, Hq, Hkv, L, dqk, dv, blk, causal=True, wl=-1, wr=-1, docs=False, seed=0):
    q = workloads.normal_bf16((B, Hq, L, dqk), seed + 1)
    k = workloads.normal_bf16((B, Hkv, L, dqk), seed + 2)
    v = workloads.normal_bf16((B, Hkv, L, dv), seed + 3)
    seg = workloads.random_segment_ids(B, L, seed + 4, 4, True) if docs else None
    segd = seg.cuda() if seg is not None else None
    mi = bsf.build_mask_info(bsf.MaskSpec(causal, wl, wr, segd, segd), L, L, blk, blk)
    ospec = oracle.MaskSpec(causal, wl, wr, seg.numpy() if seg is not None else None,
                            seg.numpy() if seg is not None else None)
    return q, k, v, mi, ospec


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_mle_matches_the_oracle(bsf, case):
    label, B, Hq, Hkv, L, dqk, dv, blk, mult, cap, c, kw = case
    q, k, v, mi, ospec = make(bsf, B, Hq, Hkv, L, dqk, dv, blk, seed=11 * CASES.index(case), **kw)
    scale = mult / math.sqrt(dqk)
    O, LSE = oracle.attention(q, k, v, ospec, scale, cap)
    out, lse = bsf.attention_fwd(q.cuda(), k.cuda(), v.cuda(), mi, scale, cap, max_logit=c)
    torch.cuda.synchronize()
    assert bsf.last_device_error() == 0, f"{label}: device error"
    compare_rows(out.float().cpu().numpy().reshape(-1, dv), lse.cpu().numpy().reshape(-1),
                 O.reshape(-1, dv), LSE.reshape(-1), label)
    mi.close()


def test_mle_agrees_with_the_plain_forward(bsf):
    q, k, v, mi, _ = make(bsf, 1, 4, 2, 2048, 128, 128, 128, wl=1000, seed=5)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out0, lse0 = bsf.attention_fwd(qd, kd, vd, mi, 128 ** -0.5, 30.0)
    out1, lse1 = bsf.attention_fwd(qd, kd, vd, mi, 128 ** -0.5, 30.0, max_logit=30.0)
    torch.cuda.synchronize()
    # the two differ by rounding only (P is rounded to bf16 against different
    # references before the PV product): well inside the output tolerance,
    # and equal on average
    d = (out0.float() - out1.float()).abs()
    assert d.max().item() <= 2e-2
    assert d.mean().item() <= 1e-3
    assert (lse0 - lse1).abs().max().item() <= 1e-4
    mi.close()


def test_mle_underflow_gives_the_masked_row_output(bsf):
    # scores ~ N(0, 1) against c = 300: every exponential flushes to zero, so
    # each row ends with l = 0 and is reported like a fully masked row
    q, k, v, mi, _ = make(bsf, 1, 2, 2, 256, 64, 64, 64, seed=9)
    out, lse = bsf.attention_fwd(q.cuda(), k.cuda(), v.cuda(), mi, 0.125, 0.0, max_logit=300.0)
    torch.cuda.synchronize()
    assert bsf.last_device_error() == 0
    assert torch.all(out == 0)
    assert torch.all(torch.isneginf(lse))
    mi.close()


@pytest.mark.parametrize("bad", [float("inf"), float("-inf"), float("nan")])
def test_mle_rejects_non_finite_constants(bsf, bad):
    q, k, v, mi, _ = make(bsf, 1, 2, 2, 256, 64, 64, 64)
    with pytest.raises(bsf.SplashError):
        bsf.attention_fwd(q.cuda(), k.cuda(), v.cuda(), mi, 0.125, 0.0, max_logit=bad)
    with pytest.raises(ValueError):
        bsf.attention_fwd(q.cuda(), k.cuda(), v.cuda(), mi, 0.125, 0.0, max_logit=1.0, num_splits=2)
    mi.close()
