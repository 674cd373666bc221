"""Backward pass on the GPU against the f64 backward oracle.

The GPU backward is fed the GPU forward's out and lse (its own product
path); the oracle differentiates the forward's definition from q, k, v and
dout (exact D).  The GPU forms D_i = dout_i . out_i from the stored bf16
output, which moves small dq rows by several per cent; each dq row's bound
therefore adds an allowance derived from that rounding (d_term_allowance).
Gradients are compared per tensor with the tolerances of the
forward's output (bf16 results of fp32 arithmetic on bf16 operands):
max |error| <= 2e-2 * max |reference| and, per row (one query's dq, one
key's dk / dv), ||error|| <= 2e-2 * max(||reference row||, 1e-2 * the
largest reference row norm)."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

GRAD_ABS = 2e-2   # relative to the tensor's largest |reference| entry
GRAD_ROW = 2e-2   # per-row relative norm


@pytest.fixture(scope="module")
def bsf():
    from block_sparse_flash_gb300 import build as b
    b.build()
    import block_sparse_flash_gb300 as m
    return m


def compare_grad(got, ref, label, extra=None):
    """extra: optional per-row absolute allowance added to the row bound."""
    g = got.float().cpu().numpy().astype(np.float64).reshape(-1, got.shape[-1])
    r = ref.reshape(-1, ref.shape[-1])
    assert np.all(np.isfinite(g)), f"{label}: non-finite"
    scale = max(float(np.abs(r).max()), 1e-30)
    err = np.abs(g - r)
    assert float(err.max()) <= GRAD_ABS * scale, f"{label}: max abs err {err.max():.3e} (max |ref| {scale:.3e})"
    rn = np.linalg.norm(r, axis=1)
    bound = GRAD_ROW * np.maximum(rn, 1e-2 * max(float(rn.max()), 1e-30))
    if extra is not None:
        bound = bound + extra.reshape(-1)
    ratio = float((np.linalg.norm(g - r, axis=1) / bound).max())
    assert ratio <= 1.0, f"{label}: row error {ratio:.3f} x its bound"
    return float(err.max()) / scale, ratio


CASES = [
    # label, B, Hq, Hkv, L, d, softcap, mask kwargs
    ("causal MHA d128", 1, 2, 2, 512, 128, 0.0, dict(causal=True)),
    ("causal GQA d128 softcap 30", 2, 4, 2, 1024, 128, 30.0, dict(causal=True)),
    ("window 300 + causal d64", 1, 4, 1, 1024, 64, 0.0, dict(causal=True, wl=299)),
    ("documents + causal, batch 2", 2, 2, 1, 768, 128, 0.0, dict(causal=True, docs=True)),
    ("two-sided window, no causal", 1, 2, 2, 640, 128, 20.0, dict(causal=False, wl=200, wr=150)),
]


def make(bsf, B, Hq, Hkv, L, d, causal=True, wl=-1, wr=-1, docs=False, seed=0, kv_seg=None, bq=128):
    q = workloads.normal_bf16((B, Hq, L, d), seed + 1)
    k = workloads.normal_bf16((B, Hkv, L, d), seed + 2)
    v = workloads.normal_bf16((B, Hkv, L, d), seed + 3)
    g = workloads.normal_bf16((B, Hq, L, d), seed + 5)
    qs = workloads.random_segment_ids(B, L, seed + 4, 4, True) if docs else None
    ks = kv_seg if kv_seg is not None else qs
    mi = bsf.build_mask_info(bsf.MaskSpec(causal, wl, wr, qs.cuda() if qs is not None else None,
                                          ks.cuda() if ks is not None else None), L, L, bq, 128)
    ospec = oracle.MaskSpec(causal, wl, wr, qs.numpy() if qs is not None else None,
                            ks.numpy() if ks is not None else None)
    return q, k, v, g, mi, ospec


def run_both(bsf, q, k, v, g, mi, ospec, scale, cap):
    qd, kd, vd, gd = q.cuda(), k.cuda(), v.cuda(), g.cuda()
    out, lse = bsf.attention_fwd(qd, kd, vd, mi, scale, cap)
    dq, dk, dv = bsf.attention_bwd(qd, kd, vd, out, lse, gd, mi, scale, cap)
    torch.cuda.synchronize()
    assert bsf.last_device_error() == 0, "device error"
    ref = oracle.attention_bwd(q, k, v, g, ospec, scale, cap)
    return (dq, dk, dv), ref


def d_term_allowance(q, k, v, g, ospec, scale, cap):
    """Per-row allowance for dq from D_i = dout_i . out_i being formed from
    the stored bf16 output instead of the exact one.  Each element of that
    output is within 2^-9 |O_id| (its bf16 rounding) plus 2^-9 sum_j P_ij
    |v_jd| (the bf16 rounding of P before the PV product) of the exact O, so
    |dD_i| <= 2^-9 sum_d |dout_id| (|O_id| + sum_j P_ij |v_jd|).  A change
    dD_i of D moves dq_i by exactly dD_i times the dq_i of a backward with
    dout = 0 and D = 1 (pinned in the oracle tests), so the allowance is
    |dD_i| * ||that row||.  The weighted sums are the oracle's own forward
    with other values (|v|)."""
    O, _ = oracle.attention(q, k, v, ospec, scale, cap)
    A, _ = oracle.attention(q, k, v.abs(), ospec, scale, cap)
    dD = 2.0 ** -9 * np.sum(np.abs(g.double().numpy()) * (np.abs(O) + A), axis=-1)
    B, Hq, Lq, _ = q.shape
    unit = oracle.attention_bwd(q, k, v, torch.zeros_like(g), ospec, scale, cap, delta=np.ones((B, Hq, Lq)))
    return dD * np.linalg.norm(unit["dq"], axis=-1)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_backward_matches_the_oracle(bsf, case):
    label, B, Hq, Hkv, L, d, cap, kw = case
    q, k, v, g, mi, ospec = make(bsf, B, Hq, Hkv, L, d, seed=13 * CASES.index(case), **kw)
    scale = 1.0 / math.sqrt(d)
    (dq, dk, dv), ref = run_both(bsf, q, k, v, g, mi, ospec, scale, cap)
    extra = d_term_allowance(q, k, v, g, ospec, scale, cap)
    errs = [compare_grad(dq, ref["dq"], f"{label}: dq", extra), compare_grad(dk, ref["dk"], f"{label}: dk"),
            compare_grad(dv, ref["dv"], f"{label}: dv")]
    print(label, errs)
    mi.close()


TALL_CASES = [
    # label, B, Hq, Hkv, L, d, softcap, mask kwargs -- tables of 256-row q-blocks
    ("256-row blocks, causal MHA d128", 1, 2, 2, 1024, 128, 0.0, dict(causal=True)),
    ("256-row blocks, documents + causal GQA, batch 2", 2, 4, 2, 768, 128, 0.0, dict(causal=True, docs=True)),
    ("256-row blocks, ragged causal 1000", 1, 2, 1, 1000, 128, 0.0, dict(causal=True)),
    ("256-row blocks, window 300 + causal d64 cap 30", 1, 2, 2, 896, 64, 30.0, dict(causal=True, wl=299)),
]


@pytest.mark.parametrize("case", TALL_CASES, ids=[c[0] for c in TALL_CASES])
def test_backward_with_256_row_blocks_matches_the_oracle(bsf, case):
    """A table of 256-row q-blocks: the backward takes each as two 128-row
    halves (the half's rows of Q, dO, LSE, D and its words of the transposed
    pattern); a half the mask leaves empty for a key block contributes
    nothing."""
    label, B, Hq, Hkv, L, d, cap, kw = case
    q, k, v, g, mi, ospec = make(bsf, B, Hq, Hkv, L, d, seed=17 * TALL_CASES.index(case) + 3, bq=256, **kw)
    assert mi.shape()["bq"] == 256
    scale = 1.0 / math.sqrt(d)
    (dq, dk, dv), ref = run_both(bsf, q, k, v, g, mi, ospec, scale, cap)
    extra = d_term_allowance(q, k, v, g, ospec, scale, cap)
    errs = [compare_grad(dq, ref["dq"], f"{label}: dq", extra), compare_grad(dk, ref["dk"], f"{label}: dk"),
            compare_grad(dv, ref["dv"], f"{label}: dv")]
    print(label, errs)
    mi.close()


def test_256_row_blocks_give_the_same_key_gradients(bsf):
    """dk and dv of a 256-row table equal those of the 128-row table bit for
    bit: both visit the same 128-row pieces of a key block's column in the
    same order, and a half that the mask leaves empty adds exact zeros."""
    B, Hq, Hkv, L, d = 1, 4, 2, 1024, 128
    grads = []
    for bq in (128, 256):
        q, k, v, g, mi, ospec = make(bsf, B, Hq, Hkv, L, d, seed=5, bq=bq)
        qd, kd, vd, gd = q.cuda(), k.cuda(), v.cuda(), g.cuda()
        mi128 = bsf.build_mask_info(bsf.MaskSpec(True), L, L, 128, 128)
        out, lse = bsf.attention_fwd(qd, kd, vd, mi128, d ** -0.5)  # same forward for both
        grads.append(bsf.attention_bwd(qd, kd, vd, out, lse, gd, mi, d ** -0.5))
        torch.cuda.synchronize()
        assert bsf.last_device_error() == 0
        mi.close()
        mi128.close()
    assert torch.equal(grads[0][1], grads[1][1]) and torch.equal(grads[0][2], grads[1][2])
    assert (grads[0][0].float() - grads[1][0].float()).abs().max().item() <= 2e-2 * grads[0][0].float().abs().max().item()


def test_keys_no_query_sees_get_zero_gradients(bsf):
    # key block 2 carries a segment ID no query has: its column of the table is
    # empty, and dk = dv = 0 there
    B, Hq, Hkv, L, d = 1, 2, 1, 512, 128
    qs = torch.zeros((B, L), dtype=torch.int32)
    ks = torch.zeros((B, L), dtype=torch.int32)
    ks[:, 256:384] = 7
    q = workloads.normal_bf16((B, Hq, L, d), 91)
    k = workloads.normal_bf16((B, Hkv, L, d), 92)
    v = workloads.normal_bf16((B, Hkv, L, d), 93)
    g = workloads.normal_bf16((B, Hq, L, d), 94)
    mi = bsf.build_mask_info(bsf.MaskSpec(False, -1, -1, qs.cuda(), ks.cuda()), L, L, 128, 128)
    ospec = oracle.MaskSpec(False, -1, -1, qs.numpy(), ks.numpy())
    (dq, dk, dv), ref = run_both(bsf, q, k, v, g, mi, ospec, d ** -0.5, 0.0)
    assert torch.all(dk[:, :, 256:384] == 0) and torch.all(dv[:, :, 256:384] == 0)
    compare_grad(dq, ref["dq"], "dq")
    compare_grad(dk, ref["dk"], "dk")
    compare_grad(dv, ref["dv"], "dv")
    mi.close()


def test_dk_dv_are_deterministic_and_dq_nearly(bsf):
    q, k, v, g, mi, _ = make(bsf, 1, 4, 2, 1024, 128, seed=40)
    qd, kd, vd, gd = q.cuda(), k.cuda(), v.cuda(), g.cuda()
    out, lse = bsf.attention_fwd(qd, kd, vd, mi, 128 ** -0.5, 0.0)
    a = bsf.attention_bwd(qd, kd, vd, out, lse, gd, mi, 128 ** -0.5, 0.0)
    b = bsf.attention_bwd(qd, kd, vd, out, lse, gd, mi, 128 ** -0.5, 0.0)
    torch.cuda.synchronize()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    # dq: fp32 atomic additions in varying order, then one bf16 rounding
    assert (a[0].float() - b[0].float()).abs().max().item() <= 1e-2 * a[0].float().abs().max().item()
    mi.close()


def test_column_table_follows_rebuilds(bsf):
    # the backward keeps the MaskInfo's column-major copy between calls and
    # must make a new one after the table is rebuilt with another mask
    B, Hq, Hkv, L, d = 1, 2, 1, 640, 128
    q = workloads.normal_bf16((B, Hq, L, d), 61)
    k = workloads.normal_bf16((B, Hkv, L, d), 62)
    v = workloads.normal_bf16((B, Hkv, L, d), 63)
    g = workloads.normal_bf16((B, Hq, L, d), 64)
    qd, kd, vd, gd = q.cuda(), k.cuda(), v.cuda(), g.cuda()
    mi = bsf.build_mask_info(bsf.MaskSpec(True), L, L, 128, 128)
    out, lse = bsf.attention_fwd(qd, kd, vd, mi, d ** -0.5)
    first = bsf.attention_bwd(qd, kd, vd, out, lse, gd, mi, d ** -0.5)
    again = bsf.attention_bwd(qd, kd, vd, out, lse, gd, mi, d ** -0.5)
    torch.cuda.synchronize()
    assert torch.equal(first[1], again[1]) and torch.equal(first[2], again[2])
    for spec, ospec in ((bsf.MaskSpec(True, 199, -1), oracle.MaskSpec(True, 199, -1)),
                        (bsf.MaskSpec(False, 100, 300), oracle.MaskSpec(False, 100, 300))):
        mi.rebuild(spec, L, L, 128, 128)
        out, lse = bsf.attention_fwd(qd, kd, vd, mi, d ** -0.5)
        dq, dk, dv = bsf.attention_bwd(qd, kd, vd, out, lse, gd, mi, d ** -0.5)
        torch.cuda.synchronize()
        assert bsf.last_device_error() == 0
        ref = oracle.attention_bwd(q, k, v, g, ospec, d ** -0.5, 0.0)
        compare_grad(dq, ref["dq"], "dq after rebuild", d_term_allowance(q, k, v, g, ospec, d ** -0.5, 0.0))
        compare_grad(dk, ref["dk"], "dk after rebuild")
        compare_grad(dv, ref["dv"], "dv after rebuild")
    mi.close()


def test_backward_rejects_unsupported_shapes(bsf):
    q, k, v, g, mi, _ = make(bsf, 1, 2, 2, 256, 128)
    qd, kd, vd, gd = q.cuda(), k.cuda(), v.cuda(), g.cuda()
    out, lse = bsf.attention_fwd(qd, kd, vd, mi, 0.1, 0.0)
    with pytest.raises(bsf.SplashError):  # workspace too small
        bsf.attention_bwd(qd, kd, vd, out, lse, gd, mi, 0.1, 0.0,
                          workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    mi.close()
    mi64 = bsf.build_mask_info(bsf.MaskSpec(True, -1, -1, None, None), 256, 256, 64, 64)
    with pytest.raises(bsf.SplashError):  # 64 x 64 blocks: unsupported by the backward
        bsf.attention_bwd(qd, kd, vd, out, lse, gd, mi64, 0.1, 0.0)
    mi64.close()
