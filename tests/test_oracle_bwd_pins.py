"""Pins for the backward oracle (gradients of masked attention).  CPU only.

The backward oracle differentiates the forward's definition by hand (the
softmax Jacobian, P recomputed from the row log-sum-exp).  These tests pin it
to things other than itself: central finite differences of an independent
dense forward written here, torch autograd in float64, closed forms (a query
that sees only itself passes its upstream gradient straight to v and none to
q or k), the zero-sum of key gradients implied by softmax shift invariance,
and consistency with the forward oracle (its LSE, and D_i = dout_i . out_i).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import MaskSpec


def dense_mask(spec: MaskSpec, b, Lq, Lk):
    i = np.arange(Lq)[:, None]
    j = np.arange(Lk)[None, :]
    m = np.ones((Lq, Lk), dtype=bool)
    if spec.causal:
        m &= j <= i
    if spec.window_left >= 0:
        m &= i - j <= spec.window_left
    if spec.window_right >= 0:
        m &= j - i <= spec.window_right
    if spec.q_segment_ids is not None:
        m &= np.asarray(spec.q_segment_ids)[b][:, None] == np.asarray(spec.kv_segment_ids)[b][None, :]
    return m


def dense_forward(q, k, v, spec, scale, cap):
    """Textbook masked softmax attention in float64 (numpy), for finite
    differences: out[b, h] = softmax(mask(s)) v with s = scale q k^T
    (capped: cap tanh(s / cap))."""
    B, Hq, Lq, _ = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Hq, Lq, v.shape[3]))
    for b in range(B):
        m = dense_mask(spec, b, Lq, Lk)
        for h in range(Hq):
            s = scale * q[b, h] @ k[b, h // G].T
            if cap > 0:
                s = cap * np.tanh(s / cap)
            s = np.where(m, s, -np.inf)
            mx = np.max(s, axis=1, keepdims=True)
            live = np.isfinite(mx)
            e = np.where(m, np.exp(s - np.where(live, mx, 0)), 0.0)
            den = np.sum(e, axis=1, keepdims=True)
            out[b, h] = np.where(live, e / np.where(den > 0, den, 1), 0) @ v[b, h // G]
    return out


SPECS = [
    ("causal", MaskSpec(True, -1, -1), 0.0),
    ("window 3 + causal + cap 2", MaskSpec(True, 2, -1), 2.0),
    ("two-sided window", MaskSpec(False, 3, 1), 0.0),
    ("documents + causal + cap 5", None, 5.0),
]


def spec_of(name, spec, B, L, seed):
    if spec is not None:
        return spec
    seg = workloads.random_segment_ids(B, L, seed, 3, True).numpy()
    return MaskSpec(True, -1, -1, seg, seg)


@pytest.mark.parametrize("case", SPECS, ids=[c[0] for c in SPECS])
def test_backward_matches_finite_differences(case):
    name, spec, cap = case
    rng = np.random.default_rng(3)
    B, Hq, Hkv, L, d, dv = 2, 2, 1, 10, 4, 3
    spec = spec_of(name, spec, B, L, 5)
    q = rng.normal(size=(B, Hq, L, d))
    k = rng.normal(size=(B, Hkv, L, d))
    v = rng.normal(size=(B, Hkv, L, dv))
    g = rng.normal(size=(B, Hq, L, dv))
    scale = 0.7
    r = oracle.attention_bwd(q, k, v, g, spec, scale, cap)
    eps = 1e-6

    def loss(qq, kk, vv):
        return float(np.sum(dense_forward(qq, kk, vv, spec, scale, cap) * g))

    for name_x, x, grad in (("q", q, r["dq"]), ("k", k, r["dk"]), ("v", v, r["dv"])):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = dict(q=q, k=k, v=v)
            args_m = dict(q=q, k=k, v=v)
            args_p[name_x], args_m[name_x] = xp, xm
            num[idx] = (loss(args_p["q"], args_p["k"], args_p["v"]) -
                        loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * eps)
        np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-7, err_msg=f"{name}: d{name_x}")


def test_backward_matches_torch_autograd_gqa_documents_softcap():
    B, Hq, Hkv, L, d, dv = 2, 4, 2, 48, 16, 8
    seg = workloads.random_segment_ids(B, L, 17, 4, True).numpy()
    spec = MaskSpec(True, 20, -1, seg, seg)
    gen = torch.Generator().manual_seed(4)
    q = torch.randn(B, Hq, L, d, generator=gen, dtype=torch.float64)
    k = torch.randn(B, Hkv, L, d, generator=gen, dtype=torch.float64)
    v = torch.randn(B, Hkv, L, dv, generator=gen, dtype=torch.float64)
    g = torch.randn(B, Hq, L, dv, generator=gen, dtype=torch.float64)
    scale, cap = 0.4, 3.0
    r = oracle.attention_bwd(q, k, v, g, spec, scale, cap)
    qt, kt, vt = (x.clone().requires_grad_(True) for x in (q, k, v))
    mask = torch.stack([torch.from_numpy(dense_mask(spec, b, L, L)) for b in range(B)])[:, None]
    kr = kt.repeat_interleave(Hq // Hkv, dim=1)
    vr = vt.repeat_interleave(Hq // Hkv, dim=1)
    s = cap * torch.tanh(scale * qt @ kr.transpose(-1, -2) / cap)
    p = torch.softmax(s.masked_fill(~mask, float("-inf")), dim=-1)
    (p @ vr * g).sum().backward()
    np.testing.assert_allclose(r["dq"], qt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(r["dk"], kt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(r["dv"], vt.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_self_only_attention_passes_the_gradient_to_v():
    # causal with a window of one key: each query sees only itself, so
    # out_i = v_i exactly, dv = dout, and q, k get no gradient
    rng = np.random.default_rng(8)
    q, k = rng.normal(size=(1, 3, 20, 8)), rng.normal(size=(1, 3, 20, 8))
    v, g = rng.normal(size=(1, 3, 20, 5)), rng.normal(size=(1, 3, 20, 5))
    r = oracle.attention_bwd(q, k, v, g, MaskSpec(True, 0, -1), 0.3, 4.0)
    np.testing.assert_array_equal(r["dq"], 0)
    np.testing.assert_array_equal(r["dk"], 0)
    np.testing.assert_allclose(r["dv"], g, rtol=0, atol=1e-15)
    np.testing.assert_allclose(r["delta"], np.sum(g * v, axis=-1), rtol=1e-14)


def test_key_gradients_sum_to_zero_without_a_cap():
    # shifting every key by the same vector shifts each row's scores by a
    # constant, which softmax ignores: the key gradients of each head sum to 0
    rng = np.random.default_rng(12)
    q, k = rng.normal(size=(1, 4, 64, 16)), rng.normal(size=(1, 2, 64, 16))
    v, g = rng.normal(size=(1, 2, 64, 16)), rng.normal(size=(1, 4, 64, 16))
    for spec in (MaskSpec(True, -1, -1), MaskSpec(False, 10, 5)):
        r = oracle.attention_bwd(q, k, v, g, spec, 0.25, 0.0)
        scale_ref = np.abs(r["dk"]).max()
        np.testing.assert_allclose(r["dk"].sum(axis=2), 0, atol=1e-12 * max(1.0, scale_ref))
        # and the value gradients of each head sum to the upstream gradient
        # over its rows (every row's weights sum to 1)
        np.testing.assert_allclose(r["dv"].sum(axis=2),
                                   g.reshape(1, 2, 2, 64, 16).sum(axis=(2, 3)), rtol=1e-12, atol=1e-12)


def test_backward_agrees_with_the_forward_oracle():
    # LSE from the backward equals the forward's; D_i = dout_i . out_i
    B, Hq, Hkv, L, d = 1, 4, 2, 256, 64
    q = workloads.normal_bf16((B, Hq, L, d), 71)
    k = workloads.normal_bf16((B, Hkv, L, d), 72)
    v = workloads.normal_bf16((B, Hkv, L, d), 73)
    g = workloads.normal_bf16((B, Hq, L, d), 74)
    spec = MaskSpec(True, 100, -1)
    O, LSE = oracle.attention(q, k, v, spec, 0.125, 10.0)
    r = oracle.attention_bwd(q, k, v, g, spec, 0.125, 10.0)
    np.testing.assert_allclose(r["lse"], LSE, rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["delta"], np.sum(O * g.double().numpy(), axis=-1), rtol=1e-11, atol=1e-12)


def test_head_subset_gives_the_same_rows():
    rng = np.random.default_rng(21)
    q, k = rng.normal(size=(2, 4, 32, 8)), rng.normal(size=(2, 1, 32, 8))
    v, g = rng.normal(size=(2, 1, 32, 8)), rng.normal(size=(2, 4, 32, 8))
    spec = MaskSpec(True, -1, -1)
    full = oracle.attention_bwd(q, k, v, g, spec, 0.5)
    part = oracle.attention_bwd(q, k, v, g, spec, 0.5, heads=[(1, 2)])
    np.testing.assert_array_equal(part["dq"][1, 2], full["dq"][1, 2])
    assert np.all(part["dq"][0] == 0)
    # one head's key contribution: the full dk minus the other heads' equals it
    others = oracle.attention_bwd(q, k, v, g, spec, 0.5, heads=[(1, 0), (1, 1), (1, 3)])
    np.testing.assert_allclose(part["dk"][1] + others["dk"][1], full["dk"][1], rtol=1e-12, atol=1e-13)


def test_given_delta_from_the_exact_output_is_the_exact_delta():
    # D_i = dout_i . out_i equals sum_j P_ij dP_ij when out is the exact
    # forward output; another D moves only dq and dk, linearly:
    # dq_i changes by -scale (D'_i - D_i) sum_j P_ij (1 - t_ij^2) k_j
    B, Hq, Hkv, L, d = 1, 2, 1, 128, 32
    q = workloads.normal_bf16((B, Hq, L, d), 81)
    k = workloads.normal_bf16((B, Hkv, L, d), 82)
    v = workloads.normal_bf16((B, Hkv, L, d), 83)
    g = workloads.normal_bf16((B, Hq, L, d), 84)
    spec = MaskSpec(True, 40, -1)
    O, _ = oracle.attention(q, k, v, spec, 0.2, 5.0)
    exact = oracle.attention_bwd(q, k, v, g, spec, 0.2, 5.0)
    given = oracle.attention_bwd(q, k, v, g, spec, 0.2, 5.0, delta=np.sum(g.double().numpy() * O, axis=-1))
    for name in ("dq", "dk", "dv", "delta"):
        np.testing.assert_allclose(given[name], exact[name], rtol=1e-11, atol=1e-12)
    shift = np.random.default_rng(5).normal(size=(B, Hq, L))
    moved = oracle.attention_bwd(q, k, v, g, spec, 0.2, 5.0, delta=exact["delta"] + shift)
    unit = oracle.attention_bwd(q, k, v, torch.zeros_like(g), spec, 0.2, 5.0, delta=np.ones((B, Hq, L)))
    np.testing.assert_array_equal(moved["dv"], exact["dv"])
    np.testing.assert_allclose(moved["dq"], exact["dq"] + shift[..., None] * unit["dq"], rtol=1e-9, atol=1e-11)
