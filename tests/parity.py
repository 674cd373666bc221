"""Shared helpers for GPU-vs-oracle parity checks (used by the -m gpu tests and
by __graft_entry__.smoke()).

Tolerances (bf16 output, fp32 LSE):
  O    max |GPU - oracle| <= 2e-2 over all compared elements, and for every
       compared row ||GPU - oracle||_2 <= 2e-2 * ||oracle||_2;
  LSE  |GPU - oracle| <= 1e-3 where the oracle is finite; rows with no allowed
       key must be -inf on both sides (and O = 0).
"""
import numpy as np
import torch

O_ABS_TOL = 2e-2
O_REL_TOL = 2e-2
LSE_ABS_TOL = 1e-3

# Error triples of the full-size workload checks, by label, printed in the
# test session's summary so that a run's record shows the margins.
MARGINS = {}


def oracle_spec(w_or_spec_kwargs, seg=None):
    import oracle
    return oracle.MaskSpec(**w_or_spec_kwargs, q_segment_ids=seg, kv_segment_ids=seg) if seg is not None \
        else oracle.MaskSpec(**w_or_spec_kwargs)


def compare_rows(out_gpu, lse_gpu, O_ref, lse_ref, label=""):
    """out_gpu [n, dv] (any float tensor/array), lse_gpu [n]; refs f64."""
    o = np.asarray(out_gpu, dtype=np.float64)
    l = np.asarray(lse_gpu, dtype=np.float64)
    masked = np.isneginf(lse_ref)
    assert np.all(np.isneginf(l[masked])), f"{label}: fully masked rows must have lse = -inf"
    assert np.all(o[masked] == 0), f"{label}: fully masked rows must have O = 0"
    keep = ~masked
    err = np.abs(o[keep] - O_ref[keep])
    max_abs = float(err.max()) if err.size else 0.0
    assert np.all(np.isfinite(o[keep])), f"{label}: non-finite O"
    num = np.linalg.norm(o[keep] - O_ref[keep], axis=1)
    den = np.maximum(np.linalg.norm(O_ref[keep], axis=1), 1e-30)
    rel = float((num / den).max()) if num.size else 0.0
    lse_err = float(np.abs(l[keep] - lse_ref[keep]).max()) if keep.any() else 0.0
    assert max_abs <= O_ABS_TOL, f"{label}: O max abs err {max_abs:.3e}"
    assert rel <= O_REL_TOL, f"{label}: O row rel err {rel:.3e}"
    assert lse_err <= LSE_ABS_TOL, f"{label}: LSE abs err {lse_err:.3e}"
    return dict(o_max_abs=max_abs, o_row_rel=rel, lse_max_abs=lse_err)


def sample_rows(B, Hq, Lq, bq, n_random, seed, extra_blocks=()):
    """Flat rows (b*Hq + h)*Lq + i: n_random random rows plus every row of the
    given (b, h, q-block) triples."""
    rng = np.random.default_rng(seed)
    rows = set(int(x) for x in rng.integers(0, B * Hq * Lq, size=n_random))
    for b, h, r in extra_blocks:
        base = (b * Hq + h) * Lq + r * bq
        rows.update(range(base, base + bq))
    return np.array(sorted(rows), dtype=np.int64)


def gather_rows(out, lse, rows):
    """Rows of GPU outputs [B, Hq, Lq, dv] / [B, Hq, Lq] as f64 numpy."""
    dv = out.shape[-1]
    idx = torch.as_tensor(rows, device=out.device)
    o = out.reshape(-1, dv).index_select(0, idx).float().cpu().numpy()
    l = lse.reshape(-1).index_select(0, idx).cpu().numpy()
    return o, l
