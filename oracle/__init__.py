"""The oracle: a plain, slow, obviously correct CPU implementation of
block-sparse masked attention (forward and backward) and of its sparse
execution table.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
CPU-baseline / reference legs of bench.py may import this package.  It
shares no code with block_sparse_flash_gb300 (the CUDA library) and never
imports it; inputs reach it as numpy arrays.

The arithmetic lives in splash_oracle.c (f64, brute force); this module
only marshals numpy arrays through ctypes.  Source passages are cited in
the C file:
  "Pallas Kernels and Splash Attention" (CMU 11-868 Lecture 13 notes)
  §5.1-§5.4 (softmax, Flash body, soft cap) and §6.1-§6.4 (MaskInfo,
  segment IDs, joint masks); "The maths and infra behind core LLM
  operations" (joto.ai), sections "Causal Mask" and "LSE and Online
  Softmax".
"""
import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import numpy as np

from . import build as _build
from .softmax_ref import (exp_limits, merge, mle_safe_range, mle_softmax, online_softmax_trace,  # noqa: F401
                          partial_state, safe_softmax)

_lib = None


class _Spec(ctypes.Structure):
    _fields_ = [
        ("causal", ctypes.c_int32),
        ("window_left", ctypes.c_int64),
        ("window_right", ctypes.c_int64),
        ("q_seg", ctypes.c_void_p),
        ("kv_seg", ctypes.c_void_p),
        ("batch", ctypes.c_int32),
    ]


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        i64, vp, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        L.oracle_mask_classify.argtypes = [ctypes.POINTER(_Spec), i64, i64, i64, i64, i32, vp,
                                           ctypes.POINTER(i64), ctypes.POINTER(i64), ctypes.POINTER(i64)]
        L.oracle_mask_table.argtypes = [ctypes.POINTER(_Spec), i64, i64, i64, i64, vp, vp, vp, vp,
                                        vp, vp, vp, vp, i64, ctypes.POINTER(i64)]
        L.oracle_attention.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, i64,
                                       ctypes.POINTER(_Spec), ctypes.c_double, ctypes.c_double,
                                       vp, i64, i32, vp, vp]
        L.oracle_allowed.argtypes = [ctypes.POINTER(_Spec), i64, i64, i64, i64, i64]
        L.oracle_attention_bwd_head.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64,
                                                ctypes.POINTER(_Spec), ctypes.c_double, ctypes.c_double,
                                                i32, vp, vp, vp, vp, vp]
        for f in (L.oracle_mask_classify, L.oracle_mask_table, L.oracle_attention, L.oracle_allowed,
                  L.oracle_attention_bwd_head):
            f.restype = ctypes.c_int
        _lib = L
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


@dataclass
class MaskSpec:
    """The joint mask: causal AND local window AND segment equality.

    window_left / window_right are inclusive distances (query i may see key
    j when i - j <= window_left and j - i <= window_right); -1 is unbounded.
    q_segment_ids / kv_segment_ids are int32 arrays [batch, L] or None.
    """
    causal: bool = False
    window_left: int = -1
    window_right: int = -1
    q_segment_ids: Optional[np.ndarray] = None
    kv_segment_ids: Optional[np.ndarray] = None

    def _c(self):
        keep = []
        qs = kvs = None
        batch = 0
        if self.q_segment_ids is not None:
            qs = np.ascontiguousarray(self.q_segment_ids, dtype=np.int32)
            kv = self.kv_segment_ids if self.kv_segment_ids is not None else self.q_segment_ids
            kvs = np.ascontiguousarray(kv, dtype=np.int32)
            if qs.ndim == 1:
                qs = qs[None]
            if kvs.ndim == 1:
                kvs = kvs[None]
            batch = qs.shape[0]
            keep = [qs, kvs]
        s = _Spec(int(bool(self.causal)), int(self.window_left), int(self.window_right),
                  qs.ctypes.data if qs is not None else None,
                  kvs.ctypes.data if kvs is not None else None, batch)
        return s, keep

    @property
    def batch_rows(self) -> int:
        if self.q_segment_ids is None:
            return 1
        a = np.asarray(self.q_segment_ids)
        return 1 if a.ndim == 1 else a.shape[0]


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def allowed(spec: MaskSpec, b, Lq, Lk, i, j) -> bool:
    s, keep = spec._c()
    return bool(lib().oracle_allowed(ctypes.byref(s), b, Lq, Lk, i, j))


@dataclass
class MaskInfo:
    """The sparse execution table, as the oracle builds it."""
    batch_rows: int
    nq: int
    nk: int
    bq: int
    bk: int
    block_mask: np.ndarray          # int8 [batch_rows, nq, nk]: 0 empty, 1 partial, 2 full
    row_ptr: np.ndarray             # int32 [batch_rows*nq + 1]
    active_rows: np.ndarray         # int32 [A]  (q-block index within its batch row)
    active_cols: np.ndarray         # int32 [A]  (kv-block index)
    mask_next: np.ndarray           # int32 [A]  (pattern index, -1 for full blocks)
    bounds_start: np.ndarray        # uint8 [A]
    bounds_end: np.ndarray          # uint8 [A]
    partial_mask_blocks: np.ndarray  # uint8 [P, bq, bk]
    allowed_pairs: int              # allowed (query, key) pairs over the batch rows

    @property
    def num_active(self):
        return int(self.active_cols.shape[0])

    @property
    def num_partial(self):
        return int(np.count_nonzero(self.mask_next >= 0))

    @property
    def num_patterns(self):
        return int(self.partial_mask_blocks.shape[0])


def mask_info(spec: MaskSpec, Lq: int, Lk: int, bq: int, bk: int, nthreads: int = 0) -> MaskInfo:
    """Builds MaskInfo by brute-force classification of every element.  When
    Lq or Lk is not a multiple of the block, the grid is padded to whole blocks
    and padding positions are masked."""
    L = lib()
    s, keep = spec._c()
    nbm = spec.batch_rows
    nq, nk = -(-Lq // bq), -(-Lk // bk)  # padded grid: the last blocks may be ragged
    bm = np.zeros((nbm, nq, nk), dtype=np.int8)
    A, Ap, npairs = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _check(L.oracle_mask_classify(ctypes.byref(s), Lq, Lk, bq, bk, nthreads or default_threads(),
                                  bm.ctypes.data, ctypes.byref(A), ctypes.byref(Ap),
                                  ctypes.byref(npairs)), "classify")
    a, ap = A.value, Ap.value
    row_ptr = np.zeros(nbm * nq + 1, dtype=np.int32)
    rows = np.zeros(max(a, 1), dtype=np.int32)
    cols = np.zeros(max(a, 1), dtype=np.int32)
    nxt = np.zeros(max(a, 1), dtype=np.int32)
    bs = np.zeros(max(a, 1), dtype=np.uint8)
    be = np.zeros(max(a, 1), dtype=np.uint8)
    pats = np.zeros((max(ap, 1), bq, bk), dtype=np.uint8)
    P = ctypes.c_int64()
    _check(L.oracle_mask_table(ctypes.byref(s), Lq, Lk, bq, bk, bm.ctypes.data, row_ptr.ctypes.data,
                               rows.ctypes.data, cols.ctypes.data, nxt.ctypes.data, bs.ctypes.data,
                               be.ctypes.data, pats.ctypes.data, ap, ctypes.byref(P)), "table")
    return MaskInfo(nbm, nq, nk, bq, bk, bm, row_ptr, rows[:a].copy(), cols[:a].copy(),
                    nxt[:a].copy(), bs[:a].copy(), be[:a].copy(), pats[:P.value].copy(),
                    int(npairs.value))


def _bits(x) -> np.ndarray:
    """bf16 data as uint16 bit patterns (accepts uint16 / int16 numpy arrays
    or torch bf16 CPU tensors)."""
    if hasattr(x, "dtype") and str(x.dtype) == "torch.bfloat16":
        import torch  # torch CPU only: a bit-level view of the caller's tensor
        return x.contiguous().view(torch.int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(x)
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError("oracle.attention wants bf16 bit patterns (uint16) or torch bf16 tensors")
    return a


def attention(q, k, v, spec: MaskSpec, scale: float, softcap: float = 0.0, rows=None,
              nthreads: int = 0):
    """Forward attention in f64.

    q [B, Hq, Lq, dqk], k [B, Hkv, Lk, dqk], v [B, Hkv, Lk, dv] as bf16 bits.
    rows: optional int64 array of flat query rows (b*Hq + h)*Lq + i.
    Returns (O, LSE): O f64 [nrows, dv] (or [B, Hq, Lq, dv] when rows is None),
    LSE f64 [nrows] (or [B, Hq, Lq]); fully masked rows give O = 0, LSE = -inf.
    """
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    B, Hq, Lq, dqk = qb.shape
    _, Hkv, Lk, _ = kb.shape
    dv = vb.shape[3]
    s, keep = spec._c()
    if rows is None:
        n = B * Hq * Lq
        rptr = None
    else:
        rws = np.ascontiguousarray(rows, dtype=np.int64)
        n = rws.shape[0]
        rptr = rws.ctypes.data
    out = np.zeros((max(n, 1), dv), dtype=np.float64)
    lse = np.zeros(max(n, 1), dtype=np.float64)
    _check(lib().oracle_attention(qb.ctypes.data, kb.ctypes.data, vb.ctypes.data, B, Hq, Hkv, Lq, Lk,
                                  dqk, dv, ctypes.byref(s), float(scale), float(softcap), rptr, n,
                                  nthreads or default_threads(), out.ctypes.data, lse.ctypes.data),
           "attention")
    out, lse = out[:n], lse[:n]
    if rows is None:
        return out.reshape(B, Hq, Lq, dv), lse.reshape(B, Hq, Lq)
    return out, lse


def _f64(x) -> np.ndarray:
    """float64 copy of a torch tensor (bf16 widens exactly) or an array."""
    if hasattr(x, "dtype") and str(x.dtype).startswith("torch."):
        import torch  # torch CPU only: widening the caller's tensor
        return np.ascontiguousarray(x.detach().to(torch.float64).cpu().numpy())
    return np.ascontiguousarray(x, dtype=np.float64)


def attention_bwd(q, k, v, dout, spec: MaskSpec, scale: float, softcap: float = 0.0, heads=None,
                  nthreads: int = 0, delta=None):
    """Backward attention in f64 (gradients of the forward with respect to q,
    k and v for the upstream gradient dout).

    q [B, Hq, Lq, dqk], k [B, Hkv, Lk, dqk], v [B, Hkv, Lk, dv],
    dout [B, Hq, Lq, dv]: torch tensors (bf16 widens exactly) or float64
    arrays.  delta (optional, [B, Hq, Lq]): D_i to use instead of the exact
    sum_j P_ij dP_ij (for instance dout_i . out_i of a stored output).  heads:
    optional list of (b, h) pairs; only those query heads are differentiated
    (dq of the others stays 0 and dk / dv then hold the listed heads'
    contributions).  Returns dict(dq, dk, dv, lse, delta) of f64 arrays shaped
    like q, k, v, [B, Hq, Lq], [B, Hq, Lq]."""
    qf, kf, vf, gf = _f64(q), _f64(k), _f64(v), _f64(dout)
    df = _f64(delta) if delta is not None else None
    B, Hq, Lq, dqk = qf.shape
    _, Hkv, Lk, _ = kf.shape
    dv = vf.shape[3]
    if Hq % Hkv or gf.shape != (B, Hq, Lq, dv):
        raise ValueError("shape mismatch")
    G = Hq // Hkv
    s, keep = spec._c()
    dq = np.zeros_like(qf)
    dk = np.zeros_like(kf)
    dvv = np.zeros_like(vf)
    lse = np.full((B, Hq, Lq), -np.inf)
    delta = np.zeros((B, Hq, Lq))
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(Hq)]
    tdk = np.zeros((Lk, dqk))
    tdv = np.zeros((Lk, dv))
    for b, h in heads:
        g = h // G
        qh, gh = np.ascontiguousarray(qf[b, h]), np.ascontiguousarray(gf[b, h])
        dh_in = np.ascontiguousarray(df[b, h]) if df is not None else None
        kh, vh = np.ascontiguousarray(kf[b, g]), np.ascontiguousarray(vf[b, g])
        dqh = np.zeros((Lq, dqk))
        lh = np.zeros(Lq)
        dh = np.zeros(Lq)
        _check(lib().oracle_attention_bwd_head(qh.ctypes.data, kh.ctypes.data, vh.ctypes.data, gh.ctypes.data,
                                               dh_in.ctypes.data if dh_in is not None else None, b, Lq, Lk, dqk, dv, ctypes.byref(s), float(scale), float(softcap),
                                               nthreads or default_threads(), dqh.ctypes.data, tdk.ctypes.data,
                                               tdv.ctypes.data, lh.ctypes.data, dh.ctypes.data),
               "attention_bwd")
        dq[b, h] = dqh
        dk[b, g] += tdk
        dvv[b, g] += tdv
        lse[b, h] = lh
        delta[b, h] = dh
    return dict(dq=dq, dk=dk, dv=dvv, lse=lse, delta=delta)
