"""block_sparse_flash_gb300 -- Python binding of libsplash.so, the sm_103a
block-sparse (Splash) masked attention forward library.

This module only marshals arguments: torch tensors become device pointers,
the current torch stream becomes the cudaStream_t.  Every step of the
computation runs in the library's CUDA kernels; there is no CPU or PyTorch
fallback.  If the library has not been built, importing works but every call
raises SplashLibraryMissing.

    spec = MaskSpec(causal=True, window_left=4095)
    mi = build_mask_info(spec, L, L, 128, 128)
    out, lse = attention_fwd(q, k, v, mi, scale=1 / 128 ** 0.5, softcap=30.0)

C ABI: include/splash.h.
"""
import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libsplash.so")

SPLASH_OK = 0
_STATUS = {
    0: "SPLASH_OK", 1: "SPLASH_ERR_INVALID_ARG", 2: "SPLASH_ERR_SHAPE", 3: "SPLASH_ERR_UNSUPPORTED",
    4: "SPLASH_ERR_CUDA", 5: "SPLASH_ERR_DEVICE_TIMEOUT", 6: "SPLASH_ERR_OOM", 7: "SPLASH_ERR_DEVICE_CHECK",
}


class SplashLibraryMissing(RuntimeError):
    pass


class SplashError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__(f"{what}: {_status_string(status)}")


class _Spec(ctypes.Structure):
    _fields_ = [
        ("causal", ctypes.c_int32),
        ("window_left", ctypes.c_int64),
        ("window_right", ctypes.c_int64),
        ("q_segment_ids", ctypes.c_void_p),
        ("kv_segment_ids", ctypes.c_void_p),
        ("batch", ctypes.c_int32),
    ]


_lib = None


def lib():
    """The loaded libsplash.so (ctypes.CDLL); raises SplashLibraryMissing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise SplashLibraryMissing(
            f"{LIB_PATH} is missing: build it with block_sparse_flash_gb300.build.build() "
            "(there is no fallback implementation)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    P = ctypes.POINTER
    L.splash_build_mask_info.argtypes = [P(_Spec), i64, i64, i32, i32, vp, P(vp)]
    L.splash_mask_info_rebuild.argtypes = [vp, P(_Spec), i64, i64, i32, i32, vp]
    L.splash_mask_info_shape.argtypes = [vp, P(i32), P(i64), P(i64), P(i32), P(i32)]
    L.splash_mask_info_counts.argtypes = [vp, P(i64), P(i64), P(i64), P(i64)]
    L.splash_mask_info_to_host.argtypes = [vp] + [vp] * 8
    L.splash_mask_info_destroy.argtypes = [vp]
    L.splash_mask_info_destroy.restype = None
    L.splash_attention_fwd.argtypes = [vp, vp, vp, i32, i32, i32, i64, i64, i32, i32, vp, vp, vp, f32, f32,
                                       vp, vp, vp]
    L.splash_attention_fwd_split.argtypes = [vp, vp, vp, i32, i32, i32, i64, i64, i32, i32, vp, vp, vp, f32, f32,
                                             i32, vp, vp, vp]
    L.splash_attention_fwd_mle.argtypes = [vp, vp, vp, i32, i32, i32, i64, i64, i32, i32, vp, vp, vp, f32, f32,
                                           f32, vp, vp, vp]
    L.splash_attention_bwd_workspace_size.argtypes = [i32, i32, i64, i32, P(ctypes.c_size_t)]
    L.splash_attention_bwd.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i64, i64, i32, i32, vp, vp, vp,
                                       f32, f32, vp, vp, vp, vp, ctypes.c_size_t, vp]
    L.splash_mask_info_set_pattern_source.argtypes = [vp, i32]
    L.splash_attention_fwd_host.argtypes = [vp, vp, vp, i32, i32, i32, i64, i64, i32, i32, vp, vp, vp, f32, f32,
                                            vp, vp, vp, vp, vp, vp, vp, vp]
    L.splash_attention_merge.argtypes = [vp, vp, i32, i64, i32, vp, vp, vp]
    L.splash_last_device_error.argtypes = [vp]
    L.splash_debug_wait_selftest.argtypes = [ctypes.c_uint64, vp]
    L.splash_status_string.argtypes = [ctypes.c_int]
    L.splash_status_string.restype = ctypes.c_char_p
    L.splash_version.argtypes = []
    L.splash_version.restype = ctypes.c_char_p
    L.splash_shard_items.argtypes = [i32, i32, i32, i32, P(i64), P(i64)]
    L.splash_kernel_launches.argtypes = []
    L.splash_kernel_launches.restype = ctypes.c_uint64
    for f in (L.splash_build_mask_info, L.splash_mask_info_rebuild, L.splash_mask_info_shape,
              L.splash_mask_info_counts, L.splash_mask_info_to_host, L.splash_attention_fwd,
              L.splash_attention_fwd_split, L.splash_attention_merge,
              L.splash_last_device_error, L.splash_debug_wait_selftest, L.splash_shard_items):
        f.restype = ctypes.c_int
    _lib = L
    return L


def _status_string(s):
    try:
        return lib().splash_status_string(int(s)).decode()
    except SplashLibraryMissing:
        return _STATUS.get(int(s), f"status {s}")


def _check(status, what):
    if status != SPLASH_OK:
        raise SplashError(status, what)


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


@dataclass
class MaskSpec:
    """Joint mask = causal AND window AND segment equality (splash_mask_spec).

    window_left / window_right: inclusive distances, -1 = unbounded.
    q_segment_ids / kv_segment_ids: int32 CUDA tensors [batch, L] (or [L]) or None.
    """
    causal: bool = False
    window_left: int = -1
    window_right: int = -1
    q_segment_ids: Optional[torch.Tensor] = None
    kv_segment_ids: Optional[torch.Tensor] = None

    def _c(self):
        qs, kvs, batch = self.q_segment_ids, self.kv_segment_ids, 0
        for t in (qs, kvs):
            if t is not None and (t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous()):
                raise ValueError("segment ids must be contiguous int32 CUDA tensors")
        if qs is not None:
            batch = 1 if qs.dim() == 1 else qs.shape[0]
        return _Spec(int(bool(self.causal)), int(self.window_left), int(self.window_right),
                     qs.data_ptr() if qs is not None else None,
                     kvs.data_ptr() if kvs is not None else None, batch)


class MaskInfo:
    """Owner of a splash_mask_info handle (device memory freed on close)."""

    def __init__(self, handle):
        self._h = ctypes.c_void_p(handle)

    @property
    def handle(self):
        if not self._h:
            raise ValueError("MaskInfo is closed")
        return self._h

    def close(self):
        if self._h:
            lib().splash_mask_info_destroy(self._h)
            self._h = ctypes.c_void_p(0)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def rebuild(self, spec: MaskSpec, Lq, Lk, bq, bk, stream=None):
        s = spec._c()
        _check(lib().splash_mask_info_rebuild(self.handle, ctypes.byref(s), Lq, Lk, bq, bk, _stream(stream)),
               "splash_mask_info_rebuild")
        return self

    def shape(self):
        bm, bq, bk = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        nq, nk = ctypes.c_int64(), ctypes.c_int64()
        _check(lib().splash_mask_info_shape(self.handle, ctypes.byref(bm), ctypes.byref(nq), ctypes.byref(nk),
                                            ctypes.byref(bq), ctypes.byref(bk)), "splash_mask_info_shape")
        return dict(batch_rows=bm.value, nq=nq.value, nk=nk.value, bq=bq.value, bk=bk.value)

    def set_pattern_source(self, source: str):
        """'stored' (default) or 'positions': the forward computes partial
        blocks' masks from positions, and for a table built with segment IDs
        from the segment arrays, which every forward call must then pass."""
        code = {"stored": 0, "positions": 1}[source]
        _check(lib().splash_mask_info_set_pattern_source(self.handle, code), "splash_mask_info_set_pattern_source")

    def counts(self):
        a, p, n, u = (ctypes.c_int64() for _ in range(4))
        _check(lib().splash_mask_info_counts(self.handle, ctypes.byref(a), ctypes.byref(p), ctypes.byref(n),
                                             ctypes.byref(u)), "splash_mask_info_counts")
        return dict(num_active=a.value, num_partial=p.value, num_patterns=n.value, allowed_pairs=u.value)

    def to_host(self):
        """All table arrays as numpy arrays (synchronous copy)."""
        sh, c = self.shape(), self.counts()
        R, A, P = sh["batch_rows"] * sh["nq"], c["num_active"], c["num_patterns"]
        out = dict(
            block_mask=np.zeros((sh["batch_rows"], sh["nq"], sh["nk"]), dtype=np.int8),
            row_ptr=np.zeros(R + 1, dtype=np.int32),
            active_rows=np.zeros(max(A, 1), dtype=np.int32),
            active_cols=np.zeros(max(A, 1), dtype=np.int32),
            mask_next=np.zeros(max(A, 1), dtype=np.int32),
            bounds_start=np.zeros(max(A, 1), dtype=np.uint8),
            bounds_end=np.zeros(max(A, 1), dtype=np.uint8),
            partial_mask_blocks=np.zeros((max(P, 1), sh["bq"], sh["bk"]), dtype=np.uint8),
        )
        order = ["block_mask", "row_ptr", "active_rows", "active_cols", "mask_next", "bounds_start",
                 "bounds_end", "partial_mask_blocks"]
        _check(lib().splash_mask_info_to_host(self.handle, *[out[k].ctypes.data for k in order]),
               "splash_mask_info_to_host")
        for k in ("active_rows", "active_cols", "mask_next", "bounds_start", "bounds_end"):
            out[k] = out[k][:A]
        out["partial_mask_blocks"] = out["partial_mask_blocks"][:P]
        out.update(c)
        out.update(sh)
        return out


def build_mask_info(spec: MaskSpec, Lq: int, Lk: int, bq: int, bk: int, stream=None) -> MaskInfo:
    """The sparse execution table of `spec` on a (Lq, Lk) grid of bq x bk
    blocks (splash_build_mask_info): bk in {64, 128}, bq in {64, 128, 256}.
    The forward takes bq == bk, or bq = 256 with bk = 128 (each 256-row
    q-block computed as two 128-row tiles of one head sharing every K/V tile,
    the faster choice for MHA); the backward takes 128 x 128."""
    h = ctypes.c_void_p()
    s = spec._c()
    _check(lib().splash_build_mask_info(ctypes.byref(s), Lq, Lk, bq, bk, _stream(stream), ctypes.byref(h)),
           "splash_build_mask_info")
    return MaskInfo(h.value)


def _qkv_shapes(q, k, v):
    for t in (q, k, v):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError("q, k, v must be contiguous 4-D bf16 CUDA tensors")
    B, Hq, Lq, dqk = q.shape
    return B, Hq, Lq, dqk, k.shape[1], k.shape[2], v.shape[3]


def attention_fwd(q, k, v, mask_info: MaskInfo, scale: float, softcap: float = 0.0, q_segment_ids=None,
                  kv_segment_ids=None, out=None, lse=None, stream=None, num_splits: int = 1,
                  max_logit=None):
    """out [B, Hq, Lq, dv] bf16 and lse [B, Hq, Lq] fp32 (allocated if not given).

    num_splits > 1 runs the split-KV forward into fp32 workspace allocated
    here, then the LSE merge (same result).  max_logit = c runs the Max Logit
    Estimate variant (the softmax reference fixed at c; same result while c
    is in the safe range, e.g. c = softcap)."""
    B, Hq, Lq, dqk, Hkv, Lk, dv = _qkv_shapes(q, k, v)
    if out is None:
        out = torch.empty((B, Hq, Lq, dv), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device)
    if max_logit is not None:
        if num_splits > 1:
            raise ValueError("max_logit is supported by the one-pass forward only (num_splits == 1)")
        _check(lib().splash_attention_fwd_mle(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Lq, Lk, dqk, dv,
                                              _ptr(q_segment_ids), _ptr(kv_segment_ids), mask_info.handle,
                                              float(scale), float(softcap), float(max_logit), _ptr(out),
                                              _ptr(lse), _stream(stream)),
               "splash_attention_fwd_mle")
        return out, lse
    if num_splits > 1:
        o_part, lse_part = attention_fwd_split(q, k, v, mask_info, scale, softcap, num_splits, q_segment_ids,
                                               kv_segment_ids, stream=stream)
        return attention_merge(o_part, lse_part, out=out, lse=lse, stream=stream)
    _check(lib().splash_attention_fwd(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Lq, Lk, dqk, dv,
                                      _ptr(q_segment_ids), _ptr(kv_segment_ids), mask_info.handle,
                                      float(scale), float(softcap), _ptr(out), _ptr(lse), _stream(stream)),
           "splash_attention_fwd")
    return out, lse


def attention_fwd_host(q_host, k_host, v_host, mask_info: MaskInfo, scale: float, softcap: float = 0.0,
                       out_host=None, lse_host=None, q=None, k=None, v=None, out=None, lse=None,
                       q_segment_ids=None, kv_segment_ids=None, stream=None):
    """attention_fwd for CPU tensors (pinned for overlap): copies in, computes
    and copies out, pipelined in chunks.  Device buffers q, k, v, out, lse are
    allocated on the current device when not given.  Returns (out_host,
    lse_host); they are complete once the stream has reached this point."""
    for t in (q_host, k_host, v_host):
        if t.dtype != torch.bfloat16 or t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError("q_host, k_host, v_host must be contiguous 4-D bf16 CPU tensors")
    B, Hq, Lq, dqk = q_host.shape
    Hkv, Lk, dv = k_host.shape[1], k_host.shape[2], v_host.shape[3]
    dev = torch.device("cuda", torch.cuda.current_device())
    if out_host is None:
        out_host = torch.empty((B, Hq, Lq, dv), dtype=torch.bfloat16).pin_memory()
    if lse_host is None:
        lse_host = torch.empty((B, Hq, Lq), dtype=torch.float32).pin_memory()
    q = torch.empty_like(q_host, device=dev) if q is None else q
    k = torch.empty_like(k_host, device=dev) if k is None else k
    v = torch.empty_like(v_host, device=dev) if v is None else v
    out = torch.empty((B, Hq, Lq, dv), dtype=torch.bfloat16, device=dev) if out is None else out
    lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=dev) if lse is None else lse
    _check(lib().splash_attention_fwd_host(_ptr(q_host), _ptr(k_host), _ptr(v_host), B, Hq, Hkv, Lq, Lk, dqk, dv,
                                           _ptr(q_segment_ids), _ptr(kv_segment_ids), mask_info.handle,
                                           float(scale), float(softcap), _ptr(out_host), _ptr(lse_host), _ptr(q),
                                           _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _stream(stream)),
           "splash_attention_fwd_host")
    return out_host, lse_host


def attention_fwd_split(q, k, v, mask_info: MaskInfo, scale: float, softcap: float, num_splits: int,
                        q_segment_ids=None, kv_segment_ids=None, o_part=None, lse_part=None, stream=None):
    """Split-KV partials: o_part [S, B, Hq, Lq, dv] fp32 and lse_part [S, B, Hq, Lq] fp32."""
    B, Hq, Lq, dqk, Hkv, Lk, dv = _qkv_shapes(q, k, v)
    if o_part is None:
        o_part = torch.empty((num_splits, B, Hq, Lq, dv), dtype=torch.float32, device=q.device)
    if lse_part is None:
        lse_part = torch.empty((num_splits, B, Hq, Lq), dtype=torch.float32, device=q.device)
    _check(lib().splash_attention_fwd_split(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Lq, Lk, dqk, dv,
                                            _ptr(q_segment_ids), _ptr(kv_segment_ids), mask_info.handle,
                                            float(scale), float(softcap), int(num_splits), _ptr(o_part),
                                            _ptr(lse_part), _stream(stream)),
           "splash_attention_fwd_split")
    return o_part, lse_part


def attention_merge(o_part, lse_part, out=None, lse=None, stream=None):
    """Merges split-KV partials [S, ..., dv] / [S, ...] into bf16 out [..., dv] and fp32 lse [...]."""
    if o_part.dtype != torch.float32 or lse_part.dtype != torch.float32 or not o_part.is_contiguous() \
            or not lse_part.is_contiguous():
        raise ValueError("o_part and lse_part must be contiguous fp32 tensors")
    S, dv = o_part.shape[0], o_part.shape[-1]
    rows = lse_part[0].numel()
    if out is None:
        out = torch.empty(o_part.shape[1:], dtype=torch.bfloat16, device=o_part.device)
    if lse is None:
        lse = torch.empty(lse_part.shape[1:], dtype=torch.float32, device=o_part.device)
    _check(lib().splash_attention_merge(_ptr(o_part), _ptr(lse_part), int(S), int(rows), int(dv), _ptr(out),
                                        _ptr(lse), _stream(stream)), "splash_attention_merge")
    return out, lse


def attention_bwd(q, k, v, out, lse, dout, mask_info: MaskInfo, scale: float, softcap: float = 0.0,
                  q_segment_ids=None, kv_segment_ids=None, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Gradients (dq, dk, dv) of attention_fwd for the upstream gradient dout,
    from the forward's out and lse (bf16 tensors shaped like q, k, v; allocated
    if not given).  workspace: optional uint8 device tensor of at least
    attention_bwd_workspace_size(...) bytes."""
    B, Hq, Lq, dqk, Hkv, Lk, dvd = _qkv_shapes(q, k, v)
    for name, t, shape, dt in (("out", out, (B, Hq, Lq, dvd), torch.bfloat16),
                               ("dout", dout, (B, Hq, Lq, dvd), torch.bfloat16),
                               ("lse", lse, (B, Hq, Lq), torch.float32)):
        if tuple(t.shape) != shape or t.dtype != dt or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous {dt} tensor of shape {shape}")
    if dq is None:
        dq = torch.empty_like(q)
    if dk is None:
        dk = torch.empty_like(k)
    if dv is None:
        dv = torch.empty_like(v)
    need = attention_bwd_workspace_size(B, Hq, Lq, dqk)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(lib().splash_attention_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), B, Hq, Hkv,
                                      Lq, Lk, dqk, dvd, _ptr(q_segment_ids), _ptr(kv_segment_ids),
                                      mask_info.handle, float(scale), float(softcap), _ptr(dq), _ptr(dk), _ptr(dv),
                                      _ptr(workspace), int(workspace.numel() * workspace.element_size()),
                                      _stream(stream)),
           "splash_attention_bwd")
    return dq, dk, dv


def attention_bwd_workspace_size(B: int, Hq: int, Lq: int, dqk: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().splash_attention_bwd_workspace_size(int(B), int(Hq), int(Lq), int(dqk), ctypes.byref(n)),
           "splash_attention_bwd_workspace_size")
    return int(n.value)


def shard_items(B: int, Hkv: int, world: int, rank: int):
    """This rank's half-open range [begin, end) of the B * Hkv (batch, KV
    head) groups when a workload is split across `world` GPUs
    (splash_shard_items)."""
    b, e = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().splash_shard_items(int(B), int(Hkv), int(world), int(rank), ctypes.byref(b), ctypes.byref(e)),
           "splash_shard_items")
    return b.value, e.value


def shard_views(q, k, v, begin: int, end: int, out=None, lse=None, segment_ids=None):
    """Sub-tensors of groups [begin, end) as a problem of (end - begin) batch
    rows, Hq / Hkv query heads and one KV head: views of q [B, Hq, L, dqk],
    k, v, out and lse (no copy), and with segment IDs [B, L] a per-group copy
    of the rows they read (row g // Hkv for group g).  Returns a dict with
    the same keys."""
    B, Hq, Lq, dqk = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    r = dict(q=q.view(B * Hkv, G, Lq, dqk)[begin:end],
             k=k.view(B * Hkv, 1, k.shape[2], k.shape[3])[begin:end],
             v=v.view(B * Hkv, 1, v.shape[2], v.shape[3])[begin:end])
    if out is not None:
        r["out"] = out.view(B * Hkv, G, Lq, out.shape[3])[begin:end]
    if lse is not None:
        r["lse"] = lse.view(B * Hkv, G, Lq)[begin:end]
    if segment_ids is not None:
        idx = torch.arange(begin, end, device=segment_ids.device) // Hkv
        r["segment_ids"] = segment_ids.index_select(0, idx).contiguous()
    return r


def last_device_error(stream=None) -> int:
    """Synchronises and returns (and clears) the device error status code."""
    return lib().splash_last_device_error(_stream(stream))


def check_device_error(stream=None):
    _check(last_device_error(stream), "device")


def debug_wait_selftest(timeout_ns: int, stream=None) -> int:
    return lib().splash_debug_wait_selftest(int(timeout_ns), _stream(stream))


def kernel_launches() -> int:
    """Kernels launched by the library in this process so far."""
    return int(lib().splash_kernel_launches())


def version() -> str:
    return lib().splash_version().decode()
