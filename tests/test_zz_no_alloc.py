"""The allocation-free classification entry point (splash_classify_blocks_noalloc),
called through the C ABI, must agree with the regular MaskInfo build.

It serves callers that may not allocate device memory themselves (their device
memory belongs to a pool allocator with a fixed budget); its working memory is a
fixed array inside the library.  Two calls run back to back, on different
masks, so that a counter left over from the previous call would show up.
This file is collected last on purpose."""
import ctypes

import numpy as np
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


def noalloc(bsf, spec, Lq, Lk, bq, bk):
    lib = bsf.lib()
    f = lib.splash_classify_blocks_noalloc
    f.argtypes = [ctypes.POINTER(bsf._Spec), ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    rows = 1 if spec.q_segment_ids is None else spec.q_segment_ids.shape[0]
    # ragged lengths are padded to whole blocks
    block_mask = torch.full((rows, -(-Lq // bq), -(-Lk // bk)), -1, dtype=torch.int8, device="cuda")
    totals = np.zeros(4, dtype=np.int64)
    s = spec._c()
    status = f(ctypes.byref(s), Lq, Lk, bq, bk, ctypes.c_void_p(block_mask.data_ptr()),
               ctypes.c_void_p(totals.ctypes.data), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert status == 0, bsf._status_string(status)
    return block_mask.cpu().numpy(), totals


def regular(bsf, spec, Lq, Lk, bq, bk):
    mi = bsf.build_mask_info(spec, Lq, Lk, bq, bk)
    h = mi.to_host()
    mi.close()
    row_counts = np.diff(h["row_ptr"])
    return h["block_mask"], [h["num_active"], h["num_partial"], h["allowed_pairs"], int(row_counts.max())]


def test_noalloc_matches_regular_build_on_consecutive_calls(bsf):
    lens = workloads.document_lengths(8192, 4242, mean=700, lo=64, hi=3000, batch_rows=2)
    seg = workloads.segment_ids_from_lengths(lens).cuda()
    cases = [
        (bsf.MaskSpec(True), 4096, 4096, 128, 128),
        (bsf.MaskSpec(True, 1023, 0, seg, seg), 8192, 8192, 64, 64),
        (bsf.MaskSpec(True), 4096, 4096, 128, 128),
    ]
    for spec, Lq, Lk, bq, bk in cases:
        got_mask, got_tot = noalloc(bsf, spec, Lq, Lk, bq, bk)
        ref_mask, ref_tot = regular(bsf, spec, Lq, Lk, bq, bk)
        np.testing.assert_array_equal(got_mask, ref_mask)
        assert got_tot.tolist() == ref_tot


def test_noalloc_ragged_segments_and_tall_query_blocks(bsf):
    # ragged lengths (padded grid) with document segments, then 256-row
    # q-blocks under a plain causal mask, back to back
    lens = workloads.document_lengths(8000, 4343, mean=500, lo=64, hi=2000, batch_rows=2)
    seg = workloads.segment_ids_from_lengths(lens).cuda()
    cases = [
        (bsf.MaskSpec(True, -1, -1, seg, seg), 8000, 8000, 128, 128),
        (bsf.MaskSpec(True), 4096, 4096, 256, 128),
        (bsf.MaskSpec(True, 700, 0, seg, seg), 8000, 8000, 64, 64),
    ]
    for spec, Lq, Lk, bq, bk in cases:
        got_mask, got_tot = noalloc(bsf, spec, Lq, Lk, bq, bk)
        ref_mask, ref_tot = regular(bsf, spec, Lq, Lk, bq, bk)
        np.testing.assert_array_equal(got_mask, ref_mask)
        assert got_tot.tolist() == ref_tot


def test_noalloc_rejects_masks_beyond_its_limit(bsf):
    lib = bsf.lib()
    f = lib.splash_classify_blocks_noalloc
    f.argtypes = [ctypes.POINTER(bsf._Spec), ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    totals = np.zeros(4, dtype=np.int64)
    s = bsf.MaskSpec(True)._c()
    L = 64 * 16385  # 16385 q-blocks of 64: one more than the scratch holds
    dummy = torch.empty(1, dtype=torch.int8, device="cuda")
    status = f(ctypes.byref(s), L, L, 64, 64, ctypes.c_void_p(dummy.data_ptr()),
               ctypes.c_void_p(totals.ctypes.data), ctypes.c_void_p(0))
    assert status == 3  # SPLASH_ERR_UNSUPPORTED, before any launch


def test_noalloc_rejects_too_many_key_blocks(bsf):
    # two batch rows of 8193 key blocks: 16386 columns against a limit of
    # 16384, with a single q-block row
    lib = bsf.lib()
    f = lib.splash_classify_blocks_noalloc
    f.argtypes = [ctypes.POINTER(bsf._Spec), ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    Lq, Lk = 64, 64 * 8193
    sq = torch.zeros((2, Lq), dtype=torch.int32, device="cuda")
    skv = torch.zeros((2, Lk), dtype=torch.int32, device="cuda")
    s = bsf.MaskSpec(False, -1, -1, sq, skv)._c()
    totals = np.zeros(4, dtype=np.int64)
    dummy = torch.empty(1, dtype=torch.int8, device="cuda")
    status = f(ctypes.byref(s), Lq, Lk, 64, 64, ctypes.c_void_p(dummy.data_ptr()),
               ctypes.c_void_p(totals.ctypes.data), ctypes.c_void_p(0))
    assert status == 3  # SPLASH_ERR_UNSUPPORTED, before any launch
