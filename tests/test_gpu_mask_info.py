"""MaskInfo built on the GPU must equal the oracle's brute-force table
bit for bit (every array), on the five workloads' masks and on fuzzed masks."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bsf():
    from block_sparse_flash_gb300 import build as b
    b.build()
    import block_sparse_flash_gb300 as m
    return m


def gpu_and_oracle(bsf, causal, wl, wr, seg_q, seg_kv, Lq, Lk, bq, bk):
    q_dev = seg_q.cuda() if seg_q is not None else None
    kv_dev = seg_kv.cuda() if seg_kv is not None else None
    mi = bsf.build_mask_info(bsf.MaskSpec(causal, wl, wr, q_dev, kv_dev), Lq, Lk, bq, bk)
    got = mi.to_host()
    mi.close()
    ref = oracle.mask_info(oracle.MaskSpec(causal, wl, wr,
                                           seg_q.numpy() if seg_q is not None else None,
                                           (seg_kv if seg_kv is not None else seg_q).numpy()
                                           if seg_q is not None else None), Lq, Lk, bq, bk)
    return got, ref


def assert_same(got, ref, label):
    np.testing.assert_array_equal(got["block_mask"], ref.block_mask, err_msg=label)
    np.testing.assert_array_equal(got["row_ptr"], ref.row_ptr, err_msg=label)
    np.testing.assert_array_equal(got["active_rows"], ref.active_rows, err_msg=label)
    np.testing.assert_array_equal(got["active_cols"], ref.active_cols, err_msg=label)
    np.testing.assert_array_equal(got["mask_next"], ref.mask_next, err_msg=label)
    np.testing.assert_array_equal(got["bounds_start"], ref.bounds_start, err_msg=label)
    np.testing.assert_array_equal(got["bounds_end"], ref.bounds_end, err_msg=label)
    np.testing.assert_array_equal(got["partial_mask_blocks"], ref.partial_mask_blocks, err_msg=label)
    assert got["num_active"] == ref.num_active, label
    assert got["num_partial"] == ref.num_partial, label
    assert got["num_patterns"] == ref.num_patterns, label
    assert got["allowed_pairs"] == ref.allowed_pairs, label


@pytest.mark.parametrize("index", [1, 2, 3, 4, 5])
def test_workload_masks_bit_exact(bsf, index):
    w = workloads.workload(index)
    seg = workloads.make_inputs(w, with_values=False).segment_ids
    got, ref = gpu_and_oracle(bsf, w.causal, w.window_left, w.window_right, seg, seg, w.L, w.L, w.bq, w.bk)
    assert_same(got, ref, w.name)


def fuzz_cases():
    rng = np.random.default_rng(1234)
    cases = []
    for n in range(40):
        L = int(rng.choice([128, 256, 512, 1024]))
        bq = int(rng.choice([64, 128]))
        bk = int(rng.choice([64, 128]))
        causal = bool(rng.integers(2))
        wl = int(rng.choice([-1, 0, 1, 63, 64, 100, 300]))
        wr = int(rng.choice([-1, 0, 5, 64, 200]))
        kind = int(rng.integers(4))  # 0 none, 1 sorted docs, 2 non-monotone ids, 3 batch of 2 with q != kv
        cases.append((n, L, bq, bk, causal, wl, wr, kind, int(rng.integers(1 << 30))))
    return cases


@pytest.mark.parametrize("n,L,bq,bk,causal,wl,wr,kind,seed", fuzz_cases())
def test_fuzzed_masks_bit_exact(bsf, n, L, bq, bk, causal, wl, wr, kind, seed):
    seg_q = seg_kv = None
    if kind == 1:
        seg_q = seg_kv = workloads.random_segment_ids(1, L, seed, 6, True)
    elif kind == 2:
        seg_q = seg_kv = workloads.random_segment_ids(1, L, seed, 3, False)
    elif kind == 3:
        seg_q = workloads.random_segment_ids(2, L, seed, 4, True)
        seg_kv = workloads.random_segment_ids(2, L, seed + 1, 4, True)
    got, ref = gpu_and_oracle(bsf, causal, wl, wr, seg_q, seg_kv, L, L, bq, bk)
    assert_same(got, ref, f"case {n}")


# Band-only masks (no segment IDs) are built either by one single-CTA kernel
# (tables up to 2048 q-block rows, 2048 kv-blocks and 65536 blocks) or by the
# one-launch persistent build; both take the block classes in closed form.
# Shapes on both sides of each limit, square and rectangular.
BAND_CASES = [
    # Lq, Lk, bq, bk, causal, wl, wr
    (131072, 2048, 64, 64, True, -1, -1),      # single CTA: 2048 rows x 32 (row limit)
    (2048, 131072, 128, 64, False, 700, 3000),  # single CTA: 16 rows x 2048 (column limit)
    (16384, 16384, 64, 64, True, 4095, 0),      # single CTA: 256 x 256 = 65536 blocks
    (16384, 16384, 64, 128, False, 100, 100),   # single CTA, bq != bk
    (20480, 20480, 64, 64, True, -1, -1),       # one launch: 320 x 320 blocks
    (8192, 139264, 64, 64, True, 2000, -1),     # one launch: 2176 kv-blocks
    (3000 * 64, 128, 64, 64, False, 10, 10),    # one launch, 3000 rows (single-CTA scan)
]


@pytest.mark.parametrize("Lq,Lk,bq,bk,causal,wl,wr", BAND_CASES)
def test_band_masks_both_build_paths(bsf, Lq, Lk, bq, bk, causal, wl, wr):
    got, ref = gpu_and_oracle(bsf, causal, wl, wr, None, None, Lq, Lk, bq, bk)
    assert_same(got, ref, f"{Lq}x{Lk} {bq}x{bk} causal={causal} window=({wl},{wr})")


# The build is one persistent launch up to 4M blocks and a bound of 65,536
# partial blocks (the blocks the band part alone leaves non-empty with segment
# IDs; 2 * (ceil((bq-1)/bk) + 1) per q-block row without them); past that it
# is the chain of nine kernels.  Inside the one launch, tables of more than
# 2048 q-block rows place their rows with a single-CTA scan.  Each path is
# compared bit for bit with the oracle.
PATH_CASES = [
    # label, Lq, Lk, bq, bk, causal, wl, wr, segments (0 none, 1 documents, 2 q and kv IDs of their own)
    ("chain: documents + causal, 512 x 512 blocks of 64", 32768, 32768, 64, 64, True, -1, -1, 1),
    ("chain: band only, 20000 rows x 8 columns", 20000 * 64, 512, 64, 64, False, 60, 100, 0),
    # (3,359 partial blocks: the pattern indices also come from the single-CTA
    # scan, where smaller tables count them in the first-occurrence bitmap)
    ("one launch, 2100 rows (single-CTA scan): q / kv IDs of their own", 2100 * 64, 256, 64, 64, False, -1, -1, 2),
]


@pytest.mark.parametrize("case", PATH_CASES, ids=[c[0] for c in PATH_CASES])
def test_build_paths_beyond_the_one_launch_limits(bsf, case):
    label, Lq, Lk, bq, bk, causal, wl, wr, segs = case
    seg_q = seg_kv = None
    if segs == 1:
        lens = workloads.document_lengths(Lq, 77, mean=1500, lo=64, hi=6000)
        seg_q = seg_kv = workloads.segment_ids_from_lengths(lens)
    elif segs == 2:
        seg_q = workloads.random_segment_ids(1, Lq, 78, 5, True)
        seg_kv = workloads.random_segment_ids(1, Lk, 79, 5, True)
    got, ref = gpu_and_oracle(bsf, causal, wl, wr, seg_q, seg_kv, Lq, Lk, bq, bk)
    assert_same(got, ref, label)


def test_rebuild_reuses_the_handle(bsf):
    seg = workloads.random_segment_ids(1, 1024, 5, 5, True).cuda()
    mi = bsf.build_mask_info(bsf.MaskSpec(True), 4096, 4096, 128, 128)
    a = mi.counts()
    mi.rebuild(bsf.MaskSpec(False, 10, 10, seg, seg), 1024, 1024, 64, 64)
    got = mi.to_host()
    ref = oracle.mask_info(oracle.MaskSpec(False, 10, 10, seg.cpu().numpy(), seg.cpu().numpy()), 1024, 1024, 64, 64)
    assert_same(got, ref, "rebuilt")
    mi.rebuild(bsf.MaskSpec(True), 4096, 4096, 128, 128)
    assert mi.counts() == a
    mi.close()


def test_everything_masked_gives_an_empty_table(bsf):
    q = torch.zeros(1, 256, dtype=torch.int32)
    kv = torch.ones(1, 256, dtype=torch.int32)
    got, ref = gpu_and_oracle(bsf, True, -1, -1, q, kv, 256, 256, 64, 64)
    assert got["num_active"] == 0
    assert_same(got, ref, "empty")


def test_async_build_then_attention_then_counts(bsf):
    # without segment IDs the build does not wait on the host; the attention
    # call may follow at once and the totals are read afterwards
    L = 2048
    q = workloads.normal_bf16((1, 2, L, 128), 11).cuda()
    k = workloads.normal_bf16((1, 2, L, 128), 12).cuda()
    v = workloads.normal_bf16((1, 2, L, 128), 13).cuda()
    mi = bsf.build_mask_info(bsf.MaskSpec(True, 300, 0), L, L, 128, 128)
    out, lse = bsf.attention_fwd(q, k, v, mi, 128 ** -0.5)
    mi.rebuild(bsf.MaskSpec(True), L, L, 128, 128)
    out2, lse2 = bsf.attention_fwd(q, k, v, mi, 128 ** -0.5)
    ref = oracle.mask_info(oracle.MaskSpec(True), L, L, 128, 128)
    c = mi.counts()
    assert (c["num_active"], c["num_partial"], c["num_patterns"], c["allowed_pairs"]) == \
        (ref.num_active, ref.num_partial, ref.num_patterns, ref.allowed_pairs)
    assert bsf.last_device_error() == 0
    O, Lr = oracle.attention(q.cpu(), k.cpu(), v.cpu(), oracle.MaskSpec(True), 128 ** -0.5, rows=np.arange(0, 2 * L, 7))
    from tests.parity import compare_rows, gather_rows
    o, l = gather_rows(out2, lse2, np.arange(0, 2 * L, 7))
    compare_rows(o, l, O, Lr, "async rebuild")
    mi.close()
