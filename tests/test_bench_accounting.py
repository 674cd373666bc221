"""bench.py's FLOP accounting (CPU): useful FLOPs count the allowed (q, k)
pairs, executed FLOPs every element of every active block, with the counts
taken from the oracle's MaskInfo of the workload's mask."""
import pytest

import bench
import oracle
import workloads


def counts_of(w):
    mi = oracle.mask_info(oracle.MaskSpec(w.causal, w.window_left, w.window_right), w.q_len, w.L, w.bq, w.bk)
    return {"allowed_pairs": mi.allowed_pairs, "num_active": mi.num_active}


def test_dense_causal_gqa_flops():
    # causal L = 4096: L (L + 1) / 2 allowed pairs per head; 528 active 128 x 128 blocks
    w = workloads.workload(2)
    useful, executed = bench.flop_counts(w, counts_of(w), 1)
    per = 2 * (128 + 128) * w.B * w.Hq
    assert useful == per * 4096 * 4097 // 2 == pytest.approx(2.7495e11, rel=1e-4)
    assert executed == per * 128 * 128 * 528 == pytest.approx(2.8347e11, rel=1e-4)


def test_wide_head_flops_with_256_row_blocks():
    # the same causal pairs; 272 active 256 x 128 blocks execute 3 % more than
    # the 528 blocks of 128 x 128 (each row's last block is masked for its
    # upper half)
    w = workloads.workload(3)
    assert (w.bq, w.bk) == (256, 128)
    c = counts_of(w)
    assert c["num_active"] == 272
    useful, executed = bench.flop_counts(w, c, 1)
    per = 2 * (192 + 128) * w.Hq
    assert useful == per * 4096 * 4097 // 2 == pytest.approx(6.8736e11, rel=1e-4)
    assert executed == per * 256 * 128 * 272
    assert executed / (per * 128 * 128 * 528) == pytest.approx(544 / 528)
