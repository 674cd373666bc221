"""The seeded input generators (CPU only)."""
import torch

import workloads


def test_document_lengths_recipe():
    for seed in (4004, 1, 2, 3):
        lens = workloads.document_lengths(32768, seed)[0]
        assert sum(lens) == 32768
        assert all(64 <= n for n in lens)
        assert all(n <= 8192 for n in lens[:-1])
        assert lens[-1] <= 8192 + 64


def test_document_workload_is_deterministic():
    w = workloads.workload(4)
    a = workloads.make_inputs(w, with_values=False)
    b = workloads.make_inputs(w, with_values=False)
    assert a.doc_lengths == b.doc_lengths
    assert torch.equal(a.segment_ids, b.segment_ids)
    seg = a.segment_ids[0]
    assert seg.shape[0] == w.L
    assert torch.all(seg[1:] >= seg[:-1])
    assert int(seg[0]) == 0 and int(seg[-1]) == len(a.doc_lengths[0]) - 1


def test_values_are_seeded_bf16():
    x = workloads.normal_bf16((2, 3, 4), 123)
    y = workloads.normal_bf16((2, 3, 4), 123)
    assert x.dtype == torch.bfloat16 and torch.equal(x, y)
    z = workloads.normal_bf16((2, 3, 4), 124)
    assert not torch.equal(x, z)


def test_workload_table():
    assert [w.index for w in workloads.WORKLOADS] == [1, 2, 3, 4, 5]
    w5 = workloads.workload(5)
    assert (w5.window_left, w5.softcap, w5.L) == (4095, 30.0, 65536)
    w3 = workloads.workload(3)
    assert (w3.dqk, w3.dv, w3.bq, w3.bk) == (192, 128, 256, 128)
