"""Seeded synthetic workloads for block-sparse masked attention.

This module only draws inputs: shapes, seeds and random numbers.  It holds
none of the method's arithmetic, so both the CUDA path and the CPU oracle
can be fed from it without sharing any computation.

The five workload shapes follow the configurations the lecture notes
discuss ("Pallas Kernels and Splash Attention", §1.1 and §6.6: 128 heads,
L = 4096, head dims 192/128, DeepSeek-V3 style) plus dense-causal GQA, a
document mask joined with causal, and a causal local window with a tanh
soft cap.  Values are N(0, 1) drawn in float32 by torch's CPU generator,
rounded to bf16 (round to nearest even).  Seeds: workload c uses 1000c+1,
1000c+2, 1000c+3 for q, k, v and 1000c+4 for the document lengths.
"""
import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch


@dataclass(frozen=True)
class Workload:
    index: int                # 1-based workload number
    name: str
    B: int
    Hq: int
    Hkv: int
    L: int
    dqk: int
    dv: int
    bq: int
    bk: int
    causal: bool = True
    window_left: int = -1     # inclusive distance, -1 = unbounded
    window_right: int = -1
    documents: bool = False   # segment IDs from seeded document lengths
    softcap: float = 0.0
    Lq: int = 0               # query length when it differs from L (L is then the key length)

    @property
    def q_len(self) -> int:
        return self.Lq or self.L

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.dqk)

    @property
    def seeds(self):
        c = self.index
        return 1000 * c + 1, 1000 * c + 2, 1000 * c + 3, 1000 * c + 4

    def describe(self) -> str:
        lens = f"L={self.L}" if not self.Lq else f"Lq={self.Lq}, Lk={self.L}"
        parts = [f"B={self.B}", f"Hq={self.Hq}", f"Hkv={self.Hkv}", lens,
                 f"dqk={self.dqk}", f"dv={self.dv}", f"blocks={self.bq}x{self.bk}"]
        mask = []
        if self.documents:
            mask.append("document")
        if self.window_left >= 0:
            mask.append(f"window {self.window_left + 1}")
        if self.causal:
            mask.append("causal")
        parts.append("mask=" + "+".join(mask or ["none"]))
        if self.softcap > 0:
            parts.append(f"softcap={self.softcap:g}")
        return f"{self.name}: " + ", ".join(parts)


WORKLOADS: List[Workload] = [
    Workload(1, "tiny causal MHA", 1, 2, 2, 256, 64, 64, 64, 64),
    Workload(2, "dense causal GQA", 2, 32, 8, 4096, 128, 128, 128, 128),
    # the configuration leaves the blocks open: 256-row q-blocks let the
    # kernel's two 128-row tiles of one head share each K / V tile
    Workload(3, "wide-head causal MHA", 1, 128, 128, 4096, 192, 128, 256, 128),
    Workload(4, "document + causal GQA", 1, 16, 8, 32768, 128, 128, 128, 128, documents=True),
    Workload(5, "local window 4096 + causal + softcap 30", 1, 32, 8, 65536, 128, 128, 128, 128,
             window_left=4095, window_right=0, softcap=30.0),
]


# Workloads beyond the five above, for the split-KV forward: few query rows
# against long keys (the shape where one item per q-block row leaves most of
# the GPU idle).  Not one of the five configurations.
EXTRA_WORKLOADS: List[Workload] = [
    Workload(6, "few queries, long keys GQA", 1, 32, 8, 65536, 128, 128, 128, 128, causal=False, Lq=512),
]


def workload(index: int) -> Workload:
    if index <= len(WORKLOADS):
        return WORKLOADS[index - 1]
    return EXTRA_WORKLOADS[index - len(WORKLOADS) - 1]


def normal_bf16(shape, seed: int) -> torch.Tensor:
    """N(0, 1) in float32 from torch's CPU generator, rounded to bf16."""
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def document_lengths(L: int, seed: int, mean: int = 2048, lo: int = 64, hi: int = 8192,
                     batch_rows: int = 1) -> List[List[int]]:
    """Seeded document lengths per batch row.

    Each length is 1 + floor(ln(U) / ln(1 - 1/mean)) for U ~ U(0, 1) (a
    geometric draw on {1, 2, ...} with the given mean), clipped to [lo, hi];
    lengths are appended until they reach L, the last one is cut so that the
    row sums to exactly L, and a last piece shorter than lo is merged into
    the document before it.
    """
    g = torch.Generator().manual_seed(seed)
    out = []
    q = math.log(1.0 - 1.0 / mean)
    for _ in range(batch_rows):
        lens: List[int] = []
        total = 0
        while total < L:
            u = float(torch.rand(1, generator=g, dtype=torch.float64).item())
            u = max(u, 1e-300)
            n = 1 + int(math.floor(math.log(u) / q))
            n = min(max(n, lo), hi)
            if total + n > L:
                n = L - total
            lens.append(n)
            total += n
        if len(lens) > 1 and lens[-1] < lo:
            last = lens.pop()
            lens[-1] += last
        out.append(lens)
    return out


def segment_ids_from_lengths(lengths: List[List[int]]) -> torch.Tensor:
    """int32 [batch_rows, L]: document d of a row gets id d (0, 1, 2, ...)."""
    rows = []
    for lens in lengths:
        ids = torch.cat([torch.full((n,), d, dtype=torch.int32) for d, n in enumerate(lens)])
        rows.append(ids)
    return torch.stack(rows)


@dataclass
class Inputs:
    q: torch.Tensor                         # bf16 [B, Hq, L, dqk] (CPU)
    k: torch.Tensor                         # bf16 [B, Hkv, L, dqk]
    v: torch.Tensor                         # bf16 [B, Hkv, L, dv]
    segment_ids: Optional[torch.Tensor]     # int32 [B, L] or None
    doc_lengths: Optional[List[List[int]]] = field(default=None)


def make_inputs(w: Workload, with_values: bool = True) -> Inputs:
    sq, sk, sv, ss = w.seeds
    if with_values:
        q = normal_bf16((w.B, w.Hq, w.q_len, w.dqk), sq)
        k = normal_bf16((w.B, w.Hkv, w.L, w.dqk), sk)
        v = normal_bf16((w.B, w.Hkv, w.L, w.dv), sv)
    else:
        q = k = v = None
    seg = lens = None
    if w.documents:
        lens = document_lengths(w.L, ss, batch_rows=w.B)
        seg = segment_ids_from_lengths(lens)
    return Inputs(q, k, v, seg, lens)


def random_segment_ids(B: int, L: int, seed: int, max_id: int, sorted_ids: bool) -> torch.Tensor:
    """Random int32 segment IDs in [0, max_id) for fuzz tests; sorted per row
    (contiguous documents) or in arbitrary order (non-monotone IDs)."""
    g = torch.Generator().manual_seed(seed)
    ids = torch.randint(0, max_id, (B, L), generator=g, dtype=torch.int64)
    if sorted_ids:
        ids, _ = torch.sort(ids, dim=1)
    return ids.to(torch.int32)
