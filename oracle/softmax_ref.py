"""Online softmax and the two-segment merge, in float64 numpy.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

These restate the softmax algebra of "Pallas Kernels and Splash Attention"
(CMU 11-868 Lecture 13 notes), §5.1 "Online softmax": the running pair
(m, l) is updated block by block as m_new = max(m, max(block)),
l <- l * exp(m - m_new) + sum(exp(block - m_new)); two partial results
(m1, l1, o1), (m2, l2, o2) merge as m = max(m1, m2),
l = l1 exp(m1 - m) + l2 exp(m2 - m), o = (o1 exp(m1 - m) + o2 exp(m2 - m)) / l,
where o1, o2 are the unnormalised weighted sums.  The safe (two-pass)
softmax follows "The maths and infra behind core LLM operations" (joto.ai),
section "Softmax".
"""
import numpy as np


def safe_softmax(x):
    """Two-pass softmax: subtract the maximum, exponentiate, normalise."""
    x = np.asarray(x, dtype=np.float64)
    m = np.max(x)
    e = np.exp(x - m)
    return e / np.sum(e)


def online_softmax_trace(x, block):
    """Scans x in blocks of `block` entries; returns the (m, l) after each
    block and the final softmax exp(x - m) / l."""
    x = np.asarray(x, dtype=np.float64)
    m, l = -np.inf, 0.0
    trace = []
    for s in range(0, len(x), block):
        blk = x[s:s + block]
        m_new = max(m, float(np.max(blk)))
        l = l * np.exp(m - m_new) + float(np.sum(np.exp(blk - m_new)))
        m = m_new
        trace.append((m, l))
    return trace, np.exp(x - m) / l


def partial_state(scores, values):
    """(m, l, o) of one segment: o is the unnormalised sum exp(s - m) v."""
    s = np.asarray(scores, dtype=np.float64)
    v = np.asarray(values, dtype=np.float64)
    m = float(np.max(s))
    p = np.exp(s - m)
    return m, float(np.sum(p)), p @ v


def merge(m1, l1, o1, m2, l2, o2):
    """Merges two segment states; returns (m, l, normalised output)."""
    m = max(m1, m2)
    a1, a2 = np.exp(m1 - m), np.exp(m2 - m)
    l = l1 * a1 + l2 * a2
    return m, l, (np.asarray(o1) * a1 + np.asarray(o2) * a2) / l
