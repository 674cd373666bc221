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
section "Softmax".  The Max Logit Estimate (§5.4 of the first page) replaces
the maximum by a constant c fixed in advance; its safe range follows from
where exp overflows and where it leaves the normal range in the working
precision (§5.4 and exercise 10).
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


def mle_softmax(x, c, dtype=np.float64):
    """Softmax with the constant reference c (Max Logit Estimate):
    exp(x - c) / sum exp(x - c), every step in `dtype`.  Returns
    (weights, l, lse) with l = sum exp(x - c) and lse = c + ln l."""
    x = np.asarray(x, dtype=dtype)
    c = dtype(c)
    with np.errstate(over="ignore", under="ignore", invalid="ignore", divide="ignore"):
        e = np.exp(x - c)
        l = np.sum(e, dtype=dtype)
        return e / l, l, c + np.log(l)


def exp_limits(dtype=np.float32):
    """(overflow, subnormal) thresholds of exp in `dtype`: exp(x) is finite
    below ln(max) and a normal number above ln(smallest normal)."""
    fi = np.finfo(dtype)
    return float(np.log(np.float64(fi.max))), float(np.log(np.float64(fi.tiny)))


def mle_safe_range(score_max, row_max_floor, dtype=np.float32, n_terms=1):
    """Open interval of constants c for which the Max Logit Estimate neither
    overflows (score_max - c below the overflow threshold) nor pushes a row
    whose maximum is row_max_floor out of the normal range
    (c - row_max_floor below minus the subnormal threshold).  The lecture
    bounds each exponential (n_terms = 1); a sum of n_terms of them stays
    finite only if c is also ln(n_terms) higher."""
    over, sub = exp_limits(dtype)
    return score_max - over + float(np.log(n_terms)), row_max_floor - sub
