"""Blockwise (online) softmax aggregation of one query row, step by step.

TEST INFRASTRUCTURE ONLY: the product path never imports this module.

This follows the update rules the pages state for one query row that sees its
scores one block at a time:

* "FlashAttention: l'attenzione che non spreca memoria", section
  "La online softmax, con i numeri": two running scalars per row, the record
  m and the running total l; when a block raises the record, whatever was
  already accumulated is re-expressed against the new record by the factor
  alpha = e^(m - m_new); at the very end o <- o / l.
* "L'attention fusionnee", section "Le softmax en ligne": per key tile,
  m' = max(m, max(s)), p = exp(s - m'), l = l*exp(m - m') + sum(p),
  o = o*exp(m - m') + p.v, m = m'; one division o / l after the last tile.
* "FlashAttention" (paweldubiel.com), section "Blockergebnisse einfach zu
  mitteln reicht nicht": the same state written as (m, l, u) with the result
  u / l.

Plain Python floats (double precision) and `math.exp`; no vectorisation.  The
function returns the full per-block trace so that the pages' worked examples
(which print the intermediate m, alpha and l) can be checked value by value.
"""

import math


def online_softmax_row(scores, values, block):
    """Aggregate `values` weighted by softmax(`scores`), `block` scores at a time.

    scores: sequence of floats (masked entries may be -inf).
    values: sequence of the same length; each item a float or a sequence of
            floats (a value vector).
    block:  positive block size; the last block may be shorter.

    Returns (out, lse, trace).  `out` = o / l (a float, or a list for vector
    values); `lse` = m + ln l; `trace` is a list with one dict per block
    holding the state after that block: m, alpha (None on the first block,
    where nothing had been accumulated), l and o.
    """
    if block < 1:
        raise ValueError("block must be >= 1")
    if len(scores) != len(values):
        raise ValueError("scores and values differ in length")
    if len(scores) == 0:
        raise ValueError("empty row")
    vector = not isinstance(values[0], (int, float))
    width = len(values[0]) if vector else 1

    def as_vec(x):
        return [float(t) for t in x] if vector else [float(x)]

    m = -math.inf
    l = 0.0
    o = [0.0] * width
    trace = []
    for start in range(0, len(scores), block):
        s = [float(x) for x in scores[start:start + block]]
        vals = [as_vec(x) for x in values[start:start + block]]
        m_new = max(m, max(s))
        if m_new == -math.inf:
            # every score seen so far is masked: nothing to accumulate yet
            trace.append({"m": m, "alpha": None, "l": l, "o": list(o)})
            continue
        first = m == -math.inf
        alpha = None if first else math.exp(m - m_new)
        p = [math.exp(x - m_new) for x in s]
        if first:
            l = sum(p)
            o = [sum(p[t] * vals[t][c] for t in range(len(p))) for c in range(width)]
        else:
            l = l * alpha + sum(p)
            o = [o[c] * alpha + sum(p[t] * vals[t][c] for t in range(len(p)))
                 for c in range(width)]
        m = m_new
        trace.append({"m": m, "alpha": alpha, "l": l,
                      "o": list(o) if vector else o[0]})
    if l == 0.0:
        return ([0.0] * width if vector else 0.0), -math.inf, trace
    out = [x / l for x in o]
    return (out if vector else out[0]), m + math.log(l), trace


def naive_block_average(scores, values, block):
    """The WRONG aggregation the paweldubiel.com note warns against.

    Each block is softmax-normalised on its own and the per-block results are
    then averaged with equal weight.  Kept only as a negative control: on the
    note's example (scores [0, 0, ln 3, ln 3], values [0, 0, 1, 1], blocks of
    two) it gives 0.5 instead of the exact 0.75.
    """
    results = []
    for start in range(0, len(scores), block):
        s = [float(x) for x in scores[start:start + block]]
        v = [float(x) for x in values[start:start + block]]
        mx = max(s)
        w = [math.exp(x - mx) for x in s]
        results.append(sum(wi * vi for wi, vi in zip(w, v)) / sum(w))
    return sum(results) / len(results)
