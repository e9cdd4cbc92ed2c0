"""Second oracle path: pure-Python loops with ``math.exp`` and ``math.fsum``.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Written separately
from ``fd_oracle.c`` so the two can pin each other on tiny inputs.  Values
arrive already widened to Python floats (float64 arrays from
``torch.Tensor.double()``), so this path also checks the C code's own bf16
and int8 widening.

Definition followed: softmax(scale * q . k_j) over the visible keys, weighted
sum of the value rows; "each seeing the cache plus the drafts before it"
(ComfyUI #16509, list item 2) gives the bottom-right causal window; the
gather attends exactly the listed cells (llama.cpp #28244, Conversation).
"""
from __future__ import annotations

import math


def visible_dense(L, cap, n_q, i, causal):
    """Cache positions query row ``i`` sees in the dense prefix mode."""
    L = max(0, min(int(L), int(cap)))
    if causal:
        # row n_q-1 is the newest token and sees all L positions; row i sees
        # the prefix that ends (n_q - 1 - i) positions earlier.
        hi = L - (n_q - 1 - i)
    else:
        hi = L
    return list(range(0, max(hi, 0)))


def visible_gather(lst, cap):
    """Listed cells, in list order, padding (<0) and out-of-range dropped."""
    return [int(j) for j in lst if 0 <= int(j) < int(cap)]


def attend_row(qrow, krows, vrows, scale):
    """One softmax-weighted average; ``krows``/``vrows`` are lists of rows."""
    d = len(vrows[0]) if vrows else len(qrow)
    if not krows:
        return [0.0] * d
    scores = [scale * math.fsum(a * b for a, b in zip(qrow, kr)) for kr in krows]
    mx = max(scores)
    w = [math.exp(s - mx) for s in scores]
    den = math.fsum(w)
    return [math.fsum(w[t] * vrows[t][c] for t in range(len(w))) / den
            for c in range(d)]


def attend(q, k, v, visible, scale):
    """Brute-force attention.

    q: nested lists / float64 array [B, n_q, Hq, d]
    k, v: [B, Hkv, cap, d] (already dequantised)
    visible(b, i) -> list of cache positions for query row i of sequence b.
    Returns nested lists [B][n_q][Hq][d].
    """
    B, n_q, Hq = len(q), len(q[0]), len(q[0][0])
    Hkv = len(k[0])
    g = Hq // Hkv
    out = []
    for b in range(B):
        ob = []
        for i in range(n_q):
            pos = visible(b, i)
            oi = []
            for h in range(Hq):
                hk = h // g
                qrow = [float(x) for x in q[b][i][h]]
                krows = [[float(x) for x in k[b][hk][j]] for j in pos]
                vrows = [[float(x) for x in v[b][hk][j]] for j in pos]
                oi.append(attend_row(qrow, krows, vrows, scale))
            ob.append(oi)
        out.append(ob)
    return out
