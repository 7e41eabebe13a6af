"""Pure-Python brute force of the differential-attention head, for tiny shapes.

Plain nested loops over Python floats with ``math.exp``; nothing vectorised,
nothing shared with the C oracle.  Used only to check the oracle on N <= 16,
d <= 8.  Source: "Differential Transformer" glossary page, section "How
differential attention works" (two softmax maps, (map1 - lambda map2) V,
per-head normalisation, times (1 - lambda_init)).
"""
import math


def _softmax_row(q_row, keys, visible_js, d):
    logits = []
    for j in visible_js:
        dot = 0.0
        for c in range(d):
            dot += q_row[c] * keys[j][c]
        logits.append(dot / math.sqrt(d))
    top = max(logits)
    ex = [math.exp(x - top) for x in logits]
    tot = sum(ex)
    return [e / tot for e in ex]


def head_forward(q1, k1, q2, k2, v, lam, causal, headnorm, w_head, eps, lambda_init):
    """One head: lists of rows in, list of output rows out.

    There may be fewer query rows than key rows (a key/value cache): the queries
    are then the last positions of the sequence, query i at position
    len(k1) - len(q1) + i.
    """
    n = len(q1)
    n_keys = len(k1)
    d = len(q1[0])
    dv = len(v[0])
    out = []
    for i in range(n):
        pos = n_keys - n + i
        js = [j for j in range(n_keys) if (j <= pos or not causal)]
        p1 = _softmax_row(q1[i], k1, js, d)
        p2 = _softmax_row(q2[i], k2, js, d)
        o = [0.0] * dv
        for t, j in enumerate(js):
            wgt = p1[t] - lam * p2[t]
            for c in range(dv):
                o[c] += wgt * v[j][c]
        if headnorm:
            ms = sum(x * x for x in o) / dv
            r = 1.0 / math.sqrt(ms + eps)
            o = [o[c] * r * (1.0 if w_head is None else w_head[c]) * (1.0 - lambda_init)
                 for c in range(dv)]
        out.append(o)
    return out
