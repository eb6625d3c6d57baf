"""Brute-force attention for tiny inputs: pure Python, math.fsum sums.

An independent second statement of softmax(scale * Q K^T [masked]) V for
n <= 8, written without numpy or the C oracle, so that a dropped term, a wrong
index or a transposed operand in either one shows up as a mismatch. Masked
keys are left out of the sums entirely (their weight is exactly zero).
"""

import math


def attention_row(q_row, keys, values, scale, visible):
    """q_row: list[d_k]; keys: list of list[d_k]; values: list of list[d_v]."""
    scores = [scale * math.fsum(a * b for a, b in zip(q_row, key)) for key in keys]
    vis_scores = [s for s, ok in zip(scores, visible) if ok]
    top = max(vis_scores)
    expo = [math.exp(s - top) if ok else 0.0 for s, ok in zip(scores, visible)]
    total = math.fsum(expo)
    weights = [e / total for e in expo]
    d_v = len(values[0])
    out = [math.fsum(weights[j] * values[j][c] for j in range(len(values))) for c in range(d_v)]
    return out, weights


def attention(q, k, v, scale, causal=False, key_lens=None):
    """q[b][t][i][c], k[b][j][i][c], v[b][j][i][c] nested lists -> out[b][t][i][c]."""
    out = []
    for b in range(len(q)):
        n_k = len(k[b])
        kv_len = key_lens[b] if key_lens is not None else n_k
        rows = []
        for t in range(len(q[b])):
            heads = []
            for i in range(len(q[b][t])):
                visible = [(not (causal and j > t)) and j < kv_len for j in range(n_k)]
                keys = [k[b][j][i] for j in range(n_k)]
                vals = [v[b][j][i] for j in range(n_k)]
                o, _ = attention_row(q[b][t][i], keys, vals, scale, visible)
                heads.append(o)
            rows.append(heads)
        out.append(rows)
    return out


def feed_forward_row(x, w1, b1, w2, b2, gamma, beta, eps):
    """One row of LayerNorm(x + max(0, x W1 + b1) W2 + b2): x list[d_model],
    w1 list of d_model lists of d_ff, w2 list of d_ff lists of d_model."""
    d_model, d_ff = len(x), len(b1)
    hid = [max(0.0, b1[j] + math.fsum(x[c] * w1[c][j] for c in range(d_model))) for j in range(d_ff)]
    z = [x[c] + b2[c] + math.fsum(hid[j] * w2[j][c] for j in range(d_ff)) for c in range(d_model)]
    mean = math.fsum(z) / d_model
    var = math.fsum((v - mean) ** 2 for v in z) / d_model
    return [gamma[c] * (z[c] - mean) / math.sqrt(var + eps) + beta[c] for c in range(d_model)]
