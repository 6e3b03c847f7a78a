"""Pure-Python brute force of the decode definition -- TEST INFRASTRUCTURE ONLY.

Loop-by-loop, on Python floats (IEEE double), for tiny inputs only.  It
restates the same definition as ``pa_oracle.c`` independently so the two can
be checked against each other:

  for sequence b, query head h, KV head k = h // G (contiguous GQA groups,
  the broadcast of one KV head over its query group in the
  "paged_attention_v2_pytorch.py" commit 15ef28e, "Key changes"):
      s_t = scale * sum_d q[b][h][d] * K[table[b][t // bs]][k][t % bs][d]
      out[d] = sum_t exp(s_t) V_t[d] / sum_t exp(s_t)

Inputs are nested lists / numpy arrays of already-decoded Python floats.
"""
from __future__ import annotations

import math


def decode(query, key_cache, value_cache, block_tables, seq_lens, scale, q_len=None):
    """query [S][H][D], or [S][Q][H][D] with q_len = Q (query i sees t <= L - Q + i)."""
    if q_len is not None:
        rows = []
        for b in range(len(query)):
            per_i = []
            for i in range(q_len):
                visible = max(0, min(int(seq_lens[b]), int(seq_lens[b]) - q_len + i + 1))
                per_i.append(decode([query[b][i]], key_cache, value_cache, [block_tables[b]],
                                    [visible], scale)[0])
            rows.append(per_i)
        return rows
    S = len(query)
    H = len(query[0])
    D = len(query[0][0])
    KV = len(key_cache[0])
    bs = len(key_cache[0][0])
    G = H // KV
    out = []
    for b in range(S):
        rows = []
        for h in range(H):
            k = h // G
            L = int(seq_lens[b])
            if L == 0:
                rows.append([0.0] * D)
                continue
            s = []
            for t in range(L):
                blk = int(block_tables[b][t // bs])
                krow = key_cache[blk][k][t % bs]
                s.append(scale * math.fsum(float(query[b][h][d]) * float(krow[d]) for d in range(D)))
            m = max(s)
            w = [math.exp(x - m) for x in s]
            z = math.fsum(w)
            o = []
            for d in range(D):
                acc = math.fsum(
                    w[t] * float(value_cache[int(block_tables[b][t // bs])][k][t % bs][d])
                    for t in range(L))
                o.append(acc / z)
            rows.append(o)
        out.append(rows)
    return out
