"""Scalar-loop restatement of paged attention, for tiny inputs only (oracle side).

Test infrastructure only (see ``oracle/__init__``).  It walks the block table
one position at a time, keeps the running maximum / running sum / running
weighted value exactly as the online-softmax update of "LLM 推理引擎 Continuous
Batching 与 PagedAttention：从 vLLM 原理到生产级部署实战" §3.3 does (new max
m' = max(m, s); l <- l * e^(m - m') + e^(s - m'); the value accumulator takes
the same rescale), with ``math.exp`` and Python floats.  It shares no code with
``attention.py`` and is used to pin it.
"""

from __future__ import annotations

import math


def attention(q, k_cache, v_cache, qsl, seq_lens, block_tables, block_size, scale, num_kv_heads):
    """Same contract as ``oracle.attention.attention``; nested lists in, nested lists out.

    ``q[t][h][d]``, ``k_cache[b][o][kh][d]``; returns ``out[t][h][d]``.
    """
    T = len(q)
    Hq = len(q[0]) if T else 0
    D = len(q[0][0]) if T else 0
    g = Hq // num_kv_heads
    out = [[[0.0] * D for _ in range(Hq)] for _ in range(T)]
    for s in range(len(seq_lens)):
        t0, t1 = int(qsl[s]), int(qsl[s + 1])
        L = int(seq_lens[s])
        cached = L - (t1 - t0)
        for t in range(t0, t1):
            last = cached + (t - t0)          # newest key this query may see
            for h in range(Hq):
                kh = h // g
                m = -math.inf
                l = 0.0
                acc = [0.0] * D
                for p in range(last + 1):
                    blk = int(block_tables[s][p // block_size])
                    off = p % block_size
                    krow = k_cache[blk][off][kh]
                    vrow = v_cache[blk][off][kh]
                    sc = 0.0
                    for d in range(D):
                        sc += float(q[t][h][d]) * float(krow[d])
                    sc *= scale
                    m_new = max(m, sc)
                    alpha = math.exp(m - m_new) if m != -math.inf else 0.0
                    e = math.exp(sc - m_new)
                    l = l * alpha + e
                    for d in range(D):
                        acc[d] = acc[d] * alpha + e * float(vrow[d])
                    m = m_new
                for d in range(D):
                    out[t][h][d] = acc[d] / l
    return out


def gather(cache, block_table_row, seq_len, block_size):
    """Per-position loop gather of one sequence's rows: ``rows[p] = cache[bt[p//bs]][p%bs]``."""
    rows = []
    for p in range(int(seq_len)):
        rows.append(cache[int(block_table_row[p // block_size])][p % block_size])
    return rows
