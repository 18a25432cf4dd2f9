"""Static ``[B, L_max]`` padded formulation with an attention mask (oracle side).

Test infrastructure only (see ``oracle/__init__``).  This is the traditional
batch that "vLLM Continuous Batching：从 Forward Shape 理解两个核心参数" §1 and
§2.1 and "vLLM 学习笔记（2）：从单请求到批处理" contrast with the flat batch:
every sequence padded to the longest one, pad positions masked out.  It takes
dense per-sequence K/V (no block table, no flat offsets) so that agreeing with
``oracle.attention`` pins the ragged slicing, the gather and the mask
alignment of the flat formulation.
"""

from __future__ import annotations

import numpy as np


def attention(q_list, k_list, v_list, scale, num_kv_heads):
    """Attention of a padded batch.

    ``q_list[s]``: ``[q_s, Hq, D]`` queries of sequence s (its newest tokens);
    ``k_list[s]``, ``v_list[s]``: ``[L_s, Hkv, D]`` all of its keys/values in
    position order.  Returns a list of ``[q_s, Hq, D]`` outputs.
    """
    S = len(q_list)
    Hq, D = q_list[0].shape[1:]
    g = Hq // num_kv_heads
    qmax = max(x.shape[0] for x in q_list)
    lmax = max(x.shape[0] for x in k_list)
    Qp = np.zeros((S, qmax, Hq, D))
    Kp = np.zeros((S, lmax, num_kv_heads, D))
    Vp = np.zeros((S, lmax, num_kv_heads, D))
    mask = np.zeros((S, qmax, lmax), dtype=bool)   # True = may attend
    for s in range(S):
        qn, L = q_list[s].shape[0], k_list[s].shape[0]
        Qp[s, :qn] = q_list[s]
        Kp[s, :L] = k_list[s]
        Vp[s, :L] = v_list[s]
        # queries are the sequence's last qn tokens: row i is at position L - qn + i
        for i in range(qn):
            mask[s, i, : L - qn + i + 1] = True
    # expand KV heads to query heads, contiguous groups of g
    Kq = np.repeat(Kp, g, axis=2)
    Vq = np.repeat(Vp, g, axis=2)
    z = scale * np.einsum("sihd,sjhd->shij", Qp, Kq)
    z = np.where(mask[:, None, :, :], z, -np.inf)
    rowmax = z.max(axis=3, keepdims=True)
    rowmax = np.where(np.isfinite(rowmax), rowmax, 0.0)   # fully padded query rows
    w = np.exp(z - rowmax)
    den = w.sum(axis=3, keepdims=True)
    w = np.divide(w, den, out=np.zeros_like(w), where=den > 0)
    o = np.einsum("shij,sjhd->sihd", w, Vq)
    return [o[s, : q_list[s].shape[0]] for s in range(S)]
