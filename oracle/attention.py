"""fp64 reference for the three hot-path operations (oracle side).

Test infrastructure only (see ``oracle/__init__``).  Arrays are numpy; the
caller converts bf16 tensors to float64 exactly (every bf16 value is an fp64
value) or passes raw ``uint16`` bit patterns to the two copy operations, which
move values without arithmetic.
"""

from __future__ import annotations

import numpy as np


def write_kv(k_cache, v_cache, k, v, slot_mapping, block_size: int):
    """Scatter each new token's K/V row into its cache slot; returns new caches.

    "vLLM Continuous Batching：从 Forward Shape 理解两个核心参数" §2.3补充 第一步:
    the K/V of flat token ``t`` go to ``(slot // block_size, slot % block_size)``
    of the ``[num_blocks, block_size, kv_heads, head_dim]`` cache ("vLLM 原理"
    §3.6, ``store_kvcache`` in §3.7).  A negative slot means "no write" (a pad
    token); the pages are silent on it.
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        b, off = divmod(int(slot), block_size)
        kc[b, off] = k[t]
        vc[b, off] = v[t]
    return kc, vc


def copy_blocks(k_cache, v_cache, pairs):
    """Copy-on-write block copies: ``cache[dst] = cache[src]`` for every pair.

    "vLLM 原理" §2.1 (Parallel Sampling): when a shared block with ref count > 1
    is about to be written, a fresh block is allocated and the old block's
    whole contents are copied into it.  Destinations are fresh blocks, so no
    pair reads a block another pair writes.
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    for src, dst in np.asarray(pairs, dtype=np.int64).reshape(-1, 2).tolist():
        kc[dst] = k_cache[src]
        vc[dst] = v_cache[src]
    return kc, vc


def swap_blocks(src_k, src_v, dst_k, dst_v, pairs):
    """Move whole blocks between two pools; returns the new destination pools.

    "LLM 推理引擎 Continuous Batching 与 PagedAttention：从 vLLM 原理到生产级部署实战"
    §4.4: swapping a request out copies its blocks from the GPU pool to the CPU
    pool, swapping in copies them back; a block is moved whole, all slots.
    """
    dk = np.array(dst_k, copy=True)
    dv = np.array(dst_v, copy=True)
    for s, d in np.asarray(pairs, dtype=np.int64).reshape(-1, 2).tolist():
        dk[d] = src_k[s]
        dv[d] = src_v[s]
    return dk, dv


def gather_sequence(cache, block_table_row, seq_len: int, block_size: int):
    """Dense ``[seq_len, kv_heads, head_dim]`` view of one sequence's paged K or V.

    "vLLM Continuous Batching：从 Forward Shape 理解两个核心参数" §2.3补充 第二步
    2): position p -> logical block p // block_size -> physical block via the
    sequence's own table -> offset p % block_size.  Only positions below
    seq_len are read, so reserved slots and other sequences' blocks never are.
    """
    p = np.arange(seq_len)
    phys = np.asarray(block_table_row)[p // block_size]
    if seq_len and (phys < 0).any():
        raise ValueError("block table has no block for a live position")
    return cache[phys, p % block_size]


def attention(q, k_cache, v_cache, qsl, seq_lens, block_tables, block_size: int,
              scale: float, num_kv_heads: int):
    """Ragged, causal, paged attention of one step's flat query batch, in fp64.

    For sequence ``s`` with ``q_s = qsl[s+1] - qsl[s]`` new tokens and
    ``L_s = seq_lens[s]`` tokens in total, local query ``i`` (flat row
    ``qsl[s] + i``) sits at position ``c_s + i`` with ``c_s = L_s - q_s``.  It
    attends to keys ``0 .. c_s + i`` of its own sequence only:
    ``o = softmax(scale * q k^T) v`` with a max-subtracted fp64 ``exp``.

    * Per-sequence isolation and causal visibility: "vLLM Continuous Batching：
      从 Forward Shape 理解两个核心参数" §0 and §2.3 (A never sees B; a_i sees
      positions 0..i).
    * New queries against the whole cached sequence ("seqlen_k 是整个 sequence
      长度"): "vLLM 原理" §3.7, which is why the causal mask is aligned to the
      bottom-right corner when ``c_s > 0``.
    * Query head ``h`` reads KV head ``h // (Hq / Hkv)`` (contiguous groups; the
      pages give only the two head counts, §2.2 of the first page).
    """
    q = np.asarray(q, dtype=np.float64)
    T, Hq, D = q.shape
    if Hq % num_kv_heads:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    g = Hq // num_kv_heads
    out = np.zeros((T, Hq, D), dtype=np.float64)
    qsl = np.asarray(qsl, dtype=np.int64)
    for s in range(len(seq_lens)):
        t0, t1 = int(qsl[s]), int(qsl[s + 1])
        qn, L = t1 - t0, int(seq_lens[s])
        if qn == 0:
            continue
        if L < qn:
            raise ValueError("seq_len shorter than the query")
        c = L - qn
        K = np.asarray(gather_sequence(k_cache, block_tables[s], L, block_size), dtype=np.float64)
        V = np.asarray(gather_sequence(v_cache, block_tables[s], L, block_size), dtype=np.float64)
        # key j is visible to local query i iff j <= c + i
        visible = np.arange(L)[None, :] <= (c + np.arange(qn))[:, None]
        for h in range(Hq):
            kh = h // g
            z = scale * (q[t0:t1, h, :] @ K[:, kh, :].T)          # [qn, L]
            z = np.where(visible, z, -np.inf)
            z = z - z.max(axis=1, keepdims=True)
            w = np.exp(z)
            w = w / w.sum(axis=1, keepdims=True)
            out[t0:t1, h, :] = w @ V[:, kh, :]
    return out


def attention_flops(qsl, seq_lens, num_q_heads: int, head_dim: int) -> int:
    """Multiply-add work of the visible (causal) score and value products.

    Each visible (query, key) pair costs ``2*D`` FLOPs for ``q . k`` and ``2*D``
    for ``w * v``; query ``i`` of sequence ``s`` sees ``c_s + i + 1`` keys.
    """
    qsl = np.asarray(qsl, dtype=np.int64)
    pairs = 0
    for s in range(len(seq_lens)):
        qn = int(qsl[s + 1] - qsl[s])
        c = int(seq_lens[s]) - qn
        pairs += qn * c + qn * (qn + 1) // 2
    return 4 * head_dim * num_q_heads * pairs
