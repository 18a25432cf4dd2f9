"""Flat-batch metadata, written out from the pages' definitions (oracle side).

Test infrastructure only (see ``oracle/__init__``).
"""

from __future__ import annotations

import numpy as np


def query_start_loc(query_lens) -> np.ndarray:
    """Offsets of each sequence's new tokens inside the flat ``[T]`` batch.

    "vLLM Continuous Batching：从 Forward Shape 理解两个核心参数" §2.1: the array
    is the running sum of the per-sequence query lengths, starting at 0 and
    ending at T, so sequence ``s`` owns ``flat[qsl[s]:qsl[s+1]]``.  The same
    array appears as ``cu_seqlens_q`` in "vLLM 原理" §3.7 and as
    ``query_start_loc`` in "vLLM 学习笔记（2）：从单请求到批处理".
    """
    out = [0]
    for n in query_lens:
        n = int(n)
        if n < 0:
            raise ValueError("negative query length")
        out.append(out[-1] + n)
    return np.asarray(out, dtype=np.int64)


def positions(qsl, seq_lens) -> np.ndarray:
    """Position of every new token inside its own sequence.

    "vLLM Continuous Batching：从 Forward Shape 理解两个核心参数" §2.1: B decodes
    its 8th token at position 7 (7 cached), C at position 2, and A's prompt
    tokens sit at 0..4.  The new tokens are the last ``q_s`` of the sequence's
    ``seq_lens[s]`` tokens, so token ``i`` of sequence ``s`` has position
    ``seq_lens[s] - q_s + i``.
    """
    qsl = np.asarray(qsl, dtype=np.int64)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    pos = []
    for s in range(len(seq_lens)):
        q = int(qsl[s + 1] - qsl[s])
        cached = int(seq_lens[s]) - q
        if cached < 0:
            raise ValueError("seq_len shorter than the query")
        pos.extend(range(cached, cached + q))
    return np.asarray(pos, dtype=np.int64)


def physical_slot(block_table_row, pos: int, block_size: int):
    """(physical block, offset) holding position ``pos`` of one sequence.

    "vLLM Continuous Batching：从 Forward Shape 理解两个核心参数" §2.3补充 第二步
    1)-2): logical block = pos // block_size, physical block =
    block_table[logical block], offset = pos % block_size.
    """
    lb = pos // block_size
    return int(block_table_row[lb]), pos % block_size


def slot_mapping(qsl, seq_lens, block_tables, block_size: int) -> np.ndarray:
    """Flat slot index each new token's K/V is written to.

    "vLLM Continuous Batching：从 Forward Shape 理解两个核心参数" §2.3补充 第一步
    maps a flat token to ``physical_slot(block, offset)``; the slot is encoded
    as the single integer ``block * block_size + offset`` (the pages print only
    the pair; "vLLM 原理" §3.7 item 1 counts ``num_blocks * block_size``
    slots, one per token).
    """
    pos = positions(qsl, seq_lens)
    qsl = np.asarray(qsl, dtype=np.int64)
    out = np.empty(len(pos), dtype=np.int64)
    for s in range(len(seq_lens)):
        for t in range(int(qsl[s]), int(qsl[s + 1])):
            pb, off = physical_slot(block_tables[s], int(pos[t]), block_size)
            out[t] = pb * block_size + off
    return out


def pad_block_tables(tables, fill: int = -1) -> np.ndarray:
    """Stack per-sequence block lists into ``[S, max_blocks]``, padded with -1.

    "vLLM 原理" §3.7 item 4: sequences owning [0,1,2], [3,4,5,6] and [7] give
    ``[0,1,2,-1, 3,4,5,6, 7,-1,-1,-1]``.
    """
    width = max((len(t) for t in tables), default=0)
    out = np.full((len(tables), width), fill, dtype=np.int64)
    for i, t in enumerate(tables):
        out[i, : len(t)] = t
    return out


def padded_slot_counts(lengths):
    """(real tokens, padded slots, padding) of a static ``[B, L_max]`` batch.

    "vLLM Continuous Batching：从 Forward Shape 理解两个核心参数" §1: lengths
    16/128/1024/2048 give 3216 real tokens in 4 * 2048 = 8192 slots.
    """
    lengths = [int(x) for x in lengths]
    real = sum(lengths)
    slots = len(lengths) * max(lengths, default=0)
    return real, slots, slots - real


def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, itemsize: int) -> int:
    """K and V bytes one token occupies across all layers.

    "LLM 推理引擎 Continuous Batching 与 PagedAttention：从 vLLM 原理到生产级部署实战"
    §1.2: 2 (K and V) x layers x heads x head_dim x bytes per element.
    """
    return 2 * num_layers * num_kv_heads * head_dim * itemsize
