"""Seeded synthetic inputs for one continuous-batching attention step.

This module is the only code that both the CUDA path (tests, ``bench.py``) and
the CPU oracle consume.  It draws lengths, block placements and tensor values
and lays them out in the metadata format the library's C ABI takes (the flat
``[T]`` batch with ``query_start_loc``, ``seq_lens``, ``-1``-padded
``block_tables`` and ``slot_mapping``).  It performs none of the attention,
scatter or copy arithmetic.

Workloads (shapes follow the pages' examples and Llama-2-7B's attention
geometry, 32 heads of 128 dims, with ``max_num_seqs = 256`` and
``max_num_batched_tokens = 8192``):

1. ``worked``  — the B/C/A step: B decodes after 7 cached tokens, C after 2,
   A prefills 5 tokens; 4/4 heads, head_dim 64, block_size 4, 16 blocks.
2. ``decode``  — 256 sequences x 1 new token, cached history uniform in
   [512, 4096]; 32/32 heads, head_dim 128, block_size 16, 70,000-block pool.
3. ``prefill`` — 16 prompts, log-uniform lengths in [16, 2048] trimmed to a
   total of 8192, no history; 32/8 heads, head_dim 128, block_size 16.
4. ``mixed``   — 240 decodes (history uniform in [128, 8192]) + two prefill
   chunks of 3976 tokens on 1024 and 3000 cached tokens (T = 8192); 32/8 heads.
5. ``shared``  — 64 sequences sharing one 16384-token prompt (1024 blocks,
   ref count 64), private tails of uniform [1, 256] tokens, 1 decode token
   each; 63 copy-on-write pairs for the last prompt block; 64/8 heads.
6. ``prefix``  — prefill on a cached prefix (a prefix-cache hit: only the
   uncached suffix is computed, against the whole cached sequence): 32
   sequences, cached history uniform in [1024, 8192], new chunks uniform in
   [64, 512] tokens; 32/8 heads, head_dim 128, block_size 16.

Placement: every sequence's logical blocks take consecutive entries of a
seeded random permutation of the pool.  Values: N(0, 1) rounded to bf16.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

CONFIG_NAMES = {1: "worked", 2: "decode", 3: "prefill", 4: "mixed", 5: "shared", 6: "prefix"}


@dataclass
class Layout:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    query_lens: np.ndarray            # int32 [S]
    seq_lens: np.ndarray              # int32 [S]
    tables: list                      # per-sequence physical block ids (after copy-on-write)
    cow_pairs: np.ndarray = field(default_factory=lambda: np.zeros((0, 2), np.int32))
    # flat metadata, filled by _finish()
    query_start_loc: np.ndarray = None
    block_tables: np.ndarray = None
    slot_mapping: np.ndarray = None
    num_decode_seqs: int = 0

    @property
    def num_seqs(self) -> int:
        return len(self.seq_lens)

    @property
    def num_tokens(self) -> int:
        return int(self.query_start_loc[-1])

    @property
    def max_query_len(self) -> int:
        return int(self.query_lens.max()) if self.num_seqs else 0

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.num_seqs else 0

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def cached_lens(self) -> np.ndarray:
        return self.seq_lens - self.query_lens

    def owned_blocks(self) -> np.ndarray:
        ids = set()
        for t in self.tables:
            ids.update(int(b) for b in t)
        return np.array(sorted(ids), dtype=np.int64)

    def reserved_slots(self) -> np.ndarray:
        """Slots of each sequence's last block that lie past its length."""
        out = []
        bs = self.block_size
        for t, L in zip(self.tables, self.seq_lens.tolist()):
            if not t:
                continue
            used = L - (len(t) - 1) * bs
            out.extend(int(t[-1]) * bs + o for o in range(used, bs))
        return np.array(out, dtype=np.int64)


def _finish(lay: Layout) -> Layout:
    """Lay the per-sequence description out as the C ABI's flat metadata."""
    q = lay.query_lens.astype(np.int64)
    lay.query_start_loc = np.concatenate([[0], np.cumsum(q)]).astype(np.int32)
    width = max((len(t) for t in lay.tables), default=0)
    bt = np.full((lay.num_seqs, max(width, 1)), -1, dtype=np.int32)
    for s, t in enumerate(lay.tables):
        bt[s, : len(t)] = t
    lay.block_tables = bt
    bs = lay.block_size
    slots = np.empty(int(q.sum()), dtype=np.int32)
    for s in range(lay.num_seqs):
        start = int(lay.seq_lens[s] - q[s])
        tab = lay.tables[s]
        base = int(lay.query_start_loc[s])
        for i in range(int(q[s])):
            p = start + i
            slots[base + i] = tab[p // bs] * bs + p % bs
    lay.slot_mapping = slots
    nd = 0
    while nd < lay.num_seqs and lay.query_lens[nd] == 1:
        nd += 1
    lay.num_decode_seqs = nd
    return lay


def _tables_from_permutation(seq_lens, block_size, num_blocks, rng, extra=()):
    perm = rng.permutation(num_blocks)
    cursor = 0
    tables = []
    for L in seq_lens:
        n = -(-int(L) // block_size)
        tables.append([int(b) for b in perm[cursor: cursor + n]])
        cursor += n
    if cursor > num_blocks:
        raise ValueError("pool too small for the batch")
    return tables, perm[cursor:]


def custom_layout(name, cached, queries, num_q_heads, num_kv_heads, head_dim, block_size,
                  num_blocks, seed, scale=None) -> Layout:
    """Arbitrary batch: sequence s has ``cached[s]`` history and ``queries[s]`` new tokens."""
    rng = np.random.default_rng(seed)
    cached = np.asarray(cached, dtype=np.int32)
    queries = np.asarray(queries, dtype=np.int32)
    seq_lens = (cached + queries).astype(np.int32)
    tables, _ = _tables_from_permutation(seq_lens, block_size, num_blocks, rng)
    lay = Layout(name, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                 scale if scale is not None else 1.0 / math.sqrt(head_dim),
                 queries, seq_lens, tables)
    return _finish(lay)


def prefill_lengths(rng, n=16, lo=16, hi=2048, total=8192):
    """Log-uniform prompt lengths in [lo, hi], rescaled to sum exactly to ``total``."""
    x = np.round(np.exp(rng.uniform(math.log(lo), math.log(hi), n))).astype(np.int64)
    y = np.clip(np.floor(x * total / x.sum()).astype(np.int64), lo, hi)
    rest = total - int(y.sum())
    order = np.argsort(-y, kind="stable")
    i = 0
    while rest != 0:
        j = order[i % n]
        if rest > 0 and y[j] < hi:
            y[j] += 1
            rest -= 1
        elif rest < 0 and y[j] > lo:
            y[j] -= 1
            rest += 1
        i += 1
        if i > 100 * n * (abs(rest) + 1) + total:
            raise ValueError("cannot trim lengths to the total")
    return y


def config_layout(cfg: int, seed: int = 0) -> Layout:
    """Layout of one of the five workloads (see the module docstring)."""
    rng = np.random.default_rng(1000 * cfg + seed)
    if cfg == 1:
        # B: 7 cached + 1, C: 2 cached + 1, A: 5-token prompt; decodes first.
        return custom_layout("worked", [7, 2, 0], [1, 1, 5], 4, 4, 64, 4, 16, 1000 + seed)
    if cfg == 2:
        cached = rng.integers(512, 4096, size=256, endpoint=True)
        return custom_layout("decode", cached, np.ones(256, np.int32), 32, 32, 128, 16,
                             70_000, 2000 + seed)
    if cfg == 3:
        lens = prefill_lengths(rng)
        return custom_layout("prefill", np.zeros(16, np.int32), lens, 32, 8, 128, 16,
                             4096, 3000 + seed)
    if cfg == 4:
        dec = rng.integers(128, 8192, size=240, endpoint=True)
        cached = np.concatenate([dec, [1024, 3000]])
        queries = np.concatenate([np.ones(240, np.int64), [3976, 3976]])
        return custom_layout("mixed", cached, queries, 32, 8, 128, 16, 70_000, 4000 + seed)
    if cfg == 5:
        return shared_prefix_layout(seed)
    if cfg == 6:
        cached = rng.integers(1024, 8192, size=32, endpoint=True)
        queries = rng.integers(64, 512, size=32, endpoint=True)
        return custom_layout("prefix", cached, queries, 32, 8, 128, 16, 16_384, 6000 + seed)
    raise ValueError(f"no workload {cfg}")


def shared_prefix_layout(seed: int = 0, num_seqs=64, prompt=16384, tail_max=256,
                         num_q_heads=64, num_kv_heads=8, head_dim=128, block_size=16,
                         num_blocks=4096) -> Layout:
    """Parallel sampling over one shared prompt, with copy-on-write of its last block.

    ``prompt`` should fill whole blocks: the tails are history that each
    sequence wrote after its copy, so a partial last prompt block would put
    the owner's tail tokens into the other sequences' copies.

    All sequences share the prompt's blocks (ref count ``num_seqs``).  Each one
    then writes into the last prompt block: sequences 0..n-2 move onto fresh
    private copies (one copy pair each), the last one keeps the original, whose
    ref count has dropped to 1 by then.  Tails (history) and the decode token
    live in private blocks after the prompt.
    """
    rng = np.random.default_rng(5000 + seed)
    perm = [int(b) for b in rng.permutation(num_blocks)]
    nprompt = -(-prompt // block_size)
    shared = perm[:nprompt]
    cursor = nprompt
    tails = rng.integers(1, tail_max, size=num_seqs, endpoint=True)
    seq_lens = (prompt + tails + 1).astype(np.int32)
    tables, pairs = [], []
    for s in range(num_seqs):
        tab = list(shared)
        if s < num_seqs - 1:
            fresh = perm[cursor]
            cursor += 1
            pairs.append((tab[-1], fresh))
            tab[-1] = fresh
        need = -(-int(seq_lens[s]) // block_size)
        while len(tab) < need:
            tab.append(perm[cursor])
            cursor += 1
        tables.append(tab)
    if cursor > num_blocks:
        raise ValueError("pool too small")
    lay = Layout("shared", num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                 1.0 / math.sqrt(head_dim), np.ones(num_seqs, np.int32), seq_lens, tables,
                 np.array(pairs, dtype=np.int32).reshape(-1, 2))
    return _finish(lay)


def literal_layout() -> Layout:
    """The B/C/A example with the pages' own physical block ids.

    B's table is [10, 21] and A's is [5, 18] as printed; C's table is not
    printed, so it takes block 0.  The pool has 34 blocks so that block 33
    (B's next block in the example) exists.  4/4 heads, head_dim 64, bs 4.
    """
    lay = Layout("literal", 4, 4, 64, 4, 34, 1.0 / 8.0,
                 np.array([1, 1, 5], np.int32), np.array([8, 3, 5], np.int32),
                 [[10, 21], [0], [5, 18]])
    return _finish(lay)


# ---------------------------------------------------------------------------
# tensor values


def make_tensors(lay: Layout, seed: int = 0, device="cpu", poison: bool = False,
                 chunk_blocks: int = 8192):
    """Draw q/k/v for the new tokens and the paged K/V pool (all bf16, N(0,1)).

    With ``poison`` every block no sequence owns, every reserved slot past a
    sequence's length, every slot the step is about to write and every
    copy-on-write destination is filled with NaN, so that a read outside a
    sequence's own live keys (or a missing write or copy) shows up as a NaN.
    """
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    T, Hq, Hkv, D = lay.num_tokens, lay.num_q_heads, lay.num_kv_heads, lay.head_dim
    bf = torch.bfloat16
    q = torch.randn((T, Hq, D), generator=g, device=device, dtype=bf)
    k = torch.randn((T, Hkv, D), generator=g, device=device, dtype=bf)
    v = torch.randn((T, Hkv, D), generator=g, device=device, dtype=bf)
    shape = (lay.num_blocks, lay.block_size, Hkv, D)
    k_cache = torch.empty(shape, device=device, dtype=bf)
    v_cache = torch.empty(shape, device=device, dtype=bf)
    for c in (k_cache, v_cache):
        for b0 in range(0, lay.num_blocks, chunk_blocks):
            b1 = min(lay.num_blocks, b0 + chunk_blocks)
            c[b0:b1] = torch.randn((b1 - b0,) + shape[1:], generator=g, device=device, dtype=bf)
    if poison:
        owned = np.zeros(lay.num_blocks, dtype=bool)
        owned[lay.owned_blocks()] = True
        for dst in lay.cow_pairs[:, 1].tolist():
            owned[dst] = True          # written by the copy; poisoned below
        unowned = torch.from_numpy(np.nonzero(~owned)[0]).to(device)
        slots = np.concatenate([lay.reserved_slots(),
                                lay.slot_mapping[lay.slot_mapping >= 0].astype(np.int64)])
        slots_t = torch.from_numpy(slots).to(device)
        dsts = torch.from_numpy(lay.cow_pairs[:, 1].astype(np.int64)).to(device)
        for c in (k_cache, v_cache):
            c.index_fill_(0, unowned, float("nan"))
            c.view(-1, Hkv, D).index_fill_(0, slots_t, float("nan"))
            c.index_fill_(0, dsts, float("nan"))
    return {"q": q, "k": k, "v": v, "k_cache": k_cache, "v_cache": v_cache}
