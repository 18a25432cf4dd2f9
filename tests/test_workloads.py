"""The seeded input generator lays out the metadata exactly as the oracle's
page-pinned definitions say, and each workload has the stated shape."""

import numpy as np
import pytest

import workloads
from oracle import blockmgr, metadata


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5, 6])
def test_generator_metadata_matches_oracle(cfg):
    lay = workloads.config_layout(cfg, 0)
    assert lay.query_start_loc.tolist() == metadata.query_start_loc(lay.query_lens).tolist()
    assert lay.block_tables.tolist() == metadata.pad_block_tables(lay.tables).tolist()
    sm = metadata.slot_mapping(lay.query_start_loc, lay.seq_lens, lay.block_tables, lay.block_size)
    assert np.array_equal(sm, lay.slot_mapping)
    # every live position has a block, blocks are in range, no block is owned twice
    # except through sharing in the shared-prefix workload
    for s, t in enumerate(lay.tables):
        assert len(t) == -(-int(lay.seq_lens[s]) // lay.block_size)
        assert all(0 <= b < lay.num_blocks for b in t)
    assert len(set(lay.slot_mapping.tolist())) == lay.num_tokens


def test_literal_layout_is_the_pages_example():
    lay = workloads.literal_layout()
    assert lay.query_start_loc.tolist() == [0, 1, 2, 7]
    assert lay.slot_mapping.tolist() == [87, 2, 20, 21, 22, 23, 72]
    assert lay.num_decode_seqs == 2


def test_workload_shapes():
    w = workloads.config_layout(1)
    assert (w.num_tokens, w.num_seqs, w.num_decode_seqs) == (7, 3, 2)
    assert w.seq_lens.tolist() == [8, 3, 5]
    d = workloads.config_layout(2)
    assert d.num_seqs == 256 and d.num_tokens == 256 and d.num_decode_seqs == 256
    assert d.cached_lens.min() >= 512 and d.cached_lens.max() <= 4096
    p = workloads.config_layout(3)
    assert p.num_seqs == 16 and p.num_tokens == 8192 and p.num_decode_seqs == 0
    assert p.query_lens.min() >= 16 and p.query_lens.max() <= 2048
    assert (p.cached_lens == 0).all() and (p.num_q_heads, p.num_kv_heads) == (32, 8)
    m = workloads.config_layout(4)
    assert m.num_tokens == 8192 and m.num_decode_seqs == 240
    assert m.query_lens[240:].tolist() == [3976, 3976]
    assert m.cached_lens[240:].tolist() == [1024, 3000]
    s = workloads.config_layout(5)
    assert s.num_seqs == 64 and (s.query_lens == 1).all() and len(s.cow_pairs) == 63
    assert s.seq_lens.min() >= 16384 + 2 and s.seq_lens.max() <= 16384 + 257
    x = workloads.config_layout(6)
    assert x.num_seqs == 32 and x.num_decode_seqs == 0
    assert x.cached_lens.min() >= 1024 and x.cached_lens.max() <= 8192
    assert x.query_lens.min() >= 64 and x.query_lens.max() <= 512


def test_shared_prefix_copy_pairs_follow_copy_on_write_rule():
    # Replaying the rule with the test-only block manager: 64 forks of one
    # prompt; each sequence in turn writes into the last prompt block.
    lay = workloads.config_layout(5)
    prompt_blocks = 1024
    shared = lay.tables[-1][:prompt_blocks]
    pool = blockmgr.BlockPool(lay.num_blocks, 16)
    base = pool.allocate(16384)
    tables = [base] + [pool.fork(base) for _ in range(63)]
    last = base[-1]
    pairs = []
    for t in tables:
        _, pair = pool.write_slot(t, 16383)
        if pair:
            pairs.append(pair)
    assert len(pairs) == len(lay.cow_pairs) == 63
    # same sources (the shared last block), fresh distinct destinations
    assert set(p[0] for p in pairs) == {last}
    assert set(lay.cow_pairs[:, 0].tolist()) == {shared[-1]}
    dst = lay.cow_pairs[:, 1].tolist()
    assert len(set(dst)) == 63 and not set(dst) & set(shared)
    # after the copies sequence 63 keeps the original block, the others their copy
    for s in range(63):
        assert lay.tables[s][prompt_blocks - 1] == dst[s]
        assert lay.tables[s][: prompt_blocks - 1] == shared[:-1]
    assert pool.ref[last] == 1 and tables[-1][-1] == last


def test_prefill_lengths_trim():
    rng = np.random.default_rng(123)
    y = workloads.prefill_lengths(rng)
    assert y.sum() == 8192 and y.min() >= 16 and y.max() <= 2048


def test_poison_marks_only_dead_slots():
    import torch
    lay = workloads.config_layout(1)
    ts = workloads.make_tensors(lay, poison=True)
    kc = ts["k_cache"].float()
    owned = set(lay.owned_blocks().tolist())
    dead = set(lay.reserved_slots().tolist()) | set(lay.slot_mapping.tolist())
    for b in range(lay.num_blocks):
        for o in range(lay.block_size):
            nan = torch.isnan(kc[b, o]).all().item()
            if b not in owned or b * lay.block_size + o in dead:
                assert nan
            else:
                assert not torch.isnan(kc[b, o]).any().item()


def test_shared_prefix_blocks_of_the_shared_workload():
    # the bench's cascade leg passes the leading table entries every sequence
    # shares: the prompt's blocks before the copied last one
    import bench
    lay = workloads.config_layout(5, 0)
    assert bench.shared_prefix_blocks(lay) == 1023
    small = workloads.shared_prefix_layout(1, num_seqs=4, prompt=160, tail_max=20,
                                           num_q_heads=8, num_kv_heads=2, head_dim=64,
                                           block_size=16, num_blocks=64)
    assert bench.shared_prefix_blocks(small) == 9
    # every key position below the shared prefix maps to the same block in every table
    for s in range(small.num_seqs):
        assert list(small.tables[s][:9]) == list(small.tables[0][:9])
    # the copied last prompt block differs for all but the last sequence
    assert len({int(small.tables[s][9]) for s in range(small.num_seqs)}) == small.num_seqs
