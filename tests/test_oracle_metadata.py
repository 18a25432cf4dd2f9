"""Pins of the oracle's metadata functions and the test-only block manager
against the integers the pages print (tests/golden/pages_examples.json)."""

import json
import os

import numpy as np
import pytest

from oracle import blockmgr, metadata

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_examples.json")))


def test_bca_query_start_loc_positions_seq_lens():
    ex = GOLDEN["bca_step"]
    qsl = metadata.query_start_loc(ex["query_lens"])
    assert qsl.tolist() == ex["query_start_loc"]
    seq_lens = [c + q for c, q in zip(ex["cached"], ex["query_lens"])]
    assert seq_lens == ex["seq_lens"]
    assert metadata.positions(qsl, seq_lens).tolist() == ex["positions"]


def test_bca_slots_and_block_reads():
    ex = GOLDEN["bca_step"]
    bs = ex["block_size"]
    B, A = ex["tables"]["B"], ex["tables"]["A"]
    assert metadata.physical_slot(B, 7, bs) == tuple(ex["b7_block_offset"])
    assert [list(metadata.physical_slot(A, p, bs)) for p in range(5)] == ex["a_block_offsets"]
    reads = ex["b_reads"]
    assert [p for p in range(8) if metadata.physical_slot(B, p, bs)[0] == 10] == reads["block_10_positions"]
    assert [p for p in range(8) if metadata.physical_slot(B, p, bs)[0] == 21] == reads["block_21_positions"]
    # full slot_mapping with C on block 0 (C's table is not printed)
    tables = metadata.pad_block_tables([B, [0], A])
    sm = metadata.slot_mapping(ex["query_start_loc"], ex["seq_lens"], tables, bs)
    expect = [21 * bs + 3, 0 * bs + 2] + [b * bs + o for b, o in ex["a_block_offsets"]]
    assert sm.tolist() == expect


def test_three_prompts_and_apple_banana():
    ex = GOLDEN["three_prompts"]
    assert metadata.query_start_loc(ex["lengths"]).tolist() == ex["query_start_loc"]
    real, slots, _ = metadata.padded_slot_counts(ex["lengths"])
    assert (real, slots) == (ex["real_tokens"], ex["padded_slots"])
    ab = GOLDEN["apple_banana"]
    assert metadata.query_start_loc(ab["lengths"]).tolist() == ab["cu_seqlens"]


def test_padded_block_tables():
    ex = GOLDEN["padded_block_tables"]
    assert metadata.pad_block_tables(ex["tables"]).reshape(-1).tolist() == ex["flat_padded"]


def test_static_padding_counts():
    ex = GOLDEN["static_padding"]
    assert metadata.padded_slot_counts(ex["lengths"]) == (ex["real_tokens"], ex["slots"], ex["padding"])


def test_kv_bytes_per_token():
    ex = GOLDEN["kv_bytes"]
    b = metadata.kv_bytes_per_token(ex["layers"], ex["kv_heads"], ex["head_dim"], ex["itemsize"])
    assert b == ex["bytes_per_token"]
    assert b * ex["tokens"] == ex["bytes_for_tokens"]


def test_positions_reject_short_seq():
    with pytest.raises(ValueError):
        metadata.positions([0, 3], [2])


# -- test-only block manager ---------------------------------------------------

def test_copy_on_write_example():
    ex = GOLDEN["copy_on_write"]
    bs = ex["block_size"]
    shared = ex["shared_physical_blocks"]
    order = shared + [3] + [b for b in range(8) if b not in shared + [3]]
    pool = blockmgr.BlockPool(8, bs, free_order=order)
    a1 = pool.allocate(ex["prompt_tokens"])
    assert a1 == shared
    a2 = pool.fork(a1)
    assert [pool.ref[b] for b in shared] == [ex["ref_count_before"]] * 2
    # A1 writes its next token at position 7 (logical block 1)
    slot, pair = pool.write_slot(a1, ex["prompt_tokens"])
    assert list(pair) == ex["first_writer_copy"]
    assert a1 == ex["first_writer_table_after"]
    assert pool.ref[shared[1]] == ex["ref_count_of_1_after"]
    assert slot == 3 * bs + 3
    # A2 writes at the same position: no copy any more
    slot2, pair2 = pool.write_slot(a2, ex["prompt_tokens"])
    assert pair2 is None and ex["second_writer_copies"] == 0
    assert slot2 == shared[1] * bs + 3


def test_b_grows_into_block_33():
    ex = GOLDEN["bca_step"]["b_growth"]
    bs = GOLDEN["bca_step"]["block_size"]
    order = [10, 21, 33] + [b for b in range(34) if b not in (10, 21, 33)]
    pool = blockmgr.BlockPool(34, bs, free_order=order)
    table = pool.allocate(8)
    assert table == [10, 21]
    assert pool.needs_new_block(ex["new_position"] + 1)
    slot, pair = pool.write_slot(table, ex["new_position"])
    assert pair is None
    assert ex["new_position"] // bs == ex["logical_block"]
    assert table == ex["table_after"]
    assert slot == ex["appended_physical_block"] * bs


def test_can_append_rule():
    ex = GOLDEN["can_append"]
    pool = blockmgr.BlockPool(4, ex["block_size"])
    for n, need in ex["new_len_needs_block"].items():
        assert pool.needs_new_block(int(n)) == need


def test_deallocate_returns_blocks():
    pool = blockmgr.BlockPool(6, 4)
    t = pool.allocate(9)
    u = pool.fork(t)
    pool.deallocate(t)
    assert len(pool.free) == 3
    pool.deallocate(u)
    assert len(pool.free) == 6 and not pool.used
