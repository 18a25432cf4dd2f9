"""Pins of the fp64 attention / scatter / copy oracle against things other than
itself: the pages' worked step, scalar brute force, the padded formulation,
torch's scaled_dot_product_attention (the textbook case it reduces to),
closed forms and invariants."""

import json
import math
import os

import numpy as np
import pytest
import torch

import workloads
from oracle import attention as ref
from oracle import brute, metadata, padded

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_examples.json")))


def _f64(t):
    return t.to(torch.float64).numpy()


def _case(lay, seed=0, poison=False):
    ts = workloads.make_tensors(lay, seed=seed, poison=poison)
    return {k: _f64(v) for k, v in ts.items()}


def _run_ref(lay, x, write=True):
    kc, vc = x["k_cache"], x["v_cache"]
    if write:
        kc, vc = ref.write_kv(kc, vc, x["k"], x["v"], lay.slot_mapping, lay.block_size)
    return ref.attention(x["q"], kc, vc, lay.query_start_loc, lay.seq_lens, lay.block_tables,
                         lay.block_size, lay.scale, lay.num_kv_heads), kc, vc


def _small_layouts():
    out = [workloads.config_layout(1, 0), workloads.literal_layout()]
    rng = np.random.default_rng(7)
    for i, (hq, hkv, d, bs) in enumerate([(4, 2, 8, 2), (6, 3, 4, 3), (2, 1, 8, 1), (4, 4, 5, 4)]):
        S = 4
        cached = rng.integers(0, 9, S)
        queries = rng.integers(1, 5, S)
        queries[1] = 0 if i % 2 else queries[1]      # an empty sequence
        cached[1] = max(cached[1], 1)
        out.append(workloads.custom_layout(f"tiny{i}", cached, queries, hq, hkv, d, bs, 40, 10 + i))
    return out


@pytest.mark.parametrize("lay", _small_layouts(), ids=lambda l: l.name)
def test_matches_scalar_brute_force(lay):
    x = _case(lay)
    o, kc, vc = _run_ref(lay, x)
    b = brute.attention(x["q"].tolist(), kc.tolist(), vc.tolist(), lay.query_start_loc.tolist(),
                        lay.seq_lens.tolist(), lay.block_tables.tolist(), lay.block_size,
                        lay.scale, lay.num_kv_heads)
    assert np.max(np.abs(o - np.array(b).reshape(o.shape))) <= 1e-12


@pytest.mark.parametrize("lay", _small_layouts(), ids=lambda l: l.name)
def test_matches_padded_formulation(lay):
    x = _case(lay)
    o, kc, vc = _run_ref(lay, x)
    qs, ks, vs, rows = [], [], [], []
    for s in range(lay.num_seqs):
        t0, t1 = int(lay.query_start_loc[s]), int(lay.query_start_loc[s + 1])
        if t1 == t0:
            continue
        L = int(lay.seq_lens[s])
        qs.append(x["q"][t0:t1])
        ks.append(np.array(brute.gather(kc, lay.block_tables[s], L, lay.block_size)))
        vs.append(np.array(brute.gather(vc, lay.block_tables[s], L, lay.block_size)))
        rows.append((t0, t1))
    po = padded.attention(qs, ks, vs, lay.scale, lay.num_kv_heads)
    for (t0, t1), y in zip(rows, po):
        assert np.max(np.abs(o[t0:t1] - y)) <= 1e-12


def _sdpa(q, k, v, scale, g, causal=True):
    # q [n, Hq, D], k/v [L, Hkv, D] -> [n, Hq, D] with a top-left causal mask on [n, L]
    qt = torch.from_numpy(q).transpose(0, 1)
    kt = torch.from_numpy(k).repeat_interleave(g, dim=1).transpose(0, 1)
    vt = torch.from_numpy(v).repeat_interleave(g, dim=1).transpose(0, 1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal, scale=scale)
    return o.transpose(0, 1).numpy()


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2)])
def test_identity_table_single_prompt_is_textbook_causal_attention(hq, hkv):
    # one sequence, no history, block table = identity: plain causal softmax attention
    L, D, bs = 37, 16, 4
    lay = workloads.custom_layout("one", [0], [L], hq, hkv, D, bs, 16, 0)
    lay.tables = [list(range(-(-L // bs)))]
    lay = workloads._finish(lay)
    x = _case(lay, seed=3)
    o, kc, vc = _run_ref(lay, x)
    expect = _sdpa(x["q"], x["k"], x["v"], lay.scale, hq // hkv)
    assert np.max(np.abs(o - expect)) <= 1e-12


def test_chunked_prefill_equals_last_rows_of_full_prefill():
    # the pages' 5000-token prompt under a 2048 budget with 10 decodes:
    # chunks [0:2038], [2038:4076], [4076:5000]; each chunk attends to the
    # whole cached prefix plus itself, so stacking the chunks' outputs must
    # give the full prompt's causal attention.
    ex = GOLDEN["chunked_prefill"]
    assert ex["budget"] - ex["decodes"] == ex["chunks"][0][1]
    P, hq, hkv, D, bs = ex["prompt"], 2, 1, 8, 16
    rng = np.random.default_rng(0)
    q = rng.standard_normal((P, hq, D))
    k = rng.standard_normal((P, hkv, D))
    v = rng.standard_normal((P, hkv, D))
    full = _sdpa(q, k, v, 1 / math.sqrt(D), hq // hkv)
    nb = -(-P // bs)
    table = np.arange(nb)[None, :]
    kc = np.zeros((nb, bs, hkv, D)); vc = np.zeros((nb, bs, hkv, D))
    kc.reshape(-1, hkv, D)[:P] = k
    vc.reshape(-1, hkv, D)[:P] = v
    for a, b in ex["chunks"]:
        o = ref.attention(q[a:b], kc, vc, [0, b - a], [b], table, bs, 1 / math.sqrt(D), hkv)
        assert np.max(np.abs(o - full[a:b])) <= 1e-12


def test_single_key_returns_its_value_exactly():
    lay = workloads.custom_layout("L1", [0, 0], [1, 1], 2, 1, 8, 4, 8, 0)
    x = _case(lay)
    o, kc, vc = _run_ref(lay, x)
    for s in range(2):
        assert np.array_equal(o[s, 0], x["v"][s, 0]) and np.array_equal(o[s, 1], x["v"][s, 0])


def test_zero_query_gives_causal_prefix_mean():
    lay = workloads.custom_layout("zq", [3], [4], 2, 2, 8, 2, 8, 0)
    x = _case(lay)
    x["q"][:] = 0.0
    o, kc, vc = _run_ref(lay, x)
    V = np.array(brute.gather(vc, lay.block_tables[0], 7, 2))
    for i in range(4):
        np.testing.assert_allclose(o[i], V[: 3 + i + 1].mean(axis=0), rtol=0, atol=1e-14)


def test_identical_keys_give_mean_and_boosted_key_dominates():
    lay = workloads.custom_layout("ik", [5], [1], 1, 1, 8, 4, 4, 0)
    x = _case(lay)
    kc, vc = ref.write_kv(x["k_cache"], x["v_cache"], x["k"], x["v"], lay.slot_mapping, 4)
    bt = lay.block_tables[0]
    kflat = kc.copy()
    for p in range(6):
        b, o_ = metadata.physical_slot(bt, p, 4)
        kflat[b, o_] = kc[bt[0], 0]           # every key equal to key 0
    o = ref.attention(x["q"], kflat, vc, lay.query_start_loc, lay.seq_lens, lay.block_tables, 4, lay.scale, 1)
    V = np.array(brute.gather(vc, bt, 6, 4))
    np.testing.assert_allclose(o[0, 0], V[:, 0].mean(axis=0), atol=1e-14)
    # boost key 2 so that its logit exceeds the others by 40
    kb = kc.copy()
    q0 = x["q"][0, 0]
    b2, o2 = metadata.physical_slot(bt, 2, 4)
    kb[b2, o2, 0] = q0 * (40.0 / lay.scale) / np.dot(q0, q0) + kb[b2, o2, 0]
    o = ref.attention(x["q"], kb, vc, lay.query_start_loc, lay.seq_lens, lay.block_tables, 4, lay.scale, 1)
    np.testing.assert_allclose(o[0, 0], V[2, 0], atol=1e-8)


def test_scale_enters_once():
    # doubling the scale equals doubling q
    lay = workloads.config_layout(1, 0)
    x = _case(lay)
    o1, kc, vc = _run_ref(lay, x)
    o2 = ref.attention(2 * x["q"], kc, vc, lay.query_start_loc, lay.seq_lens, lay.block_tables,
                       lay.block_size, lay.scale / 2, lay.num_kv_heads)
    assert np.max(np.abs(o1 - o2)) <= 1e-12


def test_block_permutation_invariance_and_isolation():
    lay = workloads.custom_layout("perm", [5, 9, 0, 3], [1, 1, 6, 2], 4, 2, 8, 4, 24, 5)
    x = _case(lay, poison=True)
    o, kc, vc = _run_ref(lay, x)
    assert np.isfinite(o).all()                        # never reads a NaN-poisoned slot
    perm = np.random.default_rng(1).permutation(lay.num_blocks)   # new id of old block b = perm[b]
    kp = np.empty_like(kc); vp = np.empty_like(vc)
    kp[perm] = kc; vp[perm] = vc
    bt = np.where(lay.block_tables >= 0, perm[np.maximum(lay.block_tables, 0)], -1)
    o2 = ref.attention(x["q"], kp, vp, lay.query_start_loc, lay.seq_lens, bt, 4, lay.scale, 2)
    assert np.array_equal(o, o2)


def test_sequence_order_permutes_rows():
    lay = workloads.custom_layout("ord", [4, 0, 7], [1, 3, 2], 2, 1, 8, 4, 16, 2)
    x = _case(lay)
    o, kc, vc = _run_ref(lay, x)
    order = [2, 0, 1]
    qsl = lay.query_start_loc
    rows = np.concatenate([np.arange(qsl[s], qsl[s + 1]) for s in order])
    qsl2 = metadata.query_start_loc([lay.query_lens[s] for s in order])
    o2 = ref.attention(x["q"][rows], kc, vc, qsl2, lay.seq_lens[order], lay.block_tables[order], 4, lay.scale, 1)
    assert np.array_equal(o2, o[rows])


def test_write_kv_pages_example():
    lay = workloads.literal_layout()
    ts = workloads.make_tensors(lay, seed=0)
    raw = {k: v.view(torch.int16).numpy() for k, v in ts.items()}
    kc, vc = ref.write_kv(raw["k_cache"], raw["v_cache"], raw["k"], raw["v"], lay.slot_mapping, 4)
    ex = GOLDEN["bca_step"]
    b, o = ex["b7_block_offset"]
    assert np.array_equal(kc[b, o], raw["k"][0]) and np.array_equal(vc[b, o], raw["v"][0])
    for i, (b, o) in enumerate(ex["a_block_offsets"]):
        assert np.array_equal(kc[b, o], raw["k"][2 + i])
    assert np.array_equal(kc[0, 2], raw["k"][1])     # C's token on its block 0
    changed = np.zeros((34, 4), bool)
    changed[21, 3] = changed[0, 2] = changed[18, 0] = True
    changed[5, :] = True
    assert np.array_equal(kc[~changed], raw["k_cache"][~changed])


def test_write_kv_skips_negative_slots():
    kc = np.zeros((2, 2, 1, 2), np.int16)
    k = np.ones((3, 1, 2), np.int16)
    out, _ = ref.write_kv(kc, kc, k, k, [1, -1, 2], 2)
    assert out.reshape(4, 2).tolist() == [[0, 0], [1, 1], [1, 1], [0, 0]]


def test_copy_blocks_pages_example():
    cache = np.arange(8 * 4 * 2 * 2, dtype=np.int16).reshape(8, 4, 2, 2)
    kc, vc = ref.copy_blocks(cache, -cache, [[1, 3]])
    assert np.array_equal(kc[3], cache[1]) and np.array_equal(vc[3], -cache[1])
    keep = [b for b in range(8) if b != 3]
    assert np.array_equal(kc[keep], cache[keep])


def test_swap_out_and_in_round_trip():
    # §4.4 of the deployment page: blocks go device -> host on swap-out and
    # come back host -> device (into whatever blocks are free) on swap-in.
    rng = np.random.default_rng(5)
    gpu = rng.integers(-1000, 1000, size=(10, 4, 2, 3)).astype(np.int16)
    cpu = rng.integers(-1000, 1000, size=(6, 4, 2, 3)).astype(np.int16)
    gpu_before, cpu_before = gpu.copy(), cpu.copy()
    out_pairs = [[3, 0], [5, 4], [1, 2]]
    hk, hv = ref.swap_blocks(gpu, -gpu, cpu, -cpu, out_pairs)
    assert np.array_equal(gpu, gpu_before) and np.array_equal(cpu, cpu_before)   # inputs kept
    for s, d in out_pairs:
        assert np.array_equal(hk[d], gpu[s]) and np.array_equal(hv[d], -gpu[s])
    for b in (1, 3, 5):                                   # host blocks no pair names
        assert np.array_equal(hk[b], cpu[b])
    in_pairs = [[0, 7], [4, 6], [2, 9]]
    dk, dv = ref.swap_blocks(hk, hv, gpu, -gpu, in_pairs)
    for (g_src, _), (_, g_dst) in zip(out_pairs, in_pairs):
        assert np.array_equal(dk[g_dst], gpu[g_src]) and np.array_equal(dv[g_dst], -gpu[g_src])
    for b in (0, 1, 2, 3, 4, 5, 8):
        assert np.array_equal(dk[b], gpu[b])


def test_swap_in_to_other_blocks_keeps_attention():
    # The block table is the only link from positions to blocks: after B's
    # blocks (10, 21 in the worked step) leave for the host and come back
    # into blocks 30, 31, attention with B's table rewritten is unchanged.
    ex = GOLDEN["bca_step"]
    rng = np.random.default_rng(9)
    nb, bs, hkv, d = 40, ex["block_size"], 2, 8
    kc = rng.standard_normal((nb, bs, hkv, d))
    vc = rng.standard_normal((nb, bs, hkv, d))
    q = rng.standard_normal((7, 4, d))
    tables = [ex["tables"]["B"], [7], ex["tables"]["A"]]
    bt = metadata.pad_block_tables(tables)
    args = (ex["query_start_loc"], ex["seq_lens"])
    before = ref.attention(q, kc, vc, *args, bt, bs, 0.3, hkv)
    host_k = np.zeros((4, bs, hkv, d))
    host_v = np.zeros((4, bs, hkv, d))
    host_k, host_v = ref.swap_blocks(kc, vc, host_k, host_v, [[10, 2], [21, 0]])
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[[10, 21]] = np.nan                                  # freed, then reused by others
    vc2[[10, 21]] = np.nan
    kc2, vc2 = ref.swap_blocks(host_k, host_v, kc2, vc2, [[2, 30], [0, 31]])
    bt2 = metadata.pad_block_tables([[30, 31], [7], ex["tables"]["A"]])
    after = ref.attention(q, kc2, vc2, *args, bt2, bs, 0.3, hkv)
    assert np.array_equal(before, after)


def test_attention_flops_closed_form():
    # decode with history c: q=1 sees c+1 keys; prefill of n sees n(n+1)/2 pairs
    assert ref.attention_flops([0, 1], [8], 1, 1) == 4 * 8
    assert ref.attention_flops([0, 5], [5], 2, 4) == 4 * 4 * 2 * 15
    assert ref.attention_flops([0, 2], [5], 1, 1) == 4 * (4 + 5)


# -- planted mistakes: each must be caught by one of the pins above ------------

def test_planted_gather_off_by_one_is_caught(monkeypatch):
    lay = workloads.config_layout(1, 0)
    x = _case(lay)
    good = ref.gather_sequence

    def shifted(cache, row, L, bs):
        out = good(cache, row, L + 1, bs) if L + 1 <= len(row) * bs else good(cache, row, L, bs)
        return out[1:] if len(out) > L else out[::-1]

    monkeypatch.setattr(ref, "gather_sequence", shifted)
    o, kc, vc = _run_ref(lay, x)
    b = brute.attention(x["q"].tolist(), kc.tolist(), vc.tolist(), lay.query_start_loc.tolist(),
                        lay.seq_lens.tolist(), lay.block_tables.tolist(), lay.block_size,
                        lay.scale, lay.num_kv_heads)
    assert np.max(np.abs(o - np.array(b).reshape(o.shape))) > 1e-3


def test_planted_wrong_exponential_is_caught(monkeypatch):
    L, D, bs, hq, hkv = 21, 16, 4, 4, 2
    lay = workloads.custom_layout("one", [0], [L], hq, hkv, D, bs, 16, 0)
    lay.tables = [list(range(-(-L // bs)))]
    lay = workloads._finish(lay)
    x = _case(lay, seed=3)
    monkeypatch.setattr(ref.np, "exp", np.exp2)
    o, _, _ = _run_ref(lay, x)
    monkeypatch.undo()
    expect = _sdpa(x["q"], x["k"], x["v"], lay.scale, hq // hkv)
    assert np.max(np.abs(o - expect)) > 1e-3
