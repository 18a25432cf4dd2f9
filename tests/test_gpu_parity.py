"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Attention: max-abs <= 2e-2 and mean-abs <= 2e-3 (bf16 inputs, fp32
accumulation, bf16 output).  Scatter and block copies: bit-exact.  Every
case runs on NaN-poisoned pools (unowned blocks, reserved slots, slots about
to be written, copy destinations), so a read outside a sequence's own live
keys or a missing write shows up as a non-finite output.
"""

import numpy as np
import pytest
import torch

import paged_kv_cache_133_gb300 as pa
import workloads
from tests import _helpers as H

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    H.ensure_built()
    torch.cuda.set_device(0)


@pytest.fixture(autouse=True)
def _no_device_errors():
    # every step a test runs without its own flag reports here; none may fire
    H.default_err().zero_()
    yield
    torch.cuda.synchronize()
    assert int(H.default_err().item()) == 0


def _small_cases():
    rng = np.random.default_rng(11)
    cases = [workloads.config_layout(1, 0), workloads.literal_layout()]
    specs = [
        # (name, Hq, Hkv, D, bs, decodes, prefills)
        ("d128_bs16_g4", 8, 2, 128, 16, 5, 3),
        ("d64_bs16_g1", 4, 4, 64, 16, 3, 2),
        ("d128_bs1", 4, 2, 128, 1, 2, 2),
        ("d128_bs2_g8", 16, 2, 128, 2, 3, 1),
        ("d64_bs8_g2", 4, 2, 64, 8, 4, 4),
        ("d128_bs32_g16", 32, 2, 128, 32, 3, 2),
        ("d128_bs64_g32", 32, 1, 128, 64, 2, 2),
        ("d64_bs256", 2, 2, 64, 256, 2, 2),
        ("d128_bs128_g6", 12, 2, 128, 128, 3, 3),
        # short chunks with a group of 4 or 8: tiles of <= 64 tokens carry two
        # heads per side on the tensor-core kernel
        ("d64_bs16_g4_short", 8, 2, 64, 16, 2, 5),
        ("d128_bs16_g8_short", 16, 2, 128, 16, 1, 6),
    ]
    for i, (name, hq, hkv, d, bs, nd, npf) in enumerate(specs):
        cached = list(rng.integers(0, 300, nd)) + list(rng.integers(0, 200, npf))
        queries = [1] * nd + list(rng.integers(1, 150, npf))
        if npf:
            cached[-1] = 0                      # a plain prompt
            queries[-1] = int(rng.integers(60, 200))
        nb = sum(-(-(c + q) // bs) for c, q in zip(cached, queries)) + 7
        cases.append(workloads.custom_layout(name, cached, queries, hq, hkv, d, bs, nb, 100 + i))
    # degenerate: single-token prompts (L = 1), and an empty sequence in the middle
    cases.append(workloads.custom_layout("L1", [0, 0, 5], [1, 1, 1], 4, 2, 128, 16, 8, 3))
    cases.append(workloads.custom_layout("empty_mid", [9, 3, 0], [1, 0, 17], 4, 1, 64, 4, 16, 4))
    # scale <= 0 is legal (the tensor-core prefill takes the row maximum before
    # scaling and leaves such steps to the general kernel)
    cases.append(workloads.custom_layout("neg_scale", [40, 0, 130], [1, 150, 70], 8, 2, 128, 16,
                                         40, 5, scale=-0.07))
    cases.append(workloads.custom_layout("zero_scale", [0, 20], [90, 33], 4, 2, 64, 16, 16, 6,
                                         scale=0.0))
    return cases


@pytest.mark.parametrize("lay", _small_cases(), ids=lambda l: l.name)
def test_small_step_matches_oracle(lay):
    ts = workloads.make_tensors(lay, seed=5, poison=True)
    g = {k: v.to(DEV) for k, v in ts.items()}
    md = H.device_meta(lay, DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = H.run_step(lay, g, md, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    expect = H.oracle_full(lay, ts)
    got = H.f64(out)
    rows = [t for s in range(lay.num_seqs)
            for t in range(lay.query_start_loc[s], lay.query_start_loc[s + 1])]
    H.assert_close(got[rows], expect[rows], lay.name)
    # the scatter is bit-exact: compare the whole pool's bits with the oracle's
    from oracle import attention as ref
    bits = {k: v.view(torch.int16).numpy() for k, v in ts.items()}
    kc, vc = bits["k_cache"], bits["v_cache"]
    if len(lay.cow_pairs):
        kc, vc = ref.copy_blocks(kc, vc, lay.cow_pairs)
    kc, vc = ref.write_kv(kc, vc, bits["k"], bits["v"], lay.slot_mapping, lay.block_size)
    assert np.array_equal(g["k_cache"].view(torch.int16).cpu().numpy(), kc)
    assert np.array_equal(g["v_cache"].view(torch.int16).cpu().numpy(), vc)


@pytest.mark.parametrize("lay", _small_cases()[2:6], ids=lambda l: l.name)
def test_decode_rows_on_prefill_kernel(lay):
    # num_decode_seqs = 0 sends the single-token rows through the general kernel
    ts = workloads.make_tensors(lay, seed=6, poison=True)
    g = {k: v.to(DEV) for k, v in ts.items()}
    md = H.device_meta(lay, DEV)
    out = H.run_step(lay, g, md, num_decode=0)
    torch.cuda.synchronize()
    H.assert_close(H.f64(out), H.oracle_full(lay, ts), lay.name)


def _sample_rows(lay, rng, n_seq, rows_per_seq=3):
    seqs = list(rng.choice(lay.num_seqs, size=min(n_seq, lay.num_seqs), replace=False))
    seqs.append(int(np.argmax(lay.seq_lens)))      # the longest sequence
    rows = []
    for s in sorted(set(int(x) for x in seqs)):
        q = int(lay.query_lens[s])
        picks = {0, q - 1} | set(int(x) for x in rng.integers(0, q, rows_per_seq))
        rows += [(s, i) for i in sorted(picks) if 0 <= i < q]
    return rows


@pytest.mark.parametrize("cfg", [2, 3, 4, 5, 6])
def test_full_size_workload(cfg):
    # Workloads 2-4 (decode batch, 16-prompt prefill, mixed step): every output
    # row against the oracle.  Workloads 5-6 (shared prefix, prefix-cached
    # prefill): sampled rows, whose oracle cost stays in seconds.
    lay = workloads.config_layout(cfg, 0)
    g = workloads.make_tensors(lay, seed=0, device=DEV, poison=True)
    md = H.device_meta(lay, DEV)
    every_row = cfg in (2, 3, 4)
    if every_row:
        full = H.FullOracle(lay, g)
    else:
        rng = np.random.default_rng(cfg)
        snap = H.Snapshot(lay, g, _sample_rows(lay, rng, 8))
    written = md["slots"].long()
    k_new, v_new = g["k"].clone(), g["v"].clone()
    src_blocks = md["pairs"][:, 0].long() if len(lay.cow_pairs) else None
    src_k = g["k_cache"].index_select(0, src_blocks).clone() if src_blocks is not None else None
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = H.run_step(lay, g, md, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # bit-exact scatter of every new token and copy of every pair
    Hkv, D = lay.num_kv_heads, lay.head_dim
    assert torch.equal(g["k_cache"].view(-1, Hkv, D)[written].view(torch.int16), k_new.view(torch.int16))
    assert torch.equal(g["v_cache"].view(-1, Hkv, D)[written].view(torch.int16), v_new.view(torch.int16))
    if src_k is not None:
        dst = g["k_cache"].index_select(0, md["pairs"][:, 1].long())
        assert torch.equal(dst.view(torch.int16), src_k.view(torch.int16))
    # every output row is finite and matches the oracle (or the sampled rows do)
    assert torch.isfinite(out.float()).all()
    if every_row:
        full.check(out, lay.name)
    else:
        H.assert_close(snap.gpu_rows(out), snap.expected(), lay.name)


def _perm_case():
    return workloads.custom_layout("perm", [700, 33, 0, 1500, 5], [1, 1, 40, 1, 90], 16, 4, 128, 16,
                                   400, 21)


def test_block_permutation_is_bitwise_invariant():
    lay = _perm_case()
    ts = workloads.make_tensors(lay, seed=9, poison=True)
    g1 = {k: v.to(DEV) for k, v in ts.items()}
    out1 = H.run_step(lay, g1, H.device_meta(lay, DEV))
    perm = np.random.default_rng(2).permutation(lay.num_blocks)
    lay2 = workloads.custom_layout("perm", [700, 33, 0, 1500, 5], [1, 1, 40, 1, 90], 16, 4, 128,
                                   16, 400, 21)
    lay2.tables = [[int(perm[b]) for b in t] for t in lay.tables]
    lay2 = workloads._finish(lay2)
    g2 = {k: v.to(DEV) for k, v in ts.items()}
    pt = torch.from_numpy(perm).to(DEV)
    for name in ("k_cache", "v_cache"):
        moved = torch.empty_like(g2[name])
        moved[pt] = g2[name]
        g2[name] = moved
    out2 = H.run_step(lay2, g2, H.device_meta(lay2, DEV))
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_run_to_run_bitwise_determinism():
    lay = workloads.config_layout(5, 0)
    g = workloads.make_tensors(lay, seed=1, device=DEV)
    md = H.device_meta(lay, DEV)
    out1 = H.run_step(lay, g, md).clone()
    out2 = H.run_step(lay, g, md).clone()
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_sequence_order_permutes_rows():
    lay = _perm_case()
    ts = workloads.make_tensors(lay, seed=3, poison=True)
    g = {k: v.to(DEV) for k, v in ts.items()}
    out = H.run_step(lay, g, H.device_meta(lay, DEV)).clone()
    # reverse the prefills and the decodes separately (decodes stay first)
    nd = lay.num_decode_seqs
    order = list(reversed(range(nd))) + list(reversed(range(nd, lay.num_seqs)))
    qsl = lay.query_start_loc
    rows = np.concatenate([np.arange(qsl[s], qsl[s + 1]) for s in order])
    lay2 = workloads.Layout("ord", lay.num_q_heads, lay.num_kv_heads, lay.head_dim, lay.block_size,
                            lay.num_blocks, lay.scale, lay.query_lens[order], lay.seq_lens[order],
                            [lay.tables[s] for s in order])
    lay2 = workloads._finish(lay2)
    g2 = {k: (v[torch.from_numpy(rows).to(DEV)] if k in ("q", "k", "v") else v) for k, v in g.items()}
    out2 = H.run_step(lay2, g2, H.device_meta(lay2, DEV))
    torch.cuda.synchronize()
    assert torch.equal(out2.view(torch.int16), out[torch.from_numpy(rows).to(DEV)].view(torch.int16))


def test_copy_on_write_copy_is_needed():
    # without the block copies the shared-prefix step reads NaN-poisoned blocks
    lay = workloads.shared_prefix_layout(0, num_seqs=4, prompt=64, tail_max=8, num_q_heads=8,
                                         num_kv_heads=2, num_blocks=64)
    ts = workloads.make_tensors(lay, seed=2, poison=True)
    g = {k: v.to(DEV) for k, v in ts.items()}
    md = H.device_meta(lay, DEV)
    pa.write_kv(g["k"], g["v"], g["k_cache"], g["v_cache"], md["slots"])
    out = pa.attention(g["q"], g["k_cache"], g["v_cache"], md["qsl"], md["seq_lens"], md["bt"],
                       num_decode_seqs=lay.num_decode_seqs, max_query_len=1,
                       max_seq_len=lay.max_seq_len, scale=lay.scale)
    torch.cuda.synchronize()
    assert not torch.isfinite(out.float()[:3]).all()     # sequences 0..2 read fresh blocks
    g = {k: v.to(DEV) for k, v in ts.items()}
    out = H.run_step(lay, g, md)
    torch.cuda.synchronize()
    H.assert_close(H.f64(out), H.oracle_full(lay, ts), "cow")


def test_many_splits_combine():
    # few long decode sequences force many key splits and the combine pass
    lay = workloads.custom_layout("splits", [9000, 20000, 300], [1, 1, 1], 8, 1, 128, 16,
                                  2000, 8)
    ws = pa.workspace_size(3, 8, 1, 128, lay.max_seq_len)
    assert ws > 0
    ts = workloads.make_tensors(lay, seed=4, poison=True)
    g = {k: v.to(DEV) for k, v in ts.items()}
    before = pa.kernel_launches()
    out = H.run_step(lay, g, H.device_meta(lay, DEV))
    torch.cuda.synchronize()
    assert pa.kernel_launches() - before == 3           # scatter, decode, combine
    H.assert_close(H.f64(out), H.oracle_full(lay, ts), "splits")


def test_empty_batch_is_a_no_op():
    lay = workloads.config_layout(1, 0)
    g = workloads.make_tensors(lay, seed=0, device=DEV)
    k0 = g["k_cache"].clone()
    before = pa.kernel_launches()
    z = torch.zeros(0, dtype=torch.int32, device=DEV)
    pa.write_kv(g["k"][:0], g["v"][:0], g["k_cache"], g["v_cache"], z)
    assert pa.kernel_launches() == before
    assert torch.equal(k0, g["k_cache"])


@pytest.fixture(params=["tc", "mma"])
def prefill_impl(request, monkeypatch):
    """Run a test once on the tcgen05 prefill kernel and once on the mma.sync one."""
    if request.param == "mma":
        monkeypatch.setenv("PA_PREFILL_IMPL", "mma")
    else:
        monkeypatch.delenv("PA_PREFILL_IMPL", raising=False)
    return request.param


def _prefill_cases():
    rng = np.random.default_rng(23)
    out = []
    for i, (hq, hkv, d, bs) in enumerate([(8, 2, 128, 16), (4, 4, 64, 16), (8, 1, 128, 8),
                                           (4, 2, 128, 256), (12, 4, 64, 32), (2, 2, 128, 128)]):
        cached = [0, int(rng.integers(1, 400)), 0, int(rng.integers(100, 900))]
        queries = [int(rng.integers(1, 300)), int(rng.integers(100, 260)), 128, int(rng.integers(2, 40))]
        nb = sum(-(-(c + q) // bs) for c, q in zip(cached, queries)) + 5
        out.append(workloads.custom_layout(f"pf{i}_h{hq}x{hkv}_d{d}_bs{bs}", cached, queries, hq, hkv,
                                           d, bs, nb, 200 + i))
    return out


@pytest.mark.parametrize("lay", _prefill_cases(), ids=lambda l: l.name)
def test_prefill_kernels_match_oracle(lay, prefill_impl):
    ts = workloads.make_tensors(lay, seed=8, poison=True)
    g = {k: v.to(DEV) for k, v in ts.items()}
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = H.run_step(lay, g, H.device_meta(lay, DEV), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    H.assert_close(H.f64(out), H.oracle_full(lay, ts), f"{lay.name}/{prefill_impl}")


def test_prefill_slot_walk_is_bitwise_identical():
    # Beyond 2046 cost levels (max_seq_len above 261,760) the scheduler walks
    # every (level, sequence, head pair) slot and skips the empty ones instead
    # of using its dense item table.  max_seq_len is only an upper bound, so
    # a small batch passed with max_seq_len 300,000 takes that path: about
    # 37,500 slots, nearly all empty, so every CTA's first slot is empty and
    # the draws come from the work counter.  The same items run in the same
    # order, so the output is bit for bit the dense list's, eagerly and
    # replayed from a CUDA graph (the counter's reset at the last draw
    # covers slots too).
    lay = _prefill_cases()[0]
    g = workloads.make_tensors(lay, seed=5, device=DEV)
    md = H.device_meta(lay, DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.write_kv(g["k"], g["v"], g["k_cache"], g["v_cache"], md["slots"], err=err)
    ws = torch.empty(1 << 16, dtype=torch.uint8, device=DEV)

    def attn(out, max_seq_len):
        pa.attention(g["q"], g["k_cache"], g["v_cache"], md["qsl"], md["seq_lens"], md["bt"],
                     num_decode_seqs=0, max_query_len=lay.max_query_len,
                     max_seq_len=max_seq_len, scale=lay.scale, out=out, workspace=ws, err=err)

    expect = torch.empty_like(g["q"])
    attn(expect, lay.max_seq_len)
    out = torch.full_like(g["q"], float("nan"))
    attn(out, 300_000)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), expect.view(torch.int16))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        attn(out, 300_000)
    torch.cuda.synchronize()
    for _ in range(3):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), expect.view(torch.int16))
    assert int(err.item()) == 0


@pytest.mark.parametrize("pad", [8, 16], ids=["16B_rows", "32B_rows"])
def test_prefill_output_with_padded_rows(pad):
    # An output whose token stride carries `pad` extra elements.  Rows that
    # are 16- but not 32-byte aligned (pad 8) take the general kernel, since
    # the tensor-core epilogue stores 32 bytes at a time; pad 16 keeps the
    # tensor-core path.  Both must write only their own rows.
    lay = _prefill_cases()[0]
    ts = workloads.make_tensors(lay, seed=9, poison=True)
    g = {k: v.to(DEV) for k, v in ts.items()}
    T, hq, d = g["q"].shape
    buf = torch.full((T, hq * d + pad), float("nan"), dtype=torch.bfloat16, device=DEV)
    if pad == 16:  # rows at the start of each padded row: 32-byte aligned
        out = buf[:, :hq * d].view(T, hq, d)
        rest = buf[:, hq * d:]
    else:  # rows 16 bytes into each padded row: 16- but not 32-byte aligned
        out = torch.as_strided(buf, (T, hq, d), (hq * d + pad, d, 1), storage_offset=pad)
        rest = buf[:, :pad]
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    H.run_step(lay, g, H.device_meta(lay, DEV), err=err, out=out)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    H.assert_close(H.f64(out), H.oracle_full(lay, ts), f"padded rows {pad}")
    assert torch.isnan(rest.float()).all(), "a kernel wrote outside the output rows"


@pytest.mark.parametrize("cfg", [3, 4, 6])
def test_prefill_full_size_both_kernels_agree(cfg, monkeypatch):
    # the tensor-core and the general kernel on the same full-size batch
    lay = workloads.config_layout(cfg, 0)
    g = workloads.make_tensors(lay, seed=0, device=DEV)
    md = H.device_meta(lay, DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    monkeypatch.delenv("PA_PREFILL_IMPL", raising=False)
    out_tc = H.run_step(lay, g, md, err=err).clone()
    monkeypatch.setenv("PA_PREFILL_IMPL", "mma")
    out_mma = H.run_step(lay, g, md, err=err).clone()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # the prefill rows (the decode rows run the same decode kernel either way)
    rows = slice(int(lay.query_start_loc[lay.num_decode_seqs]), None)
    d = (out_tc[rows].float() - out_mma[rows].float()).abs()
    assert torch.isfinite(out_tc.float()).all()
    assert d.max().item() <= 2e-2 and d.mean().item() <= 2e-3


def test_workspace_reused_across_calls():
    # the prefill work queue lives in the workspace header and must restart
    # from zero on every call, whatever the previous call left there
    lay = _prefill_cases()[0]
    ts = workloads.make_tensors(lay, seed=12, poison=True)
    g = {k: v.to(DEV) for k, v in ts.items()}
    md = H.device_meta(lay, DEV)
    need = pa.workspace_size(lay.num_decode_seqs, lay.num_q_heads, lay.num_kv_heads,
                             lay.head_dim, lay.max_seq_len)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device=DEV)
    out1 = H.run_step(lay, g, md, workspace=ws).clone()
    out2 = H.run_step(lay, g, md, workspace=ws).clone()
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    H.assert_close(H.f64(out1), H.oracle_full(lay, ts), "reused workspace")


def test_mixed_step_side_by_side_is_bitwise_identical(monkeypatch):
    # decode rows beside the prefill kernel (default) or after it: same bits
    lay = workloads.custom_layout("mix", [900, 40, 3000, 12, 0, 700], [1, 1, 1, 1, 300, 150], 16, 4,
                                  128, 16, 600, 41)
    ts = workloads.make_tensors(lay, seed=13, poison=True)
    g = {k: v.to(DEV) for k, v in ts.items()}
    md = H.device_meta(lay, DEV)
    monkeypatch.delenv("PA_MIXED_DECODE_SMS", raising=False)
    out1 = H.run_step(lay, g, md).clone()
    monkeypatch.setenv("PA_MIXED_DECODE_SMS", "0")
    out2 = H.run_step(lay, g, md).clone()
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    H.assert_close(H.f64(out1), H.oracle_full(lay, ts), "mixed")


def test_step_replays_from_a_cuda_graph():
    # every call is stream-ordered and allocation-free, so a whole step
    # (copy-on-write copies, scatter, attention with decode beside prefill)
    # can be captured once and replayed
    lay = workloads.shared_prefix_layout(0, num_seqs=6, prompt=512, tail_max=40, num_q_heads=16,
                                         num_kv_heads=4, num_blocks=256)
    lay2 = workloads.custom_layout("gmix", [300, 60, 0], [1, 1, 200], 16, 4, 128, 16, 64, 7)
    for L in (lay, lay2):
        ts = workloads.make_tensors(L, seed=14, poison=True)
        g = {k: v.to(DEV) for k, v in ts.items()}
        md = H.device_meta(L, DEV)
        need = pa.workspace_size(L.num_decode_seqs, L.num_q_heads, L.num_kv_heads, L.head_dim,
                                 L.max_seq_len)
        ws = torch.empty(need, dtype=torch.uint8, device=DEV)
        out = torch.empty_like(g["q"])
        H.run_step(L, g, md, out=out, workspace=ws)          # first call: per-device set-up
        torch.cuda.synchronize()
        expect = out.clone()
        out.zero_()
        graph = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(graph, stream=s):
                H.run_step(L, g, md, out=out, workspace=ws)
        torch.cuda.current_stream().wait_stream(s)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), expect.view(torch.int16))
