"""GPU parity of the shared-prefix (cascade) decode call against the fp64 oracle.

Layouts: several decode sequences share a cached prompt's blocks (ref counted,
with the last prompt block copied on write), then own private tails.  The
call reads the shared blocks once per group of query rows and merges the
partials with each sequence's own keys; the result must match the oracle's
plain attention (same tolerance as every attention test) on NaN-poisoned
pools, and pa_attention on the same inputs.
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


def _shared(name, num_seqs, prompt, tail_max, hq, hkv, d, bs, seed):
    nprompt = -(-prompt // bs)
    tails_blocks = num_seqs * (-(-(tail_max + 1) // bs) + 2)
    lay = workloads.shared_prefix_layout(seed, num_seqs=num_seqs, prompt=prompt, tail_max=tail_max,
                                         num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                                         block_size=bs, num_blocks=nprompt + tails_blocks + 9)
    lay.name = name
    return lay


def _cases():
    # Prompts fill whole blocks: the copy-on-write of the last prompt block
    # then carries prompt tokens only, and every tail starts in a block of its
    # own (a partial last block would carry the owner's tail into the copies).
    return [
        # (layout; prefix blocks = the prompt's blocks before the copied last one)
        _shared("g8_d128_bs16", 6, 704, 60, 16, 2, 128, 16, 1),
        _shared("g1_d128_bs16", 9, 512, 40, 8, 8, 128, 16, 2),
        _shared("g4_d64_bs8", 5, 336, 90, 8, 2, 64, 8, 3),
        _shared("g8_rows_over_64", 20, 256, 30, 16, 2, 128, 16, 4),     # 160 rows per kv head
        _shared("g16_d128_bs64", 3, 1536, 200, 32, 2, 128, 64, 5),
        _shared("g2_d128_bs1", 4, 90, 20, 4, 2, 128, 1, 6),
        _shared("long_prefix", 4, 6000, 100, 16, 2, 128, 16, 7),       # several prefix chunks
        _shared("g8_d64_bs16", 7, 896, 50, 16, 2, 64, 16, 8),
        _shared("g32_d128_bs32", 3, 416, 30, 32, 1, 128, 32, 9),
    ]


def _prefix_blocks(lay):
    tabs = [list(t) for t in lay.tables]
    n = 0
    while all(len(t) > n for t in tabs) and len({t[n] for t in tabs}) == 1:
        n += 1
    return n


def _run(lay, g, md, prefix_blocks, err):
    if len(lay.cow_pairs):
        pa.copy_blocks(g["k_cache"], g["v_cache"], md["pairs"], err=err)
    pa.write_kv(g["k"], g["v"], g["k_cache"], g["v_cache"], md["slots"], err=err)
    return pa.attention_cascade(g["q"], g["k_cache"], g["v_cache"], md["qsl"], md["seq_lens"],
                                md["bt"], prefix_blocks=prefix_blocks,
                                max_seq_len=lay.max_seq_len, scale=lay.scale, err=err)


@pytest.mark.parametrize("lay", _cases(), ids=lambda l: l.name)
def test_cascade_matches_oracle(lay):
    pb = _prefix_blocks(lay)
    assert pb >= 1 and pb * lay.block_size < int(lay.seq_lens.min())
    ts = workloads.make_tensors(lay, seed=3, poison=True)
    expect = H.oracle_full(lay, ts)
    g = {k: v.to(DEV) for k, v in ts.items()}
    md = H.device_meta(lay, DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(lay, g, md, pb, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    H.assert_close(H.f64(out), expect, f"cascade/{lay.name}")


@pytest.mark.parametrize("lay", _cases()[:3], ids=lambda l: l.name)
def test_cascade_agrees_with_plain_attention(lay):
    pb = _prefix_blocks(lay)
    g = workloads.make_tensors(lay, seed=4, device=DEV)
    md = H.device_meta(lay, DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out_c = _run(lay, g, md, pb, err).clone()
    plain = pa.attention(g["q"], g["k_cache"], g["v_cache"], md["qsl"], md["seq_lens"], md["bt"],
                         num_decode_seqs=lay.num_seqs, max_query_len=1,
                         max_seq_len=lay.max_seq_len, scale=lay.scale, err=err)
    # no prefix: the call is plain decode attention, bit for bit
    zero = pa.attention_cascade(g["q"], g["k_cache"], g["v_cache"], md["qsl"], md["seq_lens"],
                                md["bt"], prefix_blocks=0, max_seq_len=lay.max_seq_len,
                                scale=lay.scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    H.assert_close(H.f64(out_c), H.f64(plain), f"cascade vs plain/{lay.name}")
    assert torch.equal(zero.view(torch.int16), plain.view(torch.int16))


@pytest.mark.parametrize("lay", [c for c in _cases() if c.num_q_heads // c.num_kv_heads % 8 == 0],
                         ids=lambda l: l.name)
def test_cascade_tensor_core_and_mma_passes_agree(lay, monkeypatch):
    # query heads per kv head a multiple of 8: the prefix pass runs on the
    # tensor-core kernel; PA_CASCADE_IMPL=mma forces the mma.sync pass
    pb = _prefix_blocks(lay)
    g = workloads.make_tensors(lay, seed=8, device=DEV)
    md = H.device_meta(lay, DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out_tc = _run(lay, g, md, pb, err).clone()
    monkeypatch.setenv("PA_CASCADE_IMPL", "mma")
    out_mma = _run(lay, g, md, pb, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    H.assert_close(H.f64(out_tc), H.f64(out_mma), f"tc vs mma/{lay.name}")


def test_cascade_full_size_shared_workload_sampled():
    lay = workloads.config_layout(5, 0)
    pb = _prefix_blocks(lay)
    assert pb == 1023
    g = workloads.make_tensors(lay, seed=0, device=DEV, poison=True)
    md = H.device_meta(lay, DEV)
    rng = np.random.default_rng(55)
    rows = [(int(s), 0) for s in sorted(rng.choice(lay.num_seqs, 6, replace=False))]
    snap = H.Snapshot(lay, g, rows)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(lay, g, md, pb, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.isfinite(out.float()).all()
    H.assert_close(snap.gpu_rows(out), snap.expected(), "cascade/shared")


def test_cascade_sequence_without_own_keys_sets_flag():
    lay = _cases()[0]
    g = workloads.make_tensors(lay, seed=5, device=DEV)
    md = H.device_meta(lay, DEV)
    # a prefix longer than the shortest sequence: that row has no key of its
    # own (the others read blocks the promise does not cover; only the flag
    # is checked)
    short = int(lay.seq_lens.min())
    pb = short // lay.block_size + (1 if short % lay.block_size else 0)
    assert pb * lay.block_size >= short and pb * lay.block_size < lay.max_seq_len
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.attention_cascade(g["q"], g["k_cache"], g["v_cache"], md["qsl"], md["seq_lens"], md["bt"],
                         prefix_blocks=pb, max_seq_len=lay.max_seq_len, scale=lay.scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEV_BAD_LEN


def test_cascade_host_checks():
    lay = _cases()[0]
    g = workloads.make_tensors(lay, seed=6, device=DEV)
    md = H.device_meta(lay, DEV)
    args = (g["q"], g["k_cache"], g["v_cache"], md["qsl"], md["seq_lens"], md["bt"])
    with pytest.raises(pa.PaError, match="INVALID"):
        pa.attention_cascade(*args, prefix_blocks=-1, max_seq_len=lay.max_seq_len)
    too_long = -(-lay.max_seq_len // lay.block_size)
    with pytest.raises(pa.PaError, match="INVALID"):
        pa.attention_cascade(*args, prefix_blocks=too_long, max_seq_len=lay.max_seq_len)
