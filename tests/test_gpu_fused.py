"""GPU: the fused scatter + attention call (pa_write_kv_attention) against
pa_write_kv followed by pa_attention on the same inputs: both caches
bit-identical, outputs within the attention tolerance of the fp64 oracle and
of the two-call path (bit-identical where the two group keys into the same
tiles: prompts without history).

The pages run the scatter and the attention back to back ("vLLM 原理" §3.7).
On a prefill-only step the fused call is one tensor-core launch that takes
the new tokens' K/V from the inputs and stores their rows; steps with decode
rows (and steps on the general kernel) scatter first.  Cases with
num_decode_seqs = 0 and a block size of 8 or more exercise the one-launch
path, histories on and off every alignment included."""

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


def _cases():
    rng = np.random.default_rng(77)
    out = [workloads.config_layout(1, 0), workloads.literal_layout()]
    specs = [
        # (name, Hq, Hkv, D, bs, decodes, prefills, max cached)
        ("f_d128_bs16", 8, 2, 128, 16, 4, 4, 700),
        ("f_d64_bs16_g1", 4, 4, 64, 16, 3, 3, 400),
        ("f_d128_bs8", 8, 2, 128, 8, 2, 3, 300),
        ("f_d128_bs32_g8", 16, 2, 128, 32, 2, 3, 500),
        ("f_d128_bs64", 8, 4, 128, 64, 2, 2, 600),
        ("f_d128_bs128", 4, 1, 128, 128, 2, 2, 900),
        ("f_d64_bs256", 4, 2, 64, 256, 1, 3, 900),
        ("f_d128_bs4_general", 8, 2, 128, 4, 2, 2, 200),
        ("f_d128_bs1_general", 4, 2, 128, 1, 2, 2, 60),
    ]
    for i, (name, hq, hkv, d, bs, nd, npf, cmax) in enumerate(specs):
        cached = list(rng.integers(1, cmax, nd)) + list(rng.integers(0, cmax, npf))
        queries = [1] * nd + list(rng.integers(1, 300, npf))
        cached[-1] = 0                                     # one plain prompt
        nb = sum(-(-(c + q) // bs) for c, q in zip(cached, queries)) + 9
        out.append(workloads.custom_layout(name, cached, queries, hq, hkv, d, bs, nb, 300 + i))
    # chunk boundaries off every alignment, an empty sequence, single-token prompts
    out.append(workloads.custom_layout("f_ragged", [129, 1, 255, 16, 0, 7],
                                       [200, 131, 1, 0, 130, 257], 8, 2, 128, 16, 120, 9))
    out.append(workloads.custom_layout("f_L1", [0, 0, 5], [1, 1, 1], 4, 2, 128, 16, 8, 10))
    out.append(workloads.custom_layout("f_negscale", [30, 0], [1, 90], 4, 2, 128, 16, 16, 11,
                                       scale=-0.1))
    return out


def _run(lay, fused, seed, num_decode=None):
    ts = workloads.make_tensors(lay, seed=seed, poison=True)
    g = {k: v.to(DEV) for k, v in ts.items()}
    md = H.device_meta(lay, DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    nd = lay.num_decode_seqs if num_decode is None else num_decode
    if fused:
        if len(lay.cow_pairs):
            pa.copy_blocks(g["k_cache"], g["v_cache"], md["pairs"], err=err)
        out = pa.write_kv_attention(g["q"], g["k"], g["v"], g["k_cache"], g["v_cache"],
                                    md["slots"], md["qsl"], md["seq_lens"], md["bt"],
                                    num_decode_seqs=nd, max_query_len=lay.max_query_len,
                                    max_seq_len=lay.max_seq_len, scale=lay.scale, err=err)
    else:
        out = H.run_step(lay, g, md, err=err, num_decode=nd)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return ts, out, g


def _bits(t):
    return t.view(torch.int16)


def _close(a, b):
    d = (a.float() - b.float()).abs()
    assert torch.isfinite(a.float()).all() and torch.isfinite(b.float()).all()
    assert d.max().item() <= H.MAX_ABS and d.mean().item() <= H.MAX_ABS / 10


@pytest.mark.parametrize("lay", _cases(), ids=lambda l: l.name)
def test_fused_matches_the_two_calls(lay):
    _, o1, g1 = _run(lay, False, 21)
    ts, o2, g2 = _run(lay, True, 21)
    rows = [t for s in range(lay.num_seqs)
            for t in range(lay.query_start_loc[s], lay.query_start_loc[s + 1])]
    assert torch.equal(_bits(g1["k_cache"]), _bits(g2["k_cache"]))
    assert torch.equal(_bits(g1["v_cache"]), _bits(g2["v_cache"]))
    _close(o1[rows], o2[rows])
    H.assert_close(H.f64(o2)[rows], H.oracle_full(lay, ts)[rows], f"fused/{lay.name}")


@pytest.mark.parametrize("lay", _cases()[2:5], ids=lambda l: l.name)
def test_fused_decode_rows_on_prefill_kernel(lay):
    # num_decode_seqs = 0: every row, single tokens included, goes to the prefill kernel
    _, o1, g1 = _run(lay, False, 22, num_decode=0)
    ts, o2, g2 = _run(lay, True, 22, num_decode=0)
    _close(o1, o2)
    assert torch.equal(_bits(g1["k_cache"]), _bits(g2["k_cache"]))
    H.assert_close(H.f64(o2), H.oracle_full(lay, ts), f"fused-nodecode/{lay.name}")


@pytest.mark.parametrize("cfg", [2, 3, 4, 5, 6])
def test_fused_full_size(cfg):
    lay = workloads.config_layout(cfg, 0)
    outs, caches = [], []
    full = None
    for fused in (False, True):
        g = workloads.make_tensors(lay, seed=3, device=DEV)
        md = H.device_meta(lay, DEV)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        if fused and cfg in (2, 3, 4):
            full = H.FullOracle(lay, g)        # every row of the fused step vs the oracle
        if fused:
            if len(lay.cow_pairs):
                pa.copy_blocks(g["k_cache"], g["v_cache"], md["pairs"], err=err)
            o = pa.write_kv_attention(g["q"], g["k"], g["v"], g["k_cache"], g["v_cache"],
                                      md["slots"], md["qsl"], md["seq_lens"], md["bt"],
                                      num_decode_seqs=lay.num_decode_seqs,
                                      max_query_len=lay.max_query_len,
                                      max_seq_len=lay.max_seq_len, scale=lay.scale, err=err)
        else:
            o = H.run_step(lay, g, md, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        outs.append(o)
        caches.append((g["k_cache"], g["v_cache"]))
        del g
    if (lay.cached_lens[lay.num_decode_seqs:] == 0).all():
        assert torch.equal(_bits(outs[0]), _bits(outs[1]))  # same key tiles: same bits
    else:
        _close(outs[0], outs[1])
    assert torch.equal(_bits(caches[0][0]), _bits(caches[1][0]))
    assert torch.equal(_bits(caches[0][1]), _bits(caches[1][1]))
    if full is not None:
        full.check(outs[1], f"fused/{lay.name}")


def test_fused_bad_slot_sets_flag():
    lay = workloads.custom_layout("f_bad", [40, 0], [1, 70], 8, 2, 128, 16, 16, 12)
    ts = workloads.make_tensors(lay, seed=4, poison=False)
    g = {k: v.to(DEV) for k, v in ts.items()}
    md = H.device_meta(lay, DEV)
    for t in (0, 5):                                   # a decode row and a prefill row
        slots = md["slots"].clone()
        slots[t] = lay.num_blocks * lay.block_size
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        pa.write_kv_attention(g["q"], g["k"], g["v"], g["k_cache"], g["v_cache"], slots,
                              md["qsl"], md["seq_lens"], md["bt"],
                              num_decode_seqs=lay.num_decode_seqs,
                              max_query_len=lay.max_query_len, max_seq_len=lay.max_seq_len,
                              err=err)
        torch.cuda.synchronize()
        assert int(err.item()) & pa.DEV_BAD_SLOT
