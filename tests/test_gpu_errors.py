"""Failure detection on the GPU path without faulting the GPU: host-side
argument errors come back as status codes with nothing launched, and
device-side inconsistencies set bits in the error flag while every access
stays inside the buffers (bad rows are skipped, not dereferenced)."""

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


def _setup(lay):
    ts = workloads.make_tensors(lay, seed=0)
    g = {k: v.to(DEV) for k, v in ts.items()}
    return g, H.device_meta(lay, DEV), torch.zeros(1, dtype=torch.int32, device=DEV)


def test_bad_slot_sets_flag_and_writes_nothing_else():
    lay = workloads.config_layout(1, 0)
    g, md, err = _setup(lay)
    before = g["k_cache"].clone()
    slots = md["slots"].clone()
    slots[3] = lay.num_blocks * lay.block_size + 5       # past the pool
    slots[4] = -1                                         # skipped on purpose
    pa.write_kv(g["k"], g["v"], g["k_cache"], g["v_cache"], slots, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEV_BAD_SLOT
    Hkv, D = lay.num_kv_heads, lay.head_dim
    flat_new = g["k_cache"].view(-1, Hkv, D)
    flat_old = before.view(-1, Hkv, D)
    good = [0, 1, 2, 5, 6]
    for t in good:
        assert torch.equal(flat_new[lay.slot_mapping[t]], g["k"][t])
    untouched = np.ones(lay.num_blocks * lay.block_size, bool)
    untouched[lay.slot_mapping[good]] = False
    idx = torch.from_numpy(np.nonzero(untouched)[0]).to(DEV)
    assert torch.equal(flat_new[idx], flat_old[idx])


def test_bad_block_id_sets_flag():
    lay = workloads.config_layout(1, 0)
    g, md, err = _setup(lay)
    bt = md["bt"].clone()
    bt[0, 0] = lay.num_blocks + 3                         # decode row B
    bt[2, 1] = -1                                         # prefill row A, live position 4
    pa.attention(g["q"], g["k_cache"], g["v_cache"], md["qsl"], md["seq_lens"], bt,
                 num_decode_seqs=2, max_query_len=5, max_seq_len=8, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEV_BAD_BLOCK


def test_bad_lengths_set_flag():
    lay = workloads.config_layout(1, 0)
    g, md, err = _setup(lay)
    sl = md["seq_lens"].clone()
    sl[2] = 3                                             # A: 5 new tokens but seq_len 3
    pa.attention(g["q"], g["k_cache"], g["v_cache"], md["qsl"], sl, md["bt"],
                 num_decode_seqs=2, max_query_len=5, max_seq_len=8, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEV_BAD_LEN
    err.zero_()
    sl = md["seq_lens"].clone()
    sl[0] = 4 * lay.block_size                            # beyond B's 2-block table row
    pa.attention(g["q"], g["k_cache"], g["v_cache"], md["qsl"], sl, md["bt"],
                 num_decode_seqs=2, max_query_len=5, max_seq_len=64, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEV_BAD_LEN


def test_decode_row_with_several_tokens_sets_flag():
    lay = workloads.config_layout(1, 0)
    g, md, err = _setup(lay)
    # claim all three rows are decodes: A has 5 tokens
    pa.attention(g["q"], g["k_cache"], g["v_cache"], md["qsl"], md["seq_lens"], md["bt"],
                 num_decode_seqs=3, max_query_len=5, max_seq_len=8, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEV_BAD_DECODE


def test_bad_copy_pair_sets_flag():
    lay = workloads.config_layout(1, 0)
    g, md, err = _setup(lay)
    pairs = torch.tensor([[1, lay.num_blocks]], dtype=torch.int32, device=DEV)
    before = g["k_cache"].clone()
    pa.copy_blocks(g["k_cache"], g["v_cache"], pairs, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEV_BAD_PAIR
    assert torch.equal(before, g["k_cache"])


def test_bad_swap_pair_sets_flag():
    shape = (4, 16, 2, 64)
    src = torch.randn(shape, device=DEV).to(torch.bfloat16)
    dk = torch.zeros(shape, dtype=torch.bfloat16).pin_memory()
    dv = torch.zeros(shape, dtype=torch.bfloat16).pin_memory()
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pairs = torch.tensor([[0, 4], [4, 1], [-1, 2], [2, 3]], dtype=torch.int32, device=DEV)
    pa.swap_blocks(src, src, dk, dv, pairs, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEV_BAD_PAIR
    assert torch.equal(dk[3], src[2].cpu())               # the valid pair still moved
    assert not dk[:3].any() and not dv[:3].any()


def test_workspace_too_small_is_refused():
    lay = workloads.custom_layout("splits", [20000], [1], 8, 1, 128, 16, 1300, 8)
    g, md, err = _setup(lay)
    need = pa.workspace_size(1, 8, 1, 128, lay.max_seq_len)
    assert need > 0
    small = torch.empty(need - 16, dtype=torch.uint8, device=DEV)
    with pytest.raises(pa.PaError, match="WORKSPACE"):
        pa.attention(g["q"], g["k_cache"], g["v_cache"], md["qsl"], md["seq_lens"], md["bt"],
                     num_decode_seqs=1, max_query_len=1, max_seq_len=lay.max_seq_len,
                     workspace=small, err=err)


def test_unsupported_head_dim_is_refused():
    lay = workloads.custom_layout("d32", [3], [2], 2, 2, 32, 4, 4, 0)
    g, md, err = _setup(lay)
    with pytest.raises(pa.PaError, match="UNSUPPORTED"):
        pa.attention(g["q"], g["k_cache"], g["v_cache"], md["qsl"], md["seq_lens"], md["bt"],
                     num_decode_seqs=0, max_query_len=2, max_seq_len=5)


@pytest.mark.parametrize("fused", [False, True], ids=["two-calls", "fused-scatter"])
def test_pipeline_wait_gives_up_then_next_call_is_exact(fused):
    # The tensor-core prefill waits on shared-memory barriers for its copies
    # and products.  A 1 ns limit makes its first waits run out on purpose:
    # the kernel must set DEV_TIMEOUT, drain what it has in flight, free its
    # tensor memory and return, leaving the context usable.  The next call,
    # with the default limit, must then match the oracle.
    lay = workloads.custom_layout("timeout", [0, 0, 40, 0], [700, 300, 129, 64], 8, 2, 128, 16,
                                  400, 21)
    ts = workloads.make_tensors(lay, seed=5, poison=True)            # CPU copies for the oracle
    g = {k: v.to(DEV) for k, v in ts.items()}
    md = H.device_meta(lay, DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)

    def step():
        kw = dict(num_decode_seqs=lay.num_decode_seqs, max_query_len=lay.max_query_len,
                  max_seq_len=lay.max_seq_len, scale=lay.scale, err=err)
        if fused:
            return pa.write_kv_attention(g["q"], g["k"], g["v"], g["k_cache"], g["v_cache"],
                                         md["slots"], md["qsl"], md["seq_lens"], md["bt"], **kw)
        pa.write_kv(g["k"], g["v"], g["k_cache"], g["v_cache"], md["slots"], err=err)
        return pa.attention(g["q"], g["k_cache"], g["v_cache"], md["qsl"], md["seq_lens"],
                            md["bt"], **kw)

    prev = pa.set_wait_limit_ns(1)
    try:
        step()
        torch.cuda.synchronize()                     # the call returned; no CUDA error
    finally:
        pa.set_wait_limit_ns(prev)
    assert int(err.item()) & pa.DEV_TIMEOUT
    err.zero_()
    out = step()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    H.assert_close(H.f64(out), H.oracle_full(lay, ts), "after a timed-out call")
