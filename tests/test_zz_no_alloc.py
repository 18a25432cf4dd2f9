"""pa_attention_noalloc: attention for callers that cannot allocate device memory.

Some callers of this library have no allocator to call: code embedded in a
host application that owns every device allocation, a runtime whose device
memory is reserved up front, or a loop that must not call cudaMalloc because
it can wait for the whole device.  pa_attention_noalloc takes no workspace;
its split-KV scratch is a static device array inside the library.  These
tests call it through the C ABI and check that it gives the same output as
pa_attention with a caller-provided workspace and agrees with the fp64
oracle, on two calls in a row (the second call finds the first call's
partial results still in the array), and that it refuses a batch that needs
more scratch than the array holds.

This file is collected last on purpose: it only adds an entry point and must
pass both alone in a fresh process and after every other test.
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


def _layouts():
    # both batches have long decode rows, so both need split-KV scratch
    a = workloads.custom_layout("noalloc-a", [9000, 20000, 300, 40], [1, 1, 1, 25], 8, 1, 128, 16,
                                2100, 31)
    b = workloads.custom_layout("noalloc-b", [15000, 700, 12000], [1, 1, 1], 16, 2, 128, 16,
                                1800, 32)
    return [a, b]


def test_noalloc_matches_attention_on_two_calls_in_a_row():
    for i, lay in enumerate(_layouts()):
        need = pa.workspace_size(lay.num_decode_seqs, lay.num_q_heads, lay.num_kv_heads,
                                 lay.head_dim, lay.max_seq_len)
        # more than the header alone: the decode rows need split-KV partials
        header = pa.workspace_size(0, lay.num_q_heads, lay.num_kv_heads, lay.head_dim,
                                   lay.max_seq_len)
        assert header < need <= pa.NOALLOC_SCRATCH_BYTES
        ts = workloads.make_tensors(lay, seed=40 + i, poison=True)    # CPU copies for the oracle
        g = {k: v.to(DEV) for k, v in ts.items()}
        md = H.device_meta(lay, DEV)
        pa.write_kv(g["k"], g["v"], g["k_cache"], g["v_cache"], md["slots"])
        expect = pa.attention(g["q"], g["k_cache"], g["v_cache"], md["qsl"], md["seq_lens"],
                              md["bt"], num_decode_seqs=lay.num_decode_seqs,
                              max_query_len=lay.max_query_len, max_seq_len=lay.max_seq_len,
                              scale=lay.scale)
        torch.cuda.synchronize()
        oracle = H.oracle_full(lay, ts)
        for call in range(2):
            out = torch.empty_like(g["q"])
            err = torch.zeros(1, dtype=torch.int32, device=DEV)
            before = pa.kernel_launches()
            pa.attention_noalloc(g["q"], g["k_cache"], g["v_cache"], md["qsl"], md["seq_lens"],
                                 md["bt"], out=out, num_decode_seqs=lay.num_decode_seqs,
                                 max_query_len=lay.max_query_len, max_seq_len=lay.max_seq_len,
                                 scale=lay.scale, err=err)
            torch.cuda.synchronize()
            launched = pa.kernel_launches() - before
            assert int(err.item()) == 0
            # decode and the split combine (plus the prefill kernel for prefill rows):
            # the partials really go through the static array
            has_prefill = lay.num_seqs > lay.num_decode_seqs
            assert launched == 2 + int(has_prefill), launched
            H.assert_close(H.f64(out), H.f64(expect), f"{lay.name} call {call}")
            H.assert_close(H.f64(out), oracle, f"{lay.name} call {call} vs oracle")


def test_noalloc_refuses_batches_beyond_its_scratch():
    # find a decode batch whose partials exceed the static array
    nd = None
    for n in range(400, 4000, 25):
        if pa.workspace_size(n, 16, 1, 128, 1024) > pa.NOALLOC_SCRATCH_BYTES:
            nd = n
            break
    assert nd is not None
    q = torch.zeros((nd, 16, 128), dtype=torch.bfloat16, device=DEV)
    cache = torch.zeros((4, 16, 1, 128), dtype=torch.bfloat16, device=DEV)
    qsl = torch.arange(nd + 1, dtype=torch.int32, device=DEV)
    sl = torch.ones(nd, dtype=torch.int32, device=DEV)
    bt = torch.zeros((nd, 1), dtype=torch.int32, device=DEV)
    with pytest.raises(pa.PaError, match="WORKSPACE"):
        pa.attention_noalloc(q, cache, cache, qsl, sl, bt, out=torch.empty_like(q),
                             num_decode_seqs=nd, max_query_len=1, max_seq_len=1024)
