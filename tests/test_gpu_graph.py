"""Steps captured into a CUDA graph give the same results as the same calls
run eagerly.  Every call is stream-ordered with no host sync, so a serving
loop can capture one step and replay it; a mixed step forks its decode and
prefill sides onto the library's two side streams and joins them back, which
the capture records.  The kernels are deterministic, so the replayed output
is compared bitwise with the eager one (and the eager one is checked against
the oracle in the parity tests)."""

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
    return [
        # decode rows and two prefill chunks: the side-by-side dispatch
        workloads.custom_layout("mixed", [300, 900, 40, 1200, 64, 0], [1, 1, 1, 1, 700, 333],
                                16, 4, 128, 16, 400, 3),
        # prefill only (persistent tensor-core kernel and its work counter)
        workloads.custom_layout("prefill", [0, 0, 0], [500, 130, 47], 8, 2, 128, 16, 64, 4),
        # decode only (split-KV partials and their combine)
        workloads.custom_layout("decode", [5000, 17, 800], [1, 1, 1], 8, 8, 64, 16, 400, 5),
    ]


@pytest.mark.parametrize("lay", _layouts(), ids=lambda l: l.name)
@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused"])
def test_graph_replay_matches_eager(lay, fused):
    g = workloads.make_tensors(lay, seed=11, device=DEV)
    md = H.device_meta(lay, DEV)
    need = pa.workspace_size(lay.num_decode_seqs, lay.num_q_heads, lay.num_kv_heads,
                             lay.head_dim, lay.max_seq_len)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kc0, vc0 = g["k_cache"].clone(), g["v_cache"].clone()

    def step(out):
        if fused:
            pa.write_kv_attention(g["q"], g["k"], g["v"], g["k_cache"], g["v_cache"], md["slots"],
                                  md["qsl"], md["seq_lens"], md["bt"],
                                  num_decode_seqs=lay.num_decode_seqs,
                                  max_query_len=lay.max_query_len, max_seq_len=lay.max_seq_len,
                                  scale=lay.scale, out=out, workspace=ws, err=err)
        else:
            H.run_step(lay, g, md, err=err, out=out, workspace=ws)

    eager = torch.empty_like(g["q"])
    step(eager)
    torch.cuda.synchronize()
    kc1, vc1 = g["k_cache"].clone(), g["v_cache"].clone()

    replay = torch.full_like(g["q"], float("nan"))
    g["k_cache"].copy_(kc0)
    g["v_cache"].copy_(vc0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step(replay)
    torch.cuda.synchronize()
    for _ in range(3):
        replay.fill_(float("nan"))  # every replay must write every row again
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(replay.view(torch.int16), eager.view(torch.int16))
    assert int(err.item()) == 0
    assert torch.equal(g["k_cache"].view(torch.int16), kc1.view(torch.int16))
    assert torch.equal(g["v_cache"].view(torch.int16), vc1.view(torch.int16))
    assert np.isfinite(H.f64(replay)).all()


@pytest.mark.parametrize("g8", [True, False], ids=["tensor_core_prefix", "mma_prefix"])
def test_cascade_graph_replay_matches_eager(g8):
    # shared-prompt decode: prefix pass, own keys and combine in one capture
    hq, hkv = (16, 2) if g8 else (8, 4)
    lay = workloads.shared_prefix_layout(3, num_seqs=5, prompt=640, tail_max=40, num_q_heads=hq,
                                         num_kv_heads=hkv, head_dim=128, block_size=16,
                                         num_blocks=120)
    tabs = [list(t) for t in lay.tables]
    pb = 0
    while all(len(t) > pb for t in tabs) and len({t[pb] for t in tabs}) == 1:
        pb += 1
    g = workloads.make_tensors(lay, seed=12, device=DEV)
    md = H.device_meta(lay, DEV)
    need = pa.cascade_workspace_size(lay.num_seqs, hq, hkv, 128, lay.max_seq_len, pb,
                                     lay.block_size)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)

    def step(out):
        pa.attention_cascade(g["q"], g["k_cache"], g["v_cache"], md["qsl"], md["seq_lens"],
                             md["bt"], prefix_blocks=pb, max_seq_len=lay.max_seq_len,
                             scale=lay.scale, out=out, workspace=ws, err=err)

    eager = torch.empty_like(g["q"])
    step(eager)
    torch.cuda.synchronize()
    replay = torch.full_like(g["q"], float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step(replay)
    torch.cuda.synchronize()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(replay.view(torch.int16), eager.view(torch.int16))


def test_work_queue_needs_no_zeroing():
    # The persistent prefill kernel draws items from two words in the
    # workspace header that the host never zeroes: each launch tags them, a
    # word holding another launch's tag (or any bytes) is reset by the kernel,
    # and the last CTA leaves them ready for a replay of the same launch.  Two
    # captured steps with more items than CTAs share one workspace and replay
    # alternately, some replays after the header was overwritten with ones,
    # and an eager call follows a clobbered header too.
    lays = [workloads.custom_layout("qa", [0] * 6, [700, 500, 300, 129, 64, 1000], 32, 8, 128,
                                    16, 400, 21),
            workloads.custom_layout("qb", [200, 0, 900], [640, 1500, 77], 32, 8, 128, 16, 600, 22)]
    need = max(pa.workspace_size(0, l.num_q_heads, l.num_kv_heads, l.head_dim, l.max_seq_len)
               for l in lays)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    runs = []
    for lay in lays:
        g = workloads.make_tensors(lay, seed=13, device=DEV)
        md = H.device_meta(lay, DEV)
        pa.write_kv(g["k"], g["v"], g["k_cache"], g["v_cache"], md["slots"], err=err)
        out = torch.full_like(g["q"], float("nan"))

        def attn(lay=lay, g=g, md=md, out=out):
            pa.attention(g["q"], g["k_cache"], g["v_cache"], md["qsl"], md["seq_lens"], md["bt"],
                         num_decode_seqs=0, max_query_len=lay.max_query_len,
                         max_seq_len=lay.max_seq_len, scale=lay.scale, out=out, workspace=ws,
                         err=err)

        attn()
        torch.cuda.synchronize()
        runs.append((attn, out, out.clone()))
    graphs = []
    for attn, _, _ in runs:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            attn()
        torch.cuda.synchronize()
        graphs.append(gr)
    for rep in range(4):
        for (attn, out, expect), gr in zip(runs, graphs):
            if rep % 2:
                ws[:64].fill_(255)
            out.fill_(float("nan"))
            gr.replay()
            torch.cuda.synchronize()
            assert torch.equal(out.view(torch.int16), expect.view(torch.int16)), rep
    attn, out, expect = runs[1]
    ws[:64].fill_(255)
    out.fill_(float("nan"))
    attn()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), expect.view(torch.int16))
    assert int(err.item()) == 0
