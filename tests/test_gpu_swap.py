"""GPU parity of the block swap (CPU offload of the KV cache, "LLM 推理引擎
Continuous Batching 与 PagedAttention" §4.4): blocks move between the device
pool and a pool in page-locked host memory, bit-exact against the oracle, and
attention is unchanged after they come back into other device blocks."""

import zlib

import numpy as np
import pytest
import torch

import paged_kv_cache_133_gb300 as pa
import workloads
from oracle import attention as ref
from tests import _helpers as H

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    H.ensure_built()
    torch.cuda.set_device(0)


def _bits(t):
    return t.view(torch.int16).cpu().numpy()


def _pairs(src, dst):
    return torch.from_numpy(np.stack([src, dst], 1).astype(np.int32)).to(DEV)


def _pool(n, shape, where, gen):
    t = torch.randn((n,) + shape, generator=gen, dtype=torch.bfloat16)
    return t.pin_memory() if where == "host" else t.to(DEV)


@pytest.mark.parametrize("shape", [(16, 8, 128), (1, 1, 64), (2, 4, 8), (256, 2, 128), (32, 1, 24)])
@pytest.mark.parametrize("route", ["d2h", "h2d", "d2d"])
def test_swap_matches_oracle_bitwise(shape, route):
    seed = zlib.crc32(repr((shape, route)).encode())
    gen = torch.Generator().manual_seed(seed)
    rng = np.random.default_rng(seed)
    ns, nd = 37, 29
    where_s = "host" if route == "h2d" else "dev"
    where_d = "host" if route == "d2h" else "dev"
    sk, sv = _pool(ns, shape, where_s, gen), _pool(ns, shape, where_s, gen)
    dk, dv = _pool(nd, shape, where_d, gen), _pool(nd, shape, where_d, gen)
    n = 23                                          # ragged: not a multiple of anything
    src = rng.choice(ns, n, replace=False)
    dst = rng.choice(nd, n, replace=False)
    exp_k, exp_v = ref.swap_blocks(_bits(sk), _bits(sv), _bits(dk), _bits(dv),
                                   np.stack([src, dst], 1))
    sk0 = _bits(sk)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.swap_blocks(sk, sv, dk, dv, _pairs(src, dst), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(_bits(dk), exp_k) and np.array_equal(_bits(dv), exp_v)
    assert np.array_equal(_bits(sk), sk0)


def test_swap_out_and_back_keeps_attention():
    rng = np.random.default_rng(21)
    S = 24
    lay = workloads.custom_layout("swap", rng.integers(100, 3000, S), [1] * S, 32, 8, 128, 16,
                                  8000, 21)
    g = workloads.make_tensors(lay, seed=3, device=DEV, poison=True)
    md = H.device_meta(lay, DEV)
    before = H.run_step(lay, g, md).clone()
    torch.cuda.synchronize()
    assert torch.isfinite(before).all()

    # swap out the blocks of every other sequence into a host pool, in random host blocks
    out_seqs = list(range(0, S, 2))
    blocks = np.array([b for s in out_seqs for b in lay.tables[s]])
    n_host = len(blocks) + 57
    host = rng.permutation(n_host)[: len(blocks)]
    hk = torch.full((n_host,) + tuple(g["k_cache"].shape[1:]), 7.0, dtype=torch.bfloat16).pin_memory()
    hv = hk.clone().pin_memory()
    exp_k, exp_v = ref.swap_blocks(_bits(g["k_cache"]), _bits(g["v_cache"]), _bits(hk), _bits(hv),
                                   np.stack([blocks, host], 1))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.swap_blocks(g["k_cache"], g["v_cache"], hk, hv, _pairs(blocks, host), err=err)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(hk), exp_k) and np.array_equal(_bits(hv), exp_v)

    # the device blocks are freed and overwritten; the sequences come back elsewhere
    idx = torch.from_numpy(blocks).to(DEV)
    for c in (g["k_cache"], g["v_cache"]):
        c.index_fill_(0, idx, float("nan"))
    owned = np.zeros(lay.num_blocks, bool)
    owned[lay.owned_blocks()] = True
    free = rng.permutation(np.nonzero(~owned)[0])[: len(blocks)]
    pa.swap_blocks(hk, hv, g["k_cache"], g["v_cache"], _pairs(host, free), err=err)
    remap = dict(zip(blocks.tolist(), free.tolist()))
    bt = lay.block_tables.copy()
    for s in out_seqs:
        bt[s, : len(lay.tables[s])] = [remap[b] for b in lay.tables[s]]
    after = pa.attention(g["q"], g["k_cache"], g["v_cache"], md["qsl"], md["seq_lens"],
                         torch.from_numpy(bt).to(DEV), num_decode_seqs=lay.num_decode_seqs,
                         max_query_len=lay.max_query_len, max_seq_len=lay.max_seq_len,
                         scale=lay.scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(after, before)


def test_swap_full_size_bitwise():
    # 4096 blocks of the decode pool's shape (256 MiB of K+V) out to host and back.
    rng = np.random.default_rng(4)
    shape = (16, 8, 128)
    gen = torch.Generator(device=DEV).manual_seed(4)
    nd, nh, n = 12000, 8192, 4096
    dk = torch.randn((nd,) + shape, generator=gen, device=DEV, dtype=torch.bfloat16)
    dv = torch.randn((nd,) + shape, generator=gen, device=DEV, dtype=torch.bfloat16)
    hk = torch.zeros((nh,) + shape, dtype=torch.bfloat16).pin_memory()
    hv = torch.zeros((nh,) + shape, dtype=torch.bfloat16).pin_memory()
    src, host = rng.choice(nd, n, replace=False), rng.choice(nh, n, replace=False)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    dk0, dv0 = _bits(dk), _bits(dv)
    pa.swap_blocks(dk, dv, hk, hv, _pairs(src, host), err=err)
    torch.cuda.synchronize()
    exp_k, exp_v = ref.swap_blocks(dk0, dv0, np.zeros_like(_bits(hk)), np.zeros_like(_bits(hv)),
                                   np.stack([src, host], 1))
    assert np.array_equal(_bits(hk), exp_k) and np.array_equal(_bits(hv), exp_v)
    back = rng.choice(nd, n, replace=False)
    pa.swap_blocks(hk, hv, dk, dv, _pairs(host, back), err=err)
    torch.cuda.synchronize()
    exp_k, exp_v = ref.swap_blocks(exp_k, exp_v, dk0, dv0, np.stack([host, back], 1))
    assert int(err.item()) == 0
    assert np.array_equal(_bits(dk), exp_k) and np.array_equal(_bits(dv), exp_v)
