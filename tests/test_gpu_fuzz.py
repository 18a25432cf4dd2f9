"""Seeded random sweep of small ragged steps against the fp64 oracle.

Each case draws a head layout (group sizes 1-16), head_dim, block size, a
mix of decode rows and prefill chunks with random histories and lengths
(including chunk tails of a few tokens and of exactly 64, 65 and 128), and
runs copy-free write + attention on a NaN-poisoned pool; a second sweep runs
shared-prompt decode batches through pa_attention_cascade.  Same tolerance as
every attention test.
"""

import numpy as np
import pytest
import torch

import paged_kv_cache_133_gb300 as pa
import workloads
from tests import _helpers as H

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

HEADS = [(4, 4), (8, 2), (16, 2), (12, 4), (32, 8), (8, 1), (16, 4), (6, 2)]
DIMS = [64, 128]
BLOCKS = [1, 2, 8, 16, 32, 64, 128]
SPECIAL_Q = [1, 2, 7, 63, 64, 65, 127, 128, 129, 200]


@pytest.fixture(scope="module", autouse=True)
def _built():
    H.ensure_built()
    torch.cuda.set_device(0)


def _random_layout(seed):
    rng = np.random.default_rng(9000 + seed)
    hq, hkv = HEADS[rng.integers(len(HEADS))]
    d = DIMS[rng.integers(len(DIMS))]
    bs = BLOCKS[rng.integers(len(BLOCKS))]
    nd = int(rng.integers(0, 5))
    npf = int(rng.integers(0 if nd else 1, 5))
    cached = [int(rng.integers(0, 400)) for _ in range(nd)]
    queries = [1] * nd
    for _ in range(npf):
        cached.append(int(rng.integers(0, 300)) if rng.random() < 0.6 else 0)
        queries.append(int(SPECIAL_Q[rng.integers(len(SPECIAL_Q))]) if rng.random() < 0.5
                       else int(rng.integers(1, 260)))
    nb = sum(-(-(c + q) // bs) for c, q in zip(cached, queries)) + int(rng.integers(1, 9))
    return workloads.custom_layout(f"fuzz{seed}_h{hq}-{hkv}_d{d}_bs{bs}", cached, queries, hq, hkv,
                                   d, bs, nb, 700 + seed)


@pytest.mark.parametrize("seed", range(24))
def test_random_step_matches_oracle(seed):
    lay = _random_layout(seed)
    ts = workloads.make_tensors(lay, seed=seed, poison=True)
    expect = H.oracle_full(lay, ts)
    g = {k: v.to(DEV) for k, v in ts.items()}
    md = H.device_meta(lay, DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = H.run_step(lay, g, md, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    H.assert_close(H.f64(out), expect, lay.name)


def _random_shared(seed):
    rng = np.random.default_rng(9500 + seed)
    hq, hkv = HEADS[rng.integers(len(HEADS))]
    d = DIMS[rng.integers(len(DIMS))]
    bs = [8, 16, 32, 64][rng.integers(4)]
    nprompt = int(rng.integers(2, 40))
    n = int(rng.integers(2, 12))
    tail = int(rng.integers(1, 120))
    nb = nprompt + n * (-(-(tail + 1) // bs) + 2) + 5
    lay = workloads.shared_prefix_layout(seed, num_seqs=n, prompt=nprompt * bs, tail_max=tail,
                                         num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                                         block_size=bs, num_blocks=nb)
    lay.name = f"shared{seed}_h{hq}-{hkv}_d{d}_bs{bs}_p{nprompt}_n{n}"
    return lay


@pytest.mark.parametrize("seed", range(12))
def test_random_shared_prefix_matches_oracle(seed):
    lay = _random_shared(seed)
    tabs = [list(t) for t in lay.tables]
    pb = 0
    while all(len(t) > pb for t in tabs) and len({t[pb] for t in tabs}) == 1:
        pb += 1
    ts = workloads.make_tensors(lay, seed=seed, poison=True)
    expect = H.oracle_full(lay, ts)
    g = {k: v.to(DEV) for k, v in ts.items()}
    md = H.device_meta(lay, DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.copy_blocks(g["k_cache"], g["v_cache"], md["pairs"], err=err)
    pa.write_kv(g["k"], g["v"], g["k_cache"], g["v_cache"], md["slots"], err=err)
    out = pa.attention_cascade(g["q"], g["k_cache"], g["v_cache"], md["qsl"], md["seq_lens"],
                               md["bt"], prefix_blocks=pb, max_seq_len=lay.max_seq_len,
                               scale=lay.scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    H.assert_close(H.f64(out), expect, lay.name)
