"""GPU parity of the 8-bit (E4M3) KV cache: the quantising scatter is
bit-exact against the oracle's codes, and decode attention over the codes
matches the fp64 oracle run on the dequantised cache (same tolerance as the
bf16 path).  Unowned blocks and reserved slots hold the NaN code, so a read
outside a sequence's live keys shows up as a non-finite output."""

import numpy as np
import pytest
import torch

import paged_kv_cache_133_gb300 as pa
import workloads
from oracle import attention as ref
from oracle import fp8
from tests import _helpers as H

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    H.ensure_built()
    torch.cuda.set_device(0)


def _decode_layout(name, n, cmax, hq, hkv, d, bs, seed, cmin=1):
    rng = np.random.default_rng(seed)
    cached = rng.integers(cmin, cmax, n)
    nb = int(sum(-(-(c + 1) // bs) for c in cached)) + 11
    return workloads.custom_layout(name, cached, [1] * n, hq, hkv, d, bs, nb, seed)


def _f32(t):
    return t.float().cpu().numpy()


def _setup(lay, k_scale, v_scale, seed):
    """bf16 tensors drawn by the generator; the cache quantised by the oracle
    (NaN code outside live keys and in the slots about to be written)."""
    ts = workloads.make_tensors(lay, seed=seed, poison=False)
    kc = fp8.quantize(_f32(ts["k_cache"]), k_scale)
    vc = fp8.quantize(_f32(ts["v_cache"]), v_scale)
    live = np.zeros(lay.num_blocks * lay.block_size, bool)
    for s, tab in enumerate(lay.tables):
        for p in range(int(lay.seq_lens[s])):
            live[tab[p // lay.block_size] * lay.block_size + p % lay.block_size] = True
    live[lay.slot_mapping[lay.slot_mapping >= 0]] = False
    shape = kc.shape
    kc = kc.reshape(-1, *shape[2:])
    vc = vc.reshape(-1, *shape[2:])
    kc[~live] = fp8.NAN_CODE
    vc[~live] = fp8.NAN_CODE
    return ts, kc.reshape(shape), vc.reshape(shape)


@pytest.mark.parametrize("k_scale,v_scale", [(1.0, 1.0), (0.02, 0.05), (0.37, 3.0)])
def test_write_kv_fp8_codes_bit_exact(k_scale, v_scale):
    lay = _decode_layout("w8", 40, 300, 8, 4, 128, 16, 31)
    ts, kc, vc = _setup(lay, k_scale, v_scale, 3)
    ts["k"] = ts["k"] * 7                                  # some magnitudes past 448 * scale
    dk = torch.from_numpy(kc).to(DEV)
    dv = torch.from_numpy(vc).to(DEV)
    md = H.device_meta(lay, DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.write_kv_fp8(ts["k"].to(DEV), ts["v"].to(DEV), dk, dv, md["slots"], k_scale, v_scale,
                    err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ek, ev = fp8.write_kv(kc, vc, _f32(ts["k"]), _f32(ts["v"]), lay.slot_mapping, lay.block_size,
                          k_scale, v_scale)
    assert np.array_equal(dk.cpu().numpy(), ek)
    assert np.array_equal(dv.cpu().numpy(), ev)


def _cases():
    return [
        _decode_layout("d128_bs16_g4", 24, 700, 16, 4, 128, 16, 41),
        _decode_layout("d64_bs16_g1", 16, 500, 8, 8, 64, 16, 42),
        _decode_layout("d128_bs1", 8, 90, 4, 2, 128, 1, 43),
        _decode_layout("d128_bs64_g8", 12, 900, 16, 2, 128, 64, 44),
        _decode_layout("d128_bs256_g32", 6, 1200, 32, 1, 128, 256, 45),
        _decode_layout("d128_long_splits", 3, 20000, 8, 2, 128, 16, 46, cmin=12000),
        _decode_layout("d64_bs8_g2", 20, 300, 4, 2, 64, 8, 47),
    ]


@pytest.mark.parametrize("lay", _cases(), ids=lambda l: l.name)
def test_decode_fp8_matches_oracle(lay):
    k_scale, v_scale = 0.03, 0.07
    ts, kc, vc = _setup(lay, k_scale, v_scale, 5)
    # the oracle: the same scatter, then attention on the dequantised cache
    ek, ev = fp8.write_kv(kc, vc, _f32(ts["k"]), _f32(ts["v"]), lay.slot_mapping, lay.block_size,
                          k_scale, v_scale)
    expect = ref.attention(_f32(ts["q"]).astype(np.float64), fp8.dequantize(ek, k_scale),
                           fp8.dequantize(ev, v_scale), lay.query_start_loc, lay.seq_lens,
                           lay.block_tables, lay.block_size, lay.scale, lay.num_kv_heads)
    dk = torch.from_numpy(kc).to(DEV)
    dv = torch.from_numpy(vc).to(DEV)
    md = H.device_meta(lay, DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    q = ts["q"].to(DEV)
    pa.write_kv_fp8(ts["k"].to(DEV), ts["v"].to(DEV), dk, dv, md["slots"], k_scale, v_scale,
                    err=err)
    out = pa.attention_fp8(q, dk, dv, md["qsl"], md["seq_lens"], md["bt"], k_scale=k_scale,
                           v_scale=v_scale, max_seq_len=lay.max_seq_len, scale=lay.scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(dk.cpu().numpy(), ek)
    H.assert_close(H.f64(out), expect, f"fp8/{lay.name}")


def test_decode_fp8_full_size_sampled():
    # the decode workload's shape with an 8-bit pool; 24 sampled sequences
    lay = workloads.config_layout(2, 0)
    k_scale, v_scale = 0.03, 0.05
    g = workloads.make_tensors(lay, seed=7, device=DEV)
    rng = np.random.default_rng(5)
    pick = sorted(rng.choice(lay.num_seqs, 24, replace=False).tolist())
    dk = torch.empty(g["k_cache"].shape, dtype=torch.uint8, device=DEV)
    dv = torch.empty_like(dk)
    # quantise the whole pool on the GPU with the scatter itself (every slot once)
    n_slots = lay.num_blocks * lay.block_size
    all_slots = torch.arange(n_slots, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kv_rows = lambda c: c.view(n_slots, lay.num_kv_heads, lay.head_dim)
    pa.write_kv_fp8(kv_rows(g["k_cache"]), kv_rows(g["v_cache"]), dk, dv, all_slots, k_scale,
                    v_scale, err=err)
    md = H.device_meta(lay, DEV)
    pa.write_kv_fp8(g["k"], g["v"], dk, dv, md["slots"], k_scale, v_scale, err=err)
    out = pa.attention_fp8(g["q"], dk, dv, md["qsl"], md["seq_lens"], md["bt"], k_scale=k_scale,
                           v_scale=v_scale, max_seq_len=lay.max_seq_len, scale=lay.scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    q64 = g["q"].double().cpu().numpy()
    for s in pick:
        tab = torch.tensor(lay.tables[s], device=DEV, dtype=torch.long)
        kb = fp8.dequantize(dk[tab].cpu().numpy(), k_scale)
        vb = fp8.dequantize(dv[tab].cpu().numpy(), v_scale)
        L = int(lay.seq_lens[s])
        exp = ref.attention(q64[s:s + 1], kb, vb, [0, 1], [L],
                            np.arange(len(lay.tables[s]))[None, :], lay.block_size, lay.scale,
                            lay.num_kv_heads)
        H.assert_close(H.f64(out[s:s + 1]), exp, f"fp8 full/{s}")


def test_fp8_refuses_prefill_rows_and_bad_scales():
    lay = workloads.custom_layout("mix8", [30, 0], [1, 20], 4, 2, 128, 16, 16, 3)
    ts = workloads.make_tensors(lay, seed=1)
    md = H.device_meta(lay, DEV)
    dk = torch.zeros(ts["k_cache"].shape, dtype=torch.uint8, device=DEV)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=DEV)
    lib = pa.load()
    rc = lib.pa_attention_fp8(pa._ptr(ts["q"].to(DEV)), 512, pa._ptr(ts["q"].to(DEV)), 512,
                              pa._ptr(dk), pa._ptr(dk), pa._ptr(md["qsl"]), pa._ptr(md["seq_lens"]),
                              pa._ptr(md["bt"]), 2, lay.num_tokens, md["bt"].shape[1], 1, 20,
                              lay.max_seq_len, 4, 2, 128, 16, lay.num_blocks, 0.1, 0.5, 0.5,
                              pa._ptr(ws), ws.numel(), pa._ptr(None), None)
    assert rc == 2
    with pytest.raises(pa.PaError, match="INVALID"):
        pa.write_kv_fp8(ts["k"].to(DEV), ts["v"].to(DEV), dk, dk.clone(), md["slots"], 0.0, 1.0)


def test_fp8_bad_slot_sets_flag():
    lay = _decode_layout("bad8", 4, 40, 4, 2, 128, 16, 9)
    ts = workloads.make_tensors(lay, seed=2)
    dk = torch.zeros(ts["k_cache"].shape, dtype=torch.uint8, device=DEV)
    dv = dk.clone()
    slots = torch.from_numpy(lay.slot_mapping).to(DEV)
    slots[1] = lay.num_blocks * lay.block_size
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.write_kv_fp8(ts["k"].to(DEV), ts["v"].to(DEV), dk, dv, slots, 1.0, 1.0, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEV_BAD_SLOT
