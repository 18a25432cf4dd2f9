"""Shared plumbing of the GPU tests: run one step through the C ABI and build
the oracle's expected values from inputs snapshotted before the step."""

import os

import numpy as np
import torch

import paged_kv_cache_133_gb300 as pa
from oracle import attention as ref
from oracle import metadata

MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def ensure_built():
    from paged_kv_cache_133_gb300 import build as pabuild
    lib_path = pa.library_path()
    srcs = pabuild.sources() + [os.path.join(os.path.dirname(pabuild.CSRC), "..", "include", "pa.h")]
    if not os.path.exists(lib_path) or any(os.path.getmtime(s) > os.path.getmtime(lib_path)
                                           for s in srcs if os.path.exists(s)):
        pabuild.build()
    pa.load()


def device_meta(lay, dev):
    return {
        "qsl": torch.from_numpy(lay.query_start_loc).to(dev),
        "seq_lens": torch.from_numpy(lay.seq_lens).to(dev),
        "bt": torch.from_numpy(lay.block_tables).to(dev),
        "slots": torch.from_numpy(lay.slot_mapping).to(dev),
        "pairs": torch.from_numpy(np.ascontiguousarray(lay.cow_pairs, dtype=np.int32)).to(dev),
    }


_ERR = None


def default_err():
    """Error flag used by run_step when the test passes none (zero it, check it after)."""
    global _ERR
    if _ERR is None:
        _ERR = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    return _ERR


def run_step(lay, g, md, err=None, num_decode=None, out=None, workspace=None):
    """copy_blocks (if any pairs) -> write_kv -> attention, all on the current stream."""
    if err is None:
        err = default_err()
    if len(lay.cow_pairs):
        pa.copy_blocks(g["k_cache"], g["v_cache"], md["pairs"], err=err)
    pa.write_kv(g["k"], g["v"], g["k_cache"], g["v_cache"], md["slots"], err=err)
    nd = lay.num_decode_seqs if num_decode is None else num_decode
    return pa.attention(g["q"], g["k_cache"], g["v_cache"], md["qsl"], md["seq_lens"], md["bt"],
                        num_decode_seqs=nd, max_query_len=lay.max_query_len,
                        max_seq_len=lay.max_seq_len, scale=lay.scale, out=out,
                        workspace=workspace, err=err)


def f64(t):
    return t.detach().to(torch.float64).cpu().numpy()


def oracle_full(lay, ts_cpu):
    """Expected output of the whole step from CPU copies of the inputs."""
    f = {k: f64(v) for k, v in ts_cpu.items()}
    kc, vc = f["k_cache"], f["v_cache"]
    if len(lay.cow_pairs):
        kc, vc = ref.copy_blocks(kc, vc, lay.cow_pairs)
    kc, vc = ref.write_kv(kc, vc, f["k"], f["v"], lay.slot_mapping, lay.block_size)
    return ref.attention(f["q"], kc, vc, lay.query_start_loc, lay.seq_lens, lay.block_tables,
                         lay.block_size, lay.scale, lay.num_kv_heads)


class Snapshot:
    """Blocks (and new-token rows) that the oracle needs for a sample of query
    rows, copied out of the inputs BEFORE the step runs."""

    def __init__(self, lay, g, rows):
        # rows: list of (sequence, local query index)
        self.lay = lay
        self.rows = rows
        seqs = sorted({s for s, _ in rows})
        need = set()
        for s in seqs:
            need.update(lay.tables[s])
        pairs = [(int(a), int(b)) for a, b in lay.cow_pairs.tolist() if int(b) in need]
        need.update(a for a, _ in pairs)
        self.ids = sorted(need)
        remap = {b: i for i, b in enumerate(self.ids)}
        idx = torch.tensor(self.ids, device=g["k_cache"].device, dtype=torch.long)
        self.kc = f64(g["k_cache"].index_select(0, idx))
        self.vc = f64(g["v_cache"].index_select(0, idx))
        self.pairs = np.array([(remap[a], remap[b]) for a, b in pairs], dtype=np.int64).reshape(-1, 2)
        self.seqs = seqs
        self.tables = [[remap[b] for b in lay.tables[s]] for s in seqs]
        qsl = lay.query_start_loc
        trows = np.concatenate([np.arange(qsl[s], qsl[s + 1]) for s in seqs]).astype(np.int64)
        ti = torch.from_numpy(trows).to(g["q"].device)
        self.q = f64(g["q"].index_select(0, ti))
        self.k = f64(g["k"].index_select(0, ti))
        self.v = f64(g["v"].index_select(0, ti))
        self.local_start = {}
        pos = 0
        for s in seqs:
            self.local_start[s] = pos
            pos += int(qsl[s + 1] - qsl[s])

    def expected(self):
        """fp64 oracle output for each sampled row, in ``rows`` order.

        Row (s, i) of a sequence with c cached tokens is the last query of the
        same sequence cut at length c + i + 1 (its causal key range), so it is
        evaluated as a one-token query over the post-write cache.
        """
        lay = self.lay
        bs = lay.block_size
        seq_lens = [int(lay.seq_lens[s]) for s in self.seqs]
        qlens = [int(lay.query_lens[s]) for s in self.seqs]
        qsl = metadata.query_start_loc(qlens)
        bt = metadata.pad_block_tables(self.tables)
        kc, vc = self.kc, self.vc
        if len(self.pairs):
            kc, vc = ref.copy_blocks(kc, vc, self.pairs)
        slots = metadata.slot_mapping(qsl, seq_lens, bt, bs)
        kc, vc = ref.write_kv(kc, vc, self.k, self.v, slots, bs)
        out = []
        for s, i in self.rows:
            j = self.seqs.index(s)
            c = seq_lens[j] - qlens[j]
            r = self.local_start[s] + i
            o = ref.attention(self.q[r:r + 1], kc, vc, [0, 1], [c + i + 1], bt[j:j + 1], bs,
                              lay.scale, lay.num_kv_heads)
            out.append(o[0])
        return np.stack(out)

    def gpu_rows(self, out):
        qsl = self.lay.query_start_loc
        idx = torch.tensor([int(qsl[s]) + i for s, i in self.rows], device=out.device)
        return f64(out.index_select(0, idx))


def assert_close(got, expect, what=""):
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    d = np.abs(got - expect)
    assert d.max() <= MAX_ABS and d.mean() <= MEAN_ABS, \
        f"{what}: max abs {d.max():.3g} mean abs {d.mean():.3g}"
    return float(d.max()), float(d.mean())


class FullOracle:
    """Every output row of a full-size step against the oracle.

    The blocks the step's sequences read (their tables and the copy-on-write
    sources) and the new-token rows are copied on the device BEFORE the step
    runs.  ``check`` then evaluates the oracle over chunks of sequences, each
    from a host fp64 copy of just the blocks it needs, and bounds max-abs and
    mean-abs over all T x Hq x D outputs.
    """

    def __init__(self, lay, g, chunk_bytes=256 << 20):
        self.lay = lay
        ids = set()
        for t in lay.tables:
            ids.update(int(b) for b in t)
        ids.update(int(a) for a, _ in lay.cow_pairs.tolist())
        self.ids = sorted(ids)
        self.pos = {b: i for i, b in enumerate(self.ids)}
        idx = torch.tensor(self.ids, dtype=torch.long, device=g["k_cache"].device)
        self.kc = g["k_cache"].index_select(0, idx)
        self.vc = g["v_cache"].index_select(0, idx)
        self.q, self.k, self.v = g["q"].clone(), g["k"].clone(), g["v"].clone()
        per_block = lay.block_size * lay.num_kv_heads * lay.head_dim * 8
        self.max_blocks = max(1, chunk_bytes // per_block)

    def _chunks(self):
        lay = self.lay
        cur, nblk = [], 0
        for s in range(lay.num_seqs):
            n = len(lay.tables[s])
            if cur and nblk + n > self.max_blocks:
                yield cur
                cur, nblk = [], 0
            cur.append(s)
            nblk += n
        if cur:
            yield cur

    def check(self, out, what=""):
        lay = self.lay
        bs = lay.block_size
        qsl = lay.query_start_loc
        cow = {int(d): int(s) for s, d in lay.cow_pairs.tolist()}
        worst, total, count = 0.0, 0.0, 0
        for seqs in self._chunks():
            blocks = sorted({int(b) for s in seqs for b in lay.tables[s]} |
                            {cow[int(b)] for s in seqs for b in lay.tables[s] if int(b) in cow})
            local = {b: i for i, b in enumerate(blocks)}
            sel = torch.tensor([self.pos[b] for b in blocks], dtype=torch.long,
                               device=self.kc.device)
            kc = f64(self.kc.index_select(0, sel))
            vc = f64(self.vc.index_select(0, sel))
            pairs = [(local[cow[b]], local[b]) for b in blocks if b in cow]
            if pairs:
                kc, vc = ref.copy_blocks(kc, vc, np.array(pairs, dtype=np.int64))
            rows = np.concatenate([np.arange(qsl[s], qsl[s + 1]) for s in seqs]).astype(np.int64)
            slots = lay.slot_mapping[rows].astype(np.int64)
            lslots = np.array([local[int(x) // bs] * bs + int(x) % bs if x >= 0 else -1
                               for x in slots], dtype=np.int64)
            ti = torch.from_numpy(rows).to(self.q.device)
            kc, vc = ref.write_kv(kc, vc, f64(self.k.index_select(0, ti)),
                                  f64(self.v.index_select(0, ti)), lslots, bs)
            qlens = [int(qsl[s + 1] - qsl[s]) for s in seqs]
            tables = metadata.pad_block_tables([[local[int(b)] for b in lay.tables[s]]
                                                for s in seqs])
            expect = ref.attention(f64(self.q.index_select(0, ti)), kc, vc,
                                   metadata.query_start_loc(qlens),
                                   [int(lay.seq_lens[s]) for s in seqs], tables, bs, lay.scale,
                                   lay.num_kv_heads)
            got = f64(out.index_select(0, ti))
            assert np.isfinite(got).all(), f"{what}: non-finite output"
            d = np.abs(got - expect)
            worst = max(worst, float(d.max()))
            total += float(d.sum())
            count += d.size
        mean = total / max(count, 1)
        assert count == lay.num_tokens * lay.num_q_heads * lay.head_dim
        assert worst <= MAX_ABS and mean <= MEAN_ABS, f"{what}: max abs {worst:.3g} mean abs {mean:.3g}"
        return worst, mean
