"""Python binding of the paged-KV attention C ABI (``include/pa.h``).

Argument marshalling only: torch tensors become raw device pointers, strides
and sizes, and the current CUDA stream is passed through.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback.  If the
library has not been built the first call raises.

    write_kv(k, v, k_cache, v_cache, slot_mapping)
    attention(q, k_cache, v_cache, query_start_loc, seq_lens, block_tables, ...)
    attention_cascade(..., prefix_blocks=...)   # decode over a shared cached prefix
    copy_blocks(k_cache, v_cache, pairs)
"""

from __future__ import annotations

import ctypes
import math
import os

__all__ = ["write_kv", "attention", "write_kv_attention", "attention_noalloc", "copy_blocks",
           "swap_blocks", "write_kv_fp8", "attention_fp8", "attention_cascade", "workspace_size",
           "cascade_workspace_size", "kernel_launches",
           "library_path", "load", "PaError", "DEV_BAD_SLOT", "DEV_BAD_BLOCK", "DEV_BAD_LEN",
           "DEV_BAD_DECODE", "DEV_BAD_PAIR", "DEV_TIMEOUT", "set_wait_limit_ns"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_lib", "libpa133.so")
_lib = None

DEV_BAD_SLOT = 1
DEV_BAD_BLOCK = 2
DEV_BAD_LEN = 4
DEV_BAD_DECODE = 8
DEV_BAD_PAIR = 16
DEV_TIMEOUT = 32

_c_i = ctypes.c_int
_c_i64 = ctypes.c_int64
_c_p = ctypes.c_void_p
_c_sz = ctypes.c_size_t
_c_f = ctypes.c_float

_SIGNATURES = {
    "pa_write_kv": (_c_i, [_c_p, _c_p, _c_i64, _c_i64, _c_p, _c_p, _c_p, _c_i, _c_i, _c_i, _c_i,
                           _c_i, _c_p, _c_p]),
    "pa_attention_workspace_size": (_c_sz, [_c_i, _c_i, _c_i, _c_i, _c_i]),
    "pa_attention": (_c_i, [_c_p, _c_i64, _c_p, _c_i64, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i, _c_i,
                            _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_f, _c_p,
                            _c_sz, _c_p, _c_p]),
    "pa_write_kv_attention": (_c_i, [_c_p, _c_i64, _c_p, _c_i64, _c_p, _c_i64, _c_p, _c_i64, _c_p,
                                     _c_p, _c_p, _c_p, _c_p, _c_p, _c_i, _c_i, _c_i, _c_i, _c_i,
                                     _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_f, _c_p, _c_sz, _c_p,
                                     _c_p]),
    "pa_write_kv_fp8": (_c_i, [_c_p, _c_p, _c_i64, _c_i64, _c_p, _c_p, _c_p, _c_i, _c_i, _c_i, _c_i,
                               _c_i, _c_f, _c_f, _c_p, _c_p]),
    "pa_attention_fp8": (_c_i, [_c_p, _c_i64, _c_p, _c_i64, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i, _c_i,
                                _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_f, _c_f,
                                _c_f, _c_p, _c_sz, _c_p, _c_p]),
    "pa_cascade_workspace_size": (_c_sz, [_c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i]),
    "pa_attention_cascade": (_c_i, [_c_p, _c_i64, _c_p, _c_i64, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i,
                                    _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_f,
                                    _c_p, _c_sz, _c_p, _c_p]),
    "pa_copy_blocks": (_c_i, [_c_p, _c_p, _c_p, _c_i, _c_i, _c_i, _c_i, _c_i, _c_p, _c_p]),
    "pa_attention_noalloc": (_c_i, [_c_p, _c_i64, _c_p, _c_i64, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i,
                                    _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i,
                                    _c_f, _c_p, _c_p]),
    "pa_swap_blocks": (_c_i, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i,
                              _c_p, _c_p]),
    "pa_status_string": (ctypes.c_char_p, [_c_i]),
    "pa_last_cuda_error": (_c_i, []),
    "pa_kernel_launches": (ctypes.c_uint64, []),
    "pa_set_wait_limit_ns": (ctypes.c_uint64, [ctypes.c_uint64]),
}


class PaError(RuntimeError):
    pass


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load ``libpa133.so`` (raises if it is missing: build it first)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise PaError(f"CUDA library not built: {_LIB_PATH} is missing "
                      "(run `python -m paged_kv_cache_133_gb300.build`)")
    lib = ctypes.CDLL(_LIB_PATH)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(rc: int, what: str):
    if rc != 0:
        lib = load()
        msg = lib.pa_status_string(rc).decode()
        if msg == "PA_ERR_CUDA":
            msg += f" (cudaError {lib.pa_last_cuda_error()})"
        raise PaError(f"{what}: {msg}")


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _need(cond, msg):
    if not cond:
        raise ValueError(msg)


def _bf16_rows(t, name):
    import torch
    _need(t.dtype == torch.bfloat16, f"{name} must be bfloat16")
    _need(t.is_cuda, f"{name} must be on a CUDA device")
    _need(t.dim() == 3, f"{name} must be [tokens, heads, head_dim]")
    _need(t.stride(2) == 1 and t.stride(1) == t.shape[2], f"{name}: heads x head_dim must be contiguous")


def _i32(t, name):
    import torch
    _need(t.dtype == torch.int32 and t.is_cuda and t.is_contiguous(),
          f"{name} must be a contiguous int32 CUDA tensor")


def _cache(t, name):
    import torch
    _need(t.dtype == torch.bfloat16 and t.is_cuda and t.is_contiguous() and t.dim() == 4,
          f"{name} must be a contiguous bf16 CUDA tensor [num_blocks, block_size, kv_heads, head_dim]")


def _cache8(t, name):
    import torch
    _need(t.element_size() == 1 and t.dtype in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8))
          and t.is_cuda and t.is_contiguous() and t.dim() == 4,
          f"{name} must be a contiguous 8-bit CUDA tensor [num_blocks, block_size, kv_heads, head_dim]")


def kernel_launches() -> int:
    return int(load().pa_kernel_launches())


def set_wait_limit_ns(ns: int) -> int:
    """Limit of each pipeline wait inside the tensor-core kernels for later
    launches (0: the default 2 s); returns the previous setting.  A wait that
    runs out sets ``PA_DEV_TIMEOUT`` in the error flag and the kernel exits
    cleanly."""
    return int(load().pa_set_wait_limit_ns(int(ns)))


def write_kv(k, v, k_cache, v_cache, slot_mapping, err=None, stream=None):
    """Scatter new-token K/V rows into the paged cache through ``slot_mapping``."""
    _bf16_rows(k, "k")
    _bf16_rows(v, "v")
    _cache(k_cache, "k_cache")
    _cache(v_cache, "v_cache")
    _i32(slot_mapping, "slot_mapping")
    nb, bs, hkv, d = k_cache.shape
    _need(tuple(v_cache.shape) == (nb, bs, hkv, d), "k_cache and v_cache shapes differ")
    _need(k.shape[1:] == (hkv, d) and v.shape[1:] == (hkv, d), "k/v head shape mismatch")
    T = slot_mapping.numel()
    _need(k.shape[0] >= T and v.shape[0] >= T, "k/v have fewer rows than slot_mapping")
    rc = load().pa_write_kv(_ptr(k), _ptr(v), k.stride(0), v.stride(0), _ptr(k_cache), _ptr(v_cache),
                            _ptr(slot_mapping), T, nb, bs, hkv, d, _ptr(err), _stream(stream))
    _check(rc, "pa_write_kv")


def write_kv_fp8(k, v, k_cache, v_cache, slot_mapping, k_scale, v_scale, err=None, stream=None):
    """Scatter new-token K/V rows into an 8-bit (E4M3) cache: codes of x / scale."""
    _bf16_rows(k, "k")
    _bf16_rows(v, "v")
    _cache8(k_cache, "k_cache")
    _cache8(v_cache, "v_cache")
    _i32(slot_mapping, "slot_mapping")
    nb, bs, hkv, d = k_cache.shape
    _need(tuple(v_cache.shape) == (nb, bs, hkv, d), "k_cache and v_cache shapes differ")
    _need(k.shape[1:] == (hkv, d) and v.shape[1:] == (hkv, d), "k/v head shape mismatch")
    T = slot_mapping.numel()
    _need(k.shape[0] >= T and v.shape[0] >= T, "k/v have fewer rows than slot_mapping")
    rc = load().pa_write_kv_fp8(_ptr(k), _ptr(v), k.stride(0), v.stride(0), _ptr(k_cache),
                                _ptr(v_cache), _ptr(slot_mapping), T, nb, bs, hkv, d,
                                float(k_scale), float(v_scale), _ptr(err), _stream(stream))
    _check(rc, "pa_write_kv_fp8")


def attention_fp8(q, k_cache, v_cache, query_start_loc, seq_lens, block_tables, *, k_scale,
                  v_scale, max_seq_len, scale=None, out=None, workspace=None, err=None,
                  stream=None):
    """Decode attention over an 8-bit (E4M3) cache; every sequence is a decode row."""
    import torch
    _bf16_rows(q, "q")
    _cache8(k_cache, "k_cache")
    _cache8(v_cache, "v_cache")
    for t, n in ((query_start_loc, "query_start_loc"), (seq_lens, "seq_lens"),
                 (block_tables, "block_tables")):
        _i32(t, n)
    nb, bs, hkv, d = k_cache.shape
    T, hq, dq = q.shape
    _need(dq == d, "q head_dim differs from the cache's")
    S = seq_lens.numel()
    _need(query_start_loc.numel() == S + 1 and block_tables.shape[0] == S, "metadata sizes differ")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    need = workspace_size(S, hq, hkv, d, max_seq_len)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = load().pa_attention_fp8(_ptr(out), out.stride(0), _ptr(q), q.stride(0), _ptr(k_cache),
                                 _ptr(v_cache), _ptr(query_start_loc), _ptr(seq_lens),
                                 _ptr(block_tables), S, T, block_tables.shape[1], S, 1,
                                 max_seq_len, hq, hkv, d, bs, nb, float(scale), float(k_scale),
                                 float(v_scale), _ptr(workspace), wbytes, _ptr(err), _stream(stream))
    _check(rc, "pa_attention_fp8")
    return out


def cascade_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_seq_len,
                           prefix_blocks, block_size) -> int:
    return int(load().pa_cascade_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                 max_seq_len, prefix_blocks, block_size))


def attention_cascade(q, k_cache, v_cache, query_start_loc, seq_lens, block_tables, *,
                      prefix_blocks, max_seq_len, scale=None, out=None, workspace=None, err=None,
                      stream=None):
    """Decode attention when every sequence's first ``prefix_blocks`` table
    entries are the same physical blocks (a shared cached prompt); every
    sequence is a decode row."""
    import torch
    _bf16_rows(q, "q")
    _cache(k_cache, "k_cache")
    _cache(v_cache, "v_cache")
    for t, n in ((query_start_loc, "query_start_loc"), (seq_lens, "seq_lens"),
                 (block_tables, "block_tables")):
        _i32(t, n)
    _need(block_tables.dim() == 2, "block_tables must be [num_seqs, max_blocks_per_seq]")
    nb, bs, hkv, d = k_cache.shape
    T, hq, dq = q.shape
    _need(dq == d, "q head_dim differs from the cache's")
    S = seq_lens.numel()
    _need(query_start_loc.numel() == S + 1 and block_tables.shape[0] == S, "metadata sizes differ")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    else:
        _bf16_rows(out, "out")
        _need(out.shape == q.shape, "out shape differs from q")
    need = cascade_workspace_size(S, hq, hkv, d, max_seq_len, prefix_blocks, bs)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    wbytes = workspace.numel() * workspace.element_size()
    rc = load().pa_attention_cascade(_ptr(out), out.stride(0), _ptr(q), q.stride(0), _ptr(k_cache),
                                     _ptr(v_cache), _ptr(query_start_loc), _ptr(seq_lens),
                                     _ptr(block_tables), S, T, block_tables.shape[1], max_seq_len,
                                     hq, hkv, d, bs, nb, int(prefix_blocks), float(scale),
                                     _ptr(workspace), wbytes, _ptr(err), _stream(stream))
    _check(rc, "pa_attention_cascade")
    return out


def copy_blocks(k_cache, v_cache, pairs, err=None, stream=None):
    """Copy-on-write: ``cache[dst] = cache[src]`` for each row (src, dst) of ``pairs``."""
    _cache(k_cache, "k_cache")
    _cache(v_cache, "v_cache")
    _i32(pairs, "pairs")
    nb, bs, hkv, d = k_cache.shape
    n = pairs.numel() // 2
    rc = load().pa_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(pairs), n, nb, bs, hkv, d,
                               _ptr(err), _stream(stream))
    _check(rc, "pa_copy_blocks")


def _pool(t, name):
    import torch
    _need(t.dtype == torch.bfloat16 and t.is_contiguous() and t.dim() == 4,
          f"{name} must be a contiguous bf16 tensor [blocks, block_size, kv_heads, head_dim]")
    _need(t.is_cuda or t.is_pinned(), f"{name} must be on the GPU or in pinned host memory")


def swap_blocks(src_k, src_v, dst_k, dst_v, pairs, err=None, stream=None):
    """Move whole blocks between pools: ``dst[d] = src[s]`` for each row (s, d) of ``pairs``.

    Either pool may be in pinned host memory (CPU offload of the cache); the
    copy runs as one kernel reading and writing through the pointers.
    """
    for t, n in ((src_k, "src_k"), (src_v, "src_v"), (dst_k, "dst_k"), (dst_v, "dst_v")):
        _pool(t, n)
    _i32(pairs, "pairs")
    _need(src_k.shape == src_v.shape and dst_k.shape == dst_v.shape, "K and V pools differ")
    _need(src_k.shape[1:] == dst_k.shape[1:], "pools differ in block shape")
    nsrc, bs, hkv, d = src_k.shape
    n = pairs.numel() // 2
    rc = load().pa_swap_blocks(_ptr(src_k), _ptr(src_v), _ptr(dst_k), _ptr(dst_v), _ptr(pairs), n,
                               nsrc, dst_k.shape[0], bs, hkv, d, _ptr(err), _stream(stream))
    _check(rc, "pa_swap_blocks")


def workspace_size(num_decode_seqs, num_q_heads, num_kv_heads, head_dim, max_seq_len) -> int:
    """Bytes of scratch ``attention`` needs on the current device."""
    return int(load().pa_attention_workspace_size(num_decode_seqs, num_q_heads, num_kv_heads,
                                                  head_dim, max_seq_len))


def attention(q, k_cache, v_cache, query_start_loc, seq_lens, block_tables, *, num_decode_seqs,
              max_query_len, max_seq_len, scale=None, out=None, workspace=None, err=None,
              stream=None):
    """Causal paged attention of one step's flat query batch; returns ``out`` [T, Hq, D] bf16.

    ``max_query_len`` / ``max_seq_len`` are host-side upper bounds (no device
    sync happens here).  ``workspace`` is allocated with torch when not given
    and the call needs one.
    """
    import torch
    _bf16_rows(q, "q")
    _cache(k_cache, "k_cache")
    _cache(v_cache, "v_cache")
    for t, n in ((query_start_loc, "query_start_loc"), (seq_lens, "seq_lens"),
                 (block_tables, "block_tables")):
        _i32(t, n)
    _need(block_tables.dim() == 2, "block_tables must be [num_seqs, max_blocks_per_seq]")
    nb, bs, hkv, d = k_cache.shape
    T, hq, dq = q.shape
    _need(dq == d, "q head_dim differs from the cache's")
    S = seq_lens.numel()
    _need(query_start_loc.numel() == S + 1 and block_tables.shape[0] == S, "metadata sizes differ")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    else:
        _bf16_rows(out, "out")
        _need(out.shape == q.shape, "out shape differs from q")
    need = workspace_size(num_decode_seqs, hq, hkv, d, max_seq_len)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = load().pa_attention(_ptr(out), out.stride(0), _ptr(q), q.stride(0), _ptr(k_cache),
                             _ptr(v_cache), _ptr(query_start_loc), _ptr(seq_lens),
                             _ptr(block_tables), S, T, block_tables.shape[1], num_decode_seqs,
                             max_query_len, max_seq_len, hq, hkv, d, bs, nb, float(scale),
                             _ptr(workspace), wbytes, _ptr(err), _stream(stream))
    _check(rc, "pa_attention")
    return out


def write_kv_attention(q, k, v, k_cache, v_cache, slot_mapping, query_start_loc, seq_lens,
                       block_tables, *, num_decode_seqs, max_query_len, max_seq_len, scale=None,
                       out=None, workspace=None, err=None, stream=None):
    """``write_kv`` then ``attention`` in one call, the scatter folded into the kernels.

    Same result as the two calls in sequence when each new token's slot is the
    one its sequence's block table gives to its position.
    """
    import torch
    _bf16_rows(q, "q")
    _bf16_rows(k, "k")
    _bf16_rows(v, "v")
    _cache(k_cache, "k_cache")
    _cache(v_cache, "v_cache")
    for t, n in ((slot_mapping, "slot_mapping"), (query_start_loc, "query_start_loc"),
                 (seq_lens, "seq_lens"), (block_tables, "block_tables")):
        _i32(t, n)
    _need(block_tables.dim() == 2, "block_tables must be [num_seqs, max_blocks_per_seq]")
    nb, bs, hkv, d = k_cache.shape
    T, hq, dq = q.shape
    _need(dq == d and k.shape == (T, hkv, d) and v.shape == (T, hkv, d), "q / k / v shapes differ")
    _need(slot_mapping.numel() == T, "slot_mapping must have one entry per token")
    S = seq_lens.numel()
    _need(query_start_loc.numel() == S + 1 and block_tables.shape[0] == S, "metadata sizes differ")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    else:
        _bf16_rows(out, "out")
        _need(out.shape == q.shape, "out shape differs from q")
    need = workspace_size(num_decode_seqs, hq, hkv, d, max_seq_len)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = load().pa_write_kv_attention(
        _ptr(out), out.stride(0), _ptr(q), q.stride(0), _ptr(k), k.stride(0), _ptr(v), v.stride(0),
        _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), _ptr(query_start_loc), _ptr(seq_lens),
        _ptr(block_tables), S, T, block_tables.shape[1], num_decode_seqs, max_query_len,
        max_seq_len, hq, hkv, d, bs, nb, float(scale), _ptr(workspace), wbytes, _ptr(err),
        _stream(stream))
    _check(rc, "pa_write_kv_attention")
    return out


NOALLOC_SCRATCH_BYTES = 16 << 20


def attention_noalloc(q, k_cache, v_cache, query_start_loc, seq_lens, block_tables, *, out,
                      num_decode_seqs, max_query_len, max_seq_len, scale=None, err=None,
                      stream=None):
    """``attention`` for callers that cannot allocate device memory.

    Takes a caller-provided ``out`` and no workspace: the split-KV scratch is a
    static device array of ``NOALLOC_SCRATCH_BYTES`` inside the library, shared
    by every call (calls that overlap on the GPU race on it).  Nothing here
    allocates.  Raises ``PaError`` (PA_ERR_WORKSPACE) when the batch's decode
    rows need more scratch than the array holds.
    """
    _bf16_rows(q, "q")
    _bf16_rows(out, "out")
    _cache(k_cache, "k_cache")
    _cache(v_cache, "v_cache")
    for t, n in ((query_start_loc, "query_start_loc"), (seq_lens, "seq_lens"),
                 (block_tables, "block_tables")):
        _i32(t, n)
    _need(block_tables.dim() == 2, "block_tables must be [num_seqs, max_blocks_per_seq]")
    nb, bs, hkv, d = k_cache.shape
    T, hq, dq = q.shape
    _need(dq == d, "q head_dim differs from the cache's")
    _need(out.shape == q.shape, "out shape differs from q")
    S = seq_lens.numel()
    _need(query_start_loc.numel() == S + 1 and block_tables.shape[0] == S, "metadata sizes differ")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rc = load().pa_attention_noalloc(_ptr(out), out.stride(0), _ptr(q), q.stride(0), _ptr(k_cache),
                                     _ptr(v_cache), _ptr(query_start_loc), _ptr(seq_lens),
                                     _ptr(block_tables), S, T, block_tables.shape[1],
                                     num_decode_seqs, max_query_len, max_seq_len, hq, hkv, d, bs,
                                     nb, float(scale), _ptr(err), _stream(stream))
    _check(rc, "pa_attention_noalloc")
    return out
