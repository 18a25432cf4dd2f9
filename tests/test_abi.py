"""CPU checks of the C ABI boundary: the library builds, loads, exports exactly
the functions include/pa.h declares, and rejects bad host-side arguments
before touching the GPU."""

import ctypes
import os
import re
import subprocess

import pytest
import torch

import paged_kv_cache_133_gb300 as pa
from paged_kv_cache_133_gb300 import build as pabuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(pa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    srcs = pabuild.sources()
    lib_path = pa.library_path()
    if not os.path.exists(lib_path) or any(os.path.getmtime(s) > os.path.getmtime(lib_path) for s in srcs):
        pabuild.build()
    return pa.load()


def test_header_declares_the_three_calls():
    names = _declared()
    for n in ("pa_write_kv", "pa_attention", "pa_attention_workspace_size", "pa_copy_blocks",
              "pa_swap_blocks", "pa_write_kv_attention"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", pa.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = sorted(set(re.findall(r"\sT\s(pa_\w+)$", out, flags=re.M)))
    assert exported == _declared()
    for n in _declared():
        assert hasattr(lib, n)


def test_status_strings(lib):
    assert lib.pa_status_string(0) == b"PA_OK"
    assert lib.pa_status_string(3) == b"PA_ERR_WORKSPACE"


def test_host_validation_rejects_before_launch(lib):
    nul = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(1 << 20)     # never dereferenced: validation fails first
    # unsupported head_dim
    rc = lib.pa_attention(fake, 96 * 4, fake, 96 * 4, fake, fake, fake, fake, fake, 1, 1, 1, 0, 1, 1,
                          4, 4, 96, 16, 8, 1.0, nul, 0, nul, nul)
    assert rc == 2
    # q heads not a multiple of kv heads
    rc = lib.pa_attention(fake, 0, fake, 0, fake, fake, fake, fake, fake, 1, 1, 1, 0, 1, 1,
                          6, 4, 128, 16, 8, 1.0, nul, 0, nul, nul)
    assert rc == 2
    # block size not a power of two
    rc = lib.pa_attention(fake, 0, fake, 0, fake, fake, fake, fake, fake, 1, 1, 1, 0, 1, 1,
                          4, 4, 128, 12, 8, 1.0, nul, 0, nul, nul)
    assert rc == 2
    # more decode rows than sequences
    rc = lib.pa_attention(fake, 0, fake, 0, fake, fake, fake, fake, fake, 1, 1, 1, 2, 1, 1,
                          4, 4, 128, 16, 8, 1.0, nul, 0, nul, nul)
    assert rc == 1
    # null cache
    rc = lib.pa_write_kv(fake, fake, 512, 512, nul, fake, fake, 4, 8, 16, 4, 128, nul, nul)
    assert rc == 1
    # pool too large for int32 slots
    rc = lib.pa_write_kv(fake, fake, 512, 512, fake, fake, fake, 4, 1 << 28, 16, 4, 128, nul, nul)
    assert rc == 1
    # nothing to do is fine and launches nothing
    before = lib.pa_kernel_launches()
    assert lib.pa_write_kv(nul, nul, 512, 512, fake, fake, nul, 0, 8, 16, 4, 128, nul, nul) == 0
    assert lib.pa_copy_blocks(fake, fake, nul, 0, 8, 16, 4, 128, nul, nul) == 0
    assert lib.pa_swap_blocks(fake, fake, fake, fake, nul, 0, 8, 4, 16, 4, 128, nul, nul) == 0
    assert lib.pa_kernel_launches() == before
    # swap: null pool, empty destination pool, too many pairs for one call
    assert lib.pa_swap_blocks(fake, nul, fake, fake, fake, 1, 8, 4, 16, 4, 128, nul, nul) == 1
    assert lib.pa_swap_blocks(fake, fake, fake, fake, fake, 1, 8, 0, 16, 4, 128, nul, nul) == 1
    assert lib.pa_swap_blocks(fake, fake, fake, fake, fake, 70000, 8, 4, 16, 4, 128, nul, nul) == 2


def test_swap_binding_refuses_pageable_host_pools():
    # Only device memory or page-locked host memory reaches the C call.
    t = torch.zeros((2, 1, 1, 8), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="pinned"):
        pa.swap_blocks(t, t, t, t, None)


def test_fused_call_validates_its_extra_arguments(lib):
    nul = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(1 << 20)     # never dereferenced: validation fails first
    args = lambda k, ks, slots: (fake, 512, fake, 512, k, ks, fake, ks, fake, fake, slots, fake,
                                 fake, fake, 1, 4, 1, 0, 4, 4, 4, 1, 128, 16, 8, 1.0, fake,
                                 1 << 20, nul, nul)
    assert lib.pa_write_kv_attention(*args(nul, 128, fake)) == 1   # no k
    assert lib.pa_write_kv_attention(*args(fake, 128, nul)) == 1   # no slot_mapping
    assert lib.pa_write_kv_attention(*args(fake, 64, fake)) == 1   # token stride < Hkv * D
    assert lib.pa_write_kv_attention(*args(fake, 132, fake)) == 2  # stride not a multiple of 8
