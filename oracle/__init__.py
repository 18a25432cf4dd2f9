"""Plain, slow CPU oracle for paged-KV attention over one continuous-batching step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import or run it.  It shares no
code with the CUDA library (no kernels, headers, helpers or tables); the only
module both sides use is the seeded input generator in ``workloads/``, which
holds none of the method's arithmetic.

Sources (cited by page title and section):

* "vLLM Continuous Batching：从 Forward Shape 理解两个核心参数" — the flat ``[T]``
  token batch, ``query_start_loc``, ``positions``, ``seq_lens``,
  ``block_tables``, ``slot_mapping`` (§2.1, §2.3, §2.3补充 第一步 / 第二步).
* "vLLM 原理" — the paged KV tensor ``[num_blocks, block_size, heads, dim]``
  (§3.6), ``Attention.forward`` (§3.7), copy-on-write of shared blocks (§2.1),
  ``Block`` / ``BlockManager`` (§3.3, §3.4).
* "LLM 推理引擎 Continuous Batching 与 PagedAttention：从 vLLM 原理到生产级部署实战"
  — paged read through the block table and the online-softmax update (§3.3).
* "vLLM 学习笔记（2）：从单请求到批处理" — padded vs flat batches and
  ``query_start_loc = [0, 3, 8, 10]`` (section on packing ragged sequences).

Modules:

* ``metadata``  — query_start_loc, positions, slot_mapping, padded block tables.
* ``attention`` — fp64 scatter, block copy and ragged causal paged attention.
* ``brute``     — the same attention with scalar Python loops (tiny inputs only).
* ``padded``    — the ``[S, L_max]`` + attention-mask formulation.
* ``blockmgr``  — a test-only block allocator with ref counts and copy-on-write.
* ``fp8``       — the 8-bit (E4M3) cache encoding: quantise, dequantise, scatter
  (an extension; the pages' cache is bf16).

Every function here is pinned by ``tests/test_oracle_*.py`` to something other
than itself: the pages' worked integers, closed forms, a library routine it
reduces to, brute force on tiny inputs, or invariants.
"""

from . import attention, blockmgr, brute, metadata, padded  # noqa: F401
