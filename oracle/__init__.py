"""CPU oracle for paged decode attention and the cache-maintenance copies.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package. The product library (``paged_kv_cache_04_gb300``) never imports it and
shares no code with it.

* :func:`decode` / :func:`partitions` / :func:`merge` -- float64 attention, in
  plain C (``pa_oracle.c``), reading the pool through the block table.
* :func:`reshape_and_cache` / :func:`copy_blocks` / :func:`swap_blocks` -- the cache writes, element
  by element on bit patterns (``cache_ops.py``).
* :func:`kv_bytes_per_token` -- the per-token KV size formula.
* :mod:`oracle.fp8` -- the E4M3 code format and the quantised-cache write and
  attention built on it.

Every function cites the passage it follows; the pins in
``tests/test_oracle_pins.py`` tie each one to something other than itself.
"""
from .cache_ops import copy_blocks, kv_bytes_per_token, reshape_and_cache, swap_blocks  # noqa: F401
from .attention import decode, partitions, merge, f16_bits_to_f64, bf16_bits_to_f64, max_threads  # noqa: F401
from . import fp8  # noqa: F401
