"""Float64 CPU oracle for the fused LM-head scoring path.

Test infrastructure: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` import it.  It shares no code
with the CUDA library.
"""
