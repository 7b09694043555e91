"""fp64 CPU oracle for paged varlen relative-bias attention.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import or run anything in this package.  It
shares no code with the CUDA library (``paged_attention_relative_gb300``) and
neither imports the other; both are fed by the seeded input module
``paged_attention_relative_gb300.workloads``, which holds no attention
arithmetic.

Contents:
  rel_attn_oracle.c   the plain definition in C, fp64, OpenMP over (request, head)
  build.py            compiles it with gcc into oracle/librel_attn_oracle.so
  reference.py        ctypes wrapper, a pure-Python brute force for tiny
                      cases, and the pages' split-count heuristic restated

Parity status: every function here is pinned by the not-gpu tests in
tests/test_oracle_pins.py (library routines, closed forms, invariants, the
pages' own formula values).  None is "parity unpinned".
"""
