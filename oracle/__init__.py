"""Independent CPU oracle for the tcgen05 GEMM library.

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are its only users; the CUDA path neither
imports nor links anything here, and nothing here comes from the CUDA path.

* ``oracle.gemm``    -- fp64 triple-loop GEMM ``D = alpha A B + beta C``
                        (C, OpenMP over rows), per-entry evaluation for
                        full-size samples, round-to-nearest-even output.
* ``oracle.layouts`` -- swizzle functor and XOR grid, the LBO/SBO/SWZ page's
                        closed forms, descriptor encoder and interpreter,
                        TMA box placement, bank-conflict counter, TMEM
                        accumulator maps, mbarrier ring parity.

Every function cites the passage it restates. Each is pinned in
``tests/test_oracle_*.py`` against values the pages print, closed forms,
invariants or brute force.
"""
from . import gemm, layouts  # noqa: F401
