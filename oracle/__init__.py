"""Float64 CPU oracle of the decode path (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never links, calls or
reads anything here, and nothing here reads the CUDA library.
"""
