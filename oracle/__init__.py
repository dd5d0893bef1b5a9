"""Oracle: plain, slow, obviously correct CPU restatement of the paged-KV method.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import, call, link
or execute anything in this package. The product library never routes through it
and shares no code with it (no common headers, helpers, tables or generators).

Parts (each function cites the passage it follows):

* ``budget``       closed forms of the KV byte budget and of page tail waste;
* ``alloc_model``  block pool, per-sequence block tables, refcounts, fork and
                   copy-on-write of the partially filled last block (integers);
* ``cache_ops``    slot-mapped cache write and block copy as NumPy scatters;
* ``attention``    fp64 exact attention over pages gathered through a block table,
                   the online (running max/sum) recurrence, the log-sum-exp merge
                   of partial results, and a pure-Python brute force for tiny cases;
* ``native``       the same decode definition in C (binary64, OpenMP over
                   (sequence, query head)) for sizes NumPy loops cannot reach.

Every function is pinned by ``tests/test_oracle_*.py`` against values the pages
print, closed forms, library routines and invariants. Nothing in this package is
"parity unpinned" except the six-request tail example noted in ``budget``.
"""
