"""Float64 CPU oracle for causal + document-masked GQA attention on one
context-parallel rank.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this package; only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline
leg and ``--impl reference``) may import or run it.  It shares no code,
constants or helpers with the CUDA path under ``document_masked_gqa_gb300/``.

Modules:

* ``cp``        - chunk assignment, chunk order, query positions, document ids
                  (context-parallel sharding as the Llama 3 pages describe it).
* ``attention`` - explicit-softmax attention over an explicit boolean mask,
                  forward (O, row log-sum-exp) and analytic backward.
* ``blockmask`` - brute-force classification of (query tile, key tile) pairs
                  as skip / full / partial, and the derived lists.
* ``flops``     - unmasked pair counts and the FLOP convention.

Every function is pinned by the ``-m "not gpu"`` tests in ``tests/`` against
closed forms, library routines (torch SDPA in float64), finite differences,
brute force on tiny inputs and the worked examples in ``tests/golden/``.
"""
