"""ORACLE -- test infrastructure, not product code.

A plain, slow, obviously correct CPU restatement of what the shared-prefix
paged decode path computes, written from the pages' descriptions:

* ``attention``     fp64 attention over an explicitly gathered context (C, plain loops)
                    and the log-sum-exp merge of GraniKV Eq. 1;
* ``block_manager`` the refcounted copy-on-write block pool of "Paged KV cache"
                    (How it works; Code) with the slot formula;
* ``hot_pool``      GraniKV's HOT pool allocator (Section 3.2, Appendix B.8b);
* ``pool_model``    a host model of the HOT/COLD storage (reshape_and_cache
                    scatter, copy-on-write block copy, gather through a table);
* ``reference``     expected outputs of a workload, from the seeded inputs;
* ``dispatch``      GraniKV Eq. 2 and the per-step dispatch rule (Section 3.6);
* ``model``         the byte and flop model of GraniKV Appendix B.11 / Table 23.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may import
this package.  It shares no code with the CUDA library.
"""
