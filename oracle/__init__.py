"""CPU oracle for paged-KV attention over working sets.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute anything in this package: only the tests, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.

It is a plain, slow, obviously correct restatement of what the Pie pages say
the attention step computes ("How Pie thinks", section 4 "Working sets";
"Poem ops", the ``ops.attn`` row; "Write a model in Poem", section 4
"State (caches)"), written with numpy in float64, and it shares no code with
the CUDA library.  The modules:

* ``e4m3``      -- the FP8 E4M3 codec, from the OCP 8-bit floating point
                   format definition (the pages name ``dtype.e4m3`` only).
* ``kvstore``   -- page allocator, reference counts, prefix dedup table,
                   working-set state machine (create / fork / freeze /
                   rollback / match_prefix / destroy), the per-pass slot
                   reservation and the paged byte store that ``kv_append``
                   writes.
* ``attention`` -- exact softmax(q K^T / sqrt(d)) V per query row over the
                   row's working set, with grouped-query head mapping and the
                   causal rule, computed from keys gathered out of the store.
* ``rope``      -- the rotary position embedding of new K (and Q) rows that
                   precedes the append, in the kernel's float32 precision,
                   with the float64 rotation it is pinned against.

Parity status per function is listed in each module's docstring.
"""
