"""CPU oracle for one EAGLE-3 draft-and-verify step.

TEST INFRASTRUCTURE ONLY.  This package is the slow, plain reference that the
CUDA path is checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The product path (``eagle_tree_speculative_spec_gb300``) never imports it and
shares no code, table or constant generator with it.

Floating point is fp64 unless the method fixes the arithmetic (the
deterministic softmax in :mod:`oracle.dsm`, which is specified as a sequence
of IEEE fp32 round-to-nearest operations so that both sides agree bit for bit).

Modules
-------
philox      Philox4x32-10 counter-based generator (Salmon et al., SC'11).
dsm         Deterministic fixed-point softmax: EXP, LOG, weights, log-normaliser.
tree        Parent arrays -> depth, positions, ancestor mask / bitmask.
accept      Greedy longest-matching-path walk and lossless rejection sampling.
compact     Copy of the accepted path's K/V (and aux rows) into cache slots.
attention   RoPE and tree-masked verify attention.
llama       Tiny Llama target, EAGLE-3 draft head, vanilla and speculative decoding.
draft_tree  Dynamic top-k draft tree (expand, frontier select, final rerank).

Parity status per function is stated in each module header; every function
without an independent pin says "parity unpinned".
"""
