"""Plain float64 CPU oracle for SepLLM's attention hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports, links or
executes anything here; only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it.

The oracle is written from the SepLLM pages ("SepLLM: Accelerate Large
Language Models by Compressing One Segment into One Separator", arXiv
2412.12094), not from the CUDA path, and shares no code, table or constant
with it.  Its functions take every input as an argument (arrays produced by
the seeded generators); it holds no random state of its own.

Modules
-------
``sepllm``     separator detection, the SepLLM mask, keep-token compaction,
               per-query-tile block lists, masked softmax attention forward
               and its textbook backward.
``fixllm``     the FixLLM control (one kept token per fixed interval instead
               of the separators) on the same mask machinery.
``hybrid``     hybrid heads: kv groups with full causal attention beside
               groups under the SepLLM (or sliding-window) mask.
``varlen``     packed batches: several sequences in one row, the mask
               restarting at each sequence start.
``streaming``  the four-block streaming KV cache (initial, separator, past
               window, local window) with eviction into the separator cache,
               position shifting inside the cache, RoPE and decode attention.

Parity status: every function here is pinned by the ``-m "not gpu"`` tests
(brute force, reductions to textbook cases, library routines, closed forms
and the pages' worked example), except the choices the pages leave open and
that the build declares itself (RoPE theta and variant, the split of the
streaming window into past and local parts, the moment compression fires,
the block-list record format).  Those are marked "parity unpinned" where
they are defined.
"""

from . import fixllm, hybrid, sepllm, streaming, varlen  # noqa: F401
