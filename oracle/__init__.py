"""CPU oracle for the packed single->pair->single block and for
variable-length (cu_seqlens) attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
link this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It
shares no code with the CUDA library and imports nothing from it.

Everything here is plain numpy in float64, one sample (or one segment) at a
time, written to be checked against the pages by eye:

* ``partition``  -- sample offsets, pair offsets and second-level row splits
  ("DanLing NestedTensor", section 3.1 "Numerical storage" Eq. 2, Figure 2,
  Appendix A "Structural invariants").
* ``block``      -- Eq. 1 of the same paper (section 3), per sample, densely;
  plus a padded-then-gathered route that reaches the same cells through a
  B x N_max x N_max envelope.
* ``block_backward`` -- the sample-weighted squared loss of the same
  paper's Appendix A.1, Eq. 5, on the block's two outputs, and the block's
  gradients (the chain rule of Eq. 1), per sample, densely.
* ``attention``  -- softmax attention restricted to each cu_seqlens segment
  ("Variable-length attention and data packing", sections "What it is" and
  "How it works"), and the full T x T block-diagonal masked form of that
  page's "Core math" section (C).

Parity status: every function is pinned by tests under ``tests/`` marked
``not gpu`` (worked example of Figure 2, closed forms, library routines on
special cases, invariants, brute force).  No function is "parity unpinned".
"""
