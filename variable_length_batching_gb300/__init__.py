"""Packed multi-ragged single->pair->single block and variable-length
attention on GB300 (sm_103a).

The compute path is the C-ABI library ``libnt.so`` built from ``csrc/`` by
:mod:`variable_length_batching_gb300.build`; :mod:`variable_length_batching_gb300.nt`
is its thin binding.  The library is loaded on first call and its absence
raises: there is no other path.
"""
