"""Packed multi-ragged single->pair->single block and variable-length
attention on GB300 (sm_103a).

The compute path is the C-ABI library ``libnt.so`` built from ``csrc/``;
:mod:`variable_length_batching_gb300.nt` is its thin binding.  The library is
loaded on first use and its absence raises: there is no other path.
"""
__all__ = ["nt", "workloads"]


def __getattr__(name):
    if name == "nt":
        from . import nt
        return nt
    raise AttributeError(name)
