"""CPU fp64 oracle for exact scaled-dot-product attention (forward and backward).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute anything in this package: only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.
It shares no code, constants or helpers with the CUDA library in
``tiled_attention_tmem_gb300``; both sides only receive the same seeded input
arrays.

Modules
-------
attention       the plain definition: materialised S and P, analytic gradients
online_softmax  the blockwise m/l merge the tiled method relies on, written as a
                separate routine so tests can check it against the definition, and
                the split-KV route (parts finished on their own, then merged by
                their log-sum-exps)

Every function in these modules is pinned by CPU tests (``-m "not gpu"``) to
closed forms, invariants, brute force on tiny inputs and central finite
differences; none is "parity unpinned".
"""

from .attention import (
    scores,
    probabilities,
    forward,
    forward_rows,
    backward,
    backward_parts,
    backward_rows,
    row_statistics,
    visible_keys,
)
from .online_softmax import blockwise_forward, merge_partials, split_forward

__all__ = [
    "scores",
    "probabilities",
    "forward",
    "forward_rows",
    "backward",
    "backward_parts",
    "backward_rows",
    "row_statistics",
    "visible_keys",
    "blockwise_forward",
    "merge_partials",
    "split_forward",
]
