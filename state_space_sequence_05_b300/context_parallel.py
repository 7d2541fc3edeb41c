"""Context (sequence) parallelism for the SSD layer forward.

One sequence is cut into consecutive slices, one per rank of a
``torch.distributed`` group, in rank order.  Every rank

1. computes the state its slice leaves from a zero state, S_r, with the
   states-only pass (``ssd_chunk_scan_states``: segment states and state
   passing, no outputs), and the slice's total log-decay a_r
   (``ssd_segment_decay``);
2. all-gathers (a_r, S_r) from every rank: the one exchange step;
3. composes the earlier slices' affine maps h -> exp(a_k) h + S_k into the
   state entering its own slice (``ssd_segment_combine``; the composition
   rule (a2, b2) o (a1, b1) = (a2 a1, a2 b1 + b2) of the Mamba paper review,
   sec. 4);
4. runs the forward over its slice from that state: the exact y and end
   state.

The result equals the single-device forward up to rounding (the recurrence
is linear in its initial state).  Each rank does one states-only pass and
one forward over its slice ("Transformers are SSMs Review" sec. 3-2 (6):
only the boundary states move between the pieces).

This module marshals arguments and calls the collective; every step of the
computation runs in the library's kernels.  ``ops`` replaces those kernels
only for host-side tests of the exchange logic.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, Optional

import torch


@dataclass
class CPOps:
    """The per-rank device steps: forward(x, dt, A, B, C, D, chunk_size,
    init) -> (y, final); states(x, dt, A, B, chunk_size) -> final from a
    zero state; decay(dt, A) -> [b, H]; combine(decay [R, b, H], states
    [R, b, H, P, N], init) -> [R + 1, b, H, P, N]."""
    forward: Callable
    decay: Callable
    combine: Callable
    states: Optional[Callable] = None


def cuda_ops() -> CPOps:
    from . import ssd

    def forward(x, dt, A, B, C, D, chunk_size, init):
        return ssd.ssd_chunk_scan_fwd(x, dt, A, B, C, D, chunk_size, init)

    def states(x, dt, A, B, chunk_size):
        return ssd.ssd_chunk_scan_states(x, dt, A, B, chunk_size)

    return CPOps(forward, ssd.ssd_segment_decay, ssd.ssd_segment_combine, states)


def ssd_forward_context_parallel(x, dt, A, B, C, D=None, chunk_size=256, init_states=None,
                                 group=None, ops: Optional[CPOps] = None):
    """The forward of one sequence (per batch row) sliced over the ranks of
    `group` (None: the default group; a single process needs none).

    Each rank passes its own slice x [b, T_r, H, P], dt [b, T_r, H], B/C
    [b, T_r, G, N] (rank order = sequence order; slices may differ in
    length) and the same A, D and ``init_states`` [b, H, P, N] (the state
    before the first slice, or None).  Returns (y [b, T_r, H, P], final
    [b, H, P, N]): this slice's output and the state at its end (the
    sequence's final state on the last rank).
    """
    import torch.distributed as dist
    ops = ops or cuda_ops()
    world = dist.get_world_size(group) if dist.is_available() and dist.is_initialized() else 1
    if world == 1:
        return ops.forward(x, dt, A, B, C, D, chunk_size, init_states)
    rank = dist.get_rank(group)
    # 1. the state this slice leaves from a zero state (D does not enter it)
    if ops.states is not None:
        S = ops.states(x, dt, A, B, chunk_size)
    else:
        _, S = ops.forward(x, dt, A, B, C, None, chunk_size, None)
    a = ops.decay(dt, A)
    # 2. the exchange
    S_all = [torch.empty_like(S) for _ in range(world)]
    a_all = [torch.empty_like(a) for _ in range(world)]
    dist.all_gather(S_all, S.contiguous(), group=group)
    dist.all_gather(a_all, a.contiguous(), group=group)
    # 3. the state entering this slice
    if rank == 0:
        h_in = init_states
    else:
        h_in = ops.combine(torch.stack(a_all[:rank]).contiguous(),
                           torch.stack(S_all[:rank]).contiguous(), init_states)[rank].contiguous()
    # 4. the slice from its true initial state
    return ops.forward(x, dt, A, B, C, D, chunk_size, h_in)
