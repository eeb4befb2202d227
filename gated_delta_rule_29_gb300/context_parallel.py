"""Span-parallel context parallelism built on gdn_summary.

A long sequence cut into consecutive spans, one span per rank: every rank runs
gdn_summary on its span (end state S_H from a zero start and the transition
P^T), the ranks exchange those two tensors once (all-gather), and each rank
composes the state entering its span,

    S_{r+1} = einsum('ab,av->bv', transition_r, S_r) + S_H,r,     S_0 = initial state,

then runs gdn_fwd on its span from that state (cuDNN Linear Attention page,
"Summaries": the summaries compose across spans to give context parallelism).
The composition is a handful of small fp32 products per rank and runs on
whatever device the tensors live on; the exchange is the only collective.
"""
from __future__ import annotations

from typing import List, Optional

import torch


def compose(transitions: List[torch.Tensor], end_states: List[torch.Tensor],
            initial_state: Optional[torch.Tensor] = None, like: Optional[torch.Tensor] = None) -> List[torch.Tensor]:
    """States entering each span and the final state.

    transitions[j]: [..., K, K] (as returned by gdn_summary), end_states[j]: [..., K, V].
    Returns len(spans) + 1 tensors: the state entering span 0 (the initial state, or zeros
    shaped like `like` / the first end state), entering span 1, ..., and the state after the
    last span.
    """
    if initial_state is not None:
        S = initial_state
    else:
        S = torch.zeros_like(like if like is not None else end_states[0])
    out = [S]
    for tr, sh in zip(transitions, end_states):
        S = torch.einsum("...ab,...av->...bv", tr, S) + sh
        out.append(S)
    return out


def entering_state(transition: torch.Tensor, end_state: torch.Tensor,
                   initial_state: Optional[torch.Tensor] = None, group=None) -> torch.Tensor:
    """State entering this rank's span, given this rank's span summary.

    Ranks hold consecutive spans in rank order.  One all-gather of (transition, end_state);
    `initial_state` is the state entering rank 0's span (zeros when None; only rank 0's value
    is used).
    """
    import torch.distributed as dist

    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    trs = [torch.empty_like(transition) for _ in range(world)]
    shs = [torch.empty_like(end_state) for _ in range(world)]
    dist.all_gather(trs, transition.contiguous(), group=group)
    dist.all_gather(shs, end_state.contiguous(), group=group)
    s0 = initial_state
    if s0 is not None:
        s0 = s0.contiguous().clone()
        dist.broadcast(s0, src=dist.get_global_rank(group, 0) if group is not None else 0, group=group)
    return compose(trs[:rank], shs[:rank], s0, like=end_state)[rank]
