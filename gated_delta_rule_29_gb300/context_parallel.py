"""Span-parallel context parallelism built on gdn_summary.

A long sequence cut into consecutive spans, one span per rank: every rank runs
gdn_summary on its span (end state S_H from a zero start and the transition
P^T), the ranks exchange those two tensors once (all-gather), and each rank
composes the state entering its span,

    S_{r+1} = einsum('ab,av->bv', transition_r, S_r) + S_H,r,     S_0 = initial state,

then runs gdn_fwd on its span from that state (cuDNN Linear Attention page,
"Summaries": the summaries compose across spans to give context parallelism).
The backward mirrors it: each rank's state gradient from its own outputs
(gdn_summary_bwd, the summary's counterpart on the gradient side), one all-gather, and
the reverse composition dS_enter = transition dS_exit + dS_H give every rank the
cotangent of its span's end state for gdn_bwd.
The composition runs in the library's kernel (gdn_compose_spans: a handful of
small fp32 products per rank, on the CUDA device of the summaries); the exchange
is the only collective.  `entering_state` and `exit_state_grad` take an optional
`composer` with the signature of `compose` / `compose_grads` for callers whose
tensors are not on a GPU.
"""
from __future__ import annotations

from typing import Callable, List, Optional

import torch

from . import api


def compose(transitions: List[torch.Tensor], end_states: List[torch.Tensor],
            initial_state: Optional[torch.Tensor] = None, like: Optional[torch.Tensor] = None) -> List[torch.Tensor]:
    """States entering each span and the final state.

    transitions[j]: [..., K, K] (as returned by gdn_summary), end_states[j]: [..., K, V].
    Returns len(spans) + 1 tensors: the state entering span 0 (the initial state, or zeros
    shaped like `like` / the first end state), entering span 1, ..., and the state after the
    last span.
    """
    if not transitions:
        if initial_state is not None:
            return [initial_state]
        return [torch.zeros_like(like if like is not None else end_states[0])]
    trs, shs = torch.stack(list(transitions)), torch.stack(list(end_states))
    out = api.compose_spans(trs, shs, initial_state, backward=False)
    return list(out.unbind(0))


def compose_grads(transitions: List[torch.Tensor], local_grads: List[torch.Tensor],
                  d_final: Optional[torch.Tensor] = None) -> List[torch.Tensor]:
    """Backward of compose: the state gradient entering and leaving each span.

    The gradients are linear in the final-state cotangent, and through a span the state gradient
    moves as dS_enter = einsum('ab,bv->av', transition, dS_exit) (the transpose of the forward
    composition).  local_grads[r] is the entering-state gradient of span r from its own outputs
    alone (gdn_summary_bwd, or gdn_bwd with a zero final-state cotangent); d_final the cotangent
    of the state after
    the last span.  Returns len(spans) + 1 tensors: the gradient leaving each span (dS_exit_r,
    the final-state cotangent to use for span r), then the gradient entering span 0.
    """
    if not transitions:
        return [d_final]
    trs, loc = torch.stack(list(transitions)), torch.stack(list(local_grads))
    out = api.compose_spans(trs, loc, d_final, backward=True)
    return list(out.unbind(0))


def exit_state_grad(transition: torch.Tensor, local_grad: torch.Tensor,
                    d_final: Optional[torch.Tensor] = None, group=None,
                    composer: Optional[Callable] = None) -> torch.Tensor:
    """Final-state cotangent for this rank's span in the context-parallel backward.

    Ranks hold consecutive spans in rank order.  Each rank first takes its span's own state
    gradient (local_grad: gdn_summary_bwd, zero exit cotangent), then one all-gather of
    (transition, local_grad) lets every rank compose the gradient arriving at its span's end;
    running gdn_bwd again with that cotangent (or adding the contribution of the second run, the
    gradients being linear in it) completes the rank's gradients.  `d_final` is the cotangent
    of the state after the last span (only the last rank's value is used; zero when None).
    """
    import torch.distributed as dist

    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    trs = [torch.empty_like(transition) for _ in range(world)]
    lgs = [torch.empty_like(local_grad) for _ in range(world)]
    dist.all_gather(trs, transition.contiguous(), group=group)
    dist.all_gather(lgs, local_grad.contiguous(), group=group)
    dfin = d_final.contiguous().clone() if d_final is not None else torch.zeros_like(local_grad)
    last = dist.get_global_rank(group, world - 1) if group is not None else world - 1
    dist.broadcast(dfin, src=last, group=group)
    return (composer or compose_grads)(trs, lgs, dfin)[rank]


def entering_state(transition: torch.Tensor, end_state: torch.Tensor,
                   initial_state: Optional[torch.Tensor] = None, group=None,
                   composer: Optional[Callable] = None) -> torch.Tensor:
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
    # every rank takes part in the broadcast (a rank without a start state sends zeros)
    s0 = initial_state.contiguous().clone() if initial_state is not None else torch.zeros_like(end_state)
    dist.broadcast(s0, src=dist.get_global_rank(group, 0) if group is not None else 0, group=group)
    return (composer or compose)(trs[:rank], shs[:rank], s0, like=end_state)[rank]
