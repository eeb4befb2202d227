"""Autograd for the chunked GDN: gdn_fwd as the forward, gdn_bwd as its backward.

cuDNN Linear Attention page ("Semantics worth knowing"): every variant has a forward and a full
backward, exposed as PyTorch operators with autograd formulas, and the backward reuses the
forward's state checkpoints.  `gdn_attention` is that pairing: the forward keeps fp32 checkpoints
every `checkpoint_every_n` tokens for the backward (64: the chunk cadence, read directly; a larger
multiple of 64: the backward regenerates the states entering every chunk from them, segment by
segment; with save_checkpoints=False the backward recomputes them all), and the gradients flow
to q, k, v, g, beta, the initial state and, with the softplus gate, a_log and dt_bias.  Every
computation runs in the library's kernels.
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch

from . import api


class _GDN(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, g, beta, cu_seqlens, initial_state, a_log, dt_bias, scale, use_qk_l2norm,
                gate_lower_bound, beta_sigmoid, ckpt_n):
        o, fin, ck = api.gdn_fwd(q, k, v, g, beta, cu_seqlens, scale=scale, use_qk_l2norm=use_qk_l2norm,
                                 initial_state=initial_state, output_final_state=True,
                                 checkpoint_every_n=ckpt_n,
                                 checkpoint_dtype=torch.float32, a_log=a_log, dt_bias=dt_bias,
                                 gate_lower_bound=gate_lower_bound, beta_sigmoid=beta_sigmoid)
        ctx.save_for_backward(q, k, v, g, beta, cu_seqlens, initial_state, a_log, dt_bias, ck)
        ctx.opts = (scale, use_qk_l2norm, gate_lower_bound, beta_sigmoid, ckpt_n)
        return o, fin

    @staticmethod
    def backward(ctx, d_o, d_fin):
        q, k, v, g, beta, cu, s0, a_log, dt_bias, ck = ctx.saved_tensors
        scale, use_qk_l2norm, gate_lower_bound, beta_sigmoid, ckpt_n = ctx.opts
        if d_o is None:
            d_o = torch.zeros(q.shape[0], v.shape[1], v.shape[2], dtype=torch.bfloat16, device=q.device)
        out = api.gdn_bwd(q, k, v, g, beta, cu, d_o.to(torch.bfloat16).contiguous(), scale=scale,
                          use_qk_l2norm=use_qk_l2norm, initial_state=s0,
                          d_final_state=None if d_fin is None else d_fin.float().contiguous(),
                          checkpoints=ck, checkpoint_every_n=ckpt_n if ckpt_n else 64, a_log=a_log,
                          dt_bias=dt_bias, gate_lower_bound=gate_lower_bound, beta_sigmoid=beta_sigmoid)
        dq, dk, dv, dg, dbeta, ds0 = out[:6]
        d_alog, d_dt = (out[6], out[7]) if len(out) > 6 else (None, None)
        if s0 is not None and ds0 is not None:
            ds0 = ds0.to(s0.dtype)
        return (dq, dk, dv, dg, dbeta.to(beta.dtype), None, ds0, d_alog, d_dt,
                None, None, None, None, None)


def gdn_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
                  cu_seqlens: torch.Tensor, *, initial_state: Optional[torch.Tensor] = None,
                  scale: Optional[float] = None, use_qk_l2norm: bool = True, a_log: Optional[torch.Tensor] = None,
                  dt_bias: Optional[torch.Tensor] = None, gate_lower_bound: Optional[float] = None,
                  beta_sigmoid: bool = False, save_checkpoints: bool = True, checkpoint_every_n: int = 64
                  ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Differentiable chunked GDN: returns (o [T, HO, V] bf16, final_state [N, HO, K, V] fp32).

    Arguments as for gdn_fwd.  save_checkpoints keeps the forward's fp32 states every
    checkpoint_every_n tokens (a multiple of 64) for the backward: every 64 tokens costs
    N_chunks x HO x K x V x 4 bytes and is read as it is; every n tokens costs n / 64 times less
    and the backward regenerates the rest with one forward launch over the n-token segments
    (the gradients are bitwise the same).  False keeps none: the backward recomputes them all."""
    if checkpoint_every_n <= 0 or checkpoint_every_n % 64 != 0:
        raise ValueError("checkpoint_every_n must be a positive multiple of 64")
    return _GDN.apply(q, k, v, g, beta, cu_seqlens, initial_state, a_log, dt_bias, scale, use_qk_l2norm,
                      gate_lower_bound, beta_sigmoid, checkpoint_every_n if save_checkpoints else 0)
