"""Torch-facing wrappers of the liblinattn C ABI (same names: gdn_fwd, gdn_summary).

PyTorch only supplies device memory and the current stream; every step of the
computation runs in the library's CUDA kernels.  Shapes follow the cuDNN Linear
Attention page: packed THD operands [T, heads, dim], cu_seqlens [N + 1].
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional, Tuple

import torch

from . import binding as B


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _check_thd(name, x, dtype, heads_dim=True):
    if not isinstance(x, torch.Tensor) or not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if x.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {x.dtype} (dtypes are strict)")
    if x.dim() != (3 if heads_dim else 2):
        raise ValueError(f"{name} must be rank {3 if heads_dim else 2}, got shape {tuple(x.shape)}")
    if heads_dim and x.shape[-1] > 1 and x.stride(-1) != 1:
        raise ValueError(f"{name} must have a contiguous innermost axis")


def _set_transforms(p, HO, dev, a_log, dt_bias, gate_lower_bound, beta_sigmoid, beta):
    """Fills the optional input-transform fields (cudnn-frontend PR #616 in-kernel fusions):
    a_log + dt_bias select the softplus gate, gate_lower_bound the bounded sigmoid gate."""
    if (a_log is None) != (dt_bias is None):
        raise ValueError("the softplus gate needs both a_log and dt_bias")
    if a_log is not None and gate_lower_bound is not None:
        raise ValueError("choose one gate transform: (a_log, dt_bias) or gate_lower_bound")
    keep = []
    if a_log is not None:
        for name, x in (("a_log", a_log), ("dt_bias", dt_bias)):
            if not isinstance(x, torch.Tensor) or x.device != dev or x.dtype != torch.float32 or x.numel() != HO:
                raise ValueError(f"{name} must be a float32 tensor of {HO} elements on {dev}")
        a_log, dt_bias = a_log.contiguous(), dt_bias.contiguous()
        keep += [a_log, dt_bias]
        p.gate_mode, p.a_log, p.dt_bias = B.LA_GATE_SOFTPLUS, a_log.data_ptr(), dt_bias.data_ptr()
    elif gate_lower_bound is not None:
        p.gate_mode, p.gate_lower_bound = B.LA_GATE_SIGMOID_BOUND, float(gate_lower_bound)
    p.beta_sigmoid = int(bool(beta_sigmoid))
    p.beta_bf16 = int(beta.dtype == torch.bfloat16)
    return keep


def _check_beta(beta, beta_sigmoid):
    if beta_sigmoid and isinstance(beta, torch.Tensor) and beta.dtype == torch.bfloat16:
        _check_thd("beta", beta, torch.bfloat16, heads_dim=False)
    else:
        _check_thd("beta", beta, torch.float32, heads_dim=False)


def _out(name, x, shape, dtype, dev, contiguous=False):
    """A caller-provided output buffer, or a new one when x is None."""
    if x is None:
        return torch.empty(*shape, dtype=dtype, device=dev)
    if not isinstance(x, torch.Tensor) or x.device != dev or x.dtype != dtype or tuple(x.shape) != tuple(shape):
        raise ValueError(f"{name} must be a {dtype} tensor of shape {tuple(shape)} on {dev}")
    if contiguous and not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if len(shape) == 3 and shape[-1] > 1 and x.stride(-1) != 1:
        raise ValueError(f"{name} must have a contiguous innermost axis")
    return x


def _cu_bits(cu: torch.Tensor) -> int:
    if cu.dtype == torch.int32:
        return 32
    if cu.dtype == torch.int64:
        return 64
    raise TypeError("cu_seqlens must be int32 or int64")


def checkpoint_rows(cu_seqlens: torch.Tensor, n: int) -> int:
    """Rows of the checkpoint series, sum_i ceil(L_i / n) (reads cu_seqlens on the host)."""
    cu = cu_seqlens.detach().to("cpu", torch.int64).contiguous()
    out = ctypes.c_int64(0)
    B.check(B.load().la_checkpoint_rows(cu.data_ptr(), 64, cu.numel() - 1, int(n), ctypes.byref(out)),
            "la_checkpoint_rows")
    return int(out.value)


def workspace_bytes(N: int, summary: bool = False) -> int:
    return int(B.load().la_gdn_workspace_bytes(int(N), int(bool(summary))))


def gdn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
            cu_seqlens: torch.Tensor, *, scale: Optional[float] = None, use_qk_l2norm: bool = True,
            initial_state: Optional[torch.Tensor] = None, output_final_state: bool = True,
            checkpoint_every_n: int = 0, checkpoint_dtype: torch.dtype = torch.bfloat16,
            checkpoint_rows_hint: Optional[int] = None, o: Optional[torch.Tensor] = None,
            final_state: Optional[torch.Tensor] = None, checkpoints: Optional[torch.Tensor] = None,
            workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
            stream: Optional[torch.cuda.Stream] = None, a_log: Optional[torch.Tensor] = None,
            dt_bias: Optional[torch.Tensor] = None, gate_lower_bound: Optional[float] = None,
            beta_sigmoid: bool = False, state_indices: Optional[torch.Tensor] = None,
            num_householder: int = 1
            ) -> Tuple[torch.Tensor, Optional[torch.Tensor], Optional[torch.Tensor]]:
    """Chunked GDN forward.  Returns (o [T, HO, V] bf16, final_state [N, HO, K, V] fp32 or None,
    checkpoints [R, HO, K, V] or None).  Asynchronous on the current stream.

    g is the natural-log decay, unless a_log and dt_bias ([HO] fp32) are given (the kernel then
    uses -exp(a_log) softplus(g + dt_bias)) or gate_lower_bound (< 0; the kernel uses
    gate_lower_bound * sigmoid(g)).  With beta_sigmoid, beta holds logits (fp32 or bf16).

    state_indices ([N] int32): initial_state is then a contiguous state pool [P, HO, K, V]
    (fp32 or bf16); sequence i starts from pool[state_indices[i]] and its end state is
    written back into that slot in place.  No final_state or checkpoints are returned.

    num_householder n > 1 (Gated DeltaProduct): k, v and beta carry n rows per token, as the
    update timeline [T * n, ...] or token-major [T, n, ...] (contiguous per token); q, g and o
    keep one row per token."""
    n = int(num_householder)
    if n > 1:
        T_ = q.shape[0]
        if k.dim() == 4:
            k = k.reshape(T_ * n, k.shape[2], k.shape[3])
        if v.dim() == 4:
            v = v.reshape(T_ * n, v.shape[2], v.shape[3])
        if beta.dim() == 3:
            beta = beta.reshape(T_ * n, beta.shape[2])
        if k.shape[0] != T_ * n or v.shape[0] != T_ * n or beta.shape[0] != T_ * n:
            raise ValueError(f"num_householder={n}: k, v and beta need {T_ * n} update rows")
    _check_thd("q", q, torch.bfloat16)
    _check_thd("k", k, torch.bfloat16)
    _check_thd("v", v, torch.bfloat16)
    _check_thd("g", g, torch.float32, heads_dim=False)
    _check_beta(beta, beta_sigmoid)
    T, HK, K = q.shape
    HV, V = v.shape[1], v.shape[2]
    N = cu_seqlens.numel() - 1
    HO = HV
    dev = q.device
    if o is None:
        o = torch.empty(T, HO, V, dtype=torch.bfloat16, device=dev)
    if state_indices is not None:
        if initial_state is None or not initial_state.is_contiguous() or initial_state.dim() != 4:
            raise ValueError("state_indices needs initial_state as a contiguous pool [P, HO, K, V]")
        if state_indices.dtype != torch.int32 or state_indices.numel() != N or state_indices.device != dev:
            raise ValueError(f"state_indices must be int32 [{N}] on {dev}")
        if checkpoint_every_n:
            raise ValueError("state_indices and checkpoints are exclusive")
        output_final_state = False
    if output_final_state and final_state is None:
        final_state = torch.empty(N, HO, K, V, dtype=torch.float32, device=dev)
    if not output_final_state:
        final_state = None
    if checkpoint_every_n and checkpoints is None:
        R = checkpoint_rows_hint if checkpoint_rows_hint is not None else checkpoint_rows(cu_seqlens, checkpoint_every_n)
        checkpoints = torch.empty(R, HO, K, V, dtype=checkpoint_dtype, device=dev)
    if workspace is None:
        need = workspace_bytes(N) if n <= 1 else B.load().la_gdp_workspace_bytes(T, N, HK, HV, K, V, n)
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    if initial_state is not None and state_indices is None:
        initial_state = initial_state.contiguous()
    p = B.GdnFwdParams()
    p.num_householder = n
    p.q, p.q_stride_t, p.q_stride_h = q.data_ptr(), q.stride(0), q.stride(1)
    p.k, p.k_stride_t, p.k_stride_h = k.data_ptr(), k.stride(0), k.stride(1)
    p.v, p.v_stride_t, p.v_stride_h = v.data_ptr(), v.stride(0), v.stride(1)
    p.g, p.g_stride_t, p.g_stride_h = g.data_ptr(), g.stride(0), g.stride(1)
    p.beta, p.beta_stride_t, p.beta_stride_h = beta.data_ptr(), beta.stride(0), beta.stride(1)
    p.cu_seqlens, p.cu_seqlens_bits = cu_seqlens.data_ptr(), _cu_bits(cu_seqlens)
    p.T, p.N, p.HK, p.HV, p.K, p.V = T, N, HK, HV, K, V
    p.scale = float(scale) if scale is not None else 1.0 / math.sqrt(K)
    p.use_qk_l2norm = int(bool(use_qk_l2norm))
    if initial_state is not None:
        p.initial_state = initial_state.data_ptr()
        p.initial_state_dtype = B.LA_DTYPE_BF16 if initial_state.dtype == torch.bfloat16 else B.LA_DTYPE_F32
    p.o, p.o_stride_t, p.o_stride_h = o.data_ptr(), o.stride(0), o.stride(1)
    p.final_state = final_state.data_ptr() if final_state is not None else None
    if checkpoints is not None:
        p.checkpoints = checkpoints.data_ptr()
        p.checkpoint_dtype = B.LA_DTYPE_BF16 if checkpoints.dtype == torch.bfloat16 else B.LA_DTYPE_F32
        p.checkpoint_every_n = int(checkpoint_every_n)
    p.workspace, p.workspace_bytes = workspace.data_ptr(), workspace.numel()
    p.status = status.data_ptr() if status is not None else None
    keep = _set_transforms(p, HO, dev, a_log, dt_bias, gate_lower_bound, beta_sigmoid, beta)  # noqa: F841
    if state_indices is not None:
        p.state_indices, p.state_pool_size = state_indices.data_ptr(), initial_state.shape[0]
    B.check(B.load().gdn_fwd(ctypes.byref(p), _stream_ptr(stream)), "gdn_fwd")
    return o, final_state, checkpoints


def gdn_summary(k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
                cu_seqlens: torch.Tensor, *, use_qk_l2norm: bool = True,
                start_state: Optional[torch.Tensor] = None, end_state: Optional[torch.Tensor] = None,
                transition: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                status: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None,
                a_log: Optional[torch.Tensor] = None, dt_bias: Optional[torch.Tensor] = None,
                gate_lower_bound: Optional[float] = None, beta_sigmoid: bool = False
                ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Span summary.  Returns (end_state [N, HO, K, V] fp32, transition [N, HO, K, K] fp32) with
    end_state = einsum('ab,av->bv', transition, S_init) + S_H across spans.  The gate and beta
    transforms are as in gdn_fwd."""
    _check_thd("k", k, torch.bfloat16)
    _check_thd("v", v, torch.bfloat16)
    _check_thd("g", g, torch.float32, heads_dim=False)
    _check_beta(beta, beta_sigmoid)
    T, HK, K = k.shape
    HV, V = v.shape[1], v.shape[2]
    N = cu_seqlens.numel() - 1
    HO = HV
    dev = k.device
    if end_state is None:
        end_state = torch.empty(N, HO, K, V, dtype=torch.float32, device=dev)
    if transition is None:
        transition = torch.empty(N, HO, K, K, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(workspace_bytes(N, True), dtype=torch.uint8, device=dev)
    if start_state is not None:
        start_state = start_state.contiguous()
    p = B.GdnSummaryParams()
    p.k, p.k_stride_t, p.k_stride_h = k.data_ptr(), k.stride(0), k.stride(1)
    p.v, p.v_stride_t, p.v_stride_h = v.data_ptr(), v.stride(0), v.stride(1)
    p.g, p.g_stride_t, p.g_stride_h = g.data_ptr(), g.stride(0), g.stride(1)
    p.beta, p.beta_stride_t, p.beta_stride_h = beta.data_ptr(), beta.stride(0), beta.stride(1)
    p.cu_seqlens, p.cu_seqlens_bits = cu_seqlens.data_ptr(), _cu_bits(cu_seqlens)
    p.T, p.N, p.HK, p.HV, p.K, p.V = T, N, HK, HV, K, V
    p.use_qk_l2norm = int(bool(use_qk_l2norm))
    if start_state is not None:
        p.start_state = start_state.data_ptr()
        p.start_state_dtype = B.LA_DTYPE_BF16 if start_state.dtype == torch.bfloat16 else B.LA_DTYPE_F32
    p.end_state = end_state.data_ptr()
    p.transition = transition.data_ptr()
    p.workspace, p.workspace_bytes = workspace.data_ptr(), workspace.numel()
    p.status = status.data_ptr() if status is not None else None
    keep = _set_transforms(p, HO, dev, a_log, dt_bias, gate_lower_bound, beta_sigmoid, beta)  # noqa: F841
    B.check(B.load().gdn_summary(ctypes.byref(p), _stream_ptr(stream)), "gdn_summary")
    return end_state, transition


def gdn_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
            cu_seqlens: torch.Tensor, d_o: torch.Tensor, *, scale: Optional[float] = None,
            use_qk_l2norm: bool = True, initial_state: Optional[torch.Tensor] = None,
            d_final_state: Optional[torch.Tensor] = None, checkpoints: Optional[torch.Tensor] = None,
            workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
            stream: Optional[torch.cuda.Stream] = None, a_log: Optional[torch.Tensor] = None,
            dt_bias: Optional[torch.Tensor] = None, gate_lower_bound: Optional[float] = None,
            beta_sigmoid: bool = False, out: Optional[Tuple[Optional[torch.Tensor], ...]] = None):
    """Backward of gdn_fwd: returns (dq, dk, dv, dg, dbeta, d_initial_state or None) for the loss
    sum(d_o * o) + sum(d_final_state * final_state).  `checkpoints`, if given, are the forward's
    fp32 checkpoints every 64 tokens; otherwise the forward is re-run for them.  With the input
    transforms of gdn_fwd, dg and dbeta are the gradients of the raw inputs, and the softplus
    gate (a_log, dt_bias) appends (d_a_log, d_dt_bias) [HO] fp32 to the tuple.

    out: optional preallocated (dq, dk, dv, dg, dbeta, d_initial_state) buffers (any entry None
    is allocated); dq/dk/dv/dg/dbeta may be strided views, d_initial_state is contiguous."""
    _check_thd("q", q, torch.bfloat16)
    _check_thd("k", k, torch.bfloat16)
    _check_thd("v", v, torch.bfloat16)
    _check_thd("g", g, torch.float32, heads_dim=False)
    _check_beta(beta, beta_sigmoid)
    _check_thd("d_o", d_o, torch.bfloat16)
    T, HK, K = k.shape
    HV, V = v.shape[1], v.shape[2]
    N = cu_seqlens.numel() - 1
    dev = q.device
    o6 = tuple(out) + (None,) * (6 - len(out)) if out is not None else (None,) * 6
    if len(o6) != 6:
        raise ValueError("out holds at most (dq, dk, dv, dg, dbeta, d_initial_state)")
    dq = _out("dq", o6[0], (T, HK, K), torch.bfloat16, dev)
    dk = _out("dk", o6[1], (T, HK, K), torch.bfloat16, dev)
    dv = _out("dv", o6[2], (T, HV, V), torch.bfloat16, dev)
    dg = _out("dg", o6[3], (T, HV), torch.float32, dev)
    db = _out("dbeta", o6[4], (T, HV), torch.float32, dev)
    ds0 = _out("d_initial_state", o6[5], (N, HV, K, V), torch.float32, dev, contiguous=True) \
        if initial_state is not None else None
    lib = B.load()
    if workspace is None:
        need = lib.la_gdn_bwd_workspace_bytes(T, N, HK, HV, K, V, int(checkpoints is not None))
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    if initial_state is not None:
        initial_state = initial_state.contiguous()
    if d_final_state is not None:
        d_final_state = d_final_state.contiguous().float()
    if checkpoints is not None:
        if checkpoints.dtype != torch.float32 or not checkpoints.is_contiguous():
            raise ValueError("checkpoints must be the forward's contiguous fp32 rows every 64 tokens")
    p = B.GdnBwdParams()
    p.q, p.q_stride_t, p.q_stride_h = q.data_ptr(), q.stride(0), q.stride(1)
    p.k, p.k_stride_t, p.k_stride_h = k.data_ptr(), k.stride(0), k.stride(1)
    p.v, p.v_stride_t, p.v_stride_h = v.data_ptr(), v.stride(0), v.stride(1)
    p.g, p.g_stride_t, p.g_stride_h = g.data_ptr(), g.stride(0), g.stride(1)
    p.beta, p.beta_stride_t, p.beta_stride_h = beta.data_ptr(), beta.stride(0), beta.stride(1)
    p.cu_seqlens, p.cu_seqlens_bits = cu_seqlens.data_ptr(), _cu_bits(cu_seqlens)
    p.T, p.N, p.HK, p.HV, p.K, p.V = T, N, HK, HV, K, V
    p.scale = float(scale) if scale is not None else 1.0 / math.sqrt(K)
    p.use_qk_l2norm = int(bool(use_qk_l2norm))
    if initial_state is not None:
        p.initial_state = initial_state.data_ptr()
        p.initial_state_dtype = B.LA_DTYPE_BF16 if initial_state.dtype == torch.bfloat16 else B.LA_DTYPE_F32
    p.checkpoints = checkpoints.data_ptr() if checkpoints is not None else None
    p.d_o, p.d_o_stride_t, p.d_o_stride_h = d_o.data_ptr(), d_o.stride(0), d_o.stride(1)
    p.d_final_state = d_final_state.data_ptr() if d_final_state is not None else None
    p.dq, p.dq_stride_t, p.dq_stride_h = dq.data_ptr(), dq.stride(0), dq.stride(1)
    p.dk, p.dk_stride_t, p.dk_stride_h = dk.data_ptr(), dk.stride(0), dk.stride(1)
    p.dv, p.dv_stride_t, p.dv_stride_h = dv.data_ptr(), dv.stride(0), dv.stride(1)
    p.dg, p.dg_stride_t, p.dg_stride_h = dg.data_ptr(), dg.stride(0), dg.stride(1)
    p.dbeta, p.dbeta_stride_t, p.dbeta_stride_h = db.data_ptr(), db.stride(0), db.stride(1)
    p.d_initial_state = ds0.data_ptr() if ds0 is not None else None
    p.workspace, p.workspace_bytes = workspace.data_ptr(), workspace.numel()
    p.status = status.data_ptr() if status is not None else None
    keep = _set_transforms(p, HV, dev, a_log, dt_bias, gate_lower_bound, beta_sigmoid, beta)  # noqa: F841
    extra = ()
    if a_log is not None:
        da = torch.empty(HV, dtype=torch.float32, device=dev)
        ddt = torch.empty(HV, dtype=torch.float32, device=dev)
        p.d_a_log, p.d_dt_bias = da.data_ptr(), ddt.data_ptr()
        extra = (da, ddt)
    B.check(lib.gdn_bwd(ctypes.byref(p), _stream_ptr(stream)), "gdn_bwd")
    return (dq, dk, dv, dg, db, ds0) + extra


def gdn_summary_bwd(q: torch.Tensor, k: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
                    cu_seqlens: torch.Tensor, d_o: torch.Tensor, *, scale: Optional[float] = None,
                    use_qk_l2norm: bool = True, d_final_state: Optional[torch.Tensor] = None,
                    workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                    stream: Optional[torch.cuda.Stream] = None, a_log: Optional[torch.Tensor] = None,
                    dt_bias: Optional[torch.Tensor] = None, gate_lower_bound: Optional[float] = None,
                    beta_sigmoid: bool = False, d_state: Optional[torch.Tensor] = None) -> torch.Tensor:
    """State-gradient mirror of gdn_summary: for each span (sequence) the gradient of
    sum(d_o * o) + sum(d_final_state * end_state) with respect to the state entering the span,
    [N, HO, K, V] fp32.  It depends on neither that state nor v; with gdn_summary's transition,
    d_enter = einsum('ab,bv->av', transition, d_exit) + (the value for d_exit = 0).  Gate and
    beta transforms as in gdn_fwd.  d_state: optional preallocated contiguous output."""
    _check_thd("q", q, torch.bfloat16)
    _check_thd("k", k, torch.bfloat16)
    _check_thd("g", g, torch.float32, heads_dim=False)
    _check_beta(beta, beta_sigmoid)
    _check_thd("d_o", d_o, torch.bfloat16)
    T, HK, K = k.shape
    HV, V = d_o.shape[1], d_o.shape[2]
    N = cu_seqlens.numel() - 1
    dev = q.device
    d_state = _out("d_state", d_state, (N, HV, K, V), torch.float32, dev, contiguous=True)
    lib = B.load()
    if workspace is None:
        workspace = torch.empty(lib.la_gdn_summary_bwd_workspace_bytes(N, HV, K, V), dtype=torch.uint8, device=dev)
    if d_final_state is not None:
        d_final_state = d_final_state.contiguous().float()
    p = B.GdnSummaryBwdParams()
    p.q, p.q_stride_t, p.q_stride_h = q.data_ptr(), q.stride(0), q.stride(1)
    p.k, p.k_stride_t, p.k_stride_h = k.data_ptr(), k.stride(0), k.stride(1)
    p.g, p.g_stride_t, p.g_stride_h = g.data_ptr(), g.stride(0), g.stride(1)
    p.beta, p.beta_stride_t, p.beta_stride_h = beta.data_ptr(), beta.stride(0), beta.stride(1)
    p.cu_seqlens, p.cu_seqlens_bits = cu_seqlens.data_ptr(), _cu_bits(cu_seqlens)
    p.T, p.N, p.HK, p.HV, p.K, p.V = T, N, HK, HV, K, V
    p.scale = float(scale) if scale is not None else 1.0 / math.sqrt(K)
    p.use_qk_l2norm = int(bool(use_qk_l2norm))
    p.d_o, p.d_o_stride_t, p.d_o_stride_h = d_o.data_ptr(), d_o.stride(0), d_o.stride(1)
    p.d_final_state = d_final_state.data_ptr() if d_final_state is not None else None
    p.d_state = d_state.data_ptr()
    p.workspace, p.workspace_bytes = workspace.data_ptr(), workspace.numel()
    p.status = status.data_ptr() if status is not None else None
    keep = _set_transforms(p, HV, dev, a_log, dt_bias, gate_lower_bound, beta_sigmoid, beta)  # noqa: F841
    B.check(lib.gdn_summary_bwd(ctypes.byref(p), _stream_ptr(stream)), "gdn_summary_bwd")
    return d_state


def gdn_decode(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
               state_pool: torch.Tensor, *, state_indices: Optional[torch.Tensor] = None,
               scale: Optional[float] = None, use_qk_l2norm: bool = True, o: Optional[torch.Tensor] = None,
               status: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None,
               a_log: Optional[torch.Tensor] = None, dt_bias: Optional[torch.Tensor] = None,
               gate_lower_bound: Optional[float] = None, beta_sigmoid: bool = False) -> torch.Tensor:
    """One new token for each of N sequences: q, k [N, HK, K], v [N, HV, V], g, beta [N, HO].
    Sequence i steps the state pool[state_indices[i]] (pool[i] when state_indices is None) in
    place and returns o [N, HO, V] bf16.  Gate and beta transforms as in gdn_fwd."""
    _check_thd("q", q, torch.bfloat16)
    _check_thd("k", k, torch.bfloat16)
    _check_thd("v", v, torch.bfloat16)
    _check_thd("g", g, torch.float32, heads_dim=False)
    _check_beta(beta, beta_sigmoid)
    N, HK, K = k.shape
    HV, V = v.shape[1], v.shape[2]
    dev = q.device
    if state_pool.dim() != 4 or not state_pool.is_contiguous() or state_pool.shape[1:] != (HV, K, V):
        raise ValueError(f"state_pool must be a contiguous [P, {HV}, {K}, {V}] tensor")
    if state_pool.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("state_pool must be float32 or bfloat16")
    if state_indices is not None and (state_indices.dtype != torch.int32 or state_indices.numel() != N):
        raise ValueError(f"state_indices must be int32 [{N}]")
    if o is None:
        o = torch.empty(N, HV, V, dtype=torch.bfloat16, device=dev)
    p = B.GdnDecodeParams()
    p.q, p.q_stride_n, p.q_stride_h = q.data_ptr(), q.stride(0), q.stride(1)
    p.k, p.k_stride_n, p.k_stride_h = k.data_ptr(), k.stride(0), k.stride(1)
    p.v, p.v_stride_n, p.v_stride_h = v.data_ptr(), v.stride(0), v.stride(1)
    p.g, p.g_stride_n, p.g_stride_h = g.data_ptr(), g.stride(0), g.stride(1)
    p.beta, p.beta_stride_n, p.beta_stride_h = beta.data_ptr(), beta.stride(0), beta.stride(1)
    p.N, p.HK, p.HV, p.K, p.V = N, HK, HV, K, V
    p.scale = float(scale) if scale is not None else 1.0 / math.sqrt(K)
    p.use_qk_l2norm = int(bool(use_qk_l2norm))
    p.state_pool, p.state_pool_size = state_pool.data_ptr(), state_pool.shape[0]
    p.state_dtype = B.LA_DTYPE_BF16 if state_pool.dtype == torch.bfloat16 else B.LA_DTYPE_F32
    p.state_indices = state_indices.data_ptr() if state_indices is not None else None
    p.o, p.o_stride_n, p.o_stride_h = o.data_ptr(), o.stride(0), o.stride(1)
    p.status = status.data_ptr() if status is not None else None
    keep = _set_transforms(p, HV, dev, a_log, dt_bias, gate_lower_bound, beta_sigmoid, beta)  # noqa: F841
    B.check(B.load().gdn_decode(ctypes.byref(p), _stream_ptr(stream)), "gdn_decode")
    return o


def read_status(status: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronises the stream and returns the device status word (an la_status code)."""
    out = ctypes.c_int32(0)
    B.check(B.load().la_read_status(status.data_ptr(), _stream_ptr(stream), ctypes.byref(out)), "la_read_status")
    return int(out.value)


def _host_parts(lengths, groups, n):
    """The token ranges gdn_fwd_host pipelines, in packed order: runs of consecutive whole
    sequences of at most P tokens, and every sequence longer than P cut into pieces of P tokens,
    each piece a range of its own.  P is about total / groups, rounded up to a multiple of 64
    and of the checkpoint cadence n, so a cut falls on a chunk and checkpoint boundary.

    Returns (P, parts) with parts as tuples (t_a, t_b, a, b, piece, last): tokens t_a..t_b of
    the packed batch; a run holds sequences a..b-1 (piece = -1, last = True); a piece belongs to
    sequence a (b = a + 1), piece is its index within the sequence and last says whether it
    ends the sequence."""
    total = int(sum(lengths))
    unit = 64 if not n else 64 * int(n) // math.gcd(64, int(n))
    target = -(-total // max(1, int(groups))) if total else 1
    P = max(unit, -(-target // unit) * unit)
    parts = []
    t = 0
    run_a, run_t = 0, 0
    for i, L in enumerate(lengths):
        L = int(L)
        if L > P:
            if i > run_a:
                parts.append((run_t, t, run_a, i, -1, True))
            npc = -(-L // P)
            for pc in range(npc):
                parts.append((t + pc * P, t + min(L, (pc + 1) * P), i, i + 1, pc, pc == npc - 1))
            t += L
            run_a, run_t = i + 1, t
            continue
        if t + L - run_t > P and i > run_a:
            parts.append((run_t, t, run_a, i, -1, True))
            run_a, run_t = i, t
        t += L
    if len(lengths) > run_a:
        parts.append((run_t, t, run_a, len(lengths), -1, True))
    return P, parts


def gdn_fwd_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
                 cu_seqlens: torch.Tensor, *, scale: Optional[float] = None, use_qk_l2norm: bool = True,
                 initial_state: Optional[torch.Tensor] = None, output_final_state: bool = True,
                 checkpoint_every_n: int = 0, checkpoint_dtype: torch.dtype = torch.bfloat16,
                 out: Optional[Tuple[torch.Tensor, Optional[torch.Tensor], Optional[torch.Tensor]]] = None,
                 device: Optional[torch.device] = None, groups: int = 4, staging: Optional[dict] = None,
                 compute_streams: int = 8):
    """gdn_fwd on HOST tensors: copies in, computes, copies out, pipelined over token ranges.

    q, k, v, g, beta, cu_seqlens (and initial_state) are contiguous CPU tensors (pin them for
    asynchronous copies).  The packed batch is cut into ranges of about T / groups tokens (see
    _host_parts): runs of whole sequences, and long sequences cut into pieces at chunk and
    checkpoint boundaries, a piece starting from the state the previous piece ended in (fp32,
    on the device).  Each range's host-to-device copy, forward and device-to-host copy are
    ordered by events across a copy-in stream, `compute_streams` compute streams (the pieces of
    one sequence stay on one) and a copy-out stream, so copies overlap computation and the
    forward of a range starts as soon as its inputs have arrived.  Outputs are CPU tensors
    (pinned when `out` is not given).  Returns (o, final_state, checkpoints) once every copy is
    enqueued; the current stream is made to wait for them, so synchronise it (or an event
    recorded on it) before reading the outputs on the host.  The result is bitwise that of one
    gdn_fwd call: every sequence's results are independent of the batch around it, and a cut
    at a chunk boundary hands the exact fp32 state to the next piece, which continues the
    same chunk sequence with the same arithmetic.  `staging` may carry device buffers and
    streams from an earlier call of the same shapes to avoid reallocation.
    """
    dev = device or torch.device("cuda", torch.cuda.current_device())
    T, HK, K = k.shape
    HV, V = v.shape[1], v.shape[2]
    HO = HV
    N = cu_seqlens.numel() - 1
    cu = cu_seqlens.to(torch.int64)
    lengths = (cu[1:] - cu[:-1]).tolist()
    n = int(checkpoint_every_n or 0)
    rows = [(int(L) + n - 1) // n for L in lengths] if n else [0] * N
    if out is None:
        o_h = torch.empty(T, HO, V, dtype=torch.bfloat16).pin_memory()
        fin_h = torch.empty(N, HO, K, V, dtype=torch.float32).pin_memory() if output_final_state else None
        ck_h = torch.empty(sum(rows), HO, K, V, dtype=checkpoint_dtype).pin_memory() if n else None
    else:
        o_h, fin_h, ck_h = out
    st = staging if staging is not None else {}

    def dbuf(name, shape, dtype):
        t = st.get(name)
        if t is None or tuple(t.shape) != tuple(shape) or t.dtype != dtype:
            t = torch.empty(*shape, dtype=dtype, device=dev)
            st[name] = t
        return t

    qd, kd, vd = dbuf("q", q.shape, q.dtype), dbuf("k", k.shape, k.dtype), dbuf("v", v.shape, v.dtype)
    gd, bd = dbuf("g", g.shape, g.dtype), dbuf("beta", beta.shape, beta.dtype)
    s0d = dbuf("s0", initial_state.shape, initial_state.dtype) if initial_state is not None else None
    od = dbuf("o", o_h.shape, o_h.dtype)
    find = dbuf("fin", fin_h.shape, fin_h.dtype) if fin_h is not None else None
    ckd = dbuf("ck", ck_h.shape, ck_h.dtype) if ck_h is not None else None
    _, parts = _host_parts(lengths, groups, n)
    long_seqs = sorted({a for (_, _, a, _, pc, _) in parts if pc >= 0})
    # the state between two pieces of a long sequence: two fp32 slots per such sequence
    mid = dbuf("mid", (max(1, len(long_seqs)), 2, HO, K, V), torch.float32) if long_seqs else None
    slot = {j: x for x, j in enumerate(long_seqs)}
    cur = torch.cuda.current_stream(dev)
    h2d = st.setdefault("h2d_stream", torch.cuda.Stream(dev))
    d2h = st.setdefault("d2h_stream", torch.cuda.Stream(dev))
    ncs = max(1, int(compute_streams))
    css = [st.setdefault(f"compute_stream{x}", torch.cuda.Stream(dev)) for x in range(ncs)]
    h2d.wait_stream(cur)
    d2h.wait_stream(cur)
    for cs in css:
        cs.wait_stream(cur)
    row_off = [0]
    for r_ in rows:
        row_off.append(row_off[-1] + r_)
    # every range's cu_seqlens in one pinned buffer and one copy ahead of the inputs (a copy from
    # pageable memory would make the host wait for the copies already queued)
    cu_list, cu_at = [], []
    for (t_a, t_b, a, b, pc, _) in parts:
        cu_at.append(len(cu_list))
        cu_list += (cu[a:b + 1] - int(cu[a])).tolist() if pc < 0 else [0, t_b - t_a]
    with torch.cuda.stream(h2d):
        cu_all = torch.tensor(cu_list, dtype=torch.int32).pin_memory().to(dev, non_blocking=True) \
            if cu_list else None
    seq_stream = {}
    for pi, (t_a, t_b, a, b, pc, last) in enumerate(parts):
        with torch.cuda.stream(h2d):
            for dst, src in ((qd, q), (kd, k), (vd, v), (gd, g), (bd, beta)):
                dst[t_a:t_b].copy_(src[t_a:t_b], non_blocking=True)
            if s0d is not None and pc <= 0:
                s0d[a:b].copy_(initial_state[a:b], non_blocking=True)
            ev_in = torch.cuda.Event()
            ev_in.record(h2d)
        cu_d = cu_all[cu_at[pi]:cu_at[pi] + (b - a + 1 if pc < 0 else 2)]
        cs = css[seq_stream.setdefault(a, len(seq_stream) % ncs)] if pc >= 0 else css[pi % ncs]
        cs.wait_event(ev_in)
        if pc < 0:
            s_in = s0d[a:b] if s0d is not None else None
            s_out = find[a:b] if find is not None else None
            r_a, r_b = row_off[a], row_off[b]
        else:
            m = mid[slot[a]]
            s_in = (s0d[a:b] if s0d is not None else None) if pc == 0 else m[(pc - 1) % 2:(pc - 1) % 2 + 1]
            s_out = (find[a:b] if find is not None else None) if last else m[pc % 2:pc % 2 + 1]
            off = int(cu[a])
            r_a = row_off[a] + ((t_a - off) // n if n else 0)
            r_b = row_off[a] + ((t_b - off + n - 1) // n if n else 0)
        with torch.cuda.stream(cs):
            gdn_fwd(qd[t_a:t_b], kd[t_a:t_b], vd[t_a:t_b], gd[t_a:t_b], bd[t_a:t_b], cu_d, scale=scale,
                    use_qk_l2norm=use_qk_l2norm, initial_state=s_in, output_final_state=s_out is not None,
                    checkpoint_every_n=n, checkpoint_dtype=checkpoint_dtype, checkpoint_rows_hint=r_b - r_a,
                    o=od[t_a:t_b], final_state=s_out, checkpoints=ckd[r_a:r_b] if ckd is not None else None,
                    stream=cs)
            cu_all.record_stream(cs)
            ev_c = torch.cuda.Event()
            ev_c.record(cs)
        d2h.wait_event(ev_c)
        with torch.cuda.stream(d2h):
            o_h[t_a:t_b].copy_(od[t_a:t_b], non_blocking=True)
            if fin_h is not None and last:
                fin_h[a:b].copy_(find[a:b], non_blocking=True)
            if ck_h is not None and r_b > r_a:
                ck_h[r_a:r_b].copy_(ckd[r_a:r_b], non_blocking=True)
    cur.wait_stream(d2h)
    for cs in css:
        cur.wait_stream(cs)
    return o_h, fin_h, ck_h
