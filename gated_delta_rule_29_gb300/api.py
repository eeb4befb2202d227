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


def split_workspace_bytes(T: int, N: int, HV: int) -> int:
    """Workspace with which gdn_fwd may run as two passes (the same bits as the fused kernel)."""
    return int(B.load().la_gdn_fwd_split_workspace_bytes(int(T), int(N), int(HV)))


def _workspace(preferred: int, minimum: int, dev: torch.device) -> torch.Tensor:
    """A device workspace of `preferred` bytes (room for the two-pass schedules, about 272 bytes
    per token and head), or of `minimum` bytes when that allocation fails: the library then takes
    its single-kernel path, as it does for any smaller workspace."""
    try:
        return torch.empty(preferred, dtype=torch.uint8, device=dev)
    except torch.cuda.OutOfMemoryError:
        return torch.empty(minimum, dtype=torch.uint8, device=dev)


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
        need = split_workspace_bytes(T, N, HV) if n <= 1 else B.load().la_gdp_workspace_bytes(T, N, HK, HV, K, V, n)
        # n > 64 needs its whole timeline workspace; otherwise the minimum is the prologue's tables
        workspace = _workspace(need, workspace_bytes(N) if n <= 64 else need, dev)
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
        workspace = _workspace(split_workspace_bytes(k.shape[0], N, v.shape[1]), workspace_bytes(N, True), dev)
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
            beta_sigmoid: bool = False, out: Optional[Tuple[Optional[torch.Tensor], ...]] = None,
            checkpoint_every_n: int = 64):
    """Backward of gdn_fwd: returns (dq, dk, dv, dg, dbeta, d_initial_state or None) for the loss
    sum(d_o * o) + sum(d_final_state * final_state).  `checkpoints`, if given, are the forward's
    checkpoints (fp32 or bf16) every `checkpoint_every_n` tokens (a multiple of 64): rows every 64
    tokens are used directly (bf16 widened), sparser rows regenerate the states entering every
    chunk segment by segment; without them the forward is re-run.  With the input
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
    ck_n = int(checkpoint_every_n) if checkpoints is not None else 0
    ck_bf16 = checkpoints is not None and checkpoints.dtype == torch.bfloat16
    if checkpoints is not None:
        if checkpoints.dtype not in (torch.float32, torch.bfloat16) or not checkpoints.is_contiguous():
            raise ValueError("checkpoints must be the forward's contiguous fp32 or bf16 rows")
        if ck_n <= 0 or ck_n % 64 != 0:
            raise ValueError("checkpoint_every_n must be a positive multiple of 64")
    if workspace is None:
        workspace = _workspace(lib.la_gdn_bwd_workspace_bytes_ckpt(T, N, HK, HV, K, V, ck_n, int(ck_bf16)),
                               lib.la_gdn_bwd_workspace_bytes_min(T, N, HK, HV, K, V, ck_n, int(ck_bf16)), dev)
    if initial_state is not None:
        initial_state = initial_state.contiguous()
    if d_final_state is not None:
        d_final_state = d_final_state.contiguous().float()
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
    p.checkpoint_every_n, p.checkpoint_bf16 = ck_n, int(ck_bf16)
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
        # room for the tensor-core path (the forward's WY records), else the tile kernel's minimum
        tile = int(lib.la_gdn_summary_bwd_workspace_bytes(N, HV, K, V))
        workspace = _workspace(max(tile, split_workspace_bytes(q.shape[0], N, HV)), tile, dev)
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


def compose_spans(transitions: torch.Tensor, terms: torch.Tensor, start: Optional[torch.Tensor] = None, *,
                  backward: bool = False, out: Optional[torch.Tensor] = None,
                  stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Composition of span summaries on the GPU (gdn_compose_spans).  transitions [R, HO, K, K]
    and terms [R, HO, K, V] fp32 on one CUDA device; start [HO, K, V] or None (zeros).
    Forward: returns [R + 1, HO, K, V], the state entering each span and the final state.
    Backward (terms = each span's own entering-state gradient, start = the cotangent after the
    last span): the cotangent leaving each span, then the gradient entering span 0."""
    if transitions.dim() != 4 or terms.dim() != 4:
        raise ValueError("transitions [R, HO, K, K] and terms [R, HO, K, V] expected")
    R, HO, K, V = terms.shape
    if tuple(transitions.shape) != (R, HO, K, K):
        raise ValueError(f"transitions must be [{R}, {HO}, {K}, {K}], got {tuple(transitions.shape)}")
    dev = terms.device
    for name, x in (("transitions", transitions), ("terms", terms), ("start", start)):
        if x is not None and (x.dtype != torch.float32 or x.device != dev or dev.type != "cuda"):
            raise ValueError(f"{name} must be fp32 on the CUDA device of terms")
    if start is not None and tuple(start.shape) != (HO, K, V):
        raise ValueError(f"start must be [{HO}, {K}, {V}]")
    transitions, terms = transitions.contiguous(), terms.contiguous()
    start = start.contiguous() if start is not None else None
    if out is None:
        out = torch.empty(R + 1, HO, K, V, dtype=torch.float32, device=dev)
    p = B.GdnComposeParams()
    p.R, p.HO, p.K, p.V = R, HO, K, V
    p.transitions, p.terms = transitions.data_ptr(), terms.data_ptr()
    p.start = start.data_ptr() if start is not None else None
    p.out = out.data_ptr()
    p.backward = int(bool(backward))
    B.check(B.load().gdn_compose_spans(ctypes.byref(p), _stream_ptr(stream)), "gdn_compose_spans")
    return out


def read_status(status: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronises the stream and returns the device status word (an la_status code)."""
    out = ctypes.c_int32(0)
    B.check(B.load().la_read_status(status.data_ptr(), _stream_ptr(stream), ctypes.byref(out)), "la_read_status")
    return int(out.value)


def _host_parts(lengths, groups, n):
    """The token ranges gdn_fwd_host pipelines (the library's plan, la_gdn_fwd_host_plan): runs
    of whole sequences of at most P tokens, and sequences longer than P cut into pieces of P
    tokens, P about total / groups rounded up to a multiple of 64 and of the checkpoint cadence
    n.  Returns (P, parts), parts as tuples (t_a, t_b, a, b, piece, last)."""
    acc, cu = 0, [0]
    for L in lengths:
        acc += int(L)
        cu.append(acc)
    cu_t = torch.tensor(cu, dtype=torch.int64)
    lib = B.load()
    P = ctypes.c_int64(0)
    args = (cu_t.data_ptr(), 64, len(lengths), max(1, int(groups)), int(n or 0))
    cnt = lib.la_gdn_fwd_host_plan(*args, None, 0, ctypes.byref(P))
    if cnt < 0:
        raise ValueError("invalid lengths, groups or checkpoint cadence")
    rows = (ctypes.c_int64 * (6 * max(cnt, 1)))()
    lib.la_gdn_fwd_host_plan(*args, rows, cnt, ctypes.byref(P))
    parts = [tuple(int(rows[6 * i + j]) for j in range(5)) + (bool(rows[6 * i + 5]),) for i in range(cnt)]
    return int(P.value), parts


def _check_host(name, x, dtype, dims):
    if not isinstance(x, torch.Tensor) or x.is_cuda or x.dtype != dtype or x.dim() != dims or not x.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CPU {dtype} tensor of rank {dims} (pinned for overlap)")


def gdn_fwd_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
                 cu_seqlens: torch.Tensor, *, scale: Optional[float] = None, use_qk_l2norm: bool = True,
                 initial_state: Optional[torch.Tensor] = None, output_final_state: bool = True,
                 checkpoint_every_n: int = 0, checkpoint_dtype: torch.dtype = torch.bfloat16,
                 out: Optional[Tuple[torch.Tensor, Optional[torch.Tensor], Optional[torch.Tensor]]] = None,
                 device: Optional[torch.device] = None, groups: int = 16, staging: Optional[dict] = None,
                 status: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None,
                 a_log: Optional[torch.Tensor] = None, dt_bias: Optional[torch.Tensor] = None,
                 gate_lower_bound: Optional[float] = None, beta_sigmoid: bool = False):
    """gdn_fwd on HOST tensors through the library's gdn_fwd_host: copy in, forward, copy out,
    pipelined over about `groups` token ranges on the library's own streams.

    q, k, v, g, beta, initial_state are contiguous CPU tensors (pin them so the copies run
    asynchronously), cu_seqlens a CPU int32/int64 tensor; a_log and dt_bias, with the softplus
    gate, CPU float32 [HO].  Outputs (o, final_state, checkpoints) are CPU tensors (pinned when
    `out` is not given).  Returns once everything is enqueued, with the stream made to wait for
    the last copy out: synchronise it before reading the outputs, and keep the inputs alive and
    unchanged until then.  The result is bitwise that of one gdn_fwd call.  `staging` (a dict)
    keeps the device staging buffer from one call to the next: a call with the same buffer is
    ordered after the previous call that used it rather than after the stream, so alternating two
    dicts lets one call's copies run under the previous call's last forwards.  The status word, if
    given, is a device int32 tensor as for gdn_fwd."""
    dev = device or torch.device("cuda", torch.cuda.current_device())
    _check_host("q", q, torch.bfloat16, 3)
    _check_host("k", k, torch.bfloat16, 3)
    _check_host("v", v, torch.bfloat16, 3)
    _check_host("g", g, torch.float32, 2)
    beta_bf16 = beta_sigmoid and beta.dtype == torch.bfloat16
    _check_host("beta", beta, torch.bfloat16 if beta_bf16 else torch.float32, 2)
    T, HK, K = k.shape
    HV, V = v.shape[1], v.shape[2]
    HO = HV
    cu = cu_seqlens.detach().to("cpu").contiguous()
    N = cu.numel() - 1
    if N < 0 or int(cu[0]) != 0 or int(cu[-1]) != T or bool((cu[1:] < cu[:-1]).any()):
        raise ValueError("cu_seqlens must start at 0, be nondecreasing and end at T")
    n = int(checkpoint_every_n or 0)
    R = checkpoint_rows(cu, n) if n else 0
    if out is None:
        o_h = torch.empty(T, HO, V, dtype=torch.bfloat16).pin_memory()
        fin_h = torch.empty(N, HO, K, V, dtype=torch.float32).pin_memory() if output_final_state else None
        ck_h = torch.empty(R, HO, K, V, dtype=checkpoint_dtype).pin_memory() if n else None
    else:
        o_h, fin_h, ck_h = out
    _check_host("o", o_h, torch.bfloat16, 3)
    if fin_h is not None:
        _check_host("final_state", fin_h, torch.float32, 4)
    if ck_h is not None:
        _check_host("checkpoints", ck_h, checkpoint_dtype, 4)
    hp = B.GdnFwdHostParams()
    p = hp.fwd
    p.q, p.q_stride_t, p.q_stride_h = q.data_ptr(), HK * K, K
    p.k, p.k_stride_t, p.k_stride_h = k.data_ptr(), HK * K, K
    p.v, p.v_stride_t, p.v_stride_h = v.data_ptr(), HV * V, V
    p.g, p.g_stride_t, p.g_stride_h = g.data_ptr(), HO, 1
    p.beta, p.beta_stride_t, p.beta_stride_h = beta.data_ptr(), HO, 1
    p.cu_seqlens, p.cu_seqlens_bits = cu.data_ptr(), _cu_bits(cu)
    p.T, p.N, p.HK, p.HV, p.K, p.V = T, N, HK, HV, K, V
    p.scale = float(scale) if scale is not None else 1.0 / math.sqrt(K)
    p.use_qk_l2norm = int(bool(use_qk_l2norm))
    if initial_state is not None:
        _check_host("initial_state", initial_state, initial_state.dtype, 4)
        p.initial_state = initial_state.data_ptr()
        p.initial_state_dtype = B.LA_DTYPE_BF16 if initial_state.dtype == torch.bfloat16 else B.LA_DTYPE_F32
    p.o, p.o_stride_t, p.o_stride_h = o_h.data_ptr(), HO * V, V
    p.final_state = fin_h.data_ptr() if fin_h is not None else None
    if ck_h is not None:
        p.checkpoints = ck_h.data_ptr()
        p.checkpoint_dtype = B.LA_DTYPE_BF16 if ck_h.dtype == torch.bfloat16 else B.LA_DTYPE_F32
        p.checkpoint_every_n = n
    p.status = status.data_ptr() if status is not None else None
    if (a_log is None) != (dt_bias is None):
        raise ValueError("the softplus gate needs both a_log and dt_bias")
    if a_log is not None:
        if gate_lower_bound is not None:
            raise ValueError("choose one gate transform: (a_log, dt_bias) or gate_lower_bound")
        for name, x in (("a_log", a_log), ("dt_bias", dt_bias)):
            _check_host(name, x, torch.float32, 1)
            if x.numel() != HO:
                raise ValueError(f"{name} must hold {HO} elements")
        p.gate_mode, p.a_log, p.dt_bias = B.LA_GATE_SOFTPLUS, a_log.data_ptr(), dt_bias.data_ptr()
    elif gate_lower_bound is not None:
        p.gate_mode, p.gate_lower_bound = B.LA_GATE_SIGMOID_BOUND, float(gate_lower_bound)
    p.beta_sigmoid = int(bool(beta_sigmoid))
    p.beta_bf16 = int(beta_bf16)
    hp.ranges = max(1, int(groups))
    lib = B.load()
    need = int(lib.la_gdn_fwd_host_staging_bytes(ctypes.byref(hp)))
    if need == 0:
        raise ValueError("gdn_fwd_host: invalid arguments (shapes, cu_seqlens or options)")
    st = staging if staging is not None else {}
    buf = st.get("staging")
    if buf is None or buf.numel() < need or buf.device != dev:
        with torch.cuda.stream(stream if stream is not None else torch.cuda.current_stream(dev)):
            buf = torch.empty(need, dtype=torch.uint8, device=dev)
        st["staging"] = buf
    hp.staging, hp.staging_bytes = buf.data_ptr(), buf.numel()
    B.check(lib.gdn_fwd_host(ctypes.byref(hp), _stream_ptr(stream)), "gdn_fwd_host")
    return o_h, fin_h, ck_h
