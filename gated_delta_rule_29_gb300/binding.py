"""ctypes binding of liblinattn (include/liblinattn.h), argument marshalling only.

Every step of the computation runs in the library's CUDA kernels.  There is no
fallback: if the shared library cannot be built or loaded, importing the
functions below raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

LA_OK = 0
LA_ERR_INVALID_ARG = 1
LA_ERR_UNSUPPORTED = 2
LA_ERR_CUDA = 3
LA_ERR_BAD_SEQLENS = 4
LA_ERR_TIMEOUT = 5
LA_ERR_WORKSPACE = 6
LA_ERR_BAD_STATE_INDEX = 7

LA_DTYPE_BF16 = 0
LA_DTYPE_F32 = 1
LA_GATE_LOG = 0
LA_GATE_SOFTPLUS = 1
LA_GATE_SIGMOID_BOUND = 2

EXPORTED_SYMBOLS = (
    "gdn_fwd",
    "gdn_summary",
    "la_gdn_workspace_bytes",
    "la_gdn_fwd_split_workspace_bytes",
    "la_checkpoint_rows",
    "la_read_status",
    "la_status_string",
    "la_version",
    "la_set_kernel_timing_events",
    "la_test_set_wait_hooks",
    "la_test_set_fwd_pieces",
    "la_test_set_fwd_passes",
    "gdn_compose_spans",
    "gdn_fwd_static_workspace",
    "gdn_decode",
    "gdn_bwd",
    "la_gdn_bwd_workspace_bytes",
    "la_gdn_bwd_workspace_bytes_ckpt",
    "la_gdn_bwd_workspace_bytes_min",
    "la_gdp_workspace_bytes",
    "gdn_summary_bwd",
    "la_gdn_summary_bwd_workspace_bytes",
    "gdn_fwd_host",
    "la_gdn_fwd_host_staging_bytes",
    "la_gdn_fwd_host_plan",
)

_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_vp = ctypes.c_void_p


class GdnFwdParams(ctypes.Structure):
    """Mirror of la_gdn_fwd_params (same field order and types)."""
    _fields_ = [
        ("q", _vp), ("q_stride_t", _i64), ("q_stride_h", _i64),
        ("k", _vp), ("k_stride_t", _i64), ("k_stride_h", _i64),
        ("v", _vp), ("v_stride_t", _i64), ("v_stride_h", _i64),
        ("g", _vp), ("g_stride_t", _i64), ("g_stride_h", _i64),
        ("beta", _vp), ("beta_stride_t", _i64), ("beta_stride_h", _i64),
        ("cu_seqlens", _vp), ("cu_seqlens_bits", _i32),
        ("T", _i64),
        ("N", _i32), ("HK", _i32), ("HV", _i32), ("K", _i32), ("V", _i32),
        ("scale", ctypes.c_float), ("use_qk_l2norm", _i32),
        ("initial_state", _vp), ("initial_state_dtype", _i32),
        ("o", _vp), ("o_stride_t", _i64), ("o_stride_h", _i64),
        ("final_state", _vp),
        ("checkpoints", _vp), ("checkpoint_dtype", _i32), ("checkpoint_every_n", _i64),
        ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t),
        ("status", _vp),
        ("gate_mode", _i32), ("a_log", _vp), ("dt_bias", _vp), ("gate_lower_bound", ctypes.c_float),
        ("beta_sigmoid", _i32), ("beta_bf16", _i32),
        ("state_indices", _vp), ("state_pool_size", _i64),
        ("num_householder", _i32),
    ]


class GdnFwdHostParams(ctypes.Structure):
    """Mirror of la_gdn_fwd_host_params: gdn_fwd's parameters with host data pointers, the
    device staging buffer and the number of token ranges."""
    _fields_ = [("fwd", GdnFwdParams), ("staging", _vp), ("staging_bytes", ctypes.c_size_t), ("ranges", _i32)]


class GdnSummaryParams(ctypes.Structure):
    """Mirror of la_gdn_summary_params (same field order and types)."""
    _fields_ = [
        ("k", _vp), ("k_stride_t", _i64), ("k_stride_h", _i64),
        ("v", _vp), ("v_stride_t", _i64), ("v_stride_h", _i64),
        ("g", _vp), ("g_stride_t", _i64), ("g_stride_h", _i64),
        ("beta", _vp), ("beta_stride_t", _i64), ("beta_stride_h", _i64),
        ("cu_seqlens", _vp), ("cu_seqlens_bits", _i32),
        ("T", _i64),
        ("N", _i32), ("HK", _i32), ("HV", _i32), ("K", _i32), ("V", _i32),
        ("use_qk_l2norm", _i32),
        ("start_state", _vp), ("start_state_dtype", _i32),
        ("end_state", _vp),
        ("transition", _vp),
        ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t),
        ("status", _vp),
        ("gate_mode", _i32), ("a_log", _vp), ("dt_bias", _vp), ("gate_lower_bound", ctypes.c_float),
        ("beta_sigmoid", _i32), ("beta_bf16", _i32),
    ]


class GdnComposeParams(ctypes.Structure):
    """Mirror of la_gdn_compose_params (same field order and types)."""
    _fields_ = [
        ("R", _i32), ("HO", _i32), ("K", _i32), ("V", _i32),
        ("transitions", _vp), ("terms", _vp), ("start", _vp), ("out", _vp),
        ("backward", _i32),
    ]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load liblinattn.so (building it in-tree first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if build_if_missing and not _build.up_to_date():
            _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"liblinattn.so not found at {path}; run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        lib.gdn_fwd.restype = ctypes.c_int
        lib.gdn_fwd.argtypes = [ctypes.POINTER(GdnFwdParams), _vp]
        lib.gdn_bwd.restype = ctypes.c_int
        lib.gdn_bwd.argtypes = [ctypes.POINTER(GdnBwdParams), _vp]
        lib.gdn_summary_bwd.restype = ctypes.c_int
        lib.gdn_summary_bwd.argtypes = [ctypes.POINTER(GdnSummaryBwdParams), _vp]
        lib.la_gdn_summary_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.la_gdn_summary_bwd_workspace_bytes.argtypes = [_i32, _i32, _i32, _i32]
        lib.la_gdp_workspace_bytes.restype = ctypes.c_size_t
        lib.la_gdp_workspace_bytes.argtypes = [_i64, _i32, _i32, _i32, _i32, _i32, _i32]
        lib.la_gdn_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.la_gdn_bwd_workspace_bytes.argtypes = [_i64, _i32, _i32, _i32, _i32, _i32, _i32]
        lib.la_gdn_bwd_workspace_bytes_ckpt.restype = ctypes.c_size_t
        lib.la_gdn_bwd_workspace_bytes_ckpt.argtypes = [_i64, _i32, _i32, _i32, _i32, _i32, _i64, _i32]
        lib.la_gdn_bwd_workspace_bytes_min.restype = ctypes.c_size_t
        lib.la_gdn_bwd_workspace_bytes_min.argtypes = [_i64, _i32, _i32, _i32, _i32, _i32, _i64, _i32]
        lib.gdn_decode.restype = ctypes.c_int
        lib.gdn_decode.argtypes = [ctypes.POINTER(GdnDecodeParams), _vp]
        lib.gdn_summary.restype = ctypes.c_int
        lib.gdn_summary.argtypes = [ctypes.POINTER(GdnSummaryParams), _vp]
        lib.la_gdn_workspace_bytes.restype = ctypes.c_size_t
        lib.la_gdn_workspace_bytes.argtypes = [_i32, _i32]
        lib.la_gdn_fwd_split_workspace_bytes.restype = ctypes.c_size_t
        lib.la_gdn_fwd_split_workspace_bytes.argtypes = [_i64, _i32, _i32]
        lib.la_checkpoint_rows.restype = ctypes.c_int
        lib.la_checkpoint_rows.argtypes = [_vp, _i32, _i32, _i64, ctypes.POINTER(_i64)]
        lib.la_read_status.restype = ctypes.c_int
        lib.la_read_status.argtypes = [_vp, _vp, ctypes.POINTER(_i32)]
        lib.la_status_string.restype = ctypes.c_char_p
        lib.la_status_string.argtypes = [ctypes.c_int]
        lib.la_version.restype = _i32
        lib.la_version.argtypes = []
        lib.la_set_kernel_timing_events.restype = ctypes.c_int
        lib.la_set_kernel_timing_events.argtypes = [_vp, _vp]
        lib.la_test_set_wait_hooks.restype = ctypes.c_int
        lib.la_test_set_wait_hooks.argtypes = [_i32, ctypes.c_uint64]
        lib.la_test_set_fwd_pieces.restype = ctypes.c_int
        lib.la_test_set_fwd_pieces.argtypes = [_i32]
        lib.la_test_set_fwd_passes.restype = ctypes.c_int
        lib.la_test_set_fwd_passes.argtypes = [_i32]
        lib.gdn_compose_spans.restype = ctypes.c_int
        lib.gdn_compose_spans.argtypes = [ctypes.POINTER(GdnComposeParams), _vp]
        lib.gdn_fwd_host.restype = ctypes.c_int
        lib.gdn_fwd_host.argtypes = [ctypes.POINTER(GdnFwdHostParams), _vp]
        lib.la_gdn_fwd_host_staging_bytes.restype = ctypes.c_size_t
        lib.la_gdn_fwd_host_staging_bytes.argtypes = [ctypes.POINTER(GdnFwdHostParams)]
        lib.la_gdn_fwd_host_plan.restype = _i32
        lib.la_gdn_fwd_host_plan.argtypes = [_vp, _i32, _i32, _i32, _i64, ctypes.POINTER(_i64), _i32,
                                             ctypes.POINTER(_i64)]
        lib.gdn_fwd_static_workspace.restype = ctypes.c_int
        lib.gdn_fwd_static_workspace.argtypes = [ctypes.POINTER(GdnFwdParams), _vp]
        _lib = lib
        return lib


class GdnDecodeParams(ctypes.Structure):
    """Mirror of la_gdn_decode_params (same field order and types)."""
    _fields_ = [
        ("q", _vp), ("q_stride_n", _i64), ("q_stride_h", _i64),
        ("k", _vp), ("k_stride_n", _i64), ("k_stride_h", _i64),
        ("v", _vp), ("v_stride_n", _i64), ("v_stride_h", _i64),
        ("g", _vp), ("g_stride_n", _i64), ("g_stride_h", _i64),
        ("beta", _vp), ("beta_stride_n", _i64), ("beta_stride_h", _i64),
        ("N", _i32), ("HK", _i32), ("HV", _i32), ("K", _i32), ("V", _i32),
        ("scale", ctypes.c_float), ("use_qk_l2norm", _i32),
        ("state_pool", _vp), ("state_dtype", _i32), ("state_pool_size", _i64),
        ("state_indices", _vp),
        ("o", _vp), ("o_stride_n", _i64), ("o_stride_h", _i64),
        ("status", _vp),
        ("gate_mode", _i32), ("a_log", _vp), ("dt_bias", _vp), ("gate_lower_bound", ctypes.c_float),
        ("beta_sigmoid", _i32), ("beta_bf16", _i32),
    ]


class GdnBwdParams(ctypes.Structure):
    """Mirror of la_gdn_bwd_params (same field order and types)."""
    _fields_ = [
        ("q", _vp), ("q_stride_t", _i64), ("q_stride_h", _i64),
        ("k", _vp), ("k_stride_t", _i64), ("k_stride_h", _i64),
        ("v", _vp), ("v_stride_t", _i64), ("v_stride_h", _i64),
        ("g", _vp), ("g_stride_t", _i64), ("g_stride_h", _i64),
        ("beta", _vp), ("beta_stride_t", _i64), ("beta_stride_h", _i64),
        ("cu_seqlens", _vp), ("cu_seqlens_bits", _i32),
        ("T", _i64),
        ("N", _i32), ("HK", _i32), ("HV", _i32), ("K", _i32), ("V", _i32),
        ("scale", ctypes.c_float), ("use_qk_l2norm", _i32),
        ("initial_state", _vp), ("initial_state_dtype", _i32),
        ("checkpoints", _vp),
        ("d_o", _vp), ("d_o_stride_t", _i64), ("d_o_stride_h", _i64),
        ("d_final_state", _vp),
        ("dq", _vp), ("dq_stride_t", _i64), ("dq_stride_h", _i64),
        ("dk", _vp), ("dk_stride_t", _i64), ("dk_stride_h", _i64),
        ("dv", _vp), ("dv_stride_t", _i64), ("dv_stride_h", _i64),
        ("dg", _vp), ("dg_stride_t", _i64), ("dg_stride_h", _i64),
        ("dbeta", _vp), ("dbeta_stride_t", _i64), ("dbeta_stride_h", _i64),
        ("d_initial_state", _vp),
        ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t),
        ("status", _vp),
        ("gate_mode", _i32), ("a_log", _vp), ("dt_bias", _vp), ("gate_lower_bound", ctypes.c_float),
        ("beta_sigmoid", _i32), ("beta_bf16", _i32),
        ("d_a_log", _vp), ("d_dt_bias", _vp),
        ("checkpoint_every_n", _i64), ("checkpoint_bf16", _i32),
    ]


class GdnSummaryBwdParams(ctypes.Structure):
    """Mirror of la_gdn_summary_bwd_params (same field order and types)."""
    _fields_ = [
        ("q", _vp), ("q_stride_t", _i64), ("q_stride_h", _i64),
        ("k", _vp), ("k_stride_t", _i64), ("k_stride_h", _i64),
        ("g", _vp), ("g_stride_t", _i64), ("g_stride_h", _i64),
        ("beta", _vp), ("beta_stride_t", _i64), ("beta_stride_h", _i64),
        ("cu_seqlens", _vp), ("cu_seqlens_bits", _i32),
        ("T", _i64),
        ("N", _i32), ("HK", _i32), ("HV", _i32), ("K", _i32), ("V", _i32),
        ("scale", ctypes.c_float), ("use_qk_l2norm", _i32),
        ("d_o", _vp), ("d_o_stride_t", _i64), ("d_o_stride_h", _i64),
        ("d_final_state", _vp),
        ("d_state", _vp),
        ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t),
        ("status", _vp),
        ("gate_mode", _i32), ("a_log", _vp), ("dt_bias", _vp), ("gate_lower_bound", ctypes.c_float),
        ("beta_sigmoid", _i32), ("beta_bf16", _i32),
    ]


class LinAttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = load().la_status_string(code).decode()
        super().__init__(f"{where}: {msg} (la_status {code})")
        self.code = code


def check(code: int, where: str) -> None:
    if code != LA_OK:
        raise LinAttnError(code, where)
