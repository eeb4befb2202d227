"""The C ABI on the host: exports, struct layout, and argument errors (no GPU needed).

Every case here returns from the library before any CUDA call, so it runs on a
machine without a GPU.  Device pointers are fake, suitably aligned integers:
validation rejects the call before anything could dereference them.
"""
import ctypes
import os
import re
import subprocess

import pytest

from gated_delta_rule_29_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "liblinattn.h")


def _declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:la_status|size_t|const char\*|int32_t)\s+(\w+)\s*\(", text, re.M)))


def test_library_exports_every_declared_function():
    lib = B.load()
    declared = _declared_functions()
    assert set(declared) == set(B.EXPORTED_SYMBOLS), declared
    for name in declared:
        assert hasattr(lib, name), f"{name} not exported"


def _c_layout(struct_name, fields):
    src = ["#include <stdio.h>", "#include <stddef.h>", f'#include "{HEADER}"', "int main(void) {",
           f'  printf("%zu\\n", sizeof({struct_name}));']
    for f in fields:
        src.append(f'  printf("%zu\\n", offsetof({struct_name}, {f}));')
    src.append("  return 0; }")
    d = os.path.join(ROOT, "tests", "_build")
    os.makedirs(d, exist_ok=True)
    c = os.path.join(d, f"layout_{struct_name}.c")
    exe = os.path.join(d, f"layout_{struct_name}")
    open(c, "w").write("\n".join(src))
    subprocess.run(["gcc", "-std=c11", "-o", exe, c], check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout.split()
    return int(out[0]), [int(x) for x in out[1:]]


@pytest.mark.parametrize("cls,cname", [(B.GdnFwdParams, "la_gdn_fwd_params"),
                                       (B.GdnSummaryParams, "la_gdn_summary_params"),
                                       (B.GdnDecodeParams, "la_gdn_decode_params"),
                                       (B.GdnBwdParams, "la_gdn_bwd_params"),
                                       (B.GdnSummaryBwdParams, "la_gdn_summary_bwd_params"),
                                       (B.GdnFwdHostParams, "la_gdn_fwd_host_params"),
                                       (B.GdnComposeParams, "la_gdn_compose_params")])
def test_ctypes_mirror_matches_c_layout(cls, cname):
    names = [f[0] for f in cls._fields_]
    size, offs = _c_layout(cname, names)
    assert ctypes.sizeof(cls) == size
    for name, off in zip(names, offs):
        assert getattr(cls, name).offset == off, name


FAKE = 0x10000  # 64 KiB: aligned for every check; never dereferenced


def _fwd(**over):
    p = B.GdnFwdParams()
    T, N, HK, HV, K, V = 256, 2, 2, 2, 64, 64
    p.q, p.q_stride_t, p.q_stride_h = FAKE, HK * K, K
    p.k, p.k_stride_t, p.k_stride_h = FAKE, HK * K, K
    p.v, p.v_stride_t, p.v_stride_h = FAKE, HV * V, V
    p.g, p.g_stride_t, p.g_stride_h = FAKE, HV, 1
    p.beta, p.beta_stride_t, p.beta_stride_h = FAKE, HV, 1
    p.cu_seqlens, p.cu_seqlens_bits = FAKE, 32
    p.T, p.N, p.HK, p.HV, p.K, p.V = T, N, HK, HV, K, V
    p.scale, p.use_qk_l2norm = 0.0, 1
    p.o, p.o_stride_t, p.o_stride_h = FAKE, HV * V, V
    for k, v in over.items():
        setattr(p, k, v)
    return p


def _summary(**over):
    p = B.GdnSummaryParams()
    T, N, HK, HV, K, V = 256, 2, 2, 2, 64, 64
    p.k, p.k_stride_t, p.k_stride_h = FAKE, HK * K, K
    p.v, p.v_stride_t, p.v_stride_h = FAKE, HV * V, V
    p.g, p.g_stride_t, p.g_stride_h = FAKE, HV, 1
    p.beta, p.beta_stride_t, p.beta_stride_h = FAKE, HV, 1
    p.cu_seqlens, p.cu_seqlens_bits = FAKE, 32
    p.T, p.N, p.HK, p.HV, p.K, p.V = T, N, HK, HV, K, V
    p.end_state, p.transition = FAKE, FAKE
    for k, v in over.items():
        setattr(p, k, v)
    return p


FWD_ERRORS = [
    ("K not 64/128", dict(K=96), B.LA_ERR_UNSUPPORTED),
    ("V not 64/128", dict(V=32), B.LA_ERR_UNSUPPORTED),
    ("HV not a multiple of HK", dict(HK=3, HV=4), B.LA_ERR_UNSUPPORTED),
    ("more q/k heads than value heads", dict(HK=4, HV=2), B.LA_ERR_UNSUPPORTED),
    ("negative T", dict(T=-1), B.LA_ERR_INVALID_ARG),
    ("negative N", dict(N=-1), B.LA_ERR_INVALID_ARG),
    ("zero heads", dict(HK=0), B.LA_ERR_INVALID_ARG),
    ("cu_seqlens bits", dict(cu_seqlens_bits=16), B.LA_ERR_INVALID_ARG),
    ("null cu_seqlens", dict(cu_seqlens=None), B.LA_ERR_INVALID_ARG),
    ("misaligned int64 cu_seqlens", dict(cu_seqlens=FAKE + 4, cu_seqlens_bits=64), B.LA_ERR_INVALID_ARG),
    ("null q", dict(q=None), B.LA_ERR_INVALID_ARG),
    ("null k", dict(k=None), B.LA_ERR_INVALID_ARG),
    ("null v", dict(v=None), B.LA_ERR_INVALID_ARG),
    ("null o", dict(o=None), B.LA_ERR_INVALID_ARG),
    ("null g", dict(g=None), B.LA_ERR_INVALID_ARG),
    ("null beta", dict(beta=None), B.LA_ERR_INVALID_ARG),
    ("q base not 16-byte aligned", dict(q=FAKE + 8), B.LA_ERR_INVALID_ARG),
    ("k token stride not a multiple of 8", dict(k_stride_t=132), B.LA_ERR_INVALID_ARG),
    ("v head stride not a multiple of 8", dict(v_stride_h=65), B.LA_ERR_INVALID_ARG),
    ("misaligned g", dict(g=FAKE + 2), B.LA_ERR_INVALID_ARG),
    ("checkpoints without n", dict(checkpoints=FAKE, checkpoint_every_n=0), B.LA_ERR_INVALID_ARG),
    ("checkpoint n not a multiple of 64", dict(checkpoints=FAKE, checkpoint_every_n=100), B.LA_ERR_INVALID_ARG),
    ("checkpoint dtype", dict(checkpoints=FAKE, checkpoint_every_n=64, checkpoint_dtype=7), B.LA_ERR_UNSUPPORTED),
    ("initial state dtype", dict(initial_state=FAKE, initial_state_dtype=3), B.LA_ERR_UNSUPPORTED),
    ("misaligned fp32 initial state", dict(initial_state=FAKE + 2, initial_state_dtype=1), B.LA_ERR_INVALID_ARG),
    ("misaligned final state", dict(final_state=FAKE + 1), B.LA_ERR_INVALID_ARG),
    ("T beyond int32 TMA coordinates", dict(T=1 << 31), B.LA_ERR_UNSUPPORTED),
    ("unknown gate mode", dict(gate_mode=5), B.LA_ERR_INVALID_ARG),
    ("softplus gate without a_log", dict(gate_mode=1, dt_bias=FAKE), B.LA_ERR_INVALID_ARG),
    ("bounded gate with a positive bound", dict(gate_mode=2, gate_lower_bound=1.0), B.LA_ERR_INVALID_ARG),
    ("state pool without a pool", dict(state_indices=FAKE, state_pool_size=4), B.LA_ERR_INVALID_ARG),
    ("state pool and final state", dict(state_indices=FAKE, state_pool_size=4, initial_state=FAKE,
                                        initial_state_dtype=1, final_state=FAKE), B.LA_ERR_INVALID_ARG),
    ("state pool and checkpoints", dict(state_indices=FAKE, state_pool_size=4, initial_state=FAKE,
                                        initial_state_dtype=1, checkpoints=FAKE, checkpoint_every_n=64),
     B.LA_ERR_INVALID_ARG),
    ("empty state pool", dict(state_indices=FAKE, state_pool_size=0, initial_state=FAKE, initial_state_dtype=1),
     B.LA_ERR_INVALID_ARG),
]


@pytest.mark.parametrize("name,over,code", FWD_ERRORS, ids=[e[0] for e in FWD_ERRORS])
def test_gdn_fwd_rejects(name, over, code):
    lib = B.load()
    p = _fwd(**over)
    assert lib.gdn_fwd(ctypes.byref(p), None) == code


SUM_ERRORS = [
    ("K not 64/128", dict(K=80), B.LA_ERR_UNSUPPORTED),
    ("null end state", dict(end_state=None), B.LA_ERR_INVALID_ARG),
    ("null transition", dict(transition=None), B.LA_ERR_INVALID_ARG),
    ("transition not 16-byte aligned", dict(transition=FAKE + 4), B.LA_ERR_INVALID_ARG),
    ("null k", dict(k=None), B.LA_ERR_INVALID_ARG),
    ("start state dtype", dict(start_state=FAKE, start_state_dtype=9), B.LA_ERR_UNSUPPORTED),
    ("HV not a multiple of HK", dict(HK=2, HV=3), B.LA_ERR_UNSUPPORTED),
]


@pytest.mark.parametrize("name,over,code", SUM_ERRORS, ids=[e[0] for e in SUM_ERRORS])
def test_gdn_summary_rejects(name, over, code):
    lib = B.load()
    p = _summary(**over)
    assert lib.gdn_summary(ctypes.byref(p), None) == code


def _decode(**over):
    p = B.GdnDecodeParams()
    N, HK, HV, K, V = 4, 2, 4, 128, 128
    p.q, p.q_stride_n, p.q_stride_h = FAKE, HK * K, K
    p.k, p.k_stride_n, p.k_stride_h = FAKE, HK * K, K
    p.v, p.v_stride_n, p.v_stride_h = FAKE, HV * V, V
    p.g, p.g_stride_n, p.g_stride_h = FAKE, HV, 1
    p.beta, p.beta_stride_n, p.beta_stride_h = FAKE, HV, 1
    p.N, p.HK, p.HV, p.K, p.V = N, HK, HV, K, V
    p.state_pool, p.state_dtype, p.state_pool_size = FAKE, B.LA_DTYPE_F32, 8
    p.o, p.o_stride_n, p.o_stride_h = FAKE, HV * V, V
    for k, v in over.items():
        setattr(p, k, v)
    return p


DECODE_ERRORS = [
    ("K not 64/128", dict(K=96), B.LA_ERR_UNSUPPORTED),
    ("HV not a multiple of HK", dict(HK=3), B.LA_ERR_UNSUPPORTED),
    ("pool dtype", dict(state_dtype=4), B.LA_ERR_UNSUPPORTED),
    ("null pool", dict(state_pool=None), B.LA_ERR_INVALID_ARG),
    ("pool not 16-byte aligned", dict(state_pool=FAKE + 8), B.LA_ERR_INVALID_ARG),
    ("pool smaller than N without indices", dict(state_pool_size=3), B.LA_ERR_INVALID_ARG),
    ("misaligned indices", dict(state_indices=FAKE + 2), B.LA_ERR_INVALID_ARG),
    ("null q", dict(q=None), B.LA_ERR_INVALID_ARG),
    ("null o", dict(o=None), B.LA_ERR_INVALID_ARG),
    ("negative N", dict(N=-1), B.LA_ERR_INVALID_ARG),
    ("unknown gate mode", dict(gate_mode=9), B.LA_ERR_INVALID_ARG),
]


@pytest.mark.parametrize("name,over,code", DECODE_ERRORS, ids=[e[0] for e in DECODE_ERRORS])
def test_gdn_decode_rejects(name, over, code):
    lib = B.load()
    p = _decode(**over)
    assert lib.gdn_decode(ctypes.byref(p), None) == code


def test_null_params():
    lib = B.load()
    assert lib.gdn_fwd(None, None) == B.LA_ERR_INVALID_ARG
    assert lib.gdn_summary(None, None) == B.LA_ERR_INVALID_ARG
    assert lib.gdn_decode(None, None) == B.LA_ERR_INVALID_ARG
    assert lib.gdn_bwd(None, None) == B.LA_ERR_INVALID_ARG
    assert lib.gdn_summary_bwd(None, None) == B.LA_ERR_INVALID_ARG


def _summary_bwd(**over):
    p = B.GdnSummaryBwdParams()
    T, N, HK, HV, K, V = 256, 2, 2, 4, 128, 128
    p.q, p.q_stride_t, p.q_stride_h = FAKE, HK * K, K
    p.k, p.k_stride_t, p.k_stride_h = FAKE, HK * K, K
    p.g, p.g_stride_t, p.g_stride_h = FAKE, HV, 1
    p.beta, p.beta_stride_t, p.beta_stride_h = FAKE, HV, 1
    p.cu_seqlens, p.cu_seqlens_bits = FAKE, 32
    p.T, p.N, p.HK, p.HV, p.K, p.V = T, N, HK, HV, K, V
    p.d_o, p.d_o_stride_t, p.d_o_stride_h = FAKE, HV * V, V
    p.d_state = FAKE
    for k, v in over.items():
        setattr(p, k, v)
    return p


SUM_BWD_ERRORS = [
    ("K not 64/128", dict(K=96), B.LA_ERR_UNSUPPORTED),
    ("HV not a multiple of HK", dict(HK=3), B.LA_ERR_UNSUPPORTED),
    ("null d_state", dict(d_state=None), B.LA_ERR_INVALID_ARG),
    ("misaligned d_state", dict(d_state=FAKE + 2), B.LA_ERR_INVALID_ARG),
    ("misaligned d_final_state", dict(d_final_state=FAKE + 2), B.LA_ERR_INVALID_ARG),
    ("null q", dict(q=None), B.LA_ERR_INVALID_ARG),
    ("q not 16-byte aligned", dict(q=FAKE + 8), B.LA_ERR_INVALID_ARG),
    ("null d_o", dict(d_o=None), B.LA_ERR_INVALID_ARG),
    ("negative N", dict(N=-1), B.LA_ERR_INVALID_ARG),
    ("small workspace", dict(workspace=FAKE, workspace_bytes=16), B.LA_ERR_WORKSPACE),
]


@pytest.mark.parametrize("name,over,code", SUM_BWD_ERRORS, ids=[e[0] for e in SUM_BWD_ERRORS])
def test_gdn_summary_bwd_rejects(name, over, code):
    lib = B.load()
    p = _summary_bwd(**over)
    assert lib.gdn_summary_bwd(ctypes.byref(p), None) == code


def _bwd(**over):
    p = B.GdnBwdParams()
    T, N, HK, HV, K, V = 256, 2, 2, 4, 128, 128
    p.q, p.q_stride_t, p.q_stride_h = FAKE, HK * K, K
    p.k, p.k_stride_t, p.k_stride_h = FAKE, HK * K, K
    p.v, p.v_stride_t, p.v_stride_h = FAKE, HV * V, V
    p.g, p.g_stride_t, p.g_stride_h = FAKE, HV, 1
    p.beta, p.beta_stride_t, p.beta_stride_h = FAKE, HV, 1
    p.cu_seqlens, p.cu_seqlens_bits = FAKE, 32
    p.T, p.N, p.HK, p.HV, p.K, p.V = T, N, HK, HV, K, V
    p.d_o, p.d_o_stride_t, p.d_o_stride_h = FAKE, HV * V, V
    p.dq, p.dq_stride_t, p.dq_stride_h = FAKE, HK * K, K
    p.dk, p.dk_stride_t, p.dk_stride_h = FAKE, HK * K, K
    p.dv, p.dv_stride_t, p.dv_stride_h = FAKE, HV * V, V
    p.dg, p.dg_stride_t, p.dg_stride_h = FAKE, HV, 1
    p.dbeta, p.dbeta_stride_t, p.dbeta_stride_h = FAKE, HV, 1
    p.workspace, p.workspace_bytes = FAKE, 16  # too small: reached only after every argument check
    for k, v in over.items():
        setattr(p, k, v)
    return p


BWD_ERRORS = [
    ("valid arguments reach the workspace check", dict(), B.LA_ERR_WORKSPACE),
    ("K not 64/128", dict(K=96), B.LA_ERR_UNSUPPORTED),
    ("null dg", dict(dg=None), B.LA_ERR_INVALID_ARG),
    ("softplus gate without a_log", dict(gate_mode=B.LA_GATE_SOFTPLUS, dt_bias=FAKE), B.LA_ERR_INVALID_ARG),
    ("bounded gate with a positive bound", dict(gate_mode=B.LA_GATE_SIGMOID_BOUND, gate_lower_bound=1.0),
     B.LA_ERR_INVALID_ARG),
    ("unknown gate mode", dict(gate_mode=7), B.LA_ERR_INVALID_ARG),
    ("misaligned d_a_log", dict(gate_mode=B.LA_GATE_SOFTPLUS, a_log=FAKE, dt_bias=FAKE, d_a_log=FAKE + 2),
     B.LA_ERR_INVALID_ARG),
    ("softplus gate with outputs reaches the workspace check",
     dict(gate_mode=B.LA_GATE_SOFTPLUS, a_log=FAKE, dt_bias=FAKE, d_a_log=FAKE, d_dt_bias=FAKE), B.LA_ERR_WORKSPACE),
    ("checkpoint cadence not a multiple of 64", dict(checkpoints=FAKE, checkpoint_every_n=100), B.LA_ERR_INVALID_ARG),
    ("negative checkpoint cadence", dict(checkpoints=FAKE, checkpoint_every_n=-64), B.LA_ERR_INVALID_ARG),
    ("misaligned fp32 checkpoints", dict(checkpoints=FAKE + 2), B.LA_ERR_INVALID_ARG),
    ("bf16 checkpoints every 1024 tokens reach the workspace check",
     dict(checkpoints=FAKE + 2, checkpoint_bf16=1, checkpoint_every_n=1024), B.LA_ERR_WORKSPACE),
]


@pytest.mark.parametrize("name,over,code", BWD_ERRORS, ids=[e[0] for e in BWD_ERRORS])
def test_gdn_bwd_rejects(name, over, code):
    lib = B.load()
    p = _bwd(**over)
    assert lib.gdn_bwd(ctypes.byref(p), None) == code


def test_bwd_workspace_bytes_by_checkpoint_kind():
    """Given fp32 rows every 64 tokens need the least; bf16 rows add the widened copy; sparse
    rows also the regenerating forward's output, segment boundaries and start states."""
    lib = B.load()
    args = (65536, 8, 32, 32, 128, 128)
    none = lib.la_gdn_bwd_workspace_bytes(*args, 0)
    direct = lib.la_gdn_bwd_workspace_bytes(*args, 1)
    assert lib.la_gdn_bwd_workspace_bytes_ckpt(*args, 0, 0) == none
    assert lib.la_gdn_bwd_workspace_bytes_ckpt(*args, 64, 0) == direct
    widen = lib.la_gdn_bwd_workspace_bytes_ckpt(*args, 64, 1)
    sparse = lib.la_gdn_bwd_workspace_bytes_ckpt(*args, 1024, 0)
    assert direct < widen < none < sparse
    rows = 65536 // 64 + 8
    assert widen - direct >= rows * 32 * 128 * 128 * 4
    assert lib.la_gdn_bwd_workspace_bytes_ckpt(*args, 100, 0) == 0


def test_bwd_workspace_min_is_the_tile_kernels():
    """K = V = 128: the default size adds the tensor-core schedule's areas (the WY records, T's
    residual and the gradient leaving every (chunk, head)) to the tile kernel's minimum; other
    head sizes have the tile kernel only, so the two sizes agree."""
    lib = B.load()
    for ck in ((0, 0), (64, 0), (64, 1), (1024, 0)):
        args = (65536, 8, 32, 32, 128, 128, *ck)
        full, least = lib.la_gdn_bwd_workspace_bytes_ckpt(*args), lib.la_gdn_bwd_workspace_bytes_min(*args)
        items = (65536 // 64 + 8) * 32
        assert least > 0 and full - least >= items * (17408 + 8192 + 65536)
        small = (65536, 8, 32, 32, 64, 64, *ck)
        assert lib.la_gdn_bwd_workspace_bytes_ckpt(*small) == lib.la_gdn_bwd_workspace_bytes_min(*small) > 0
    assert lib.la_gdn_bwd_workspace_bytes_min(65536, 8, 32, 32, 128, 128, 100, 0) == 0


def _compose(**over):
    p = B.GdnComposeParams()
    p.R, p.HO, p.K, p.V = 3, 2, 128, 64
    p.transitions, p.terms, p.start, p.out = FAKE, FAKE, FAKE, FAKE
    for k_, v_ in over.items():
        setattr(p, k_, v_)
    return p


@pytest.mark.parametrize("name,over,code", [
    ("no out", dict(out=None), B.LA_ERR_INVALID_ARG),
    ("negative spans", dict(R=-1), B.LA_ERR_INVALID_ARG),
    ("no heads", dict(HO=0), B.LA_ERR_INVALID_ARG),
    ("no transitions", dict(transitions=None), B.LA_ERR_INVALID_ARG),
    ("no terms", dict(terms=None), B.LA_ERR_INVALID_ARG),
    ("misaligned out", dict(out=FAKE + 2), B.LA_ERR_INVALID_ARG),
    ("misaligned start", dict(start=FAKE + 1), B.LA_ERR_INVALID_ARG),
    ("K = 96", dict(K=96), B.LA_ERR_UNSUPPORTED),
    ("V = 32", dict(V=32), B.LA_ERR_UNSUPPORTED),
])
def test_gdn_compose_rejects(name, over, code):
    assert B.load().gdn_compose_spans(ctypes.byref(_compose(**over)), None) == code, name


def test_fwd_pieces_hook_range():
    """The scheduling test hook takes 0 (automatic) .. 16 and rejects the rest; it only stores
    the setting (no device work), so it is callable without a GPU."""
    lib = B.load()
    for bad in (-1, 17):
        assert lib.la_test_set_fwd_pieces(bad) == B.LA_ERR_INVALID_ARG
    for ok in (16, 1, 0):
        assert lib.la_test_set_fwd_pieces(ok) == B.LA_OK


def test_summary_bwd_workspace_bytes():
    lib = B.load()
    a = lib.la_gdn_summary_bwd_workspace_bytes(8, 32, 128, 128)
    b = lib.la_gdn_summary_bwd_workspace_bytes(16, 32, 128, 128)
    assert b > a >= 8 * 32 * 128 * 128 * 4
    assert lib.la_gdn_summary_bwd_workspace_bytes(-1, 32, 128, 128) == 0


def test_checkpoint_rows_host_helper():
    lib = B.load()
    for bits, ctype in ((32, ctypes.c_int32), (64, ctypes.c_int64)):
        cu = (ctype * 5)(0, 100, 100, 1124, 1125)
        out = ctypes.c_int64(-1)
        assert lib.la_checkpoint_rows(ctypes.addressof(cu), bits, 4, 64, ctypes.byref(out)) == B.LA_OK
        assert out.value == 2 + 0 + 16 + 1
        bad = (ctype * 3)(0, 5, 3)
        assert lib.la_checkpoint_rows(ctypes.addressof(bad), bits, 2, 64, ctypes.byref(out)) == B.LA_ERR_INVALID_ARG
    assert lib.la_checkpoint_rows(ctypes.addressof(cu), 64, 4, 0, ctypes.byref(out)) == B.LA_ERR_INVALID_ARG


def test_status_strings_and_version():
    lib = B.load()
    for code in range(8):
        assert lib.la_status_string(code) != b"unknown status"
    assert lib.la_status_string(99) == b"unknown status"
    assert lib.la_version() >= 100
    assert lib.la_read_status(None, None, ctypes.byref(ctypes.c_int32())) == B.LA_ERR_INVALID_ARG


def test_workspace_bytes_grows_with_batch():
    lib = B.load()
    small = lib.la_gdn_workspace_bytes(4, 0)
    big = lib.la_gdn_workspace_bytes(100000, 0)
    assert small >= 256 and small % 256 == 0
    assert big > small and big % 256 == 0
    assert big >= 256 + 4 * 100000 + 8 * 100000 + 8 * 131072


def _host(cu, **over):
    """gdn_fwd_host parameters over a real host cu_seqlens (the call reads it on the host)."""
    hp = B.GdnFwdHostParams()
    p = _fwd()
    p.cu_seqlens, p.cu_seqlens_bits = ctypes.addressof(cu), 32
    p.T, p.N = cu[len(cu) - 1], len(cu) - 1
    for k, v in over.items():
        if k in ("staging", "staging_bytes", "ranges"):
            setattr(hp, k, v)
        else:
            setattr(p, k, v)
    hp.fwd = p
    if "staging" not in over:
        hp.staging = FAKE
    if "staging_bytes" not in over:
        hp.staging_bytes = 1 << 40
    if "ranges" not in over:
        hp.ranges = 4
    return hp


HOST_ERRORS = [
    ("decreasing cu_seqlens", [0, 200, 100, 256], {}, B.LA_ERR_BAD_SEQLENS),
    ("cu_seqlens not ending at T", [0, 100, 256], dict(T=300), B.LA_ERR_BAD_SEQLENS),
    ("cu_seqlens not starting at 0", [4, 100, 256], {}, B.LA_ERR_BAD_SEQLENS),
    ("zero ranges", [0, 100, 256], dict(ranges=0), B.LA_ERR_INVALID_ARG),
    ("Gated DeltaProduct", [0, 100, 256], dict(num_householder=2), B.LA_ERR_UNSUPPORTED),
    ("state pool", [0, 100, 256], dict(state_indices=FAKE, state_pool_size=4), B.LA_ERR_UNSUPPORTED),
    ("HV not a multiple of HK", [0, 100, 256], dict(HK=3, HV=4), B.LA_ERR_UNSUPPORTED),
    ("K not 64/128", [0, 100, 256], dict(K=96), B.LA_ERR_UNSUPPORTED),
    ("strided q", [0, 100, 256], dict(q_stride_t=256), B.LA_ERR_INVALID_ARG),
    ("strided g", [0, 100, 256], dict(g_stride_t=4), B.LA_ERR_INVALID_ARG),
    ("null o", [0, 100, 256], dict(o=None), B.LA_ERR_INVALID_ARG),
    ("checkpoint n not a multiple of 64", [0, 100, 256], dict(checkpoints=FAKE, checkpoint_every_n=100),
     B.LA_ERR_INVALID_ARG),
    ("softplus gate without dt_bias", [0, 100, 256], dict(gate_mode=1, a_log=FAKE), B.LA_ERR_INVALID_ARG),
    ("staging too small", [0, 100, 256], dict(staging_bytes=1024), B.LA_ERR_WORKSPACE),
    ("staging misaligned", [0, 100, 256], dict(staging=FAKE + 16), B.LA_ERR_WORKSPACE),
    ("no staging", [0, 100, 256], dict(staging=None), B.LA_ERR_WORKSPACE),
]


@pytest.mark.parametrize("name,cu,over,code", HOST_ERRORS, ids=[e[0] for e in HOST_ERRORS])
def test_gdn_fwd_host_rejects(name, cu, over, code):
    """Every rejection of the host-buffer entry happens on the host, before any CUDA call."""
    lib = B.load()
    cu_arr = (ctypes.c_int32 * len(cu))(*cu)
    hp = _host(cu_arr, **over)
    assert lib.gdn_fwd_host(ctypes.byref(hp), None) == code


def test_gdn_fwd_host_staging_bytes():
    """The staging size covers the device copies of every input and output: it grows with the
    checkpoints and the start state, and is 0 for invalid parameters."""
    lib = B.load()
    cu = (ctypes.c_int32 * 3)(0, 100, 256)
    base = lib.la_gdn_fwd_host_staging_bytes(ctypes.byref(_host(cu)))
    T, HK, HV, K, V = 256, 2, 2, 64, 64
    assert base >= T * (2 * HK * K + 2 * HV * V) * 2 + 2 * T * HV * 4
    ck = lib.la_gdn_fwd_host_staging_bytes(ctypes.byref(_host(cu, checkpoints=FAKE, checkpoint_every_n=64,
                                                                   checkpoint_dtype=1)))
    assert ck >= base + (2 + 3) * HV * K * V * 4
    s0 = lib.la_gdn_fwd_host_staging_bytes(ctypes.byref(_host(cu, initial_state=FAKE, initial_state_dtype=1)))
    assert s0 >= base + 2 * HV * K * V * 4
    assert lib.la_gdn_fwd_host_staging_bytes(ctypes.byref(_host(cu, K=96))) == 0
