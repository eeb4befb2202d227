"""State pool (state_indices) and the one-token decode kernel vs the fp64 oracle, through the
C ABI.  Tolerances as in test_gpu_parity: o 1e-2, fp32 states 2e-3, bf16 states 1e-2
(max|x - ref| / max|ref| per tensor); slots no sequence names must come back bitwise
unchanged."""
import numpy as np
import pytest
import torch

import oracle
import gated_delta_rule_29_gb300 as la
from gated_delta_rule_29_gb300 import workloads as W

pytestmark = pytest.mark.gpu

O_TOL = 1e-2
S_TOL = 2e-3
BF16_STATE_TOL = 1e-2


def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def rel(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.abs(ref).max()
    assert den > 0, "reference is all zero: the comparison would be vacuous"
    return float(np.abs(got - ref).max() / den)


def decode_case(N, HK, HV, K, V, P, seed, pool_dtype=torch.float32, indices=True):
    """One token per sequence (the decode workload's shape), a pool of P slots holding
    0.1 N(0,1) states, and a random injective slot assignment."""
    w = W.draw("decode", [1] * N, HK, HV, K, V, seed=seed)
    gen = torch.Generator().manual_seed(seed + 1)
    pool = (0.1 * torch.randn(P, HV, K, V, generator=gen)).to(pool_dtype)
    idx = torch.randperm(P, generator=gen)[:N].to(torch.int32) if indices else None
    return w, pool, idx


def run_decode(w, pool, idx, **kw):
    d = dev()
    pool_d = pool.to(d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    o = la.gdn_decode(w.q.to(d), w.k.to(d), w.v.to(d), w.g.to(d), w.beta.to(d), pool_d,
                      state_indices=None if idx is None else idx.to(d), status=status, **kw)
    assert la.read_status(status) == 0
    return o.float().cpu().numpy(), pool_d.float().cpu().numpy()


def check_pool(w, pool, idx, o, pool_out, ref, tol):
    N = w.N
    slots = np.arange(N) if idx is None else idx.numpy().astype(np.int64)
    errs = {"o": rel(o, ref["o"]), "pool": rel(pool_out[slots], ref["state_pool"][slots])}
    others = np.setdiff1d(np.arange(pool.shape[0]), slots)
    if len(others):
        assert np.array_equal(pool_out[others], pool.float().numpy()[others]), "untouched slots changed"
    print(f"[parity] {w.name}: " + ", ".join(f"{k_} {v_:.2e}" for k_, v_ in errs.items()))
    assert errs["o"] <= O_TOL and errs["pool"] <= tol, errs


def test_decode_serving_batch():
    """512 sequences, 16 q/k heads shared by 32 value heads, K = V = 128, fp32 pool of 1024 slots."""
    w, pool, idx = decode_case(512, 16, 32, 128, 128, 1024, seed=301)
    o, pool_out = run_decode(w, pool, idx)
    ref = oracle.gdn_fwd(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, initial_state=pool, state_indices=idx)
    check_pool(w, pool, idx, o, pool_out, ref, S_TOL)


@pytest.mark.parametrize("K,V", [(64, 64), (64, 128), (128, 64), (128, 128)])
def test_decode_head_dims_bf16_pool_transforms(K, V):
    """bf16 pool, no index array (slot i), softplus gate and beta logits in the kernel."""
    w, pool, _ = decode_case(37, 2, 4, K, V, 40, seed=311 + K + V, pool_dtype=torch.bfloat16, indices=False)
    gen = torch.Generator().manual_seed(7)
    g_raw = torch.randn(w.N, 4, generator=gen)
    beta_raw = torch.randn(w.N, 4, generator=gen)
    a_log = torch.log(torch.tensor([0.5, 1.0, 2.0, 4.0]))
    dt_bias = torch.tensor([-1.0, 0.0, 0.5, 1.0])
    d = dev()
    pool_d = pool.to(d)
    o = la.gdn_decode(w.q.to(d), w.k.to(d), w.v.to(d), g_raw.to(d), beta_raw.to(d), pool_d, a_log=a_log.to(d),
                      dt_bias=dt_bias.to(d), beta_sigmoid=True)
    ref = oracle.gdn_fwd(w.q, w.k, w.v, g_raw, beta_raw, w.cu_seqlens, initial_state=pool.float(),
                         state_indices=np.arange(w.N), gate="softplus", a_log=a_log, dt_bias=dt_bias,
                         beta_sigmoid=True)
    check_pool(w, pool, None, o.float().cpu().numpy(), pool_d.float().cpu().numpy(), ref, BF16_STATE_TOL)


def test_decode_steps_match_prefill():
    """Eight decode steps, each feeding the pool forward, equal one 8-token forward per sequence."""
    N, HK, HV, K, V, L = 24, 2, 4, 128, 128, 8
    w = W.draw("steps", [L] * N, HK, HV, K, V, seed=331)
    gen = torch.Generator().manual_seed(332)
    pool = 0.1 * torch.randn(2 * N, HV, K, V, generator=gen)
    idx = torch.randperm(2 * N, generator=gen)[:N].to(torch.int32)
    d = dev()
    pool_d, idx_d = pool.to(d), idx.to(d)
    q, k, v, g, b = (x.to(d).view(N, L, *x.shape[1:]) for x in (w.q, w.k, w.v, w.g, w.beta))
    outs = []
    for t in range(L):
        outs.append(la.gdn_decode(q[:, t], k[:, t], v[:, t], g[:, t], b[:, t], pool_d, state_indices=idx_d))
    o = torch.stack(outs, 1).reshape(N * L, HV, V).float().cpu().numpy()
    ref = oracle.gdn_fwd(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, initial_state=pool, state_indices=idx)
    check_pool(w, pool, idx, o, pool_d.cpu().numpy(), ref, S_TOL)


@pytest.mark.parametrize("pool_dtype", [torch.float32, torch.bfloat16])
def test_fwd_with_state_pool(pool_dtype):
    """gdn_fwd over ragged sequences starting from, and writing back into, a state pool."""
    lengths = [1, 63, 0, 200, 64, 129]
    w = W.draw("pool prefill", lengths, 2, 4, 128, 128, seed=341, slow_decay=True)
    gen = torch.Generator().manual_seed(342)
    pool = (0.1 * torch.randn(9, 4, 128, 128, generator=gen)).to(pool_dtype)
    idx = torch.tensor([8, 0, 3, 5, 1, 6], dtype=torch.int32)
    d = dev()
    pool_d = pool.to(d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    o, fin, ck = la.gdn_fwd(w.q.to(d), w.k.to(d), w.v.to(d), w.g.to(d), w.beta.to(d), w.cu_seqlens.to(d),
                            initial_state=pool_d, state_indices=idx.to(d), status=status)
    assert la.read_status(status) == 0 and fin is None and ck is None
    ref = oracle.gdn_fwd(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, initial_state=pool.float(), state_indices=idx)
    tol = S_TOL if pool_dtype == torch.float32 else BF16_STATE_TOL
    check_pool(w, pool, idx, o.float().cpu().numpy(), pool_d.float().cpu().numpy(), ref, tol)


def test_bad_state_index_sets_status():
    w, pool, idx = decode_case(8, 1, 2, 64, 64, 8, seed=351)
    d = dev()
    bad = idx.clone()
    bad[3] = 8  # one past the pool
    status = torch.zeros(1, dtype=torch.int32, device=d)
    la.gdn_decode(w.q.to(d), w.k.to(d), w.v.to(d), w.g.to(d), w.beta.to(d), pool.to(d), state_indices=bad.to(d),
                  status=status)
    assert la.read_status(status) == la.binding.LA_ERR_BAD_STATE_INDEX
    status.zero_()
    la.gdn_fwd(w.q.to(d), w.k.to(d), w.v.to(d), w.g.to(d), w.beta.to(d), w.cu_seqlens.to(d),
               initial_state=pool.to(d), state_indices=bad.to(d), status=status)
    assert la.read_status(status) == la.binding.LA_ERR_BAD_STATE_INDEX
    status.zero_()
    run = la.gdn_decode(w.q.to(d), w.k.to(d), w.v.to(d), w.g.to(d), w.beta.to(d), pool.to(d),
                        state_indices=idx.to(d), status=status)
    assert la.read_status(status) == 0 and torch.isfinite(run.float()).all()


def test_decode_fused_projection_views_and_strided_output():
    """q, k, v as column slices of one fused [N, 2 HK K + HV V] projection, g and beta as slices
    of one [N, 2 HV] buffer, o written into a column slice of a wider buffer: the same bits as
    with contiguous tensors, and within tolerance of the oracle."""
    N, HK, HV, K, V, P = 48, 2, 4, 128, 64, 64
    w, pool, idx = decode_case(N, HK, HV, K, V, P, seed=351)
    d = dev()
    a, b = HK * K, 2 * HK * K
    fused = torch.cat([w.q.reshape(N, -1), w.k.reshape(N, -1), w.v.reshape(N, -1)], dim=1).to(d)
    q, k, v = fused[:, :a].view(N, HK, K), fused[:, a:b].view(N, HK, K), fused[:, b:].view(N, HV, V)
    gb = torch.cat([w.g, w.beta], dim=1).to(d)
    g, beta = gb[:, :HV], gb[:, HV:]
    assert not q.is_contiguous() and not g.is_contiguous()
    wide = torch.full((N, HV, V + 32), 7.0, dtype=torch.bfloat16, device=d)
    o = wide[:, :, :V]
    pool_s = pool.to(d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    la.gdn_decode(q, k, v, g, beta, pool_s, state_indices=idx.to(d), o=o, status=status)
    assert la.read_status(status) == 0
    assert bool((wide[:, :, V:] == 7.0).all()), "a write outside the output view"
    o_c, pool_c = run_decode(w, pool, idx)
    assert np.array_equal(o.float().cpu().numpy(), o_c)
    assert np.array_equal(pool_s.float().cpu().numpy(), pool_c)
    ref = oracle.gdn_fwd(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, initial_state=pool, state_indices=idx)
    check_pool(w, pool, idx, o_c, pool_c, ref, S_TOL)
