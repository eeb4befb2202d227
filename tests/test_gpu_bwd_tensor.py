"""The tensor-core schedule of gdn_bwd (K = V = 128): the forward's WY pass, the state-gradient
pass storing the gradient leaving every chunk, and the chunk-parallel gradient pass.

Each case runs the default schedule (the tensor-core one when the workspace has room, as the
API's default workspace does) and, where it says so, the tile kernel (the passes hook set to 1),
both against the fp64 oracle with the tolerances of tests/test_gpu_bwd.py (max|x - ref| /
max|ref|: bf16 gradients 1e-2, fp32 gradients 2e-3)."""
import numpy as np
import pytest
import torch

import oracle
import gated_delta_rule_29_gb300 as la
from gated_delta_rule_29_gb300 import workloads as W

from test_gpu_bwd import compare, cotangents, dev

pytestmark = pytest.mark.gpu

NAMES = ["dq", "dk", "dv", "dg", "dbeta", "d_initial_state"]


def bwd(w, do, dfin, passes=0, **kw):
    """gdn_bwd through the API; passes 1 forces the tile kernel."""
    d = dev()
    lib = la.binding.load()
    status = torch.zeros(1, dtype=torch.int32, device=d)
    assert lib.la_test_set_fwd_passes(passes) == 0
    try:
        out = la.gdn_bwd(w.q.to(d), w.k.to(d), w.v.to(d), kw.pop("g", w.g).to(d), kw.pop("beta", w.beta).to(d),
                         w.cu_seqlens.to(d), do.to(d),
                         initial_state=None if w.initial_state is None else w.initial_state.to(d),
                         d_final_state=None if dfin is None else dfin.to(d), status=status, **kw)
        assert la.read_status(status) == 0
    finally:
        assert lib.la_test_set_fwd_passes(0) == 0
    return out


def host(out):
    return [None if x is None else x.float().cpu().numpy() for x in out]


def test_bwd_tensor_and_tile_schedules_against_oracle():
    """Ragged sequences (one token, a chunk +- 1, an empty one, several chunks: partial last
    chunks take the per-thread stores, full ones the TMA stores), grouped value heads (per-head
    dq, dk summed afterwards), a start state and a final-state cotangent: both schedules within
    tolerance, and they are distinct code paths (their rounding differs)."""
    w = W.draw("bwd tc ragged", [1, 63, 0, 64, 65, 200, 130], 2, 4, 128, 128, seed=601, initial_state=True,
               slow_decay=True)
    do, dfin = cotangents(w, 602)
    ref = oracle.gdn_bwd(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, do, initial_state=w.initial_state,
                         d_final_state=dfin)
    tc = host(bwd(w, do, dfin))
    tile = host(bwd(w, do, dfin, passes=1))
    compare(w, tc, ref, label=" tensor cores")
    compare(w, tile, ref, label=" tile kernel")
    assert any(not np.array_equal(a, b) for a, b in zip(tc, tile))


def test_bwd_tensor_page_distributions_one_key_head():
    """The pages' fast decay, one key head shared by four value heads, no start state and no
    final-state cotangent."""
    w = W.draw("bwd tc page", [300, 129, 1000], 1, 4, 128, 128, seed=611)
    do, _ = cotangents(w, 612, with_final=False)
    ref = oracle.gdn_bwd(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, do)
    compare(w, host(bwd(w, do, None)), ref, label=" tensor cores, one key head")


def test_bwd_tensor_batch_invariant_every_sequence():
    """Every sequence's gradients (dq, dk, dv, dg, dbeta and the start state's) are bitwise the
    same alone and inside the batch, on the tensor-core schedule."""
    w = W.draw("bwd tc batch", [90, 200, 33, 128, 64, 1], 1, 2, 128, 128, seed=621, initial_state=True,
               slow_decay=True)
    do, dfin = cotangents(w, 622)
    full = host(bwd(w, do, dfin))
    cu = w.cu_seqlens.numpy().astype(np.int64)
    for i in range(w.N):
        sl = slice(cu[i], cu[i + 1])
        sub = W.Workload(name="one", cu_seqlens=torch.tensor([0, cu[i + 1] - cu[i]]), q=w.q[sl], k=w.k[sl],
                         v=w.v[sl], g=w.g[sl].contiguous(), beta=w.beta[sl].contiguous(),
                         initial_state=w.initial_state[i:i + 1])
        alone = host(bwd(sub, do[sl], dfin[i:i + 1]))
        for name, x, y in zip(NAMES[:5], full[:5], alone[:5]):
            assert np.array_equal(x[sl], y), (i, name)
        assert np.array_equal(full[5][i], alone[5][0]), i


def test_bwd_tensor_bounded_gate_bf16_beta_logits():
    """The bounded sigmoid gate and bf16 beta logits through the sigmoid: the chain rules of the
    chunk-parallel pass."""
    w = W.draw("bwd tc bounded", [70, 129, 64], 1, 2, 128, 128, seed=631, initial_state=True)
    gen = torch.Generator().manual_seed(632)
    g_raw = torch.randn(w.T, w.HV, generator=gen)
    b_logit = torch.randn(w.T, w.HV, generator=gen).to(torch.bfloat16)
    do, dfin = cotangents(w, 633)
    got = host(bwd(w, do, dfin, g=g_raw, beta=b_logit, gate_lower_bound=-0.1, beta_sigmoid=True))
    ref = oracle.gdn_bwd(w.q, w.k, w.v, g_raw, b_logit.float(), w.cu_seqlens, do, initial_state=w.initial_state,
                         d_final_state=dfin, gate="sigmoid_bound", gate_lower_bound=-0.1, beta_sigmoid=True)
    compare(w, got, ref, label=" tensor cores, bounded gate + bf16 beta logits")


def test_bwd_tensor_softplus_gate_parameter_sums():
    """The softplus gate: d_a_log and d_dt_bias from the per-(chunk, head) sums, added per head in
    chunk order, against the oracle."""
    w = W.draw("bwd tc softplus", [1, 100, 64, 250], 2, 4, 128, 128, seed=641, initial_state=True)
    gen = torch.Generator().manual_seed(642)
    g_raw = torch.randn(w.T, w.HV, generator=gen)
    a_log = torch.log(0.02 + 0.08 * torch.rand(w.HV, generator=gen))  # rates that carry state across chunks
    dt_bias = 0.5 * torch.randn(w.HV, generator=gen)
    do, dfin = cotangents(w, 643)
    d = dev()
    out = host(bwd(w, do, dfin, g=g_raw, a_log=a_log.to(d), dt_bias=dt_bias.to(d)))
    ref = oracle.gdn_bwd(w.q, w.k, w.v, g_raw, w.beta, w.cu_seqlens, do, initial_state=w.initial_state,
                         d_final_state=dfin, gate="softplus", a_log=a_log, dt_bias=dt_bias)
    compare(w, out[:6], ref, label=" tensor cores, softplus gate")
    for name, x in zip(["d_a_log", "d_dt_bias"], out[6:]):
        r = np.asarray(ref[name], dtype=np.float64)
        e = float(np.abs(x - r).max() / np.abs(r).max())
        print(f"[parity] bwd tensor cores {name}: {e:.2e}")
        assert e <= 2e-3, (name, e)


def test_bwd_tensor_without_l2norm():
    """The norm off (keys and queries scaled to unit-order norms by hand), scale 0.5."""
    w = W.draw("bwd tc no-norm", [150, 70, 64], 1, 2, 128, 128, seed=651, initial_state=True, slow_decay=True)
    w.q = (w.q.float() / 11.0).to(torch.bfloat16)
    w.k = (w.k.float() / 11.0).to(torch.bfloat16)
    do, dfin = cotangents(w, 652)
    got = host(bwd(w, do, dfin, use_qk_l2norm=False, scale=0.5))
    ref = oracle.gdn_bwd(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, do, scale=0.5, use_qk_l2norm=False,
                         initial_state=w.initial_state, d_final_state=dfin)
    compare(w, got, ref, label=" tensor cores, no norm")


def test_bwd_tensor_unaligned_outputs_take_thread_stores_same_bits():
    """dq, dk, dv as views whose head stride is not a multiple of 8 elements: no TMA stores, the
    same arithmetic, so bitwise the results of the aligned outputs."""
    w = W.draw("bwd tc views", [128, 64, 77], 2, 2, 128, 128, seed=661, initial_state=True, slow_decay=True)
    do, dfin = cotangents(w, 662)
    d = dev()
    base = host(bwd(w, do, dfin))
    dq = torch.empty(w.T, w.HK, w.K + 1, dtype=torch.bfloat16, device=d)[..., :w.K]
    dk = torch.empty(w.T, w.HK, w.K + 1, dtype=torch.bfloat16, device=d)[..., :w.K]
    dv = torch.empty(w.T, w.HV, w.V + 1, dtype=torch.bfloat16, device=d)[..., :w.V]
    got = host(bwd(w, do, dfin, out=(dq, dk, dv)))
    for name, x, y in zip(NAMES, base, got):
        assert np.array_equal(x, y), name


def test_bwd_tensor_small_workspace_takes_the_tile_kernel():
    """A workspace of la_gdn_bwd_workspace_bytes_min runs the tile kernel: bitwise the forced
    tile schedule."""
    w = W.draw("bwd tc small ws", [200, 64], 2, 2, 128, 128, seed=671, initial_state=True, slow_decay=True)
    do, dfin = cotangents(w, 672)
    lib = la.binding.load()
    least = lib.la_gdn_bwd_workspace_bytes_min(w.T, w.N, w.HK, w.HV, w.K, w.V, 0, 0)
    assert least < lib.la_gdn_bwd_workspace_bytes_ckpt(w.T, w.N, w.HK, w.HV, w.K, w.V, 0, 0)
    ws = torch.empty(least, dtype=torch.uint8, device=dev())
    small = host(bwd(w, do, dfin, workspace=ws))
    tile = host(bwd(w, do, dfin, passes=1))
    for name, x, y in zip(NAMES, small, tile):
        assert np.array_equal(x, y), name


def test_bwd_tensor_state_gradient_ranges_same_bits():
    """More (sequence, head) units than SMs: the state-gradient pass walks every unit in four
    chunk ranges over co-resident CTAs, each range starting from the exact fp32 gradient its
    successor left; the gradient entering every sequence is bitwise the summary backward's (one
    walk per unit), and the chunk pass's gradients match the oracle on sampled units."""
    sms = torch.cuda.get_device_properties(dev()).multi_processor_count
    n_seq = sms // 2 + 8
    lengths = [200 + 7 * (i % 5) for i in range(n_seq)]
    w = W.draw("bwd tc ranges", lengths, 1, 2, 128, 128, seed=681, initial_state=True, slow_decay=True)
    assert w.N * w.HV > sms
    do, dfin = cotangents(w, 682)
    d = dev()
    got = bwd(w, do, dfin)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    ds = la.gdn_summary_bwd(w.q.to(d), w.k.to(d), w.g.to(d), w.beta.to(d), w.cu_seqlens.to(d), do.to(d),
                            d_final_state=dfin.to(d), status=status)
    assert la.read_status(status) == 0
    assert torch.equal(got[5], ds)
    # two sequences against the oracle (all of their heads)
    cu = w.cu_seqlens.numpy().astype(np.int64)
    for i in (0, n_seq - 1):
        sl = slice(cu[i], cu[i + 1])
        sub = W.Workload(name="one", cu_seqlens=torch.tensor([0, cu[i + 1] - cu[i]]), q=w.q[sl], k=w.k[sl],
                         v=w.v[sl], g=w.g[sl].contiguous(), beta=w.beta[sl].contiguous(),
                         initial_state=w.initial_state[i:i + 1])
        ref = oracle.gdn_bwd(sub.q, sub.k, sub.v, sub.g, sub.beta, sub.cu_seqlens, do[sl],
                             initial_state=sub.initial_state, d_final_state=dfin[i:i + 1])
        part = [got[0][sl].float().cpu().numpy(), got[1][sl].float().cpu().numpy(), got[2][sl].float().cpu().numpy(),
                got[3][sl].float().cpu().numpy(), got[4][sl].float().cpu().numpy(), got[5][i:i + 1].float().cpu().numpy()]
        compare(sub, part, ref, label=f" tensor cores, ranged state gradient, sequence {i}")


def test_bwd_tensor_bounded_wait_timeout_reports_and_context_survives():
    """The chunk-parallel pass's failure path, made on the host: the library's test hook stops its
    tile loads, so every CTA's first tile wait runs out after a 20 ms budget; the call reports
    LA_ERR_TIMEOUT and returns, and the next call on the same context matches the oracle."""
    w = W.draw("bwd tc timeout", [130, 64], 1, 2, 128, 128, seed=691, initial_state=True, slow_decay=True)
    do, dfin = cotangents(w, 692)
    d = dev()
    lib = la.binding.load()
    status = torch.zeros(1, dtype=torch.int32, device=d)
    assert lib.la_test_set_wait_hooks(1, 20000000) == 0
    try:
        la.gdn_bwd(w.q.to(d), w.k.to(d), w.v.to(d), w.g.to(d), w.beta.to(d), w.cu_seqlens.to(d), do.to(d),
                   initial_state=w.initial_state.to(d), d_final_state=dfin.to(d), status=status)
        assert la.read_status(status) == la.binding.LA_ERR_TIMEOUT
    finally:
        assert lib.la_test_set_wait_hooks(0, 0) == 0
    torch.cuda.synchronize()
    got = host(bwd(w, do, dfin))
    ref = oracle.gdn_bwd(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, do, initial_state=w.initial_state,
                         d_final_state=dfin)
    compare(w, got, ref, label=" tensor cores, after a timed-out call")
