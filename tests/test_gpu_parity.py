"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Tolerances (max|x - ref| / max|ref| over each output tensor):
  o (bf16)                         1e-2
  fp32 states, checkpoints, transitions   2e-3
  bf16 checkpoints / bf16-start states     1e-2   (bf16 storage alone is 2^-9 relative)
Full-size workloads are compared on sampled (sequence, head) units, in the same
launch configuration as the benchmark (one call over the whole batch).
"""
import numpy as np
import pytest
import torch

import oracle
import gated_delta_rule_29_gb300 as la
from gated_delta_rule_29_gb300 import context_parallel as cp
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


def to_dev(w, d):
    return dict(q=w.q.to(d), k=w.k.to(d), v=w.v.to(d), g=w.g.to(d), beta=w.beta.to(d),
                cu=w.cu_seqlens.to(d),
                s0=None if w.initial_state is None else w.initial_state.to(d))


def gpu_fwd(w, d=None, **kw):
    d = d or dev()
    t = to_dev(w, d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    args = dict(use_qk_l2norm=w.use_qk_l2norm, initial_state=t["s0"],
                output_final_state=w.output_final_state, checkpoint_every_n=w.checkpoint_every_n,
                checkpoint_dtype=w.checkpoint_dtype, status=status)
    args.update(kw)
    o, fin, ck = la.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu"], **args)
    assert la.read_status(status) == 0
    f = lambda x: None if x is None else x.float().cpu().numpy()
    return f(o), f(fin), f(ck)


def oracle_fwd(w, units=None):
    mask = None
    if units is not None:
        mask = np.zeros((w.N, w.HV), dtype=bool)
        for i, h in units:
            mask[i, h] = True
    return oracle.gdn_fwd(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, use_qk_l2norm=w.use_qk_l2norm,
                          initial_state=w.initial_state, checkpoint_every_n=w.checkpoint_every_n,
                          unit_mask=mask)


def compare_units(w, got, ref, units, ck_tol=S_TOL):
    o, fin, ck = got
    cu = w.cu_seqlens.numpy().astype(np.int64)
    go = np.concatenate([o[cu[i]:cu[i + 1], h] for i, h in units])
    ro = np.concatenate([ref["o"][cu[i]:cu[i + 1], h] for i, h in units])
    errs = {"o": rel(go, ro)}
    if fin is not None:
        errs["final"] = rel(np.stack([fin[i, h] for i, h in units]),
                            np.stack([ref["final_state"][i, h] for i, h in units]))
    if ck is not None:
        off, _ = oracle.checkpoint_offsets(cu, w.checkpoint_every_n)
        rows = [(off[i] + j, h) for i, h in units for j in range(-(-(cu[i + 1] - cu[i]) // w.checkpoint_every_n))]
        errs["ckpt"] = rel(np.stack([ck[r_, h] for r_, h in rows]), np.stack([ref["checkpoints"][r_, h] for r_, h in rows]))
    print(f"[parity] {w.name}: " + ", ".join(f"{k_} {v_:.2e}" for k_, v_ in errs.items()))
    assert errs["o"] <= O_TOL, errs
    assert errs.get("final", 0) <= S_TOL, errs
    assert errs.get("ckpt", 0) <= ck_tol, errs
    return errs


def all_units(w):
    return [(i, h) for i in range(w.N) for h in range(w.HV) if w.lengths()[i] > 0]


# ------------------------------------------------------------------ the five workloads
@pytest.mark.parametrize("slow", [False, True])
def test_tiny_workload(slow):
    w = W.config(1, slow_decay=slow)
    got = gpu_fwd(w)
    compare_units(w, got, oracle_fwd(w), all_units(w))


@pytest.mark.parametrize("slow", [False, True])
def test_varlen_workload(slow):
    w = W.config(2, slow_decay=slow)
    got = gpu_fwd(w)
    compare_units(w, got, oracle_fwd(w), all_units(w))


_C3 = {}


def c3(slow):
    if slow not in _C3:
        _C3[slow] = W.config(3, slow_decay=slow)
    return _C3[slow]


@pytest.mark.parametrize("slow", [False, True])
def test_dense_batch_full_size_sampled(slow):
    """T = 65536, H = 32, K = V = 128, fp32 start state, final state and fp32 checkpoints every
    1024 tokens: the benchmark's launch; the oracle recomputes sampled units."""
    w = c3(slow)
    got = gpu_fwd(w)
    units = [(0, 0), (3, 17), (7, 31), (5, 8)]
    compare_units(w, got, oracle_fwd(w, units), units)
    assert np.isfinite(got[0]).all() and np.isfinite(got[1]).all()


def _ck_offsets(lengths, n):
    rows = [-(-int(L) // n) for L in lengths]
    return np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)


def _fwd_dev(w, ckpt_n, d):
    """gdn_fwd on the device, results kept on the device (o bf16, final and checkpoints fp32)."""
    t = to_dev(w, d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    o, fin, ck = la.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu"], use_qk_l2norm=True,
                            initial_state=t["s0"], output_final_state=True, checkpoint_every_n=ckpt_n,
                            checkpoint_dtype=torch.float32, status=status)
    assert la.read_status(status) == 0
    return o, fin, ck


def test_skewed_gva_sampled_and_batch_invariant():
    """The skewed grouped-head batch: parity on sampled units, then bitwise batch invariance of
    EVERY sequence (page, "Semantics worth knowing": batch_invariant): each of the 64 sequences
    run alone and inside three shuffled copies of the whole batch gives the same bits in o, the
    final state and its fp32 checkpoints as in the original batch."""
    w = W.config(4)
    d = dev()
    lens = w.lengths()
    order = np.argsort(lens)
    picks = [int(order[0]), int(order[len(order) // 2]), int(order[-1])]
    units = [(i, h) for i in picks for h in (0, 1, 31)]
    n = 512
    full = _fwd_dev(w, n, d)
    host = (full[0].float().cpu().numpy(), full[1].cpu().numpy(), None)
    compare_units(w, host, oracle_fwd(w, units), units)
    del host
    cu = w.cu_seqlens.numpy().astype(np.int64)
    off = _ck_offsets(lens, n)

    def check_batch(seqs, tag):
        idx = np.concatenate([np.arange(cu[i], cu[i + 1]) for i in seqs])
        sub = W.Workload(name=tag, cu_seqlens=W._cu([lens[i] for i in seqs]), q=w.q[idx], k=w.k[idx],
                         v=w.v[idx], g=w.g[idx].contiguous(), beta=w.beta[idx].contiguous())
        o2, f2, c2 = _fwd_dev(sub, n, d)
        cu2 = sub.cu_seqlens.numpy().astype(np.int64)
        off2 = _ck_offsets([lens[i] for i in seqs], n)
        for j, i in enumerate(seqs):
            assert torch.equal(o2[cu2[j]:cu2[j + 1]], full[0][cu[i]:cu[i + 1]]), (tag, i, "o")
            assert torch.equal(f2[j], full[1][i]), (tag, i, "final")
            assert torch.equal(c2[off2[j]:off2[j + 1]], full[2][off[i]:off[i + 1]]), (tag, i, "ckpt")

    for i in range(w.N):
        check_batch([i], f"alone {i}")
    rng = np.random.default_rng(7)
    for trial in range(3):
        check_batch([int(x) for x in rng.permutation(w.N)], f"shuffle {trial}")


@pytest.mark.parametrize("slow", [False, True])
def test_summary_span_composition(slow):
    """One 131072-token sequence cut into 8 spans: composing the span summaries with the
    library's kernel (S <- transition^T S + S_H, gdn_compose_spans) reproduces the unsplit
    forward's final state."""
    w = W.config(5, slow_decay=slow)
    d = dev()
    t = to_dev(w, d)
    spans = w.spans.to(d)
    # a nonzero state entering the sequence, S_init ~ 0.1 N(0, 1), so that the first span's
    # transition is applied to a state (page, "Summaries": S_final = S_init * transition + S_H)
    gen = torch.Generator().manual_seed(5005)
    S_init = 0.1 * torch.randn((1, w.HV, w.K, w.V), generator=gen, dtype=torch.float32)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    end, tr = la.gdn_summary(t["k"], t["v"], t["g"], t["beta"], spans, use_qk_l2norm=True, status=status)
    assert la.read_status(status) == 0
    _, fin, _ = la.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu"], use_qk_l2norm=True,
                           initial_state=S_init.to(d))
    S = cp.compose(list(tr), list(end), S_init[0].to(d))[-1].double().cpu().numpy()
    end = end.double().cpu().numpy()
    tr = tr.double().cpu().numpy()
    fin = fin.double().cpu().numpy()[0]
    errs = {"composed_vs_unsplit": rel(S, fin)}
    assert errs["composed_vs_unsplit"] <= S_TOL
    # the oracle on two sampled heads: span end states, transitions, the composed state and the
    # unsplit run from the same start
    heads = [0, 11]
    mask = np.zeros((8, w.HV), dtype=bool)
    mask[:, heads] = True
    ref = oracle.gdn_summary(w.k, w.v, w.g, w.beta, w.spans, unit_mask=mask)
    errs["end_state"] = rel(end[:, heads], ref["end_state"][:, heads])
    if slow:
        errs["transition"] = rel(tr[:, heads], ref["transition"][:, heads])
    refS = oracle.compose_spans(ref["transition"], ref["end_state"], S_init.double().numpy()[0])[-1]
    errs["composed_vs_oracle"] = rel(S[heads], refS[heads])
    umask = np.zeros((1, w.HV), dtype=bool)
    umask[0, heads] = True
    unsplit = oracle.gdn_fwd(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, initial_state=S_init, want_o=False,
                             unit_mask=umask)["final_state"][0]
    errs["oracle_composed_vs_oracle_unsplit"] = rel(refS[heads], unsplit[heads])
    errs["unsplit_vs_oracle"] = rel(fin[heads], unsplit[heads])
    print(f"[parity] summary slow={slow}: " + ", ".join(f"{k_} {v_:.2e}" for k_, v_ in errs.items()))
    assert max(errs.values()) <= S_TOL, errs


# ------------------------------------------------------------------ edge cases
def small(lengths, HK=2, HV=2, K=64, V=64, seed=5, **kw):
    return W.draw("edge", lengths, HK, HV, K, V, seed=seed, **kw)


@pytest.mark.parametrize("K,V", [(64, 128), (128, 64), (128, 128), (64, 64)])
def test_head_dims(K, V):
    w = small([1, 63, 64, 65, 200], K=K, V=V, seed=K + V, initial_state=True, checkpoint_every_n=64,
              checkpoint_dtype=torch.float32, slow_decay=True)
    compare_units(w, gpu_fwd(w), oracle_fwd(w), all_units(w))


def test_empty_and_ragged_sequences():
    w = small([0, 1, 64, 0, 129, 0], initial_state=True, checkpoint_every_n=64,
              checkpoint_dtype=torch.float32, slow_decay=True)
    got = gpu_fwd(w)
    compare_units(w, got, oracle_fwd(w), all_units(w))
    s0 = w.initial_state.numpy()
    for i in (0, 3, 5):
        assert np.array_equal(got[1][i], s0[i])  # empty sequence: final = initial state


def test_bf16_checkpoints_and_bf16_initial_state():
    w = small([300, 128, 70], initial_state=True, checkpoint_every_n=128, slow_decay=True)
    w.initial_state = w.initial_state.to(torch.bfloat16).float()  # the oracle sees the rounded start
    d = dev()
    got = gpu_fwd(w, initial_state=w.initial_state.to(d).to(torch.bfloat16), checkpoint_dtype=torch.bfloat16)
    compare_units(w, got, oracle_fwd(w), all_units(w), ck_tol=BF16_STATE_TOL)


def test_grouped_heads_hk1():
    w = small([130, 77], HK=1, HV=4, seed=9, slow_decay=True)
    compare_units(w, gpu_fwd(w), oracle_fwd(w), all_units(w))


def test_no_l2norm():
    w = small([150, 90], seed=11)
    w.q = (w.q.float() * 0.05).to(torch.bfloat16)
    w.k = (w.k.float() * 0.05).to(torch.bfloat16)
    w.use_qk_l2norm = False
    compare_units(w, gpu_fwd(w), oracle_fwd(w), all_units(w))


def test_strided_fused_projection_views():
    """q, k, v as column slices of one fused [T, 2*HK*K + HV*V] projection (no copies)."""
    w = small([100, 156], HK=2, HV=4, K=64, V=64, seed=13, slow_decay=True)
    d = dev()
    T = w.T
    fused = torch.cat([w.q.reshape(T, -1), w.k.reshape(T, -1), w.v.reshape(T, -1)], dim=1).to(d)
    a, b = w.HK * w.K, 2 * w.HK * w.K
    q = fused[:, :a].view(T, w.HK, w.K)
    k = fused[:, a:b].view(T, w.HK, w.K)
    v = fused[:, b:].view(T, w.HV, w.V)
    assert not q.is_contiguous()
    o, fin, _ = la.gdn_fwd(q, k, v, w.g.to(d), w.beta.to(d), w.cu_seqlens.to(d))
    compare_units(w, (o.float().cpu().numpy(), fin.cpu().numpy(), None), oracle_fwd(w), all_units(w))


def test_int64_cu_seqlens_and_explicit_scale():
    w = small([77, 200], seed=17, slow_decay=True)
    d = dev()
    t = to_dev(w, d)
    o, fin, _ = la.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu"].long(), scale=0.3)
    ref = oracle.gdn_fwd(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, scale=0.3)
    assert rel(o.float().cpu().numpy(), ref["o"]) <= O_TOL
    assert rel(fin.cpu().numpy(), ref["final_state"]) <= S_TOL


def test_bad_cu_seqlens_sets_status():
    w = small([100, 156], seed=19)
    d = dev()
    t = to_dev(w, d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    for bad in ([0, 300, 256], [1, 100, 256], [0, 100, 255]):
        cu = torch.tensor(bad, dtype=torch.int32, device=d)
        la.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], cu, status=status)
        assert la.read_status(status) == la.binding.LA_ERR_BAD_SEQLENS
    la.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu"], status=status)
    assert la.read_status(status) == 0


def test_bounded_wait_timeout_reports_and_context_survives():
    """The failure path of the bounded waits, made on the host: the library's test hook stops
    the K/Q tile loads, so every CTA's first wait runs out after a 20 ms budget.  The kernel
    must report LA_ERR_TIMEOUT and return; the next normal call on the same context must
    succeed and match the oracle."""
    w = small([100, 156, 64], seed=37)
    d = dev()
    t = to_dev(w, d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    lib = la.binding.load()
    assert lib.la_test_set_wait_hooks(1, 20000000) == 0
    try:
        la.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu"], status=status)
        assert la.read_status(status) == la.binding.LA_ERR_TIMEOUT
    finally:
        assert lib.la_test_set_wait_hooks(0, 0) == 0
    torch.cuda.synchronize()
    status.zero_()
    o, fin, _ = la.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu"], status=status)
    assert la.read_status(status) == 0
    ref = oracle.gdn_fwd(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens)
    assert rel(o.float().cpu().numpy(), ref["o"]) <= O_TOL
    assert rel(fin.cpu().numpy(), ref["final_state"]) <= S_TOL


def test_many_sequences_global_sort_path():
    """More than 8192 sequences: the prologue sorts in global memory."""
    rng = np.random.default_rng(23)
    lengths = [int(x) for x in rng.integers(0, 4, size=9000)] + [150]
    w = small(lengths, HK=1, HV=1, K=64, V=64, seed=23)
    got = gpu_fwd(w)
    ref = oracle_fwd(w)
    compare_units(w, got, ref, all_units(w))


def test_summary_start_state_and_empty_spans():
    w = small([0, 150, 0, 64], HK=1, HV=2, K=64, V=64, seed=29, initial_state=True, slow_decay=True)
    d = dev()
    t = to_dev(w, d)
    end, tr = la.gdn_summary(t["k"], t["v"], t["g"], t["beta"], t["cu"], start_state=t["s0"])
    ref = oracle.gdn_summary(w.k, w.v, w.g, w.beta, w.cu_seqlens, start_state=w.initial_state)
    assert rel(end.cpu().numpy(), ref["end_state"]) <= S_TOL
    assert rel(tr.cpu().numpy(), ref["transition"]) <= S_TOL
    eye = np.eye(64)
    for i in (0, 2):
        assert np.array_equal(tr[i].cpu().numpy(), np.stack([eye, eye]).astype(np.float32))


@pytest.mark.parametrize("groups", [1, 3, 8])
def test_host_pipeline_matches_device_call(groups):
    """gdn_fwd_host (host buffers, pipelined over token ranges: 3 and 8 ranges cut the longer
    sequences into pieces that hand their fp32 state on) gives the same bits as gdn_fwd."""
    w = small([300, 1, 0, 200, 129, 64], HK=2, HV=4, K=128, V=128, seed=37, initial_state=True,
              checkpoint_every_n=64, checkpoint_dtype=torch.float32, slow_decay=True)
    o_d, f_d, c_d = gpu_fwd(w)
    pin = lambda x: x.contiguous().pin_memory()
    o_h, f_h, c_h = la.gdn_fwd_host(pin(w.q), pin(w.k), pin(w.v), pin(w.g), pin(w.beta), w.cu_seqlens,
                                    initial_state=pin(w.initial_state), checkpoint_every_n=64,
                                    checkpoint_dtype=torch.float32, groups=groups)
    torch.cuda.synchronize()
    assert np.array_equal(o_h.float().numpy(), o_d)
    assert np.array_equal(f_h.numpy(), f_d)
    assert np.array_equal(c_h.numpy(), c_d)


# ------------------------------------------------------------------ in-kernel input transforms
def _raw_gate_inputs(w, seed, beta_dtype=torch.float32):
    """Raw gate and beta logits of a workload's shape (the layer's projections, N(0,1))."""
    gen = torch.Generator().manual_seed(seed)
    T = int(w.cu_seqlens[-1])
    g_raw = torch.randn(T, w.HV, generator=gen)
    beta_raw = torch.randn(T, w.HV, generator=gen).to(beta_dtype)
    return g_raw, beta_raw


@pytest.mark.parametrize("rate,beta_dtype", [(1.0, torch.float32), (0.01, torch.bfloat16)])
def test_softplus_gate_and_beta_sigmoid(rate, beta_dtype):
    """g = -exp(a_log) softplus(g_raw + dt_bias) and beta = sigmoid(beta_raw) computed in the
    kernel, against the oracle applying the same transforms in fp64.  rate scales exp(a_log):
    1.0 gives the layer's usual fast decay, 0.01 a slow one that keeps the start state alive."""
    w = small([1, 63, 64, 65, 200], HK=2, HV=4, K=128, V=128, seed=41, initial_state=True,
              checkpoint_every_n=64, checkpoint_dtype=torch.float32)
    g_raw, beta_raw = _raw_gate_inputs(w, 43, beta_dtype)
    a_log = torch.log(rate * torch.tensor([1.0, 2.0, 4.0, 8.0]))
    dt_bias = torch.tensor([-4.0, -2.0, 0.0, 1.0])
    d = dev()
    t = to_dev(w, d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    o, fin, ck = la.gdn_fwd(t["q"], t["k"], t["v"], g_raw.to(d), beta_raw.to(d), t["cu"],
                            initial_state=t["s0"], checkpoint_every_n=64, checkpoint_dtype=torch.float32,
                            a_log=a_log.to(d), dt_bias=dt_bias.to(d), beta_sigmoid=True, status=status)
    assert la.read_status(status) == 0
    ref = oracle.gdn_fwd(w.q, w.k, w.v, g_raw, beta_raw.float(), w.cu_seqlens, initial_state=w.initial_state,
                         checkpoint_every_n=64, gate="softplus", a_log=a_log, dt_bias=dt_bias, beta_sigmoid=True)
    got = (o.float().cpu().numpy(), fin.cpu().numpy(), ck.cpu().numpy())
    compare_units(w, got, ref, all_units(w))


def test_bounded_gate_summary_and_forward():
    """g = lower_bound * sigmoid(g_raw) with lower_bound = -0.05 (slow decay, so the start state
    and the transitions stay large) and fp32 beta logits: summary and forward against the oracle."""
    w = small([0, 150, 64, 300], HK=1, HV=2, K=64, V=128, seed=47, initial_state=True)
    g_raw, beta_raw = _raw_gate_inputs(w, 53)
    d = dev()
    t = to_dev(w, d)
    kw = dict(gate_lower_bound=-0.05, beta_sigmoid=True)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    end, tr = la.gdn_summary(t["k"], t["v"], g_raw.to(d), beta_raw.to(d), t["cu"], start_state=t["s0"],
                             status=status, **kw)
    assert la.read_status(status) == 0
    o, fin, _ = la.gdn_fwd(t["q"], t["k"], t["v"], g_raw.to(d), beta_raw.to(d), t["cu"], initial_state=t["s0"],
                           status=status, **kw)
    assert la.read_status(status) == 0
    okw = dict(gate="sigmoid_bound", gate_lower_bound=-0.05, beta_sigmoid=True)
    ref_s = oracle.gdn_summary(w.k, w.v, g_raw, beta_raw, w.cu_seqlens, start_state=w.initial_state, **okw)
    ref_f = oracle.gdn_fwd(w.q, w.k, w.v, g_raw, beta_raw, w.cu_seqlens, initial_state=w.initial_state, **okw)
    errs = {"end": rel(end.cpu().numpy(), ref_s["end_state"]), "transition": rel(tr.cpu().numpy(), ref_s["transition"]),
            "o": rel(o.float().cpu().numpy(), ref_f["o"]), "final": rel(fin.cpu().numpy(), ref_f["final_state"])}
    print("[parity] bounded gate: " + ", ".join(f"{k_} {v_:.2e}" for k_, v_ in errs.items()))
    assert errs["o"] <= O_TOL and max(errs["end"], errs["transition"], errs["final"]) <= S_TOL, errs


def test_transform_arguments_rejected():
    w = small([64], seed=59)
    d = dev()
    t = to_dev(w, d)
    with pytest.raises(la.binding.LinAttnError):
        la.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu"], gate_lower_bound=0.5)
    with pytest.raises(ValueError):
        la.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu"], a_log=torch.zeros(2, device=d))


def test_host_pipeline_transforms_and_options_bitwise():
    """gdn_fwd_host with the softplus gate (host a_log, dt_bias), bf16 beta logits, a bf16 start
    state, bf16 checkpoints every 128 tokens, no final state, int64 cu_seqlens and 7 ranges: the
    same bits as gdn_fwd on device buffers."""
    w = small([700, 64, 1, 0, 389, 129], HK=1, HV=4, K=128, V=64, seed=43, initial_state=True)
    g_raw, beta_raw = _raw_gate_inputs(w, 44, torch.bfloat16)
    a_log = torch.log(torch.tensor([0.02, 0.05, 0.1, 0.5]))
    dt_bias = torch.tensor([-3.0, -1.0, 0.0, 0.5])
    s0 = w.initial_state.to(torch.bfloat16)
    d = dev()
    t = to_dev(w, d)
    kw = dict(checkpoint_every_n=128, checkpoint_dtype=torch.bfloat16, output_final_state=False, beta_sigmoid=True)
    o_d, _, c_d = la.gdn_fwd(t["q"], t["k"], t["v"], g_raw.to(d), beta_raw.to(d), t["cu"], initial_state=s0.to(d),
                             a_log=a_log.to(d), dt_bias=dt_bias.to(d), **kw)
    pin = lambda x: x.contiguous().pin_memory()
    o_h, f_h, c_h = la.gdn_fwd_host(pin(w.q), pin(w.k), pin(w.v), pin(g_raw), pin(beta_raw),
                                    w.cu_seqlens.to(torch.int64), initial_state=pin(s0), a_log=a_log, dt_bias=dt_bias,
                                    groups=7, **kw)
    torch.cuda.synchronize()
    assert f_h is None
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(c_h, c_d.cpu())


@pytest.mark.parametrize("nstaging", [1, 2])
def test_host_pipeline_back_to_back_calls(nstaging):
    """Four gdn_fwd_host calls enqueued without a host synchronisation, on two different input
    sets and into four output sets, with one staging buffer or two used in turn (a call is then
    ordered only after the last call on its buffer): every output equals its device call."""
    lengths = [300, 1, 129, 450]
    ws = [small(lengths, HK=2, HV=2, K=128, V=128, seed=51 + i, initial_state=True, checkpoint_every_n=64,
                checkpoint_dtype=torch.float32, slow_decay=True) for i in range(2)]
    pin = lambda x: x.contiguous().pin_memory()
    host = [[pin(x) for x in (w.q, w.k, w.v, w.g, w.beta, w.initial_state)] for w in ws]
    refs = [gpu_fwd(w) for w in ws]
    stagings = [{} for _ in range(nstaging)]
    outs = []
    for call in range(4):
        q, k, v, g, b, s0 = host[call % 2]
        outs.append(la.gdn_fwd_host(q, k, v, g, b, ws[0].cu_seqlens, initial_state=s0, checkpoint_every_n=64,
                                    checkpoint_dtype=torch.float32, groups=5, staging=stagings[call % nstaging]))
    torch.cuda.synchronize()
    for call, (o_h, f_h, c_h) in enumerate(outs):
        o_d, f_d, c_d = refs[call % 2]
        assert np.array_equal(o_h.float().numpy(), o_d), call
        assert np.array_equal(f_h.numpy(), f_d) and np.array_equal(c_h.numpy(), c_d), call


def test_host_pipeline_pageable_buffers_and_two_threads():
    """gdn_fwd_host on pageable (not pinned) host tensors, outputs included, and two host
    threads calling it at once with their own staging buffers: the same bits as gdn_fwd."""
    import threading
    ws = [small([260, 64, 3], HK=1, HV=2, K=64, V=128, seed=61 + i, initial_state=True, checkpoint_every_n=64,
                checkpoint_dtype=torch.float32, slow_decay=True) for i in range(2)]
    refs = [gpu_fwd(w) for w in ws]

    def run(w, out):
        o = torch.empty(w.T, w.HV, w.V, dtype=torch.bfloat16)
        f = torch.empty(w.N, w.HV, w.K, w.V)
        c = torch.empty(la.checkpoint_rows(w.cu_seqlens, 64), w.HV, w.K, w.V)
        s = torch.cuda.Stream()
        la.gdn_fwd_host(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, initial_state=w.initial_state, checkpoint_every_n=64,
                        checkpoint_dtype=torch.float32, out=(o, f, c), groups=3, staging={}, stream=s)
        s.synchronize()
        out.extend([o, f, c])

    outs = [[], []]
    threads = [threading.Thread(target=run, args=(w, out)) for w, out in zip(ws, outs)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    for (o, f, c), (o_d, f_d, c_d) in zip(outs, refs):
        assert np.array_equal(o.float().numpy(), o_d) and np.array_equal(f.numpy(), f_d)
        assert np.array_equal(c.numpy(), c_d)


@pytest.mark.parametrize("K,V", [(128, 128), (64, 64)])
def test_extreme_but_valid_values(K, V):
    """Gates from 0 down to -30 (decays spanning far more than fp32's range within a chunk: the
    kernel's factorised decays must fall back to direct ones), beta exactly 0 or 1, all-zero q
    and k rows under the L2 norm (the norm's epsilon keeps them zero), and a start state."""
    w = small([300, 77, 64], HK=2, HV=2, K=K, V=V, seed=71 + K, initial_state=True, checkpoint_every_n=64,
              checkpoint_dtype=torch.float32)
    gen = torch.Generator().manual_seed(72)
    T = w.T
    u = torch.rand(T, w.HV, generator=gen)
    g = torch.where(u < 0.1, torch.full_like(u, -30.0), torch.where(u < 0.5, torch.zeros_like(u), -0.01 * u))
    r = torch.rand(T, w.HV, generator=gen)
    beta = torch.where(r < 0.2, torch.zeros_like(r), torch.where(r < 0.4, torch.ones_like(r), r))
    q, k = w.q.clone(), w.k.clone()
    zq = torch.rand(T, generator=gen) < 0.05
    zk = torch.rand(T, generator=gen) < 0.05
    q[zq] = 0
    k[zk] = 0
    w.q, w.k, w.g, w.beta = q, k, g.contiguous(), beta.contiguous()
    got = gpu_fwd(w)
    compare_units(w, got, oracle_fwd(w), all_units(w))


@pytest.mark.parametrize("cut", [128, 200])
def test_state_round_trip_split_run(cut):
    """Running tokens [0, m) and then [m, L) from the first part's fp32 final state equals the
    unsplit run: bitwise when m is a chunk boundary (the second run continues the same chunk
    sequence from the exact state), within tolerance of the oracle otherwise (the chunk grid
    restarts at m)."""
    L = 450
    w = small([L], HK=2, HV=4, K=128, V=128, seed=41, initial_state=True, slow_decay=True)
    d = dev()
    t = to_dev(w, d)
    o, fin, _ = la.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu"], initial_state=t["s0"])
    parts = []
    s_in = t["s0"]
    for a, b in ((0, cut), (cut, L)):
        cu = torch.tensor([0, b - a], dtype=torch.int32, device=d)
        oo, ff, _ = la.gdn_fwd(t["q"][a:b], t["k"][a:b], t["v"][a:b], t["g"][a:b], t["beta"][a:b], cu,
                               initial_state=s_in)
        parts.append(oo)
        s_in = ff
    o2 = torch.cat(parts)
    if cut % 64 == 0:
        assert torch.equal(o2, o) and torch.equal(s_in, fin)
    ref = oracle_fwd(w)
    e_o, e_f = rel(o2.float().cpu().numpy(), ref["o"]), rel(s_in.cpu().numpy(), ref["final_state"])
    print(f"[parity] split run at {cut}: o {e_o:.2e}, final {e_f:.2e}")
    assert e_o <= O_TOL and e_f <= S_TOL
