"""Gated DeltaProduct (num_householder n > 1) through gdn_fwd vs the fp64 oracle's gdp_fwd.
Tolerances as in test_gpu_parity: o 1e-2, fp32 states and checkpoints 2e-3."""
import numpy as np
import pytest
import torch

import oracle
import gated_delta_rule_29_gb300 as la

pytestmark = pytest.mark.gpu

O_TOL = 1e-2
S_TOL = 2e-3


def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def rel(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.abs(ref).max()
    assert den > 0, "reference is all zero: the comparison would be vacuous"
    return float(np.abs(got - ref).max() / den)


def gdp_case(lengths, n, HK, HV, K, V, seed, slow=True):
    """The pages' distributions on both timelines: q, g per token; k, v, beta per update."""
    gen = torch.Generator().manual_seed(seed)
    T = sum(lengths)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    q = torch.randn(T, HK, K, generator=gen).to(torch.bfloat16)
    k = torch.randn(T * n, HK, K, generator=gen).to(torch.bfloat16)
    v = torch.randn(T * n, HV, V, generator=gen).to(torch.bfloat16)
    g = -torch.nn.functional.softplus(torch.randn(T, HV, generator=gen))
    beta = torch.sigmoid(torch.randn(T * n, HV, generator=gen))
    if slow:
        g, beta = g * 1e-3, beta * 0.2
    s0 = 0.1 * torch.randn(len(lengths), HV, K, V, generator=gen)
    return dict(q=q, k=k, v=v, g=g.contiguous(), beta=beta.contiguous(), cu=cu, s0=s0)


def test_gdp_two_updates_checkpoints_grouped_heads():
    n = 2
    c = gdp_case([1, 31, 32, 33, 100], n, 2, 4, 128, 128, seed=501)
    d = dev()
    status = torch.zeros(1, dtype=torch.int32, device=d)
    o, fin, ck = la.gdn_fwd(c["q"].to(d), c["k"].to(d), c["v"].to(d), c["g"].to(d), c["beta"].to(d), c["cu"].to(d),
                            initial_state=c["s0"].to(d), checkpoint_every_n=32, checkpoint_dtype=torch.float32,
                            num_householder=n, status=status)
    assert la.read_status(status) == 0
    ref = oracle.gdp_fwd(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu"], n, initial_state=c["s0"],
                         checkpoint_every_n=32)
    errs = {"o": rel(o.float().cpu(), ref["o"]), "final": rel(fin.cpu(), ref["final_state"]),
            "ckpt": rel(ck.cpu(), ref["checkpoints"])}
    print("[parity] gdp n=2: " + ", ".join(f"{k_} {v_:.2e}" for k_, v_ in errs.items()))
    assert errs["o"] <= O_TOL and errs["final"] <= S_TOL and errs["ckpt"] <= S_TOL, errs


@pytest.mark.parametrize("n,K,V", [(4, 128, 128), (8, 64, 128), (4, 64, 64), (3, 128, 128), (5, 64, 64),
                                   (7, 128, 64), (16, 128, 128), (33, 64, 128), (64, 64, 64), (65, 64, 64)])
def test_gdp_native_timeline_ragged(n, K, V):
    """The chunk kernel reads the queries and gates per token and writes the outputs per token
    (n = 4, 8, 16, 64: 64 / n tokens per chunk; n = 3, 5, 7, 33: chunks begin and end inside
    tokens; n = 65: the timeline build, one token longer than a chunk): ragged sequences that end
    inside a chunk, a one-token sequence, grouped heads, checkpoints, a start state."""
    c = gdp_case([1, 15, 16, 17, 70], n, 2, 4, K, V, seed=521 + n + K + V)
    d = dev()
    status = torch.zeros(1, dtype=torch.int32, device=d)
    ck_n = 64 // n if 64 % n == 0 else 64
    o, fin, ck = la.gdn_fwd(c["q"].to(d), c["k"].to(d), c["v"].to(d), c["g"].to(d), c["beta"].to(d), c["cu"].to(d),
                            initial_state=c["s0"].to(d), checkpoint_every_n=ck_n, checkpoint_dtype=torch.float32,
                            num_householder=n, status=status)
    assert la.read_status(status) == 0
    ref = oracle.gdp_fwd(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu"], n, initial_state=c["s0"],
                         checkpoint_every_n=ck_n)
    errs = {"o": rel(o.float().cpu(), ref["o"]), "final": rel(fin.cpu(), ref["final_state"]),
            "ckpt": rel(ck.cpu(), ref["checkpoints"])}
    print(f"[parity] gdp n={n} K={K} V={V}: " + ", ".join(f"{k_} {v_:.2e}" for k_, v_ in errs.items()))
    assert errs["o"] <= O_TOL and errs["final"] <= S_TOL and errs["ckpt"] <= S_TOL, errs


def test_gdp_native_bounded_gate_beta_logits_page_distributions():
    """n = 2 with the pages' fast decay, the bounded sigmoid gate and beta logits."""
    n = 2
    c = gdp_case([200, 64, 33], n, 1, 1, 128, 128, seed=531, slow=False)
    gen = torch.Generator().manual_seed(532)
    g_raw = torch.randn(c["q"].shape[0], 1, generator=gen)
    b_raw = torch.randn(c["k"].shape[0], 1, generator=gen)
    d = dev()
    status = torch.zeros(1, dtype=torch.int32, device=d)
    o, fin, _ = la.gdn_fwd(c["q"].to(d), c["k"].to(d), c["v"].to(d), g_raw.to(d), b_raw.to(d), c["cu"].to(d),
                           initial_state=c["s0"].to(d), num_householder=n, gate_lower_bound=-3.0,
                           beta_sigmoid=True, status=status)
    assert la.read_status(status) == 0
    g_log = oracle.gate_transform(g_raw, gate="sigmoid_bound", gate_lower_bound=-3.0)
    b = oracle.beta_transform(b_raw, beta_sigmoid=True)
    ref = oracle.gdp_fwd(c["q"], c["k"], c["v"], g_log, b, c["cu"], n, initial_state=c["s0"])
    errs = {"o": rel(o.float().cpu(), ref["o"]), "final": rel(fin.cpu(), ref["final_state"])}
    print("[parity] gdp n=2 bounded gate: " + ", ".join(f"{k_} {v_:.2e}" for k_, v_ in errs.items()))
    assert errs["o"] <= O_TOL and errs["final"] <= S_TOL, errs


def test_gdp_three_updates_token_major_transforms():
    """n = 3 (chunks end inside tokens), token-major [T, n, H, D] inputs, the softplus gate and
    beta logits in the kernel."""
    n = 3
    c = gdp_case([50, 7, 130], n, 1, 2, 64, 64, seed=511, slow=False)
    gen = torch.Generator().manual_seed(512)
    T = c["q"].shape[0]
    g_raw = torch.randn(T, 2, generator=gen)
    b_raw = torch.randn(T * n, 2, generator=gen)
    a_log, dt_bias = torch.log(torch.tensor([0.05, 0.2])), torch.tensor([-1.0, 0.5])
    d = dev()
    k4 = c["k"].view(T, n, 1, 64).to(d)
    v4 = c["v"].view(T, n, 2, 64).to(d)
    b4 = b_raw.view(T, n, 2).to(d)
    o, fin, _ = la.gdn_fwd(c["q"].to(d), k4, v4, g_raw.to(d), b4, c["cu"].to(d), initial_state=c["s0"].to(d),
                           num_householder=n, a_log=a_log.to(d), dt_bias=dt_bias.to(d), beta_sigmoid=True)
    g_log = oracle.gate_transform(g_raw, gate="softplus", a_log=a_log, dt_bias=dt_bias)
    b = oracle.beta_transform(b_raw, beta_sigmoid=True)
    ref = oracle.gdp_fwd(c["q"], c["k"], c["v"], g_log, b, c["cu"], n, initial_state=c["s0"])
    errs = {"o": rel(o.float().cpu(), ref["o"]), "final": rel(fin.cpu(), ref["final_state"])}
    print("[parity] gdp n=3: " + ", ".join(f"{k_} {v_:.2e}" for k_, v_ in errs.items()))
    assert errs["o"] <= O_TOL and errs["final"] <= S_TOL, errs


def test_gdp_one_update_is_gdn_bitwise():
    c = gdp_case([100, 64], 1, 2, 2, 64, 64, seed=521)
    d = dev()
    args = [x.to(d) for x in (c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu"])]
    o1, f1, _ = la.gdn_fwd(*args, initial_state=c["s0"].to(d))
    o2, f2, _ = la.gdn_fwd(*args, initial_state=c["s0"].to(d), num_householder=1)
    assert torch.equal(o1, o2) and torch.equal(f1, f2)


def test_gdp_native_with_state_pool():
    """n = 2 natively with a state pool: each sequence starts from its slot and its end state goes
    back into that slot (the other slots untouched)."""
    n = 2
    c = gdp_case([40, 1, 97], n, 1, 2, 128, 128, seed=541)
    d = dev()
    gen = torch.Generator().manual_seed(542)
    P = 6
    pool = 0.1 * torch.randn(P, 2, 128, 128, generator=gen)
    idx = torch.tensor([4, 0, 2], dtype=torch.int32)
    pool_d = pool.to(d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    o, _, _ = la.gdn_fwd(c["q"].to(d), c["k"].to(d), c["v"].to(d), c["g"].to(d), c["beta"].to(d), c["cu"].to(d),
                         initial_state=pool_d, state_indices=idx.to(d), num_householder=n, status=status)
    assert la.read_status(status) == 0
    ref = oracle.gdp_fwd(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu"], n, initial_state=pool[idx.long()])
    got_pool = pool_d.cpu()
    errs = {"o": rel(o.float().cpu(), ref["o"]), "slots": rel(got_pool[idx.long()], ref["final_state"])}
    print("[parity] gdp n=2 state pool: " + ", ".join(f"{k_} {v_:.2e}" for k_, v_ in errs.items()))
    assert errs["o"] <= O_TOL and errs["slots"] <= S_TOL, errs
    untouched = [i for i in range(P) if i not in idx.tolist()]
    assert torch.equal(got_pool[untouched], pool[untouched])
