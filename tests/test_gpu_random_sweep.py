"""Seeded random sweep over the forward's and the backward's options, against the fp64 oracle.

Each case draws, from its own seed: 1-5 sequences with lengths mixing the edge cases (empty,
one token, a chunk +- 1) with random ones; 1 or 2 key heads shared by 1, 2 or 4 value heads;
K, V in {64, 128}; the q/k L2 norm on or off; an explicit scale or the default; no start
state, an fp32 or a bf16 one; checkpoints every 64, 128 or 192 tokens in fp32 or bf16, or
none; the plain log gate (the pages' fast decay or a slow one), the softplus gate or the
bounded sigmoid gate; beta as values or as fp32 / bf16 logits; int32 or int64 cu_seqlens.
Tolerances as in test_gpu_parity / test_gpu_bwd (max|x - ref| / max|ref| per tensor)."""
import numpy as np
import pytest
import torch

import oracle
import gated_delta_rule_29_gb300 as la

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


def draw_case(seed, backward=False):
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    N = int(rng.integers(1, 6))
    pool = [0, 1, 63, 64, 65, 128, 129]
    lengths = [int(rng.choice(pool)) if rng.random() < 0.5 else int(rng.integers(2, 400)) for _ in range(N)]
    if sum(lengths) == 0:
        lengths[0] = 100
    HK = int(rng.choice([1, 2]))
    HV = HK * int(rng.choice([1, 2, 4]))
    K, V = int(rng.choice([64, 128])), int(rng.choice([64, 128]))
    T = sum(lengths)
    c = dict(seed=seed, lengths=lengths, HK=HK, HV=HV, K=K, V=V)
    c["l2"] = bool(rng.random() < 0.75)
    c["scale"] = None if rng.random() < 0.5 else float(rng.uniform(0.1, 1.0))
    c["s0"] = str(rng.choice(["none", "f32", "bf16"]))
    c["ck"] = 0 if backward else int(rng.choice([0, 64, 128, 192]))
    c["ck_dtype"] = torch.float32 if rng.random() < 0.5 else torch.bfloat16
    c["gate"] = str(rng.choice(["log_fast", "log_slow", "softplus", "bound"]))
    c["beta"] = str(rng.choice(["plain", "logit_f32", "logit_bf16"]))
    c["cu64"] = bool(rng.random() < 0.5)
    c["gb_fused"] = bool(rng.random() < 0.3)
    q = torch.randn(T, HK, K, generator=gen)
    k = torch.randn(T, HK, K, generator=gen)
    if not c["l2"]:
        q, k = q * 0.05, k * 0.05
    c["q"], c["k"] = q.to(torch.bfloat16), k.to(torch.bfloat16)
    c["v"] = torch.randn(T, HV, V, generator=gen).to(torch.bfloat16)
    graw = torch.randn(T, HV, generator=gen)
    braw = torch.randn(T, HV, generator=gen)
    okw, kw = {}, {}
    if c["gate"] == "log_fast":
        c["g"] = -torch.nn.functional.softplus(graw)
    elif c["gate"] == "log_slow":
        c["g"] = -torch.nn.functional.softplus(graw) * 1e-3
    elif c["gate"] == "softplus":
        c["g"] = graw
        a_log = torch.log(torch.tensor(rng.uniform(0.005, 1.0, size=HV), dtype=torch.float32))
        dt_bias = torch.tensor(rng.uniform(-4.0, 1.0, size=HV), dtype=torch.float32)
        okw.update(gate="softplus", a_log=a_log, dt_bias=dt_bias)
        kw.update(a_log=a_log, dt_bias=dt_bias)
    else:
        c["g"] = graw
        lb = -float(rng.uniform(0.01, 1.0))
        okw.update(gate="sigmoid_bound", gate_lower_bound=lb)
        kw.update(gate_lower_bound=lb)
    if c["beta"] == "plain":
        c["b"] = torch.sigmoid(braw) * (0.2 if c["gate"] == "log_slow" else 1.0)
    else:
        c["b"] = braw.to(torch.bfloat16) if c["beta"] == "logit_bf16" else braw
        okw.update(beta_sigmoid=True)
        kw.update(beta_sigmoid=True)
    if c["gb_fused"] and c["b"].dtype == torch.float32:
        # g and beta as column slices of one [T, 2 HV] projection output (strided views)
        c["gb"] = torch.cat([c["g"].reshape(T, HV), c["b"].reshape(T, HV)], dim=1)
    else:
        c["gb_fused"] = False
    s0 = None
    if c["s0"] != "none":
        s0 = 0.1 * torch.randn(N, HV, K, V, generator=gen)
        if c["s0"] == "bf16":
            s0 = s0.to(torch.bfloat16)
    c["s0t"] = s0
    c["cu"] = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]),
                           dtype=torch.int64 if c["cu64"] else torch.int32)
    c["okw"], c["kw"] = okw, kw
    return c


def gate_beta_on(c, d):
    """g and beta on the device: two tensors, or two column slices of one fused buffer."""
    if c["gb_fused"]:
        gb = c["gb"].to(d)
        HV = c["HV"]
        g, b = gb[:, :HV], gb[:, HV:]
        assert not g.is_contiguous() and g.stride(0) == 2 * HV
        return g, b
    return c["g"].to(d), c["b"].to(d)


def label(c):
    keys = ("seed", "lengths", "HK", "HV", "K", "V", "l2", "scale", "s0", "ck", "gate", "beta", "cu64", "gb_fused")
    return " ".join(f"{x}={c[x]}" for x in keys) + (f" ck_dtype={c['ck_dtype']}" if c["ck"] else "")


@pytest.mark.parametrize("case", range(64))
def test_forward_random_case(case):
    c = draw_case(7000 + case)
    d = dev()
    status = torch.zeros(1, dtype=torch.int32, device=d)
    kw = {x: (y.to(d) if isinstance(y, torch.Tensor) else y) for x, y in c["kw"].items()}
    o, fin, ck = la.gdn_fwd(c["q"].to(d), c["k"].to(d), c["v"].to(d), *gate_beta_on(c, d), c["cu"].to(d),
                            scale=c["scale"], use_qk_l2norm=c["l2"],
                            initial_state=None if c["s0t"] is None else c["s0t"].to(d),
                            checkpoint_every_n=c["ck"], checkpoint_dtype=c["ck_dtype"], status=status, **kw)
    assert la.read_status(status) == 0
    s0 = None if c["s0t"] is None else c["s0t"].float()
    ref = oracle.gdn_fwd(c["q"], c["k"], c["v"], c["g"], c["b"].float(), c["cu"], scale=c["scale"],
                         use_qk_l2norm=c["l2"], initial_state=s0, checkpoint_every_n=c["ck"], **c["okw"])
    errs = {"o": rel(o.float().cpu(), ref["o"]), "final": rel(fin.cpu(), ref["final_state"])}
    if c["ck"]:
        if np.abs(ref["checkpoints"]).max() == 0:  # only entry rows from a zero start: exact zeros
            assert not ck.float().cpu().numpy().any()
        else:
            errs["ckpt"] = rel(ck.float().cpu(), ref["checkpoints"])
    print(f"[parity] sweep fwd {label(c)}: " + ", ".join(f"{x} {y:.2e}" for x, y in errs.items()))
    ck_tol = S_TOL if c["ck_dtype"] == torch.float32 else BF16_STATE_TOL
    assert errs["o"] <= O_TOL and errs["final"] <= S_TOL and errs.get("ckpt", 0.0) <= ck_tol, (label(c), errs)


@pytest.mark.parametrize("case", range(20))
def test_backward_random_case(case):
    c = draw_case(7500 + case, backward=True)
    d = dev()
    gen = torch.Generator().manual_seed(7500 + case)
    T, N = sum(c["lengths"]), len(c["lengths"])
    do = torch.randn(T, c["HV"], c["V"], generator=gen).to(torch.bfloat16)
    dfin = torch.randn(N, c["HV"], c["K"], c["V"], generator=gen) if case % 2 == 0 else None
    status = torch.zeros(1, dtype=torch.int32, device=d)
    kw = {x: (y.to(d) if isinstance(y, torch.Tensor) else y) for x, y in c["kw"].items()}
    out = la.gdn_bwd(c["q"].to(d), c["k"].to(d), c["v"].to(d), *gate_beta_on(c, d), c["cu"].to(d), do.to(d),
                     scale=c["scale"], use_qk_l2norm=c["l2"],
                     initial_state=None if c["s0t"] is None else c["s0t"].to(d),
                     d_final_state=None if dfin is None else dfin.to(d), status=status, **kw)
    assert la.read_status(status) == 0
    s0 = None if c["s0t"] is None else c["s0t"].float()
    ref = oracle.gdn_bwd(c["q"], c["k"], c["v"], c["g"], c["b"].float(), c["cu"], do, scale=c["scale"],
                         use_qk_l2norm=c["l2"], initial_state=s0, d_final_state=dfin, **c["okw"])
    names = ["dq", "dk", "dv", "dg", "dbeta"] + (["d_initial_state"] if s0 is not None else [])
    errs = {x: rel(y.float().cpu(), ref[x]) for x, y in zip(names, out)}
    if "a_log" in c["okw"]:
        errs["d_a_log"] = rel(out[6].cpu(), ref["d_a_log"])
        errs["d_dt_bias"] = rel(out[7].cpu(), ref["d_dt_bias"])
    print(f"[parity] sweep bwd {label(c)} dfinal={dfin is not None}: "
          + ", ".join(f"{x} {y:.2e}" for x, y in errs.items()))
    for x, e in errs.items():
        assert e <= (O_TOL if x in ("dq", "dk", "dv") else S_TOL), (label(c), errs)
