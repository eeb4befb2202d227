"""The backward (gdn_bwd) vs the fp64 oracle's reverse-mode gradients, through the C ABI.

Tolerances (max|x - ref| / max|ref| per tensor): bf16 gradients (dq, dk, dv) 1e-2, as for o;
fp32 gradients (dg, dbeta, d_initial_state) 2e-3, as for the fp32 states.  The loss is
sum(d_o * o) + sum(d_final_state * final_state) with seeded N(0,1) cotangents."""
import numpy as np
import pytest
import torch

import oracle
import gated_delta_rule_29_gb300 as la
from gated_delta_rule_29_gb300 import workloads as W

pytestmark = pytest.mark.gpu

BF16_TOL = 1e-2
F32_TOL = 2e-3


def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def rel(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.abs(ref).max()
    assert den > 0, "reference is all zero: the comparison would be vacuous"
    return float(np.abs(got - ref).max() / den)


def cotangents(w, seed, with_final=True):
    gen = torch.Generator().manual_seed(seed)
    T = int(w.cu_seqlens[-1])
    do = torch.randn(T, w.HV, w.V, generator=gen).to(torch.bfloat16)
    dfin = torch.randn(w.N, w.HV, w.K, w.V, generator=gen) if with_final else None
    return do, dfin


def run_bwd(w, do, dfin, l2=True, checkpoints=None, scale=None, checkpoint_every_n=64):
    d = dev()
    status = torch.zeros(1, dtype=torch.int32, device=d)
    out = la.gdn_bwd(w.q.to(d), w.k.to(d), w.v.to(d), w.g.to(d), w.beta.to(d), w.cu_seqlens.to(d), do.to(d),
                     use_qk_l2norm=l2, scale=scale,
                     initial_state=None if w.initial_state is None else w.initial_state.to(d),
                     d_final_state=None if dfin is None else dfin.to(d), checkpoints=checkpoints, status=status,
                     checkpoint_every_n=checkpoint_every_n)
    assert la.read_status(status) == 0
    return [None if x is None else x.float().cpu().numpy() for x in out]


def compare(w, got, ref, units=None, label="", f32_tol=F32_TOL):
    names = ["dq", "dk", "dv", "dg", "dbeta", "d_initial_state"]
    errs = {}
    for name, x in zip(names, got):
        if x is None or (name == "d_initial_state" and w.initial_state is None):
            continue
        r = ref[name]
        if units is not None and name in ("dv", "dg", "dbeta"):
            cu = w.cu_seqlens.numpy().astype(np.int64)
            x = np.concatenate([x[cu[i]:cu[i + 1], h] for i, h in units])
            r = np.concatenate([r[cu[i]:cu[i + 1], h] for i, h in units])
        errs[name] = rel(x, r)
    print(f"[parity] bwd {w.name}{label}: " + ", ".join(f"{k_} {v_:.2e}" for k_, v_ in errs.items()))
    for name, e in errs.items():
        assert e <= (BF16_TOL if name in ("dq", "dk", "dv") else f32_tol), errs
    return errs


@pytest.mark.parametrize("K,V", [(64, 64), (128, 128), (64, 128), (128, 64)])
def test_bwd_ragged_grouped_heads(K, V):
    """Ragged sequences (one token, a chunk +- 1, an empty one, several chunks), grouped heads,
    a start state and a final-state cotangent, slow decay."""
    w = W.draw("bwd ragged", [1, 63, 0, 64, 65, 200], 2, 4, K, V, seed=401 + K + V, initial_state=True,
               slow_decay=True)
    do, dfin = cotangents(w, 402)
    got = run_bwd(w, do, dfin)
    ref = oracle.gdn_bwd(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, do, initial_state=w.initial_state,
                         d_final_state=dfin)
    compare(w, got, ref)


def test_bwd_page_distributions_no_final_no_start():
    """The pages' gate and beta distributions (fast decay), no start state, no final-state
    cotangent."""
    w = W.draw("bwd page", [300, 129, 1000], 4, 4, 128, 128, seed=411)
    do, _ = cotangents(w, 412, with_final=False)
    got = run_bwd(w, do, None)
    ref = oracle.gdn_bwd(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, do)
    compare(w, got, ref)


def test_bwd_without_l2norm():
    """Keys and queries scaled to unit-order norms by hand, the kernel's norm off."""
    w = W.draw("bwd no-norm", [150, 70], 1, 2, 64, 64, seed=421, initial_state=True, slow_decay=True)
    w.q = (w.q.float() / 8.0).to(torch.bfloat16)
    w.k = (w.k.float() / 8.0).to(torch.bfloat16)
    do, dfin = cotangents(w, 422)
    got = run_bwd(w, do, dfin, l2=False, scale=0.5)
    ref = oracle.gdn_bwd(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, do, scale=0.5, use_qk_l2norm=False,
                         initial_state=w.initial_state, d_final_state=dfin)
    compare(w, got, ref)


def test_bwd_reuses_forward_checkpoints_bitwise():
    """Checkpoints every 64 tokens from gdn_fwd give bitwise the gradients of the regenerated path."""
    w = W.draw("bwd ckpt", [130, 64, 257], 2, 2, 128, 128, seed=431, initial_state=True, slow_decay=True)
    do, dfin = cotangents(w, 432)
    d = dev()
    _, _, ck = la.gdn_fwd(w.q.to(d), w.k.to(d), w.v.to(d), w.g.to(d), w.beta.to(d), w.cu_seqlens.to(d),
                          initial_state=w.initial_state.to(d), checkpoint_every_n=64, checkpoint_dtype=torch.float32)
    a = run_bwd(w, do, dfin)
    b = run_bwd(w, do, dfin, checkpoints=ck)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def fwd_checkpoints(w, n, dtype):
    d = dev()
    _, _, ck = la.gdn_fwd(w.q.to(d), w.k.to(d), w.v.to(d), w.g.to(d), w.beta.to(d), w.cu_seqlens.to(d),
                          initial_state=None if w.initial_state is None else w.initial_state.to(d),
                          checkpoint_every_n=n, checkpoint_dtype=dtype)
    return ck


@pytest.mark.parametrize("n", [128, 256])
def test_bwd_sparse_fp32_checkpoints_regenerate_the_same_bits(n):
    """Page, "States and checkpoints": the backward regenerates the states entering every chunk
    from sparser rows.  The segments start from the forward's exact fp32 states, so the
    gradients are bitwise those computed from the rows every 64 tokens (and from a full re-run).
    Ragged lengths: partial last segments and chunks, an empty sequence, one-chunk sequences."""
    w = W.draw("bwd sparse ckpt", [300, 0, 64, 1000, 129, 1, 520], 2, 4, 128, 128, seed=471, initial_state=True,
               slow_decay=True)
    do, dfin = cotangents(w, 472)
    dense = run_bwd(w, do, dfin, checkpoints=fwd_checkpoints(w, 64, torch.float32))
    sparse = run_bwd(w, do, dfin, checkpoints=fwd_checkpoints(w, n, torch.float32), checkpoint_every_n=n)
    regen = run_bwd(w, do, dfin)
    for name, x, y, z in zip(["dq", "dk", "dv", "dg", "dbeta", "d_initial_state"], dense, sparse, regen):
        assert np.array_equal(x, y), name
        assert np.array_equal(x, z), name


@pytest.mark.parametrize("n,KV", [(64, 64), (192, 64), (64, 128), (192, 128)])
def test_bwd_bf16_checkpoints_against_oracle(n, KV):
    """bf16 rows (the io dtype) at the chunk cadence are widened; at n = 192 the dense series is
    regenerated from them.  The states then carry bf16's 2^-9 relative rounding before the
    backward starts, so every gradient is held to the bf16 bound 1e-2 (as bf16 checkpoints are);
    the oracle differentiates the exact recurrence.  K = V = 64: the tile kernel; 128: the
    tensor-core schedule."""
    w = W.draw("bwd bf16 ckpt", [200, 64, 450, 77], 2, 2, KV, KV, seed=481, initial_state=True, slow_decay=True)
    do, dfin = cotangents(w, 482)
    got = run_bwd(w, do, dfin, checkpoints=fwd_checkpoints(w, n, torch.bfloat16), checkpoint_every_n=n)
    ref = oracle.gdn_bwd(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, do, initial_state=w.initial_state,
                         d_final_state=dfin)
    compare(w, got, ref, label=f" bf16 rows every {n}", f32_tol=BF16_TOL)


def test_bwd_dense_batch_reuses_its_1024_token_checkpoints_bitwise():
    """The dense batch's forward keeps fp32 rows every 1024 tokens; the backward from them equals
    the backward from rows every 64 tokens bit for bit."""
    w = W.config(3, slow_decay=True)
    do, dfin = cotangents(w, 491)
    a = run_bwd(w, do, dfin, checkpoints=fwd_checkpoints(w, 64, torch.float32))
    b = run_bwd(w, do, dfin, checkpoints=fwd_checkpoints(w, 1024, torch.float32), checkpoint_every_n=1024)
    for name, x, y in zip(["dq", "dk", "dv", "dg", "dbeta", "d_initial_state"], a, b):
        assert np.array_equal(x, y), name


def test_bwd_batch_invariant():
    """A sequence's gradients are bitwise the same alone and inside a batch."""
    w = W.draw("bwd batch", [90, 200, 33, 128], 2, 2, 64, 64, seed=441, initial_state=True, slow_decay=True)
    do, dfin = cotangents(w, 442)
    full = run_bwd(w, do, dfin)
    cu = w.cu_seqlens.numpy().astype(np.int64)
    i = 1
    sl = slice(cu[i], cu[i + 1])
    sub = W.Workload(name="one", cu_seqlens=torch.tensor([0, cu[i + 1] - cu[i]]), q=w.q[sl], k=w.k[sl], v=w.v[sl],
                     g=w.g[sl].contiguous(), beta=w.beta[sl].contiguous(), initial_state=w.initial_state[i:i + 1])
    alone = run_bwd(sub, do[sl], dfin[i:i + 1])
    for name, x, y in zip(["dq", "dk", "dv", "dg", "dbeta"], full[:5], alone[:5]):
        assert np.array_equal(x[sl], y), name
    assert np.array_equal(full[5][i], alone[5][0])


def test_bwd_dense_batch_sampled():
    """The dense batch (T = 65536, H = 32, K = V = 128, start state): the oracle recomputes two
    sampled (sequence, head) units."""
    w = W.config(3)
    do, dfin = cotangents(w, 451)
    got = run_bwd(w, do, dfin)
    units = [(0, 0), (6, 21)]
    mask = np.zeros((w.N, w.HV), dtype=bool)
    for i, h in units:
        mask[i, h] = True
    ref = oracle.gdn_bwd(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, do, initial_state=w.initial_state,
                         d_final_state=dfin, unit_mask=mask)
    cu = w.cu_seqlens.numpy().astype(np.int64)
    # per-unit rows of every gradient (dq / dk rows of a unit's q/k head: H = HK here)
    errs = {}
    for name, x in zip(["dq", "dk", "dv", "dg", "dbeta"], got[:5]):
        xs = np.concatenate([x[cu[i]:cu[i + 1], h] for i, h in units])
        rs = np.concatenate([ref[name][cu[i]:cu[i + 1], h] for i, h in units])
        errs[name] = rel(xs, rs)
    errs["d_initial_state"] = rel(np.stack([got[5][i, h] for i, h in units]),
                                  np.stack([ref["d_initial_state"][i, h] for i, h in units]))
    print("[parity] bwd dense batch sampled: " + ", ".join(f"{k_} {v_:.2e}" for k_, v_ in errs.items()))
    for name, e in errs.items():
        assert e <= (BF16_TOL if name in ("dq", "dk", "dv") else F32_TOL), errs


def test_bwd_softplus_gate_and_beta_sigmoid():
    """The backward through the forward's input transforms: softplus gate with a_log, dt_bias
    (raw gate inputs N(0,1), rates exp(a_log) in [0.02, 0.1] so that state crosses chunks) and
    beta logits through the sigmoid; gradients of the raw inputs, d_a_log and d_dt_bias."""
    w = W.draw("bwd softplus", [1, 100, 64, 250], 2, 4, 128, 128, seed=461, initial_state=True)
    gen = torch.Generator().manual_seed(462)
    g_raw = torch.randn(w.T, w.HV, generator=gen)
    b_logit = torch.randn(w.T, w.HV, generator=gen)
    a_log = torch.log(0.02 + 0.08 * torch.rand(w.HV, generator=gen))
    dt_bias = 0.5 * torch.randn(w.HV, generator=gen)
    do, dfin = cotangents(w, 463)
    d = dev()
    status = torch.zeros(1, dtype=torch.int32, device=d)
    out = la.gdn_bwd(w.q.to(d), w.k.to(d), w.v.to(d), g_raw.to(d), b_logit.to(d), w.cu_seqlens.to(d), do.to(d),
                     initial_state=w.initial_state.to(d), d_final_state=dfin.to(d), status=status,
                     a_log=a_log.to(d), dt_bias=dt_bias.to(d), beta_sigmoid=True)
    assert la.read_status(status) == 0
    assert len(out) == 8
    got = [x.float().cpu().numpy() for x in out]
    ref = oracle.gdn_bwd(w.q, w.k, w.v, g_raw, b_logit, w.cu_seqlens, do, initial_state=w.initial_state,
                         d_final_state=dfin, gate="softplus", a_log=a_log, dt_bias=dt_bias, beta_sigmoid=True)
    compare(w, got[:6], ref, label=" softplus gate + beta sigmoid")
    errs = {name: rel(x, ref[name]) for name, x in zip(["d_a_log", "d_dt_bias"], got[6:])}
    print("[parity] bwd gate parameters: " + ", ".join(f"{k_} {v_:.2e}" for k_, v_ in errs.items()))
    assert max(errs.values()) <= F32_TOL, errs


def test_bwd_bounded_gate_bf16_beta_logits():
    """The bounded sigmoid gate (lower bound -0.1) and bf16 beta logits through the sigmoid."""
    w = W.draw("bwd bounded", [70, 129], 1, 2, 64, 64, seed=471, initial_state=True)
    gen = torch.Generator().manual_seed(472)
    g_raw = torch.randn(w.T, w.HV, generator=gen)
    b_logit = torch.randn(w.T, w.HV, generator=gen).to(torch.bfloat16)
    do, dfin = cotangents(w, 473)
    d = dev()
    status = torch.zeros(1, dtype=torch.int32, device=d)
    out = la.gdn_bwd(w.q.to(d), w.k.to(d), w.v.to(d), g_raw.to(d), b_logit.to(d), w.cu_seqlens.to(d), do.to(d),
                     initial_state=w.initial_state.to(d), d_final_state=dfin.to(d), status=status,
                     gate_lower_bound=-0.1, beta_sigmoid=True)
    assert la.read_status(status) == 0
    got = [x.float().cpu().numpy() for x in out]
    ref = oracle.gdn_bwd(w.q, w.k, w.v, g_raw, b_logit.float(), w.cu_seqlens, do, initial_state=w.initial_state,
                         d_final_state=dfin, gate="sigmoid_bound", gate_lower_bound=-0.1, beta_sigmoid=True)
    compare(w, got, ref, label=" bounded gate + bf16 beta logits")


def test_bwd_bf16_start_state_regenerated_checkpoints():
    """A bf16 start state: the regenerated forward reads it as given, and the gradient with
    respect to it comes back in fp32."""
    w = W.draw("bwd bf16 s0", [96, 200], 2, 2, 128, 64, seed=481, initial_state=True, slow_decay=True)
    w.initial_state = w.initial_state.to(torch.bfloat16)
    do, dfin = cotangents(w, 482)
    got = run_bwd(w, do, dfin)
    ref = oracle.gdn_bwd(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, do, initial_state=w.initial_state.float(),
                         d_final_state=dfin)
    compare(w, got, ref, label=" bf16 start state")


@pytest.mark.parametrize("save_checkpoints,n,KV", [(True, 64, 64), (True, 128, 64), (False, 64, 64),
                                                    (True, 64, 128), (False, 64, 128)])
def test_autograd_matches_oracle_gradients(save_checkpoints, n, KV):
    """gdn_attention under torch.autograd: a scalar loss of o and the final state, backward through
    the library's kernels, gradients of every input against the oracle's reverse mode (the forward
    keeping fp32 states every 64 or 128 tokens, or none; K = V = 128 takes the tensor-core
    backward)."""
    w = W.draw("autograd", [70, 129, 1, 300], 2, 4, KV, KV, seed=491, initial_state=True, slow_decay=True)
    d = dev()
    gen = torch.Generator().manual_seed(492)
    wo = torch.randn(w.T, w.HV, w.V, generator=gen).to(torch.bfloat16)
    wf = torch.randn(w.N, w.HV, w.K, w.V, generator=gen)
    leaves = [x.to(d).requires_grad_(True) for x in (w.q, w.k, w.v, w.g, w.beta, w.initial_state)]
    q, k, v, g, beta, s0 = leaves
    o, fin = la.gdn_attention(q, k, v, g, beta, w.cu_seqlens.to(d), initial_state=s0,
                              save_checkpoints=save_checkpoints, checkpoint_every_n=n)
    loss = (o.float() * wo.to(d).float()).sum() + (fin * wf.to(d)).sum()
    loss.backward()
    ref = oracle.gdn_bwd(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, wo, initial_state=w.initial_state,
                         d_final_state=wf)
    got = [x.grad.float().cpu().numpy() for x in leaves]
    compare(w, got, ref, label=f" autograd (saved checkpoints: {save_checkpoints}, every {n})")


def test_bwd_fused_projection_views_int64_cu_single_key_head():
    """q, k, v as column slices of one fused projection, gradients written into column slices of
    one fused gradient buffer (the layout a fused projection's backward consumes), int64
    cu_seqlens, one key head shared by four value heads, explicit scale, K != V."""
    w = W.draw("bwd fused views", [150, 64, 1, 93], 1, 4, 128, 64, seed=451, initial_state=True, slow_decay=True)
    do, dfin = cotangents(w, 452)
    d = dev()
    T = w.T
    a, b = w.HK * w.K, 2 * w.HK * w.K
    fused = torch.cat([w.q.reshape(T, -1), w.k.reshape(T, -1), w.v.reshape(T, -1)], dim=1).to(d)
    q, k, v = fused[:, :a].view(T, w.HK, w.K), fused[:, a:b].view(T, w.HK, w.K), fused[:, b:].view(T, w.HV, w.V)
    assert not q.is_contiguous() and not v.is_contiguous()
    grad = torch.full_like(fused, float("nan"))
    gb = torch.full((T, 2 * w.HV), float("nan"), dtype=torch.float32, device=d)
    out = (grad[:, :a].view(T, w.HK, w.K), grad[:, a:b].view(T, w.HK, w.K), grad[:, b:].view(T, w.HV, w.V),
           gb[:, :w.HV], gb[:, w.HV:], None)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    res = la.gdn_bwd(q, k, v, w.g.to(d), w.beta.to(d), w.cu_seqlens.to(torch.int64).to(d), do.to(d), scale=0.3,
                     initial_state=w.initial_state.to(d), d_final_state=dfin.to(d), status=status, out=out)
    assert la.read_status(status) == 0
    for x, y in zip(res[:5], out[:5]):
        assert x.data_ptr() == y.data_ptr()
    assert not torch.isnan(grad).any() and not torch.isnan(gb).any()
    got = [x.float().cpu().numpy() for x in res[:6]]
    ref = oracle.gdn_bwd(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, do, scale=0.3, initial_state=w.initial_state,
                         d_final_state=dfin)
    compare(w, got, ref)
    # the same gradients as through freshly allocated contiguous outputs, bitwise
    plain = run_bwd(w, do, dfin, scale=0.3)
    for name, x, y in zip(["dq", "dk", "dv", "dg", "dbeta", "d_initial_state"], got, plain):
        assert np.array_equal(x, y), name


def test_bwd_out_buffers_rejected_when_mismatched():
    """A preallocated output of the wrong shape or dtype is an argument error, raised before launch."""
    w = W.draw("bwd out check", [64], 1, 1, 64, 64, seed=461)
    do, _ = cotangents(w, 462, with_final=False)
    d = dev()
    args = [x.to(d) for x in (w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, do)]
    with pytest.raises(ValueError):
        la.gdn_bwd(*args, out=(torch.empty(w.T, w.HK, w.K + 1, dtype=torch.bfloat16, device=d),))
    with pytest.raises(ValueError):
        la.gdn_bwd(*args, out=(None, None, None, torch.empty(w.T, w.HV, dtype=torch.float64, device=d)))


def test_bwd_extreme_but_valid_values():
    """Gates from 0 down to -30, beta exactly 0 or 1, all-zero q and k rows under the norm, a
    start state and a final-state cotangent: finite gradients within tolerance of the oracle."""
    w = W.draw("bwd extreme", [200, 77, 64], 2, 2, 128, 128, seed=471, initial_state=True)
    gen = torch.Generator().manual_seed(472)
    T = w.T
    u = torch.rand(T, w.HV, generator=gen)
    w.g = torch.where(u < 0.1, torch.full_like(u, -30.0), torch.where(u < 0.5, torch.zeros_like(u), -0.01 * u))
    r = torch.rand(T, w.HV, generator=gen)
    w.beta = torch.where(r < 0.2, torch.zeros_like(r), torch.where(r < 0.4, torch.ones_like(r), r)).contiguous()
    w.g = w.g.contiguous()
    q, k = w.q.clone(), w.k.clone()
    q[torch.rand(T, generator=gen) < 0.05] = 0
    k[torch.rand(T, generator=gen) < 0.05] = 0
    w.q, w.k = q, k
    do, dfin = cotangents(w, 473)
    got = run_bwd(w, do, dfin)
    for x in got:
        if x is not None:
            assert np.isfinite(x).all()
    ref = oracle.gdn_bwd(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, do, initial_state=w.initial_state,
                         d_final_state=dfin)
    compare(w, got, ref)
