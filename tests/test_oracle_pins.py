"""Pins for the fp64 oracle: checks against facts fixed by the pages and by mathematics.

Every check below is an independent statement of what the Gated DeltaNet forward
(cuDNN Linear Attention page: the GDN recurrence, "States and checkpoints",
"Summaries") must produce, evaluated without the oracle's own loop:
  * a hand-derived worked example (tests/golden/gdn_hand_3tok.json);
  * brute-force dense products of the explicit K x K factors on tiny inputs;
  * closed forms: exact retrieval with orthonormal keys, pure decay (beta = 0),
    a single token from a zero start;
  * invariants: joint linearity in (v, S0), scale linearity, L2-norm invariance
    under positive row rescaling, grouped heads == duplicated heads;
  * summaries: span composition and the transition product order;
  * checkpoints: entry j equals the final state of the prefix of length j*n;
  * state round trip: [0, m) then [m, L) equals the unsplit run;
  * empty sequences;
  * the optional input transforms (softplus gate, bounded sigmoid gate, beta
    sigmoid) at arguments where they take exact values (ln 2, 1, 1/2, 3/4);
  * the state pool (state_indices): one-token updates against the explicit
    factor form, written back to the named slots, other slots untouched;
  * the backward: every gradient against central finite differences of the
    pinned forward (with and without the L2 norm, grouped heads, start state);
  * GDP (several updates per token) against its definition as dense products of
    the token's Householder-like factors, and n = 1 against GDN.
test_planted_mistakes_are_caught plants each of the oracle's known mutations
and requires at least one check to fail, so a plausible slip anywhere (a dropped
term, a flipped sign, a wrong index or orientation) cannot pass unnoticed.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(12345)


def _rand_case(lengths, HK, HV, K, V, seed, s0=False, gscale=1.0):
    rng = np.random.default_rng(seed)
    T = int(sum(lengths))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    q = rng.standard_normal((T, HK, K))
    k = rng.standard_normal((T, HK, K))
    v = rng.standard_normal((T, HV, V))
    g = -np.log1p(np.exp(rng.standard_normal((T, HV)))) * gscale
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, HV))))
    S0 = 0.3 * rng.standard_normal((len(lengths), HV, K, V)) if s0 else None
    return q, k, v, g, beta, cu, S0


def _rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = max(np.abs(b).max(), 1e-300)
    return float(np.abs(a - b).max() / den)


# --------------------------------------------------------------------------------------
# checks: each returns the worst relative error it saw for the given oracle mutation
# --------------------------------------------------------------------------------------

def check_golden(mutation=0):
    d = json.load(open(os.path.join(GOLDEN, "gdn_hand_3tok.json")))
    q = np.array(d["q"], dtype=np.float64)[:, None, :]
    k = np.array(d["k"], dtype=np.float64)[:, None, :]
    v = np.array(d["v"], dtype=np.float64)[:, None, :]
    g = np.log(np.array(d["decay"]))[:, None]
    beta = np.array(d["beta"], dtype=np.float64)[:, None]
    cu = np.array(d["cu_seqlens"])
    r = oracle.gdn_fwd(q, k, v, g, beta, cu, scale=d["scale"], use_qk_l2norm=False,
                       checkpoint_every_n=d["checkpoint_every_n"], mutation=mutation)
    s = oracle.gdn_summary(k, v, g, beta, cu, use_qk_l2norm=False, mutation=mutation)
    errs = [
        np.abs(r["o"][:, 0, :] - np.array(d["o"])).max(),
        np.abs(r["final_state"][0, 0] - np.array(d["final_state"])).max(),
        np.abs(r["checkpoints"][:, 0] - np.array(d["checkpoints"])).max(),
        np.abs(s["transition"][0, 0] - np.array(d["transition"])).max(),
        np.abs(s["end_state"][0, 0] - np.array(d["final_state"])).max(),
    ]
    return float(max(errs))


def _dense_reference(q, k, v, g, beta, cu, S0, scale, l2norm, HK, HV):
    """Explicit K x K factors multiplied densely: S_t = M_t S_{t-1} + beta k v^T."""
    T, _, K = k.shape
    V = v.shape[2]
    N = len(cu) - 1
    o = np.zeros((T, HV, V))
    fin = np.zeros((N, HV, K, V))
    trans = np.zeros((N, HV, K, K))
    for i in range(N):
        for h in range(HV):
            hk = h // (HV // HK)
            S = np.zeros((K, V)) if S0 is None else S0[i, h].copy()
            P = np.eye(K)
            for t in range(cu[i], cu[i + 1]):
                kt, qt = k[t, hk].copy(), q[t, hk].copy()
                if l2norm:
                    kt = kt / math.sqrt(kt @ kt + 1e-6)
                    qt = qt / math.sqrt(qt @ qt + 1e-6)
                M = math.exp(g[t, h]) * (np.eye(K) - beta[t, h] * np.outer(kt, kt))
                S = M @ S + beta[t, h] * np.outer(kt, v[t, h])
                P = M @ P
                o[t, h] = scale * S.T @ qt
            fin[i, h] = S
            trans[i, h] = P.T
    return o, fin, trans


def check_brute_force(mutation=0):
    worst = 0.0
    for l2 in (False, True):
        for (lengths, HK, HV, K, V, s0) in (([5, 3], 1, 1, 3, 4, True), ([4, 0, 6], 2, 4, 4, 3, False)):
            q, k, v, g, beta, cu, S0 = _rand_case(lengths, HK, HV, K, V, seed=7 + K, s0=s0)
            o, fin, tr = _dense_reference(q, k, v, g, beta, cu, S0, 0.7, l2, HK, HV)
            r = oracle.gdn_fwd(q, k, v, g, beta, cu, scale=0.7, use_qk_l2norm=l2,
                               initial_state=S0, mutation=mutation)
            s = oracle.gdn_summary(k, v, g, beta, cu, use_qk_l2norm=l2, mutation=mutation)
            _, fin0, _ = _dense_reference(q, k, v, g, beta, cu, None, 0.7, l2, HK, HV)
            worst = max(worst, _rel(r["o"], o), _rel(r["final_state"], fin),
                        _rel(s["transition"], tr), _rel(s["end_state"], fin0))
    return worst


def check_retrieval(mutation=0):
    """g = 0, beta = 1, orthonormal keys: o_t = scale * (newest value written under q's key)."""
    K = V = 8
    rng = np.random.default_rng(3)
    order = [0, 3, 5, 3, 7, 0, 1]           # key indices written, with rewrites
    T = len(order)
    basis = np.eye(K)
    k = basis[order][:, None, :]
    q = k.copy()                             # query the key just written
    v = rng.standard_normal((T, 1, V))
    g = np.zeros((T, 1))
    beta = np.ones((T, 1))
    cu = np.array([0, T])
    r = oracle.gdn_fwd(q, k, v, g, beta, cu, scale=1.5, use_qk_l2norm=False, mutation=mutation)
    err = _rel(r["o"][:, 0], 1.5 * v[:, 0])
    # the final state holds, in row j, the newest value written under key j
    expect = np.zeros((K, V))
    for t, j in enumerate(order):
        expect[j] = v[t, 0]
    err = max(err, _rel(r["final_state"][0, 0], expect))
    # querying an older key after later writes still returns its newest value
    q2 = basis[[0] * T][:, None, :]
    r2 = oracle.gdn_fwd(q2, k, v, g, beta, cu, scale=1.0, use_qk_l2norm=False, mutation=mutation)
    newest0 = [v[max(s for s in range(t + 1) if order[s] == 0), 0] for t in range(T)]
    err = max(err, _rel(r2["o"][:, 0], np.array(newest0)))
    return err


def check_pure_decay(mutation=0):
    """beta = 0: S_t = exp(sum g) S0 and o_t = scale exp(b_t) S0^T q_hat_t."""
    q, k, v, g, beta, cu, S0 = _rand_case([9, 4], 1, 2, 5, 3, seed=11, s0=True, gscale=0.3)
    beta[:] = 0.0
    r = oracle.gdn_fwd(q, k, v, g, beta, cu, scale=0.9, use_qk_l2norm=True, initial_state=S0,
                       mutation=mutation)
    worst = 0.0
    for i in range(2):
        for h in range(2):
            b = 0.0
            for t in range(cu[i], cu[i + 1]):
                b += g[t, h]
                qh = q[t, 0] / math.sqrt(q[t, 0] @ q[t, 0] + 1e-6)
                worst = max(worst, _rel(r["o"][t, h], 0.9 * math.exp(b) * S0[i, h].T @ qh))
            worst = max(worst, _rel(r["final_state"][i, h], math.exp(b) * S0[i, h]))
    return worst


def check_single_token(mutation=0):
    """One token from zero: S1 = beta k_hat v^T, o = scale beta (k_hat . q_hat) v."""
    rng = np.random.default_rng(5)
    K, V = 6, 4
    q = rng.standard_normal((1, 1, K))
    k = rng.standard_normal((1, 1, K))
    v = rng.standard_normal((1, 1, V))
    g = np.array([[-0.4]])
    beta = np.array([[0.6]])
    r = oracle.gdn_fwd(q, k, v, g, beta, np.array([0, 1]), scale=0.5, use_qk_l2norm=True,
                       mutation=mutation)
    kh = k[0, 0] / math.sqrt(k[0, 0] @ k[0, 0] + 1e-6)
    qh = q[0, 0] / math.sqrt(q[0, 0] @ q[0, 0] + 1e-6)
    return max(_rel(r["final_state"][0, 0], 0.6 * np.outer(kh, v[0, 0])),
               _rel(r["o"][0, 0], 0.5 * 0.6 * (kh @ qh) * v[0, 0]))


def check_linearity(mutation=0):
    """o and the final state are jointly linear in (v, S0); o is linear in scale."""
    q, k, v, g, beta, cu, S0 = _rand_case([7, 5], 1, 1, 4, 3, seed=21, s0=True)
    _, _, v2, _, _, _, S02 = _rand_case([7, 5], 1, 1, 4, 3, seed=22, s0=True)
    f = lambda vv, ss, sc=1.0, qq=q, kk=k: oracle.gdn_fwd(
        qq, kk, vv, g, beta, cu, scale=sc, initial_state=ss, use_qk_l2norm=True, mutation=mutation)
    a, b = 0.7, -1.3
    r = f(a * v + b * v2, a * S0 + b * S02)
    r1, r2 = f(v, S0), f(v2, S02)
    err = max(_rel(r["o"], a * r1["o"] + b * r2["o"]),
              _rel(r["final_state"], a * r1["final_state"] + b * r2["final_state"]))
    err = max(err, _rel(f(v, S0, sc=2.5)["o"], 2.5 * r1["o"]))
    return err


def check_norm_invariance(mutation=0):
    """With the L2 norm on, positive per-row rescaling of q and k leaves o unchanged
    up to the 1e-6 inside the square root (rows here have |x|^2 >= 0.5)."""
    q, k, v, g, beta, cu, S0 = _rand_case([7, 5], 1, 1, 4, 3, seed=21, s0=True)
    rs = np.random.default_rng(23).uniform(1.0, 5.0, size=(q.shape[0], 1, 1))
    f = lambda qq, kk: oracle.gdn_fwd(qq, kk, v, g, beta, cu, initial_state=S0,
                                      use_qk_l2norm=True, mutation=mutation)["o"]
    return _rel(f(q * rs, k * rs[::-1]), f(q, k))


def check_gva(mutation=0):
    """HK = 2, HV = 6 equals HK = HV = 6 with q/k heads duplicated in contiguous groups."""
    q, k, v, g, beta, cu, S0 = _rand_case([6, 3], 2, 6, 4, 3, seed=31, s0=True)
    idx = [h // 3 for h in range(6)]
    r = oracle.gdn_fwd(q, k, v, g, beta, cu, initial_state=S0, mutation=mutation)
    rd = oracle.gdn_fwd(q[:, idx], k[:, idx], v, g, beta, cu, initial_state=S0, mutation=mutation)
    return max(_rel(r["o"], rd["o"]), _rel(r["final_state"], rd["final_state"]))


def check_span_composition(mutation=0):
    """Summaries of consecutive spans compose to the unsplit end state and transition."""
    lengths = [5, 7, 4]
    q, k, v, g, beta, _, _ = _rand_case([sum(lengths)], 1, 2, 4, 3, seed=41, gscale=0.2)
    S_init = 0.5 * np.random.default_rng(42).standard_normal((1, 2, 4, 3))
    whole_cu = np.array([0, sum(lengths)])
    span_cu = np.concatenate([[0], np.cumsum(lengths)])
    full = oracle.gdn_fwd(q, k, v, g, beta, whole_cu, initial_state=S_init, mutation=mutation)
    s = oracle.gdn_summary(k, v, g, beta, span_cu, mutation=mutation)
    sw = oracle.gdn_summary(k, v, g, beta, whole_cu, mutation=mutation)
    S = oracle.compose_spans(s["transition"], s["end_state"], S_init[0], mutation=mutation)[-1]
    tr_prod = np.stack([np.eye(4)] * 2)
    for j in range(len(lengths)):
        tr_prod = np.einsum("hab,hbc->hac", tr_prod, s["transition"][j])
    err = max(_rel(S, full["final_state"][0]), _rel(tr_prod, sw["transition"][0]))
    # summary from a non-zero start equals transition applied to the start plus S_H
    st = oracle.gdn_summary(k, v, g, beta, whole_cu, start_state=S_init, mutation=mutation)
    err = max(err, _rel(st["end_state"][0],
                        np.einsum("hab,hav->hbv", sw["transition"][0], S_init[0]) + sw["end_state"][0]))
    return err


def check_checkpoints(mutation=0):
    """Checkpoint entry j of a sequence equals the final state of its first j*n tokens."""
    n = 3
    lengths = [7, 3, 0, 5]
    q, k, v, g, beta, cu, S0 = _rand_case(lengths, 1, 1, 3, 2, seed=51, s0=True, gscale=0.2)
    r = oracle.gdn_fwd(q, k, v, g, beta, cu, initial_state=S0, checkpoint_every_n=n,
                       mutation=mutation)
    off, R = oracle.checkpoint_offsets(cu, n)
    assert R == 3 + 1 + 0 + 2
    worst = 0.0
    for i, L in enumerate(lengths):
        for j in range(-(-L // n)):
            m = j * n
            if m == 0:
                expect = S0[i]
            else:
                sl = slice(cu[i], cu[i] + m)
                pr = oracle.gdn_fwd(q[sl], k[sl], v[sl], g[sl], beta[sl], np.array([0, m]),
                                    initial_state=S0[i:i + 1], mutation=0)
                expect = pr["final_state"][0]
            worst = max(worst, _rel(r["checkpoints"][off[i] + j], expect))
    return worst


def check_round_trip(mutation=0):
    """Running [0, m) then [m, L) with final -> initial equals the unsplit run."""
    L, m = 13, 6
    q, k, v, g, beta, _, S0 = _rand_case([L], 1, 2, 4, 3, seed=61, s0=True, gscale=0.2)
    full = oracle.gdn_fwd(q, k, v, g, beta, np.array([0, L]), initial_state=S0, mutation=mutation)
    a = oracle.gdn_fwd(q[:m], k[:m], v[:m], g[:m], beta[:m], np.array([0, m]),
                       initial_state=S0, mutation=mutation)
    b = oracle.gdn_fwd(q[m:], k[m:], v[m:], g[m:], beta[m:], np.array([0, L - m]),
                       initial_state=a["final_state"], mutation=mutation)
    return max(_rel(b["final_state"], full["final_state"]), _rel(b["o"], full["o"][m:]),
               _rel(a["o"], full["o"][:m]))


def check_empty(mutation=0):
    """Empty sequences: final = initial, no checkpoint rows, transition = identity."""
    lengths = [0, 4, 0]
    q, k, v, g, beta, cu, S0 = _rand_case(lengths, 1, 1, 3, 2, seed=71, s0=True)
    r = oracle.gdn_fwd(q, k, v, g, beta, cu, initial_state=S0, checkpoint_every_n=2,
                       mutation=mutation)
    s = oracle.gdn_summary(k, v, g, beta, cu, mutation=mutation)
    off, R = oracle.checkpoint_offsets(cu, 2)
    assert R == 2 and list(off) == [0, 0, 2]
    return max(_rel(r["final_state"][0], S0[0]), _rel(r["final_state"][2], S0[2]),
               _rel(s["transition"][0, 0], np.eye(3)), _rel(s["transition"][2, 0], np.eye(3)),
               float(np.abs(s["end_state"][[0, 2]]).max()))


def check_gate_softplus(mutation=0):
    """Softplus gate -exp(a_log) softplus(g + dt_bias), with beta = 0 so only the decay acts.

    Head 0: a_log = 0, dt_bias = 0, g = 0 gives log decay -ln 2 per token (softplus(0) = ln 2).
    Head 1: a_log = ln 3, dt_bias = ln(e - 1), g = 0 gives -3 per token (softplus = ln e = 1).
    Head 2: a_log = -3, g = 50 checks the large-argument branch: softplus(50) = 50 + log1p(e^-50).
    Head 3: a_log = 0, dt_bias = -ln 3, g = 0 checks the negative branch: softplus(-ln 3) =
    ln(1 + 1/3) = ln(4/3), a decay of exactly 3/4 per token.
    Head 4: a_log = 0, g = -5: softplus(-5) = ln(1 + e^-5).
    The state after L tokens is exp(sum of log decays) S0, and the transition that factor times I.
    """
    L, K, V, H = 5, 3, 2, 5
    rng = np.random.default_rng(91)
    q = rng.standard_normal((L, 1, K))
    k = rng.standard_normal((L, 1, K))
    v = rng.standard_normal((L, H, V))
    S0 = rng.standard_normal((1, H, K, V))
    g_raw = np.zeros((L, H))
    g_raw[:, 2] = 50.0
    g_raw[:, 4] = -5.0
    a_log = np.array([0.0, math.log(3.0), -3.0, 0.0, 0.0])
    dt_bias = np.array([0.0, math.log(math.e - 1.0), 0.0, -math.log(3.0), 0.0])
    beta = np.zeros((L, H))
    cu = np.array([0, L])
    kw = dict(gate="softplus", a_log=a_log, dt_bias=dt_bias, mutation=mutation)
    r = oracle.gdn_fwd(q, k, v, g_raw, beta, cu, initial_state=S0, **kw)
    s = oracle.gdn_summary(k, v, g_raw, beta, cu, **kw)
    per_token = np.array([-math.log(2.0), -3.0, -math.exp(-3.0) * (50.0 + math.log1p(math.exp(-50.0))),
                          math.log(0.75), -math.log1p(math.exp(-5.0))])
    factor = np.exp(L * per_token)
    errs = [_rel(r["final_state"][0, h], factor[h] * S0[0, h]) for h in range(H)]
    errs += [_rel(s["transition"][0, h], factor[h] * np.eye(K)) for h in range(H)]
    return max(errs)


def check_gate_sigmoid_bound(mutation=0):
    """Bounded gate lower_bound * sigmoid(g) with lower_bound = -2 ln 2 and beta = 0:
    g = 0 gives sigmoid 1/2, a decay of exactly 1/2 per token; g = ln 3 gives sigmoid 3/4,
    a decay of 2^-1.5; g = -ln 3 (the negative branch) gives sigmoid 1/4, a decay of 2^-0.5."""
    L, K, V = 4, 2, 3
    rng = np.random.default_rng(92)
    q = rng.standard_normal((L, 1, K))
    k = rng.standard_normal((L, 1, K))
    v = rng.standard_normal((L, 3, V))
    S0 = rng.standard_normal((1, 3, K, V))
    g_raw = np.zeros((L, 3))
    g_raw[:, 1] = math.log(3.0)
    g_raw[:, 2] = -math.log(3.0)
    beta = np.zeros((L, 3))
    r = oracle.gdn_fwd(q, k, v, g_raw, beta, np.array([0, L]), initial_state=S0, gate="sigmoid_bound",
                       gate_lower_bound=-2.0 * math.log(2.0), mutation=mutation)
    return max(_rel(r["final_state"][0, 0], 0.5 ** L * S0[0, 0]),
               _rel(r["final_state"][0, 1], 2.0 ** (-1.5 * L) * S0[0, 1]),
               _rel(r["final_state"][0, 2], 2.0 ** (-0.5 * L) * S0[0, 2]))


def check_beta_sigmoid(mutation=0):
    """beta given as logits: beta_raw = ln 3 is beta = 3/4 (head 0) and beta_raw = -ln 3, the
    negative branch, is beta = 1/4 (head 1).  One token from a zero start with k = q = e_0, no
    norm, scale 1: S_1 = beta e_0 v^T and o_0 = beta v."""
    K, V = 3, 2
    k = np.zeros((1, 1, K))
    k[0, 0, 0] = 1.0
    v = np.array([[[1.0, -2.0], [3.0, 0.5]]])
    g = np.array([[-0.3, -0.7]])
    beta_raw = np.array([[math.log(3.0), -math.log(3.0)]])
    r = oracle.gdn_fwd(k, k, v, g, beta_raw, np.array([0, 1]), scale=1.0, use_qk_l2norm=False,
                       beta_sigmoid=True, mutation=mutation)
    errs = []
    for h, b in ((0, 0.75), (1, 0.25)):
        expect_S = np.zeros((K, V))
        expect_S[0] = b * v[0, h]
        errs += [_rel(r["o"][0, h], b * v[0, h]), _rel(r["final_state"][0, h], expect_S)]
    return max(errs)


def check_state_pool(mutation=0):
    """Decode from a state pool: N sequences of one token each start from pool[state_indices[i]]
    and write back there.  Each update is checked against the explicit one-token form
    S' = e^g (I - beta k k^T) S + beta k v^T, o = scale S'^T q (no norm), and the slots that
    no sequence names must come back unchanged."""
    rng = np.random.default_rng(97)
    N, P, HV, K, V = 3, 5, 2, 4, 3
    idx = np.array([3, 0, 4])
    q = rng.standard_normal((N, 1, K))
    k = rng.standard_normal((N, 1, K))
    v = rng.standard_normal((N, HV, V))
    g = -0.1 * rng.random((N, HV))
    beta = rng.random((N, HV))
    pool = rng.standard_normal((P, HV, K, V))
    r = oracle.gdn_fwd(q, k, v, g, beta, np.arange(N + 1), scale=0.7, use_qk_l2norm=False,
                       initial_state=pool, state_indices=idx, mutation=mutation)
    errs = []
    for i in range(N):
        for h in range(HV):
            kk = k[i, 0]
            S1 = math.exp(g[i, h]) * (np.eye(K) - beta[i, h] * np.outer(kk, kk)) @ pool[idx[i], h] \
                + beta[i, h] * np.outer(kk, v[i, h])
            errs.append(_rel(r["state_pool"][idx[i], h], S1))
            errs.append(_rel(r["o"][i, h], 0.7 * S1.T @ q[i, 0]))
    errs.append(float(np.abs(r["state_pool"][[1, 2]] - pool[[1, 2]]).max()))
    return max(errs)


def _fd_case(l2norm, seed):
    rng = np.random.default_rng(seed)
    lengths = [4, 5]
    T, HK, HV, K, V = sum(lengths), 1, 2, 3, 2
    cu = np.array([0, 4, 9])
    q = rng.standard_normal((T, HK, K))
    k = rng.standard_normal((T, HK, K))
    v = rng.standard_normal((T, HV, V))
    g = -0.3 * rng.random((T, HV))
    beta = rng.random((T, HV))
    S0 = 0.5 * rng.standard_normal((2, HV, K, V))
    do = rng.standard_normal((T, HV, V))
    dfin = rng.standard_normal((2, HV, K, V))
    return dict(q=q, k=k, v=v, g=g, beta=beta, S0=S0), cu, do, dfin, l2norm


def check_backward_finite_differences(mutation=0):
    """Every gradient of L = sum(do * o) + sum(dS_T * S_final) against central differences of
    the (pinned) forward, with and without the L2 norm, grouped heads and a start state."""
    worst = 0.0
    names = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta": "dbeta", "S0": "d_initial_state"}
    for l2norm, seed in ((True, 101), (False, 102)):
        x, cu, do, dfin, l2 = _fd_case(l2norm, seed)

        def loss(xx):
            r = oracle.gdn_fwd(xx["q"], xx["k"], xx["v"], xx["g"], xx["beta"], cu, scale=0.8, use_qk_l2norm=l2,
                               initial_state=xx["S0"], nthreads=1)
            return float((r["o"] * do).sum() + (r["final_state"] * dfin).sum())

        grads = oracle.gdn_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, do, scale=0.8, use_qk_l2norm=l2,
                               initial_state=x["S0"], d_final_state=dfin, nthreads=1, mutation=mutation)
        eps = 1e-6
        for name, gname in names.items():
            fd = np.zeros_like(x[name])
            for idx in np.ndindex(x[name].shape):
                xp = {kk: vv.copy() for kk, vv in x.items()}
                xm = {kk: vv.copy() for kk, vv in x.items()}
                xp[name][idx] += eps
                xm[name][idx] -= eps
                fd[idx] = (loss(xp) - loss(xm)) / (2 * eps)
            worst = max(worst, _rel(grads[gname], fd))
    return worst


def check_backward_transforms_finite_differences(mutation=0):
    """The backward through the input transforms (softplus gate with a_log and dt_bias, bounded
    sigmoid gate, beta sigmoid) against central differences of the (pinned) forward with the same
    transforms: the raw gate and beta inputs, a_log and dt_bias."""
    worst = 0.0
    x, cu, do, dfin, l2 = _fd_case(True, 141)
    rng = np.random.default_rng(142)
    HV = x["g"].shape[1]
    x["g"] = rng.standard_normal(x["g"].shape)          # raw gate inputs
    x["beta"] = rng.standard_normal(x["beta"].shape)    # beta logits
    x["a_log"] = 0.3 * rng.standard_normal(HV)
    x["dt_bias"] = 0.5 * rng.standard_normal(HV)
    for kw, names in ((dict(gate="softplus", beta_sigmoid=True), ("g", "beta", "a_log", "dt_bias")),
                      (dict(gate="sigmoid_bound", gate_lower_bound=-2.5), ("g",))):
        def fw(xx):
            extra = dict(kw)
            if kw["gate"] == "softplus":
                extra.update(a_log=xx["a_log"], dt_bias=xx["dt_bias"])
            return extra

        def loss(xx):
            r = oracle.gdn_fwd(xx["q"], xx["k"], xx["v"], xx["g"], xx["beta"], cu, scale=0.8, use_qk_l2norm=l2,
                               initial_state=xx["S0"], nthreads=1, **fw(xx))
            return float((r["o"] * do).sum() + (r["final_state"] * dfin).sum())

        grads = oracle.gdn_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, do, scale=0.8, use_qk_l2norm=l2,
                               initial_state=x["S0"], d_final_state=dfin, nthreads=1, mutation=mutation, **fw(x))
        gname = {"g": "dg", "beta": "dbeta", "a_log": "d_a_log", "dt_bias": "d_dt_bias"}
        eps = 1e-6
        for name in names:
            fd = np.zeros_like(x[name])
            for idx in np.ndindex(x[name].shape):
                xp = {kk: vv.copy() for kk, vv in x.items()}
                xm = {kk: vv.copy() for kk, vv in x.items()}
                xp[name][idx] += eps
                xm[name][idx] -= eps
                fd[idx] = (loss(xp) - loss(xm)) / (2 * eps)
            worst = max(worst, _rel(grads[gname[name]], fd))
    return worst


def check_gdp_dense_products(mutation=0):
    """GDP against its definition written as dense products: per token, S_t = exp(g_t) H_t S_{t-1}
    + sum_j (prod_{i > j} (I - beta_i k_i k_i^T)) beta_j k_j v_j^T with H_t the product of the
    token's n Householder-like factors (later updates on the left); o_t = scale S_t^T q_t.
    Also num_householder = 1 against gdn_fwd."""
    rng = np.random.default_rng(111)
    n, lengths, HK, HV, K, V = 3, [4, 2], 1, 2, 3, 2
    T = sum(lengths)
    cu = np.array([0, 4, 6])
    q = rng.standard_normal((T, HK, K))
    k = rng.standard_normal((T * n, HK, K))
    v = rng.standard_normal((T * n, HV, V))
    g = -0.4 * rng.random((T, HV))
    beta = rng.random((T * n, HV))
    S0 = rng.standard_normal((2, HV, K, V))
    r = oracle.gdp_fwd(q, k, v, g, beta, cu, n, scale=0.9, use_qk_l2norm=True, initial_state=S0, mutation=mutation)
    worst = 0.0
    for i in range(2):
        for h in range(HV):
            S = S0[i, h].copy()
            for t in range(cu[i], cu[i + 1]):
                H = np.eye(K)
                add = np.zeros((K, V))
                for j in range(n):
                    kk = k[t * n + j, 0] / np.sqrt((k[t * n + j, 0] ** 2).sum() + 1e-6)
                    F = np.eye(K) - beta[t * n + j, h] * np.outer(kk, kk)
                    H = F @ H
                    add = F @ add + beta[t * n + j, h] * np.outer(kk, v[t * n + j, h])
                S = math.exp(g[t, h]) * H @ S + add
                qq = q[t, 0] / np.sqrt((q[t, 0] ** 2).sum() + 1e-6)
                worst = max(worst, _rel(r["o"][t, h], 0.9 * S.T @ qq))
            worst = max(worst, _rel(r["final_state"][i, h], S))
    # n = 1 is GDN
    k1, v1, b1 = k[::n], v[::n], beta[::n]
    r1 = oracle.gdp_fwd(q, k1, v1, g, b1, cu, 1, initial_state=S0, mutation=mutation)
    f1 = oracle.gdn_fwd(q, k1, v1, g, b1, cu, initial_state=S0)
    worst = max(worst, _rel(r1["o"], f1["o"]), _rel(r1["final_state"], f1["final_state"]))
    return worst


def check_summary_bwd(mutation=0):
    """The summary's state-gradient mirror against (1) the entering-state gradient of the
    (finite-difference pinned) backward, with and without a final-state cotangent, grouped heads,
    the L2 norm on and off and an empty sequence; (2) the closed form with beta = 0,
    G = exp(b_L) dS_exit + sum_t exp(b_t) scale q_t do_t^T (b_t the cumulative gate from the span
    start); (3) span composition: the whole sequence's gradient equals the per-span gradients
    composed right to left with the summary's transitions, d_enter = transition d_exit + (the
    span's own value)."""
    worst = 0.0
    rng = np.random.default_rng(121)
    cu = np.array([0, 5, 5, 12])
    T, HK, HV, K, V = 12, 1, 2, 3, 4
    q = rng.standard_normal((T, HK, K))
    k = rng.standard_normal((T, HK, K))
    v = rng.standard_normal((T, HV, V))
    g = -0.4 * rng.random((T, HV))
    beta = rng.random((T, HV))
    do = rng.standard_normal((T, HV, V))
    S0 = rng.standard_normal((3, HV, K, V))
    dfin = rng.standard_normal((3, HV, K, V))
    for l2 in (True, False):
        for df in (None, dfin):
            ref = oracle.gdn_bwd(q, k, v, g, beta, cu, do, scale=0.7, use_qk_l2norm=l2, initial_state=S0,
                                 d_final_state=df, nthreads=1)["d_initial_state"]
            got = oracle.gdn_summary_bwd(q, k, g, beta, cu, do, scale=0.7, use_qk_l2norm=l2, d_final_state=df,
                                         mutation=mutation)
            worst = max(worst, _rel(got, ref))
    # (2) beta = 0 closed form (no L2 norm)
    b0 = np.zeros_like(beta)
    got = oracle.gdn_summary_bwd(q, k, g, b0, cu, do, scale=0.7, use_qk_l2norm=False, d_final_state=dfin,
                                 mutation=mutation)
    for i in range(3):
        for h in range(HV):
            s_, e_ = cu[i], cu[i + 1]
            G = np.exp(g[s_:e_, h].sum()) * dfin[i, h]
            for t in range(s_, e_):
                G = G + np.exp(g[s_:t + 1, h].sum()) * 0.7 * np.outer(q[t, h // (HV // HK)], do[t, h])
            worst = max(worst, _rel(got[i, h], G))
    # (3) span composition of the state gradient
    L = 11
    whole = np.array([0, L])
    spans = np.array([0, 4, 7, L])
    qs, ks, gs, bs, ds = q[:L], k[:L], g[:L], beta[:L], do[:L]
    dF = dfin[:1]
    full = oracle.gdn_summary_bwd(qs, ks, gs, bs, whole, ds, scale=0.7, d_final_state=dF, mutation=mutation)
    loc = oracle.gdn_summary_bwd(qs, ks, gs, bs, spans, ds, scale=0.7, mutation=mutation)
    trs = oracle.gdn_summary(ks, v[:L], gs, bs, spans)["transition"]
    d = oracle.compose_span_grads(trs, loc, dF[0], mutation=mutation)[-1]
    return max(worst, _rel(d, full[0]))


def check_summary_bwd_finite_differences(mutation=0):
    """The summary's state-gradient mirror against central differences of the (pinned) forward's
    loss sum(do * o) + sum(dS_T * S_final) in the start state."""
    x, cu, do, dfin, l2 = _fd_case(True, 131)
    got = oracle.gdn_summary_bwd(x["q"], x["k"], x["g"], x["beta"], cu, do, scale=0.8, use_qk_l2norm=l2,
                                 d_final_state=dfin, mutation=mutation)

    def loss(S0):
        r = oracle.gdn_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, scale=0.8, use_qk_l2norm=l2,
                           initial_state=S0, nthreads=1)
        return float((r["o"] * do).sum() + (r["final_state"] * dfin).sum())

    eps = 1e-6
    fd = np.zeros_like(x["S0"])
    for idx in np.ndindex(x["S0"].shape):
        sp, sm = x["S0"].copy(), x["S0"].copy()
        sp[idx] += eps
        sm[idx] -= eps
        fd[idx] = (loss(sp) - loss(sm)) / (2 * eps)
    return _rel(got, fd)


CHECKS = {
    "golden": (check_golden, 1e-12),
    "brute_force": (check_brute_force, 1e-12),
    "retrieval": (check_retrieval, 1e-12),
    "pure_decay": (check_pure_decay, 1e-12),
    "single_token": (check_single_token, 1e-12),
    "linearity": (check_linearity, 1e-10),
    "norm_invariance": (check_norm_invariance, 2e-5),
    "gva": (check_gva, 1e-13),
    "span_composition": (check_span_composition, 1e-12),
    "checkpoints": (check_checkpoints, 1e-13),
    "round_trip": (check_round_trip, 1e-12),
    "empty": (check_empty, 1e-15),
    "gate_softplus": (check_gate_softplus, 1e-12),
    "gate_sigmoid_bound": (check_gate_sigmoid_bound, 1e-12),
    "beta_sigmoid": (check_beta_sigmoid, 1e-14),
    "state_pool": (check_state_pool, 1e-13),
    "backward_finite_differences": (check_backward_finite_differences, 1e-6),
    "backward_transforms_finite_differences": (check_backward_transforms_finite_differences, 1e-6),
    "gdp_dense_products": (check_gdp_dense_products, 1e-12),
    "summary_bwd": (check_summary_bwd, 1e-12),
    "summary_bwd_finite_differences": (check_summary_bwd_finite_differences, 1e-6),
}


@pytest.mark.parametrize("name", sorted(CHECKS))
def test_oracle_pin(name):
    fn, tol = CHECKS[name]
    err = fn(0)
    assert err <= tol, f"{name}: relative error {err:.3e} > {tol:.1e}"


@pytest.mark.parametrize("mutation", sorted(oracle.MUTATIONS))
def test_planted_mistakes_are_caught(mutation):
    failed = []
    for name, (fn, tol) in CHECKS.items():
        try:
            err = fn(mutation)
        except (AssertionError, ValueError):
            err = float("inf")
        if not err <= tol:
            failed.append(name)
    assert failed, f"planted mistake '{oracle.MUTATIONS[mutation]}' passed every pin"


def test_retrieval_with_l2norm_close():
    """With the L2 norm on, unit keys are rescaled by 1/sqrt(1 + 1e-6): retrieval holds to ~1e-6."""
    K = V = 4
    k = np.eye(K)[[0, 1, 2, 1]][:, None, :]
    v = np.random.default_rng(9).standard_normal((4, 1, V))
    r = oracle.gdn_fwd(k, k, v, np.zeros((4, 1)), np.ones((4, 1)), np.array([0, 4]), scale=1.0)
    assert _rel(r["o"][:, 0], v[:, 0]) < 2e-6


def test_unit_mask_computes_only_marked_units():
    q, k, v, g, beta, cu, S0 = _rand_case([4, 5], 1, 2, 3, 2, seed=81, s0=True)
    full = oracle.gdn_fwd(q, k, v, g, beta, cu, initial_state=S0)
    mask = np.array([[False, True], [True, False]])
    part = oracle.gdn_fwd(q, k, v, g, beta, cu, initial_state=S0, unit_mask=mask)
    assert np.array_equal(part["final_state"][0, 1], full["final_state"][0, 1])
    assert np.array_equal(part["final_state"][1, 0], full["final_state"][1, 0])
    assert not part["final_state"][0, 0].any()


def test_rejects_bad_cu_seqlens():
    q, k, v, g, beta, cu, _ = _rand_case([3, 2], 1, 1, 2, 2, seed=91)
    with pytest.raises(ValueError):
        oracle.gdn_fwd(q, k, v, g, beta, np.array([0, 4, 3]))
