"""Parity oracle -- TEST INFRASTRUCTURE ONLY.

A plain fp64 CPU restatement of the Gated DeltaNet forward (``gdn_fwd``), of
the span summary (``gdn_summary``), of the forward's backward (``gdn_bwd``,
reverse-mode differentiation of the token recurrence) and of the summary's
state-gradient mirror (``gdn_summary_bwd``), following the cuDNN "Linear Attention"
operations page (sections "Layout", "Semantics worth knowing" and "Summaries").  The
arithmetic lives in ``gdn_oracle.c`` (token-by-token recurrence, fp64); this
module only compiles it with gcc, converts inputs to fp64 and marshals
arguments.  The optional in-kernel input transforms of cudnn-frontend PR #616
(the softplus gate -exp(a_log) softplus(g + dt_bias), the bounded gate
lower_bound * sigmoid(g), and beta = sigmoid(beta)) are applied here in fp64
before the recurrence.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does, and this
package imports nothing from the library: the two share no code.

``compose_spans`` / ``compose_span_grads`` restate the page's composition of span summaries
(numpy products, fp64); they serve the context-parallel tests.

Parity pins: every entry point is pinned in ``tests/test_oracle_pins.py``
(brute-force dense products, closed forms, linearity, span composition,
hand-derived golden values in ``tests/golden/``; the backward against central
finite differences of the forward).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None

# planted mistakes understood by gdn_oracle.c (0 = the correct oracle)
MUTATIONS = {
    1: "decay dropped",
    2: "erase sign flipped",
    3: "erase term dropped",
    4: "exclusive output (reads the previous state)",
    5: "L2 norm without the square root",
    6: "interleaved grouped-head mapping",
    7: "transition stored untransposed",
    8: "checkpoints taken one token late",
    # planted in the gate / beta transforms below (applied before the C recurrence)
    9: "softplus gate without dt_bias",
    10: "softplus gate rate a_log instead of exp(a_log)",
    11: "beta sigmoid of the negated logit",
    12: "bounded gate without the sigmoid",
    13: "state pool written back to slot i instead of state_indices[i]",
    16: "GDP: decay applied before every update instead of once per token",
    17: "GDP: output read after the first update of the token instead of the last",
    # planted in the backward
    14: "backward: decay gradient misses the erase path (uses dS instead of dS')",
    15: "backward: key gradient misses the S' dx term",
    18: "summary backward: a token's output term added after its erase step instead of before",
    19: "backward of the softplus gate: d_dt_bias without the sigmoid factor",
    20: "backward of the beta sigmoid: the logit gradient scaled by beta instead of beta (1 - beta)",
    # planted in the negative-argument branches of the two scalar functions below
    21: "sigmoid at x < 0 evaluated as 1 / (1 + e^x), the positive branch's formula",
    22: "softplus at x < 0 evaluated as x + log1p(e^-|x|), dropping the max(x, 0)",
    # planted in the span composition below
    23: "span composition applies the transition untransposed",
    24: "backward span composition adds the span's own gradient after moving through the span",
}


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c into oracle/_build/libgdn_oracle.so (plain gcc, -O2)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            d = ctypes.POINTER(ctypes.c_double)
            i64 = ctypes.POINTER(ctypes.c_int64)
            lib.gdn_oracle_run.restype = ctypes.c_int
            lib.gdn_oracle_run.argtypes = [
                d, d, d, d, d, i64,
                ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_double, ctypes.c_int, d,
                d, d,
                d, ctypes.c_int64, i64,
                d, ctypes.c_void_p,
                ctypes.c_int, ctypes.c_int,
            ]
            lib.gdn_oracle_bwd.restype = ctypes.c_int
            lib.gdn_oracle_bwd.argtypes = [
                d, d, d, d, d, i64,
                ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_double, ctypes.c_int, d,
                d, d,
                d, d, d, d, d, d,
                ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
            ]
            _lib = lib
    return _lib


def _f64(x):
    """Exact conversion of a torch tensor (bf16/fp32) or array to contiguous fp64."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().float().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i64(x):
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int64))


def _ptr(a, ctype=ctypes.c_double):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def checkpoint_offsets(cu_seqlens, n: int):
    """First checkpoint row of each sequence and the total row count.

    A sequence of length L owns ceil(L / n) rows: the states entering token
    offsets 0, n, 2n, ... < L (cuDNN page, "States and checkpoints").
    """
    cu = _i64(cu_seqlens)
    lens = np.diff(cu)
    rows = (lens + n - 1) // n
    off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)
    return off[:-1].copy(), int(off[-1])


def _default_threads():
    return max(1, os.cpu_count() or 1)


def softplus(x, mutation=0):
    """log(1 + e^x) in fp64, evaluated as max(x, 0) + log1p(e^-|x|) so it never overflows."""
    x = np.asarray(x, dtype=np.float64)
    head = x if mutation == 22 else np.maximum(x, 0.0)
    return head + np.log1p(np.exp(-np.abs(x)))


def sigmoid(x, mutation=0):
    """1 / (1 + e^-x) in fp64, evaluated without overflow for either sign of x: with
    e = e^-|x|, 1 / (1 + e) for x >= 0 and e / (1 + e) = 1 / (1 + e^-x) for x < 0."""
    x = np.asarray(x, dtype=np.float64)
    e = np.exp(-np.abs(x))
    neg = 1.0 / (1.0 + e) if mutation == 21 else e / (1.0 + e)
    return np.where(x >= 0, 1.0 / (1.0 + e), neg)


def gate_transform(g, *, gate="log", a_log=None, dt_bias=None, gate_lower_bound=None, mutation=0):
    """Per-token log decay from the raw gate input (cudnn-frontend PR #616, in-kernel gate fusion).

    gate="log":           g is already the natural-log decay.
    gate="softplus":      g[t,h] = -exp(a_log[h]) * softplus(g_raw[t,h] + dt_bias[h])   (a_log, dt_bias: [HO]).
    gate="sigmoid_bound": g[t,h] = gate_lower_bound * sigmoid(g_raw[t,h]): a log decay bounded
                          below by the (negative) lower bound.
    """
    g = _f64(g)
    if gate == "log":
        return g
    if gate == "softplus":
        a = _f64(a_log).reshape(1, -1)
        dt = _f64(dt_bias).reshape(1, -1)
        rate = a if mutation == 10 else np.exp(a)
        return -rate * softplus(g if mutation == 9 else g + dt, mutation)
    if gate == "sigmoid_bound":
        lb = float(gate_lower_bound)
        return lb * (g if mutation == 12 else sigmoid(g, mutation))
    raise ValueError(f"unknown gate mode {gate!r}")


def beta_transform(beta, *, beta_sigmoid=False, mutation=0):
    """beta, or sigmoid(beta) when the logits are given (PR #616, in-kernel beta sigmoid)."""
    beta = _f64(beta)
    if not beta_sigmoid:
        return beta
    return sigmoid(-beta if mutation == 11 else beta, mutation)


def gdn_fwd(q, k, v, g, beta, cu_seqlens, *, scale=None, use_qk_l2norm=True,
            initial_state=None, output_final_state=True, checkpoint_every_n=0,
            want_o=True, unit_mask=None, nthreads=None, mutation=0,
            gate="log", a_log=None, dt_bias=None, gate_lower_bound=None, beta_sigmoid=False,
            state_indices=None):
    """fp64 forward: returns dict(o [T,HO,V], final_state [N,HO,K,V], checkpoints [R,HO,K,V]).

    q, k: [T, HK, K]; v: [T, HV, V]; g, beta: [T, HO] (g in natural-log space unless a gate
    transform is named; beta the logits when beta_sigmoid); cu_seqlens: [N + 1];
    initial_state: [N, HO, K, V] or None (zero start).
    scale defaults to 1/sqrt(K) and multiplies the (normalised) query.
    unit_mask: optional bool [N, HO]; unmarked units are left at zero.

    state_indices ([N] ints; cuDNN page, "States and checkpoints"): initial_state is then a
    pool [N_pool, HO, K, V]; sequence i starts from pool[state_indices[i]] and its end state
    is written back to that slot.  The result then also holds "state_pool", the pool after
    the write-back (untouched slots unchanged).  Exclusive with checkpoints.
    """
    g = gate_transform(g, gate=gate, a_log=a_log, dt_bias=dt_bias, gate_lower_bound=gate_lower_bound,
                       mutation=mutation)
    beta = beta_transform(beta, beta_sigmoid=beta_sigmoid, mutation=mutation)
    pool = idx = None
    if state_indices is not None:
        if checkpoint_every_n:
            raise ValueError("state_indices and checkpoints are exclusive")
        pool = _f64(initial_state)
        idx = _i64(state_indices)
        if idx.shape != (_i64(cu_seqlens).shape[0] - 1,) or (idx < 0).any() or (idx >= pool.shape[0]).any():
            raise ValueError("state_indices must hold one slot in [0, N_pool) per sequence")
        initial_state = pool[idx]
        output_final_state = True
    r = _run(q, k, v, g, beta, cu_seqlens, scale=scale, use_qk_l2norm=use_qk_l2norm,
             s0=initial_state, want_final=output_final_state,
             checkpoint_every_n=checkpoint_every_n, want_o=want_o,
             want_transition=False, unit_mask=unit_mask, nthreads=nthreads,
             mutation=mutation if mutation < 9 else 0)
    if pool is not None:
        out = pool.copy()
        dst = np.arange(idx.shape[0]) if mutation == 13 else idx
        out[dst] = r["final_state"]
        r["state_pool"] = out
    return r


def gdp_fwd(q, k, v, g, beta, cu_seqlens, num_householder, *, scale=None, use_qk_l2norm=True,
            initial_state=None, checkpoint_every_n=0, unit_mask=None, nthreads=None, mutation=0):
    """Gated DeltaProduct forward (cuDNN Linear Attention page: GDP runs on two timelines).

    q: [T, HK, K] and g: [T, HO] have one row per token; k: [T*n, HK, K], v: [T*n, HV, V] and
    beta: [T*n, HO] have n rows per token, update-major (token t's updates are rows t*n .. t*n+n-1).
    Per token t: S <- exp(g_t) S, then for j = 0 .. n-1 the delta step
    S <- S + beta_{t,j} k_{t,j} (v_{t,j} - S^T k_{t,j})^T, then o_t = scale S^T q_t.
    num_householder == 1 is exactly gdn_fwd.  Written as that recurrence on the update timeline:
    the gate enters at each token's first update (exp(0) = 1 at the others) and the query at its
    last (the outputs at the other updates are not part of the result).
    Checkpoints every n tokens: the states entering tokens 0, n, 2n, ... of each sequence.
    """
    n = int(num_householder)
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    cu = _i64(cu_seqlens)
    T, HK, K = q.shape
    HO = g.shape[1]
    assert k.shape[0] == T * n and v.shape[0] == T * n and beta.shape[0] == T * n
    ge = np.zeros((T * n, HO))
    ge[0::n] = g
    if mutation == 16:
        ge[:] = np.repeat(g, n, axis=0)
    qe = np.zeros((T * n, HK, K))
    qe[(n - 1 if mutation != 17 else 0)::n] = q
    if scale is None:
        scale = 1.0 / np.sqrt(K)
    r = _run(qe, k, v, ge, beta, cu * n, scale=scale, use_qk_l2norm=use_qk_l2norm, s0=initial_state,
             want_final=True, checkpoint_every_n=checkpoint_every_n * n, want_o=True, want_transition=False,
             unit_mask=unit_mask, nthreads=nthreads, mutation=0)
    r["o"] = r["o"][(n - 1 if mutation != 17 else 0)::n]
    return r


def gdn_bwd(q, k, v, g, beta, cu_seqlens, do, *, scale=None, use_qk_l2norm=True, initial_state=None,
            d_final_state=None, unit_mask=None, nthreads=None, mutation=0,
            gate="log", a_log=None, dt_bias=None, gate_lower_bound=None, beta_sigmoid=False):
    """fp64 backward of gdn_fwd by reverse-mode differentiation of the token recurrence: the
    gradients of L = sum(do * o) + sum(d_final_state * S_final).

    Returns dict(dq [T,HK,K], dk [T,HK,K], dv [T,HV,V], dg [T,HO], dbeta [T,HO],
    d_initial_state [N,HO,K,V]).  Grouped heads: dq, dk sum the contributions of every value
    head of the group.  With the input transforms of gdn_fwd, dg and dbeta are the gradients of
    the raw inputs (the chain rule through the transform, applied to the gradients of the
    recurrence's log decay and beta), and the softplus gate adds d_a_log, d_dt_bias [HO]:
    with z = g_raw + dt_bias and A = -exp(a_log), g = A softplus(z) gives dg_raw = dg A sigmoid(z),
    d_dt_bias = sum_t dg_raw and d_a_log = sum_t dg g (since dg/da_log = g); the bounded gate
    g = lb sigmoid(x) gives dx = dg lb sigmoid(x) (1 - sigmoid(x)); beta = sigmoid(y) gives
    dy = dbeta beta (1 - beta).
    """
    g_raw, beta_raw = _f64(g), _f64(beta)
    g = gate_transform(g_raw, gate=gate, a_log=a_log, dt_bias=dt_bias, gate_lower_bound=gate_lower_bound)
    beta = beta_transform(beta_raw, beta_sigmoid=beta_sigmoid)
    q, k, v, do = (_f64(x) for x in (q, k, v, do))
    cu = _i64(cu_seqlens)
    T, HK, K = k.shape
    HV, V = v.shape[1], v.shape[2]
    N = cu.shape[0] - 1
    HO = HV
    if scale is None:
        scale = 1.0 / np.sqrt(K)
    s0 = _f64(initial_state)
    dfin = _f64(d_final_state)
    dqh = np.zeros((T, HO, K))
    dkh = np.zeros((T, HO, K))
    dv = np.zeros((T, HV, V))
    dg = np.zeros((T, HO))
    db = np.zeros((T, HO))
    ds0 = np.zeros((N, HO, K, V))
    mask = None
    if unit_mask is not None:
        mask = np.ascontiguousarray(np.asarray(unit_mask, dtype=np.uint8).reshape(N * HO))
    rc = _load().gdn_oracle_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu, ctypes.c_int64),
        T, N, HK, HV, K, V, float(scale), int(bool(use_qk_l2norm)), _ptr(s0),
        _ptr(do), _ptr(dfin),
        _ptr(dqh), _ptr(dkh), _ptr(dv), _ptr(dg), _ptr(db), _ptr(ds0),
        mask.ctypes.data if mask is not None else None, int(nthreads or _default_threads()),
        int(mutation if mutation < 19 else 0))
    if rc != 0:
        raise ValueError("oracle rejected its arguments (cu_seqlens or shapes)")
    grp = HV // HK
    dq = dqh.reshape(T, HK, grp, K).sum(axis=2)
    dk = dkh.reshape(T, HK, grp, K).sum(axis=2)
    out = {"dq": dq, "dk": dk, "dv": dv, "dg": dg, "dbeta": db, "d_initial_state": ds0}
    if gate == "softplus":
        z = g_raw + _f64(dt_bias).reshape(1, -1)
        A = -np.exp(_f64(a_log)).reshape(1, -1)
        dg_raw = dg * A * (1.0 if mutation == 19 else sigmoid(z))
        out["d_a_log"] = (dg * g).sum(axis=0)
        out["d_dt_bias"] = dg_raw.sum(axis=0)
        out["dg"] = dg_raw
    elif gate == "sigmoid_bound":
        sx = sigmoid(g_raw)
        out["dg"] = dg * float(gate_lower_bound) * sx * (1.0 - sx)
    if beta_sigmoid:
        out["dbeta"] = db * (beta if mutation == 20 else beta * (1.0 - beta))
    return out


def gdn_summary_bwd(q, k, g, beta, cu_seqlens, do, *, scale=None, use_qk_l2norm=True, d_final_state=None,
                    mutation=0, gate="log", a_log=None, dt_bias=None, gate_lower_bound=None, beta_sigmoid=False):
    """fp64 state-gradient counterpart of the summary (cuDNN Linear Attention page, "Summaries":
    each summary op has a backward partner acting on the state gradient).  For each span (sequence) and output
    head: the gradient of L = sum(do * o) + sum(d_final_state * S_end) with respect to the state
    entering the span, [N, HO, K, V].

    Walking the span backwards with G the gradient with respect to the state after token t:
    G <- G + scale q_t do_t^T (from o_t = scale S_t^T q_t), then G <- exp(g_t)(I - beta_t k_t k_t^T) G,
    the transposed Jacobian of S_t = exp(g_t)(I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
    (the factor is symmetric).  G after the span's first token is the result; it involves neither
    v nor any state value.  q, k are L2-normalised first when use_qk_l2norm is set; the input
    transforms of gdn_fwd apply to g and beta as there.
    """
    g = gate_transform(g, gate=gate, a_log=a_log, dt_bias=dt_bias, gate_lower_bound=gate_lower_bound)
    beta = beta_transform(beta, beta_sigmoid=beta_sigmoid)
    q, k, g, beta, do = (_f64(x) for x in (q, k, g, beta, do))
    cu = _i64(cu_seqlens)
    T, HK, K = k.shape
    HO, V = do.shape[1], do.shape[2]
    N = cu.shape[0] - 1
    grp = HO // HK
    if scale is None:
        scale = 1.0 / np.sqrt(K)
    if use_qk_l2norm:
        q = q / np.sqrt((q * q).sum(axis=-1, keepdims=True) + 1e-6)
        k = k / np.sqrt((k * k).sum(axis=-1, keepdims=True) + 1e-6)
    out = np.zeros((N, HO, K, V))
    if d_final_state is not None:
        out[:] = _f64(d_final_state)
    for i in range(N):
        G = out[i].copy()
        for t in range(int(cu[i + 1]) - 1, int(cu[i]) - 1, -1):
            qh = np.repeat(q[t], grp, axis=0)  # [HO, K]: head h reads q/k head h // grp
            kh = np.repeat(k[t], grp, axis=0)
            out_term = scale * qh[:, :, None] * do[t][:, None, :]
            if mutation != 18:
                G = G + out_term
            kG = np.einsum("hk,hkv->hv", kh, G)
            G = np.exp(g[t])[:, None, None] * (G - beta[t][:, None, None] * kh[:, :, None] * kG[:, None, :])
            if mutation == 18:
                G = G + out_term
        out[i] = G
    return out


def gdn_summary(k, v, g, beta, cu_seqlens, *, use_qk_l2norm=True, start_state=None,
                unit_mask=None, nthreads=None, mutation=0,
                gate="log", a_log=None, dt_bias=None, gate_lower_bound=None, beta_sigmoid=False):
    """fp64 span summary: returns dict(end_state [N,HO,K,V], transition [N,HO,K,K]).

    end_state is the state after each span's last token from ``start_state``
    (zero when None); transition = P^T with P the product of the span's decayed
    erase steps exp(g_t)(I - beta_t k_t k_t^T), later steps on the left, so that
    end_state = einsum('ab,av->bv', transition, S_init) + S_H.
    """
    g = gate_transform(g, gate=gate, a_log=a_log, dt_bias=dt_bias, gate_lower_bound=gate_lower_bound,
                       mutation=mutation)
    beta = beta_transform(beta, beta_sigmoid=beta_sigmoid, mutation=mutation)
    mutation = mutation if mutation < 9 else 0
    T = k.shape[0]
    HK, K = k.shape[1], k.shape[2]
    q = np.zeros((T, HK, K), dtype=np.float64)
    r = _run(q, k, v, g, beta, cu_seqlens, scale=1.0, use_qk_l2norm=use_qk_l2norm,
             s0=start_state, want_final=True, checkpoint_every_n=0, want_o=False,
             want_transition=True, unit_mask=unit_mask, nthreads=nthreads,
             mutation=mutation)
    return {"end_state": r["final_state"], "transition": r["transition"]}


def compose_spans(transitions, end_states, start, mutation=0):
    """States entering consecutive spans from their summaries (page, "Summaries": the state after
    a span is the state before it times the span's transition plus the span's own end state,
    S_final = S_init * transition + S_H).  With states [.., K, V] and transition = P^T
    [.., K, K] as gdn_summary returns them: S_{r+1}[b][v] = sum_a transition_r[a][b] S_r[a][v]
    + end_r[b][v].  Returns [S_0 = start, S_1, ..., S_R] (fp64)."""
    S = np.asarray(start, dtype=np.float64)
    out = [S]
    for tr, sh in zip(transitions, end_states):
        tr = np.asarray(tr, dtype=np.float64)
        M = np.swapaxes(tr, -1, -2) if mutation != 23 else tr
        S = M @ S + np.asarray(sh, dtype=np.float64)
        out.append(S)
    return out


def compose_span_grads(transitions, local_grads, d_final, mutation=0):
    """The reverse of compose_spans for a state gradient: leaving span r the cotangent is d_r;
    through the span it becomes d_enter = transition_r d_r + g_r, g_r the span's own
    entering-state gradient (the state is linear in the entering state with Jacobian
    transition^T).  Returns [d leaving span 0, ..., d leaving span R-1, d entering span 0]."""
    d = np.asarray(d_final, dtype=np.float64)
    R = len(transitions)
    leaving = [None] * R
    for r in range(R - 1, -1, -1):
        leaving[r] = d
        tr = np.asarray(transitions[r], dtype=np.float64)
        loc = np.asarray(local_grads[r], dtype=np.float64)
        d = loc + tr @ d if mutation != 24 else tr @ (d + loc)
    return leaving + [d]


def _run(q, k, v, g, beta, cu_seqlens, *, scale, use_qk_l2norm, s0, want_final,
         checkpoint_every_n, want_o, want_transition, unit_mask, nthreads, mutation):
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    cu = _i64(cu_seqlens)
    T, HK, K = k.shape
    HV, V = v.shape[1], v.shape[2]
    N = cu.shape[0] - 1
    HO = HV
    assert q.shape == (T, HK, K) and v.shape[0] == T
    assert g.shape == (T, HO) and beta.shape == (T, HO)
    if scale is None:
        scale = 1.0 / np.sqrt(K)
    s0 = _f64(s0)
    if s0 is not None:
        assert s0.shape == (N, HO, K, V)
    o = np.zeros((T, HO, V)) if want_o else None
    fin = np.zeros((N, HO, K, V)) if want_final else None
    ck = ck_off = None
    if checkpoint_every_n:
        ck_off, R = checkpoint_offsets(cu, checkpoint_every_n)
        ck = np.zeros((R, HO, K, V))
    tr = np.zeros((N, HO, K, K)) if want_transition else None
    mask = None
    if unit_mask is not None:
        mask = np.ascontiguousarray(np.asarray(unit_mask, dtype=np.uint8).reshape(N * HO))
    rc = _load().gdn_oracle_run(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu, ctypes.c_int64),
        T, N, HK, HV, K, V, float(scale), int(bool(use_qk_l2norm)), _ptr(s0),
        _ptr(o), _ptr(fin), _ptr(ck), int(checkpoint_every_n or 0),
        _ptr(ck_off, ctypes.c_int64), _ptr(tr),
        mask.ctypes.data if mask is not None else None,
        int(nthreads or _default_threads()), int(mutation))
    if rc != 0:
        raise ValueError("oracle rejected its arguments (cu_seqlens or shapes)")
    return {"o": o, "final_state": fin, "checkpoints": ck, "transition": tr}
