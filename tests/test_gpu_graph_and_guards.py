"""CUDA-graph capture of the library's calls, and guard regions around their outputs.

The boundary enqueues its launches on the caller's stream with no host synchronisation, and
allocates nothing when the caller passes a workspace, so a call can be captured in a CUDA graph
and replayed with new input contents (the serving pattern for decode steps).  Guard regions
filled with a sentinel around every output buffer check that no launch writes outside its
output, ragged tails and partial chunks included."""
import numpy as np
import pytest
import torch

import oracle
import gated_delta_rule_29_gb300 as la
from gated_delta_rule_29_gb300 import workloads as W

pytestmark = pytest.mark.gpu

GUARD = 4096


def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def rel(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.abs(ref).max()
    assert den > 0, "reference is all zero: the comparison would be vacuous"
    return float(np.abs(got - ref).max() / den)


def capture(fn):
    """Warm up on a side stream (library load, kernel attributes), then capture fn in a graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn(warm=True)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn(warm=False)
    return g


def test_forward_captured_in_cuda_graph_replays_new_inputs():
    lengths = [100, 64, 257]
    w = W.draw("graph fwd", lengths, 2, 4, 128, 128, seed=601, initial_state=True, slow_decay=True)
    w2 = W.draw("graph fwd 2", lengths, 2, 4, 128, 128, seed=602, initial_state=True, slow_decay=True)
    d = dev()
    ins = [x.to(d) for x in (w.q, w.k, w.v, w.g, w.beta)]
    s0 = w.initial_state.to(d)
    cu = w.cu_seqlens.to(d)
    R = la.checkpoint_rows(cu, 64)
    o = torch.empty(w.T, w.HV, w.V, dtype=torch.bfloat16, device=d)
    fin = torch.empty(w.N, w.HV, w.K, w.V, dtype=torch.float32, device=d)
    ck = torch.empty(R, w.HV, w.K, w.V, dtype=torch.float32, device=d)
    ws = torch.empty(la.workspace_bytes(w.N), dtype=torch.uint8, device=d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    scratch = [torch.empty_like(x) for x in (o, fin, ck)]

    def call(warm=False):
        oo, ff, cc = scratch if warm else (o, fin, ck)
        la.gdn_fwd(*ins, cu, initial_state=s0, o=oo, final_state=ff, checkpoints=cc, checkpoint_every_n=64,
                   checkpoint_dtype=torch.float32, workspace=ws, status=status)

    call()
    torch.cuda.synchronize()
    eager = [x.clone() for x in (o, fin, ck)]
    g = capture(call)
    for x in (o, fin, ck):
        x.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert la.read_status(status) == 0
    for x, y in zip((o, fin, ck), eager):
        assert torch.equal(x, y)
    # new contents in the same input buffers: the replay reads them at replay time
    for dst, src in zip(ins, (w2.q, w2.k, w2.v, w2.g, w2.beta)):
        dst.copy_(src.to(d))
    s0.copy_(w2.initial_state.to(d))
    g.replay()
    torch.cuda.synchronize()
    replayed = [x.clone() for x in (o, fin, ck)]
    call()
    torch.cuda.synchronize()
    for x, y in zip(replayed, (o, fin, ck)):
        assert torch.equal(x, y)
    ref = oracle.gdn_fwd(w2.q, w2.k, w2.v, w2.g, w2.beta, w2.cu_seqlens, initial_state=w2.initial_state)
    e_o, e_f = rel(replayed[0].float().cpu(), ref["o"]), rel(replayed[1].cpu(), ref["final_state"])
    print(f"[parity] graph replay, new inputs: o {e_o:.2e}, final {e_f:.2e}")
    assert e_o <= 1e-2 and e_f <= 2e-3


def test_decode_steps_captured_in_cuda_graph():
    """One decode step captured once and replayed for several steps with new token inputs: the
    state pool evolves exactly as under eager calls."""
    d = dev()
    gen = torch.Generator().manual_seed(611)
    N, HK, HV, K, V, P, steps = 64, 2, 4, 128, 128, 96, 3
    pool0 = 0.1 * torch.randn(P, HV, K, V, generator=gen)
    idx = torch.randperm(P, generator=gen)[:N].to(torch.int32).to(d)
    toks = []
    for _ in range(steps):
        toks.append((torch.randn(N, HK, K, generator=gen).to(torch.bfloat16),
                     torch.randn(N, HK, K, generator=gen).to(torch.bfloat16),
                     torch.randn(N, HV, V, generator=gen).to(torch.bfloat16),
                     -torch.nn.functional.softplus(torch.randn(N, HV, generator=gen)) * 0.1,
                     torch.sigmoid(torch.randn(N, HV, generator=gen)) * 0.5))
    # eager
    pool_e = pool0.to(d)
    outs_e = []
    for t in toks:
        outs_e.append(la.gdn_decode(*(x.to(d) for x in t), pool_e, state_indices=idx).clone())
    # graph: fixed input buffers, replayed once per step
    bufs = [x.to(d).clone() for x in toks[0]]
    pool_g = pool0.to(d)
    pool_w = pool0.to(d)
    o = torch.empty(N, HV, V, dtype=torch.bfloat16, device=d)

    def step(warm=False):
        la.gdn_decode(*bufs, pool_w if warm else pool_g, state_indices=idx, o=o)

    g = capture(step)
    for t, oe in zip(toks, outs_e):
        for dst, src in zip(bufs, t):
            dst.copy_(src.to(d))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o, oe)
    assert torch.equal(pool_g, pool_e)


def guarded(shape, dtype, sentinel, d):
    n = int(np.prod(shape))
    big = torch.full((GUARD + n + GUARD,), sentinel, dtype=dtype, device=d)
    return big, big[GUARD:GUARD + n].view(*shape)


def intact(big, sentinel):
    return bool((big[:GUARD] == sentinel).all()) and bool((big[-GUARD:] == sentinel).all())


@pytest.mark.parametrize("K,V", [(128, 128), (64, 128)])
def test_forward_and_summary_write_only_their_outputs(K, V):
    """Ragged sequences (one token, chunk +- 1, an empty one, partial last chunks) with fp32
    checkpoints every 64 tokens: the 4096 elements on either side of o, the final state, the
    checkpoints, the summary's end states and transitions keep their sentinel."""
    lengths = [1, 63, 65, 200, 0, 129]
    w = W.draw("guards", lengths, 2, 4, K, V, seed=621 + K + V, initial_state=True, slow_decay=True)
    d = dev()
    cu = w.cu_seqlens.to(d)
    R = la.checkpoint_rows(cu, 64)
    s = -77.0
    o_big, o = guarded((w.T, w.HV, V), torch.bfloat16, s, d)
    f_big, fin = guarded((w.N, w.HV, K, V), torch.float32, s, d)
    c_big, ck = guarded((R, w.HV, K, V), torch.float32, s, d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    la.gdn_fwd(w.q.to(d), w.k.to(d), w.v.to(d), w.g.to(d), w.beta.to(d), cu, initial_state=w.initial_state.to(d),
               o=o, final_state=fin, checkpoints=ck, checkpoint_every_n=64, checkpoint_dtype=torch.float32,
               status=status)
    e_big, end = guarded((w.N, w.HV, K, V), torch.float32, s, d)
    t_big, tr = guarded((w.N, w.HV, K, K), torch.float32, s, d)
    la.gdn_summary(w.k.to(d), w.v.to(d), w.g.to(d), w.beta.to(d), cu, end_state=end, transition=tr, status=status)
    torch.cuda.synchronize()
    assert la.read_status(status) == 0
    for name, big in (("o", o_big), ("final_state", f_big), ("checkpoints", c_big), ("end_state", e_big),
                      ("transition", t_big)):
        assert intact(big, s), f"{name}: a write outside the buffer"
    ref = oracle.gdn_fwd(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, initial_state=w.initial_state,
                         checkpoint_every_n=64)
    assert rel(o.float().cpu(), ref["o"]) <= 1e-2
    assert rel(ck.cpu(), ref["checkpoints"]) <= 2e-3


def test_backward_writes_only_its_outputs_and_replays_in_a_graph():
    """The backward with the forward's checkpoints, grouped heads and ragged sequences (an empty
    one, one token, chunk +- 1): the guard regions around dq, dk, dv, dg, dbeta and the
    start-state gradient keep their sentinel, and the same call captured in a CUDA graph (caller
    workspace and outputs) replays bitwise and reads new cotangents at replay time."""
    lengths = [65, 0, 1, 63, 200]
    w = W.draw("bwd guards", lengths, 2, 4, 128, 64, seed=631, initial_state=True, slow_decay=True)
    d = dev()
    ins = [x.to(d) for x in (w.q, w.k, w.v, w.g, w.beta)]
    cu = w.cu_seqlens.to(d)
    s0 = w.initial_state.to(d)
    gen = torch.Generator().manual_seed(632)
    do1 = torch.randn(w.T, w.HV, w.V, generator=gen).to(torch.bfloat16)
    do2 = torch.randn(w.T, w.HV, w.V, generator=gen).to(torch.bfloat16)
    dfin = torch.randn(w.N, w.HV, w.K, w.V, generator=gen)
    _, _, ck = la.gdn_fwd(*ins, cu, initial_state=s0, checkpoint_every_n=64, checkpoint_dtype=torch.float32)
    s = -77.0
    shapes = [((w.T, w.HK, w.K), torch.bfloat16), ((w.T, w.HK, w.K), torch.bfloat16),
              ((w.T, w.HV, w.V), torch.bfloat16), ((w.T, w.HV), torch.float32), ((w.T, w.HV), torch.float32),
              ((w.N, w.HV, w.K, w.V), torch.float32)]
    bigs, outs = zip(*[guarded(shape, dt, s, d) for shape, dt in shapes])
    d_o = do1.to(d)
    dfin_d = dfin.to(d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    import gated_delta_rule_29_gb300.binding as B
    ws = torch.empty(B.load().la_gdn_bwd_workspace_bytes(w.T, w.N, w.HK, w.HV, w.K, w.V, 1), dtype=torch.uint8,
                     device=d)
    scratch = [torch.empty_like(x) for x in outs]

    def call(warm=False):
        la.gdn_bwd(*ins, cu, d_o, initial_state=s0, d_final_state=dfin_d, checkpoints=ck, workspace=ws,
                   status=status, out=tuple(scratch) if warm else outs)

    call()
    torch.cuda.synchronize()
    assert la.read_status(status) == 0
    for name, big in zip(("dq", "dk", "dv", "dg", "dbeta", "d_initial_state"), bigs):
        assert intact(big, s), f"{name}: a write outside the buffer"
    ref = oracle.gdn_bwd(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, do1, initial_state=w.initial_state,
                         d_final_state=dfin)
    for name, x in zip(("dq", "dk", "dv", "dg", "dbeta", "d_initial_state"), outs):
        assert rel(x.float().cpu(), ref[name]) <= (1e-2 if name in ("dq", "dk", "dv") else 2e-3), name
    eager = [x.clone() for x in outs]
    g = capture(call)
    for x in outs:
        x.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert la.read_status(status) == 0
    for x, y in zip(outs, eager):
        assert torch.equal(x, y)
    # new cotangent contents: the replay reads them at replay time
    d_o.copy_(do2.to(d))
    g.replay()
    torch.cuda.synchronize()
    replayed = [x.clone() for x in outs]
    call()
    torch.cuda.synchronize()
    for x, y in zip(replayed, outs):
        assert torch.equal(x, y)
    ref2 = oracle.gdn_bwd(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, do2, initial_state=w.initial_state,
                          d_final_state=dfin)
    e = rel(replayed[2].float().cpu(), ref2["dv"])
    print(f"[parity] backward graph replay, new cotangent: dv {e:.2e}")
    assert e <= 1e-2
    for name, big in zip(("dq", "dk", "dv", "dg", "dbeta", "d_initial_state"), bigs):
        assert intact(big, s), f"{name}: a write outside the buffer (graph replay)"


def test_summary_bwd_writes_only_its_output():
    """gdn_summary_bwd into a caller buffer with guard regions: ragged spans, an empty one."""
    w = W.draw("sbwd guards", [1, 130, 0, 64], 2, 2, 64, 128, seed=641, slow_decay=True)
    d = dev()
    gen = torch.Generator().manual_seed(642)
    do = torch.randn(w.T, w.HV, w.V, generator=gen).to(torch.bfloat16)
    dfin = torch.randn(w.N, w.HV, w.K, w.V, generator=gen)
    s = -77.0
    big, out = guarded((w.N, w.HV, w.K, w.V), torch.float32, s, d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    res = la.gdn_summary_bwd(w.q.to(d), w.k.to(d), w.g.to(d), w.beta.to(d), w.cu_seqlens.to(d), do.to(d),
                             d_final_state=dfin.to(d), status=status, d_state=out)
    assert la.read_status(status) == 0
    assert res.data_ptr() == out.data_ptr()
    assert intact(big, s)
    ref = oracle.gdn_summary_bwd(w.q, w.k, w.g, w.beta, w.cu_seqlens, do, d_final_state=dfin)
    assert rel(out.cpu(), ref) <= 2e-3
