"""Multi-rank path on CPU: span-parallel composition over gloo (world size 2), and the
benchmark's rank helpers.  The span summaries, forwards and the composition itself come from
the fp64 oracle (passed to the exchange as its `composer`; the library's composition kernel is
tested on the GPU), so no GPU is involved; the exchange, the choice of spans each rank composes
and the broadcasts of the start state and the final cotangent are the code under test."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from gated_delta_rule_29_gb300 import context_parallel as cp


def _case():
    rng = np.random.default_rng(99)
    L, HV, K, V = 96, 2, 8, 4
    q = rng.standard_normal((L, 1, K))
    k = rng.standard_normal((L, 1, K))
    v = rng.standard_normal((L, HV, V))
    g = -np.log1p(np.exp(rng.standard_normal((L, HV)))) * 0.05
    beta = 0.3 / (1.0 + np.exp(-rng.standard_normal((L, HV))))
    s0 = 0.2 * rng.standard_normal((1, HV, K, V))
    return q, k, v, g, beta, s0


def _oracle_compose(trs, shs, s0, like=None):
    return [torch.from_numpy(x) for x in oracle.compose_spans([t.numpy() for t in trs], [s.numpy() for s in shs],
                                                              s0.numpy())]


def _oracle_compose_grads(trs, lgs, dfin):
    return [torch.from_numpy(x) for x in oracle.compose_span_grads([t.numpy() for t in trs],
                                                                   [x.numpy() for x in lgs], dfin.numpy())]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q, k, v, g, beta, s0 = _case()
        L = q.shape[0]
        a, b = rank * L // world, (rank + 1) * L // world
        sl = slice(a, b)
        summ = oracle.gdn_summary(k[sl], v[sl], g[sl], beta[sl], np.array([0, b - a]), nthreads=1)
        tr = torch.from_numpy(summ["transition"][0])
        sh = torch.from_numpy(summ["end_state"][0])
        s_in = cp.entering_state(tr, sh, initial_state=torch.from_numpy(s0[0]) if rank == 0 else
                                 torch.zeros_like(torch.from_numpy(s0[0])), composer=_oracle_compose)
        fw = oracle.gdn_fwd(q[sl], k[sl], v[sl], g[sl], beta[sl], np.array([0, b - a]),
                            initial_state=s_in.numpy()[None], nthreads=1)
        # the benchmark's rank helpers: barrier and max over ranks
        import bench
        bench.barrier(world)
        mx = bench.max_over_ranks(float(rank + 1), world)
        results[rank] = {"s_in": s_in.numpy(), "final": fw["final_state"][0], "o": fw["o"], "max": mx}
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_rank_span_composition_matches_unsplit():
    world = 2
    mgr = mp.Manager()
    results = mgr.dict()
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
    for p_ in procs:
        p_.start()
    for p_ in procs:
        p_.join(240)
        assert p_.exitcode == 0
    q, k, v, g, beta, s0 = _case()
    L = q.shape[0]
    full = oracle.gdn_fwd(q, k, v, g, beta, np.array([0, L]), initial_state=s0, checkpoint_every_n=L // world,
                          nthreads=1)
    # rank 1 enters with the state at the span boundary: checkpoint entry 1 of the unsplit run
    np.testing.assert_allclose(results[1]["s_in"], full["checkpoints"][1], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(results[0]["s_in"], s0[0], rtol=0, atol=0)
    np.testing.assert_allclose(results[world - 1]["final"], full["final_state"][0], rtol=1e-10, atol=1e-12)
    o = np.concatenate([results[r]["o"] for r in range(world)])
    np.testing.assert_allclose(o, full["o"], rtol=1e-9, atol=1e-12)
    assert results[0]["max"] == results[1]["max"] == float(world)


def test_compose_single_process():
    q, k, v, g, beta, s0 = _case()
    L = q.shape[0]
    cuts = [0, 30, 31, 70, L]
    trs, shs = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        s = oracle.gdn_summary(k[a:b], v[a:b], g[a:b], beta[a:b], np.array([0, b - a]), nthreads=1)
        trs.append(torch.from_numpy(s["transition"][0]))
        shs.append(torch.from_numpy(s["end_state"][0]))
    states = _oracle_compose(trs, shs, torch.from_numpy(s0[0]))
    full = oracle.gdn_fwd(q, k, v, g, beta, np.array([0, L]), initial_state=s0, checkpoint_every_n=1, nthreads=1)
    np.testing.assert_allclose(states[-1].numpy(), full["final_state"][0], rtol=1e-10, atol=1e-12)
    for j, c in enumerate(cuts[:-1]):  # the state entering span j is the unsplit run's state at its cut
        np.testing.assert_allclose(states[j].numpy(), full["checkpoints"][c], rtol=1e-10, atol=1e-12)


def _bwd_worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q, k, v, g, beta, s0 = _case()
        L = q.shape[0]
        do = np.random.default_rng(98).standard_normal(v.shape)
        dfin = np.random.default_rng(97).standard_normal(s0.shape)
        a, b = rank * L // world, (rank + 1) * L // world
        sl = slice(a, b)
        cu = np.array([0, b - a])
        # forward composition (summaries + all-gather) gives the entering state
        summ = oracle.gdn_summary(k[sl], v[sl], g[sl], beta[sl], cu, nthreads=1)
        tr = torch.from_numpy(summ["transition"][0])
        s_in = cp.entering_state(tr, torch.from_numpy(summ["end_state"][0]),
                                 initial_state=torch.from_numpy(s0[0]) if rank == 0 else None,
                                 composer=_oracle_compose)
        # the span's own state gradient (the summary's mirror: zero exit cotangent), then the
        # composed exit cotangent
        loc = oracle.gdn_summary_bwd(q[sl], k[sl], g[sl], beta[sl], cu, do[sl])
        d_exit = cp.exit_state_grad(tr, torch.from_numpy(loc[0]),
                                    d_final=torch.from_numpy(dfin[0]) if rank == world - 1 else None,
                                    composer=_oracle_compose_grads)
        full = oracle.gdn_bwd(q[sl], k[sl], v[sl], g[sl], beta[sl], cu, do[sl], initial_state=s_in.numpy()[None],
                              d_final_state=d_exit.numpy()[None], nthreads=1)
        results[rank] = {k_: full[k_] for k_ in ("dq", "dk", "dv", "dg", "dbeta", "d_initial_state")}
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_rank_backward_composition_matches_unsplit():
    """Context-parallel backward on two gloo ranks: each span's own state gradient (the summary's
    mirror), one all-gather, the reverse composition of the state gradient, and the span
    backwards from it reproduce the unsplit backward of the whole sequence."""
    world = 2
    mgr = mp.Manager()
    results = mgr.dict()
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_bwd_worker, args=(r, world, port, results)) for r in range(world)]
    for p_ in procs:
        p_.start()
    for p_ in procs:
        p_.join(240)
        assert p_.exitcode == 0
    q, k, v, g, beta, s0 = _case()
    L = q.shape[0]
    do = np.random.default_rng(98).standard_normal(v.shape)
    dfin = np.random.default_rng(97).standard_normal(s0.shape)
    ref = oracle.gdn_bwd(q, k, v, g, beta, np.array([0, L]), do, initial_state=s0, d_final_state=dfin, nthreads=1)
    for name in ("dq", "dk", "dv", "dg", "dbeta"):
        got = np.concatenate([results[r][name] for r in range(world)])
        np.testing.assert_allclose(got, ref[name], rtol=1e-8, atol=1e-10)
    np.testing.assert_allclose(results[0]["d_initial_state"], ref["d_initial_state"], rtol=1e-8, atol=1e-10)
