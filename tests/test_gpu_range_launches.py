"""Range launches against single walks, bitwise.

When a batch holds more (sequence, head) units than the GPU runs at once, gdn_summary and
gdn_bwd cut every unit's chunks into consecutive ranges and launch the ranges wave by wave, and
so does gdn_fwd when its units fill one to four waves; a later range restarts from the exact
fp32 state (the forward's final state or pool slot, the summary's end state and transition,
the backward's carried state gradient) that the previous range left behind.  The page requires a
sequence's results to be bitwise independent of the batch it runs in ("Semantics worth
knowing": batch_invariant), so every sequence of such a batch must give the same bits as the
same sequence run alone, which takes the single-walk path.  The batches below are ragged:
empty sequences, sequences of one to three chunks (whose first range can be empty) and longer
ones.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_29_gb300 as la
from gated_delta_rule_29_gb300 import workloads as W

pytestmark = pytest.mark.gpu

# 48 sequences x 8 heads = 384 units for the backward and 768 summary tiles: more than one
# wave of either kernel on a 152-SM GPU (one CTA per SM for both at these sizes)
LENGTHS = [0, 1, 63, 64, 65, 127, 128, 129, 191, 192, 0, 700, 255, 256, 257, 3, 511, 640,
           130, 0, 65, 200, 1000, 64, 2, 450, 129, 320, 0, 190, 66, 777,
           128, 1, 256, 380, 0, 193, 64, 900, 40, 129, 600, 192, 5, 333, 70, 128]


def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def workload():
    assert len(LENGTHS) == 48
    return W.draw("ranges", LENGTHS, 8, 8, 64, 64, seed=611, initial_state=True, slow_decay=True)


def one(w, i):
    cu = w.cu_seqlens.numpy().astype(np.int64)
    sl = slice(int(cu[i]), int(cu[i + 1]))
    return W.Workload(name=f"seq {i}", cu_seqlens=torch.tensor([0, cu[i + 1] - cu[i]], dtype=torch.int32),
                      q=w.q[sl], k=w.k[sl], v=w.v[sl], g=w.g[sl].contiguous(), beta=w.beta[sl].contiguous(),
                      initial_state=w.initial_state[i:i + 1].contiguous())


def summary(w, d):
    status = torch.zeros(1, dtype=torch.int32, device=d)
    end, tr = la.gdn_summary(w.k.to(d), w.v.to(d), w.g.to(d), w.beta.to(d), w.cu_seqlens.to(d),
                             start_state=w.initial_state.to(d), use_qk_l2norm=True, status=status)
    assert la.read_status(status) == 0
    return end, tr


def test_summary_ranges_match_single_walks_bitwise():
    d = dev()
    w = workload()
    end, tr = summary(w, d)
    assert torch.isfinite(end).all() and torch.isfinite(tr).all()
    eye = torch.eye(w.K, device=d).expand(w.HV, w.K, w.K)
    for i in range(w.N):
        if LENGTHS[i] == 0:  # an empty span: end state = start state, transition = I
            assert torch.equal(end[i], w.initial_state[i].to(d)) and torch.equal(tr[i], eye), i
            continue
        e1, t1 = summary(one(w, i), d)
        assert torch.equal(end[i], e1[0]), ("end state", i, LENGTHS[i])
        assert torch.equal(tr[i], t1[0]), ("transition", i, LENGTHS[i])


def bwd(w, do, dfin, d):
    status = torch.zeros(1, dtype=torch.int32, device=d)
    out = la.gdn_bwd(w.q.to(d), w.k.to(d), w.v.to(d), w.g.to(d), w.beta.to(d), w.cu_seqlens.to(d), do.to(d),
                     use_qk_l2norm=True, initial_state=w.initial_state.to(d), d_final_state=dfin.to(d),
                     status=status)
    assert la.read_status(status) == 0
    return out


def test_bwd_ranges_match_single_walks_bitwise():
    d = dev()
    w = workload()
    gen = torch.Generator().manual_seed(612)
    do = torch.randn(w.T, w.HV, w.V, generator=gen).to(torch.bfloat16)
    dfin = torch.randn(w.N, w.HV, w.K, w.V, generator=gen)
    full = bwd(w, do, dfin, d)
    cu = w.cu_seqlens.numpy().astype(np.int64)
    names = ["dq", "dk", "dv", "dg", "dbeta"]
    for i in range(w.N):
        sl = slice(int(cu[i]), int(cu[i + 1]))
        if LENGTHS[i] == 0:  # an empty sequence passes the final-state cotangent straight through
            assert torch.equal(full[5][i], dfin[i].to(d)), i
            continue
        alone = bwd(one(w, i), do[sl], dfin[i:i + 1], d)
        for name, x, y in zip(names, full[:5], alone[:5]):
            assert torch.equal(x[sl], y), (name, i, LENGTHS[i])
        assert torch.equal(full[5][i], alone[5][0]), ("d_initial_state", i, LENGTHS[i])


# ---------------------------------------------------------------- forward


def ckpt_offsets(lengths, n):
    return np.concatenate([[0], np.cumsum([(L + n - 1) // n for L in lengths])]).astype(np.int64)


def fwd(w, d, pieces, n=0, ckpt_dtype=torch.float32):
    lib = la.binding.load()
    assert lib.la_test_set_fwd_pieces(pieces) == 0
    try:
        status = torch.zeros(1, dtype=torch.int32, device=d)
        o, fin, ck = la.gdn_fwd(w.q.to(d), w.k.to(d), w.v.to(d), w.g.to(d), w.beta.to(d), w.cu_seqlens.to(d),
                                initial_state=w.initial_state.to(d), checkpoint_every_n=n,
                                checkpoint_dtype=ckpt_dtype, status=status)
        assert la.read_status(status) == 0
    finally:
        assert lib.la_test_set_fwd_pieces(0) == 0
    return o, fin, ck


@pytest.mark.parametrize("n,ckpt_dtype", [(64, torch.float32), (192, torch.bfloat16)])
def test_fwd_forced_ranges_match_single_walks_bitwise(n, ckpt_dtype):
    """Every sequence of a ragged 384-unit batch (empty sequences, one-chunk ones whose first
    ranges are empty, ranges ending on and between checkpoint rows), walked in 2, 3 and 8
    ranges: o, the final state and every checkpoint row equal the sequence run alone."""
    d = dev()
    w = workload()
    assert w.N * w.HV > 2 * torch.cuda.get_device_properties(0).multi_processor_count
    cu = w.cu_seqlens.numpy().astype(np.int64)
    off = ckpt_offsets(LENGTHS, n)
    alone = [fwd(one(w, i), d, 1, n, ckpt_dtype) for i in range(w.N)]
    for pieces in (2, 3, 8):
        o, fin, ck = fwd(w, d, pieces, n, ckpt_dtype)
        for i in range(w.N):
            a_o, a_fin, a_ck = alone[i]
            sl = slice(int(cu[i]), int(cu[i + 1]))
            assert torch.equal(o[sl], a_o), ("o", pieces, i, LENGTHS[i])
            assert torch.equal(fin[i], a_fin[0]), ("final state", pieces, i, LENGTHS[i])
            assert torch.equal(ck[int(off[i]):int(off[i + 1])], a_ck), ("checkpoints", pieces, i, LENGTHS[i])


def test_fwd_automatic_ranges_equal_whole_walks():
    """A uniform batch whose 320 units fill just over one wave (the case the automatic choice
    cuts into ranges) gives the same bits as whole walks, with and without checkpoints."""
    d = dev()
    w = W.draw("fwd ranges", [2048] * 40, 8, 8, 64, 64, seed=613, initial_state=True, slow_decay=True)
    for n in (0, 256):
        auto = fwd(w, d, 0, n)
        whole = fwd(w, d, 1, n)
        assert torch.equal(auto[0], whole[0]) and torch.equal(auto[1], whole[1]), n
        if n:
            assert torch.equal(auto[2], whole[2]), n


def test_fwd_ranges_through_an_fp32_state_pool():
    """With a state pool the hand-over goes through the sequences' own pool slots (a permuted
    slot map): the pool after a ranged call equals the pool after whole walks."""
    d = dev()
    w = workload()
    gen = torch.Generator().manual_seed(614)
    slots = torch.randperm(w.N + 5, generator=gen)[:w.N].to(torch.int32)
    pool0 = 0.1 * torch.randn(w.N + 5, w.HV, w.K, w.V, generator=gen)
    lib = la.binding.load()
    outs = []
    for pieces in (1, 4):
        pool = pool0.clone().to(d)
        status = torch.zeros(1, dtype=torch.int32, device=d)
        assert lib.la_test_set_fwd_pieces(pieces) == 0
        try:
            o, _, _ = la.gdn_fwd(w.q.to(d), w.k.to(d), w.v.to(d), w.g.to(d), w.beta.to(d), w.cu_seqlens.to(d),
                                 initial_state=pool, state_indices=slots.to(d), status=status)
            assert la.read_status(status) == 0
        finally:
            assert lib.la_test_set_fwd_pieces(0) == 0
        outs.append((o, pool))
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1], outs[1][1])
    untouched = torch.ones(w.N + 5, dtype=torch.bool)
    untouched[slots.long()] = False
    assert torch.equal(outs[1][1][untouched.to(d)], pool0[untouched].to(d))
