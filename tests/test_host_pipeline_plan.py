"""The token-range plan of gdn_fwd_host (host logic, no GPU): the ranges tile the packed batch
in order, every sequence is covered once (whole inside a run, or by consecutive pieces), and
every cut inside a sequence falls on a multiple of the piece length P, itself a multiple of
the 64-token chunk and of the checkpoint cadence."""
import math

import numpy as np
import pytest

from gated_delta_rule_29_gb300.api import _host_parts


def check_plan(lengths, groups, n):
    P, parts = _host_parts(lengths, groups, n)
    assert P % 64 == 0 and (n == 0 or P % n == 0)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    t = 0
    covered = []
    for (t_a, t_b, a, b, pc, last) in parts:
        assert t_a == t and t_b >= t_a
        t = t_b
        if pc < 0:
            assert last and b > a
            assert t_a == cu[a] and t_b == cu[b]
            assert b - a == 1 or t_b - t_a <= P
            covered += list(range(a, b))
        else:
            assert b == a + 1 and lengths[a] > P
            assert t_a - cu[a] == pc * P and 0 < t_b - t_a <= P
            assert last == (t_b == cu[a + 1])
            if pc == 0:
                covered.append(a)
    assert t == cu[-1]
    assert covered == list(range(len(lengths)))
    return P, parts


@pytest.mark.parametrize("groups", [1, 2, 3, 8, 32, 1000])
@pytest.mark.parametrize("n", [0, 64, 128, 1024])
def test_plan_random_batches(groups, n):
    rng = np.random.default_rng(groups * 7 + n)
    for _ in range(20):
        N = int(rng.integers(1, 12))
        lengths = [int(x) for x in rng.integers(0, 3000, size=N)]
        lengths[int(rng.integers(0, N))] = 0 if rng.random() < 0.3 else lengths[0]
        check_plan(lengths, groups, n)


def test_plan_dense_batch():
    """8 sequences of 8192 tokens in 32 ranges: 2048-token pieces, four per sequence."""
    P, parts = check_plan([8192] * 8, 32, 1024)
    assert P == 2048 and len(parts) == 32
    assert all(pc == i % 4 for i, (_, _, _, _, pc, _) in enumerate(parts))


def test_plan_one_range_and_empty():
    P, parts = check_plan([300, 1, 0, 200], 1, 64)
    assert parts == [(0, 501, 0, 4, -1, True)]
    assert check_plan([0, 0], 4, 0)[1] == [(0, 0, 0, 2, -1, True)]
    assert check_plan([], 4, 0)[1] == []


def test_plan_checkpoint_cadence_sets_the_cut():
    """With checkpoints every 192 tokens the cut is a multiple of lcm(64, 192) = 192."""
    P, _ = check_plan([1000, 1000], 8, 192)
    assert P % math.lcm(64, 192) == 0


def test_host_entry_rejects_bad_seqlens_before_any_device_work():
    """A cu_seqlens that is not 0, nondecreasing, T makes gdn_fwd_host raise on the host before
    any device work (the library's own entry returns LA_ERR_BAD_SEQLENS for it too, see
    test_abi)."""
    import torch

    import gated_delta_rule_29_gb300 as la
    T, H, D = 128, 1, 64
    q = torch.zeros(T, H, D, dtype=torch.bfloat16)
    v = torch.zeros(T, H, D, dtype=torch.bfloat16)
    g = torch.zeros(T, H)
    b = torch.zeros(T, H)
    for cu in ([0, 100, 64, 128], [0, 64, 100], [8, 64, 128]):
        with pytest.raises(ValueError):
            la.gdn_fwd_host(q, q, v, g, b, torch.tensor(cu, dtype=torch.int32), device=torch.device("cuda", 0))
