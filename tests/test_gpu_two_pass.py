"""The two-pass forward against the fused kernel, bitwise.

gdn_fwd may form the state-independent half of every chunk (G, the norms, A, P and
T = (I + A)^{-1}) for the whole batch first and then walk each sequence with only the
state-dependent products on its serial chain (when its workspace has room for the per-chunk
records), or do both in one fused kernel.  The two run the same arithmetic, so every output
must be the same bits: o, the final state, the checkpoints and a state pool written back in
place.  The oracle parity of the path itself is covered by the other forward tests, which take
the two-pass schedule by default.  The cases span the options the chunk's first half depends
on: head dims, grouped heads, the gate and beta transforms, no l2 norm, ragged and empty
sequences, a bf16 start state, bf16 checkpoints, and range launches on top.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_29_gb300 as la
from gated_delta_rule_29_gb300 import workloads as W

pytestmark = pytest.mark.gpu

RAGGED = [0, 1, 63, 64, 65, 300, 0, 129, 1000, 7]


def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def run(w, d, passes, pieces=0, **kw):
    lib = la.binding.load()
    assert lib.la_test_set_fwd_passes(passes) == 0 and lib.la_test_set_fwd_pieces(pieces) == 0
    try:
        status = torch.zeros(1, dtype=torch.int32, device=d)
        s0 = kw.pop("initial_state", w.initial_state)
        out = la.gdn_fwd(w.q.to(d), w.k.to(d), w.v.to(d), w.g.to(d), w.beta.to(d), w.cu_seqlens.to(d),
                         initial_state=None if s0 is None else s0.to(d), status=status, **kw)
        assert la.read_status(status) == 0
    finally:
        assert lib.la_test_set_fwd_passes(0) == 0 and lib.la_test_set_fwd_pieces(0) == 0
    return out


def bits(x):
    return x.view(torch.int16) if x.element_size() == 2 else x.view(torch.int32)


def same(a, b, tag):
    for name, x, y in zip(("o", "final state", "checkpoints"), a, b):
        assert (x is None) == (y is None), (tag, name)
        if x is not None:
            assert torch.isfinite(x.float()).all(), (tag, name, "non-finite values: the case is ill-posed")
            assert torch.equal(bits(x), bits(y)), (tag, name, float((x.float() - y.float()).abs().max()))


CASES = {
    "ragged K=V=128": dict(lengths=RAGGED, HK=2, HV=2, K=128, V=128),
    "ragged K=V=64": dict(lengths=RAGGED, HK=2, HV=2, K=64, V=64),
    "K=64 V=128 grouped 1:4": dict(lengths=[200, 64, 1, 511], HK=1, HV=4, K=64, V=128),
    "K=128 V=64 grouped 2:6": dict(lengths=[130, 70, 1024], HK=2, HV=6, K=128, V=64),
    "one long sequence": dict(lengths=[4096 + 17], HK=4, HV=4, K=128, V=128),
}


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("slow", [False, True])
def test_two_pass_equals_fused(name, slow):
    c = CASES[name]
    d = dev()
    w = W.draw(name, c["lengths"], c["HK"], c["HV"], c["K"], c["V"], seed=701 + len(name), initial_state=True,
               slow_decay=slow)
    kw = dict(checkpoint_every_n=128, checkpoint_dtype=torch.float32)
    same(run(w, d, 1, **kw), run(w, d, 2, **kw), name)


def raw_gates(w, seed, beta_dtype=torch.float32):
    gen = torch.Generator().manual_seed(seed)
    g_raw = torch.randn(w.T, w.HV, generator=gen)
    beta_logit = torch.randn(w.T, w.HV, generator=gen).to(beta_dtype)
    a_log = torch.randn(w.HV, generator=gen) * 0.5
    dt_bias = torch.randn(w.HV, generator=gen) * 0.5
    return g_raw.contiguous(), beta_logit.contiguous(), a_log, dt_bias


@pytest.mark.parametrize("beta_dtype", [torch.float32, torch.bfloat16])
def test_two_pass_equals_fused_with_transforms(beta_dtype):
    d = dev()
    w = W.draw("transforms", [300, 64, 0, 129], 2, 4, 128, 128, seed=711, initial_state=True)
    g_raw, beta_logit, a_log, dt_bias = raw_gates(w, 712, beta_dtype)
    w.g, w.beta = g_raw, beta_logit
    soft = dict(a_log=a_log.to(d), dt_bias=dt_bias.to(d), beta_sigmoid=True)
    same(run(w, d, 1, **soft), run(w, d, 2, **soft), "softplus gate, beta logits")
    bound = dict(gate_lower_bound=-5.0, beta_sigmoid=True)
    same(run(w, d, 1, **bound), run(w, d, 2, **bound), "bounded gate, beta logits")


def test_two_pass_equals_fused_options():
    """No l2 norm with an explicit scale, a bf16 start state, bf16 checkpoints every 64 tokens."""
    d = dev()
    w = W.draw("options", RAGGED, 2, 2, 128, 64, seed=721, initial_state=True)
    # without the in-kernel norm the keys and queries are given at unit scale (|k|^2 ~ 1)
    w.q, w.k = ((x.float() * 128 ** -0.5).to(torch.bfloat16) for x in (w.q, w.k))
    kw = dict(use_qk_l2norm=False, scale=0.5)
    same(run(w, d, 1, **kw), run(w, d, 2, **kw), "no l2 norm")
    s0 = w.initial_state.to(torch.bfloat16)
    kw = dict(initial_state=s0, checkpoint_every_n=64, checkpoint_dtype=torch.bfloat16)
    same(run(w, d, 1, **kw), run(w, d, 2, **kw), "bf16 start state, bf16 checkpoints")
    kw = dict(output_final_state=False)
    same(run(w, d, 1, **kw), run(w, d, 2, **kw), "no final state")


def test_two_pass_state_pool_and_ranges():
    """A permuted fp32 state pool written back in place, and forced chunk ranges (2 and 5) on a
    batch of more units than one wave: all equal to the fused whole walks."""
    d = dev()
    lengths = [0, 1, 63, 64, 65, 127, 128, 129, 191, 192, 0, 700, 255, 256, 257, 3, 511, 640,
               130, 0, 65, 200, 1000, 64, 2, 450, 129, 320, 0, 190, 66, 777,
               128, 1, 256, 380, 0, 193, 64, 900, 40, 129, 600, 192, 5, 333, 70, 128]
    w = W.draw("pool", lengths, 8, 8, 64, 64, seed=731, initial_state=True, slow_decay=True)
    gen = torch.Generator().manual_seed(732)
    slots = torch.randperm(w.N + 3, generator=gen)[:w.N].to(torch.int32).to(d)
    pool0 = 0.1 * torch.randn(w.N + 3, w.HV, w.K, w.V, generator=gen)
    outs = []
    for passes in (1, 2):
        pool = pool0.clone().to(d)
        o, _, _ = run(w, d, passes, initial_state=pool, state_indices=slots)
        outs.append((o, pool))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    kw = dict(checkpoint_every_n=192, checkpoint_dtype=torch.float32)
    ref = run(w, d, 1, 1, **kw)
    for pieces in (2, 5):
        same(ref, run(w, d, 2, pieces, **kw), f"two passes in {pieces} ranges")


def test_minimal_workspace_takes_the_fused_kernel():
    """A caller workspace of la_gdn_workspace_bytes(N, 0) has no room for the records: the call
    still succeeds (fused kernel) with the same bits."""
    d = dev()
    w = W.draw("small ws", RAGGED, 2, 2, 64, 64, seed=741, initial_state=True)
    ws = torch.empty(la.workspace_bytes(w.N), dtype=torch.uint8, device=d)
    assert la.api.split_workspace_bytes(w.T, w.N, w.HV) > ws.numel()
    same(run(w, d, 2, workspace=ws), run(w, d, 2), "minimal workspace")


# ---------------------------------------------------------------- summary


def summary(w, d, passes, start=None, **kw):
    lib = la.binding.load()
    assert lib.la_test_set_fwd_passes(passes) == 0
    try:
        status = torch.zeros(1, dtype=torch.int32, device=d)
        end, tr = la.gdn_summary(w.k.to(d), w.v.to(d), w.g.to(d), w.beta.to(d), w.cu_seqlens.to(d),
                                 start_state=None if start is None else start.to(d), status=status, **kw)
        assert la.read_status(status) == 0
    finally:
        assert lib.la_test_set_fwd_passes(0) == 0
    return end, tr


SUMMARY_CASES = {
    "ragged spans K=V=128": dict(lengths=RAGGED, HK=2, HV=2, K=128, V=128),
    "ragged spans K=V=64": dict(lengths=RAGGED, HK=1, HV=3, K=64, V=64),
    "K=128 V=64 grouped 2:4": dict(lengths=[700, 64, 1, 2000], HK=2, HV=4, K=128, V=64),
    "K=64 V=128": dict(lengths=[130, 1500], HK=2, HV=2, K=64, V=128),
}


@pytest.mark.parametrize("name", list(SUMMARY_CASES))
@pytest.mark.parametrize("slow", [False, True])
def test_two_pass_summary_equals_fused(name, slow):
    """End states (from a nonzero start) and transitions: the same bits."""
    c = SUMMARY_CASES[name]
    d = dev()
    w = W.draw(name, c["lengths"], c["HK"], c["HV"], c["K"], c["V"], seed=751 + len(name), initial_state=True,
               slow_decay=slow)
    for start in (None, w.initial_state):
        a, b = summary(w, d, 1, start), summary(w, d, 2, start)
        assert torch.equal(bits(a[0]), bits(b[0])), (name, "end state")
        assert torch.equal(bits(a[1]), bits(b[1])), (name, "transition")


def test_two_pass_summary_transforms_and_ranges():
    """The gate and beta transforms, and a batch of spans whose (span, head, tile) units exceed
    a wave even at two CTAs per SM (the range launches on top of the two passes)."""
    d = dev()
    w = W.draw("sum transforms", [300, 64, 0, 129], 2, 4, 128, 128, seed=761, initial_state=True)
    g_raw, beta_logit, a_log, dt_bias = raw_gates(w, 762)
    w.g, w.beta = g_raw, beta_logit
    kw = dict(a_log=a_log.to(d), dt_bias=dt_bias.to(d), beta_sigmoid=True)
    a, b = summary(w, d, 1, w.initial_state, **kw), summary(w, d, 2, w.initial_state, **kw)
    assert torch.equal(bits(a[0]), bits(b[0])) and torch.equal(bits(a[1]), bits(b[1]))
    lengths = [0, 1, 63, 64, 65, 127, 128, 129, 191, 192, 0, 700, 255, 256, 257, 3, 511, 640,
               130, 0, 65, 200, 1000, 64, 2, 450, 129, 320, 0, 190, 66, 777,
               128, 1, 256, 380, 0, 193, 64, 900, 40, 129, 600, 192, 5, 333, 70, 128]
    w = W.draw("sum ranges", lengths, 8, 8, 64, 64, seed=763, initial_state=True, slow_decay=True)
    assert w.N * w.HV * 2 > 2 * torch.cuda.get_device_properties(0).multi_processor_count
    a, b = summary(w, d, 1, w.initial_state), summary(w, d, 2, w.initial_state)
    assert torch.equal(bits(a[0]), bits(b[0])) and torch.equal(bits(a[1]), bits(b[1]))


# ---------------------------------------------------------------- Gated DeltaProduct


@pytest.mark.parametrize("n", [2, 3, 5, 16, 64])
def test_two_pass_gdp_equals_fused(n):
    """GDP natively on the update timeline (n updates per token): two passes and the fused kernel
    give the same outputs, final states and checkpoints (every 64 tokens)."""
    d = dev()
    lengths = [0, 1, 33, 64, 100, 257]
    w = W.draw(f"gdp {n}", lengths, 2, 4, 64, 64, seed=771 + n, initial_state=True, slow_decay=True)
    gen = torch.Generator().manual_seed(772 + n)
    T = w.T
    k = torch.randn(T * n, w.HK, w.K, generator=gen).to(torch.bfloat16)
    v = torch.randn(T * n, w.HV, w.V, generator=gen).to(torch.bfloat16)
    beta = (0.1 * torch.rand(T * n, w.HV, generator=gen)).contiguous()
    outs = []
    lib = la.binding.load()
    for passes in (1, 2):
        assert lib.la_test_set_fwd_passes(passes) == 0
        try:
            status = torch.zeros(1, dtype=torch.int32, device=d)
            outs.append(la.gdn_fwd(w.q.to(d), k.to(d), v.to(d), w.g.to(d), beta.to(d), w.cu_seqlens.to(d),
                                   initial_state=w.initial_state.to(d), checkpoint_every_n=64,
                                   checkpoint_dtype=torch.float32, num_householder=n, status=status))
            assert la.read_status(status) == 0
        finally:
            assert lib.la_test_set_fwd_passes(0) == 0
    same(outs[0], outs[1], f"GDP n={n}")


def test_api_workspace_falls_back_when_the_two_pass_room_cannot_be_allocated():
    """The wrappers allocate room for the two passes (about 272 bytes per token and head); when
    that allocation fails they hand the library the minimal workspace, which takes the fused
    kernel, instead of failing the call."""
    d = dev()
    ws = la.api._workspace(1 << 50, 4096, d)  # a petabyte: refused by the allocator, nothing launched
    assert ws.numel() == 4096
