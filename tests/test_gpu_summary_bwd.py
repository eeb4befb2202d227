"""gdn_summary_bwd (the state-gradient mirror of the span summary) vs the fp64 oracle, through
the C ABI.

Tolerance (max|x - ref| / max|ref| per tensor): 2e-3, as for the fp32 states.  The loss is
sum(d_o * o) + sum(d_final_state * end_state) with seeded N(0,1) cotangents; the result is its
gradient with respect to the state entering each span."""
import numpy as np
import pytest
import torch

import oracle
import gated_delta_rule_29_gb300 as la
from gated_delta_rule_29_gb300 import context_parallel as CP
from gated_delta_rule_29_gb300 import workloads as W

pytestmark = pytest.mark.gpu

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
    do = torch.randn(w.T, w.HV, w.V, generator=gen).to(torch.bfloat16)
    dfin = torch.randn(w.N, w.HV, w.K, w.V, generator=gen) if with_final else None
    return do, dfin


def run(w, do, dfin, l2=True, scale=None, cu=None, passes=0):
    """passes 0: the automatic path (the tensor-core state-gradient pass when the workspace has
    room, as the API's default workspace does); 1: the tile kernel's state-only mode."""
    d = dev()
    status = torch.zeros(1, dtype=torch.int32, device=d)
    cu = w.cu_seqlens if cu is None else cu
    lib = la.binding.load()
    assert lib.la_test_set_fwd_passes(passes) == 0
    try:
        out = la.gdn_summary_bwd(w.q.to(d), w.k.to(d), w.g.to(d), w.beta.to(d), cu.to(d), do.to(d),
                                 use_qk_l2norm=l2, scale=scale, d_final_state=None if dfin is None else dfin.to(d),
                                 status=status)
        assert la.read_status(status) == 0
    finally:
        assert lib.la_test_set_fwd_passes(0) == 0
    return out


def check(w, got, ref, label):
    e = rel(got.cpu().numpy(), ref)
    print(f"[parity] summary_bwd {w.name}{label}: d_state {e:.2e}")
    assert e <= F32_TOL
    return e


@pytest.mark.parametrize("K,V", [(64, 64), (128, 128), (64, 128), (128, 64)])
def test_summary_bwd_ragged_grouped_heads(K, V):
    """Ragged spans (one token, one chunk +- 1, several chunks, an empty span), grouped heads,
    a final-state cotangent, slow decay so that every chunk reaches the span start."""
    w = W.draw("sbwd ragged", [1, 63, 64, 0, 65, 200], 2, 4, K, V, seed=501 + K + V, slow_decay=True)
    do, dfin = cotangents(w, 502)
    got = run(w, do, dfin)
    ref = oracle.gdn_summary_bwd(w.q, w.k, w.g, w.beta, w.cu_seqlens, do, d_final_state=dfin)
    check(w, got, ref, f" K={K} V={V}")
    # the empty span passes the exit cotangent through unchanged
    assert torch.equal(got[3].cpu(), dfin[3].float())


def test_summary_bwd_page_distributions_no_final():
    """The pages' gate and beta distributions (fast decay) and no exit cotangent."""
    w = W.draw("sbwd page", [300, 129, 1000], 4, 4, 128, 128, seed=511)
    do, _ = cotangents(w, 512, with_final=False)
    got = run(w, do, None)
    ref = oracle.gdn_summary_bwd(w.q, w.k, w.g, w.beta, w.cu_seqlens, do)
    check(w, got, ref, "")


def test_summary_bwd_without_l2norm():
    """Keys and queries scaled to unit-order norms by hand, the kernel's norm off, explicit scale."""
    w = W.draw("sbwd no-norm", [150, 70], 1, 2, 64, 64, seed=521, slow_decay=True)
    w.q = (w.q.float() / 8.0).to(torch.bfloat16)
    w.k = (w.k.float() / 8.0).to(torch.bfloat16)
    do, dfin = cotangents(w, 522)
    got = run(w, do, dfin, l2=False, scale=0.5)
    ref = oracle.gdn_summary_bwd(w.q, w.k, w.g, w.beta, w.cu_seqlens, do, scale=0.5, use_qk_l2norm=False,
                                 d_final_state=dfin)
    check(w, got, ref, "")


def test_summary_bwd_equals_backward_state_gradient_bitwise():
    """Each path of gdn_summary_bwd is bitwise the entering-state gradient of the full backward
    on the same path (the tile kernel's state-only mode and the tile backward; the state-gradient
    pass, which the tensor-core backward runs too); the two paths agree to fp32-level tolerance."""
    w = W.draw("sbwd vs bwd", [130, 64, 257], 2, 2, 128, 128, seed=531, initial_state=True, slow_decay=True)
    do, dfin = cotangents(w, 532)
    d = dev()
    lib = la.binding.load()

    def full_bwd(passes):
        assert lib.la_test_set_fwd_passes(passes) == 0
        try:
            return la.gdn_bwd(w.q.to(d), w.k.to(d), w.v.to(d), w.g.to(d), w.beta.to(d), w.cu_seqlens.to(d),
                              do.to(d), initial_state=w.initial_state.to(d), d_final_state=dfin.to(d))[5]
        finally:
            assert lib.la_test_set_fwd_passes(0) == 0

    a = run(w, do, dfin, passes=1)
    assert torch.equal(a, full_bwd(1))
    c = run(w, do, dfin)
    assert torch.equal(c, full_bwd(0))
    e = rel(c.cpu().numpy(), a.cpu().numpy())
    print(f"[parity] summary_bwd tensor-core pass vs tile kernel: {e:.2e}")
    assert e <= F32_TOL


def test_summary_bwd_batch_invariant():
    """A span's state gradient is bitwise the same alone and inside a batch."""
    w = W.draw("sbwd batch", [90, 200, 33, 128], 2, 2, 64, 64, seed=541, slow_decay=True)
    do, dfin = cotangents(w, 542)
    full = run(w, do, dfin)
    cu = w.cu_seqlens.numpy().astype(np.int64)
    i = 1
    sl = slice(cu[i], cu[i + 1])
    sub = W.Workload(name="one", cu_seqlens=torch.tensor([0, cu[i + 1] - cu[i]]), q=w.q[sl], k=w.k[sl], v=w.v[sl],
                     g=w.g[sl].contiguous(), beta=w.beta[sl].contiguous())
    alone = run(sub, do[sl], dfin[i:i + 1])
    assert torch.equal(full[i], alone[0])


def test_summary_bwd_span_composition():
    """Context-parallel backward on one GPU: per-span state gradients (zero exit cotangent),
    composed right to left with gdn_summary's transitions, equal the whole sequence's."""
    L = 2048
    w = W.draw("sbwd spans", [L], 4, 4, 128, 128, seed=551, slow_decay=True)
    do, dfin = cotangents(w, 552)
    spans = torch.tensor([0, 512, 1024, 1536, L], dtype=torch.int32)
    d = dev()
    loc = run(w, do, None, cu=spans)
    _, trs = la.gdn_summary(w.k.to(d), w.v.to(d), w.g.to(d), w.beta.to(d), spans.to(d))
    full = run(w, do, dfin)
    composed = CP.compose_grads(list(trs), list(loc), dfin[0].to(d))[-1]
    e = rel(composed.cpu().numpy(), full[0].cpu().numpy())
    print(f"[parity] summary_bwd span composition: {e:.2e}")
    assert e <= F32_TOL


def test_summary_bwd_long_spans_sampled():
    """The long-sequence span workload (131072 tokens, 8 spans of 16384, H = 16, K = V = 128): the
    oracle recomputes two sampled (span, head) units."""
    w = W.config(5)
    do, _ = cotangents(w, 561, with_final=False)
    got = run(w, do, None, cu=w.spans).cpu().numpy()
    cu = w.spans.numpy().astype(np.int64)
    errs = []
    for i, h in [(0, 0), (7, 11)]:
        sl = slice(cu[i], cu[i + 1])
        ref = oracle.gdn_summary_bwd(w.q[sl, h:h + 1], w.k[sl, h:h + 1], w.g[sl, h:h + 1], w.beta[sl, h:h + 1],
                                     np.array([0, cu[i + 1] - cu[i]]), do[sl, h:h + 1])
        errs.append(rel(got[i, h], ref[0, 0]))
    print("[parity] summary_bwd long spans sampled: " + ", ".join(f"{e:.2e}" for e in errs))
    assert max(errs) <= F32_TOL


def test_summary_bwd_bad_cu_seqlens_sets_status():
    """A decreasing cu_seqlens is a value error: the status word says so and nothing is computed."""
    d = dev()
    w = W.draw("sbwd bad", [64, 64], 1, 1, 64, 64, seed=571)
    do, _ = cotangents(w, 572, with_final=False)
    bad = torch.tensor([0, 100, 64], dtype=torch.int32, device=d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    la.gdn_summary_bwd(w.q.to(d), w.k.to(d), w.g.to(d), w.beta.to(d), bad, do.to(d), status=status)
    assert la.read_status(status) != 0


def test_summary_bwd_with_input_transforms():
    """The forward's input transforms on g and beta (softplus gate, beta sigmoid) apply here too."""
    w = W.draw("sbwd transforms", [300, 64, 129], 2, 2, 128, 128, seed=581)
    gen = torch.Generator().manual_seed(582)
    g_raw = torch.randn(w.T, w.HV, generator=gen)
    b_logit = torch.randn(w.T, w.HV, generator=gen)
    a_log = torch.log(0.02 + 0.08 * torch.rand(w.HV, generator=gen))
    dt_bias = 0.5 * torch.randn(w.HV, generator=gen)
    do, dfin = cotangents(w, 583)
    d = dev()
    status = torch.zeros(1, dtype=torch.int32, device=d)
    got = la.gdn_summary_bwd(w.q.to(d), w.k.to(d), g_raw.to(d), b_logit.to(d), w.cu_seqlens.to(d), do.to(d),
                             d_final_state=dfin.to(d), status=status, a_log=a_log.to(d), dt_bias=dt_bias.to(d),
                             beta_sigmoid=True)
    assert la.read_status(status) == 0
    ref = oracle.gdn_summary_bwd(w.q, w.k, g_raw, b_logit, w.cu_seqlens, do, d_final_state=dfin, gate="softplus",
                                 a_log=a_log, dt_bias=dt_bias, beta_sigmoid=True)
    check(w, got, ref, " softplus gate + beta sigmoid")


def test_summary_bwd_tensor_core_pass_many_units_per_cta():
    """More (span, head) units than SMs (one state-gradient CTA per SM), so CTAs walk several
    units in turn, ragged spans included: the tensor-core pass against the tile kernel, and every
    span bitwise the same alone as inside the batch."""
    lengths = [0, 1, 63, 64, 65, 127, 128, 129, 191, 192, 0, 700, 255, 256, 257, 3, 511, 640,
               130, 0, 65, 200, 1000, 64, 2, 450, 129, 320, 0, 190, 66, 777,
               128, 1, 256, 380, 0, 193, 64, 900, 40, 129, 600, 192, 5, 333, 70, 128]
    w = W.draw("sbwd many units", lengths, 4, 8, 64, 64, seed=561, slow_decay=True)
    assert w.N * w.HV > torch.cuda.get_device_properties(0).multi_processor_count
    do, dfin = cotangents(w, 562)
    tc = run(w, do, dfin)
    tile = run(w, do, dfin, passes=1)
    e = rel(tc.cpu().numpy(), tile.cpu().numpy())
    print(f"[parity] summary_bwd many units: tensor-core pass vs tile kernel {e:.2e}")
    assert e <= F32_TOL
    cu = w.cu_seqlens.numpy().astype(np.int64)
    for i in (2, 11, 22, 39):
        sl = slice(cu[i], cu[i + 1])
        sub = W.Workload(name="one", cu_seqlens=torch.tensor([0, cu[i + 1] - cu[i]]), q=w.q[sl], k=w.k[sl], v=w.v[sl],
                         g=w.g[sl].contiguous(), beta=w.beta[sl].contiguous())
        alone = run(sub, do[sl], dfin[i:i + 1])
        assert torch.equal(tc[i], alone[0]), i


def test_summary_bwd_unaligned_d_o_takes_the_tile_kernel():
    """d_o whose rows are not in 16-byte units cannot be read by TMA: the call takes the tile
    kernel, with the tile kernel's exact result."""
    w = W.draw("sbwd odd d_o", [70, 129], 2, 2, 64, 64, seed=571, slow_decay=True)
    do, dfin = cotangents(w, 572)
    d = dev()
    wide = torch.zeros(w.T, w.HV, w.V + 1, dtype=torch.bfloat16)
    wide[:, :, :w.V] = do
    view = wide.to(d)[:, :, :w.V]  # row stride HV * (V + 1) elements: not a multiple of 8
    assert view.stride(0) % 8 != 0
    status = torch.zeros(1, dtype=torch.int32, device=d)
    got = la.gdn_summary_bwd(w.q.to(d), w.k.to(d), w.g.to(d), w.beta.to(d), w.cu_seqlens.to(d), view,
                             d_final_state=dfin.to(d), status=status)
    assert la.read_status(status) == 0
    assert torch.equal(got, run(w, do, dfin, passes=1))
