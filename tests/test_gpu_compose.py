"""Composition of span summaries on the GPU (gdn_compose_spans) and context parallelism on one GPU.

The page ("Summaries") composes consecutive spans as S_final = S_init * transition + S_H; the
library's kernel does it for the forward (the state entering every span) and, in reverse, for
a state gradient.  It is checked against the oracle's fp64 composition on random inputs, then
end to end: a sequence cut into spans, each span's gdn_summary, the composed entering states
and a gdn_fwd per span from them reproduce the unsplit forward, and the composed state
gradients reproduce the unsplit backward's entering-state gradient.
"""
import numpy as np
import pytest
import torch

import oracle
import gated_delta_rule_29_gb300 as la
from gated_delta_rule_29_gb300 import context_parallel as cp
from gated_delta_rule_29_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def rel(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


@pytest.mark.parametrize("K,V", [(128, 128), (64, 128), (128, 64), (64, 64)])
@pytest.mark.parametrize("R", [0, 1, 5])
@pytest.mark.parametrize("with_start", [True, False])
def test_compose_matches_oracle(K, V, R, with_start):
    d = dev()
    HO = 3
    gen = torch.Generator().manual_seed(801 + K + V + R)
    trs = torch.randn(R, HO, K, K, generator=gen) / K ** 0.5
    terms = torch.randn(R, HO, K, V, generator=gen)
    start = torch.randn(HO, K, V, generator=gen) if with_start else None
    s_np = start.numpy() if with_start else np.zeros((HO, K, V))
    for backward in (False, True):
        got = la.api.compose_spans(trs.to(d), terms.to(d), None if start is None else start.to(d),
                                   backward=backward).cpu().numpy()
        if backward:
            ref = oracle.compose_span_grads(list(trs.numpy()), list(terms.numpy()), s_np)
        else:
            ref = oracle.compose_spans(list(trs.numpy()), list(terms.numpy()), s_np)
        assert got.shape == (R + 1, HO, K, V)
        for j in range(R + 1):
            assert rel(got[j], ref[j]) <= 1e-5, (backward, j, rel(got[j], ref[j]))


def test_context_parallel_forward_on_one_gpu():
    """Spans of one sequence: summaries, composition, a forward per span from its entering state:
    the outputs and the final state match the unsplit forward from the same nonzero start."""
    d = dev()
    L = 3000
    w = W.draw("cp spans", [L], 2, 4, 128, 128, seed=811, slow_decay=True)
    cuts = [0, 640, 1000, 1001, 2048, L]  # a one-token span, spans not on chunk boundaries
    gen = torch.Generator().manual_seed(812)
    s_init = (0.1 * torch.randn(1, w.HV, w.K, w.V, generator=gen)).to(d)
    t = {n: getattr(w, n).to(d) for n in ("q", "k", "v", "g", "beta")}
    spans = torch.tensor(cuts, dtype=torch.int32, device=d)
    end, tr = la.gdn_summary(t["k"], t["v"], t["g"], t["beta"], spans)
    entering = cp.compose(list(tr), list(end), s_init[0])
    assert len(entering) == len(cuts)
    o_parts, fin = [], None
    for j, (a, b) in enumerate(zip(cuts[:-1], cuts[1:])):
        cu = torch.tensor([0, b - a], dtype=torch.int32, device=d)
        o, fin, _ = la.gdn_fwd(t["q"][a:b], t["k"][a:b], t["v"][a:b], t["g"][a:b].contiguous(),
                               t["beta"][a:b].contiguous(), cu, initial_state=entering[j][None])
        o_parts.append(o)
    cu_all = torch.tensor([0, L], dtype=torch.int32, device=d)
    o_full, fin_full, _ = la.gdn_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], cu_all, initial_state=s_init)
    e_fin = rel(fin.cpu().numpy(), fin_full.cpu().numpy())
    e_cmp = rel(entering[-1].cpu().numpy(), fin_full[0].cpu().numpy())
    e_o = rel(torch.cat(o_parts).float().cpu().numpy(), o_full.float().cpu().numpy())
    print(f"[parity] context parallel on one GPU: final {e_fin:.2e}, composed final {e_cmp:.2e}, o {e_o:.2e}")
    assert e_fin <= 2e-3 and e_cmp <= 2e-3 and e_o <= 1e-2


def test_context_parallel_backward_on_one_gpu():
    """The reverse composition of per-span state gradients (gdn_summary_bwd, zero exit cotangent)
    with the spans' transitions equals the unsplit summary backward's entering-state gradient."""
    d = dev()
    L = 2500
    w = W.draw("cp bwd spans", [L], 2, 4, 128, 64, seed=821, slow_decay=True)
    cuts = [0, 700, 701, 1600, L]
    gen = torch.Generator().manual_seed(822)
    do = torch.randn(L, w.HV, w.V, generator=gen).to(torch.bfloat16).to(d)
    dfin = torch.randn(1, w.HV, w.K, w.V, generator=gen).to(d)
    t = {n: getattr(w, n).to(d) for n in ("q", "k", "v", "g", "beta")}
    spans = torch.tensor(cuts, dtype=torch.int32, device=d)
    loc = la.gdn_summary_bwd(t["q"], t["k"], t["g"], t["beta"], spans, do)
    _, tr = la.gdn_summary(t["k"], t["v"], t["g"], t["beta"], spans)
    composed = cp.compose_grads(list(tr), list(loc), dfin[0])
    whole = la.gdn_summary_bwd(t["q"], t["k"], t["g"], t["beta"], torch.tensor([0, L], dtype=torch.int32, device=d),
                               do, d_final_state=dfin)
    e = rel(composed[-1].cpu().numpy(), whole[0].cpu().numpy())
    print(f"[parity] context-parallel backward on one GPU: {e:.2e}")
    assert e <= 2e-3
