"""The internal workspace grows without synchronising, and refuses to grow under capture.

A call with workspace = NULL uses one buffer per device that the library grows on demand.
The header promises that no call synchronises: growth must not wait for work already on the
GPU (here a spin kernel on another stream), and inside a stream capture, where allocation is
not allowed, a call that would need a larger buffer must return LA_ERR_WORKSPACE and launch
nothing.  The growth itself is checked on the fused forward (whose workspace depends on N
alone); then, with the automatic choice back, a captured call whose two-pass workspace does
not fit the buffer but whose fused one does falls back to the fused kernel and succeeds.  The
scenario runs in a fresh process so that the buffer starts empty whatever the other tests did.
"""
import os
import subprocess
import sys
import textwrap

import pytest
import torch

pytestmark = pytest.mark.gpu

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent(r"""
    import ctypes, sys, time
    import torch
    sys.path.insert(0, sys.argv[1])
    from gated_delta_rule_29_gb300 import binding as B

    lib = B.load()
    assert lib.la_test_set_fwd_passes(1) == 0  # the fused forward: a workspace of N alone
    d = torch.device("cuda:0")
    gen = torch.Generator(device=d).manual_seed(3)

    def inputs(N):
        # N one-token sequences, one head, K = V = 64
        T = N
        q, k, v = (torch.randn(T, 1, 64, device=d, generator=gen).to(torch.bfloat16) for _ in range(3))
        g = -torch.rand(T, 1, device=d, generator=gen)
        beta = torch.rand(T, 1, device=d, generator=gen)
        cu = torch.arange(N + 1, dtype=torch.int32, device=d)
        o = torch.empty(T, 1, 64, dtype=torch.bfloat16, device=d)
        status = torch.full((1,), -1, dtype=torch.int32, device=d)
        return q, k, v, g, beta, cu, o, status

    def call(t, stream):
        q, k, v, g, beta, cu, o, status = t
        p = B.GdnFwdParams()
        p.q, p.q_stride_t, p.q_stride_h = q.data_ptr(), q.stride(0), q.stride(1)
        p.k, p.k_stride_t, p.k_stride_h = k.data_ptr(), k.stride(0), k.stride(1)
        p.v, p.v_stride_t, p.v_stride_h = v.data_ptr(), v.stride(0), v.stride(1)
        p.g, p.g_stride_t, p.g_stride_h = g.data_ptr(), g.stride(0), g.stride(1)
        p.beta, p.beta_stride_t, p.beta_stride_h = beta.data_ptr(), beta.stride(0), beta.stride(1)
        p.cu_seqlens, p.cu_seqlens_bits = cu.data_ptr(), 32
        p.T, p.N, p.HK, p.HV, p.K, p.V = q.shape[0], cu.numel() - 1, 1, 1, 64, 64
        p.scale, p.use_qk_l2norm = 0.125, 1
        p.o, p.o_stride_t, p.o_stride_h = o.data_ptr(), o.stride(0), o.stride(1)
        p.status = status.data_ptr()
        return lib.gdn_fwd(ctypes.byref(p), stream)   # workspace NULL: the internal buffer

    main = torch.cuda.current_stream()
    small = inputs(16)
    assert call(small, main.cuda_stream) == B.LA_OK          # first use: a 1 MB buffer
    torch.cuda.synchronize()
    big = inputs(100000)                                      # needs ~2.3 MB: the buffer grows
    huge = inputs(200000)                                     # needs ~4.5 MB
    torch.cuda.synchronize()

    # growth while a spin kernel runs on another stream: the call must not wait for it
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        torch.cuda._sleep(3_000_000_000)
    spin_done = torch.cuda.Event()
    spin_done.record(side)
    t0 = time.perf_counter()
    rc = call(big, main.cuda_stream)
    dt = time.perf_counter() - t0
    still_spinning = not spin_done.query()
    assert rc == B.LA_OK, rc
    assert still_spinning, "the spin kernel finished before the growing call returned"
    assert dt < 0.5, dt
    torch.cuda.synchronize()
    assert int(big[7].item()) == B.LA_OK
    assert torch.isfinite(big[6].float()).all()

    # under stream capture: no growth (LA_ERR_WORKSPACE, nothing launched); a call that fits
    # the current buffer is captured and replays
    cap = torch.cuda.Stream()
    cap.wait_stream(main)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        rc_huge = call(huge, cap.cuda_stream)
        rc_small = call(small, cap.cuda_stream)
    assert rc_huge == B.LA_ERR_WORKSPACE, rc_huge
    assert rc_small == B.LA_OK, rc_small
    small[7].fill_(-1)
    graph.replay()
    torch.cuda.synchronize()
    assert int(small[7].item()) == B.LA_OK
    # outside the capture the same large call grows the buffer and runs
    assert call(huge, main.cuda_stream) == B.LA_OK
    torch.cuda.synchronize()
    assert int(huge[7].item()) == B.LA_OK

    # automatic choice: the two-pass workspace of `big` (about 1.8 GB) is beyond the buffer, so
    # under capture the call takes the fused kernel, whose workspace fits, and succeeds
    assert lib.la_test_set_fwd_passes(0) == 0
    need = lib.la_gdn_fwd_split_workspace_bytes(100000, 100000, 1)
    assert need > 1 << 30
    big[7].fill_(-1)
    graph2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph2, stream=cap):
        rc_fallback = call(big, cap.cuda_stream)
    assert rc_fallback == B.LA_OK, rc_fallback
    graph2.replay()
    torch.cuda.synchronize()
    assert int(big[7].item()) == B.LA_OK
    print("growth ok", round(dt * 1e3, 2), "ms")
""")


def test_internal_workspace_grows_without_sync_and_refuses_under_capture():
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    r = subprocess.run([sys.executable, "-c", SCRIPT, REPO], capture_output=True, text=True, timeout=600)
    print(r.stdout[-2000:], r.stderr[-4000:])
    assert r.returncode == 0, r.stderr[-4000:]
    assert "growth ok" in r.stdout
