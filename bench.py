"""Benchmark: chunked GDN forward tokens/s and fraction of the GB300 roofline.

Workload (one step = one gdn_fwd over the whole batch: the prologue, the WY pass and the
state pass): the dense batch of 8 sequences x 8192 tokens (T = 65536), 32 heads,
K = V = 128, bf16 q/k/v, fp32 g/beta, fp32 initial state, final state and fp32
checkpoints every 1024 tokens, q/k L2-normalised in kernel.  Inputs are seeded
synthetic tensors with the cuDNN page's distributions; q/k/v alone are 1.6 GB per
step, far larger than the 129 MB L2, so no flush is needed between steps.

Multi-GPU (torchrun): every rank runs its own copy of the batch (independent
sequences, no data-path collective: weak scaling); value = tokens of all ranks /
the slowest rank's time.

--impl reference times the fp64 CPU oracle (the parity oracle, untuned) on a
bounded sample of the same workload on the host cores (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GDN fwd tokens/s and % of GB300 roofline (T=65536,H=32,K=V=128 bf16)"
WORKLOAD = "dense batch: N=8 x 8192 tokens (T=65536), H=32, K=V=128, bf16 q/k/v, fp32 start state, " \
           "final state and fp32 checkpoints every 1024 tokens, q/k L2 norm in kernel"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def algorithmic_bytes(T, N, HK, HV, K, V, ckpt_rows, s0=True, final=True, ckpt_bytes=4):
    """Bytes the forward must move at least once: inputs read, outputs written."""
    HO = HV
    b = T * (2 * HK * K + HV * V) * 2      # q, k, v
    b += T * HO * V * 2                    # o
    b += 2 * T * HO * 4                    # g, beta
    b += N * HO * K * V * 4 if s0 else 0   # initial state
    b += N * HO * K * V * 4 if final else 0
    b += ckpt_rows * HO * K * V * ckpt_bytes
    b += (N + 1) * 4                       # cu_seqlens
    return b


def algorithmic_flops(lengths, HO, K, V):
    """Chunked-form tensor work per 64-token chunk and head: KK^T, QK^T, T*(beta V),
    T*(beta gamma K), the intra-chunk output (5 x 2 C^2 d) plus W S, Q S and the
    state update (3 x 2 C d^2), with d = K = V."""
    chunks = sum((int(L) + 63) // 64 for L in lengths)
    C = 64
    per = 2 * C * C * K * 2 + 2 * C * C * V * 3 + 2 * C * K * V * 3
    return chunks * HO * per


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", FALLBACK_BF16_TFLOPS)), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


# the sources that decide the forward's two kernels' code and launch (their DRAM traffic)
TRAFFIC_SOURCES = ("gdn_chunk.cu", "gdn_prologue.cu", "ptx.cuh", "la_api.cu")


def _code_only(text):
    """C++ source without comments or blank lines (a comment edit does not change the kernel)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = [re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines()]
    return "\n".join(ln for ln in lines if ln.strip())


def kernel_source_hash():
    h = hashlib.sha256()
    d = os.path.join(ROOT, "gated_delta_rule_29_gb300", "csrc")
    for name in TRAFFIC_SOURCES:
        h.update(_code_only(open(os.path.join(d, name)).read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per call of the forward's two passes (the WY pass and the state pass) from the
    committed ncu summary, if it was taken from the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "gdn_fwd_two_pass_dense_batch.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    return d.get("traffic_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n_, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n_)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def oracle_sample(w, units, nthreads):
    """Runs the CPU oracle on the given (sequence, head) units; returns (seconds, token-heads).

    Only the sampled sequences are sliced out and converted to fp64 before the clock starts;
    the timed call is the oracle's recurrence on exactly those units."""
    import oracle
    seqs = sorted({i for i, _ in units})
    cu = w.cu_seqlens.numpy().astype(np.int64)
    idx = np.concatenate([np.arange(cu[i], cu[i + 1]) for i in seqs])
    lens = [int(cu[i + 1] - cu[i]) for i in seqs]
    sub_cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    f64 = lambda x: np.ascontiguousarray(x.float().numpy(), dtype=np.float64)
    q, k, v, g, b = (f64(x[idx]) for x in (w.q, w.k, w.v, w.g, w.beta))
    s0 = None if w.initial_state is None else f64(w.initial_state[seqs])
    mask = np.zeros((len(seqs), w.HV), dtype=bool)
    for i, h in units:
        mask[seqs.index(i), h] = True
    t0 = time.perf_counter()
    oracle.gdn_fwd(q, k, v, g, b, sub_cu, initial_state=s0, checkpoint_every_n=w.checkpoint_every_n,
                   unit_mask=mask, nthreads=nthreads)
    dt = time.perf_counter() - t0
    return dt, int(sum(lens[seqs.index(i)] for i, _ in units))


def cpu_units(w, count):
    """The first `count` (sequence, head) units of a fixed interleaved order over the batch
    (all of them when count >= N * HO)."""
    units = [(i, h) for h in range(w.HV) for i in range(w.N)]
    return units[:min(count, len(units))]


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    from gated_delta_rule_29_gb300 import workloads as W
    w = W.config(3)
    cores = os.cpu_count() or 1
    # one (sequence, head) unit per host core per step unless told otherwise: every core works
    units = cpu_units(w, args.ref_units if args.ref_units else min(cores, w.N * w.HV))
    cores = min(cores, len(units))  # threads that actually run
    for _ in range(args.warmup):
        oracle_sample(w, units[:1], cores)
    times, th = [], 0
    for _ in range(args.steps):
        dt, n = oracle_sample(w, units, cores)
        times.append(dt)
        th += n
    total = sum(times)
    tokens_per_s = th / w.HV / total  # token-heads -> tokens of all HO heads
    line = {
        "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": WORKLOAD, "sample": f"{len(units)} (sequence, head) units x 8192 tokens per step"},
        "cpu_baseline": {"value": tokens_per_s, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{len(units)} of 256 (sequence, head) units of the workload per step, "
                                   f"fp64 token-by-token C recurrence, {cores} threads"},
        "e2e": {"value": tokens_per_s, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, world, rank, local):
    import gated_delta_rule_29_gb300 as la
    from gated_delta_rule_29_gb300 import binding as B
    from gated_delta_rule_29_gb300 import workloads as W

    assert torch.cuda.is_available(), "bench needs a CUDA device (there is no CPU fallback)"
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lib = B.load()
    if args.seq_len == 8192:
        w = W.config(3)
    else:  # a smaller dense batch of the same shape family (profiling captures)
        w = W.draw(f"dense batch N=8 x {args.seq_len}", [args.seq_len] * 8, 32, 32, 128, 128, seed=1003,
                   initial_state=True, checkpoint_every_n=1024, checkpoint_dtype=torch.float32)
    T, N, HK, HV, K, V = w.T, w.N, w.HK, w.HV, w.K, w.V
    HO = HV
    n_ck = w.checkpoint_every_n
    R = la.checkpoint_rows(w.cu_seqlens, n_ck)

    # device-resident inputs and outputs
    q, k, v = w.q.to(dev), w.k.to(dev), w.v.to(dev)
    g, beta = w.g.to(dev), w.beta.to(dev)
    cu = w.cu_seqlens.to(dev)
    s0 = w.initial_state.to(dev)
    o = torch.empty(T, HO, V, dtype=torch.bfloat16, device=dev)
    fin = torch.empty(N, HO, K, V, dtype=torch.float32, device=dev)
    ck = torch.empty(R, HO, K, V, dtype=torch.float32, device=dev)
    ws = torch.empty(la.api.split_workspace_bytes(T, N, HV), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step(qq=q, kk=k, vv=v, gg=g, bb=beta, cc=cu, ss=s0, oo=o, ff=fin, kc=ck):
        la.gdn_fwd(qq, kk, vv, gg, bb, cc, initial_state=ss, checkpoint_every_n=n_ck,
                   checkpoint_dtype=torch.float32, checkpoint_rows_hint=R, o=oo, final_state=ff,
                   checkpoints=kc, workspace=ws, status=status)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert la.read_status(status) == 0, "device status after warm-up"

    stream = torch.cuda.current_stream()
    k_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a_, b_ in k_ev:  # torch creates the underlying cudaEvent_t on first record
        a_.record(stream)
        b_.record(stream)
    torch.cuda.synchronize()
    assert all(a_.cuda_event and b_.cuda_event for a_, b_ in k_ev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(args.steps):
            lib.la_set_kernel_timing_events(k_ev[i][0].cuda_event, k_ev[i][1].cuda_event)
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    ms_local = e0.elapsed_time(e1) / args.steps
    kern_ms = statistics.mean(a.elapsed_time(b) for a, b in k_ev)
    ms = max_over_ranks(ms_local, world)
    assert la.read_status(status) == 0, "device status after the timed region"

    tokens = T * world
    value = tokens / (ms * 1e-3)
    hbm_peak, tc_peak, peak_src = load_peaks()
    alg_bytes = algorithmic_bytes(T, N, HK, HV, K, V, R)
    alg_flops = algorithmic_flops(w.lengths(), HO, K, V)
    achieved = alg_bytes / (kern_ms * 1e-3) / 1e9
    tflops = alg_flops / (kern_ms * 1e-3) / 1e12

    # end to end through the public API with host buffers: gdn_fwd_host copies the step's inputs
    # from pinned host memory, runs the forward and copies o, the final state and the checkpoints
    # back, pipelined over token ranges (long sequences cut into pieces that hand their fp32
    # state on); all of it inside the timed region
    host_in = [x.pin_memory() for x in (w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, w.initial_state)]
    host_out = (torch.empty(o.shape, dtype=o.dtype).pin_memory(), torch.empty(fin.shape).pin_memory(),
                torch.empty(ck.shape, dtype=ck.dtype).pin_memory())
    h2d = sum(x.numel() * x.element_size() for x in host_in)
    d2h = sum(x.numel() * x.element_size() for x in host_out)
    # two staging buffers used in turn: a step's copies in only wait for the step before last
    # (the one that used the same buffer), so they run under the previous step's last forward
    staging = ({}, {})
    e2e_count = [0]

    def e2e_step():
        hq, hk, hv, hg, hb, hcu, hs0 = host_in
        la.gdn_fwd_host(hq, hk, hv, hg, hb, hcu, initial_state=hs0, checkpoint_every_n=n_ck,
                        checkpoint_dtype=torch.float32, out=host_out, device=dev, groups=args.e2e_groups,
                        staging=staging[e2e_count[0] % 2])
        e2e_count[0] += 1

    e2e = None
    if not args.no_e2e:
        e2e_steps = max(3, min(args.steps, 10))
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        x0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        x1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        e2e_ms = max_over_ranks(x0.elapsed_time(x1) / e2e_steps, world)
        e2e = {"value": tokens / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "ranges": args.e2e_groups,
               "staging_buffers": 2, "entry": "gdn_fwd_host (C ABI, host buffers)"}
        assert torch.equal(host_out[0].view(torch.int16), o.cpu().view(torch.int16)), "e2e output differs"
        assert torch.equal(host_out[1], fin.cpu()) and torch.equal(host_out[2], ck.cpu()), "e2e states differ"

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = os.cpu_count() or 1
        units = cpu_units(w, args.cpu_units)
        dt, th = oracle_sample(w, units, cores)
        cpu = {"value": th / HO / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{len(units)} of {N * HO} (sequence, head) units x {w.lengths()[0]} tokens of the same "
                         f"workload ({dt:.1f} s), fp64 token-by-token C recurrence on {cores} threads"}

    qkv_bytes = sum(t.numel() * t.element_size() for t in (w.q, w.k, w.v))
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD if args.seq_len == 8192 else w.name, "global_batch": N * world,
                       "seq_len": args.seq_len,
                       "parallelism": f"independent batches per GPU x{world}" if world > 1 else "single GPU",
                       "l2": f"inputs larger than L2 ({qkv_bytes / 1e9:.2f} GB of q/k/v per step); no flush"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak,
                         # (the recorded traffic is the dense batch's: another length has none)
                         "traffic": (None if args.fwd_passes == "fused" or args.seq_len != 8192
                                     else profiled_traffic()),
                         "peak_source": peak_src,
                         "kernel": ("gdn_chunk_kernel<128, fwd> (fused)" if args.fwd_passes == "fused" else
                                    "gdn_wy_kernel<128> + gdn_chunk_kernel<128, state pass> (timed together)"),
                         "kernel_ms": kern_ms, "algorithmic_bytes": alg_bytes,
                         "tensor_tflops": tflops, "tensor_frac": tflops / tc_peak},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": (2 if args.fwd_passes == "fused" else 3) * args.steps,  # prologue, (WY pass,) state pass
            "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    return 0


DECODE_METRIC = "GDN decode tokens/s and % of GB300 HBM roofline (N=1024 sequences, H=32, K=V=128, fp32 state pool)"


def run_decode(args, world, rank, local):
    """One decode step = gdn_decode over N = 1024 sequences (one new token each), 32 heads,
    K = V = 128, against an fp32 state pool of 2048 slots (4.3 GB) with a random slot per
    sequence: the state is read and written once (4.3 GB of the 4.3 GB moved per step)."""
    import gated_delta_rule_29_gb300 as la
    from gated_delta_rule_29_gb300 import binding as B
    from gated_delta_rule_29_gb300 import workloads as W

    assert torch.cuda.is_available(), "bench needs a CUDA device (there is no CPU fallback)"
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lib = B.load()
    N, H, K, V, P = 1024, 32, 128, 128, 2048
    w = W.draw("decode step", [1] * N, H, H, K, V, seed=1006)
    gen = torch.Generator().manual_seed(1007)
    idx = torch.randperm(P, generator=gen)[:N].to(torch.int32)
    pool = torch.empty(P, H, K, V, dtype=torch.float32, device=dev)
    for s_ in range(0, P, 256):  # 0.1 N(0,1) states, drawn in slices on the device
        pool[s_:s_ + 256].normal_(0.0, 0.1, generator=torch.Generator(device=dev).manual_seed(1008 + s_))
    q, k, v, g, b, ix = (x.to(dev) for x in (w.q, w.k, w.v, w.g, w.beta, idx))
    o = torch.empty(N, H, V, dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        la.gdn_decode(q, k, v, g, b, pool, state_indices=ix, o=o, status=status)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert la.read_status(status) == 0
    stream = torch.cuda.current_stream()
    k_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a_, b_ in k_ev:
        a_.record(stream)
        b_.record(stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(args.steps):
            lib.la_set_kernel_timing_events(k_ev[i][0].cuda_event, k_ev[i][1].cuda_event)
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
    kern_ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in k_ev)
    assert la.read_status(status) == 0
    state_bytes = 2 * N * H * K * V * 4
    io_bytes = N * H * (2 * K * 2 + 2 * V * 2 + 2 * 4) + N * 4
    alg_bytes = state_bytes + io_bytes
    hbm_peak, _, peak_src = load_peaks()
    achieved = alg_bytes / (kern_ms * 1e-3) / 1e9

    # end to end: the step's token inputs from pinned host memory, o back to pinned host memory;
    # the pool is the serving state and stays on the device
    host_in = [x.pin_memory() for x in (w.q, w.k, w.v, w.g, w.beta, idx)]
    host_o = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in host_in)
    d2h = host_o.numel() * host_o.element_size()

    def e2e_step():
        qq, kk, vv, gg, bb, ii = (x.to(dev, non_blocking=True) for x in host_in)
        la.gdn_decode(qq, kk, vv, gg, bb, pool, state_indices=ii, o=o, status=status)
        host_o.copy_(o, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    x0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    x1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(x0.elapsed_time(x1) / args.steps, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle  # CPU baseline only
        cores = os.cpu_count() or 1
        m = 256  # sequences in the sample
        pool_s = pool[idx[:m].long().to(dev)].double().cpu().numpy()
        t0 = time.perf_counter()
        oracle.gdn_fwd(w.q[:m], w.k[:m], w.v[:m], w.g[:m], w.beta[:m], torch.arange(m + 1), initial_state=pool_s,
                       state_indices=torch.arange(m), nthreads=cores)
        dt = time.perf_counter() - t0
        cpu = {"value": m / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{m} of {N} sequences x {H} heads, one decode step ({dt:.2f} s), fp64 C recurrence "
                         f"on {cores} threads"}
    if rank == 0:
        line = {
            "metric": DECODE_METRIC, "value": N * world / (ms * 1e-3), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"decode step: N={N} sequences x 1 token, H={H}, K=V={K}, fp32 state pool of "
                                   f"{P} slots (random slot per sequence)", "global_batch": N * world,
                       "parallelism": "single GPU" if world == 1 else f"independent pools per GPU x{world}",
                       "l2": f"state moved per step {state_bytes / 1e9:.2f} GB > L2; no flush"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": None, "peak_source": peak_src,
                         "kernel": "gdn_decode_kernel<128, 128>", "kernel_ms": kern_ms, "algorithmic_bytes": alg_bytes},
            "cpu_baseline": cpu,
            "e2e": {"value": N * world / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": args.steps,
            "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    return 0


BWD_METRIC = "GDN bwd tokens/s (T=65536,H=32,K=V=128; gradients of q,k,v,g,beta,initial state)"
TF32_PER_BF16 = 1.1 / 2.25  # nominal dense tf32 / bf16 tensor rates of the part


def bwd_algorithmic_flops(lengths, HO, K, V, C=64):
    """Arithmetic of the chunked backward per (chunk, head), counted from its products: G and P
    (lower halves), the triangular inverse, K S / Q S / K dS, T Y, P^T dO, T^T dD, dA and dP
    (lower halves), the dK / dQ tile terms, the dS update and the A / P backward."""
    per = (2 * (C * (C + 1) // 2) * K * 2 + C ** 3 // 3 * 2 + 3 * C * K * V * 2 + 3 * C * C * V * 2
           + 2 * (C * (C + 1) // 2) * V * 2 + 3 * C * K * V * 2 + 2 * K * C * V * 2 + 3 * C * C * K * 2)
    chunks = sum((L + C - 1) // C for L in lengths)
    return int(per * chunks * HO)


def run_bwd_bench(args, world, rank, local):
    """One step = gdn_bwd over the dense batch, reusing the forward's fp32 checkpoints every 64
    tokens (the training flow: the forward dumps them, the backward reads them)."""
    import gated_delta_rule_29_gb300 as la
    from gated_delta_rule_29_gb300 import binding as B
    from gated_delta_rule_29_gb300 import workloads as W

    assert torch.cuda.is_available(), "bench needs a CUDA device (there is no CPU fallback)"
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lib = B.load()
    if args.seq_len == 8192:
        w = W.config(3)
    else:  # a smaller dense batch of the same shape family (profiling captures)
        w = W.draw(f"dense batch N=8 x {args.seq_len}", [args.seq_len] * 8, 32, 32, 128, 128, seed=1003,
                   initial_state=True)
    T, N, HK, HV, K, V = w.T, w.N, w.HK, w.HV, w.K, w.V
    L = args.seq_len
    gen = torch.Generator().manual_seed(1009)
    do_h = torch.randn(T, HV, V, generator=gen).to(torch.bfloat16)
    dfin_h = torch.randn(N, HV, K, V, generator=gen)
    q, k, v, g, b, cu, s0, do, dfin = (x.to(dev) for x in (w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens,
                                                            w.initial_state, do_h, dfin_h))
    # the checkpoints the backward is given: the forward's fp32 rows every --bwd-ckpt tokens (64:
    # the chunk cadence, read directly; larger: the dense series is regenerated segment by segment)
    # or none (the whole forward re-runs)
    ck_n = 0 if args.bwd_ckpt == "none" else int(args.bwd_ckpt)
    ck = None
    if ck_n:
        _, _, ck = la.gdn_fwd(q, k, v, g, b, cu, initial_state=s0, checkpoint_every_n=ck_n,
                              checkpoint_dtype=torch.float32)
    ws = torch.empty(lib.la_gdn_bwd_workspace_bytes_ckpt(T, N, HK, HV, K, V, ck_n, 0), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        return la.gdn_bwd(q, k, v, g, b, cu, do, initial_state=s0, d_final_state=dfin, checkpoints=ck,
                          checkpoint_every_n=ck_n if ck_n else 64, workspace=ws, status=status)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert la.read_status(status) == 0
    stream = torch.cuda.current_stream()
    k_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a_, b_ in k_ev:
        a_.record(stream)
        b_.record(stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(args.steps):
            lib.la_set_kernel_timing_events(k_ev[i][0].cuda_event, k_ev[i][1].cuda_event)
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
    kern_ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in k_ev)
    assert la.read_status(status) == 0
    flops = bwd_algorithmic_flops(w.lengths(), HV, K, V)
    _, bf16_peak, peak_src = load_peaks()
    # the tensor-core schedule (the default) computes on bf16 hi + lo tcgen05 operands (its peak:
    # the bf16 rate); the tile kernel (--fwd-passes fused) on split tf32 warp MMAs (the tf32 rate)
    tile = args.fwd_passes == "fused"
    tf32_peak = bf16_peak * TF32_PER_BF16
    tc_peak = tf32_peak if tile else bf16_peak
    achieved = flops / (kern_ms * 1e-3) / 1e12
    # launches per step: the prologue and the tile kernel's range launches (four ranges per unit
    # in one-wave launches when the units outnumber the SMs), or the prologue, the WY pass, the
    # state-gradient pass and the chunk-parallel pass
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    units = N * HV
    launches = (1 + (-(-units * 4 // sms) if units > sms else 1)) if tile else 4

    # end to end: the step's inputs, cotangents and checkpoints copied from pinned host memory,
    # the gradients copied back, all inside the timed region
    host_in = [x.pin_memory() for x in (w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, w.initial_state, do_h, dfin_h)]
    host_ck = ck.cpu().pin_memory() if ck is not None else None
    outs = step()
    host_out = [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in outs]
    h2d = sum(x.numel() * x.element_size() for x in host_in) + (host_ck.numel() * 4 if host_ck is not None else 0)
    d2h = sum(x.numel() * x.element_size() for x in host_out)

    def e2e_step():
        xs = [x.to(dev, non_blocking=True) for x in host_in]
        ckd = host_ck.to(dev, non_blocking=True) if host_ck is not None else None
        r = la.gdn_bwd(xs[0], xs[1], xs[2], xs[3], xs[4], xs[5], xs[7], initial_state=xs[6], d_final_state=xs[8],
                       checkpoints=ckd, checkpoint_every_n=ck_n if ck_n else 64, workspace=ws, status=status)
        for hbuf, dbuf in zip(host_out, r):
            hbuf.copy_(dbuf, non_blocking=True)

    e2e = None
    if not args.no_e2e:
        e2e_step()
        torch.cuda.synchronize()
        x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2e_steps = max(3, min(args.steps, 5))
        x0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        x1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(x0.elapsed_time(x1) / e2e_steps, world)
        e2e = {"value": T * world / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle  # CPU baseline only
        cores = os.cpu_count() or 1
        units = [(0, 0), (3, 5)]
        mask = np.zeros((N, HV), dtype=bool)
        for i_, h_ in units:
            mask[i_, h_] = True
        t0 = time.perf_counter()
        oracle.gdn_bwd(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, do_h, initial_state=w.initial_state,
                       d_final_state=dfin_h, unit_mask=mask, nthreads=cores)
        dt = time.perf_counter() - t0
        cpu = {"value": len(units) * L / HV / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{len(units)} of {N * HV} (sequence, head) units x {L} tokens ({dt:.1f} s), fp64 reverse "
                         f"mode of the token recurrence, up to {cores} threads (one per unit)"}
    if rank == 0:
        line = {
            "metric": BWD_METRIC, "value": T * world / (ms * 1e-3), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": (WORKLOAD if L == 8192 else w.name) + (
                           f"; bwd with the forward's fp32 checkpoints every {ck_n} tokens" if ck_n else
                           "; bwd without checkpoints (the forward re-runs)"), "global_batch": N * world, "seq_len": L,
                       "parallelism": "single GPU" if world == 1 else f"independent batches per GPU x{world}",
                       "l2": "inputs larger than L2 (1.6 GB of q/k/v + 2.1 GB of checkpoints per step); no flush"},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s",
                         "frac": achieved / tc_peak, "traffic": None,
                         "peak_source": (f"{peak_src} bf16 x {TF32_PER_BF16:.3f} (nominal dense tf32 / bf16); "
                                         "each fp32 product is 2-3 tf32 MMAs (head and remainder splits)" if tile else
                                         f"{peak_src} bf16; fp32-level products are 2-3 bf16 tcgen05 MMAs (hi and lo "
                                         "splits)"),
                         "kernel": ("gdn_bwd_kernel<128, 128>" if tile else
                                    "gdn_wy_kernel<128> + gdn_grad_kernel<128> + gdn_dchunk_kernel (timed together)"),
                         "kernel_ms": kern_ms, "algorithmic_flops": flops},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": args.steps * launches,
            "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    return 0


GDP_METRIC = "GDP fwd tokens/s and % of GB300 HBM roofline (T=65536 tokens x 2 updates, H=32, K=V=128)"


def run_gdp_bench(args, world, rank, local):
    """Gated DeltaProduct with 2 updates per token on the dense batch's shape: 8 x 8192 tokens,
    32 heads, K = V = 128, q and g per token, k, v and beta per update, start and final state."""
    import gated_delta_rule_29_gb300 as la
    from gated_delta_rule_29_gb300 import binding as B

    assert torch.cuda.is_available(), "bench needs a CUDA device (there is no CPU fallback)"
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lib = B.load()
    n, N, L, H, K, V = 2, 8, 8192, 32, 128, 128
    T = N * L
    gen = torch.Generator().manual_seed(1010)
    q_h = torch.randn(T, H, K, generator=gen).to(torch.bfloat16)
    k_h = torch.randn(T * n, H, K, generator=gen).to(torch.bfloat16)
    v_h = torch.randn(T * n, H, V, generator=gen).to(torch.bfloat16)
    g_h = -torch.nn.functional.softplus(torch.randn(T, H, generator=gen))
    b_h = torch.sigmoid(torch.randn(T * n, H, generator=gen))
    s0_h = 0.1 * torch.randn(N, H, K, V, generator=gen)
    cu_h = torch.arange(0, T + 1, L, dtype=torch.int32)
    q, k, v, g, b, cu, s0 = (x.to(dev) for x in (q_h, k_h, v_h, g_h, b_h, cu_h, s0_h))
    o = torch.empty(T, H, V, dtype=torch.bfloat16, device=dev)
    fin = torch.empty(N, H, K, V, dtype=torch.float32, device=dev)
    ws = torch.empty(lib.la_gdp_workspace_bytes(T, N, H, H, K, V, n), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        la.gdn_fwd(q, k, v, g, b, cu, initial_state=s0, o=o, final_state=fin, workspace=ws, status=status,
                   num_householder=n)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert la.read_status(status) == 0
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
    # algorithmic bytes: q, o, g per token; k, v, beta per update; start and final state
    alg = T * H * K * 2 + T * H * V * 2 + T * H * 4 + T * n * H * (K * 2 + V * 2 + 4) + 2 * N * H * K * V * 4
    hbm_peak, _, peak_src = load_peaks()
    achieved = alg / (ms * 1e-3) / 1e9
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle  # CPU baseline only
        cores = os.cpu_count() or 1
        mask = np.zeros((N, H), dtype=bool)
        mask[0, :cores] = True
        t0 = time.perf_counter()
        oracle.gdp_fwd(q_h, k_h, v_h, g_h, b_h, cu_h, n, initial_state=s0_h, unit_mask=mask, nthreads=cores)
        dt = time.perf_counter() - t0
        cpu = {"value": int(mask.sum()) * L / H / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{int(mask.sum())} of {N * H} (sequence, head) units x {L} tokens ({dt:.1f} s)"}
    if rank == 0:
        line = {
            "metric": GDP_METRIC, "value": T * world / (ms * 1e-3), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"GDP n={n}: N={N} x {L} tokens, H={H}, K=V={K}, fp32 start and final state",
                       "global_batch": N * world, "seq_len": L, "parallelism": "single GPU",
                       "l2": "inputs larger than L2; no flush"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": None, "peak_source": peak_src,
                         "kernel": "gdn_chunk_kernel<128, gdp> (whole step: prologue + kernel)",
                         "algorithmic_bytes": alg},
            "cpu_baseline": cpu,
            "e2e": None,
            "gpu_launches": 2 * args.steps,
            "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    return 0


SUM_METRIC = "GDN summary tokens/s and % of GB300 roofline (one 131072-token sequence, 8 spans, H=16, K=V=128)"


def run_summary_bench(args, world, rank, local):
    """gdn_summary over the context-parallel workload: one 131072-token sequence cut into 8 spans
    of 16384, 16 heads, K = V = 128: per span and head the end state from a zero start and the
    fp32 K x K transition."""
    import gated_delta_rule_29_gb300 as la
    from gated_delta_rule_29_gb300 import binding as B
    from gated_delta_rule_29_gb300 import workloads as W

    assert torch.cuda.is_available(), "bench needs a CUDA device (there is no CPU fallback)"
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lib = B.load()
    w = W.config(5)
    T, HK, HV, K, V = w.T, w.HK, w.HV, w.K, w.V
    k, v, g, b, spans = (x.to(dev) for x in (w.k, w.v, w.g, w.beta, w.spans))
    S = spans.numel() - 1
    end = torch.empty(S, HV, K, V, dtype=torch.float32, device=dev)
    tr = torch.empty(S, HV, K, K, dtype=torch.float32, device=dev)
    ws = torch.empty(la.api.split_workspace_bytes(T, S, HV), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        la.gdn_summary(k, v, g, b, spans, end_state=end, transition=tr, workspace=ws, status=status)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert la.read_status(status) == 0
    stream = torch.cuda.current_stream()
    k_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a_, b_ in k_ev:
        a_.record(stream)
        b_.record(stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(args.steps):
            lib.la_set_kernel_timing_events(k_ev[i][0].cuda_event, k_ev[i][1].cuda_event)
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
    kern_ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in k_ev)
    # algorithmic bytes: k, v (bf16), g, beta (fp32) in; end states and transitions (fp32) out
    alg = T * (HK * K + HV * V) * 2 + 2 * T * HV * 4 + S * HV * (K * V + K * K) * 4 + (S + 1) * 4
    # algorithmic tensor work per 64-token chunk and head: the value tile and the transition tile
    # each take K K^T, the K S product, T X, and the state update (K = V = 128)
    C = 64
    per_chunk = 2 * (2 * C * C * K + 2 * C * K * V + 2 * C * C * V + 2 * C * K * V)
    flops = per_chunk * (T // C) * HV
    hbm_peak, tc_peak, peak_src = load_peaks()
    achieved = alg / (kern_ms * 1e-3) / 1e9
    tflops = flops / (kern_ms * 1e-3) / 1e12
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle  # CPU baseline only
        cores = os.cpu_count() or 1
        mask = np.zeros((S, HV), dtype=bool)
        mask[0, :min(HV, cores)] = True
        t0 = time.perf_counter()
        oracle.gdn_summary(w.k, w.v, w.g, w.beta, w.spans, unit_mask=mask, nthreads=cores)
        dt = time.perf_counter() - t0
        cpu = {"value": int(mask.sum()) * (T // S) / HV / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{int(mask.sum())} of {S * HV} (span, head) units x {T // S} tokens ({dt:.1f} s), fp64 "
                         f"state and K x K transition recurrence"}
    if rank == 0:
        line = {
            "metric": SUM_METRIC, "value": T * world / (ms * 1e-3), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "summary: one sequence of 131072 tokens, 8 spans of 16384, H=16, K=V=128, zero start",
                       "global_batch": 1, "seq_len": T, "parallelism": "single GPU",
                       "l2": "inputs larger than L2 (1.07 GB of k/v per step); no flush"},
            # the binding roof: bytes at the copy bandwidth or the products at the bf16 rate
            "roofline": ({"bound": "tensor", "achieved": tflops, "peak": tc_peak, "unit": "TFLOP/s",
                          "frac": tflops / tc_peak, "hbm_gbs": achieved, "hbm_frac": achieved / hbm_peak}
                         if flops / (tc_peak * 1e12) > alg / (hbm_peak * 1e9) else
                         {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                          "frac": achieved / hbm_peak, "tensor_tflops": tflops, "tensor_frac": tflops / tc_peak})
                        | {"traffic": None, "peak_source": peak_src, "kernel": ("gdn_chunk_kernel<128, summary> (fused)" if args.fwd_passes == "fused" else
                                              "gdn_wy_kernel<128, summary> + gdn_chunk_kernel<128, summary state pass>"),
                           "kernel_ms": kern_ms, "algorithmic_bytes": alg, "algorithmic_flops": flops},
            "cpu_baseline": cpu,
            "e2e": None,
            "gpu_launches": 2 * args.steps,
            "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    return 0


def run_table(args, world, rank, local):
    """One line per configuration of the benchmark table: the forward on the tiny, varlen, dense-batch
    and skewed grouped-head workloads, and the summary on the span workload.  For each, the GPU
    call's and the fused kernel's time (CUDA events, mean over --steps after --warmup), tokens/s,
    the algorithmic bytes and FLOPs over the kernel time against the measured peaks, and the fp64
    oracle's rate on the host cores at one thread and at all cores, each on a bounded sample of
    the workload's (sequence, head) units, with the whole-workload oracle time those rates imply."""
    import oracle  # the CPU baseline columns only
    import gated_delta_rule_29_gb300 as la
    from gated_delta_rule_29_gb300 import binding as B
    from gated_delta_rule_29_gb300 import workloads as W

    assert torch.cuda.is_available(), "bench needs a CUDA device (there is no CPU fallback)"
    if rank != 0:
        return 0
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lib = B.load()
    hbm_peak, tc_peak, peak_src = load_peaks()
    cores = os.cpu_count() or 1
    stream = torch.cuda.current_stream()

    clock_log = []  # one clock record per timed configuration

    def timed(step):
        with ClockSampler(local) as clk:
            out = timed_inner(step)
        clock_log.append(clk.summary())
        return out

    def timed_inner(step):
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for a_, b_ in evs:
            a_.record(stream)
            b_.record(stream)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.steps):
            lib.la_set_kernel_timing_events(evs[i][0].cuda_event, evs[i][1].cuda_event)
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps, statistics.mean(a_.elapsed_time(b_) for a_, b_ in evs)

    def oracle_rates(w, units_1t, units_all, summary=False):
        def one(units, nthreads):
            if not summary:
                dt, th = oracle_sample(w, units, nthreads)
                return th / dt
            mask = np.zeros((w.N, w.HV), dtype=bool)
            for i, h in units:
                mask[i, h] = True
            t0 = time.perf_counter()
            oracle.gdn_summary(w.k, w.v, w.g, w.beta, w.cu_seqlens, unit_mask=mask, nthreads=nthreads)
            dt = time.perf_counter() - t0
            lens = w.lengths()
            return sum(int(lens[i]) for i, _ in units) / dt
        r1 = one(units_1t, 1)
        ra = one(units_all, cores)
        total = sum(int(L) for L in w.lengths()) * w.HV  # token-heads of the whole workload
        return {"tokens_per_s_1_thread": r1 / w.HV, "tokens_per_s_all_cores": ra / w.HV, "cores": cores,
                "sample_1_thread": f"{len(units_1t)} (sequence, head) units",
                "sample_all_cores": f"{len(units_all)} (sequence, head) units",
                "workload_s_1_thread": total / r1, "workload_s_all_cores": total / ra}

    def spread(w, count):
        """`count` (sequence, head) units spread over the batch (sequences of every length)."""
        units = [(i, h) for i in range(w.N) for h in range(w.HV) if w.lengths()[i] > 0]
        step_ = max(1, len(units) // count)
        return units[::step_][:count]

    rows = []
    for cfg in (1, 2, 3, 4):
        w = W.config(cfg)
        T, N, HK, HV, K, V = w.T, w.N, w.HK, w.HV, w.K, w.V
        t = [x.to(dev) for x in (w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens)]
        s0 = None if w.initial_state is None else w.initial_state.to(dev)
        n_ck = w.checkpoint_every_n
        R = la.checkpoint_rows(w.cu_seqlens, n_ck) if n_ck else 0
        o = torch.empty(T, HV, V, dtype=torch.bfloat16, device=dev)
        fin = torch.empty(N, HV, K, V, dtype=torch.float32, device=dev)
        ck = torch.empty(R, HV, K, V, dtype=torch.float32, device=dev) if n_ck else None
        ws = torch.empty(la.api.split_workspace_bytes(T, N, HV), dtype=torch.uint8, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)

        def step():
            la.gdn_fwd(*t, initial_state=s0, checkpoint_every_n=n_ck, checkpoint_dtype=torch.float32,
                       checkpoint_rows_hint=R, o=o, final_state=fin, checkpoints=ck, workspace=ws, status=status)

        call_ms, kern_ms = timed(step)
        assert la.read_status(status) == 0
        alg = algorithmic_bytes(T, N, HK, HV, K, V, R, s0=s0 is not None, final=True)
        flops = algorithmic_flops(w.lengths(), HV, K, V)
        units = [(i, h) for i in range(N) for h in range(HV) if w.lengths()[i] > 0]
        n1 = {1: len(units), 2: 8, 3: 2, 4: 8}[cfg]
        na = {1: len(units), 2: len(units), 3: 32, 4: 64}[cfg]
        rows.append({"workload": w.name, "op": "gdn_fwd", "T": T, "N": N, "HK": HK, "HV": HV, "K": K, "V": V,
                     "call_ms": call_ms, "kernel_ms": kern_ms, "tokens_per_s": T / (call_ms * 1e-3),
                     "algorithmic_bytes": alg, "hbm_gbs": alg / (kern_ms * 1e-3) / 1e9,
                     "hbm_frac": alg / (kern_ms * 1e-3) / 1e9 / hbm_peak,
                     "tensor_tflops": flops / (kern_ms * 1e-3) / 1e12,
                     "tensor_frac": flops / (kern_ms * 1e-3) / 1e12 / tc_peak, "clocks": clock_log[-1],
                     "oracle": oracle_rates(w, spread(w, n1), spread(w, na))})
        del t, o, fin, ck
    w = W.config(5)
    T, HK, HV, K, V = w.T, w.HK, w.HV, w.K, w.V
    k, v, g, b, spans = (x.to(dev) for x in (w.k, w.v, w.g, w.beta, w.spans))
    S = spans.numel() - 1
    end = torch.empty(S, HV, K, V, dtype=torch.float32, device=dev)
    tr = torch.empty(S, HV, K, K, dtype=torch.float32, device=dev)
    ws = torch.empty(la.api.split_workspace_bytes(T, S, HV), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    call_ms, kern_ms = timed(lambda: la.gdn_summary(k, v, g, b, spans, end_state=end, transition=tr, workspace=ws,
                                                    status=status))
    assert la.read_status(status) == 0
    alg = T * (HK * K + HV * V) * 2 + 2 * T * HV * 4 + S * HV * (K * V + K * K) * 4 + (S + 1) * 4
    C = 64
    flops = 2 * (2 * C * C * K + 2 * C * K * V + 2 * C * C * V + 2 * C * K * V) * (T // C) * HV
    ws5 = W.Workload(name=w.name + " (span summaries)", cu_seqlens=w.spans, q=w.k, k=w.k, v=w.v, g=w.g, beta=w.beta)
    rows.append({"workload": w.name, "op": "gdn_summary (8 spans)", "T": T, "N": S, "HK": HK, "HV": HV, "K": K,
                 "V": V, "call_ms": call_ms, "kernel_ms": kern_ms, "tokens_per_s": T / (call_ms * 1e-3),
                 "algorithmic_bytes": alg, "hbm_gbs": alg / (kern_ms * 1e-3) / 1e9,
                 "hbm_frac": alg / (kern_ms * 1e-3) / 1e9 / hbm_peak,
                 "tensor_tflops": flops / (kern_ms * 1e-3) / 1e12, "tensor_frac": flops / (kern_ms * 1e-3) / 1e12 / tc_peak,
                 "clocks": clock_log[-1],
                 "oracle": oracle_rates(ws5, [(0, 0)], [(0, h) for h in range(min(HV, cores))], summary=True)})
    for r_ in rows:
        r_["peak_source"] = peak_src
        print(json.dumps(r_), flush=True)
    return 0


SUM_BWD_METRIC = ("GDN summary_bwd tokens/s (state gradient entering each span; one 131072-token sequence, "
                  "8 spans, H=16, K=V=128)")


def summary_bwd_algorithmic_flops(lengths, HO, K, V, C=64):
    """Arithmetic of the state-gradient recursion per (chunk, head): K K^T and Q K^T (lower
    halves), the triangular inverse, K dS, P^T dO, T^T dD and the dS update K^T dx + Q^T dO."""
    per = (2 * (C * (C + 1) // 2) * K * 2 + C ** 3 // 3 * 2 + C * K * V * 2 + 2 * (C * (C + 1) // 2) * V * 2
           + 2 * K * C * V * 2)
    chunks = sum((int(L) + C - 1) // C for L in lengths)
    return int(per * chunks * HO)


def run_summary_bwd_bench(args, world, rank, local):
    """gdn_summary_bwd over the context-parallel workload: one 131072-token sequence cut into 8
    spans of 16384, 16 heads, K = V = 128: per span and head the gradient of the span's outputs
    with respect to the state entering it (zero exit cotangent)."""
    import gated_delta_rule_29_gb300 as la
    from gated_delta_rule_29_gb300 import binding as B
    from gated_delta_rule_29_gb300 import workloads as W

    assert torch.cuda.is_available(), "bench needs a CUDA device (there is no CPU fallback)"
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lib = B.load()
    w = W.config(5)
    T, HK, HV, K, V = w.T, w.HK, w.HV, w.K, w.V
    gen = torch.Generator().manual_seed(1013)
    do_h = torch.randn(T, HV, V, generator=gen).to(torch.bfloat16)
    q, k, g, b, spans, do = (x.to(dev) for x in (w.q, w.k, w.g, w.beta, w.spans, do_h))
    S = spans.numel() - 1
    ws = torch.empty(max(lib.la_gdn_summary_bwd_workspace_bytes(S, HV, K, V), la.api.split_workspace_bytes(T, S, HV)),
                     dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        return la.gdn_summary_bwd(q, k, g, b, spans, do, workspace=ws, status=status)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert la.read_status(status) == 0
    stream = torch.cuda.current_stream()
    k_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a_, b_ in k_ev:
        a_.record(stream)
        b_.record(stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(args.steps):
            lib.la_set_kernel_timing_events(k_ev[i][0].cuda_event, k_ev[i][1].cuda_event)
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
    kern_ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in k_ev)
    assert la.read_status(status) == 0
    alg = T * (2 * HK * K + HV * V) * 2 + 2 * T * HV * 4 + S * HV * K * V * 4 + (S + 1) * 4
    flops = summary_bwd_algorithmic_flops([T // S] * S, HV, K, V)
    hbm_peak, bf16_peak, peak_src = load_peaks()
    tf32_peak = bf16_peak * TF32_PER_BF16
    tile = args.fwd_passes == "fused"
    tc_peak = tf32_peak if tile else bf16_peak
    tflops = flops / (kern_ms * 1e-3) / 1e12
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle  # CPU baseline only
        n_tok = 4096
        t0 = time.perf_counter()
        oracle.gdn_summary_bwd(w.q[:n_tok, :1], w.k[:n_tok, :1], w.g[:n_tok, :1], w.beta[:n_tok, :1],
                               np.array([0, n_tok]), do_h[:n_tok, :1])
        dt = time.perf_counter() - t0
        cpu = {"value": n_tok / HV / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": f"1 head x the first {n_tok} tokens of span 0 ({dt:.1f} s), fp64 token-by-token "
                         f"reverse recursion of the state gradient (numpy, one thread)"}
    if rank == 0:
        line = {
            "metric": SUM_BWD_METRIC, "value": T * world / (ms * 1e-3), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "summary_bwd: one sequence of 131072 tokens, 8 spans of 16384, H=16, K=V=128, "
                                   "zero exit cotangent", "global_batch": 1, "seq_len": T, "parallelism": "single GPU",
                       "l2": "inputs larger than L2 (1.1 GB of q/k/dO per step); no flush"},
            # the tensor-core path computes on bf16 hi + lo operands (its peak: the bf16 rate); the
            # tile kernel (--fwd-passes fused) on split tf32 warp MMAs (the tf32 rate)
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": tc_peak, "unit": "TFLOP/s",
                         "frac": tflops / tc_peak, "traffic": None,
                         "peak_source": (f"{peak_src} bf16 x {TF32_PER_BF16:.3f} (nominal dense tf32 / bf16)" if tile
                                         else f"{peak_src} bf16"),
                         "kernel": ("gdn_bwd_kernel<128, 128> (state-gradient mode)" if tile else
                                    "gdn_wy_kernel<128> + gdn_grad_kernel<128> (timed together)"), "kernel_ms": kern_ms,
                         "algorithmic_flops": flops, "algorithmic_bytes": alg,
                         "hbm_frac": alg / (kern_ms * 1e-3) / 1e9 / hbm_peak},
            "cpu_baseline": cpu,
            "e2e": None,
            "gpu_launches": 2 * args.steps,
            "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-units", type=int, default=256,
                    help="(sequence, head) units in the CPU-baseline sample (256 = the whole batch)")
    ap.add_argument("--ref-units", type=int, default=0,
                    help="(sequence, head) units per step of the reference arm (0: one per host core)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--e2e-groups", type=int, default=16, help="token ranges pipelined by gdn_fwd_host")
    ap.add_argument("--workload", choices=["dense", "decode", "bwd", "gdp", "summary", "summary_bwd", "table"],
                    default="dense",
                    help="dense: the chunked forward over the dense batch (the headline); "
                         "decode: one decode step against a state pool; bwd: the backward of the dense batch; "
                         "gdp: Gated DeltaProduct with 2 updates per token; summary: gdn_summary over 8 spans; "
                         "summary_bwd: the summary's state-gradient mirror over the same spans; "
                         "table: one line per workload of the five configurations, with the oracle at one "
                         "thread and at all cores")
    ap.add_argument("--bwd-ckpt", choices=["64", "128", "256", "512", "1024", "none"], default="64",
                    help="bwd: cadence of the forward's fp32 checkpoints the backward is given (none: re-run)")
    ap.add_argument("--fwd-passes", choices=["auto", "fused", "two"], default="auto",
                    help="forward schedule: the automatic choice (two passes when the workspace allows), "
                         "the fused kernel, or the two passes (the same bits either way)")
    ap.add_argument("--seq-len", type=int, default=8192,
                    help="tokens per sequence of the dense batch (8192 is the benchmark workload)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    world, rank, local = dist_setup()
    if args.impl == "ours" and args.fwd_passes != "auto":
        from gated_delta_rule_29_gb300 import binding as B
        B.load().la_test_set_fwd_passes({"fused": 1, "two": 2}[args.fwd_passes])
    try:
        if args.impl == "reference":
            return run_reference(args, world, rank)
        if args.workload == "decode":
            return run_decode(args, world, rank, local)
        if args.workload == "bwd":
            return run_bwd_bench(args, world, rank, local)
        if args.workload == "gdp":
            return run_gdp_bench(args, world, rank, local)
        if args.workload == "summary":
            return run_summary_bench(args, world, rank, local)
        if args.workload == "summary_bwd":
            return run_summary_bwd_bench(args, world, rank, local)
        if args.workload == "table":
            return run_table(args, world, rank, local)
        return run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
