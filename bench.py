"""Benchmark of the causal differential-attention forward on GB300.

One step = the whole path over one batch of the long-context workload
(B = 1, T = 16384, 16 diff heads, d = 64, dv = 128, no kv grouping, depth 12):
the lambda kernel, then the fused tcgen05 forward. Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Throughput counts 768 tensor flop per unmasked (query, key) pair per diff head
(2 components x 2d for the scores + 2 components x 2dv for P V). N > 1 runs
one rank per GPU under torchrun, each on its own copy of the workload (weak
scaling, no data-path collective); `value` is all ranks' flop over the
slowest rank's time. `--impl reference` times the fp64 CPU oracle on bounded
row samples of the same workload (rank 0 only).

The default run (one GPU, no workload flags) also measures, after the headline
line's timed region, the other forward workloads (`per_config`) and the rows
beyond the forward (`next`: cache forward, backward, rotary embedding, o_proj,
context-parallel merge), each with its own clock record; `--no-extras` skips
them.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "diff-attn fwd TFLOP/s (causal) & % of GB300 bf16 tensor peak; tokens/s"
L2_BYTES = 129 * 10**6  # GB300 L2 capacity
FLOP_PER_PAIR = 768
WORKLOAD = "long_t16384"
KERNEL_SRC = os.path.join(ROOT, "differential_attention_diffattn_gb300", "csrc", "fwd_sm103a.cu")
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "fwd_bf16_sm103a_long_t16384.md")
# rotary placements: (rot_dim in units of d, interleaved)
ROPE_PLACEMENTS = {"row2d_half": (2, False), "comp_interleaved": (1, True)}
ROPE_THETA = 10000.0
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return FALLBACK_PEAKS, "fallback"


def check_device(da, where):
    """Raise if the library's device status word reports an error (it is read and cleared)."""
    st = da.diffattn_get_device_status()
    if st != 0:
        raise RuntimeError(f"device reported {da.diffattn_status_string(st)} {where}")


def dense_view(t, inp):
    """Token-major [tokens, ...] as [B, T, ...] for a dense batch of equal
    sequences (several sequences, no cu_seqlens); unchanged otherwise."""
    if inp.wl.varlen or len(inp.seq_lens) <= 1:
        return t
    return t.view(len(inp.seq_lens), inp.seq_lens[0], *t.shape[1:])


def causal_pairs(seq_lens, heads):
    return sum(n * (n + 1) // 2 for n in seq_lens) * heads


def kernel_sha():
    with open(KERNEL_SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu summary, only while the
    kernel source still matches the one that was profiled."""
    try:
        txt = open(PROFILE_SUMMARY).read()
    except OSError:
        return None
    m_sha = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", txt)
    m_b = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not m_sha or not m_b or m_sha.group(1) != kernel_sha():
        return None
    return float(m_b.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", self.gpu_id], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# dense bf16 tensor-core rate of one SM per clock (M128 N128 K16 in 64 cycles)
BF16_FLOP_PER_CLK_SM = 8192


def clock_peak_tflops(clocks):
    """SMs x 8192 flop per clock x the largest SM clock nvidia-smi reported
    during the timed region: the tensor pipe's ceiling at that clock (the
    measured cuBLAS figure is the headline denominator; this one is for
    information)."""
    import torch
    if not clocks or not clocks.get("sm_max_mhz"):
        return None
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return sms * BF16_FLOP_PER_CLK_SM * clocks["sm_max_mhz"] * 1e6 / 1e12


# ------------------------------------------------------------ ours (GPU) ---

def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import differential_attention_diffattn_gb300 as da
    from differential_attention_diffattn_gb300 import shard
    from differential_attention_diffattn_gb300 import workloads as W

    da.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = W.WORKLOADS[args.workload]
    inp = W.generate(wl, seed=args.seed)
    tokens = inp.tokens
    pairs = causal_pairs(inp.seq_lens, wl.num_heads)
    flop_per_pair = 4 * (wl.d + wl.dv)  # 768 at d = 64, dv = 128
    flops_step = flop_per_pair * pairs
    packed = wl.varlen
    # algorithmic bytes of the forward: q, k, v read once, out written once
    alg_bytes = (inp.q.numel() + inp.k.numel() + inp.v.numel()) * inp.q.element_size() + \
        tokens * wl.num_heads * wl.dv * inp.q.element_size()
    li = da.diffattn_lambda_init(wl.depth)
    stream = torch.cuda.current_stream()

    # Two input/output sets, used alternately: each is larger than the 129 MB
    # L2, so a step never starts on tensors the previous step left in L2.
    sets = []
    for _ in range(2):
        s = dict(q=dense_view(inp.q.to(dev), inp), k=dense_view(inp.k.to(dev), inp), v=dense_view(inp.v.to(dev), inp))
        s["out"] = dense_view(torch.empty(tokens, wl.num_heads, wl.dv, dtype=s["q"].dtype, device=dev), inp)
        sets.append(s)
    lvec = [x.to(dev) for x in (inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2)]
    w = inp.subln_w.to(dev)
    cu = inp.cu_seqlens.to(dev)
    lam = torch.empty(1 if not wl.lambda_per_head else wl.num_heads, dtype=torch.float32, device=dev)

    rope = ROPE_PLACEMENTS.get(args.rope)
    if rope is not None:
        # q, k arrive before the rotary embedding: each step rotates k into a
        # scratch tensor (one pass), and the forward rotates each query tile of q
        # in shared memory as it loads it
        rot_dim = rope[0] * wl.d
        cos, sin = da.diffattn_rope_tables(ROPE_THETA, inp.max_seqlen, rot_dim)
        for s in sets:
            s["kr"] = torch.empty_like(s["k"])
    rope_bytes = 2 * inp.k.numel() * inp.k.element_size()  # the k pass: read and write k once
    hidden = wl.num_heads * wl.dv
    if args.out_proj:
        # o_proj = Linear(H * dv, hidden, bias=False) after the attention, hidden = H * dv
        w_o = (torch.randn(hidden, hidden, generator=torch.Generator().manual_seed(args.seed + 7)) *
               hidden ** -0.5).to(torch.bfloat16).to(dev)
        for s in sets:
            s["y"] = torch.empty(tokens, hidden, dtype=torch.bfloat16, device=dev)
    proj_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)] if args.out_proj else None
    rope_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)] if rope is not None else None

    def fwd(s, i=None, lam=lam, w=w, cu=cu, st=None):
        st = stream if st is None else st
        q, k = s["q"], s["k"]
        pk = dict(cu_seqlens=cu, max_seqlen=inp.max_seqlen) if packed else {}
        if rope is not None:
            if i is not None:
                rope_ev[i][0].record(st)
            da.diffattn_rope_k(k, cos, sin, rot_dim, rope[1], cu_seqlens=cu if packed else None, k_out=s["kr"],
                               stream=st)
            if i is not None:
                rope_ev[i][1].record(st)
            da.diffattn_fwd_rope_q(q, s["kr"], s["v"], lam, li, w, cos, sin, rot_dim, rope[1], causal=wl.causal,
                                   eps=wl.eps, out=s["out"], stream=st, **pk)
        else:
            da.diffattn_fwd(q, k, s["v"], lam, li, w, causal=wl.causal, eps=wl.eps, out=s["out"], stream=st, **pk)
        if args.out_proj:
            if i is not None:
                proj_ev[i][0].record(st)
            da.diffattn_out_proj(s["out"], w_o, out=s["y"], stream=st)
            if i is not None:
                proj_ev[i][1].record(st)

    # One pass of the hot path: lambda and the forward. The plain forward takes the
    # combined call (diffattn_fwd_lambda: the lambda kernel, then the forward whose
    # reads of lambda alone wait for it); with the rotary embedding or o_proj the
    # two calls run one after the other.
    plain = rope is None and not args.out_proj

    def step_on(s, st, lvec=lvec, lam=lam, w=w, cu=cu):
        if plain:
            pk = dict(cu_seqlens=cu, max_seqlen=inp.max_seqlen) if packed else {}
            da.diffattn_fwd_lambda(s["q"], s["k"], s["v"], *lvec, li, w, causal=wl.causal, eps=wl.eps, lam_out=lam,
                                   out=s["out"], stream=st, **pk)
        else:
            da.diffattn_lambda(*lvec, li, out=lam, stream=st)
            fwd(s, lam=lam, w=w, cu=cu, st=st)

    def step(i):
        step_on(sets[i % 2], stream)

    # Workloads whose input/output set is not well above the 129 MB L2 get an L2
    # flush (a 256 MB memset) before every timed step, outside the step's events;
    # their value then comes from the sum of the per-step events, and a warm
    # (unflushed) figure is reported beside it.
    set_bytes = sum(t.numel() * t.element_size() for n, t in sets[0].items() if n in ("q", "k", "v", "out"))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if set_bytes < 2 * L2_BYTES else None

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    check_device(da, "during warm-up")
    warm = None
    graphs = fwd_graphs = None
    if flush is not None:
        # Steps of these workloads take a few to a hundred microseconds, about what the
        # host needs to launch them from Python (argument checks, tensor maps, two
        # launches): launched one by one, the events would time the host. Each step is
        # therefore captured once per input set as a CUDA graph (lambda + forward, and
        # the forward alone for the launch time) and replayed, the L2 flushed before
        # every replay; the warm figure replays them back to back.
        graphs, fwd_graphs = [], []
        for b in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step_on(sets[b], torch.cuda.current_stream())
            graphs.append(g)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fwd(sets[b], st=torch.cuda.current_stream())
            fwd_graphs.append(g)
        for i in range(3):
            graphs[i % 2].replay()
        torch.cuda.synchronize()
        w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        w0.record(stream)
        for i in range(args.steps):
            graphs[i % 2].replay()
        w1.record(stream)
        torch.cuda.synchronize()
        check_device(da, "in the graph replays")
        warm_ms = w0.elapsed_time(w1) / args.steps
        warm = {"ms_per_step": round(warm_ms, 5), "value": round(flops_step / (warm_ms * 1e-3) / 1e12, 2),
                "l2": "warm: consecutive steps, no flush", "launch": "CUDA graph replay per step"}

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = None
    if rank == 0:
        visible = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
        sampler = ClockSampler(visible[local_rank].strip() if local_rank < len(visible) else str(local_rank))
        sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        sev[i][0].record(stream)
        if graphs is not None:
            graphs[i % 2].replay()
        elif plain:
            step(i)
        else:
            da.diffattn_lambda(*lvec, li, out=lam, stream=stream)
            ev[i][0].record(stream)
            fwd(sets[i % 2], i)
            ev[i][1].record(stream)
        sev[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    # the forward launch alone (lambda already computed), for the roofline
    if fwd_graphs is not None:  # flushed L2 before each
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            fwd_graphs[i % 2].replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    elif plain:
        for i in range(args.steps):
            ev[i][0].record(stream)
            fwd(sets[i % 2])
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    step_times = [a.elapsed_time(b) for a, b in sev]
    elapsed_ms = sum(step_times) if flush is not None else t0.elapsed_time(t1)
    fwd_ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    rope_ms = sum(a.elapsed_time(b) for a, b in rope_ev) / args.steps if rope is not None else 0.0
    proj_ms = sum(a.elapsed_time(b) for a, b in proj_ev) / args.steps if args.out_proj else 0.0
    fwd_ms -= rope_ms + proj_ms  # the attention kernel alone
    check_device(da, "in the timed region")
    elapsed_ms = shard.max_over_ranks(elapsed_ms)
    ms_step = elapsed_ms / args.steps
    step_flops = flops_step + (2 * tokens * hidden * hidden if args.out_proj else 0)
    value = step_flops * world * args.steps / (elapsed_ms * 1e-3) / 1e12

    # ---- end to end through the public API with host buffers ----------------
    # Every step copies its inputs from pinned host memory, runs lambda + forward
    # and reads its output back into pinned host memory. The copies run on two
    # copy streams (host -> device, device -> host) over the two device sets, so
    # step i + 1's inputs and step i - 1's output move while step i computes;
    # events keep a set's inputs until its forward has read them and its output
    # until it has been read back.
    host = {n: getattr(inp, n).pin_memory() for n in ("q", "k", "v", "subln_w", "cu_seqlens")}
    host_l = [x.pin_memory() for x in (inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2)]
    out_hs = [torch.empty(tokens, wl.num_heads, wl.dv, dtype=sets[0]["q"].dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in list(host.values()) + host_l)
    d2h = out_hs[0].numel() * out_hs[0].element_size()
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    e2e = [dict(lvec=[torch.empty_like(x) for x in lvec], w=torch.empty_like(w), cu=torch.empty_like(cu),
                lam=torch.empty_like(lam)) for _ in range(2)]
    ev_in, ev_done, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))
    for e in ev_done + ev_out:
        e.record(stream)

    def e2e_h2d(b):
        s, x = sets[b], e2e[b]
        s_in.wait_event(ev_done[b])  # the set's previous forward has read its inputs
        with torch.cuda.stream(s_in):
            for n in ("q", "k", "v"):
                s[n].copy_(dense_view(host[n], inp), non_blocking=True)
            for dst, src in zip(x["lvec"], host_l):
                dst.copy_(src, non_blocking=True)
            x["w"].copy_(host["subln_w"], non_blocking=True)
            x["cu"].copy_(host["cu_seqlens"], non_blocking=True)
        ev_in[b].record(s_in)

    def e2e_compute(b):
        x = e2e[b]
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])  # the set's previous output has been read back
        step_on(sets[b], stream, lvec=x["lvec"], lam=x["lam"], w=x["w"], cu=x["cu"])
        ev_done[b].record(stream)

    def e2e_d2h(b):
        s_out.wait_event(ev_done[b])
        with torch.cuda.stream(s_out):
            res = sets[b]["y"] if args.out_proj else sets[b]["out"]  # the step's result
            out_hs[b].copy_(res.view(out_hs[b].shape), non_blocking=True)
        ev_out[b].record(s_out)

    def e2e_run(n, start=None, end=None):
        if start is not None:
            start.record(s_in)
        e2e_h2d(0)
        for i in range(n):
            if i + 1 < n:
                e2e_h2d((i + 1) % 2)
            e2e_compute(i % 2)
            e2e_d2h(i % 2)
        if end is not None:
            end.record(s_out)

    e2e_run(2)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    e2e_run(args.e2e_steps, e0, e1)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms = shard.max_over_ranks(e2e_ms)
    e2e_value = step_flops * world * args.e2e_steps / (e2e_ms * 1e-3) / 1e12
    check_device(da, "in the end-to-end region")
    if not torch.isfinite(out_hs[(args.e2e_steps - 1) % 2][:: max(1, tokens // 64)].float()).all():
        raise RuntimeError("non-finite output")

    if rank != 0:
        return None
    pk, pk_kind = peaks()
    achieved = flops_step / (fwd_ms * 1e-3) / 1e12
    peak = float(pk["bf16_tflops"])
    s0 = sets[0]
    kernel_name = (da.diffattn_fwd_kernel(s0["q"], s0["k"], s0["v"], lam, w, cu_seqlens=cu, max_seqlen=inp.max_seqlen)
                   if packed else da.diffattn_fwd_kernel(s0["q"], s0["k"], s0["v"], lam, w))
    # the committed capture is of this kernel on the default workload
    traffic = (profiled_traffic() if kernel_name == "diffattn_fwd_bf16_sm103a_kernel" and args.workload == WORKLOAD
               else None)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "batch": len(inp.seq_lens) if not packed else None,
                   "seq_len": inp.max_seqlen, "tokens": tokens, "diff_heads": wl.num_heads,
                   "kv_heads": wl.num_kv_heads, "d": wl.d, "dv": wl.dv, "depth": wl.depth,
                   "causal": wl.causal, "flop_per_pair": flop_per_pair, "flop_per_step": step_flops,
                   "l2": (f"L2 flushed before every step (256 MB memset outside the step events; two rotating "
                          f"{set_bytes / 2**20:.0f} MB input/output sets)") if flush is not None else
                         f"inputs larger than L2: two rotating {set_bytes / 2**20:.0f} MB input/output sets",
                   "inputs": "seeded N(0,1) q/k/v rounded to bf16, lambda vectors N(0,0.1^2) fp32, subln w = 1"},
        "per_step_ms": {"median": round(statistics.median(step_times), 5), "min": round(min(step_times), 5),
                        "covers": ("one diffattn_fwd_lambda call (lambda + forward kernels) per step, CUDA events"
                                   if plain else "lambda + forward launches of one step, CUDA events")},
        **({"launch": "each step a CUDA graph replay (lambda + forward), L2 flushed before it"}
           if graphs is not None else {}),
        # the same rate under the other counts of the pages' workloads, for information:
        # T^2 / 2 pairs per head instead of T (T + 1) / 2, and the 512 flop per pair of
        # the probability-map form (which one pass cannot run: it needs the row
        # statistics before P V)
        "other_flop_counts": {
            "tflops_t2_over_2_pairs": round(value * sum(L * L / 2 for L in inp.seq_lens) /
                                            sum(L * (L + 1) / 2 for L in inp.seq_lens), 2),
            "tflops_512_per_pair": round(value * 512 / flop_per_pair, 2)} if not args.out_proj else None,
        "tokens_per_s": round(tokens * world * args.steps / (elapsed_ms * 1e-3), 1),
        "pct_of_bf16_peak": round(100.0 * value / world / peak, 2),
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": args.e2e_steps, "ms_per_step": round(e2e_ms / args.e2e_steps, 4)},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_kind": f"{pk_kind} bf16 dense burst",
                     "frac_of_sustained": round(achieved / float(pk["bf16_tflops_sustained"]), 4),
                     "frac_of_clock_peak": (round(achieved / clock_peak_tflops(clocks), 4)
                                            if clock_peak_tflops(clocks) else None),
                     "kernel": kernel_name, "launch_ms": round(fwd_ms, 4),
                     "algorithmic_flop_per_launch": flops_step,
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "hbm_gbs": round(alg_bytes / (fwd_ms * 1e-3) / 1e9, 1),
                     "frac_of_hbm": round(alg_bytes / (fwd_ms * 1e-3) / 1e9 / float(pk["hbm_gbs"]), 4)},
        "clocks": clocks,
        **({"warm": warm} if warm is not None else {}),
        "gpu_launches": (2 + (rope is not None) + bool(args.out_proj)) * args.steps,
        "impl": "ours",
    }
    if args.out_proj:
        proj_flop = 2 * tokens * hidden * hidden
        line["metric"] = METRIC + " (with o_proj)"
        line["config"]["o_proj"] = {"in_features": hidden, "out_features": hidden}
        line["out_proj"] = {"kernel": "diffattn_out_proj_kernel", "ms": round(proj_ms, 5), "flop": proj_flop,
                            "tflops": round(proj_flop / (proj_ms * 1e-3) / 1e12, 1),
                            "frac_of_bf16_peak": round(proj_flop / (proj_ms * 1e-3) / 1e12 / peak, 4)}
    if rope is not None:
        line["metric"] = METRIC + " (with rotary embedding of q, k)"
        line["config"]["rope"] = {"placement": args.rope, "rot_dim": rot_dim, "interleaved": rope[1],
                                  "theta": ROPE_THETA}
        line["config"]["rope"]["q"] = "rotated inside the forward kernels (diffattn_fwd_rope_q)"
        line["rope"] = {"kernel": "diffattn_rope_qk_kernel (k only)", "ms": round(rope_ms, 5), "bytes": rope_bytes,
                        "gbs": round(rope_bytes / (rope_ms * 1e-3) / 1e9, 1),
                        "frac_of_hbm": round(rope_bytes / (rope_ms * 1e-3) / 1e9 / float(pk["hbm_gbs"]), 4)}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp, args.cpu_stride)
    return line


# ------------------------------------------------ training step (GPU) ---

BWD_FLOP_PER_PAIR = 1280  # S_1, S_2 recomputed once, dP, dV, dQ_1, dQ_2, dK_1, dK_2


def run_ours_bwd(args, rank, world, local_rank):
    """Forward with saved statistics + backward (all gradients, including the
    lambda vectors and the norm weight). Algorithmic flop per visible pair and
    diff head: 768 forward + 1280 backward."""
    import torch

    import differential_attention_diffattn_gb300 as da
    from differential_attention_diffattn_gb300 import shard
    from differential_attention_diffattn_gb300 import workloads as W

    da.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = W.WORKLOADS[args.workload]
    inp = W.generate(wl, seed=args.seed)
    tokens, H, dvv = inp.tokens, wl.num_heads, wl.dv
    pairs = causal_pairs(inp.seq_lens, H)
    fwd_flop, bwd_flop = FLOP_PER_PAIR * pairs, BWD_FLOP_PER_PAIR * pairs
    li = da.diffattn_lambda_init(wl.depth)
    stream = torch.cuda.current_stream()
    g = torch.Generator().manual_seed(args.seed + 1)
    dout_h = torch.randn(tokens, H, dvv, generator=g).to(torch.bfloat16)
    cu = inp.cu_seqlens.to(dev) if wl.varlen else None
    kw = dict(causal=wl.causal, cu_seqlens=cu, max_seqlen=inp.max_seqlen if wl.varlen else None, eps=wl.eps)
    sets = []
    for _ in range(2):  # two rotating sets, each far larger than L2
        s = {n: dense_view(t.to(dev), inp) for n, t in (("q", inp.q), ("k", inp.k), ("v", inp.v), ("dout", dout_h))}
        s["out"] = dense_view(torch.empty(tokens, H, dvv, dtype=torch.bfloat16, device=dev), inp)
        s["lse"] = dense_view(torch.empty(tokens, H, 2, dtype=torch.float32, device=dev), inp)
        s["o1"] = dense_view(torch.empty(tokens, H, dvv, dtype=torch.float32, device=dev), inp)
        s["o2"] = torch.empty_like(s["o1"])
        s["grads"] = (torch.empty_like(s["q"]), torch.empty_like(s["k"]), torch.empty_like(s["v"]),
                      torch.empty(H if wl.lambda_per_head else 1, dtype=torch.float32, device=dev),
                      torch.empty(dvv, dtype=torch.float32, device=dev))
        sets.append(s)
    lvec = [x.to(dev) for x in (inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2)]
    w = inp.subln_w.to(dev)
    lam = torch.empty(H if wl.lambda_per_head else 1, dtype=torch.float32, device=dev)
    ws = torch.empty(max(16, da.diffattn_bwd_workspace_size(sets[0]["q"], sets[0]["k"], sets[0]["v"], lam, w, cu,
                                                          kw["max_seqlen"], wl.eps)), dtype=torch.uint8, device=dev)

    def fwd(s):
        da.diffattn_fwd_train(s["q"], s["k"], s["v"], lam, li, w, out=s["out"], lse=s["lse"], o1=s["o1"],
                              o2=s["o2"], stream=stream, **kw)

    def bwd(s):
        da.diffattn_bwd(s["q"], s["k"], s["v"], lam, li, w, s["dout"], s["lse"], s["o1"], s["o2"], workspace=ws,
                        grads=s["grads"], stream=stream, **kw)

    def lam_bwd(s):
        return da.diffattn_lambda_bwd(*lvec, s["grads"][3], stream=stream)

    for i in range(args.warmup):
        s = sets[i % 2]
        da.diffattn_lambda(*lvec, li, out=lam, stream=stream)
        fwd(s)
        bwd(s)
        lam_bwd(s)
    torch.cuda.synchronize()
    check_device(da, "during warm-up")
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    ev = [(mk(), mk(), mk()) for _ in range(args.steps)]
    t0, t1 = mk(), mk()
    sampler = None
    if rank == 0:
        visible = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
        sampler = ClockSampler(visible[local_rank].strip() if local_rank < len(visible) else str(local_rank))
        sampler.start()
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(args.steps):
        s = sets[i % 2]
        da.diffattn_lambda(*lvec, li, out=lam, stream=stream)
        ev[i][0].record(stream)
        fwd(s)
        ev[i][1].record(stream)
        bwd(s)
        ev[i][2].record(stream)
        lam_bwd(s)
    t1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    check_device(da, "in the timed region")
    elapsed_ms = shard.max_over_ranks(t0.elapsed_time(t1))
    fwd_ms = sum(a.elapsed_time(b) for a, b, _ in ev) / args.steps
    bwd_ms = sum(b.elapsed_time(c) for _, b, c in ev) / args.steps
    value = (fwd_flop + bwd_flop) * world * args.steps / (elapsed_ms * 1e-3) / 1e12

    # end to end: q, k, v, dout and the parameters from pinned host memory, all
    # gradients back to pinned host memory
    hq = {n: getattr(inp, n).pin_memory() for n in ("q", "k", "v", "subln_w")}
    hq["dout"] = dout_h.pin_memory()
    hl = [x.pin_memory() for x in (inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2)]
    hg = [t.cpu().pin_memory() for t in sets[0]["grads"][:3]] + [x.cpu().pin_memory() for x in lvec] + \
        [sets[0]["grads"][4].cpu().pin_memory()]
    h2d = sum(t.numel() * t.element_size() for t in list(hq.values()) + hl)
    d2h = sum(t.numel() * t.element_size() for t in hg)

    def e2e_step():
        s = sets[0]
        for n in ("q", "k", "v", "dout"):
            s[n].copy_(dense_view(hq[n], inp), non_blocking=True)
        for dst, src in zip(lvec, hl):
            dst.copy_(src, non_blocking=True)
        w.copy_(hq["subln_w"], non_blocking=True)
        da.diffattn_lambda(*lvec, li, out=lam, stream=stream)
        fwd(s)
        bwd(s)
        lg = lam_bwd(s)
        for dst, src in zip(hg, list(s["grads"][:3]) + list(lg) + [s["grads"][4]]):
            dst.copy_(src.view(dst.shape), non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    e0, e1 = mk(), mk()
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = shard.max_over_ranks(e0.elapsed_time(e1))
    check_device(da, "in the end-to-end region")
    if not all(torch.isfinite(t.float()).all() for t in hg):
        raise RuntimeError("non-finite gradient")
    if rank != 0:
        return None
    pk, pk_kind = peaks()
    peak = float(pk["bf16_tflops"])
    bwd_achieved = bwd_flop / (bwd_ms * 1e-3) / 1e12
    return {
        "metric": "diff-attn fwd+bwd TFLOP/s (causal)", "value": round(value, 2), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(elapsed_ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "tokens": tokens, "seq_len": inp.max_seqlen, "diff_heads": H,
                   "kv_heads": wl.num_kv_heads, "d": wl.d, "dv": dvv, "causal": wl.causal,
                   "flop_per_pair": FLOP_PER_PAIR + BWD_FLOP_PER_PAIR, "flop_per_step": fwd_flop + bwd_flop,
                   "l2": "two rotating input/output sets, each larger than L2"},
        "fwd_train": {"ms": round(fwd_ms, 4), "tflops": round(fwd_flop / (fwd_ms * 1e-3) / 1e12, 2)},
        "e2e": {"value": round((fwd_flop + bwd_flop) * world * args.e2e_steps / (e2e_ms * 1e-3) / 1e12, 2),
                "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": args.e2e_steps, "ms_per_step": round(e2e_ms / args.e2e_steps, 4)},
        "roofline": {"bound": "tensor", "achieved": round(bwd_achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(bwd_achieved / peak, 4), "traffic": None,
                     "peak_kind": f"{pk_kind} bf16 dense burst",
                     "frac_of_sustained": round(bwd_achieved / float(pk["bf16_tflops_sustained"]), 4),
                     "frac_of_clock_peak": (round(bwd_achieved / clock_peak_tflops(clocks), 4)
                                            if clock_peak_tflops(clocks) else None),
                     "kernel": "diffattn_bwd (preprocessing + dQ + dK/dV kernels)", "launch_ms": round(bwd_ms, 4),
                     "algorithmic_flop_per_launch": bwd_flop},
        "clocks": clocks, "gpu_launches": 6 * args.steps, "impl": "ours",
    }


# ------------------------------------------- context-parallel split (GPU) ---

def run_ours_cp(args, rank, world, local_rank):
    """One long sequence split into 2N zigzag chunks. With one process the N
    ranks' blocks (training-forward partials + merges) run one rank after
    another on this GPU; under torchrun each rank runs its own chunks and the
    K/V chunks go around an NCCL ring."""
    import torch

    import differential_attention_diffattn_gb300 as da
    from differential_attention_diffattn_gb300 import context_parallel as cp
    from differential_attention_diffattn_gb300 import shard
    from differential_attention_diffattn_gb300 import workloads as W

    da.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = W.WORKLOADS[args.workload]
    inp = W.generate(wl, seed=args.seed)
    if len(inp.seq_lens) != 1:
        raise SystemExit("--cp splits one sequence: pick a single-sequence workload")
    n_ranks = world if world > 1 else args.cp
    T = inp.tokens
    chunk = T // (2 * n_ranks)
    if chunk * 2 * n_ranks != T or chunk % 128 != 0:
        raise SystemExit(f"{T} tokens do not split into {2 * n_ranks} chunks of a multiple of 128")
    flops = FLOP_PER_PAIR * causal_pairs(inp.seq_lens, wl.num_heads)
    li = da.diffattn_lambda_init(wl.depth)
    lvec = [x.to(dev) for x in (inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2)]
    lam = da.diffattn_lambda(*lvec, li)
    w = inp.subln_w.to(dev)
    stream = torch.cuda.current_stream()
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    kern = cp.GpuKernels(lam, li, w, wl.eps, stream=stream)
    merge_ev = []

    class Timed(cp.GpuKernels):
        def merge(self, parts, n):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            y = super().merge(parts, n)
            b.record(stream)
            merge_ev.append((a, b, n))
            return y
    kern = Timed(lam, li, w, wl.eps, stream=stream)
    kv = {b: (k[b * chunk:(b + 1) * chunk], v[b * chunk:(b + 1) * chunk]) for b in range(2 * n_ranks)}

    def step():
        if world > 1:
            return cp.ring_forward(cp.split_zigzag(q, world, rank), cp.split_zigzag(k, world, rank),
                                   cp.split_zigzag(v, world, rank), kern)
        outs = {}
        for r in range(n_ranks):
            outs.update(cp.local_forward(cp.split_zigzag(q, n_ranks, r), kv, kern))
        return outs

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    merge_ev.clear()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    sampler = None
    if rank == 0:
        visible = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
        sampler = ClockSampler(visible[local_rank].strip() if local_rank < len(visible) else str(local_rank))
        sampler.start()
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(args.steps):
        outs = step()
    t1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    check_device(da, "in the timed region")
    elapsed = shard.max_over_ranks(t0.elapsed_time(t1))
    merge_ms = sum(a.elapsed_time(b) for a, b, _ in merge_ev) / args.steps
    merge_bytes = sum(n * chunk * wl.num_heads * (2 * wl.dv * 4 + 8) + chunk * wl.num_heads * wl.dv * 2
                      for _, _, n in merge_ev) // args.steps
    # End to end: q, k, v of the sequence from pinned host memory each step, every
    # output chunk back to pinned host memory, on the compute stream.
    host_in = [x.pin_memory() for x in (inp.q, inp.k, inp.v)]
    host_out = {a: torch.empty(y.shape, dtype=y.dtype).pin_memory() for a, y in outs.items()}
    h2d = sum(x.numel() * x.element_size() for x in host_in)
    d2h = sum(x.numel() * x.element_size() for x in host_out.values())
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.e2e_steps):
        for dst, src in zip((q, k, v), host_in):
            dst.copy_(src, non_blocking=True)
        for a, y in step().items():
            host_out[a].copy_(y, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    check_device(da, "in the end-to-end region")
    e2e_ms = shard.max_over_ranks(e0.elapsed_time(e1))
    if rank != 0:
        return None
    if not all(torch.isfinite(y.float()).all() for y in outs.values()):
        raise RuntimeError("non-finite output")
    pk, pk_kind = peaks()
    return {
        "metric": "diff-attn fwd TFLOP/s (causal), context-parallel split", "value":
            round(flops * args.steps / (elapsed * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(elapsed / args.steps, 4),
        "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "tokens": T, "diff_heads": wl.num_heads, "kv_heads": wl.num_kv_heads,
                   "cp_ranks": n_ranks, "chunk": chunk,
                   "emulated_on_one_gpu": world == 1, "flop_per_step": flops},
        "e2e": {"value": round(flops * args.e2e_steps / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
                "ms_per_step": round(e2e_ms / args.e2e_steps, 4)},
        "roofline": {"bound": "hbm", "unit": "GB/s", "kernel": "diffattn_merge_kernel", "traffic": None,
                     "achieved": round(merge_bytes / (merge_ms * 1e-3) / 1e9, 1) if merge_ms > 0 else None,
                     "peak": float(pk["hbm_gbs"]), "peak_kind": f"{pk_kind} HBM copy bandwidth",
                     "frac": round(merge_bytes / (merge_ms * 1e-3) / 1e9 / float(pk["hbm_gbs"]), 4)
                     if merge_ms > 0 else None},
        "clocks": clocks,
        "merge": {"kernel": "diffattn_merge_kernel", "ms": round(merge_ms, 5), "bytes": merge_bytes,
                  "gbs": round(merge_bytes / (merge_ms * 1e-3) / 1e9, 1) if merge_ms > 0 else None,
                  "frac_of_hbm": round(merge_bytes / (merge_ms * 1e-3) / 1e9 / float(pk["hbm_gbs"]), 4)
                  if merge_ms > 0 else None},
        # per rank: 2N + 1 training-forward partials and 2 merges
        "gpu_launches": (n_ranks if world == 1 else 1) * (2 * n_ranks + 3) * args.steps, "impl": "ours",
    }


# ------------------------------------------------- cache forward (GPU) ---

def run_ours_kv(args, rank, world, local_rank):
    """Decode / short query block against a key/value cache. HBM-bound: the
    metric is algorithmic bytes (valid cache rows of K and V read once, q read,
    out written) per second."""
    import torch

    import differential_attention_diffattn_gb300 as da
    from differential_attention_diffattn_gb300 import shard
    from differential_attention_diffattn_gb300 import workloads as W

    da.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = W.KV_WORKLOADS[args.workload]
    inp = W.generate_kv(wl, seed=args.seed)
    lens = [int(x) for x in inp.cache_seqlens]
    kv_row_bytes = wl.num_kv_heads * (2 * wl.d + wl.dv) * 2
    bytes_step = (sum(lens) * kv_row_bytes + wl.batch * wl.q_len * wl.num_heads * (2 * wl.d + wl.dv) * 2)
    li = da.diffattn_lambda_init(wl.depth)
    stream = torch.cuda.current_stream()
    sets = []
    for _ in range(2):  # two caches used alternately: a step never starts on an L2-resident cache
        s = dict(q=inp.q.to(dev), k=inp.k_cache.to(dev), v=inp.v_cache.to(dev))
        s["out"] = torch.empty(inp.q.shape[:-1] + (wl.dv,), dtype=torch.bfloat16, device=dev)
        sets.append(s)
    lvec = [x.to(dev) for x in (inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2)]
    w = inp.subln_w.to(dev)
    lens_d = inp.cache_seqlens.to(dev)
    lam = torch.empty(wl.num_heads if wl.lambda_per_head else 1, dtype=torch.float32, device=dev)
    # the caller's host copy of the lengths goes to the split plan (a serving loop has it)
    desc = da.kv_desc(inp.q, inp.k_cache, inp.v_cache, wl.eps, host_seqlens=lens)
    ws = torch.empty(da.diffattn_fwd_kvcache_workspace_size(desc), dtype=torch.uint8, device=dev)
    splits = da.diffattn_fwd_kvcache_workspace_size(desc) // (wl.batch * wl.q_len * wl.num_heads * 2 * (wl.dv + 2) * 4)

    def fwd(s, st=stream):
        da.diffattn_fwd_kvcache(s["q"], s["k"], s["v"], lam, li, w, cache_seqlens=lens_d, causal=wl.causal,
                                eps=wl.eps, workspace=ws, out=s["out"], stream=st, host_seqlens=lens)

    # One step: lambda and the cache forward in one call (two launches: the combine
    # kernel, the only one that uses lambda, forms it).
    def step(s, st=stream):
        da.diffattn_fwd_kvcache_lambda(s["q"], s["k"], s["v"], *lvec, li, w, cache_seqlens=lens_d,
                                       causal=wl.causal, eps=wl.eps, workspace=ws, lam_out=lam, out=s["out"],
                                       stream=st, host_seqlens=lens)

    for i in range(args.warmup):
        step(sets[i % 2])
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = None
    if rank == 0:
        visible = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
        sampler = ClockSampler(visible[local_rank].strip() if local_rank < len(visible) else str(local_rank))
        sampler.start()
    torch.cuda.synchronize()
    # A loop of steps launched one by one from Python, then the per-call time of the
    # cache forward alone (lambda precomputed) with events around each call.
    t0.record(stream)
    for i in range(args.steps):
        step(sets[i % 2])
    t1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    check_device(da, "in the timed region")
    elapsed_ms = shard.max_over_ranks(t0.elapsed_time(t1))
    for i in range(args.steps):
        da.diffattn_lambda(*lvec, li, out=lam, stream=stream)
        ev[i][0].record(stream)
        fwd(sets[i % 2])
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    check_device(da, "in the per-call timing")
    fwd_ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    host_value = bytes_step * world * args.steps / (elapsed_ms * 1e-3) / 1e9
    host_ms = elapsed_ms / args.steps

    # The same steps replayed from CUDA graphs (a serving loop captures its decode
    # step): launched from Python, a ragged step's host work (argument checks, the
    # split plan, two tensor maps, three launches) takes longer than its ~33 us on
    # the GPU, so the Python loop above measures the host. Each graph holds
    # GRAPH_STEPS steps over the two cache sets; the calls alone are timed the same way.
    GRAPH_STEPS = 10

    def capture(with_lambda):
        gs = []
        for b in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                st = torch.cuda.current_stream()
                for r in range(GRAPH_STEPS):
                    (step if with_lambda else fwd)(sets[(b + r) % 2], st=st)
            gs.append(g)
        return gs

    def replay_ms(gs, n_graphs):
        for i in range(3):
            gs[i % 2].replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(n_graphs):
            gs[i % 2].replay()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / (n_graphs * GRAPH_STEPS)

    n_graphs = max(2, args.steps // GRAPH_STEPS)
    step_graphs, call_graphs = capture(True), capture(False)
    if rank == 0:
        sampler = ClockSampler(visible[local_rank].strip() if local_rank < len(visible) else str(local_rank))
        sampler.start()
    torch.cuda.synchronize()
    graph_ms = shard.max_over_ranks(replay_ms(step_graphs, n_graphs))
    clocks = sampler.stop() if sampler else clocks
    call_ms = replay_ms(call_graphs, n_graphs)
    check_device(da, "in the graph replays")
    value = bytes_step * world / (graph_ms * 1e-3) / 1e9

    # End to end through the public API: each step's queries arrive from pinned host
    # memory and the output is read back to pinned host memory, on the compute
    # stream. The cache stays resident; the new tokens' K / V rows are written
    # into it on the device (by the projection, in serving), not copied from the host.
    host_q = inp.q.pin_memory()
    host_out = torch.empty(sets[0]["out"].shape, dtype=torch.bfloat16).pin_memory()
    h2d = host_q.numel() * 2
    d2h = host_out.numel() * 2
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(args.e2e_steps):
        s = sets[i % 2]
        s["q"].copy_(host_q, non_blocking=True)
        step(s)
        host_out.copy_(s["out"], non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    check_device(da, "in the end-to-end region")
    e2e_ms = shard.max_over_ranks(e0.elapsed_time(e1))
    if rank != 0:
        return None
    pk, pk_kind = peaks()
    achieved = bytes_step / (call_ms * 1e-3) / 1e9
    return {
        "metric": "diff-attn kv-cache fwd HBM GB/s (decode)", "value": round(value, 1), "unit": "GB/s",
        "launch": f"CUDA graph replay ({GRAPH_STEPS} steps of diffattn_fwd_kvcache_lambda per graph)",
        "host_launched": {"value": round(host_value, 1), "ms_per_step": round(host_ms, 5),
                          "call_ms_between_events": round(fwd_ms, 5),
                          "note": "steps launched one by one from Python: bound by the host's work per call"},
        "e2e": {"value": round(bytes_step * world * args.e2e_steps / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
                "ms_per_step": round(e2e_ms / args.e2e_steps, 5),
                "covers": "queries from pinned host memory, the call, the output back (cache resident)"},
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(graph_ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "batch": wl.batch, "q_len": wl.q_len, "cache_capacity": wl.capacity,
                   "cache_tokens": sum(lens), "diff_heads": wl.num_heads, "kv_heads": wl.num_kv_heads, "d": wl.d,
                   "dv": wl.dv, "causal": wl.causal, "bytes_per_step": bytes_step,
                   "key_splits": int(splits), "split_plan": "from the host copy of the cache lengths",
                   "l2": "two rotating caches, each larger than L2"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": float(pk["hbm_gbs"]), "unit": "GB/s",
                     "frac": round(achieved / float(pk["hbm_gbs"]), 4), "traffic": None,
                     "peak_kind": f"{pk_kind} HBM copy bandwidth",
                     "kernel": "diffattn_decode_tc_kernel + diffattn_decode_combine_kernel",
                     "launch_ms": round(call_ms, 5), "launch_timing": "call alone, CUDA graph replay"},
        "clocks": clocks, "gpu_launches": 2 * n_graphs * GRAPH_STEPS, "impl": "ours",
    }


# ------------------------------------- every workload in one run (GPU) ---

# The other configurations of the forward (parity workloads of the same method)
# and the rows beyond it, each measured in the default run so that one command
# records every figure with its clocks.
EXTRA_FWD = ("tiny_f32", "b2_t512_gqa", "llama1b_b4_t2048", "varlen_32k")


def run_extras(args, local_rank):
    import torch

    from differential_attention_diffattn_gb300 import workloads as W
    W_KV = set(W.KV_WORKLOADS)

    def sub(**over):
        a = argparse.Namespace(**vars(args))
        a.steps, a.warmup, a.e2e_steps = args.extra_steps, max(3, min(args.warmup, 5)), 3
        # calls of tens of microseconds get more steps, so that the figure is not a few launches'
        if over.get("workload") in ("tiny_f32", "b2_t512_gqa") or over.get("workload") in W_KV:
            a.steps = max(args.extra_steps, 200)
        a.no_cpu_baseline, a.rope, a.out_proj, a.backward, a.cp = True, None, False, False, 0
        for k, v in over.items():
            setattr(a, k, v)
        return a

    def guarded(fn):
        try:
            return fn()
        except Exception as e:  # recorded in the line, not hidden
            log(f"extra measurement failed: {e!r}")
            return {"error": repr(e)[:300]}
        finally:
            torch.cuda.synchronize()
            torch.cuda.empty_cache()

    per_config = {}
    for name in EXTRA_FWD:
        def one(name=name):
            ln = run_ours(sub(workload=name), 0, 1, local_rank)
            rf = ln["roofline"]
            d = {"kernel": rf["kernel"], "ms_per_step": ln["ms_per_step"], "tflops_per_step": ln["value"],
                 "tokens_per_s": ln["tokens_per_s"], "launch_ms": rf["launch_ms"], "kernel_tflops": rf["achieved"],
                 "frac_of_bf16_peak": rf["frac"], "hbm_gbs": rf["hbm_gbs"], "frac_of_hbm": rf["frac_of_hbm"],
                 "flop_per_step": ln["config"]["flop_per_step"], "l2": ln["config"]["l2"],
                 "e2e": ln["e2e"], "clocks": ln["clocks"], "steps": ln["steps"]}
            if "warm" in ln:
                d["warm"] = ln["warm"]
            if name == "tiny_f32":
                d["note"] = "fp32 parity path on the CUDA cores: a latency figure, not a tensor-core rate"
            if name == "b2_t512_gqa":
                d["bound"] = "latency (neither roof): HBM GB/s reported"
            return d
        per_config[name] = guarded(one)

    nxt = {}

    def kv(name):
        ln = run_ours_kv(sub(workload=name), 0, 1, local_rank)
        return {"gbs_per_step": ln["value"], "launch": ln["launch"], "host_launched": ln["host_launched"],
                "call_ms": ln["roofline"]["launch_ms"],
                "key_splits": ln["config"]["key_splits"],
                "call_gbs": ln["roofline"]["achieved"], "frac_of_hbm": ln["roofline"]["frac"],
                "bytes_per_step": ln["config"]["bytes_per_step"], "e2e": ln["e2e"], "clocks": ln["clocks"]}
    for name in ("decode_b8_c16384", "decode_b16_q4_ragged"):
        nxt[name] = guarded(lambda name=name: kv(name))

    def bwd():
        ln = run_ours_bwd(sub(workload=WORKLOAD), 0, 1, local_rank)
        rf = ln["roofline"]
        return {"workload": WORKLOAD, "bwd_ms": rf["launch_ms"], "bwd_tflops": rf["achieved"],
                "frac_of_bf16_peak": rf["frac"], "train_step_tflops": ln["value"], "fwd_train": ln["fwd_train"],
                "flop_per_pair": "768 forward + 1280 backward (algorithmic)", "clocks": ln["clocks"]}
    nxt["backward"] = guarded(bwd)

    def rope(placement):
        ln = run_ours(sub(workload=WORKLOAD, rope=placement), 0, 1, local_rank)
        return dict(ln["rope"], step_tflops=ln["value"], attention_launch_ms=ln["roofline"]["launch_ms"],
                    clocks=ln["clocks"])
    for pl in sorted(ROPE_PLACEMENTS):
        nxt[f"rope_{pl}"] = guarded(lambda pl=pl: rope(pl))

    def proj():
        ln = run_ours(sub(workload=WORKLOAD, out_proj=True), 0, 1, local_rank)
        return dict(ln["out_proj"], step_tflops=ln["value"], clocks=ln["clocks"])
    nxt["o_proj"] = guarded(proj)

    def cp2():
        ln = run_ours_cp(sub(workload=WORKLOAD, cp=2), 0, 1, local_rank)
        return dict(ln["merge"], step_tflops=ln["value"], cp_ranks=2, emulated_on_one_gpu=True, clocks=ln["clocks"])
    nxt["cp_merge"] = guarded(cp2)
    return per_config, nxt


# --------------------------------------------------------- CPU / oracle ---

def oracle_sample(inp, positions):
    """Oracle rows for the given in-sequence query positions of every sequence
    and every head; returns (seconds, pairs)."""
    import numpy as np

    from oracle import oracle as orc
    wl = inp.wl
    cu = inp.cu_seqlens.tolist()
    toks = []
    for s in range(len(cu) - 1):
        n = cu[s + 1] - cu[s]
        toks.extend(cu[s] + p for p in positions if p < n)
    toks = np.asarray(toks, dtype=np.int32)
    tt = np.repeat(toks, wl.num_heads)
    hh = np.tile(np.arange(wl.num_heads, dtype=np.int32), toks.size)
    keys = [(p + 1 if wl.causal else cu[s + 1] - cu[s]) for s in range(len(cu) - 1) for p in positions
            if p < cu[s + 1] - cu[s]]
    pairs = int(sum(keys)) * wl.num_heads
    li = orc.lambda_init(wl.depth)
    lam = orc.lambda_values(inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2, li)
    t = time.perf_counter()
    orc.forward_rows(inp.cu_seqlens, inp._f64_q, inp._f64_k, inp._f64_v, lam, li, inp.subln_w, wl.eps,
                     wl.causal, rows=(tt, hh))
    return time.perf_counter() - t, pairs


def _prep_f64(inp):
    from oracle import oracle as orc
    if not hasattr(inp, "_f64_q"):
        inp._f64_q, inp._f64_k, inp._f64_v = orc._f64(inp.q), orc._f64(inp.k), orc._f64(inp.v)


def cpu_baseline(inp, stride):
    from oracle import oracle as orc
    _prep_f64(inp)
    positions = list(range(stride // 2, inp.max_seqlen, stride))
    sec, pairs = oracle_sample(inp, positions)
    return {"value": round(FLOP_PER_PAIR * pairs / sec / 1e12, 6), "unit": "TFLOP/s", "cores": orc.num_threads(),
            "kind": "oracle", "seconds": round(sec, 2),
            "sample": f"fp64 C oracle (OpenMP) on every {stride}th query row of every head "
                      f"({len(positions) * inp.wl.num_heads} rows, {pairs} causal pairs) of {inp.wl.name}"}


def run_reference(args):
    from differential_attention_diffattn_gb300 import workloads as W
    from oracle import oracle as orc
    wl = W.WORKLOADS[args.workload]
    inp = W.generate(wl, seed=args.seed)
    _prep_f64(inp)
    L = inp.max_seqlen
    budget_s = args.reference_budget_s
    # rows per step: start at 64 query positions, shrink so the run fits the budget
    per_step = 64
    sec, _ = oracle_sample(inp, list(range(0, L, L // per_step)))
    est = sec * (args.steps + args.warmup)
    while est > budget_s and per_step > 2:
        per_step //= 2
        est /= 2
    stride = L // per_step
    for i in range(args.warmup):
        oracle_sample(inp, list(range(i % stride, L, stride)))
    tot_s, tot_pairs = 0.0, 0
    for i in range(args.steps):
        s, p = oracle_sample(inp, list(range((i * 37) % stride, L, stride)))
        tot_s += s
        tot_pairs += p
    value = FLOP_PER_PAIR * tot_pairs / tot_s / 1e12
    sample = (f"fp64 C oracle (OpenMP) per step on {per_step} query positions (stride {stride}, rotating offset) "
              f"x {wl.num_heads} heads of {wl.name}")
    return {
        "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * tot_s / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "seq_len": L, "diff_heads": wl.num_heads, "kv_heads": wl.num_kv_heads,
                   "d": wl.d, "dv": wl.dv, "depth": wl.depth, "causal": wl.causal, "flop_per_pair": FLOP_PER_PAIR},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": orc.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
        "impl": "reference",
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-stride", type=int, default=2, help="CPU baseline: every n-th query row")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--reference-budget-s", type=float, default=150.0)
    ap.add_argument("--backward", action="store_true", help="time forward + backward (training step)")
    ap.add_argument("--out-proj", action="store_true", help="run o_proj (H*dv -> H*dv) after the attention")
    ap.add_argument("--cp", type=int, default=0,
                    help="context-parallel split of one sequence over N ranks (emulated on one GPU when run alone)")
    ap.add_argument("--rope", choices=sorted(ROPE_PLACEMENTS), default=None,
                    help="rotate q, k (pre-rotary inputs) inside each step before the attention")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other workloads and rows that the default run also measures")
    ap.add_argument("--extra-steps", type=int, default=50, help="timed steps of each extra measurement")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        line = run_reference(args)
        line["n_gpus"] = world
        print(json.dumps(line), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        from differential_attention_diffattn_gb300 import workloads as W
        if args.workload in W.KV_WORKLOADS:
            runner = run_ours_kv
        elif args.cp:
            runner = run_ours_cp
        else:
            runner = run_ours_bwd if args.backward else run_ours
        line = runner(args, rank, world, local_rank)
        default_run = (runner is run_ours and args.workload == WORKLOAD and args.rope is None and
                       not args.out_proj)
        if line is not None and world == 1 and default_run and not args.no_extras:
            line["per_config"], line["next"] = run_extras(args, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
