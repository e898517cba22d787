"""Benchmark of the KDA hot path on GB300: prefill tokens/s and decode tokens/s.

One step = one pass of the whole path over one batch of synthetic input:
  * an L2 flush (a 256 MB write, larger than the 129 MB L2; the prefill
    inputs of this workload would otherwise stay cached between steps),
  * one kda_chunk_prefill over the 4096-token prefill workload
    (B=1, H=16, dk=dv=128, bf16, float32 initial state 0.1*N(0,1)),
  * 128 consecutive kda_decode_step calls over the decode workload
    (256 sequences, H=32, dk=dv=128, bf16 inputs, 537 MB float32 state,
    read and written in place every step; the state is larger than L2).
`value` is prefill tokens/s (tokens of the sequence per second of device time
of the prefill calls); `decode.value` is decode tokens/s (sequences x steps per
second of device time of the decode calls).  `e2e` repeats both through the
same C ABI with the per-step inputs in pinned host memory, the host->device
copies of inputs and the device->host copies of outputs inside the timed
region.

`--impl reference` times the fp64 CPU oracle (the correctness yardstick, not
a tuned program) on bounded samples of the same workloads.

Multi-GPU (torchrun): every rank runs its own independent copy of the
workloads (seeded by rank), no collective on the data path; timings are
bracketed by barriers and the max over ranks is reported.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA prefill tokens/s and decode tokens/s on 1 GB300; % of tensor/HBM roofline"
HBM_FALLBACK_GBS = 6800.0


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return HBM_FALLBACK_GBS, "fallback"


def _src_sha(name):
    path = os.path.join(ROOT, "gated_delta_rule_46_gb300", "csrc", name)
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def _packed_layout(tensors):
    """Byte offsets of named tensors packed into one buffer (256-byte aligned
    pieces): (layout, total bytes, views(buf) -> the tensors as views of buf).
    One pinned buffer per step then crosses to the device in one copy."""
    layout, nbytes = {}, 0
    for n, t in tensors.items():
        size = t.numel() * t.element_size()
        layout[n] = (nbytes, t.dtype, tuple(t.shape), size)
        nbytes += (size + 255) // 256 * 256

    def views(buf):
        return {n: buf[o:o + sz].view(dt).view(shp) for n, (o, dt, shp, sz) in layout.items()}
    return layout, nbytes, views


def _ncu_traffic(kernel_key, src_file):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel source has changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)[kernel_key]
        if d.get("source_sha") != _src_sha(src_file):
            return None
        return int(d["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.result = {"sm_mhz": None, "sm_max_mhz": None, "reasons": []}
        if self.proc is None:
            return False
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if sm:
            self.result = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                           "reasons": sorted(reasons), "samples": len(sm)}
        return False


def max_over_ranks(x, world, device):
    """The largest of every rank's x (the slowest rank's time): one all-reduce
    on `device` (the GPU under NCCL, the CPU under gloo); x itself when alone."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# --------------------------------------------------------------------------- CPU arms

def _oracle_sample(budget_s=12.0, threads=None):
    """The oracle on bounded samples: the full prefill workload repeated until
    about half the budget is spent, and a slice of the decode workload."""
    import numpy as np
    import oracle
    from gated_delta_rule_46_gb300 import inputs
    threads = threads or (os.cpu_count() or 1)
    oracle.build()
    w1 = inputs.workload(1)
    d = inputs.prefill_inputs(w1)
    reps, t_pref = 0, 0.0
    while t_pref < budget_s / 2 or reps == 0:
        t0 = time.perf_counter()
        oracle.prefill(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], d["cu_seqlens"],
                       d["initial_state"], threads=threads)
        t_pref += time.perf_counter() - t0
        reps += 1
    pref_tps = reps * w1.total_tokens / t_pref
    w4 = inputs.workload(4)
    A = inputs.decode_A(w4)
    st = inputs.initial_state(w4).double().numpy()
    steps, t_dec = 0, 0.0
    while t_dec < budget_s / 2 or steps == 0:
        dd = inputs.decode_inputs(w4, steps % w4.decode_steps)
        t0 = time.perf_counter()
        _, st = oracle.decode_step(dd["q"], dd["k"], dd["v"], dd["z"], A, dd["beta"], st,
                                   threads=threads)
        t_dec += time.perf_counter() - t0
        steps += 1
    dec_tps = steps * w4.decode_N / t_dec
    sample = (f"prefill workload (1 x 4096 tokens, H=16, d=128) run in full {reps}x; "
              f"decode workload (256 seqs, H=32, d=128) {steps} of its 128 steps; fp64 "
              f"token-serial oracle, one thread per (sequence, head) chain")
    return pref_tps, dec_tps, threads, sample, t_pref + t_dec, reps, steps


def run_reference(args):
    rank, world, _ = _dist()
    if rank != 0:
        return 0
    t_start = time.perf_counter()
    pref_tps, dec_tps, cores, sample, cpu_s, reps, steps = _oracle_sample(
        budget_s=max(4.0, 3.0 * (args.steps + args.warmup)))
    wall = time.perf_counter() - t_start
    line = {
        "impl": "reference", "metric": METRIC, "value": pref_tps, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * 4096 / pref_tps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "KDA prefill B=1 H=16 T=4096 dk=dv=128 (oracle on host cores); "
                               "decode N=256 H=32 dk=dv=128",
                   "global_batch": 1, "seq_len": 4096, "parallelism": "none (CPU threads)"},
        "decode": {"value": dec_tps, "unit": "tokens/s"},
        "cpu_baseline": {"value": pref_tps, "unit": "tokens/s", "cores": cores,
                         "kind": "oracle", "sample": sample, "decode_value": dec_tps},
        "e2e": {"value": pref_tps, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "wall_s": wall,
    }
    print(json.dumps(line))
    return 0


# --------------------------------------------------------------------------- GPU arm

def run_gpu(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import gated_delta_rule_46_gb300 as kda
    from gated_delta_rule_46_gb300 import inputs

    rank, world, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    seed = rank
    kda.lib()

    # ---- prefill workload, resident in HBM
    w1 = inputs.workload(1)
    d1 = inputs.prefill_inputs(w1, seed)
    g1 = {n: (t.to(dev) if isinstance(t, torch.Tensor) else t) for n, t in d1.items()}
    T1, H1 = w1.total_tokens, w1.H
    out1 = torch.empty((T1, H1, 128), dtype=torch.bfloat16, device=dev)
    fin1 = torch.empty((1, H1, 128, 128), dtype=torch.float32, device=dev)
    ws1 = torch.zeros(kda.workspace_size(T1, 1, H1, 128, 128), dtype=torch.uint8, device=dev)
    L_pref = kda.prefill_kernel_launches(T1, 1, H1, 128, 128, torch.bfloat16, ws1.numel())
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)   # 256 MB > L2

    # ---- decode workload: 128 steps of inputs pre-generated on the device
    w4 = inputs.workload(4)
    NS = w4.decode_steps
    A4 = inputs.decode_A(w4, seed).to(dev)
    state = inputs.initial_state(w4, seed).to(dev)
    host_steps = [inputs.decode_inputs(w4, s, seed) for s in range(NS)]
    dsteps = [{n: t.to(dev) for n, t in hs.items()} for hs in host_steps]
    out4 = torch.empty((w4.decode_N, w4.H, 128), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def prefill():
        kda.chunk_prefill(g1["q"], g1["k"], g1["v"], g1["z"], g1["A"], g1["beta"],
                          g1["cu_seqlens"], g1["initial_state"], final_state=fin1, out=out1,
                          workspace=ws1)

    def decode_all():
        for s in range(NS):
            x = dsteps[s]
            kda.decode_step(x["q"], x["k"], x["v"], x["z"], A4, x["beta"], state, out=out4)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        flush.fill_(1.0)
        prefill()
        decode_all()
    barrier()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        e_start.record(stream)
        for i in range(K):
            flush.fill_(float(i))
            ev[i][0].record(stream)
            prefill()
            ev[i][1].record(stream)
            ev[i][2].record(stream)
            decode_all()
            ev[i][3].record(stream)
        e_end.record(stream)
        barrier()
    t_pref = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    t_dec = [ev[i][2].elapsed_time(ev[i][3]) for i in range(K)]
    t_total = e_start.elapsed_time(e_end)

    # ---- end to end through the C ABI with host buffers.  Every step copies its
    # inputs in from pinned host memory and its outputs back out.  The copies run
    # on two copy streams, double-buffered against the compute stream: step i's
    # inputs travel while step i - 1 computes and step i - 1's outputs travel
    # back.  e2e = work / wall time of the whole pipelined run (first copy in to
    # last copy out), so a copy that does not overlap counts in full.
    # the prefill's inputs in one pinned buffer (one copy per step), device
    # buffers of the same layout
    pref_t = {n: t for n, t in d1.items() if isinstance(t, torch.Tensor)}
    _, pref_bytes, pref_views = _packed_layout(pref_t)
    pin = torch.empty(pref_bytes, dtype=torch.uint8).pin_memory()
    for n, v in pref_views(pin).items():
        v.copy_(pref_t[n])
    host_out1 = [torch.empty((T1, H1, 128), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    host_fin1 = [torch.empty((1, H1, 128, 128), dtype=torch.float32).pin_memory() for _ in range(2)]
    # each decode step's inputs (q, k, v, z, beta) likewise
    _, step_bytes, step_views = _packed_layout(host_steps[0])
    pin_steps = []
    for hs in host_steps:
        buf = torch.empty(step_bytes, dtype=torch.uint8).pin_memory()
        for n, v in step_views(buf).items():
            v.copy_(hs[n])
        pin_steps.append(buf)
    host_out4 = [torch.empty((w4.decode_N, w4.H, 128), dtype=torch.bfloat16).pin_memory()
                 for _ in range(NS)]
    h2d_pref = pref_bytes
    d2h_pref = host_out1[0].numel() * 2 + host_fin1[0].numel() * 4
    h2d_dec = NS * step_bytes
    d2h_dec = NS * host_out4[0].numel() * 2
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    gbuf = [torch.empty(pref_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    gb = [pref_views(buf) for buf in gbuf]
    ob = [torch.empty_like(out1) for _ in range(2)]
    fb = [torch.empty_like(fin1) for _ in range(2)]
    dbuf = [torch.empty(step_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    db = [step_views(buf) for buf in dbuf]
    dob = [torch.empty_like(out4) for _ in range(2)]

    def ev():
        return torch.cuda.Event()

    def pipelined(n_items, copy_in, compute, copy_out):
        """n_items steps through the three streams, buffers b = i % 2; returns
        the wall time in seconds (events on the compute stream)."""
        in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        used = [False, False]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        e0.record(stream)
        s_in.wait_event(e0)
        s_out.wait_event(e0)
        for i in range(n_items):
            b = i % 2
            with torch.cuda.stream(s_in):
                if used[b]:
                    s_in.wait_event(comp_done[b])     # compute i - 2 has read buffer b
                copy_in(i, b)
                in_done[b].record(s_in)
            stream.wait_event(in_done[b])
            if used[b]:
                stream.wait_event(out_done[b])        # outputs of i - 2 have left buffer b
            compute(i, b)
            comp_done[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[b])
                copy_out(i, b)
                out_done[b].record(s_out)
            used[b] = True
        stream.wait_event(out_done[0])
        stream.wait_event(out_done[1])
        e1.record(stream)
        barrier()
        return e0.elapsed_time(e1) / 1000.0

    def pref_in(i, b):
        gbuf[b].copy_(pin, non_blocking=True)

    def pref_compute(i, b):
        flush.fill_(float(i))
        x = gb[b]
        kda.chunk_prefill(x["q"], x["k"], x["v"], x["z"], x["A"], x["beta"], x["cu_seqlens"],
                          x["initial_state"], final_state=fb[b], out=ob[b], workspace=ws1)

    def pref_out(i, b):
        host_out1[b].copy_(ob[b], non_blocking=True)
        host_fin1[b].copy_(fb[b], non_blocking=True)

    def dec_in(i, b):
        dbuf[b].copy_(pin_steps[i % NS], non_blocking=True)

    def dec_compute(i, b):
        x = db[b]
        kda.decode_step(x["q"], x["k"], x["v"], x["z"], A4, x["beta"], state, out=dob[b])

    def dec_out(i, b):
        host_out4[i % NS].copy_(dob[b], non_blocking=True)

    pipelined(2, pref_in, pref_compute, pref_out)            # warm-up of the streams
    e2e_pref_s = pipelined(K, pref_in, pref_compute, pref_out)
    e2e_dec_s = pipelined(K * NS, dec_in, dec_compute, dec_out)
    # the copies alone (no compute), for the achieved host<->device rate
    t_copy = pipelined(K, pref_in, lambda i, b: None, pref_out)
    copy_gbs = K * (h2d_pref + d2h_pref) / t_copy / 1e9

    def agg_max(x):
        return max_over_ranks(x, world, dev)

    tp = agg_max(sum(t_pref) / 1000.0)
    td = agg_max(sum(t_dec) / 1000.0)
    tt = agg_max(t_total / 1000.0)
    e2p = agg_max(e2e_pref_s)
    e2d = agg_max(e2e_dec_s)
    ok_status = kda.check_device_status(ws1)

    pref_tokens = world * K * T1
    dec_tokens = world * K * NS * w4.decode_N
    value = pref_tokens / tp
    dec_value = dec_tokens / td

    peak, peak_kind = _peaks()
    alg_pref = (T1 * H1 * inputs.bytes_per_token_head(128, 128, 2)
                + 2 * H1 * 128 * 128 * 4 + H1 * 128 * 4 + 8)
    alg_dec = (w4.decode_N * w4.H * (2 * 128 * 128 * 4 + inputs.bytes_per_token_head(128, 128, 2))
               + w4.H * 128 * 4)
    per_launch_pref = (sum(t_pref) / K) / 1000.0
    per_launch_dec = (sum(t_dec) / (K * NS)) / 1000.0
    ach_pref = alg_pref / per_launch_pref / 1e9
    ach_dec = alg_dec / per_launch_dec / 1e9
    traffic_dec = _ncu_traffic("decode_kernel", "kda_simt.cu")
    roof_dec = {"kernel": "decode_kernel<bf16,128,128>", "bound": "hbm", "achieved": ach_dec,
                "peak": peak, "unit": "GB/s", "frac": ach_dec / peak,
                "traffic": traffic_dec,
                "algorithmic_bytes_per_launch": alg_dec, "peak_source": peak_kind,
                "us_per_launch": per_launch_dec * 1e6}
    if traffic_dec:   # the same launch time over the DRAM bytes ncu counted
        roof_dec["frac_dram"] = traffic_dec / per_launch_dec / 1e9 / peak
    plan = {2: "schedule + fused prefill_tc_kernel",
            5: "schedule, intra-chunk, segment maps, scan, segment state pass"}.get(
                L_pref, "schedule, then an intra-chunk and a state-pass kernel per window")
    traffic_pref = _ncu_traffic("kda_chunk_prefill_T4096_H16", "kda_prefill_tc.cu")
    roof_pref = {"kernel": f"kda_chunk_prefill ({L_pref} launches: {plan})", "bound": "hbm",
                 "achieved": ach_pref, "peak": peak, "unit": "GB/s", "frac": ach_pref / peak,
                 "traffic": traffic_pref,
                 "algorithmic_bytes_per_launch": alg_pref, "peak_source": peak_kind,
                 "us_per_launch": per_launch_pref * 1e6}
    if traffic_pref:
        roof_pref["frac_dram"] = traffic_pref / per_launch_pref / 1e9 / peak

    # ---- the decode workload through kda_decode_tokens: 8 tokens per call from a
    # slot pool (the 256 states scattered over 512 slots), 16 calls = 128 tokens
    multi = _time_decode_tokens(kda, inputs, w4, dev, seed, barrier, agg_max, peak, peak_kind)

    # ---- ablation: the same prefill through the unbounded log-decay entry point
    # (token-serial kernel), g taken from the bounded gate so both compute one layer
    ablation = _time_unbounded_gate(kda, g1, fin1, out1, ws1, flush, barrier, agg_max, stream,
                                    T1, tp / K)
    # ---- the same prefill without a workspace (kda_chunk_prefill_noalloc)
    noalloc = _time_noalloc(kda, g1, fin1, out1, flush, barrier, agg_max, stream, T1, tp / K)

    # ---- the two large prefill workloads, inputs generated on the device
    extra = {}
    if not args.no_extra_workloads:
        del dsteps, pin_steps, host_steps
        torch.cuda.empty_cache()
        for wid in (2, 3):
            extra[inputs.workload(wid).name] = _time_large_prefill(kda, inputs, wid, dev, seed,
                                                                   flush, barrier, agg_max, peak,
                                                                   peak_kind)
        # the varlen batch through the unbounded-decay path (fused kernel, unbounded mode)
        ablation["varlen"] = _time_large_prefill(kda, inputs, 2, dev, seed, flush, barrier, agg_max,
                                                 peak, peak_kind, unbounded=True)
        # the 4096-token layer in float32 and with 64-channel heads (the chunkwise
        # float32 kernel on the CUDA cores)
        for case in ("prefill-f32", "prefill-d64"):
            name, lens, H = CASES[case]
            dn, dd = CASE_DTYPE[case]
            extra[case] = _time_large_prefill(kda, inputs, 77, dev, seed, flush, barrier, agg_max, peak,
                                              peak_kind, reps=3, lens=lens, H=H, name=name,
                                              dtype_name=dn, d=dd)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        pt, dt, cores, sample, _, _, _ = _oracle_sample(budget_s=12.0)
        cpu = {"value": pt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": sample, "decode_value": dt}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": 1000.0 * tt / K,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "KDA prefill B=1 H=16 T=4096 dk=dv=128 bf16, fp32 init "
                                   "state; + 128 decode steps N=256 H=32 dk=dv=128",
                       "global_batch": world, "seq_len": T1,
                       "parallelism": f"replicas x{world} (independent problems)",
                       "l2": "flushed before every prefill (256 MB write); decode state 537 MB > L2"},
            "decode": {"value": dec_value, "unit": "tokens/s", "us_per_step": per_launch_dec * 1e6,
                       "roofline": roof_dec},
            # `value` is the prefill's tokens/s, so `roofline` is the prefill call's;
            # the decode kernel (most of the step's time) is beside it
            "roofline": roof_pref,
            "roofline_decode": roof_dec,
            "prefill_us_per_call": per_launch_pref * 1e6,
            "e2e": {"value": pref_tokens / e2p, "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d_pref + h2d_dec, "d2h_bytes_per_step": d2h_pref + d2h_dec,
                    "decode_value": dec_tokens / e2d,
                    "copies": "two copy streams, double-buffered against compute",
                    "copy_gbs_alone": copy_gbs},
            "decode_tokens": multi,
            "prefill_large": extra,
            "prefill_unbounded_gate": ablation,
            "prefill_noalloc": noalloc,
            "gpu_launches": K * (L_pref + NS),   # the timed step; decode_tokens and prefill_large are timed apart
            "clocks": clk.result,
            "device_status": ok_status,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def _time_decode_tokens(kda, inputs, w4, dev, seed, barrier, agg_max, peak, peak_kind,
                        n_tok=8, reps=3):
    """The decode workload's 256 sequences x 32 heads stepped n_tok tokens per
    kda_decode_tokens call through a pool of 512 slots (a seeded permutation
    names each sequence's slot), 128 / n_tok calls per pass: the state is read
    and written once per call instead of once per token."""
    import torch
    N, H, d = w4.decode_N, w4.H, 128
    calls = w4.decode_steps // n_tok
    g = torch.Generator(device=dev)
    g.manual_seed(2000 + seed)

    def normal(shape):
        return torch.randn(shape, generator=g, device=dev, dtype=torch.float32)

    q = torch.nn.functional.normalize(normal((calls, N, n_tok, H, d)), dim=-1).to(torch.bfloat16)
    k = torch.nn.functional.normalize(normal((calls, N, n_tok, H, d)), dim=-1).to(torch.bfloat16)
    v = normal((calls, N, n_tok, H, d)).to(torch.bfloat16)
    z = normal((calls, N, n_tok, H, d)).to(torch.bfloat16)
    beta = torch.sigmoid(normal((calls, N, n_tok, H)))
    A = torch.rand((H, d), generator=g, device=dev) * 2 - 1
    pool = 0.1 * normal((2 * N, H, d, d))
    slots = torch.randperm(2 * N, generator=g, device=dev)[:N].to(torch.int32)
    out = torch.empty((N, n_tok, H, d), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def run_pass():
        for c in range(calls):
            kda.decode_tokens(q[c], k[c], v[c], z[c], A, beta[c], pool, slot_ids=slots, out=out)

    run_pass()
    barrier()
    times = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run_pass()
        e1.record(stream)
        barrier()
        times.append(e0.elapsed_time(e1) / 1000.0)
    t = agg_max(min(times))
    per_call = t / calls
    alg = N * H * (2 * d * d * 4 + n_tok * inputs.bytes_per_token_head(d, d, 2)) + H * d * 4 + 4 * N
    ach = alg / per_call / 1e9
    del q, k, v, z, beta, pool
    torch.cuda.empty_cache()
    return {"workload": f"decode {N} seqs x {w4.decode_steps} tokens, H={H}, d={d}, bf16, {n_tok} tokens "
                        f"per kda_decode_tokens call, states in a {2 * N}-slot pool",
            "value": N * w4.decode_steps / t, "unit": "tokens/s", "us_per_call": per_call * 1e6,
            "roofline": {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s",
                         "frac": ach / peak, "algorithmic_bytes_per_launch": alg,
                         "peak_source": peak_kind}}


def _time_unbounded_gate(kda, g1, fin1, out1, ws1, flush, barrier, agg_max, stream, T1,
                        t_bounded, reps=5):
    """The 4096-token prefill through kda_chunk_prefill_logdecay on g = the
    bounded gate's output: the token-serial kernel that an unbounded log-decay
    needs, against the chunked tensor-core path that the bound allows."""
    import torch
    g = kda.gate(g1["z"], g1["A"])
    T, H = g.shape[0], g.shape[1]
    ws_chunked = torch.zeros(kda.logdecay_workspace_size(T, 1, H, 128, 128), dtype=torch.uint8,
                             device=g.device)
    ws_serial = torch.zeros(256, dtype=torch.uint8, device=g.device)

    def timed(ws):
        def call():
            kda.chunk_prefill_logdecay(g1["q"], g1["k"], g1["v"], g, g1["beta"], g1["cu_seqlens"],
                                       g1["initial_state"], final_state=fin1, out=out1, workspace=ws)
        call()
        barrier()
        times = []
        for i in range(reps):
            flush.fill_(float(i))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call()
            e1.record(stream)
            barrier()
            times.append(e0.elapsed_time(e1) / 1000.0)
        return agg_max(min(times))

    t = timed(ws_chunked)
    t_serial = timed(ws_serial)
    del ws_chunked, ws_serial
    return {"workload": f"the same prefill (T={T1}) with the log-decay passed in (g from the bounded "
                        "gate): chunked path with the diagonal tiles summed pair by pair; the L2 "
                        "flushed before each call",
            "us_per_call": t * 1e6, "value": T1 / t, "unit": "tokens/s",
            "token_serial_us_per_call": t_serial * 1e6,
            "bounded_chunked_us_per_call": t_bounded * 1e6}


def _time_noalloc(kda, g1, fin1, out1, flush, barrier, agg_max, stream, T1, t_plan, reps=5):
    """The 4096-token prefill through kda_chunk_prefill_noalloc: no caller
    workspace, so always the one-kernel plan (here 16 chains on 16 CTA
    slots), against the segment-scan plan that the workspace allows."""
    import torch

    def call():
        kda.chunk_prefill_noalloc(g1["q"], g1["k"], g1["v"], g1["z"], g1["A"], g1["beta"], g1["cu_seqlens"],
                                  g1["initial_state"], final_state=fin1, out=out1)
    call()
    barrier()
    times = []
    for i in range(reps):
        flush.fill_(float(i))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        barrier()
        times.append(e0.elapsed_time(e1) / 1000.0)
    t = agg_max(min(times))
    return {"workload": f"the same prefill (T={T1}) through kda_chunk_prefill_noalloc: no workspace, "
                        "so the one-kernel plan (one CTA per chain); the L2 flushed before each call",
            "us_per_call": t * 1e6, "value": T1 / t, "unit": "tokens/s",
            "segment_scan_us_per_call": t_plan * 1e6}


# Prefill cases timed on their own (`--case`), e.g. as the command an ncu
# capture runs: (name, workload id or sequence lengths, H).
CASES = {
    "prefill": ("prefill", 1, None),
    "varlen": ("varlen", 2, None),
    "long": ("long", 3, None),
    # the fused (many-chain) plan at a size an ncu capture can replay: 1.4 GB
    "fused-16x2048": ("fused-16x2048: 16 seqs x 2048 tokens", [2048] * 16, 32),
    # the 4096-token workload through kda_chunk_prefill_logdecay (g from the
    # bounded gate): the chunked path for an unbounded log-decay
    "prefill-unbounded": ("prefill-unbounded", 1, None),
    # a 65,536-token sequence with 32 heads: the windowed split plan (as the
    # 1M-token workload runs it) at a size an ncu capture can replay
    "long-64k": ("long-64k: 1 seq x 65536 tokens", [65536], 32),
    # the 4096-token layer in float32 and with 64-channel heads: the chunkwise
    # float32 kernel on the CUDA cores
    "prefill-f32": ("prefill-f32: 1 seq x 4096 tokens, float32", [4096], 16),
    "prefill-d64": ("prefill-d64: 1 seq x 4096 tokens, dk=dv=64", [4096], 16),
}
CASE_DTYPE = {"prefill-f32": ("float32", 128), "prefill-d64": ("bfloat16", 64)}
UNBOUNDED_CASES = {"prefill-unbounded"}


def _time_large_prefill(kda, inputs, wid, dev, seed, flush, barrier, agg_max, peak, peak_kind,
                        reps=2, warm=1, lens=None, H=None, name=None, unbounded=False,
                        dtype_name="bfloat16", d=128):
    """One KDA layer over a packed batch (by default the varlen or the 1M-token
    workload `wid`): inputs drawn on the device with the same distributions as
    the parity inputs (bf16 q/k L2-normalised, v/z N(0,1), beta = sigmoid(N(0,1)),
    A ~ U(-1,1), zero initial state), outputs and final states written."""
    import torch
    if lens is None:
        w = inputs.workload(wid)
        lens, H, name = list(w.seq_lens), w.H, w.name
    T = sum(lens)
    dt = getattr(torch, dtype_name)
    g = torch.Generator(device=dev)
    g.manual_seed(1000 + 7 * wid + seed)

    def normal(shape):
        return torch.randn(shape, generator=g, device=dev, dtype=torch.float32)

    q = torch.nn.functional.normalize(normal((T, H, d)), dim=-1).to(dt)
    k = torch.nn.functional.normalize(normal((T, H, d)), dim=-1).to(dt)
    v = normal((T, H, d)).to(dt)
    z = normal((T, H, d)).to(dt)
    beta = torch.sigmoid(normal((T, H)))
    A = torch.rand((H, d), generator=g, device=dev) * 2 - 1
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32, device=dev)
    cu[1:] = torch.cumsum(torch.tensor(lens, device=dev), 0)
    N = len(lens)
    out = torch.empty((T, H, d), dtype=dt, device=dev)
    fin = torch.empty((N, H, d, d), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    if unbounded:   # the log-decay passed in (here the bounded gate's values)
        gd = kda.gate(z, A)
        ws = torch.zeros(kda.logdecay_workspace_size(T, N, H, d, d), dtype=torch.uint8, device=dev)

        def call():
            kda.chunk_prefill_logdecay(q, k, v, gd, beta, cu, None, final_state=fin, out=out, workspace=ws)
    else:
        ws = torch.zeros(kda.workspace_size(T, N, H, d, d), dtype=torch.uint8, device=dev)

        def call():
            kda.chunk_prefill(q, k, v, z, A, beta, cu, None, final_state=fin, out=out, workspace=ws)

    for _ in range(warm):
        call()
    barrier()
    times = []
    for _ in range(reps):
        flush.fill_(0.5)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        barrier()
        times.append(e0.elapsed_time(e1) / 1000.0)
    t = agg_max(min(times))
    alg = T * H * inputs.bytes_per_token_head(d, d, dt.itemsize) + N * H * d * d * 4 + H * d * 4 + 4 * (N + 1)
    ach = alg / t / 1e9
    status = kda.check_device_status(ws)
    del q, k, v, z, out, ws
    torch.cuda.empty_cache()
    return {"workload": f"{name}: {N} seqs, {T} tokens, H={H}, dk=dv={d}, {dtype_name}, zero state",
            "value": T / t, "unit": "tokens/s", "ms_per_call": 1000 * t,
            "roofline": {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s",
                         "frac": ach / peak, "algorithmic_bytes_per_launch": alg,
                         "peak_source": peak_kind},
            "device_status": status}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-workloads", action="store_true",
                    help="skip the varlen and 1M-token prefill measurements")
    ap.add_argument("--case", choices=sorted(CASES),
                    help="time one prefill case alone (--warmup untimed, --steps timed calls) "
                         "and print its JSON line; no decode, no CPU baseline")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.case:
        return run_case(args)
    return run_gpu(args)


def run_case(args):
    import torch
    import gated_delta_rule_46_gb300 as kda
    from gated_delta_rule_46_gb300 import inputs
    dev = torch.device("cuda", 0)
    kda.lib()
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)   # 256 MB > L2
    name, spec, H = CASES[args.case]
    peak, peak_kind = _peaks()
    kw = {} if isinstance(spec, int) else {"lens": spec, "H": H, "name": name}
    if args.case in CASE_DTYPE:
        kw["dtype_name"], kw["d"] = CASE_DTYPE[args.case]
    wid = spec if isinstance(spec, int) else 77
    r = _time_large_prefill(kda, inputs, wid, dev, 0, flush, torch.cuda.synchronize,
                            lambda x: x, peak, peak_kind, reps=args.steps, warm=args.warmup,
                            unbounded=args.case in UNBOUNDED_CASES, **kw)
    r.update({"case": args.case, "steps": args.steps, "warmup": args.warmup,
              "l2": "flushed before every timed call (256 MB write)"})
    print(json.dumps(r))
    return 0


if __name__ == "__main__":
    sys.exit(main())
