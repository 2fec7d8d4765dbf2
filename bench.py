"""Benchmark: KDA prefill tokens/s on the K3-shaped layer (B=1, T=4096, H=96,
d_k=d_v=128, bf16 q/k/v, fp32 log_alpha/beta/state; the kernel walks 32-token
chunks, which gives the same result as any other chunk length), with the
roofline of the prefill kernel, plus the decode step (B=256, H=96, 64 in-place
steps) in GB/s against HBM, the fp64 CPU oracle timed on this host, and an
end-to-end number through host buffers. Prints ONE JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torch.distributed (one process per GPU): every rank runs its
own independent copy of the workload (weak scaling, no collective on the data
path); the timed region is bracketed by barriers and the max over ranks is kept.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

PREFILL = dict(workload="prefill_k3_T4096_H96", T=4096, H=96, d_k=128, d_v=128, chunk=32)
# the recipe both CPU baselines (ours' cpu_baseline and the reference arm) time, one step each
ORACLE_SAMPLE = ("{heads} of {H} heads x {T} tokens per step: the whole workload, fp64 token-recurrent C oracle "
                 "on the host's cores (the reference arm and cpu_baseline time this same sample)")
DECODE = dict(B=256, H=96, d_k=128, d_v=128, steps=64)
METRIC = "KDA prefill tokens/s (H=96,d=128) & % tensor roofline; decode GB/s vs HBM"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, 1700.0, "fallback"


# Algorithmic work of the chunked prefill (chunk C = 64, d_k = d_v = 128), per token-head:
#   bytes: q, k, v bf16 (3 x 256) + log_alpha fp32 (512) + beta (4) + out fp32 (512) = 1796
#   flops: 6 d_k d_v + C (3 d_k + 2 d_v) with C = 64 = 139,264 (the pages' chunk; triangular work once)
# plus the fp32 state read once and written once per (sequence, head): 2 x 64 KiB.
PREFILL_BYTES_PER_TOKEN_HEAD = 1796
PREFILL_STATE_BYTES_PER_SEQ_HEAD = 2 * 128 * 128 * 4
PREFILL_FLOPS_PER_TOKEN_HEAD = 6 * 128 * 128 + 64 * (3 * 128 + 2 * 128)
# the gated log-decay form reads bf16 logits z instead of fp32 log_alpha: 768 + 256 + 4 + 512 = 1540
GATED_BYTES_PER_TOKEN_HEAD = 1540
# gated decay + output gate (bf16 gate logits in, bf16 output): 768 + 256 + 4 + 256 + 256 = 1540
OUTGATE_BYTES_PER_TOKEN_HEAD = 1540
# input prologue: raw q, k, v read + processed q, k, v written, bf16: 2 x 3 x 256 = 1536
PROLOGUE_BYTES_PER_TOKEN_HEAD = 1536
# decode, per (sequence, head): state read + write (131,072) + q,k,v bf16 (768) + log_alpha (512)
# + beta (4) + out fp32 (512) = 132,868 bytes
DECODE_BYTES_PER_SEQ_HEAD = 2 * 128 * 128 * 4 + 3 * 256 + 512 + 4 + 512
# fused decode step: state read + write (131,072) + raw q,k,v (768) + z (256) + beta (4) + gate logits
# (256) + out bf16 (256) + conv state read + write (2 x 3 x 384 x 2 = 4,608) = 137,220 bytes
FUSED_DECODE_BYTES_PER_SEQ_HEAD = 2 * 128 * 128 * 4 + 3 * 256 + 256 + 4 + 256 + 256 + 2 * 3 * 384 * 2


class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device="cuda") -> float:
    """The slowest rank's time: every rank's timed region ends at the same barrier."""
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(world: int, tokens_per_rank: int, ms_per_step: float) -> float:
    """Whole-job tokens/s: every rank processes its own copy of the workload."""
    return world * tokens_per_rank / (ms_per_step / 1e3)


def prefill_traffic():
    """DRAM bytes (read + write) of one prefill launch on the headline workload, from the ncu
    capture recorded in profiles/prefill_traffic.json, or None when the kernel sources have
    changed since that capture (the record carries a hash of them)."""
    path = os.path.join(ROOT, "profiles", "prefill_traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh)
        h = hashlib.sha256()
        for rel in rec["sources"]:
            with open(os.path.join(ROOT, rel), "rb") as fh:
                h.update(fh.read())
    except (OSError, KeyError, ValueError):
        return None
    return rec.get("bytes_per_launch") if h.hexdigest() == rec.get("sources_sha256") else None


def time_prefill(case, steps, warmup, world, gated=False, out_gate=False, unbounded=False, recurrent=False):
    from kimi_delta_attention_02_gb300 import binding
    out_dtype = torch.float32
    if unbounded:  # the earlier models' unbounded decay map (chunked kernel, or forced token-recurrent)
        args = ()

        def fn(out, final_state, stream):
            binding.prefill_ex(case.q, case.k, case.v, case.beta, case.cu_seqlens, z=case.z, A_log=case.A_log,
                               init_state=case.init_state, unbounded=True, recurrent=recurrent, out=out,
                               final_state=final_state, stream=stream)
    elif out_gate:  # gated decay, output gate, bf16 output: the parameter-block entry point
        out_dtype = torch.bfloat16
        args = ()

        def fn(out, final_state, stream):
            binding.prefill_ex(case.q, case.k, case.v, case.beta, case.cu_seqlens, z=case.z, A_log=case.A_log,
                               init_state=case.init_state, out_gate=case.out_gate, norm_weight=case.norm_weight,
                               out=out, final_state=final_state, stream=stream)
    elif gated:
        fn = binding.prefill_gated
        args = (case.q, case.k, case.v, case.z, case.A_log, case.beta, case.cu_seqlens, case.init_state)
    else:
        fn = binding.prefill
        args = (case.q, case.k, case.v, case.log_alpha, case.beta, case.cu_seqlens, case.init_state)
    out = torch.empty(case.v.shape, dtype=out_dtype, device=case.v.device)
    fin = torch.empty_like(case.init_state)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        fn(*args, out=out, final_state=fin, stream=stream)
    binding.check_device_error(stream)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(steps):
        starts[i].record(stream)
        fn(*args, out=out, final_state=fin, stream=stream)
        ends[i].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    binding.check_device_error(stream)
    total_ms = t0.elapsed_time(t1)
    launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return total_ms, launch_ms


def time_named_prefill(name, steps, warmup, world, seed=0, workspace="auto"):
    """kda_prefill on one named workload (built on the device, freed afterwards): per-launch ms,
    total tokens, heads and sequences."""
    from kimi_delta_attention_02_gb300 import binding, workloads
    case = workloads.prefill_workload(name, device="cuda", seed=seed)
    out = torch.empty(case.v.shape, dtype=torch.float32, device="cuda")
    fin = torch.empty((case.num_seqs,) + tuple(case.q.shape[1:]) + (case.v.shape[-1],), dtype=torch.float32,
                      device="cuda")
    stream = torch.cuda.current_stream()

    def run():
        binding.prefill(case.q, case.k, case.v, case.log_alpha, case.beta, case.cu_seqlens, case.init_state,
                        out=out, final_state=fin, stream=stream, workspace=workspace)
    for _ in range(warmup):
        run()
    binding.check_device_error(stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    for a, b in ev:
        a.record(stream)
        run()
        b.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    binding.check_device_error(stream)
    T, H, N = case.total_tokens, case.num_heads, case.num_seqs
    in_bytes = sum(t.numel() * t.element_size() for t in (case.q, case.k, case.v, case.log_alpha, case.beta))
    del case, out, fin
    torch.cuda.empty_cache()
    return [a.elapsed_time(b) for a, b in ev], T, H, N, in_bytes


def prefill_line(name, ms, T, H, N, world, hbm_gbs, tf_burst, in_bytes, note):
    """One workload's numbers: launch time, tokens/s and the HBM and tensor fractions of the
    algorithmic work (fp32 output; 1,796 B per token-head with fp32 log_alpha, plus the states)."""
    launch = sum(ms) / len(ms)
    alg = T * H * PREFILL_BYTES_PER_TOKEN_HEAD + N * H * PREFILL_STATE_BYTES_PER_SEQ_HEAD
    if in_bytes != T * H * (PREFILL_BYTES_PER_TOKEN_HEAD - 512):  # fp32 q/k/v: count the bytes read
        alg = in_bytes + T * H * 512 + N * H * PREFILL_STATE_BYTES_PER_SEQ_HEAD
    gbs = alg / (launch / 1e3) / 1e9
    tf = T * H * PREFILL_FLOPS_PER_TOKEN_HEAD / (launch / 1e3) / 1e12
    return {"workload": name, "launch_ms": launch, "tokens_per_s": world * T / (launch / 1e3),
            "token_heads_per_s": world * T * H / (launch / 1e3), "GB/s": gbs, "peak": hbm_gbs,
            "frac": gbs / hbm_gbs, "tensor_frac": tf / tf_burst, "alg_bytes": alg, "launches": len(ms),
            "hbm_bound_ms": alg / hbm_gbs / 1e6, "kernel": note}


def time_decode(steps_per_rep, reps, warmup, world, seed=0, fused=False):
    """Decode steps on B=256 sequences, H=96. ``fused``: the whole layer step between the
    projections -- the prologue on raw q, k, v (conv state shifted in place), the gated decay,
    the recurrence and the output gate (bf16 out) -- in one kernel per step."""
    from kimi_delta_attention_02_gb300 import binding, workloads
    B, H = DECODE["B"], DECODE["H"]
    state = workloads.make_decode_state(B, H, device="cuda", seed=seed)
    inputs = [workloads.make_decode_step(s, B, H, dtype=torch.bfloat16, device="cuda", seed=seed, gated=fused,
                                         out_gate=fused) for s in range(steps_per_rep)]
    out = torch.empty((B, H, 128), dtype=torch.bfloat16 if fused else torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    if fused:
        conv_w = workloads.make_conv_weight(H, device="cuda", seed=seed)
        conv_state = workloads.make_conv_state(B, H, device="cuda", seed=seed)

        def step_fn(st):
            binding.decode_ex(st.q, st.k, st.v, st.beta, state, z=st.z, A_log=st.A_log, out_gate=st.out_gate,
                              norm_weight=st.norm_weight, conv_weight=conv_w, conv_state=conv_state, out=out,
                              stream=stream)
    else:
        def step_fn(st):
            binding.decode(st.q, st.k, st.v, st.log_alpha, st.beta, state, out=out, stream=stream)
    for _ in range(warmup):
        for st in inputs:
            step_fn(st)
    binding.check_device_error(stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps * steps_per_rep)]
    barrier(world)
    torch.cuda.synchronize()
    i = 0
    for _ in range(reps):
        for st in inputs:
            ev[i][0].record(stream)
            step_fn(st)
            ev[i][1].record(stream)
            i += 1
    torch.cuda.synchronize()
    barrier(world)
    binding.check_device_error(stream)
    return [a.elapsed_time(b) for a, b in ev]


def time_prologue(steps, warmup, world, seed=0, H=None):
    """The input prologue (ShortConv, Swish, L2 norm) on the K3-shaped layer's raw projections,
    T=4096, H=96 (or H), bf16, with initial and final convolution states. Returns per-launch ms."""
    from kimi_delta_attention_02_gb300 import binding, workloads
    case = workloads.make_prologue([PREFILL["T"]], H=H or PREFILL["H"], device="cuda", seed=seed)
    q, k, v = torch.empty_like(case.q_raw), torch.empty_like(case.k_raw), torch.empty_like(case.v_raw)
    fin = torch.empty_like(case.conv_init)
    stream = torch.cuda.current_stream()

    def run():
        binding.prologue(case.q_raw, case.k_raw, case.v_raw, case.conv_weight, case.cu_seqlens, case.conv_init,
                         q=q, k=k, v=v, conv_final=fin, stream=stream)
    for _ in range(warmup):
        run()
    binding.check_device_error(stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    for a, b in ev:
        a.record(stream)
        run()
        b.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    binding.check_device_error(stream)
    return [a.elapsed_time(b) for a, b in ev]


def time_e2e(case_cpu, steps, warmup):
    """Prefill through pinned host buffers: every step copies its inputs host -> device, runs
    kda_prefill and copies out + final state back to pinned host memory. Steps are streamed
    (binding.HostPrefillStream): the next step's inputs travel while the current one computes.
    Also timed: the same with one copy stream for both directions ("half duplex": the kernel
    still overlaps the copies, the two directions never do), and one step at a time.
    Returns ({mode: ms per step}, h2d bytes, d2h bytes)."""
    from kimi_delta_attention_02_gb300 import binding
    hp = binding.HostPrefillStream(case_cpu.q, case_cpu.k, case_cpu.v, case_cpu.log_alpha, case_cpu.beta,
                                   case_cpu.cu_seqlens, case_cpu.init_state)
    ms = {}
    for mode in ("streamed", "half duplex"):
        hp.run(warmup, duplex=mode == "streamed")
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        hp.run(steps, duplex=mode == "streamed")
        torch.cuda.synchronize()
        ms[mode] = (time.perf_counter() - t0) * 1e3 / steps
    t0 = time.perf_counter()
    for _ in range(steps):
        hp.run(1)
    ms["one step at a time"] = (time.perf_counter() - t0) * 1e3 / steps
    return ms, hp.h2d_bytes, hp.d2h_bytes


def cpu_oracle_sample(case_cpu, heads: int, threads: int = 0):
    """fp64 oracle on the first `heads` heads of the workload on `threads` host threads (0: every
    core); returns (seconds, threads used, token-heads)."""
    from oracle import kda_recurrent
    threads = threads or os.cpu_count() or 1
    sl = lambda t: t[:, :heads].contiguous()
    init = case_cpu.init_state[:, :heads].contiguous()
    cu = case_cpu.cu_seqlens.long().numpy()
    t0 = time.perf_counter()
    kda_recurrent(sl(case_cpu.q), sl(case_cpu.k), sl(case_cpu.v), sl(case_cpu.log_alpha), sl(case_cpu.beta), cu,
                  init_state=init, num_threads=threads)
    dt = time.perf_counter() - t0
    return dt, min(threads, heads * (cu.shape[0] - 1)), case_cpu.total_tokens * heads


def run_reference(args, world, rank):
    """The reference arm: the fp64 CPU oracle as it stands, on host cores, rank 0 only."""
    if rank != 0:
        return None
    from kimi_delta_attention_02_gb300 import workloads
    case = workloads.prefill_workload(PREFILL["workload"], device="cpu", seed=0)
    heads = PREFILL["H"]  # the same sample as ours' cpu_baseline: every head, about a second per step
    for _ in range(args.warmup):
        cpu_oracle_sample(case, heads)
    times = []
    cores = 0
    for _ in range(args.steps):
        dt, cores, th = cpu_oracle_sample(case, heads)
        times.append(dt)
    step_s = sum(times) / len(times)
    tok_s = PREFILL["T"] * heads / PREFILL["H"] / step_s  # full-workload tokens/s equivalent
    line = {"impl": "reference", "metric": METRIC, "value": tok_s, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": PREFILL["workload"], "global_batch": 1, "seq_len": PREFILL["T"],
                       "heads": PREFILL["H"], "d_k": 128, "d_v": 128, "parallelism": "cpu threads"},
            "cpu_baseline": {"value": tok_s, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": ORACLE_SAMPLE.format(heads=heads, H=PREFILL["H"], T=PREFILL["T"])},
            "e2e": {"value": tok_s, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--heads", type=int, default=PREFILL["H"],
                    help="prefill heads (a smaller value is for profiler captures; the headline uses 96)")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time the prefill kernel only (no decode, e2e or CPU baseline): for profiler captures")
    ap.add_argument("--form", choices=["clamped", "gated", "outgate", "unbounded", "unbounded-steep", "fused"],
                    default="clamped",
                    help="with --prefill-only: the decay form timed (unbounded-steep: logits +40 on every "
                         "third channel, so that every chunk takes the position-pair step)")
    ap.add_argument("--decode-only", type=int, default=0, metavar="STEPS",
                    help="run STEPS decode steps on B=256, H=96 (plain, or with --form fused the whole layer "
                         "step) after 3 warm-up ones and print their mean time: for profiler captures")
    ap.add_argument("--prologue-only", action="store_true",
                    help="time the input prologue pass only (T=4096, --heads heads): for profiler captures")
    ap.add_argument("--workload", default=None,
                    help="with --prefill-only: time kda_prefill on this named workload instead (e.g. "
                         "prefill_f32_T256_H2, prefill_varlen8_H96), with the workspace it asks for")
    args = ap.parse_args()
    if args.form != "clamped" and not (args.prefill_only or args.decode_only):
        ap.error("--form goes with --prefill-only or --decode-only")
    if args.decode_only and args.form not in ("clamped", "fused"):
        ap.error("--decode-only takes --form clamped (plain) or fused")
    if args.form == "fused" and not args.decode_only:
        ap.error("--form fused goes with --decode-only")
    if sum(map(bool, (args.prefill_only, args.decode_only, args.prologue_only))) > 1:
        ap.error("--prefill-only, --decode-only and --prologue-only exclude one another")
    args.warmup = max(args.warmup, 3)

    if args.impl == "reference":
        # rank 0 alone times the CPU oracle; other ranks exit without work
        run_reference(args, int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")))
        return
    world, rank, local = dist_setup(args)

    from kimi_delta_attention_02_gb300 import binding, workloads
    binding.lib()
    hbm_gbs, tf_burst, tf_sust, peak_src = peaks()

    if args.prologue_only:
        p_ms = time_prologue(args.steps, args.warmup, world, seed=rank, H=args.heads)
        if rank == 0:
            print(json.dumps({"prologue_only": True, "heads": args.heads, "launch_ms": sum(p_ms) / len(p_ms)}),
                  flush=True)
        return
    if args.workload is not None:
        if not args.prefill_only:
            ap.error("--workload goes with --prefill-only")
        ms, *_ = time_named_prefill(args.workload, args.steps, args.warmup, world, seed=rank)
        if rank == 0:
            print(json.dumps({"prefill_only": True, "workload": args.workload, "launch_ms": sum(ms) / len(ms)}),
                  flush=True)
        return
    if args.decode_only:
        ms = time_decode(args.decode_only, 1, 3, world, seed=rank, fused=args.form == "fused")
        if rank == 0:
            print(json.dumps({"decode_only": True, "form": args.form, "steps": args.decode_only,
                              "ms_per_step": sum(ms) / len(ms)}), flush=True)
        return
    logits = args.form != "clamped"
    if args.heads == PREFILL["H"]:
        name = {"clamped": PREFILL["workload"], "outgate": "prefill_k3_outgate_T4096_H96"}.get(
            args.form, "prefill_k3_gated_T4096_H96")
        case = workloads.prefill_workload(name, device="cuda", seed=rank)
    else:
        case = workloads.make_prefill([PREFILL["T"]], H=args.heads, device="cuda", seed=rank, gated=logits,
                                      out_gate=args.form == "outgate")
    if args.form == "unbounded-steep":
        case.z[:, :, ::3] = 40.0
    T, H = case.total_tokens, case.num_heads
    with ClockSampler(local) as clocks:
        total_ms, launch_ms = time_prefill(case, args.steps, args.warmup, world, gated=args.form == "gated",
                                           out_gate=args.form == "outgate",
                                           unbounded=args.form.startswith("unbounded"))
        dec_ms = None if args.prefill_only else time_decode(DECODE["steps"], 1, 1, world, seed=rank)
        gated_ms = outgate_ms = prologue_ms = unbounded_ms = unbounded_rec_ms = unbounded_steep_ms = fdec_ms = None
        extra = {}
        if not args.prefill_only and args.heads == PREFILL["H"]:
            gcase = workloads.prefill_workload("prefill_k3_gated_T4096_H96", device="cuda", seed=rank)
            _, g_launch = time_prefill(gcase, args.steps, args.warmup, world, gated=True)
            gated_ms = sum(g_launch) / len(g_launch)
            del gcase
            ocase = workloads.prefill_workload("prefill_k3_outgate_T4096_H96", device="cuda", seed=rank)
            _, o_launch = time_prefill(ocase, args.steps, args.warmup, world, out_gate=True)
            outgate_ms = sum(o_launch) / len(o_launch)
            del ocase
            p_launch = time_prologue(args.steps, args.warmup, world, seed=rank)
            prologue_ms = sum(p_launch) / len(p_launch)
            fdec_ms = time_decode(DECODE["steps"], 1, 1, world, seed=rank, fused=True)
            ucase = workloads.prefill_workload("prefill_k3_gated_T4096_H96", device="cuda", seed=rank)
            _, u_launch = time_prefill(ucase, args.steps, args.warmup, world, unbounded=True)
            unbounded_ms = sum(u_launch) / len(u_launch)
            _, u_launch = time_prefill(ucase, 3, 1, world, unbounded=True, recurrent=True)  # a few ms per launch
            unbounded_rec_ms = sum(u_launch) / len(u_launch)
            ucase.z[:, :, ::3] = 40.0  # -40 e^{A_h} per step on every third channel: every chunk has wide channels
            _, u_launch = time_prefill(ucase, args.steps, args.warmup, world, unbounded=True)
            unbounded_steep_ms = sum(u_launch) / len(u_launch)
            del ucase
            torch.cuda.empty_cache()
            # the other graded prefill shapes: config 0 (fp32, token-recurrent kernel), the varlen
            # pack and the 1M-token sequence
            extra = {}
            # each with the schedule kda_prefill takes given the workspace it asks for, and without
            # one (one CTA per (sequence, head) chain, in sequence order) for comparison
            for key, name, st, wu, note in (
                    ("config0", "prefill_f32_T256_H2", args.steps, args.warmup, "fp32 token-recurrent"),
                    ("varlen", "prefill_varlen8_H96", 5, 2, "chunked, chains longest sequence first"),
                    ("long_context", "prefill_long_T1M_H32", 3, 1, "chunked, segmented: 3 segments per head")):
                ms, T_, H_, N_, ib = time_named_prefill(name, st, wu, world, seed=rank, workspace="auto")
                extra[key] = prefill_line(name, ms, T_, H_, N_, world, hbm_gbs, tf_burst, ib, note)
                if key != "config0":
                    ms1, *_ = time_named_prefill(name, st, wu, world, seed=rank, workspace=None)
                    one = sum(ms1) / len(ms1)
                    extra[key]["without_workspace"] = {
                        "launch_ms": one, "kernel": "chunked, one CTA per (sequence, head), sequence order",
                        "speedup_of_schedule": one / extra[key]["launch_ms"]}
    if args.prefill_only:
        if rank == 0:
            print(json.dumps({"prefill_only": True, "form": args.form, "heads": H, "ms_per_step": total_ms / args.steps,
                              "launch_ms": sum(launch_ms) / len(launch_ms)}), flush=True)
        return
    total_ms = max_over_ranks(total_ms, world)
    ms_per_step = total_ms / args.steps
    value = weak_scaling_value(world, T, ms_per_step)

    # roofline of the prefill kernel (one launch per step)
    launch_avg_ms = sum(launch_ms) / len(launch_ms)
    alg_bytes = T * H * PREFILL_BYTES_PER_TOKEN_HEAD + case.num_seqs * H * PREFILL_STATE_BYTES_PER_SEQ_HEAD
    alg_flops = T * H * PREFILL_FLOPS_PER_TOKEN_HEAD
    achieved_gbs = alg_bytes / (launch_avg_ms / 1e3) / 1e9
    achieved_tf = alg_flops / (launch_avg_ms / 1e3) / 1e12
    traffic = prefill_traffic() if H == PREFILL["H"] else None

    gated = None
    if gated_ms is not None:
        g_bytes = T * H * GATED_BYTES_PER_TOKEN_HEAD + case.num_seqs * H * (PREFILL_STATE_BYTES_PER_SEQ_HEAD + 4)
        g_gbs = g_bytes / (gated_ms / 1e3) / 1e9
        gated = {"workload": "prefill_k3_gated_T4096_H96", "launch_ms": gated_ms,
                 "tokens_per_s": world * T / (gated_ms / 1e3), "GB/s": g_gbs, "peak": hbm_gbs,
                 "frac": g_gbs / hbm_gbs, "alg_bytes": g_bytes,
                 "tensor_frac": alg_flops / (gated_ms / 1e3) / 1e12 / tf_burst}
    outgate = None
    if outgate_ms is not None:
        o_bytes = T * H * OUTGATE_BYTES_PER_TOKEN_HEAD + case.num_seqs * H * (PREFILL_STATE_BYTES_PER_SEQ_HEAD + 4) + 512
        o_gbs = o_bytes / (outgate_ms / 1e3) / 1e9
        outgate = {"workload": "prefill_k3_outgate_T4096_H96", "launch_ms": outgate_ms,
                   "tokens_per_s": world * T / (outgate_ms / 1e3), "GB/s": o_gbs, "peak": hbm_gbs,
                   "frac": o_gbs / hbm_gbs, "alg_bytes": o_bytes, "out_dtype": "bf16",
                   "tensor_frac": alg_flops / (outgate_ms / 1e3) / 1e12 / tf_burst}
    prologue = None
    if prologue_ms is not None:
        # raw q, k, v read + q, k, v written (bf16) per token-head, weights, states read and written
        p_bytes = T * H * PROLOGUE_BYTES_PER_TOKEN_HEAD + H * 384 * 16 + 2 * case.num_seqs * H * 3 * 384 * 2
        p_gbs = p_bytes / (prologue_ms / 1e3) / 1e9
        prologue = {"workload": "prologue_k3_T4096_H96", "launch_ms": prologue_ms, "GB/s": p_gbs, "peak": hbm_gbs,
                    "frac": p_gbs / hbm_gbs, "alg_bytes": p_bytes, "tokens_per_s": world * T / (prologue_ms / 1e3)}
    unbounded = None
    if unbounded_ms is not None:
        unbounded = {"workload": "prefill_k3_gated_T4096_H96 through g = -e^A Softplus(z)",
                     "kernel": "chunked, position pairs for channels wide in a diagonal block",
                     "launch_ms": unbounded_ms, "tokens_per_s": world * T / (unbounded_ms / 1e3),
                     "vs_bounded_chunked": (gated_ms / unbounded_ms) if gated_ms else None,
                     "steep_launch_ms": unbounded_steep_ms,
                     "steep": "logits +40 on every third channel (every chunk takes the position-pair step)",
                     "token_recurrent_launch_ms": unbounded_rec_ms}
    fdec = None
    if fdec_ms is not None:
        f_avg = sum(fdec_ms) / len(fdec_ms)
        f_bytes = DECODE["B"] * DECODE["H"] * FUSED_DECODE_BYTES_PER_SEQ_HEAD
        fdec = {"workload": "decode_B256_H96, prologue + gated decay + output gate, bf16 out",
                "ms_per_step": f_avg, "GB/s": f_bytes / (f_avg / 1e3) / 1e9, "peak": hbm_gbs,
                "frac": f_bytes / (f_avg / 1e3) / 1e9 / hbm_gbs, "alg_bytes": f_bytes, "launches": len(fdec_ms)}
    dec_avg_ms = sum(dec_ms) / len(dec_ms)
    dec_bytes = DECODE["B"] * DECODE["H"] * DECODE_BYTES_PER_SEQ_HEAD
    dec_gbs = dec_bytes / (dec_avg_ms / 1e3) / 1e9

    e2e = None
    cpu_base = None
    if rank == 0:
        case_cpu = workloads.prefill_workload(PREFILL["workload"], device="cpu", seed=0)
        modes, h2d, d2h = time_e2e(case_cpu, max(4, args.steps // 2), 2)
        # three ways of driving the host-buffer path are timed; the fastest is the line's value (on
        # some hosts the link carries both directions at once more slowly than one after another)
        best = min(modes, key=modes.get)
        e2e = {"value": T / (modes[best] / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": modes[best], "mode": best,
               "modes_ms_per_step": modes}
        if not args.no_cpu_baseline:
            heads = H  # the whole workload, as the reference arm times it: about a second on the host's cores
            dt, cores, th = cpu_oracle_sample(case_cpu, heads)
            cpu_base = {"value": T * heads / H / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                        "sample": ORACLE_SAMPLE.format(heads=heads, H=H, T=T), "seconds": dt}
            # and on one thread, for the per-core rate (2 heads: a fraction of a second)
            dt1, _, _ = cpu_oracle_sample(case_cpu, 2, threads=1)
            cpu_base["one_thread"] = {"value": T * 2 / H / dt1, "unit": "tokens/s", "cores": 1,
                                      "sample": f"2 of {H} heads x {T} tokens, one host thread", "seconds": dt1}

    if rank == 0:
        clk = clocks.summary()
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": PREFILL["workload"], "global_batch": world, "out_dtype": "f32", "seq_len": T, "heads": H,
                       "d_k": 128, "d_v": 128, "chunk": PREFILL["chunk"], "parallelism": f"replicas x{world}",
                       "l2": f"inputs {alg_bytes / 1e6:.0f} MB > 129 MB L2 per step, no flush"},
            "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm_gbs, "unit": "GB/s",
                         "frac": achieved_gbs / hbm_gbs, "traffic": traffic,
                         "peak_source": peak_src, "kernel": "prefill",
                         "tensor": {"achieved": achieved_tf, "peak": tf_burst, "unit": "TFLOP/s",
                                    "frac": achieved_tf / tf_burst},
                         "launch_ms": launch_avg_ms, "alg_bytes": alg_bytes, "alg_flops": alg_flops},
            "decode": {"workload": "decode_B256_H96", "ms_per_step": dec_avg_ms, "GB/s": dec_gbs,
                       "peak": hbm_gbs, "frac": dec_gbs / hbm_gbs,
                       "tokens_per_s": DECODE["B"] / (dec_avg_ms / 1e3), "alg_bytes": dec_bytes,
                       "launches": len(dec_ms)},
            "gated_decay": gated,
            "output_gate": outgate,
            "prologue": prologue,
            "decode_fused": fdec,
            "unbounded_decay": unbounded,
            **extra,
            "cpu_baseline": cpu_base, "e2e": e2e, "clocks": clk,
            "gpu_launches": args.steps,  # one prefill launch per timed step (decode: its own region)
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
