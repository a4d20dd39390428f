#!/usr/bin/env python3
"""Benchmark of the KDA hot path on GB300.

Default workload (one "step"): kda_prefill over B=1, H=96, T=8192, bf16
q/k/v, fp32 log_alpha/beta, S0 = 0, bf16 output and fp32 S_final, with the
inputs resident in HBM.  The same JSON line also carries the decode step
(256 requests x 96 heads, 1.6 GB of fp32 state updated in place), measured the
same way.

Prints ONE JSON line (rank 0).  Multi-GPU (torchrun): every rank runs its own
replica of the workload (weak scaling, no collective on the data path).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "KDA prefill tokens/s (% bf16 TC peak); decode tokens/s (% HBM GB/s)"
UNIT = "tokens/s"
D = 128
# Algorithmic cost per (token, head), d = 128 (bf16 q/k/v/o, fp32 log_alpha, beta); the FLOP
# count is the chunked form's at chunk 64 (the figure the roofline targets are quoted at):
PREFILL_BYTES_PER_TOKEN_HEAD = 3 * D * 2 + D * 4 + 4 + D * 2          # 1540 B
PREFILL_FLOP_PER_TOKEN_HEAD = 2 * (3 * D * D + 2.5 * 64 * D)          # 139,264 FLOP
STATE_BYTES = D * D * 4                                               # 64 KiB per (seq, head)
# Decode, per (request, head): state read + write, q/k/v bf16, log_alpha fp32, beta, o bf16
DECODE_BYTES_PER_UNIT = 2 * STATE_BYTES + 3 * D * 2 + D * 4 + 4 + D * 2  # 132,612 B
DECODE_FLOP_PER_UNIT = 2 * 4 * D * D
# Decode step of the layer core, per (request, head): state read + write, the short-convolution
# state (3 streams x 3 taps x 128 bf16) read + write, q^p, k^p, v^p, z, g bf16, beta_logit, o^g
# bf16; plus, once per step and head, the convolution weights and the decay parameters.
DECODE_LAYER_BYTES_PER_UNIT = 2 * STATE_BYTES + 2 * 9 * D * 2 + 5 * D * 2 + 2 + D * 2  # 137,218 B
DECODE_LAYER_BYTES_PER_HEAD = 3 * D * 4 * 4 + 4 + D * 4
# Several tokens per request from a pooled state, per (request, head) and token: q, k, v bf16,
# log_alpha fp32, beta, o bf16; per (request, head): the state read, and written back when the
# accepted tokens are replayed.
DECODE_TOKENS_BYTES_PER_TOKEN = 3 * D * 2 + D * 4 + 4 + D * 2           # 1,540 B
# Fused layer core, per (token, head): q^p, k^p, v^p, z, g bf16 in, o^g bf16 out, beta_logit.
LAYER_BYTES_PER_TOKEN_HEAD = 5 * D * 2 + 2 + D * 2                      # 1,538 B
E2E_SEGMENTS = 8  # end-to-end leg: token ranges per step (copies overlap the kernels)


# DRAM traffic per unit (token-head for the prefill, request-head for decode) from the
# committed ncu captures (profiles/prefill_tc_kernel_T2048_H96.md,
# profiles/decode_traffic_B64_B128_H96.md), taken on a smaller case and scaled by units.
# Valid only for the kernel source the capture was taken on: a changed kernel reports traffic
# null until it is captured again (a digest is carried over only across edits whose compiled
# kernel is byte-identical: comments, host code).
TRAFFIC = {
    "prefill": ("gated_delta_rule_kda_gb300/csrc/kda_prefill_tc.cu",
                "96aa5677145d985ef43f0bd70fb60eebd6361d95ec47882349e5b26bf6da0c78",
                (252.561408e6 + 37.64352e6) / (2048 * 96)),
    # decode kernels: the difference of captures at 128 and 64 requests (both above L2), so
    # that the written lines still in L2 at the end of a launch cancel
    # (profiles/decode_traffic_B64_B128_H96.md)
    "decode": ("gated_delta_rule_kda_gb300/csrc/kda_decode.cu",
               "4f47ecc70fd8e33c0ec569aac50f1129b3d6081242acc9ab4771f3a7c4dbd441",
               ((821180416 - 410643456) + (747280896 - 343196928)) / (64 * 96)),
    "decode_layer": ("gated_delta_rule_kda_gb300/csrc/kda_decode_layer.cu",
                     "ddc9ce806309fbe1eccc963b5e42462607fb2f0ef96d742145ab25207c53c72c",
                     ((857602560 - 431563008) + (775423232 - 357278464)) / (64 * 96)),
    # a few tokens per request (4, the bench leg's draft), same difference method
    # (profiles/decode_tokens_traffic_B64_B128_H96.md)
    "decode_tokens_verify": ("gated_delta_rule_kda_gb300/csrc/kda_decode_tokens.cu",
                             "3232adf7ab34665c383f704299e401b80f84f6d70b26b44cb953a7491b6aa8f0",
                             ((868494080 - 434240256) + (14455040 - 7170560)) / (64 * 96)),
    "decode_tokens_replay": ("gated_delta_rule_kda_gb300/csrc/kda_decode_tokens.cu",
                             "3232adf7ab34665c383f704299e401b80f84f6d70b26b44cb953a7491b6aa8f0",
                             ((868481024 - 434250752) + (755483136 - 346855936)) / (64 * 96)),
    "decode_layer_tokens_verify": ("gated_delta_rule_kda_gb300/csrc/kda_decode_layer_tokens.cu",
                                   "a264d1f312ef272f361cf3e1ae5a121e93ce66e1d325810b841455ed33228cc7",
                                   ((897339648 - 449056000) + (12546304 - 6044928)) / (64 * 96)),
    "decode_layer_tokens_replay": ("gated_delta_rule_kda_gb300/csrc/kda_decode_layer_tokens.cu",
                                   "a264d1f312ef272f361cf3e1ae5a121e93ce66e1d325810b841455ed33228cc7",
                                   ((902062080 - 450789632) + (784907008 - 361729792)) / (64 * 96)),
    # the per-head decay instantiation (one log alpha per (token, head)) and the contents
    # check: differences of captures at two sizes above L2
    # (profiles/head_decay_prefill_and_check_traffic_H96.md)
    "prefill_head_decay": ("gated_delta_rule_kda_gb300/csrc/kda_prefill_tc.cu",
                           "96aa5677145d985ef43f0bd70fb60eebd6361d95ec47882349e5b26bf6da0c78",
                           ((305234688 - 152663808) + (81304576 - 31443200)) / (2048 * 96)),
    "check": ("gated_delta_rule_kda_gb300/csrc/kda_checks.cu",
              "7b0b2e284c9fb61fdb605e513724e58d4e1da61af677c2a0e2a024e48482c146",
              ((805327360 - 402670336) + (2753024 - 2741504)) / (8192 * 96)),
    # the layer mode of the tensor-core kernel (profiles/layer_core_kernel_T2048_H96.md)
    "layer": ("gated_delta_rule_kda_gb300/csrc/kda_prefill_tc.cu",
              "96aa5677145d985ef43f0bd70fb60eebd6361d95ec47882349e5b26bf6da0c78",
              (252.79872e6 + 37.424384e6) / (2048 * 96)),
}
# GB300's nominal HBM3e bandwidth (NVIDIA's product figure), reported beside the measured copy
# bandwidth: a kernel that streams a little faster than torch's copy_ reads above 1.0 of the
# measured figure but stays below the nominal one.
HBM_NOMINAL_GBS = 7900.0


def traffic_bytes(kind, units):
    import hashlib
    path, digest, per_unit = TRAFFIC[kind]
    try:
        with open(os.path.join(ROOT, path), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != digest:
                return None
    except OSError:
        return None
    return per_unit * units


def hbm_roofline(bytes_, launch_ms, hbm, peak_kind, kernel, traffic=None):
    """Roofline object of an HBM-bound kernel: algorithmic bytes per launch over the mean
    CUDA-event launch time, against the measured copy bandwidth (frac) and the nominal one."""
    ach = bytes_ / (launch_ms / 1e3) / 1e9
    r = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
         "traffic": traffic, "peak_kind": peak_kind, "kernel": kernel,
         "nominal_peak": HBM_NOMINAL_GBS, "frac_of_nominal": ach / HBM_NOMINAL_GBS}
    if ach > hbm:
        r["note"] = ("above 1.0 of the measured peak: that peak is torch's copy_, which this "
                     "kernel outstreams; frac_of_nominal is against the datasheet figure")
    return r


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), \
            "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        self.start_wait_s = None
        self.gpu = gpu_index
        if shutil.which("nvidia-smi") is None:
            return
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        self.f = open(self.path, "w")
        self.proc = subprocess.Popen(
            ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
             "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
            stderr=subprocess.DEVNULL)
        # nvidia-smi takes a while to start: wait (up to 5 s) for its first sample, so that
        # the samples cover the timed region that follows
        t0 = time.time()
        while time.time() < t0 + 5.0 and os.path.getsize(self.path) == 0:
            if self.proc.poll() is not None:
                break
            time.sleep(0.02)
        self.start_wait_s = round(time.time() - t0, 3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for nm, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        med = statistics.median(sm) if sm else None
        return {"sm_mhz": med, "sm_max_mhz": smax, "samples": len(sm), "reasons": sorted(reasons),
                "sampler_start_s": self.start_wait_s}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The slowest rank's time (every rank gets it).  The tensor lives where the
    process group's backend expects it: on the GPU for NCCL, on the host for gloo."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(units_per_rank_step: float, ms_per_step_max: float, world: int) -> float:
    """Whole-job throughput of `world` replicas (weak scaling): every rank processes
    the same units per step; the job's step time is the slowest rank's."""
    return world * units_per_rank_step / (ms_per_step_max / 1e3)


def time_launches(fn, steps, warmup, world):
    """Per-launch CUDA-event times on the launching (current) stream."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s, e in ev:
        s.record(stream)
        fn()
        e.record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    total_ms = t0.elapsed_time(t1)
    per = [s.elapsed_time(e) for s, e in ev]
    return total_ms, per


def cpu_baseline_prefill(inp, heads, tokens, n_threads=None):
    """The fp64 oracle as it stands, on a bounded sample of the prefill workload."""
    import numpy as np
    import oracle
    f = lambda t: t[:tokens, heads].double().cpu().numpy()
    args = [f(inp.q), f(inp.k), f(inp.v), f(inp.log_alpha), f(inp.beta)]
    cores = n_threads or oracle.default_threads()
    t = time.perf_counter()
    oracle.kda_prefill(*args, np.array([0, tokens], np.int32), n_threads=cores)
    dt = time.perf_counter() - t
    head_tokens = tokens * len(heads)
    return dt, head_tokens, min(cores, len(heads))


def run_reference(args, world, rank):
    """Reference arm: the fp64 CPU oracle, timed on the host cores."""
    if rank != 0:
        return
    from gated_delta_rule_kda_gb300 import synthetic
    import oracle
    oracle.build()
    H_sample, T_sample = 16, 1024
    inp = synthetic.prefill_inputs([T_sample], H_sample, torch.bfloat16,
                                   seed=synthetic.BASE_SEED + 2, device="cpu")
    times = []
    for i in range(args.warmup + args.steps):
        dt, head_tokens, cores = cpu_baseline_prefill(inp, list(range(H_sample)), T_sample)
        if i >= args.warmup:
            times.append(dt)
    mean = sum(times) / len(times)
    value = head_tokens / mean / 96.0
    sample = (f"oracle on {H_sample} heads x {T_sample} tokens per step, "
              f"scaled to 96-head tokens")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": mean * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.gpus),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(n):
    return {"workload": "KDA prefill B=1 H=96 T=8192 d=128 bf16 (kernel chunk 32; the result "
                        "does not depend on the chunk size), S0=0, "
                        "bf16 o + fp32 S_final", "global_batch": n, "seq_len": 8192,
            "heads": 96, "head_dim": 128, "parallelism": f"replicas x{n}",
            "l2": "inputs larger than L2 (1.2 GB per step), no flush",
            "decode_workload": "256 requests x 96 heads, fp32 state 1.61 GB in place"}


def run_ours(args, world, rank, local):
    from gated_delta_rule_kda_gb300 import kda, synthetic
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    hbm, tc, tc_sus, peak_kind = peaks()

    # ---------------- prefill (the step) ----------------
    inp = synthetic.workload(2, device=dev)
    T, H = inp.q.shape[:2]
    o = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
    Sf = torch.empty((1, H, D, D), dtype=torch.float32, device=dev)

    def prefill_step():
        kda.kda_prefill(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.cu_seqlens, None,
                        o=o, S_final=Sf)

    clocks = ClockSampler(local if world > 1 else torch.cuda.current_device())
    total_ms, per = time_launches(prefill_step, args.steps, args.warmup, world)
    clk = clocks.stop()
    ms_step = max_over_ranks(total_ms / args.steps, world)
    tokens_per_step = T
    value = aggregate_rate(tokens_per_step, ms_step, world)
    launch_ms = sum(per) / len(per)
    alg_bytes = T * H * PREFILL_BYTES_PER_TOKEN_HEAD + H * STATE_BYTES
    alg_flop = T * H * PREFILL_FLOP_PER_TOKEN_HEAD
    achieved = alg_bytes / (launch_ms / 1e3) / 1e9
    tflops = alg_flop / (launch_ms / 1e3) / 1e12
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": traffic_bytes("prefill", T * H),
                "peak_kind": peak_kind,
                "kernel": "kda_prefill", "tc_achieved_tflops": tflops, "tc_peak_tflops": tc,
                "tc_frac": tflops / tc,
                "binding_roofline_frac": max(alg_bytes / (hbm * 1e9),
                                             alg_flop / (tc * 1e12)) / (launch_ms / 1e3)}

    # ---------------- the same prefill leaving a state snapshot every 1024 tokens ----------------
    ck_every = 1024
    ck_base = kda.checkpoint_offsets(inp.cu_seqlens, ck_every).to(dev)
    ck_states = torch.empty((int(ck_base[-1]), H, D, D), dtype=torch.float32, device=dev)

    def checkpoint_step():
        kda.kda_prefill_with_checkpoints(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta,
                                         inp.cu_seqlens, ck_every, None, ckpt_base=ck_base,
                                         ckpt_states=ck_states, o=o, S_final=Sf)

    ck_total, _ = time_launches(checkpoint_step, args.steps, args.warmup, world)
    ck_ms = max_over_ranks(ck_total / args.steps, world)
    checkpoints = {"entry_point": "kda_prefill_with_checkpoints", "every_tokens": ck_every,
                   "snapshots": int(ck_base[-1]) * H,
                   "snapshot_bytes": ck_states.numel() * 4, "ms_per_step": ck_ms,
                   "tokens_per_s": aggregate_rate(tokens_per_step, ck_ms, world),
                   "overhead_vs_prefill": ck_ms / ms_step - 1.0}
    del ck_states

    # ---------------- contents checks of the prefill inputs (one pass over log alpha) ----------------
    def check_step():
        kda.kda_check_prefill_inputs(inp.cu_seqlens, inp.log_alpha)

    ch_total, ch_per = time_launches(check_step, args.steps, args.warmup, world)
    ch_launch = sum(ch_per) / len(ch_per)
    check_bytes = inp.log_alpha.numel() * 4 + inp.cu_seqlens.numel() * 4
    if kda.kda_get_device_status()[0] != 0:
        raise RuntimeError("the contents checks flagged the bench's own inputs")
    contents_check = {"entry_point": "kda_check_prefill_inputs",
                      "ms_per_step": max_over_ranks(ch_total / args.steps, world),
                      "roofline": {"bound": "hbm",
                                   "achieved": check_bytes / (ch_launch / 1e3) / 1e9,
                                   "peak": hbm, "unit": "GB/s",
                                   "frac": check_bytes / (ch_launch / 1e3) / 1e9 / hbm,
                                   "traffic": traffic_bytes("check", T * H),
                                   "peak_kind": peak_kind,
                                   "kernel": "kda_check_prefill_inputs"}}

    # ---------------- the Gated DeltaNet case: one decay per (token, head) ----------------
    la_head = inp.log_alpha[:, :, 0].contiguous()  # [T, H]: one channel's draws as the head's decay

    def head_decay_step():
        kda.kda_prefill_head_decay(inp.q, inp.k, inp.v, la_head, inp.beta, inp.cu_seqlens, None,
                                   o=o, S_final=Sf)

    hd_total, hd_per = time_launches(head_decay_step, args.steps, args.warmup, world)
    hd_ms = max_over_ranks(hd_total / args.steps, world)
    hd_launch = sum(hd_per) / len(hd_per)
    hd_bytes = T * H * (PREFILL_BYTES_PER_TOKEN_HEAD - D * 4 + 4) + H * STATE_BYTES
    head_decay = {"entry_point": "kda_prefill_head_decay", "ms_per_step": hd_ms,
                  "tokens_per_s": aggregate_rate(tokens_per_step, hd_ms, world),
                  "roofline": {"bound": "hbm", "achieved": hd_bytes / (hd_launch / 1e3) / 1e9,
                               "peak": hbm, "unit": "GB/s",
                               "frac": hd_bytes / (hd_launch / 1e3) / 1e9 / hbm,
                               "traffic": traffic_bytes("prefill_head_decay", T * H),
                               "peak_kind": peak_kind,
                               "kernel": "kda_prefill_head_decay"}}
    del la_head

    # ---------------- no decay floor (Kimi Linear): kda_prefill_unbounded_decay ----------------
    def unbounded_step():
        kda.kda_prefill_unbounded_decay(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta,
                                        inp.cu_seqlens, None, o=o, S_final=Sf)

    ub_total, _ = time_launches(unbounded_step, args.steps, args.warmup, world)
    ub_ms = max_over_ranks(ub_total / args.steps, world)
    la_strong = -40.0 * torch.rand(inp.log_alpha.shape, generator=torch.Generator(device=dev)
                                   .manual_seed(7), device=dev)

    def strong_step():
        kda.kda_prefill_unbounded_decay(inp.q, inp.k, inp.v, la_strong, inp.beta,
                                        inp.cu_seqlens, None, o=o, S_final=Sf)

    st_steps = max(1, min(args.steps, 3))
    st_total, _ = time_launches(strong_step, st_steps, args.warmup, world)
    st_ms = max_over_ranks(st_total / st_steps, world)
    del la_strong
    prefill_unbounded = {"entry_point": "kda_prefill_unbounded_decay",
                         "in_range": {"decays": "the bench step's (every chunk takes the "
                                                "tensor-core form)", "ms_per_step": ub_ms,
                                      "tokens_per_s": aggregate_rate(tokens_per_step, ub_ms, world)},
                         "strong_decay": {"decays": "log alpha uniform in [-40, 0] (every chunk "
                                                    "runs token by token in the kernel)",
                                          "ms_per_step": st_ms,
                                          "tokens_per_s": aggregate_rate(tokens_per_step, st_ms,
                                                                         world)}}

    # ---------------- the long prefill: 1 x 131,072 tokens x 96 heads, carried S0 ----------------
    long_prefill = None
    if not args.skip_long_prefill:
        linp4 = synthetic.workload(4, device=dev)
        T4 = linp4.q.shape[0]
        o4 = torch.empty((T4, H, D), dtype=torch.bfloat16, device=dev)
        S4 = torch.empty((1, H, D, D), dtype=torch.float32, device=dev)

        def long_step():
            kda.kda_prefill(linp4.q, linp4.k, linp4.v, linp4.log_alpha, linp4.beta,
                            linp4.cu_seqlens, linp4.S0, o=o4, S_final=S4)

        l4_steps = max(1, min(args.steps, 5))
        l4_total, l4_per = time_launches(long_step, l4_steps, args.warmup, world)
        l4_ms = max_over_ranks(l4_total / l4_steps, world)
        l4_launch = sum(l4_per) / len(l4_per)
        l4_bytes = T4 * H * PREFILL_BYTES_PER_TOKEN_HEAD + 2 * H * STATE_BYTES
        long_prefill = {"workload": "B=1 H=96 T=131072 bf16, S0 ~ N(0, 0.1), log alpha from "
                                    "x ~ N(1, 1)", "entry_point": "kda_prefill",
                        "ms_per_step": l4_ms, "tokens_per_s": aggregate_rate(T4, l4_ms, world),
                        "roofline": {"bound": "hbm",
                                     "achieved": l4_bytes / (l4_launch / 1e3) / 1e9,
                                     "peak": hbm, "unit": "GB/s",
                                     "frac": l4_bytes / (l4_launch / 1e3) / 1e9 / hbm,
                                     "traffic": traffic_bytes("prefill", T4 * H),
                                     "peak_kind": peak_kind, "kernel": "kda_prefill"}}
        del linp4, o4, S4
        torch.cuda.empty_cache()

    # ---------------- end to end through the C ABI with host buffers ----------------
    host = {n: getattr(inp, n).cpu().pin_memory() for n in ("q", "k", "v", "log_alpha", "beta")}
    dev_bufs = {n: getattr(inp, n) for n in host}
    o_host = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    S_host = torch.empty(Sf.shape, dtype=Sf.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = o_host.numel() * o_host.element_size() + S_host.numel() * S_host.element_size()

    # The step is split into E2E_SEGMENTS consecutive token ranges that resume from
    # S_final (chunk boundaries stay aligned, so the result is the single call's): the
    # inputs of segment i+1 travel host -> device on a copy stream while segment i
    # runs, and each finished segment's output goes back on two device -> host
    # streams (one stream has measured as low as ~70 GB/s device -> host).
    seg = T // E2E_SEGMENTS
    cu_seg = torch.tensor([0, seg], dtype=torch.int32, device=dev)
    h2d_stream = torch.cuda.Stream(device=dev)
    d2h_streams = [torch.cuda.Stream(device=dev) for _ in range(2)]

    def e2e_step():
        main = torch.cuda.current_stream()
        start = torch.cuda.Event()
        start.record(main)
        h2d_stream.wait_event(start)
        for st in d2h_streams:
            st.wait_event(start)
        landed = []
        with torch.cuda.stream(h2d_stream):
            for i in range(E2E_SEGMENTS):
                for n, t in host.items():
                    dev_bufs[n][i * seg:(i + 1) * seg].copy_(t[i * seg:(i + 1) * seg],
                                                             non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(h2d_stream)
                landed.append(ev)
        for i in range(E2E_SEGMENTS):
            main.wait_event(landed[i])
            sl = slice(i * seg, (i + 1) * seg)
            kda.kda_prefill(inp.q[sl], inp.k[sl], inp.v[sl], inp.log_alpha[sl], inp.beta[sl],
                            cu_seg, None if i == 0 else Sf, o=o[sl], S_final=Sf)
            done = torch.cuda.Event()
            done.record(main)
            st = d2h_streams[i % 2]
            st.wait_event(done)
            with torch.cuda.stream(st):
                o_host[sl].copy_(o[sl], non_blocking=True)
                if i == E2E_SEGMENTS - 1:
                    S_host.copy_(Sf, non_blocking=True)
        for st in d2h_streams:
            main.wait_stream(st)

    # the segmented step must reproduce the single call (checked once, outside the timing)
    prefill_step()
    ref_o, ref_S = o.cpu(), Sf.cpu()
    e2e_step()
    torch.cuda.synchronize()
    e2e_exact = bool(torch.equal(o_host, ref_o) and torch.equal(S_host, ref_S))
    del ref_o, ref_S
    e2e_steps = max(2, min(args.steps, 5))
    e2e_total, _ = time_launches(e2e_step, e2e_steps, 1, world)
    e2e_ms = max_over_ranks(e2e_total / e2e_steps, world)
    e2e = {"value": aggregate_rate(tokens_per_step, e2e_ms, world), "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
           "pipeline": f"{E2E_SEGMENTS} resumed segments; copies overlap the kernels",
           "matches_single_call": e2e_exact}
    del host, o_host, S_host

    # ---------------- decode (second half of the metric) ----------------
    del inp, o, Sf
    torch.cuda.empty_cache()
    dinp = synthetic.workload(3, device=dev)
    od = torch.empty((256, 96, D), dtype=torch.bfloat16, device=dev)

    def decode_step():
        kda.kda_decode_step(dinp.q, dinp.k, dinp.v, dinp.log_alpha, dinp.beta, dinp.S, o=od)

    d_total, d_per = time_launches(decode_step, args.steps, args.warmup, world)
    d_ms = max_over_ranks(d_total / args.steps, world)
    d_launch = sum(d_per) / len(d_per)
    units = 256 * 96
    d_bytes = units * DECODE_BYTES_PER_UNIT
    decode = {"tokens_per_s": aggregate_rate(256, d_ms, world), "ms_per_step": d_ms,
              "roofline": hbm_roofline(d_bytes, d_launch, hbm, peak_kind, "kda_decode_step",
                                       traffic_bytes("decode", units))}
    del dinp, od
    torch.cuda.empty_cache()

    # ---------------- decode step of the whole layer core over state pools ----------------
    linp1 = synthetic.decode_layer_inputs(256, 96, 256, device=dev)
    odl = torch.empty((256, 96, D), dtype=torch.bfloat16, device=dev)

    def decode_layer_step():
        kda.kda_decode_layer(linp1.qp, linp1.kp, linp1.vp, linp1.conv_w, linp1.z, linp1.A,
                             linp1.b, linp1.beta_logit, linp1.g, linp1.slot, linp1.S_pool,
                             linp1.conv_pool, o=odl)

    dl_total, dl_per = time_launches(decode_layer_step, args.steps, args.warmup, world)
    dl_ms = max_over_ranks(dl_total / args.steps, world)
    dl_launch = sum(dl_per) / len(dl_per)
    dl_bytes = 256 * 96 * DECODE_LAYER_BYTES_PER_UNIT + 96 * DECODE_LAYER_BYTES_PER_HEAD
    decode_layer = {"tokens_per_s": aggregate_rate(256, dl_ms, world), "ms_per_step": dl_ms,
                    "entry_point": "kda_decode_layer",
                    "workload": "256 requests x 96 heads in shuffled rows of 256-row state and "
                                "convolution pools; front end + recurrence + gate",
                    "roofline": hbm_roofline(dl_bytes, dl_launch, hbm, peak_kind,
                                             "kda_decode_layer",
                                             traffic_bytes("decode_layer", 256 * 96))}
    del linp1, odl
    torch.cuda.empty_cache()

    # ---------------- a 4-token draft per request: verify, then replay ----------------
    ntok = 4
    tinp = synthetic.decode_tokens_inputs([ntok] * 256, 96, 256, device=dev)
    ot = torch.empty((256 * ntok, 96, D), dtype=torch.bfloat16, device=dev)
    spec = {"workload": f"256 requests x {ntok} tokens x 96 heads from shuffled rows of a "
                        "256-row state pool", "entry_point": "kda_decode_tokens"}
    for mode, wb in (("verify", False), ("replay", True)):
        def tokens_step():
            kda.kda_decode_tokens(tinp.q, tinp.k, tinp.v, tinp.log_alpha, tinp.beta,
                                  tinp.cu_tokens, tinp.slot, tinp.S_pool, wb, o=ot)

        t_total, t_per = time_launches(tokens_step, args.steps, args.warmup, world)
        t_ms = max_over_ranks(t_total / args.steps, world)
        t_launch = sum(t_per) / len(t_per)
        t_bytes = 256 * 96 * ((2 if wb else 1) * STATE_BYTES + ntok * DECODE_TOKENS_BYTES_PER_TOKEN)
        spec[mode] = {"tokens_per_s": aggregate_rate(256 * ntok, t_ms, world), "ms_per_step": t_ms,
                      "write_back": wb,
                      "roofline": hbm_roofline(t_bytes, t_launch, hbm, peak_kind,
                                               "kda_decode_tokens",
                                               traffic_bytes("decode_tokens_" + mode, 256 * 96))}
    del tinp, ot
    torch.cuda.empty_cache()

    # the same draft through the whole layer core (convolution state included)
    linp2 = synthetic.decode_layer_tokens_inputs([ntok] * 256, 96, 256, device=dev)
    og2 = torch.empty((256 * ntok, 96, D), dtype=torch.bfloat16, device=dev)
    spec_layer = {"workload": f"256 requests x {ntok} tokens x 96 heads from shuffled rows of "
                              "256-row state and convolution pools; front end + recurrence + gate",
                  "entry_point": "kda_decode_layer_tokens"}
    for mode, wb in (("verify", False), ("replay", True)):
        def layer_tokens_step():
            kda.kda_decode_layer_tokens(linp2.qp, linp2.kp, linp2.vp, linp2.conv_w, linp2.z,
                                        linp2.A, linp2.b, linp2.beta_logit, linp2.g,
                                        linp2.cu_tokens, linp2.slot, linp2.S_pool,
                                        linp2.conv_pool, wb, o=og2)

        t_total, t_per = time_launches(layer_tokens_step, args.steps, args.warmup, world)
        t_ms = max_over_ranks(t_total / args.steps, world)
        t_launch = sum(t_per) / len(t_per)
        per_unit = (2 if wb else 1) * (STATE_BYTES + 9 * D * 2) + ntok * LAYER_BYTES_PER_TOKEN_HEAD
        t_bytes = 256 * 96 * per_unit + 96 * DECODE_LAYER_BYTES_PER_HEAD
        spec_layer[mode] = {"tokens_per_s": aggregate_rate(256 * ntok, t_ms, world),
                            "ms_per_step": t_ms, "write_back": wb,
                            "roofline": hbm_roofline(t_bytes, t_launch, hbm, peak_kind,
                                                     "kda_decode_layer_tokens",
                                                     traffic_bytes("decode_layer_tokens_" + mode,
                                                                   256 * 96))}
    spec["layer"] = spec_layer
    del linp2, og2
    torch.cuda.empty_cache()

    # ---------------- layer core (varlen, 16 sequences) ----------------
    layer = None
    if not args.skip_layer_core:
        linp = synthetic.workload(5, device=dev)
        LT = linp.qp.shape[0]
        og = torch.empty((LT, 96, D), dtype=torch.bfloat16, device=dev)
        Sl = torch.empty((16, 96, D, D), dtype=torch.float32, device=dev)

        def fused_step():
            kda.kda_layer_core_fused(linp.qp, linp.kp, linp.vp, linp.conv_w, linp.z, linp.A,
                                     linp.b, linp.beta_logit, linp.g, linp.cu_seqlens, None,
                                     o=og, S_final=Sl)

        l_steps = max(1, min(args.steps, 10))
        l_total, l_per = time_launches(fused_step, l_steps, args.warmup, world)
        l_ms = max_over_ranks(l_total / l_steps, world)
        l_launch = sum(l_per) / len(l_per)
        # q^p, k^p, v^p, z, g, beta_logit in, o^g out per (token, head); S_final per (sequence,
        # head); the convolution weights and gate parameters once per head
        l_bytes = (LT * 96 * LAYER_BYTES_PER_TOKEN_HEAD + 16 * 96 * STATE_BYTES
                   + 96 * DECODE_LAYER_BYTES_PER_HEAD)
        layer = {"tokens_per_s": aggregate_rate(LT, l_ms, world), "ms_per_step": l_ms,
                 "tokens": LT, "workload": "16 sequences, lengths log-uniform in [1K, 64K], "
                                           "96 heads, front end + recurrence + gate",
                 "entry_point": "kda_layer_core_fused", "launches_per_step": 1,
                 "hbm_bytes_per_token_head": LAYER_BYTES_PER_TOKEN_HEAD,
                 "roofline": hbm_roofline(l_bytes, l_launch, hbm, peak_kind,
                                          "kda_layer_core_fused", traffic_bytes("layer", LT * 96))}
        if not args.skip_staged_layer_core:
            ws = torch.empty(kda.kda_layer_core_workspace_size(16, LT, 96), dtype=torch.uint8,
                             device=dev)

            def staged_step():
                kda.kda_layer_core(linp.qp, linp.kp, linp.vp, linp.conv_w, linp.z, linp.A,
                                   linp.b, linp.beta_logit, linp.g, linp.cu_seqlens, None, o=og,
                                   S_final=Sl, workspace=ws)

            s_total, _ = time_launches(staged_step, 2, 1, world)
            s_ms = max_over_ranks(s_total / 2, world)
            layer["staged"] = {"entry_point": "kda_layer_core", "ms_per_step": s_ms,
                               "tokens_per_s": aggregate_rate(LT, s_ms, world),
                               "launches_per_step": 3}

            def unbounded_step():  # Kimi Linear's gate: no decay floor, token-by-token kernel
                kda.kda_layer_core_unbounded_decay(linp.qp, linp.kp, linp.vp, linp.conv_w, linp.z,
                                                   linp.A, linp.b, linp.beta_logit, linp.g,
                                                   linp.cu_seqlens, None, o=og, S_final=Sl,
                                                   workspace=ws)

            u_total, _ = time_launches(unbounded_step, 2, 1, world)
            u_ms = max_over_ranks(u_total / 2, world)
            layer["unbounded_decay"] = {"entry_point": "kda_layer_core_unbounded_decay",
                                        "ms_per_step": u_ms,
                                        "tokens_per_s": aggregate_rate(LT, u_ms, world),
                                        "launches_per_step": 3}
            del ws

        def unbounded_fused_step():  # the same gate in the tensor-core kernel (chunk fallback)
            kda.kda_layer_core_fused_unbounded_decay(linp.qp, linp.kp, linp.vp, linp.conv_w,
                                                     linp.z, linp.A, linp.b, linp.beta_logit,
                                                     linp.g, linp.cu_seqlens, None, o=og,
                                                     S_final=Sl)

        uf_total, _ = time_launches(unbounded_fused_step, l_steps, args.warmup, world)
        uf_ms = max_over_ranks(uf_total / l_steps, world)
        layer["unbounded_decay_fused"] = {"entry_point": "kda_layer_core_fused_unbounded_decay",
                                          "ms_per_step": uf_ms,
                                          "tokens_per_s": aggregate_rate(LT, uf_ms, world),
                                          "vs_bounded_fused": uf_ms / l_ms,
                                          "launches_per_step": 1}
        del linp, og, Sl
        torch.cuda.empty_cache()

    # ---------------- CPU baseline: the oracle on a bounded sample ----------------
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from gated_delta_rule_kda_gb300 import synthetic as syn
        cinp = syn.workload(2, device="cpu")
        dt, head_tokens, cores = cpu_baseline_prefill(cinp, list(range(96)), 8192)
        # one core: 12 of the 96 heads over all 8192 tokens on one thread, scaled per head
        dt1, head_tokens1, _ = cpu_baseline_prefill(cinp, list(range(12)), 8192, n_threads=1)
        cpu = {"value": head_tokens / dt / 96.0, "unit": UNIT, "cores": cores,
               "kind": "oracle",
               "sample": f"the whole prefill workload (96 heads x 8192 tokens), {dt:.1f} s wall "
                         f"on {cores} threads",
               "one_core": {"value": head_tokens1 / dt1 / 96.0, "unit": UNIT, "cores": 1,
                            "sample": f"12 heads x 8192 tokens on one thread ({dt1:.1f} s), "
                                      f"scaled to 96-head tokens"}}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic", "config": workload_config(world),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "prefill_checkpoints": checkpoints, "prefill_head_decay": head_decay,
            "prefill_unbounded_decay": prefill_unbounded,
            "long_prefill": long_prefill, "contents_check": contents_check,
            "decode": decode,
            "decode_layer": decode_layer, "speculative": spec, "layer_core": layer,
            "clocks": clk, "gpu_launches": args.steps,
            "kernel_ms_mean": launch_ms,
        }
        print(json.dumps(line), flush=True)


def run_only(args, local):
    """One kernel on its own (for ncu): W warm-up + K launches, one summary line."""
    from gated_delta_rule_kda_gb300 import kda, synthetic
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if args.only == "prefill":
        T = 2048 if args.small else 8192
        inp = synthetic.prefill_inputs([T], 96, torch.bfloat16, seed=synthetic.BASE_SEED + 2,
                                       device=dev)
        o = torch.empty((T, 96, D), dtype=torch.bfloat16, device=dev)
        Sf = torch.empty((1, 96, D, D), dtype=torch.float32, device=dev)
        fn = lambda: kda.kda_prefill(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta,
                                     inp.cu_seqlens, None, o=o, S_final=Sf)
        units = T
    elif args.only == "prefill_head_decay":
        # kda_prefill_head_decay on the prefill workload's inputs, one decay per (token, head):
        # 2048 (--small) or 8192 tokens, or --tokens, 96 heads
        T = args.tokens or (2048 if args.small else 8192)
        inp = synthetic.prefill_inputs([T], 96, torch.bfloat16, seed=synthetic.BASE_SEED + 2,
                                       device=dev)
        la_head = inp.log_alpha[:, :, 0].contiguous()
        o = torch.empty((T, 96, D), dtype=torch.bfloat16, device=dev)
        Sf = torch.empty((1, 96, D, D), dtype=torch.float32, device=dev)
        fn = lambda: kda.kda_prefill_head_decay(inp.q, inp.k, inp.v, la_head, inp.beta,
                                                inp.cu_seqlens, None, o=o, S_final=Sf)
        units = T
    elif args.only == "check":
        # kda_check_prefill_inputs over the prefill workload's log alpha (8192 tokens, or
        # --tokens, 96 heads)
        T = args.tokens or 8192
        inp = synthetic.prefill_inputs([T], 96, torch.bfloat16, seed=synthetic.BASE_SEED + 2,
                                       device=dev)
        fn = lambda: kda.kda_check_prefill_inputs(inp.cu_seqlens, inp.log_alpha)
        units = T
    elif args.only == "prefill_fp32":
        # the token-by-token kernel (fp32 inputs): 8 sequences x 1024 tokens (--small) or
        # 16 x 8192, 96 heads
        lens = [1024] * 8 if args.small else [8192] * 16
        inp = synthetic.prefill_inputs(lens, 96, torch.float32, seed=synthetic.BASE_SEED + 1,
                                       device=dev)
        T = inp.q.shape[0]
        o = torch.empty((T, 96, D), dtype=torch.float32, device=dev)
        Sf = torch.empty((len(lens), 96, D, D), dtype=torch.float32, device=dev)
        fn = lambda: kda.kda_prefill(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta,
                                     inp.cu_seqlens, None, o=o, S_final=Sf)
        units = T
    elif args.only == "layer":
        lens = [2048] if args.small else synthetic.varlen_lengths(seed=synthetic.BASE_SEED + 5)
        linp = synthetic.layer_inputs(lens, 96, seed=synthetic.BASE_SEED + 5, device=dev)
        LT = linp.qp.shape[0]
        og = torch.empty((LT, 96, D), dtype=torch.bfloat16, device=dev)
        fn = lambda: kda.kda_layer_core_fused(linp.qp, linp.kp, linp.vp, linp.conv_w, linp.z,
                                              linp.A, linp.b, linp.beta_logit, linp.g,
                                              linp.cu_seqlens, None, o=og, want_state=False)
        units = LT
    elif args.only == "staged_layer":
        # front end -> token-by-token prefill -> gate through a workspace (kda_layer_core):
        # 2 x 2048 tokens (--small) or workload 5's lengths, 96 heads
        lens = [2048, 2048] if args.small else synthetic.varlen_lengths(seed=synthetic.BASE_SEED + 5)
        linp = synthetic.layer_inputs(lens, 96, seed=synthetic.BASE_SEED + 5, device=dev)
        LT = linp.qp.shape[0]
        og = torch.empty((LT, 96, D), dtype=torch.bfloat16, device=dev)
        Sl = torch.empty((len(lens), 96, D, D), dtype=torch.float32, device=dev)
        ws = torch.empty(kda.kda_layer_core_workspace_size(len(lens), LT, 96), dtype=torch.uint8,
                         device=dev)
        fn = lambda: kda.kda_layer_core(linp.qp, linp.kp, linp.vp, linp.conv_w, linp.z, linp.A,
                                        linp.b, linp.beta_logit, linp.g, linp.cu_seqlens, None,
                                        o=og, S_final=Sl, workspace=ws)
        units = LT
    elif args.only == "decode_layer":
        B = args.batch or (32 if args.small else 256)
        linp1 = synthetic.decode_layer_inputs(B, 96, B, device=dev)
        odl = torch.empty((B, 96, D), dtype=torch.bfloat16, device=dev)
        fn = lambda: kda.kda_decode_layer(linp1.qp, linp1.kp, linp1.vp, linp1.conv_w, linp1.z,
                                          linp1.A, linp1.b, linp1.beta_logit, linp1.g, linp1.slot,
                                          linp1.S_pool, linp1.conv_pool, o=odl)
        units = B
    elif args.only == "decode_layer_tokens":
        B = args.batch or (32 if args.small else 256)
        linp2 = synthetic.decode_layer_tokens_inputs([4] * B, 96, B, device=dev)
        og2 = torch.empty((4 * B, 96, D), dtype=torch.bfloat16, device=dev)
        fn = lambda: kda.kda_decode_layer_tokens(linp2.qp, linp2.kp, linp2.vp, linp2.conv_w,
                                                 linp2.z, linp2.A, linp2.b, linp2.beta_logit,
                                                 linp2.g, linp2.cu_tokens, linp2.slot,
                                                 linp2.S_pool, linp2.conv_pool,
                                                 bool(args.write_back), o=og2)
        units = B
    elif args.only == "decode_tokens":
        B = args.batch or (32 if args.small else 256)
        tinp = synthetic.decode_tokens_inputs([4] * B, 96, B, device=dev)
        ot = torch.empty((4 * B, 96, D), dtype=torch.bfloat16, device=dev)
        fn = lambda: kda.kda_decode_tokens(tinp.q, tinp.k, tinp.v, tinp.log_alpha, tinp.beta,
                                           tinp.cu_tokens, tinp.slot, tinp.S_pool,
                                           bool(args.write_back), o=ot)
        units = B
    else:
        B = args.batch or (32 if args.small else 256)
        dinp = synthetic.decode_inputs(B, 96, torch.bfloat16, device=dev)
        od = torch.empty((B, 96, D), dtype=torch.bfloat16, device=dev)
        fn = lambda: kda.kda_decode_step(dinp.q, dinp.k, dinp.v, dinp.log_alpha, dinp.beta,
                                         dinp.S, o=od)
        units = B
    total, per = time_launches(fn, args.steps, args.warmup, 1)
    print(json.dumps({"only": args.only, "small": args.small, "units": units,
                      "ms_mean": sum(per) / len(per), "ms_min": min(per)}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--skip-layer-core", action="store_true")
    ap.add_argument("--skip-long-prefill", action="store_true",
                    help="skip the 131,072-token prefill leg (19 GB of inputs)")
    ap.add_argument("--skip-staged-layer-core", action="store_true",
                    help="time only the fused layer core, not the three-launch composition")
    ap.add_argument("--only", choices=["prefill", "prefill_head_decay", "check", "prefill_fp32",
                                       "decode", "decode_layer",
                                       "decode_tokens", "decode_layer_tokens", "layer",
                                       "staged_layer"],
                    default=None,
                    help="profiling aid: run just this kernel (no baseline, no e2e)")
    ap.add_argument("--small", action="store_true",
                    help="with --only: a smaller case sized for ncu captures")
    ap.add_argument("--batch", type=int, default=0,
                    help="with --only and a decode kind: this many requests")
    ap.add_argument("--tokens", type=int, default=0,
                    help="with --only prefill_head_decay / check: this many tokens")
    ap.add_argument("--write-back", type=int, default=1,
                    help="with --only decode_tokens / decode_layer_tokens: 0 verify, 1 replay")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, world, rank)
        return
    world, rank, local = dist_setup()
    if args.only:
        run_only(args, local)
        return
    run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
