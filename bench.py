"""Benchmark of the whole hot path on one GB300 (or N replicas).

One step = prefill quantize of the layer's K/V (all streams, full context),
append of one token per stream, and fused dequant decode attention of one
query token per (batch, query head) over the whole cache -- every step of the
codec and of the attention, through the C ABI. Inputs are seeded synthetic
fp16 tensors already resident in HBM; they are larger than L2 (129 MB), so no
L2 flush is needed between timed steps.

Prints one JSON line (rank 0). ``value`` is the whole-step algorithmic
throughput in GB/s (bytes read + written by prefill, append and decode per
step, divided by the step time); the line also carries the decode-attention
and quantize throughputs, the roofline of the dominant kernel, clocks, the
end-to-end number through host buffers and the CPU oracle baseline.

``--impl reference`` times the CPU oracle instead (the reference arm).
Under torchrun (N > 1) each rank runs an independent replica (the path has
no exchange step); value = bytes of all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from bit_quantized_kv_kvq_gb300 import accounting as A  # noqa: E402
from bit_quantized_kv_kvq_gb300 import workloads as W  # noqa: E402

METRIC = "fused dequant decode-attention KV GB/s (% of GB300 HBM peak); quantize GB/s"
DEFAULT_WORKLOAD = W.LLAMA7B_16K.name
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# distributed helpers (host logic; tested with gloo on CPU)
# ---------------------------------------------------------------------------

def dist_env():
    """(rank, world, local_rank) from the torchrun environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def reduce_max(value, device=None):
    """Max of a float over ranks (identity without a process group)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value, device=None):
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def replica_seed(wl, rank):
    """Each replica draws its own inputs (weak scaling, independent problems)."""
    return wl.seed + 7919 * rank


# ---------------------------------------------------------------------------
# peaks and clocks
# ---------------------------------------------------------------------------

def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
        except Exception:
            pass
        finally:
            try:
                os.unlink(self.path)
            except Exception:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")
        sm = [num(r[1]) for r in rows]
        pw = [num(r[3]) for r in rows]
        load = [s for s, p in zip(sm, pw) if p == p and p > 0.4 * max(pw)] or sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = []
        for i, nm in enumerate(names):
            if any(r[5 + i].lower().startswith("active") for r in rows):
                reasons.append(nm)
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": max(num(r[2]) for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_gpu(args, wl, rank, world, device):
    import bit_quantized_kv_kvq_gb300 as kvq
    from bit_quantized_kv_kvq_gb300.synth import LayerSource

    torch.cuda.set_device(device)
    S = wl.seq_len
    cache = kvq.QuantizedKVCache(1, wl.batch, wl.num_kv_heads, wl.head_dim, S + 1, wl.k_bits,
                                 wl.v_bits, wl.k_mode, wl.v_mode, wl.k_group, wl.v_group,
                                 wl.outliers_per_row, device=device)
    src = LayerSource(wl, 0, device=device, seed=replica_seed(wl, rank))
    k, v = src.kv(S)
    q, k1, v1 = src.step(0)
    out = torch.empty((wl.batch, wl.num_q_heads, wl.head_dim), dtype=torch.float32, device=device)
    ws = cache.workspace(wl.num_q_heads)
    scale = 1.0 / math.sqrt(wl.head_dim)
    stream = torch.cuda.current_stream(device)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        cache.prefill(0, k, v)
        if ev:
            ev[1].record(stream)
        cache.append(0, k1, v1)
        if ev:
            ev[2].record(stream)
        cache.decode(0, q, scale, out=out, workspace=ws)
        if ev:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)
    assert cache.status() == 0

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    launches0 = kvq.kernel_launches()
    with ClockSampler(device.index) as clk:
        barrier(device)
        torch.cuda.synchronize(device)
        t0.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t1.record(stream)
        torch.cuda.synchronize(device)
        barrier(device)
    launches = kvq.kernel_launches() - launches0
    clocks = clk.summary()
    assert cache.status() == 0
    total_ms = t0.elapsed_time(t1)
    pre = [e[0].elapsed_time(e[1]) for e in evs]
    app = [e[1].elapsed_time(e[2]) for e in evs]
    dec = [e[2].elapsed_time(e[3]) for e in evs]

    b_pre = A.prefill_bytes(wl, S)
    b_app = A.append_bytes(wl, S)
    b_dec = A.decode_bytes(wl, S + 1)
    b_step = b_pre + b_app + b_dec
    max_ms = reduce_max(total_ms, device)
    all_bytes = reduce_sum(b_step * args.steps, device)
    value = all_bytes / (max_ms * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()
    m_pre, m_dec, m_app = statistics.mean(pre), statistics.mean(dec), statistics.mean(app)

    # decode alone, L2 scrubbed before each launch (kernel timed in isolation)
    scrub = torch.empty(512 << 20, dtype=torch.uint8, device=device)
    alone = []
    for i in range(max(5, args.steps)):
        scrub.zero_()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        cache.decode(0, q, scale, out=out, workspace=ws)
        a1.record(stream)
        torch.cuda.synchronize(device)
        alone.append(a0.elapsed_time(a1))
    m_alone = statistics.median(alone)
    del scrub

    e2e = run_e2e(args, wl, cache, k, v, q, k1, v1, out, ws, scale, device, b_step)

    # dominant kernel of the step (by time): the quantize (prefill) step
    dom = max((("prefill_quantize", m_pre, b_pre), ("decode_attention", m_dec, b_dec),
               ("append_quantize", m_app, b_app)), key=lambda t: t[1])
    gbs = lambda b, ms: b / (ms * 1e-3) / 1e9  # noqa: E731
    traffic = load_traffic(wl, dom[0])
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(max_ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded fp16, distribution of the workload)",
        "config": {"workload": wl.name, "batch": wl.batch, "q_heads": wl.num_q_heads,
                   "kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim, "seq_len": S,
                   "k_codec": codec_name(wl.k_bits, wl.k_mode, wl.k_group),
                   "v_codec": codec_name(wl.v_bits, wl.v_mode, wl.v_group),
                   "outliers_per_row": wl.outliers_per_row,
                   "step": "prefill_quantize + append_quantize + decode_attention",
                   "l2": "inputs larger than L2 (%.2f GiB fp16 K/V per step); decode_alone scrubs L2"
                         % (2 * k.numel() * 2 / 2 ** 30)},
        "decode_attention": {"gbs": round(gbs(b_dec, m_dec), 1), "ms": round(m_dec, 4),
                             "bytes": b_dec, "frac": round(gbs(b_dec, m_dec) / peak, 4),
                             "alone_l2_scrubbed_gbs": round(gbs(b_dec, m_alone), 1),
                             "alone_frac": round(gbs(b_dec, m_alone) / peak, 4)},
        "quantize": {"gbs": round(gbs(b_pre, m_pre), 1), "ms": round(m_pre, 4), "bytes": b_pre,
                     "frac": round(gbs(b_pre, m_pre) / peak, 4)},
        "append_us": round(m_app * 1e3, 2),
        "roofline": {"kernel": dom[0], "bound": "hbm", "achieved": round(gbs(dom[2], dom[1]), 1),
                     "peak": peak, "peak_kind": peak_kind + " (hbm_gbs, copy)", "unit": "GB/s",
                     "frac": round(gbs(dom[2], dom[1]) / peak, 4), "traffic": traffic,
                     "algorithmic_bytes": dom[2]},
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": launches,
    }
    return line


def codec_name(bits, mode, group):
    kind = {0: "sym int%d per-token G=%d", 1: "asym %d-bit per-token G=%d",
            2: "asym %d-bit per-channel T=%d"}[mode]
    return kind % (bits, group)


def load_traffic(wl, kernel):
    """DRAM bytes per launch (read + write) from the committed ncu summary
    profiles/traffic.txt, lines "<workload> <kernel> <bytes>", when it holds
    this workload and kernel; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        with open(p) as f:
            for ln in f:
                parts = ln.split()
                if len(parts) == 3 and parts[0] == wl.name and parts[1] == kernel:
                    return int(float(parts[2]))
    except OSError:
        pass
    return None


def run_e2e(args, wl, cache, k, v, q, k1, v1, out, ws, scale, device, b_step):
    """The same step through host buffers: pinned host -> device copies of the
    step's inputs, the three C-ABI calls, and a device -> host read of the
    output, all inside the timed region."""
    hk = torch.empty_like(k, device="cpu").pin_memory()
    hv = torch.empty_like(v, device="cpu").pin_memory()
    hq = torch.empty_like(q, device="cpu").pin_memory()
    hk1 = torch.empty_like(k1, device="cpu").pin_memory()
    hv1 = torch.empty_like(v1, device="cpu").pin_memory()
    hout = torch.empty_like(out, device="cpu").pin_memory()
    for h, d in ((hk, k), (hv, v), (hq, q), (hk1, k1), (hv1, v1)):
        h.copy_(d)
    dk, dv = torch.empty_like(k), torch.empty_like(v)
    dq, dk1, dv1 = torch.empty_like(q), torch.empty_like(k1), torch.empty_like(v1)
    h2d = sum(t.numel() * t.element_size() for t in (hk, hv, hq, hk1, hv1))
    d2h = hout.numel() * hout.element_size()

    def step():
        dk.copy_(hk, non_blocking=True)
        dv.copy_(hv, non_blocking=True)
        dq.copy_(hq, non_blocking=True)
        dk1.copy_(hk1, non_blocking=True)
        dv1.copy_(hv1, non_blocking=True)
        cache.prefill(0, dk, dv)
        cache.append(0, dk1, dv1)
        cache.decode(0, dq, scale, out=out, workspace=ws)
        hout.copy_(out, non_blocking=True)

    n = max(3, min(args.steps, 10))
    for _ in range(2):
        step()
    torch.cuda.synchronize(device)
    barrier(device)
    t = time.perf_counter()
    for _ in range(n):
        step()
    torch.cuda.synchronize(device)
    dt = reduce_max(time.perf_counter() - t, device)
    tot = reduce_sum(b_step * n, device)
    return {"value": round(tot / dt / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(dt / n * 1e3, 3), "steps": n}


# ---------------------------------------------------------------------------
# CPU oracle (the baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_step_on_sample(wl, n_streams, seed):
    """One full step of the oracle over the first n_streams (batch, kv-head)
    streams of the workload; returns (seconds, algorithmic bytes)."""
    import numpy as np
    from bit_quantized_kv_kvq_gb300.synth import LayerSource
    from oracle import kvq_oracle as O

    src = LayerSource(wl, 0, device="cpu", seed=seed)
    k, v = src.kv(wl.seq_len, batch=1)
    q, k1, v1 = src.step(0, batch=1)
    hk = k.shape[1]
    n_streams = min(n_streams, hk)
    kk = k[0, :n_streams].numpy()
    vv = v[0, :n_streams].numpy()
    g = wl.gqa
    qq = q[0, :n_streams * g].double().numpy().reshape(n_streams, g, wl.head_dim)
    spec = O.CodecSpec(wl.head_dim, wl.k_bits, wl.v_bits, wl.k_mode, wl.v_mode, wl.k_group,
                       wl.v_group, wl.outliers_per_row)
    t = time.perf_counter()
    oc = O.OracleCache(spec, n_streams)
    oc.prefill(kk, vv)
    oc.append(k1[0, :n_streams].numpy(), v1[0, :n_streams].numpy())
    oc.decode(qq, 1.0 / math.sqrt(wl.head_dim))
    dt = time.perf_counter() - t
    frac = n_streams / float(wl.batch * wl.num_kv_heads)
    S = wl.seq_len
    b = (A.prefill_bytes(wl, S) + A.append_bytes(wl, S) + A.decode_bytes(wl, S + 1)) * frac
    del np
    return dt, b


def cpu_sample(wl, budget_s):
    """Times the oracle on a bounded sample of the workload: as many (batch,
    kv-head) streams as one batch holds, repeated until about budget_s seconds
    of CPU work have been spent."""
    dt1, _ = oracle_step_on_sample(wl, 1, wl.seed)
    n = max(1, min(wl.num_kv_heads, int(budget_s / max(dt1, 1e-3))))
    tot_s, tot_b, reps = 0.0, 0.0, 0
    while reps == 0 or tot_s < 0.8 * budget_s:
        dt, b = oracle_step_on_sample(wl, n, wl.seed + reps)
        tot_s += dt
        tot_b += b
        reps += 1
    return {"value": round(tot_b / tot_s / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": "%d x %d of %d (batch, kv-head) streams at the full context %d, one full "
                      "step each (prefill + append + decode), numpy single thread"
                      % (reps, n, wl.batch * wl.num_kv_heads, wl.seq_len),
            "seconds": round(tot_s, 2)}


def run_reference(args, wl, rank, world):
    if rank != 0:
        return None
    dt1, _ = oracle_step_on_sample(wl, 1, wl.seed)
    budget_total = 150.0
    per_step = budget_total / max(1, args.steps + args.warmup)
    n = max(1, min(wl.num_kv_heads, int(per_step / max(dt1, 1e-3))))
    for _ in range(args.warmup):
        oracle_step_on_sample(wl, n, wl.seed)
    times, byts = [], []
    for _ in range(args.steps):
        dt, b = oracle_step_on_sample(wl, n, wl.seed)
        times.append(dt)
        byts.append(b)
    total = sum(times)
    value = sum(byts) / total / 1e9
    sample = ("%d of %d (batch, kv-head) streams at the full context %d per step, numpy single "
              "thread" % (n, wl.batch * wl.num_kv_heads, wl.seq_len))
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded fp16, distribution of the workload)",
        "config": {"workload": wl.name, "batch": wl.batch, "q_heads": wl.num_q_heads,
                   "kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim, "seq_len": wl.seq_len,
                   "step": "prefill_quantize + append_quantize + decode_attention"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def profile_case(args, wl):
    """A short untimed run for profilers: prefill, append and decode of the
    workload's codec and shape at a reduced batch, args.reps times."""
    import dataclasses
    import bit_quantized_kv_kvq_gb300 as kvq
    from bit_quantized_kv_kvq_gb300.synth import LayerSource

    if args.batch:
        wl = dataclasses.replace(wl, batch=args.batch)
    if args.seq:
        wl = dataclasses.replace(wl, seq_len=args.seq)
    device = torch.device("cuda", 0)
    S = wl.seq_len
    cache = kvq.QuantizedKVCache(1, wl.batch, wl.num_kv_heads, wl.head_dim, S + 1, wl.k_bits,
                                 wl.v_bits, wl.k_mode, wl.v_mode, wl.k_group, wl.v_group,
                                 wl.outliers_per_row, device=device)
    src = LayerSource(wl, 0, device=device)
    k, v = src.kv(S)
    q, k1, v1 = src.step(0)
    for _ in range(args.reps):
        cache.prefill(0, k, v)
        cache.append(0, k1, v1)
        cache.decode(0, q, 1.0 / math.sqrt(wl.head_dim))
    torch.cuda.synchronize(device)
    if cache.status() != 0:
        raise RuntimeError("device status word %#x" % cache.status())
    print(json.dumps({"profile_case": wl.name, "batch": wl.batch, "seq_len": wl.seq_len, "reps": args.reps}),
          flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.BY_NAME))
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-case", action="store_true",
                    help="untimed prefill/append/decode repetitions for a profiler")
    ap.add_argument("--batch", type=int, default=0, help="batch of --profile-case (0: workload's)")
    ap.add_argument("--reps", type=int, default=2, help="repetitions of --profile-case")
    ap.add_argument("--seq", type=int, default=0, help="context length of --profile-case (0: workload's)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    wl = W.BY_NAME[args.workload]
    if args.profile_case:
        profile_case(args, wl)
        return 0
    rank, world, local = dist_env()
    if args.impl == "reference":
        line = run_reference(args, wl, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(device)
        dist.init_process_group("nccl", device_id=device)
    line = run_gpu(args, wl, rank, world, device)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_sample(wl, args.cpu_budget)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
