"""Benchmark of the hot path on one GB300 (or N replicas).

The default workload is the full 8B-shaped decode: 32 layers x 8 kv-heads (32
query heads), head_dim 128, batch 1, a 131072-token context prefill-quantized
into the cache (4-bit per-channel keys, 8-bit per-token values), then decode
steps that each append one token and run fused dequant decode attention on
every layer. One timed step = append on all layers, then decode attention on
all layers, through the C ABI, with inputs resident in HBM. Each layer's
packed cache (218 MB) is larger than L2 (129 MB), so consecutive decodes read
from HBM; single-layer workloads flush L2 between steps (outside the decode's
own timing).

Prints one JSON line (rank 0). ``value`` is the fused dequant decode-attention
throughput in GB/s: the algorithmic bytes the decode attention of all layers
reads and writes per step (packed codes, fp16 scales and zero points, outlier
lists, fp16 residual keys, q, output), divided by the decode time of the step
(CUDA events around the block of decode calls). The line also carries the
whole-step time, the prefill quantize and append throughputs, the roofline of
the decode kernel, clocks, the end-to-end number through host buffers and the
CPU oracle baseline.

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
DEFAULT_WORKLOAD = W.LLAMA8B_FULL.name
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


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


def tensor_peak():
    """Dense fp16/bf16 tensor-core peak (TFLOP/s): the measured cuBLAS bf16
    burst figure (fp16 inputs with fp32 accumulation run at the same rate)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def prefill_attention_timing(wl, model, device, flush, chunk=1024, reps=3):
    """kvq_prefill_attention of the queries of layer 0's last `chunk`
    positions over its whole cache, L2 flushed before each run. Algorithmic
    flops: 4 D per (query head, query, visible token) (QK^T and PV, 2 D
    each)."""
    cache = model.cache
    S = model.length()
    rows = cache.seq_lengths(0)  # each batch row's tokens (ragged batches: its own)
    chunk = min(chunk, min(rows))
    gen = torch.Generator(device=device)
    gen.manual_seed(wl.seed + 77)
    q = torch.randn((wl.batch, chunk, wl.num_q_heads, wl.head_dim), generator=gen, device=device).half()
    out = torch.empty(q.shape, dtype=torch.float32, device=device)
    cache.prefill_attention(0, q, model.scale, out=out)
    ts = []
    for i in range(reps):
        if flush is not None:
            flush(i)
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record()
        cache.prefill_attention(0, q, model.scale, out=out)
        a1.record()
        torch.cuda.synchronize(device)
        ts.append(a0.elapsed_time(a1))
    assert cache.status() == 0
    visible = sum(chunk * (n - chunk) + chunk * (chunk + 1) // 2 for n in rows)
    flops = 4 * wl.head_dim * wl.num_q_heads * visible
    m = statistics.median(ts)
    peak, kind = tensor_peak()
    tf = flops / (m * 1e-3) / 1e12
    return {"ms": round(m, 3), "chunk": chunk, "context": S, "flops": flops, "tflops": round(tf, 1),
            "frac": round(tf / peak, 4), "peak": peak, "peak_kind": kind + " (bf16_tflops, dense; of " + kind + ")",
            "bound": "tensor",
            "what": "causal attention of the queries of layer 0's last %d positions of every batch row over the "
                    "row's cached tokens (%d at most; kvq_prefill_attention, fp32 out)" % (chunk, S)}


def gpu_id(device):
    """nvidia-smi's name for a torch device: its UUID (the torch index is a
    logical one under CUDA_VISIBLE_DEVICES and need not match nvidia-smi's)."""
    try:
        u = str(torch.cuda.get_device_properties(device).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(device.index)


class ClockSampler:
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu):
        self.gpu = gpu
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
            return {"gpu": str(self.gpu), "sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"],
                    "samples": 0}

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
        return {"gpu": rows[0][0], "sm_mhz": statistics.median(load),
                "sm_max_mhz": max(num(r[2]) for r in rows), "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def gbs(b, ms):
    return b / (ms * 1e-3) / 1e9


class Model:
    """The workload's layers in one packed cache: every layer prefilled with
    its seeded context, then decode steps (append one token per stream and
    layer, decode attention of every layer)."""

    def __init__(self, wl, device, seed, max_steps):
        import bit_quantized_kv_kvq_gb300 as kvq
        from bit_quantized_kv_kvq_gb300.synth import LayerSource
        self.wl, self.device = wl, device
        self.S = wl.seq_len
        self.cache = kvq.QuantizedKVCache(wl.num_layers, wl.batch, wl.num_kv_heads, wl.head_dim,
                                          self.S + max_steps, wl.k_bits, wl.v_bits, wl.k_mode,
                                          wl.v_mode, wl.k_group, wl.v_group, wl.outliers_per_row,
                                          device=device, codebook=wl.codebook)
        self.src = [LayerSource(wl, l, device=device, seed=seed) for l in range(wl.num_layers)]
        self.ws = self.cache.workspace(wl.num_q_heads)
        self.scale = 1.0 / math.sqrt(wl.head_dim)
        self.out = torch.empty((wl.num_layers, wl.batch, wl.num_q_heads, wl.head_dim),
                               dtype=torch.float32, device=device)
        # per step and layer: (q, k1, v1), drawn ahead of time
        self.inputs = [[self.src[l].step(st) for l in range(wl.num_layers)] for st in range(max_steps)]

    def prefill_all(self):
        """Prefills every layer; returns the K/V of layer 0 (kept for the
        quantize timing)."""
        kv0 = None
        for l in range(self.wl.num_layers):
            k, v = self.src[l].kv(self.S)
            if self.wl.lens:  # a ragged batch: each row keeps its own tokens
                self.cache.prefill_varlen(l, k, v, list(self.wl.lens))
            else:
                self.cache.prefill(l, k, v)
            if l == 0:
                kv0 = (k, v)
            else:
                del k, v
        return kv0

    def length(self):
        return self.cache.length(0)


def l2_flush_buffers(device):
    """Two 256 MB buffers: writing one and then reading it back into the other
    leaves L2 (129 MB) holding clean lines unrelated to the cache."""
    a = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    b = torch.empty(256 << 20, dtype=torch.uint8, device=device)

    def flush(i):
        a.fill_(i & 255)
        b.copy_(a)
    return flush


def run_gpu(args, wl, rank, world, device):
    import bit_quantized_kv_kvq_gb300 as kvq

    torch.cuda.set_device(device)
    stream = torch.cuda.current_stream(device)
    L = wl.num_layers
    steps, warm = args.steps, args.warmup
    model = Model(wl, device, replica_seed(wl, rank), warm + 2 * steps + 14)
    cache, ws, scale, out = model.cache, model.ws, model.scale, model.out
    k0, v0 = model.prefill_all()
    torch.cuda.synchronize(device)
    assert cache.status() == 0
    # each layer's cache larger than L2 makes consecutive decodes cold; a
    # single layer that fits in L2 gets a flush before each step
    per_layer = A.cache_read_bytes(wl, model.S)
    need_flush = L == 1 or per_layer < 2 * (129 << 20)
    flush = l2_flush_buffers(device) if need_flush else None

    def decode_step(st, ev=None):
        if flush is not None:
            flush(st)
        if ev:
            ev[2].record(stream)
        for l in range(L):
            _, k1, v1 = model.inputs[st][l]
            cache.append(l, k1, v1)
        if ev:
            ev[0].record(stream)
        for l in range(L):
            q, _, _ = model.inputs[st][l]
            cache.decode(l, q, scale, out=out[l], workspace=ws)
        if ev:
            ev[1].record(stream)

    st = 0
    for _ in range(warm):
        decode_step(st)
        st += 1
    torch.cuda.synchronize(device)
    assert cache.status() == 0

    len0 = model.length()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    launches0 = kvq.kernel_launches()
    with ClockSampler(gpu_id(device)) as clk:
        barrier(device)
        torch.cuda.synchronize(device)
        t0.record(stream)
        for i in range(steps):
            decode_step(st + i, evs[i])
        t1.record(stream)
        torch.cuda.synchronize(device)
        barrier(device)
    launches = kvq.kernel_launches() - launches0
    clocks = clk.summary()
    assert cache.status() == 0
    st += steps
    total_ms = t0.elapsed_time(t1)

    # the same step with the appends on a second stream, where they overlap
    # the decodes of earlier layers (kvq_decode_step); flushed as above
    aux = torch.cuda.Stream(device)
    ov_ms = []
    for i in range(steps):
        if flush is not None:
            flush(st + i)
        ins = model.inputs[st + i]
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        cache.decode_step([x[0] for x in ins], [x[1] for x in ins], [x[2] for x in ins], scale, list(out),
                          workspace=ws, aux_stream=aux)
        e1.record(stream)
        torch.cuda.synchronize(device)
        ov_ms.append(e0.elapsed_time(e1))
    assert cache.status() == 0
    st += steps
    two_stream = {"ms_per_step": round(reduce_max(statistics.median(ov_ms), device), 4),
                  "serial_ms_per_step": round(reduce_max(total_ms, device) / steps, 4),
                  "what": "append on a second stream, each layer's decode waiting for its own append "
                          "(kvq_decode_step); both times include the L2 flush"}
    dec_ms = [e[0].elapsed_time(e[1]) for e in evs]
    app_ms = [e[2].elapsed_time(e[0]) for e in evs]
    # decode bytes of each timed step (the cache grows by one token per step)
    b_dec = [L * A.decode_bytes(wl, len0 + i + 1) for i in range(steps)]
    all_dec_bytes = reduce_sum(sum(b_dec), device)
    max_dec_ms = reduce_max(sum(dec_ms), device)
    value = all_dec_bytes / (max_dec_ms * 1e-3) / 1e9
    max_ms = reduce_max(total_ms, device)
    peak, peak_kind = hbm_peak()
    launch_ms = sum(dec_ms) / (steps * L)  # average decode launch (one layer)
    b_launch = sum(b_dec) / (steps * L)

    # prefill quantize of layer 0 (K/V of the whole context), timed apart
    qt = []
    for i in range(3 + max(3, min(steps, 10))):
        if flush is not None:
            flush(i)
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        if wl.lens:
            cache.prefill_varlen(0, k0, v0, list(wl.lens))
        else:
            cache.prefill(0, k0, v0)
        a1.record(stream)
        torch.cuda.synchronize(device)
        if i >= 3:
            qt.append(a0.elapsed_time(a1))
    b_pre = A.prefill_bytes(wl, model.S)
    m_pre = statistics.median(qt)
    # append of one token on layer 0 (restores the layer's length first)
    del k0, v0
    torch.cuda.synchronize(device)

    pattn = prefill_attention_timing(wl, model, device, flush)
    e2e = run_e2e(args, wl, model, st, device)
    err = e2e_error(wl, model, device)

    traffic = load_traffic(wl, "decode_attention")
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": steps, "warmup": warm, "ms_per_step": round(max_ms / steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded fp16, distribution of the workload)",
        "config": {"workload": wl.name, "layers": L, "batch": wl.batch, "q_heads": wl.num_q_heads,
                   "kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim, "context": model.S,
                   "k_codec": codec_name(wl.k_bits, wl.k_mode, wl.k_group),
                   "v_codec": codec_name(wl.v_bits, wl.v_mode, wl.v_group),
                   "outliers_per_row": wl.outliers_per_row,
                   "row_lengths": list(wl.lens) if wl.lens else None,
                   "step": "append_quantize on every layer, then decode_attention on every layer",
                   "l2": ("flushed before each step (256 MB written then read); one layer's cache is %.0f MB"
                          % (per_layer / 1e6)) if need_flush else
                         ("inputs larger than L2: each layer's packed cache is %.0f MB and the %d layers are "
                          "decoded in turn" % (per_layer / 1e6, L))},
        "decode_attention": {"gbs": round(value, 1), "ms_per_step": round(max_dec_ms / steps, 4),
                             "bytes_per_step": int(sum(b_dec) / steps),
                             "frac": round(value / peak, 4),
                             "launch_ms": round(launch_ms, 4), "launch_bytes": int(b_launch)},
        "step_gbs": round(all_dec_bytes / (max_ms * 1e-3) / 1e9, 1),
        "quantize": {"gbs": round(gbs(b_pre, m_pre), 1), "ms": round(m_pre, 4), "bytes": b_pre,
                     "frac": round(gbs(b_pre, m_pre) / peak, 4), "what": "prefill of one layer"},
        "append_us_per_layer": round(statistics.mean(app_ms) / L * 1e3, 2),
        "prefill_attention": pattn,
        "two_stream_step": two_stream,
        "roofline": {"kernel": "decode_attention", "bound": "hbm",
                     "achieved": round(gbs(b_launch, launch_ms), 1), "peak": peak,
                     "peak_kind": peak_kind + " (hbm_gbs, copy; of measured)", "unit": "GB/s",
                     "frac": round(gbs(b_launch, launch_ms) / peak, 4), "traffic": traffic,
                     "algorithmic_bytes": int(b_launch)},
        "e2e_error": err,
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": launches,
    }
    return line


def e2e_error(wl, model, device):
    """Error of the decoded attention against fp64 attention on the
    unquantized fp16 K/V (the inputs the cache was built from), for the
    first stream of layer 0, by bit width: max over the stream's query heads
    of max_d |o - o_ref| / max_d |o_ref|. The fp64 reference is plain torch
    (softmax(q k^T scale) v) on the host. Reported, not gated."""
    cache = model.cache
    src = model.src[0]
    n_len = model.length()
    k, v = src.kv(model.S)
    ks = [k[0, 0].cpu()]
    vs = [v[0, 0].cpu()]
    del k, v
    for st in range(n_len - model.S):
        _, k1, v1 = model.inputs[st][0]
        ks.append(k1[0, 0:1].cpu())
        vs.append(v1[0, 0:1].cpu())
    kf = torch.cat(ks, 0).double()
    vf = torch.cat(vs, 0).double()
    q, _, _ = model.inputs[0][0]
    o = cache.decode(0, q.to(device), model.scale).cpu().double()[0, :wl.gqa]
    qf = q[0, :wl.gqa].cpu().double()
    ref = torch.softmax((qf @ kf.T) * model.scale, dim=-1) @ vf
    e = float(((o - ref).abs().amax(-1) / ref.abs().amax(-1).clamp_min(1e-30)).max())
    return {"k%dv%d" % (wl.k_bits, wl.v_bits): round(e, 6),
            "what": "max row error of layer 0, stream 0 (%d query heads, %d tokens) against fp64 attention "
                    "on the unquantized fp16 K/V" % (wl.gqa, n_len)}


def codec_name(bits, mode, group):
    kind = {0: "sym int%d per-token G=%d", 1: "asym %d-bit per-token G=%d",
            2: "asym %d-bit per-channel T=%d", 3: "codebook %d-bit per-token G=%d"}[mode]
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


def run_e2e(args, wl, model, st0, device):
    """The same decode step through host buffers, as a caller would run it:
    every layer's q and appended K/V rows for the step packed in one pinned
    host buffer and copied host -> device at once, one kvq_decode_step (the
    appends on a second stream, each layer's decode after its own append),
    and a device -> host read of every layer's output, all inside the timed
    region."""
    L = wl.num_layers
    cache, ws, scale = model.cache, model.ws, model.scale
    n = max(3, min(args.steps, 10))
    shapes = [tuple(t.shape) for t in model.inputs[0][0]]  # q, k1, v1
    sizes = [math.prod(sh) for sh in shapes]
    offs = [0, sizes[0], sizes[0] + sizes[1]]
    width = sum(sizes)
    host = []
    for i in range(n + 1):
        h = torch.empty((L, width), dtype=torch.float16).pin_memory()
        for l in range(L):
            for j, t in enumerate(model.inputs[st0 + i][l]):
                h[l, offs[j]:offs[j] + sizes[j]].copy_(t.reshape(-1).cpu())
        host.append(h)
    dev = torch.empty((L, width), dtype=torch.float16, device=device)
    views = [[dev[l, offs[j]:offs[j] + sizes[j]].view(shapes[j]) for l in range(L)] for j in range(3)]
    hout = torch.empty_like(model.out, device="cpu").pin_memory()
    outs = list(model.out)
    aux = torch.cuda.Stream(device)
    h2d = host[0].numel() * host[0].element_size()
    d2h = hout.numel() * hout.element_size()

    def step(i):
        dev.copy_(host[i], non_blocking=True)
        cache.decode_step(views[0], views[1], views[2], scale, outs, workspace=ws, aux_stream=aux)
        hout.copy_(model.out, non_blocking=True)

    step(0)
    torch.cuda.synchronize(device)
    len0 = model.length()
    barrier(device)
    t = time.perf_counter()
    for i in range(1, n + 1):
        step(i)
    torch.cuda.synchronize(device)
    dt = reduce_max(time.perf_counter() - t, device)
    assert cache.status() == 0
    b = sum(L * A.decode_bytes(wl, len0 + i + 1) for i in range(n))
    tot = reduce_sum(b, device)
    return {"value": round(tot / dt / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(dt / n * 1e3, 3), "steps": n,
            "what": "one pinned host->device copy of every layer's q and new K/V rows, kvq_decode_step "
                    "(appends on a second stream), one device->host read of every layer's output"}


# ---------------------------------------------------------------------------
# CPU oracle (the baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(wl, n_streams, seed):
    """The oracle's cache for the first n_streams (batch, kv-head) streams of
    layer 0 at the full context (prefill, untimed)."""
    from bit_quantized_kv_kvq_gb300.synth import LayerSource
    from oracle import kvq_oracle as O
    src = LayerSource(wl, 0, device="cpu", seed=seed)
    k, v = src.kv(wl.seq_len, batch=1)
    n_streams = min(n_streams, wl.num_kv_heads)
    spec = O.CodecSpec(wl.head_dim, wl.k_bits, wl.v_bits, wl.k_mode, wl.v_mode, wl.k_group,
                       wl.v_group, wl.outliers_per_row, 0, wl.codebook)
    oc = O.OracleCache(spec, n_streams)
    t = time.perf_counter()
    oc.prefill(k[0, :n_streams].numpy(), v[0, :n_streams].numpy())
    return oc, src, n_streams, time.perf_counter() - t


def oracle_decode_step(wl, oc, src, n_streams, st):
    """One decode step of the oracle on its sample: append one token per
    stream, then decode attention; returns (seconds, decode bytes)."""
    q, k1, v1 = src.step(st, batch=1)
    g = wl.gqa
    qq = q[0, :n_streams * g].double().numpy().reshape(n_streams, g, wl.head_dim)
    t = time.perf_counter()
    oc.append(k1[0, :n_streams].numpy(), v1[0, :n_streams].numpy())
    oc.decode(qq, 1.0 / math.sqrt(wl.head_dim))
    dt = time.perf_counter() - t
    frac = n_streams / float(wl.batch * wl.num_kv_heads)
    return dt, A.decode_bytes(wl, oc.length) * frac


def cpu_sample(wl, budget_s):
    """Times the oracle on a bounded sample: one (batch, kv-head) stream of
    layer 0 at the full context, decode steps until about budget_s seconds
    of CPU work; reports decode-attention GB/s scaled to the sample."""
    oc, src, n, _ = oracle_sample(wl, 1, wl.seed)
    tot_s, tot_b, st = 0.0, 0.0, 0
    while st == 0 or tot_s < budget_s:
        dt, b = oracle_decode_step(wl, oc, src, n, st)
        tot_s += dt
        tot_b += b
        st += 1
    return {"value": round(tot_b / tot_s / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": "%d decode steps (append + attention) of 1 of %d (batch, kv-head) streams of one "
                      "layer at the full %d-token context, numpy single thread"
                      % (st, wl.batch * wl.num_kv_heads, wl.seq_len),
            "seconds": round(tot_s, 2)}


def run_reference(args, wl, rank, world):
    if rank != 0:
        return None
    oc, src, n, _ = oracle_sample(wl, 1, wl.seed)
    for st in range(args.warmup):
        oracle_decode_step(wl, oc, src, n, st)
    times, byts = [], []
    for i in range(args.steps):
        dt, b = oracle_decode_step(wl, oc, src, n, args.warmup + i)
        times.append(dt)
        byts.append(b)
    total = sum(times)
    value = sum(byts) / total / 1e9
    sample = ("one decode step (append + attention) per step on 1 of %d (batch, kv-head) streams of "
              "one layer at the full %d-token context, numpy single thread"
              % (wl.batch * wl.num_kv_heads, wl.seq_len))
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded fp16, distribution of the workload)",
        "config": {"workload": wl.name, "layers": wl.num_layers, "batch": wl.batch,
                   "q_heads": wl.num_q_heads, "kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim,
                   "context": wl.seq_len,
                   "step": "append_quantize + decode_attention (oracle sample)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def profile_case(args, wl):
    """A short untimed run for profilers: prefill, append and decode of the
    workload's codec and shape at a reduced batch, args.reps times; with
    --chunk C, then the prefill attention of the last C positions."""
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
                                 wl.outliers_per_row, device=device, codebook=wl.codebook)
    src = LayerSource(wl, 0, device=device)
    k, v = src.kv(S)
    q, k1, v1 = src.step(0)
    for _ in range(args.reps):
        cache.prefill(0, k, v)
        cache.append(0, k1, v1)
        cache.decode(0, q, 1.0 / math.sqrt(wl.head_dim))
    if args.chunk:
        gen = torch.Generator(device=device)
        gen.manual_seed(wl.seed + 77)
        qc = torch.randn((wl.batch, min(args.chunk, S + 1), wl.num_q_heads, wl.head_dim), generator=gen,
                         device=device).half()
        cache.prefill_attention(0, qc, 1.0 / math.sqrt(wl.head_dim))
    torch.cuda.synchronize(device)
    if cache.status() != 0:
        raise RuntimeError("device status word %#x" % cache.status())
    print(json.dumps({"profile_case": wl.name, "batch": wl.batch, "seq_len": wl.seq_len, "reps": args.reps}),
          flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.BY_NAME))
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-case", action="store_true",
                    help="untimed prefill/append/decode repetitions for a profiler")
    ap.add_argument("--batch", type=int, default=0, help="batch of --profile-case (0: workload's)")
    ap.add_argument("--reps", type=int, default=2, help="repetitions of --profile-case")
    ap.add_argument("--seq", type=int, default=0, help="context length of --profile-case (0: workload's)")
    ap.add_argument("--chunk", type=int, default=0,
                    help="--profile-case: then prefill attention of the last CHUNK positions (0: none)")
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
