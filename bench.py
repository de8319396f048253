"""Benchmark of the hot path: blockwise ring attention + Ulysses permutation.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one pass of the whole path over one batch of synthetic input.
The default workload is the causal Llama-3.1-8B-shaped attention the metric
names (llama8b_32k: B=1, S=32768, Hq=32, Hkv=8, d=128, P=8 contiguous ring
blocks, position_ids 0..S-1, bf16): a step is the doc_start scan of
position_ids plus causal blockwise attention (one library call).  The
ulysses_4k workload (--workload ulysses_4k) times the Ulysses layer instead:
    seq_to_head(q, k, v)                                 Ulysses all-to-all #1
    blockwise attention, batch P*B, H/P heads, P ring blocks (online merge)
    head_to_seq(out)                                     Ulysses all-to-all #2

Reported value: attention TFLOP/s over the whole step (algorithmic FLOPs:
4*d per allowed (query, key) pair per query head), aggregated over ranks.
L2 (129 MB) is flushed between timed steps, outside the timed events, by
writing a 512 MiB buffer and then reading another 512 MiB buffer: the read
evicts the dirty lines the write leaves behind, so that their write-back does
not land in the next timed kernel (the flush leaves L2 cold and clean).
The JSON line also carries the attention kernel's roofline, an end-to-end
number with host buffers, the CPU oracle baseline and the SM clocks sampled
during the timed region; under "extra", each other timed workload with its
own roofline fraction and clock record: the Ulysses layer of ulysses_4k
(with the permutation's bandwidth in both directions, also reported under
"permute"), packed_128k in both block orders, halfmil_512k striped, the
llama8b_32k backward in both dQ forms, the packed_128k and halfmil_512k
striped backwards,
the forward and backward of an 8-device ring simulated through the per-device
calls, the
fused Ulysses path, the Ulysses + Ring hybrid, two merges of partials and two
large permutations.

Multi-GPU: every rank runs its own independent replica of the step (the
head groups / batches of the path are independent; no collective on the data
path), weak scaling; time = max over ranks.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("causal blockwise-attention TFLOP/s (% BF16 peak); seq↔head permute GB/s")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DEFAULT_WORKLOAD = "llama8b_32k"
# dram__bytes_read.sum + dram__bytes_write.sum per launch of the attention
# kernel, recorded from an ncu capture together with a SHA-256 of the kernel's
# sources at capture time; reported only while the sources still match.
TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "dram_traffic.json")
KERNEL_SOURCES = ("attn_bf16.cu", "attn_common.cuh", "ptx.cuh", "common.cuh")


def _code_only(text):
    """C++ source without comments and whitespace: what the compiler sees of
    it (a comment edit leaves the recorded capture valid, a code edit does not)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return re.sub(r"\s+", "", text)


def kernel_sources_sha256(read=None):
    """SHA-256 of the attention kernel's sources (code only).  `read(name)`
    returns a file's text (default: the working tree)."""
    import hashlib
    if read is None:
        def read(name):
            with open(os.path.join(ROOT, "sequence_parallelism_gb300", "csrc", name)) as f:
                return f.read()
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        h.update(_code_only(read(name)).encode())
    return h.hexdigest()


def recorded_traffic(workload):
    """(bytes per launch or None, note)."""
    try:
        with open(TRAFFIC_RECORD) as f:
            rec = json.load(f)["attn_bf16_kernel"].get(workload)
    except (OSError, ValueError, KeyError):
        return None, "no capture recorded"
    if rec is None:
        return None, "no capture recorded for this workload"
    if rec.get("sources_sha256") != kernel_sources_sha256():
        return None, "kernel sources changed since the capture"
    return rec["bytes_per_launch"], rec.get("note", "ncu capture of the current sources")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def attention_flops(cfg, pos):
    """4*d FLOPs per allowed (query, key) pair per query head."""
    B, S, Hq, d = cfg["B"], cfg["S"], cfg["Hq"], cfg["d"]
    if cfg.get("ulysses"):
        return 4.0 * d * S * S * Hq * B
    if pos is None:
        pairs = float(S) * S
    else:
        # pairs per document: L(L+1)/2 (position_ids restart per document)
        pairs = 0.0
        row = pos[0]
        starts = np.flatnonzero(np.concatenate([[1], row[1:] != row[:-1] + 1]))
        ends = np.concatenate([starts[1:], [S]])
        for a, b in zip(starts, ends):
            L = float(b - a)
            pairs += L * (L + 1) / 2
    return 4.0 * d * pairs * Hq * B


# ------------------------------------------------------ multi-rank logic
def rank_seed(seed, rank):
    """Each rank draws its own replica of the workload (weak scaling)."""
    return seed + 7919 * rank


class L2Flush:
    """Evicts L2 (129 MB) between timed iterations: write 512 MiB, then read
    512 MiB of another buffer so that no dirty line of the write is left to be
    written back inside the next timed kernel."""

    def __init__(self, device="cuda"):
        import torch
        self.wr = torch.empty(512 << 20, dtype=torch.uint8, device=device)
        self.rd = torch.zeros(128 << 20, dtype=torch.float32, device=device)

    def __call__(self):
        self.wr.zero_()
        self.rd.sum()


def max_over_ranks(value, world, device=None):
    """Slowest rank's value (the job takes as long as its slowest rank)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_step, world, steps, max_ms):
    """Whole-job throughput: every rank's FLOPs over the slowest rank's time."""
    return flops_per_step * world * steps / (max_ms * 1e-3) / 1e12


# --------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ our arm
def _attn_roofline(flops, ms, peaks, peak_kind, workload):
    achieved = flops / (ms * 1e-3) / 1e12
    traffic, note = recorded_traffic(workload)
    sustained = peaks.get("bf16_tflops_sustained")
    return {"kernel": "attn_bf16_kernel", "bound": "tensor", "achieved": round(achieved, 1),
            "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": round(achieved / peaks["bf16_tflops"], 4),
            "peak_source": f"{peak_kind} bf16 dense (burst)",
            # a run of thousands of back-to-back launches holds the GPU at its
            # power cap: the sustained GEMM figure is measured under the same
            "frac_of_sustained": round(achieved / sustained, 4) if sustained else None,
            "traffic": traffic, "traffic_note": note,
            "algorithmic_flops_per_launch": flops}


def run_ours(args, rank, world, local_rank):
    import torch

    import sequence_parallelism_gb300 as sp
    import workloads
    from sequence_parallelism_gb300 import _lib

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    cfg = dict(workloads.CONFIGS[args.workload])
    B, S, Hq, Hkv, d, P = (cfg[k] for k in ("B", "S", "Hq", "Hkv", "d", "P"))
    order = cfg["orders"][-1] if args.order is None else args.order
    if cfg["dtype"] != "bf16":
        raise SystemExit("bench.py times the bf16 tensor-core path")
    q, k, v = workloads.qkv_torch(B, S, Hq, Hkv, d, rank_seed(cfg["seed"], rank), torch.bfloat16,
                                  dev)
    pos_np = workloads.position_ids(cfg)
    pos = None if pos_np is None else torch.from_numpy(pos_np).to(dev)
    flops = attention_flops(cfg, pos_np)
    ulysses = bool(cfg.get("ulysses"))
    stream = torch.cuda.current_stream()

    if ulysses:
        G = Hq // P
        yq = torch.empty((P, B, S, G, d), dtype=torch.bfloat16, device=dev)
        yk, yv, yo = torch.empty_like(yq), torch.empty_like(yq), torch.empty_like(yq)
        ylse = torch.empty((P * B, G, S), dtype=torch.float32, device=dev)
        out = torch.empty_like(q)
        ws = sp.attention_workspace(P * B, S, False, dev)
        perm_bytes = 2.0 * 3 * q.numel() * 2  # read + write of q, k, v
        inv_bytes = 2.0 * q.numel() * 2

        def enqueue(qq, kk, vv, pp, oo, ev=None):
            n = 0
            if ev:
                ev[0].record(stream)
            _lib.sp_ulysses_seq_to_head_qkv(qq, kk, vv, yq, yk, yv, P)
            n += _lib.sp_last_launch_count()
            if ev:
                ev[1].record(stream)
            _lib.sp_blockwise_attn_fwd(yq.view(P * B, S, G, d), yk.view(P * B, S, G, d),
                                       yv.view(P * B, S, G, d), None, P, order, 0.0,
                                       yo.view(P * B, S, G, d), ylse, ws)
            n += _lib.sp_last_launch_count()
            if ev:
                ev[2].record(stream)
            _lib.sp_ulysses_head_to_seq(yo, oo, P)
            n += _lib.sp_last_launch_count()
            if ev:
                ev[3].record(stream)
            return n
    else:
        out = torch.empty_like(q)
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=dev)
        ws = sp.attention_workspace(B, S, pos is not None, dev)
        perm_bytes = inv_bytes = 0.0

        def enqueue(qq, kk, vv, pp, oo, ev=None):
            if ev:
                ev[0].record(stream)
                ev[1].record(stream)
            _lib.sp_blockwise_attn_fwd(qq, kk, vv, pp, P, order, 0.0, oo, lse, ws)
            n = _lib.sp_last_launch_count()
            if ev:
                ev[2].record(stream)
                ev[3].record(stream)
            return n

    def step(ev=None):
        return enqueue(q, k, v, pos, out, ev)

    flush = L2Flush(dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st, code = _lib.sp_get_device_error(ws)
    if st != 0:
        raise RuntimeError(f"device error word {code:#x} after warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    launches = 0
    for i in range(args.steps):
        flush()  # evict L2 between steps (outside the timed events)
        launches += step(evs[i])
    torch.cuda.synchronize()
    barrier()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    st, code = _lib.sp_get_device_error(ws)
    if st != 0:
        raise RuntimeError(f"device error word {code:#x} in the timed region")

    step_ms = [e[0].elapsed_time(e[3]) for e in evs]
    attn_ms = [e[1].elapsed_time(e[2]) for e in evs]
    perm_ms = [e[0].elapsed_time(e[1]) for e in evs]
    inv_ms = [e[2].elapsed_time(e[3]) for e in evs]
    tot_ms = max_over_ranks(float(sum(step_ms)), world, dev)
    ms_per_step = tot_ms / args.steps
    value = job_tflops(flops, world, args.steps, tot_ms)

    peaks, peak_kind = load_peaks()
    roofline = _attn_roofline(flops, statistics.mean(attn_ms), peaks, peak_kind, args.workload)
    roofline["timed_segment"] = ("the library call: doc_start scan + attention kernel" if pos
                                 is not None else "the attention call (kernel + tail-split merge)")

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 q/k/v; seeded packed-document position_ids)",
        "config": dict(workload_config(args.workload, cfg, order, world),
                       l2="flushed between timed steps (512 MiB write, then 512 MiB read)"),
        "roofline": roofline,
        "gpu_launches": launches,
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 3),
    }
    if ulysses:
        result["permute"] = permute_summary(perm_bytes / (statistics.mean(perm_ms) * 1e-3) / 1e9,
                                            inv_bytes / (statistics.mean(inv_ms) * 1e-3) / 1e9,
                                            peaks)
    result["e2e"] = e2e(args, inputs=(q, k, v, pos), out=out, enqueue=enqueue, flops=flops,
                        world=world, dev=dev)
    if not args.skip_extra and rank == 0 and world == 1:
        del q, k, v, out
        if ulysses:
            del yq, yk, yv, yo
        result["extra"] = extra_measurements(args, peaks, peak_kind, flush)
        if "permute" not in result and "ulysses_4k_layer" in result["extra"]:
            result["permute"] = result["extra"]["ulysses_4k_layer"]["permute"]
    if rank == 0 and world == 1 and not args.skip_cpu:
        result["cpu_baseline"] = cpu_baseline(cfg, args.workload, order, budget_s=args.cpu_budget)
    return result


def permute_summary(s2h_gbs, h2s_gbs, peaks):
    """Both directions of the Ulysses permutation against measured HBM
    bandwidth; `frac` is the slower direction's."""
    f1, f2 = s2h_gbs / peaks["hbm_gbs"], h2s_gbs / peaks["hbm_gbs"]
    return {"kernel": "permute_kernel (vector copy; launches reading < 128 MiB): seq_to_head of "
                      "q,k,v in one launch, head_to_seq of the output",
            "bound": "hbm", "seq_to_head_GBps": round(s2h_gbs, 1),
            "head_to_seq_GBps": round(h2s_gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac_seq_to_head": round(f1, 4), "frac_head_to_seq": round(f2, 4),
            "frac": round(min(f1, f2), 4),
            "note": "ulysses_4k: 3 x 32 MiB seq->head, 32 MiB head->seq; L2 flushed before each "
                    "step; bytes = read + write"}


def e2e(args, inputs, out, enqueue, flops, world, dev):
    """Same step through the public API with host buffers: every step uploads
    its inputs (q, k, v and, for causal workloads, position_ids) from pinned
    host memory and downloads its output to pinned host memory, all inside
    the timed region.  The copies run on their own streams against
    double-buffered device tensors, so step n+1's upload and step n-1's
    download overlap step n's kernels (the host link, ~210 GB/s per direction
    on this machine, is the bound when the kernels are short)."""
    import torch
    inputs = [t for t in inputs if t is not None]
    comp = torch.cuda.current_stream()
    torch.cuda.synchronize()
    ref = out.cpu()  # the device-timed steps' result on the same inputs
    hosts = [t.cpu().pin_memory() for t in inputs]
    bufs_in = [tuple(inputs), tuple(torch.empty_like(t) for t in inputs)]
    bufs_out = [out, torch.empty_like(out)]
    hout = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    s_up, s_down = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]     # upload of buffer b landed
    ev_done = [torch.cuda.Event() for _ in range(2)]   # step on buffer b finished
    ev_out = [torch.cuda.Event() for _ in range(2)]    # download of buffer b finished

    def issue(i):
        b = i % 2
        s_up.wait_event(ev_done[b])          # the step that last read buffer b is done
        with torch.cuda.stream(s_up):
            for h, t in zip(hosts, bufs_in[b]):
                t.copy_(h, non_blocking=True)
        ev_in[b].record(s_up)
        comp.wait_event(ev_in[b])
        comp.wait_event(ev_out[b])           # its output buffer has been downloaded
        bi = bufs_in[b]
        enqueue(bi[0], bi[1], bi[2], bi[3] if len(bi) > 3 else None, bufs_out[b])
        ev_done[b].record(comp)
        s_down.wait_event(ev_done[b])
        with torch.cuda.stream(s_down):
            hout[b].copy_(bufs_out[b], non_blocking=True)
        ev_out[b].record(s_down)

    n = max(3, min(args.steps, 200))
    for i in range(3):
        issue(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    s_up.wait_event(e0)
    for i in range(n):
        issue(i)
    comp.wait_stream(s_down)
    e1.record(comp)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    # what came back to the host is what the device-timed steps computed
    # (the kernels are deterministic): both download buffers, bit for bit
    for b in range(2):
        if not torch.equal(hout[b], ref):
            raise RuntimeError(f"end-to-end output (buffer {b}) differs from the device result")
    h2d = sum(t.numel() * t.element_size() for t in inputs)
    d2h = out.numel() * out.element_size()
    return {"value": round(job_tflops(flops, world, n, ms), 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(ms / n, 4), "steps": n, "checked": True,
            "note": "uploads and downloads on two copy streams, double-buffered, overlapping "
                    "the kernels of the neighbouring steps"}


def _timed(call, flush, stream, reps, warm=3):
    """Median and list of CUDA-event times (ms) of `call` over reps, L2
    flushed before each, with the SM clocks sampled meanwhile."""
    import torch
    for _ in range(warm):
        call()
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.2)
    ms = []
    for _ in range(reps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        call()
        b.record(stream)
        ms.append((a, b))
    torch.cuda.synchronize()
    clocks = sampler.stop()
    t = [a.elapsed_time(b) for a, b in ms]
    return statistics.median(t), t, clocks


def causal_attention_measurement(name, order, peaks, peak_kind, flush, stream, reps):
    """One causal workload's attention call (doc_start scan + kernel), with
    its roofline fraction and clock record."""
    import torch

    import sequence_parallelism_gb300 as sp
    import workloads
    from sequence_parallelism_gb300 import _lib

    cfg = workloads.CONFIGS[name]
    B, S, Hq, Hkv, d, P = (cfg[k] for k in ("B", "S", "Hq", "Hkv", "d", "P"))
    q, k, v = workloads.qkv_torch(B, S, Hq, Hkv, d, cfg["seed"], torch.bfloat16, "cuda")
    pos_np = workloads.position_ids(cfg)
    pos = torch.from_numpy(pos_np).cuda()
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
    ws = sp.attention_workspace(B, S, True)
    t, _, clocks = _timed(lambda: _lib.sp_blockwise_attn_fwd(q, k, v, pos, P, order, 0.0, out,
                                                              lse, ws), flush, stream, reps)
    st, code = _lib.sp_get_device_error(ws)
    if st != 0:
        raise RuntimeError(f"device error word {code:#x} in {name} {order}")
    fl = attention_flops(cfg, pos_np)
    rl = _attn_roofline(fl, t, peaks, peak_kind, name)
    sustained = peaks.get("bf16_tflops_sustained")
    return {"workload": name, "order": order, "P": P, "ms": round(t, 4),
            "TFLOP/s": rl["achieved"], "frac_of_bf16_peak": rl["frac"],
            "frac_of_sustained_bf16_peak": round(rl["achieved"] / sustained, 4) if sustained
            else None, "roofline": rl,
            "flops": fl, "reps": reps, "clocks": clocks,
            "note": "doc_start scan + attention kernel, median of reps, L2 flushed"}


def ulysses_layer_measurement(peaks, peak_kind, flush, stream, reps=50):
    """The Ulysses layer of ulysses_4k: seq->head of q, k, v (one launch),
    attention per head group, head->seq; each segment timed with events."""
    import torch

    import sequence_parallelism_gb300 as sp
    import workloads
    from sequence_parallelism_gb300 import _lib

    cfg = workloads.CONFIGS["ulysses_4k"]
    B, S, Hq, Hkv, d, P = (cfg[k] for k in ("B", "S", "Hq", "Hkv", "d", "P"))
    G = Hq // P
    q, k, v = workloads.qkv_torch(B, S, Hq, Hkv, d, cfg["seed"], torch.bfloat16, "cuda")
    yq = torch.empty((P, B, S, G, d), dtype=torch.bfloat16, device="cuda")
    yk, yv, yo = torch.empty_like(yq), torch.empty_like(yq), torch.empty_like(yq)
    ylse = torch.empty((P * B, G, S), dtype=torch.float32, device="cuda")
    out = torch.empty_like(q)
    ws = sp.attention_workspace(P * B, S, False)

    def layer(ev=None):
        if ev:
            ev[0].record(stream)
        _lib.sp_ulysses_seq_to_head_qkv(q, k, v, yq, yk, yv, P)
        if ev:
            ev[1].record(stream)
        _lib.sp_blockwise_attn_fwd(yq.view(P * B, S, G, d), yk.view(P * B, S, G, d),
                                   yv.view(P * B, S, G, d), None, P, "contiguous", 0.0,
                                   yo.view(P * B, S, G, d), ylse, ws)
        if ev:
            ev[2].record(stream)
        _lib.sp_ulysses_head_to_seq(yo, out, P)
        if ev:
            ev[3].record(stream)

    for _ in range(3):
        layer()
    torch.cuda.synchronize()
    # the same layer captured once into a CUDA graph and replayed (the launch
    # gaps between its kernels shrink; the kernels are the same)
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        layer()
    torch.cuda.synchronize()
    graph_ms, _, _ = _timed(graph.replay, flush, stream, reps)
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.2)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(reps)]
    for i in range(reps):
        flush()
        layer(evs[i])
    torch.cuda.synchronize()
    clocks = sampler.stop()
    seg = lambda a, b: statistics.mean([e[a].elapsed_time(e[b]) for e in evs])
    step, perm, attn, inv = seg(0, 3), seg(0, 1), seg(1, 2), seg(2, 3)
    fl = attention_flops(cfg, None)
    rl = _attn_roofline(fl, attn, peaks, peak_kind, "ulysses_4k")
    perm_gbs = 2.0 * 3 * q.numel() * 2 / (perm * 1e-3) / 1e9
    inv_gbs = 2.0 * q.numel() * 2 / (inv * 1e-3) / 1e9
    return {"ms_per_step": round(step, 4), "TFLOP/s_step": round(fl / (step * 1e-3) / 1e12, 1),
            "graph_ms_per_step": round(graph_ms, 4),
            "graph_TFLOP/s_step": round(fl / (graph_ms * 1e-3) / 1e12, 1),
            "attention_ms": round(attn, 4), "frac_of_bf16_peak": rl["frac"], "roofline": rl,
            "permute": permute_summary(perm_gbs, inv_gbs, peaks), "reps": reps,
            "clocks": clocks, "note": "mean of reps, L2 flushed before each step"}


def extra_measurements(args, peaks, peak_kind, flush):
    """Every other timed workload, each with its own roofline fraction and
    clock record (events, L2 flushed between reps)."""
    import torch

    import workloads
    from sequence_parallelism_gb300 import _lib

    res = {}
    stream = torch.cuda.current_stream()
    if args.workload != "ulysses_4k":
        res["ulysses_4k_layer"] = ulysses_layer_measurement(peaks, peak_kind, flush, stream)
    for name, order, reps in (("llama8b_32k", "contiguous", 20), ("packed_128k", "contiguous", 20),
                              ("packed_128k", "striped", 20), ("halfmil_512k", "striped", 5)):
        if name == args.workload and order == (args.order or workloads.CONFIGS[name]["orders"][-1]):
            continue
        res[f"{name}_{order}"] = causal_attention_measurement(name, order, peaks, peak_kind, flush,
                                                              stream, reps)
    res["llama8b_32k_causal_backward"] = backward_measurement(peaks, flush, stream)
    res["packed_128k_striped_backward"] = backward_measurement(
        peaks, flush, stream, "packed_128k", "striped", reps=10, two_forms=False)
    res["halfmil_512k_striped_backward"] = backward_measurement(
        peaks, flush, stream, "halfmil_512k", "striped", reps=3, two_forms=False)
    res["llama8b_32k_ring_forward_per_device"] = ring_forward_measurement(peaks, flush, stream)
    res["llama8b_32k_ring_backward_per_device"] = ring_backward_measurement(peaks, flush, stream)
    res.update(next_row_measurements(peaks, flush, stream))
    res["merge_partials"] = merge_measurement(peaks, flush, stream)
    # the q shapes of llama8b_32k (256 MiB) and packed_128k (1 GiB)
    for S_, label in ((32768, "permute_256MiB"), (131072, "permute_1GiB")):
        x = torch.randn((1, S_, 32, 128), device="cuda").to(torch.bfloat16)
        y = torch.empty((8, 1, S_, 4, 128), dtype=torch.bfloat16, device="cuda")
        t1, _, _ = _timed(lambda: _lib.sp_ulysses_seq_to_head(x, y, 8), flush, stream, 20)
        t2, _, _ = _timed(lambda: _lib.sp_ulysses_head_to_seq(y, x, 8), flush, stream, 20)
        g1 = 2.0 * x.numel() * 2 / (t1 * 1e-3) / 1e9
        g2 = 2.0 * x.numel() * 2 / (t2 * 1e-3) / 1e9
        res[label] = {"kernel": "permute_bulk_kernel (TMA-staged: launches reading >= 128 MiB)",
                      "seq_to_head_GBps": round(g1, 1), "head_to_seq_GBps": round(g2, 1),
                      "frac_of_hbm": round(min(g1, g2) / peaks["hbm_gbs"], 4),
                      "shape": f"[1][{S_}][32][128] bf16, P=8"}
        del x, y
    return res


def merge_measurement(peaks, flush, stream, reps=20):
    """sp_attn_merge_partials against measured HBM bandwidth on inputs larger
    than L2: a 2-way merge of full llama8b_32k-shaped partials and an 8-way
    merge of 8192-token partials.  Bytes per row: P partial rows of 2d bytes
    and P log-sum-exps read, one row and one log-sum-exp written."""
    import torch

    from sequence_parallelism_gb300 import _lib

    res = {"kernel": "merge_vec_kernel", "bound": "hbm", "peak": peaks["hbm_gbs"],
           "unit": "GB/s"}
    fr = []
    for P_, S_ in ((2, 32768), (8, 8192)):
        H, d = 32, 128
        g = torch.Generator(device="cuda").manual_seed(11 + P_)
        outs = torch.randn((P_, 1, S_, H, d), device="cuda", generator=g).to(torch.bfloat16)
        lses = torch.randn((P_, 1, H, S_), device="cuda", generator=g)
        out = torch.empty((1, S_, H, d), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((1, H, S_), dtype=torch.float32, device="cuda")
        t, _, clocks = _timed(lambda: _lib.sp_attn_merge_partials(outs, lses, out, lse), flush,
                              stream, reps)
        rows = S_ * H
        nbytes = rows * ((P_ + 1) * (2 * d + 4))
        gbs = nbytes / (t * 1e-3) / 1e9
        f = gbs / peaks["hbm_gbs"]
        fr.append(f)
        res[f"P{P_}"] = {"shape": f"{P_} x [1][{S_}][{H}][{d}] bf16", "us": round(t * 1e3, 1),
                         "bytes": nbytes, "achieved": round(gbs, 1), "frac": round(f, 4),
                         "clocks": clocks}
        del outs, lses, out, lse
    res["frac"] = round(min(fr), 4)
    res["note"] = "L2 flushed before each rep; median of reps; frac is the lower of the two"
    return res


def next_row_measurements(peaks, flush, stream):
    """The permutation-free Ulysses path (attention run directly on the
    sequence-sharded ulysses_4k tensors: every head group in place, output
    already in sequence-sharded layout) and the Ulysses + Ring hybrid on
    halfmil_512k (P_u = 8 head groups x P_r = 2 striped ring blocks), timed
    like the rest (events, L2 flushed, median of reps)."""
    import torch

    import sequence_parallelism_gb300 as sp
    import workloads
    from sequence_parallelism_gb300 import _lib

    res = {}
    cfg = workloads.CONFIGS["ulysses_4k"]
    B, S, Hq, Hkv, d, P = (cfg[k] for k in ("B", "S", "Hq", "Hkv", "d", "P"))
    q, k, v = workloads.qkv_torch(B, S, Hq, Hkv, d, cfg["seed"], torch.bfloat16, "cuda")
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
    ws = sp.attention_workspace(B, S, False)
    t, _, clocks = _timed(lambda: _lib.sp_blockwise_attn_fwd(q, k, v, None, P, "contiguous", 0.0,
                                                              out, lse, ws), flush, stream, 50)
    fl = attention_flops(cfg, None)
    tf = fl / (t * 1e-3) / 1e12
    res["ulysses_4k_fused"] = {
        "ms": round(t, 4), "TFLOP/s": round(tf, 1),
        "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4), "flops": fl, "clocks": clocks,
        "note": "attention on the sequence-sharded tensors, no permutation launches"}
    del q, k, v, out, lse, ws
    cfg = workloads.CONFIGS["halfmil_512k"]
    B, S, Hq, Hkv, d = (cfg[k] for k in ("B", "S", "Hq", "Hkv", "d"))
    P_u, P_r = 8, 2
    q, k, v = workloads.qkv_torch(B, S, Hq, Hkv, d, cfg["seed"], torch.bfloat16, "cuda")
    pos_np = workloads.position_ids(cfg)
    pos = torch.from_numpy(pos_np).cuda()
    out = torch.empty_like(q)
    lse = torch.empty((P_u, B, Hq // P_u, S), dtype=torch.float32, device="cuda")
    ws = torch.empty(_lib.sp_ulysses_ring_attn_workspace_bytes(B, S, Hq, Hkv, d, True,
                                                               _lib._dtype(q)),
                     dtype=torch.uint8, device="cuda")
    t, _, clocks = _timed(lambda: _lib.sp_ulysses_ring_attn_fwd(q, k, v, pos, P_u, P_r, "striped",
                                                                 0.0, out, lse, ws),
                          flush, stream, 3)
    fl = attention_flops(cfg, pos_np)
    tf = fl / (t * 1e-3) / 1e12
    res["halfmil_512k_hybrid_8x2"] = {
        "ms": round(t, 2), "TFLOP/s": round(tf, 1),
        "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4), "flops": fl, "clocks": clocks,
        "note": "seq->head with 8 groups, striped ring attention over 2 blocks per group, "
                "head->seq; one call"}
    del q, k, v, out, lse, ws
    return res


def backward_measurement(peaks, flush, stream, name="llama8b_32k", order="contiguous", reps=20,
                         two_forms=True):
    """Attention backward (dq, dk, dv), L2 flushed between reps, in the
    default form (doc_start scan, prep, the fused kernel -- S^T and dP^T
    once per pair of tiles, dQ pieces summed by TMA bulk reductions -- and
    the dq conversion) and, with two_forms, the bit-reproducible two-kernel
    form (dQ recomputed by its own kernel).  Algorithmic FLOPs = 2.5 x the
    forward's (five d-long products per allowed pair: S, dP, dV, dQ, dK)."""
    import torch

    import sequence_parallelism_gb300 as sp
    import workloads
    from sequence_parallelism_gb300 import _lib

    cfg = workloads.CONFIGS[name]
    B, S, Hq, Hkv, d, P = (cfg[k] for k in ("B", "S", "Hq", "Hkv", "d", "P"))
    q, k, v = workloads.qkv_torch(B, S, Hq, Hkv, d, cfg["seed"], torch.bfloat16, "cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(cfg["seed"] + 7)
    dout = torch.randn(q.shape, generator=g, device="cuda").to(torch.bfloat16)
    pos_np = workloads.position_ids(cfg)
    pos = torch.from_numpy(pos_np).cuda()
    out, lse = sp.blockwise_attention(q, k, v, P, order, pos)
    ws = torch.empty(_lib.sp_blockwise_attn_bwd_workspace_bytes(B, S, Hq, P, True),
                     dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    call = lambda: _lib.sp_blockwise_attn_bwd(q, k, v, out, dout, lse, pos, P, order, 0.0,
                                              dq, dk, dv, ws)
    fl = 2.5 * attention_flops(cfg, pos_np)

    def one(form_reduction):
        prev = _lib.sp_set_bwd_dq_reduction(form_reduction)
        try:
            t, _, clocks = _timed(call, flush, stream, reps)
            launches = _lib.sp_last_launch_count()
        finally:
            _lib.sp_set_bwd_dq_reduction(prev)
        tf = fl / (t * 1e-3) / 1e12
        return {"ms": round(t, 4), "TFLOP/s": round(tf, 1),
                "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
                "frac_of_sustained_bf16_peak": (round(tf / peaks["bf16_tflops_sustained"], 4)
                                                if peaks.get("bf16_tflops_sustained") else None),
                "launches_per_call": launches, "clocks": clocks}

    res = one(True)
    res.update({"workload": name, "order": order, "flops": fl, "reps": reps,
                "note": "doc_start scan + prep + fused dK/dV/dQ kernel (dQ pieces summed "
                        "by TMA bulk reductions into float32) + dq conversion, median of "
                        "reps; flops = 2.5 x forward (S, dP, dV, dQ, dK)"})
    if two_forms:
        res["two_kernel_form"] = dict(one(False), note="doc_start scan + prep + dQ + dK/dV "
                                      "kernels (dQ recomputed; bit-reproducible)")
    return res


def ring_forward_measurement(peaks, flush, stream, reps=10, compare=True):
    """The forward of an 8-device ring simulated on one GPU (llama8b_32k,
    contiguous blocks), as dist.ring_attention runs it on each device: step 0
    by sp_ring_block_step, steps 1..P-1 folded into the running result by
    sp_ring_block_step_accumulate (P^2 = 64 calls per rep).  Also timed: the
    same ring with every step written by sp_ring_block_step and folded by
    sp_attn_merge_partials (56 merges), unless compare is False.  FLOPs: the
    attention's algorithmic count."""
    import torch

    import sequence_parallelism_gb300 as sp
    import workloads
    from sequence_parallelism_gb300 import _lib

    cfg = workloads.CONFIGS["llama8b_32k"]
    B, S, Hq, Hkv, d, P = (cfg[k] for k in ("B", "S", "Hq", "Hkv", "d", "P"))
    q, k, v = workloads.qkv_torch(B, S, Hq, Hkv, d, cfg["seed"], torch.bfloat16, "cuda")
    pos_np = workloads.position_ids(cfg)
    pos = torch.from_numpy(pos_np).cuda()
    Lb = S // P
    rows = [torch.arange(p * Lb, (p + 1) * Lb, device="cuda") for p in range(P)]
    qb = [q.index_select(1, r).contiguous() for r in rows]
    kb = [k.index_select(1, r).contiguous() for r in rows]
    vb = [v.index_select(1, r).contiguous() for r in rows]
    del q, k, v
    outs = [torch.empty((2, B, Lb, Hq, d), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    lses = [torch.empty((2, B, Hq, Lb), dtype=torch.float32, device="cuda") for _ in range(2)]
    ws = sp.attention_workspace(B, S, True)

    def ring_accumulate():
        for i in range(P):
            for s_ in range(P):
                j = (i - s_) % P
                if s_ == 0:
                    _lib.sp_ring_block_step(qb[i], kb[j], vb[j], pos, S, P, "contiguous", i, j,
                                            0.0, outs[0][0], lses[0][0], ws)
                else:
                    _lib.sp_ring_block_step_accumulate(qb[i], kb[j], vb[j], pos, S, P,
                                                       "contiguous", i, j, 0.0, outs[0][0],
                                                       lses[0][0], ws)

    def ring_merge():
        for i in range(P):
            cur = 0
            for s_ in range(P):
                j = (i - s_) % P
                slot = 0 if s_ == 0 else 1
                _lib.sp_ring_block_step(qb[i], kb[j], vb[j], pos, S, P, "contiguous", i, j, 0.0,
                                        outs[cur][slot], lses[cur][slot], ws)
                if s_ > 0:
                    _lib.sp_attn_merge_partials(outs[cur], lses[cur], outs[1 - cur][0],
                                                lses[1 - cur][0])
                    cur = 1 - cur

    t, _, clocks = _timed(ring_accumulate, flush, stream, reps)
    fl = attention_flops(cfg, pos_np)
    tf = fl / (t * 1e-3) / 1e12
    res = {"ms": round(t, 4), "TFLOP/s": round(tf, 1),
           "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
           "calls_per_rep": P * P, "reps": reps, "clocks": clocks,
           "note": "8 simulated devices x 8 ring steps; causal contiguous pairs with j > i add "
                   "nothing (the accumulating call returns without a launch); median of reps"}
    if compare:
        t2, _, clocks2 = _timed(ring_merge, flush, stream, reps)
        tf2 = fl / (t2 * 1e-3) / 1e12
        res["step_and_merge"] = {"ms": round(t2, 4), "TFLOP/s": round(tf2, 1),
                                 "frac_of_bf16_peak": round(tf2 / peaks["bf16_tflops"], 4),
                                 "merges_per_rep": P * (P - 1), "clocks": clocks2}
    st_, code = _lib.sp_get_device_error(ws)
    if st_ != 0:
        raise RuntimeError(f"device error word {code:#x} in the ring forward")
    return res


def ring_backward_measurement(peaks, flush, stream, reps=5):
    """The backward of an 8-device ring simulated on one GPU (llama8b_32k,
    contiguous blocks): every device's P steps as sp_ring_block_step_bwd
    calls on block tensors, P^2 = 64 calls per rep, float32 accumulators;
    what one device of a real ring computes is 1/P of it.  Same FLOP rule
    as the whole-sequence backward."""
    import torch

    import sequence_parallelism_gb300 as sp
    import workloads
    from sequence_parallelism_gb300 import _lib

    cfg = workloads.CONFIGS["llama8b_32k"]
    B, S, Hq, Hkv, d, P = (cfg[k] for k in ("B", "S", "Hq", "Hkv", "d", "P"))
    q, k, v = workloads.qkv_torch(B, S, Hq, Hkv, d, cfg["seed"], torch.bfloat16, "cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(cfg["seed"] + 7)
    dout = torch.randn(q.shape, generator=g, device="cuda").to(torch.bfloat16)
    pos_np = workloads.position_ids(cfg)
    pos = torch.from_numpy(pos_np).cuda()
    out, lse = sp.blockwise_attention(q, k, v, P, "contiguous", pos)
    Lb = S // P
    rows = [torch.arange(p * Lb, (p + 1) * Lb, device="cuda") for p in range(P)]
    blk = lambda t, p, ax=1: t.index_select(ax, rows[p]).contiguous()
    qb, kb, vb = [blk(q, p) for p in range(P)], [blk(k, p) for p in range(P)], [blk(v, p) for p in range(P)]
    ob, db, lb = [blk(out, p) for p in range(P)], [blk(dout, p) for p in range(P)], [blk(lse, p, 2) for p in range(P)]
    del q, k, v, out, dout, lse
    acc = [(torch.zeros((B, Lb, Hq, d), device="cuda"), torch.zeros((B, Lb, Hkv, d), device="cuda"),
            torch.zeros((B, Lb, Hkv, d), device="cuda")) for _ in range(P)]
    ws = torch.empty(_lib.sp_ring_block_step_bwd_workspace_bytes(B, S, Hq, P, True),
                     dtype=torch.uint8, device="cuda")

    def ring():
        for i in range(P):
            for s_ in range(P):
                j = (i - s_) % P
                _lib.sp_ring_block_step_bwd(qb[i], kb[j], vb[j], ob[i], db[i], lb[i], pos, S, P,
                                            "contiguous", i, j, 0.0, acc[i][0], acc[j][1],
                                            acc[j][2], ws)

    t, _, clocks = _timed(ring, flush, stream, reps)
    st_, code = _lib.sp_get_device_error(ws)
    if st_ != 0:
        raise RuntimeError(f"device error word {code:#x} in the ring backward")
    fl = 2.5 * attention_flops(cfg, pos_np)
    tf = fl / (t * 1e-3) / 1e12
    return {"ms": round(t, 4), "TFLOP/s": round(tf, 1),
            "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
            "calls_per_rep": P * P, "reps": reps, "clocks": clocks,
            "note": "64 sp_ring_block_step_bwd calls (8 simulated devices x 8 ring steps; "
                    "causal pairs with j > i find no allowed tile), median of reps"}


# ------------------------------------------------------- CPU oracle leg
def _oracle_inputs(cfg):
    import workloads
    B, S, Hq, Hkv, d = (cfg[k] for k in ("B", "S", "Hq", "Hkv", "d"))
    rng = np.random.default_rng(cfg["seed"])
    q = rng.standard_normal((B, S, Hq, d)).astype(np.float32)
    k = rng.standard_normal((B, S, Hkv, d)).astype(np.float32)
    v = rng.standard_normal((B, S, Hkv, d)).astype(np.float32)
    return q, k, v, workloads.position_ids(cfg)


def _oracle_sample(cfg, order, rows, inputs):
    """One bounded sample of the workload through the oracle (inputs drawn
    beforehand); returns (algorithmic FLOPs done, seconds)."""
    import oracle
    import workloads

    B, S, Hq, Hkv, d, P = (cfg[k] for k in ("B", "S", "Hq", "Hkv", "d", "P"))
    q, k, v, pos = inputs
    sel = workloads.sample_rows(S, P, rows, cfg["seed"], order)
    t0 = time.perf_counter()
    if cfg.get("ulysses"):
        yq, yk, yv = (oracle.seq_to_head(t, P) for t in (q, k, v))
        G = Hq // P
        full = np.zeros((P, B, S, G, d))
        for r in range(P):
            o, _ = oracle.attention_rows(yq[r], yk[r], yv[r], sel, None)
            full[r][:, sel] = o
        oracle.head_to_seq(full)
        fl = 4.0 * d * S * len(sel) * Hq * B
    else:
        oracle.attention_rows(q, k, v, sel, pos)
        sec = time.perf_counter() - t0
        starts = oracle.doc_starts(pos[:, :int(sel.max()) + 1])
        allowed = (sel - starts[0, sel] + 1).astype(np.float64)
        return 4.0 * d * float(allowed.sum()) * Hq * B, sec
    return fl, time.perf_counter() - t0


def _calibrated_rows(cfg, order, inputs, seconds):
    """Rows whose oracle time is about `seconds`: t(rows) = a + b * rows from
    two small samples."""
    _, t1 = _oracle_sample(cfg, order, 8, inputs)
    _, t2 = _oracle_sample(cfg, order, 40, inputs)
    b = max((t2 - t1) / 32.0, 1e-6)
    a = max(t1 - 8 * b, 0.0)
    return int(max(1, min(cfg["S"], (seconds - a) / b)))


def cpu_baseline(cfg, workload, order, budget_s=15.0):
    inputs = _oracle_inputs(cfg)
    rows = _calibrated_rows(cfg, order, inputs, budget_s)
    fl, sec = _oracle_sample(cfg, order, rows, inputs)
    return {"value": round(fl / sec / 1e12, 6), "unit": "TFLOP/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{workload}: {rows} seeded query rows x all heads "
                      f"(float64 NumPy oracle{', plus full q/k/v/out permutations' if cfg.get('ulysses') else ''}),"
                      f" {sec:.1f} s; BLAS threads = library default (all cores)",
            "seconds": round(sec, 2)}


def workload_config(name, cfg, order, world):
    """The `config` keys both arms report for a workload."""
    return {"workload": name, "B": cfg["B"], "S": cfg["S"], "Hq": cfg["Hq"], "Hkv": cfg["Hkv"],
            "d": cfg["d"], "P": cfg["P"], "order": order, "causal": bool(cfg.get("causal")),
            "parallelism": f"replicas{world}" if world > 1 else "single GPU"}


def run_reference(args, rank, world):
    """The oracle as it stands, timed on the host cores: each step one bounded
    sample of the workload, sized so K + W steps take about two minutes."""
    if rank != 0:
        return None
    import workloads
    cfg = dict(workloads.CONFIGS[args.workload])
    order = cfg["orders"][-1] if args.order is None else args.order
    inputs = _oracle_inputs(cfg)
    per_step = 120.0 / max(1, args.steps + args.warmup)
    rows = _calibrated_rows(cfg, order, inputs, per_step)
    for _ in range(args.warmup):
        _oracle_sample(cfg, order, rows, inputs)
    tot_fl, tot_s = 0.0, 0.0
    for _ in range(args.steps):
        fl, s = _oracle_sample(cfg, order, rows, inputs)
        tot_fl += fl
        tot_s += s
    value = tot_fl / tot_s / 1e12
    sample = f"{args.workload}: {rows} seeded query rows x all heads per step (float64 NumPy oracle)"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tot_s * 1e3 / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(workload_config(args.workload, cfg, order, world),
                           l2="not applicable (host cores)"),
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "kind": "oracle",
                             "cores": os.cpu_count(), "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--order", default=None, choices=[None, "contiguous", "striped"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--skip-extra", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if not os.path.exists(os.path.join(ROOT, "sequence_parallelism_gb300", "libsp_gb300.so")):
        if rank == 0:  # one rank compiles; the others wait for it
            import __graft_entry__
            __graft_entry__.build()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
