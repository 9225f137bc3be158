#!/usr/bin/env python
"""Benchmark of one absorbed MLA decode step on GB300.

A step is one pass of the whole path over one batch: append the n_q new tokens,
absorb the query, split attention, log-sum-exp combine, output up-projection.
The default workload is the batched decode (B=32, prior context 4096, one new
token per sequence, 64-token pages with a shuffled page table).

Printed (rank 0, one JSON line): ``value`` = latent-cache bytes the step reads
(every cached token once per sequence, 1152 B per token) summed over ranks,
divided by the mean step time (device time from CUDA events on the launching
stream, L2 flushed before every step, inputs resident in HBM).  ``e2e`` repeats
the measurement through the same calls with the step's inputs copied from
pinned host memory and the output copied back inside the timed region (the
upload by ``mla_copy_async``, the GPU's own loads over the host link; the
decode step's out-projection stores its result straight into the pinned
host buffer, other steps download it with ``mla_copy_async``).
``roofline`` rates the split-attention kernel against the measured HBM copy
bandwidth (or dense bf16 peak when FLOPs bind).  ``cpu_baseline`` times the
fp64 CPU oracle on a bounded sample of the same workload.

``--impl reference`` times that CPU oracle alone (rank 0 only) as the
reference arm.  Multi-GPU runs (torchrun) are independent replicas: each rank
decodes its own batch of the same workload, no collective on the data path.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from mla_absorbed_decode_absorb_gb300 import accounting as A  # noqa: E402
from mla_absorbed_decode_absorb_gb300 import workloads as W  # noqa: E402

METRIC = "MLA absorbed decode µs/step, latent-cache GB/s and TFLOP/s vs GB300 roofline"
METRIC_LAYER = "MLA decode layer (projections + absorbed attention) µs/step, HBM GB/s of weights and cache"
METRIC_PREFILL = "MLA non-absorbed chunked prefill, new tokens/s and TFLOP/s vs GB300 roofline"
PREFILL_KERNEL = "prefill attention (mla_prefill_attn)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
DOMINANT_KERNEL = "split attention (mla_decode_attn_partial)"
DOMINANT_KERNEL_FP8 = "split attention over the FP8 cache (mla_decode_attn_fp8_partial)"


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=400)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=W.DEFAULT_BENCH_WORKLOAD,
                   choices=sorted(W.WORKLOADS) + sorted(W.PREFILL_WORKLOADS) + sorted(W.FP8_WORKLOADS)
                   + sorted(W.LAYER_WORKLOADS))
    p.add_argument("--split-pages", type=int, default=None, help="override the workload's KV split size")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="CPU-oracle sample budget")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-per-workload", action="store_true",
                   help="skip the short per-workload pass over the other decode workloads")
    p.add_argument("--per-workload-steps", type=int, default=20)
    p.add_argument("--launch-overlap", type=int, default=2, choices=[0, 1, 2],
                   help="mla_set_launch_overlap level (2: weights are constant, read ahead)")
    return p.parse_args(argv)


# --------------------------------------------------------------------------- helpers
def reduce_over_ranks(times_ms, nbytes, device="cpu"):
    """Across ranks: the max of each per-rank time (ms) and the sum of the bytes processed.

    With one process (no process group) the inputs come back unchanged.
    """
    import torch.distributed as dist
    t = torch.tensor([float(x) for x in times_ms], dtype=torch.float64, device=device)
    n = torch.tensor([float(nbytes)], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return [float(x) for x in t.tolist()], float(n.item())


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_cores_info():
    """Threads the oracle's BLAS runs on (its ``cores``) and the cores this process may use."""
    return {"cores": blas_threads(), "blas_threads": blas_threads(), "host_cores": host_cores()}


def blas_threads():
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(k, "").isdigit():
            return int(os.environ[k])
    return host_cores()


def workload_config(wl: W.Workload, inp: W.Inputs | None, world: int, extra=None):
    cfg = {"workload": wl.name, "description": wl.description, "B": wl.batch, "n_q": wl.n_q,
           "n_h": W.N_HEADS, "d_c": W.D_LATENT, "d_rope": W.D_ROPE, "page_size": W.PAGE,
           "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
           "l2": ("flushed before every timed step: 256 MiB written, then another 256 MiB read, so that no line "
                  "of the step's inputs is in L2 and no dirty line of the flush is written back inside the step; "
                  "each step timed by CUDA events at its boundaries")}
    if wl.ragged:
        cfg["L_range"] = list(wl.ragged)
    else:
        cfg["L"] = wl.context
    if inp is not None:
        cfg["kv_tokens"] = int(inp.kv_lens.sum())
    cfg.update(extra or {})
    return cfg


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples taken while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.t0 = self.t1 = None
        self.path = os.path.join("/tmp", f"mla_bench_clocks_{os.getpid()}.csv")
        sel = []
        try:
            bus = torch.cuda.get_device_properties(device_index).pci_bus_id
            sel = ["-i", str(bus)]
        except Exception:
            pass
        self.cmd = ["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(self.cmd, stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------------------- CPU oracle timing
def oracle_sample(inp: W.Inputs, budget_s: float, max_seqs: int | None = None, absorbed: bool = False):
    """Run the fp64 oracle over whole sequences until the budget is spent; returns (bytes, seconds, seqs).

    ``absorbed`` times the oracle's absorbed fp64 form instead of the plain definition
    (a second CPU row: the same mathematics without decompressing K and V)."""
    import numpy as np

    from oracle import mla_oracle as O

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    w_uk, w_uv = O.bf16_bits_to_f64(bits(inp.w_uk)), O.bf16_bits_to_f64(bits(inp.w_uv))
    done, nbytes, t = 0, 0, 0.0
    for b in range(inp.batch if max_seqs is None else min(max_seqs, inp.batch)):
        c_bits, k_bits = (bits(x) for x in inp.sequence(b))
        q_nope, q_rope = O.bf16_bits_to_f64(bits(inp.q_nope[b])), O.bf16_bits_to_f64(bits(inp.q_rope[b]))
        t0 = time.perf_counter()
        kv = c_bits.shape[0]
        if inp.workload.cache_format == "fp8":
            pages = (kv + 63) // 64
            img = (np.full((pages, 64, 512), 0x7F, np.uint8), np.full((pages, 64), np.nan, np.float32),
                   np.full((pages, 64, 64), 0x7E00, np.uint16))
            img = O.append_kv_fp8(*img, c_bits[None], k_bits[None], [0], np.arange(pages)[None])
            c, kr = O.gather_sequence_fp8(*img, np.arange(pages), kv)
        else:
            c = O.bf16_bits_to_f64(c_bits)
            kr = O.bf16_bits_to_f64(O.rope_key_bf16_bits(k_bits, np.arange(kv)))
        (O.decode_absorbed if absorbed else O.decode_mha)(q_nope, q_rope, w_uk, w_uv, c, kr, int(inp.prior_lens[b]))
        t += time.perf_counter() - t0
        done += 1
        nbytes += kv * A.cache_bytes_per_token(cache_format=inp.workload.cache_format)
        if t >= budget_s:
            break
    return nbytes, t, done


def oracle_layer_sample(li, budget_s: float, max_seqs=None):
    """The fp64 layer oracle on whole sequences until ``budget_s`` is spent; returns
    (sequences done, seconds).  A step of the workload costs B times one sequence."""
    import numpy as np

    from oracle import mla_oracle as O

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)
    f64 = lambda t: O.bf16_bits_to_f64(bits(t))  # noqa: E731
    inp = li.base
    ws = [f64(w) for w in (li.w_dkv, li.w_kr, li.w_dq, li.w_uq, li.w_qr)]
    w_uk, w_uv, w_o = f64(inp.w_uk), f64(inp.w_uv), f64(li.w_o)
    done, t = 0, 0.0
    for b in range(inp.batch if max_seqs is None else min(max_seqs, inp.batch)):
        hc, hk = inp.history(b)
        L = int(inp.prior_lens[b])
        t0 = time.perf_counter()
        kr = O.bf16_bits_to_f64(O.rope_key_bf16_bits(bits(hk), np.arange(L)))
        O.decode_layer(f64(li.x[b]), *ws, w_uk, w_uv, w_o, f64(hc), kr, L)
        t += time.perf_counter() - t0
        done += 1
        if t >= budget_s:
            break
    return done, t


def oracle_prefill_sample(inp: W.Inputs, budget_s: float):
    """The fp64 oracle on a bounded sample of a many-token step: the first new
    tokens of sequence 0 on 16 heads, as many 8-token groups as the budget
    allows; returns (new tokens scaled to all 128 heads, seconds, description)."""
    import numpy as np

    from oracle import mla_oracle as O

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    heads = list(range(16))
    w_uk, w_uv = O.bf16_bits_to_f64(bits(inp.w_uk)), O.bf16_bits_to_f64(bits(inp.w_uv))
    c_bits, k_bits = (bits(x) for x in inp.sequence(0))
    kv = c_bits.shape[0]
    c = O.bf16_bits_to_f64(c_bits)
    kr = O.bf16_bits_to_f64(O.rope_key_bf16_bits(k_bits, np.arange(kv)))
    q_nope, q_rope = O.bf16_bits_to_f64(bits(inp.q_nope[0])), O.bf16_bits_to_f64(bits(inp.q_rope[0]))
    L = int(inp.prior_lens[0])
    done, t = 0, 0.0
    while done < q_nope.shape[0] and (done == 0 or t < budget_s):
        j0 = done
        t0 = time.perf_counter()
        # queries j0 .. j0+7 of the chunk: the oracle's definition with the prior context shifted
        O.decode_mha(q_nope[j0:j0 + 8], q_rope[j0:j0 + 8], w_uk, w_uv, c[:L + j0 + 8], kr[:L + j0 + 8], L + j0, heads)
        t += time.perf_counter() - t0
        done = min(q_nope.shape[0], j0 + 8)
    tokens = done * len(heads) / 128
    return tokens, t, f"first {done} new tokens of sequence 0 on 16 of 128 heads ({t:.1f} s), scaled to 128 heads"


def run_reference(args, wl):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    inp = W.generate(wl, seed=0)
    prefill = wl.name in W.PREFILL_WORKLOADS
    if prefill:  # the oracle on 8 new tokens x 16 heads per step, scaled to tokens of all heads
        sample_fn = lambda: oracle_prefill_sample(inp, 0.0)[:2]  # noqa: E731
        sample = "8 new tokens of sequence 0 on 16 of 128 heads per step, scaled to 128 heads"
        metric, unit, scale = METRIC_PREFILL, "tokens/s", 1.0
    elif wl.d_model > 0:  # one sequence through the layer oracle per step, a step costing B of them
        li = W.generate_layer(wl, seed=0)
        inp = li.base
        units_step = A.step_cache_bytes(inp.kv_lens.tolist()) + A.layer_weight_bytes(wl.d_model, fold=wl.fold)

        def sample_fn():
            _, t = oracle_layer_sample(li, 0.0, max_seqs=1)
            return units_step, t * inp.batch
        sample = f"one sequence of the layer workload per step, a step costing {inp.batch} of them"
        metric, unit, scale = METRIC_LAYER, "GB/s", 1e9
    else:
        sample_fn = lambda: oracle_sample(inp, 0.0, max_seqs=1)[:2]  # noqa: E731
        sample = f"one sequence ({int(inp.kv_lens[0])} cached tokens, all 128 heads) of the workload per step"
        metric, unit, scale = METRIC, "GB/s", 1e9
    for _ in range(args.warmup):
        sample_fn()
    per_step = []
    units = 0
    for _ in range(args.steps):
        u, t = sample_fn()
        per_step.append(t)
        units = u
    mean_t = sum(per_step) / len(per_step)
    value = units / mean_t / scale
    line = {
        "impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_t * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl, inp, world, {"sample": sample}),
        "cpu_baseline": {"value": value, "unit": unit, **cpu_cores_info(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# --------------------------------------------------------------------------- our path
def kernel_source_hash():
    src = os.path.join(ROOT, "mla_absorbed_decode_absorb_gb300", "csrc", "decode_attn.cu")
    with open(src, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the split-attention kernel from the committed ncu summary, if it is current."""
    path = os.path.join(ROOT, "profiles", "decode_attn_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("source_sha256_16") != kernel_source_hash():
            return None
        rec = d.get("workloads", {}).get(workload)
        return None if rec is None else float(rec["dram_bytes_per_launch"])
    except Exception:
        return None


def measure_decode_workload(name, dev, stream, flush_l2, steps, peaks):
    """A short pass over one more decode workload, measured like the headline one:
    whole steps and the split attention between CUDA events with L2 flushed
    before every step, plus warm-L2 steps back to back, eager and replayed from
    a CUDA graph (the number that matters for a cache that fits in L2)."""
    from mla_absorbed_decode_absorb_gb300.runtime import DecodeSession

    wl = W.WORKLOADS[name]
    inp = W.generate(wl, seed=0)
    s = DecodeSession(inp, device=dev)
    kv_list = inp.kv_lens.tolist()
    step_bytes = A.step_cache_bytes(kv_list)
    step_flops = A.step_attention_flops(kv_list, wl.n_q)
    for _ in range(3):
        flush_l2()
        s.step()
    torch.cuda.synchronize()
    stages = s.stage_names()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)] for _ in range(steps)]
    tot = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for k in range(steps):
        flush_l2()
        tot[k][0].record(stream)
        s.step()
        tot[k][1].record(stream)
    for k in range(steps):
        flush_l2()
        ev[k][0].record(stream)
        for i, st in enumerate(stages):
            getattr(s, st)()
            ev[k][i + 1].record(stream)
    torch.cuda.synchronize()
    step_ms = sum(a.elapsed_time(b) for a, b in tot) / steps
    stage_ms = {st: sum(ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(steps)) / steps
                for i, st in enumerate(stages)}
    attn_ms = stage_ms["attend_partial"]
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0.record(stream)
    for _ in range(steps):
        s.step()
    w1.record(stream)
    torch.cuda.synchronize()
    warm_ms = w0.elapsed_time(w1) / steps
    g = s.capture()
    torch.cuda.synchronize()
    w0.record(stream)
    for _ in range(steps):
        g.replay()
    w1.record(stream)
    torch.cuda.synchronize()
    graph_ms = w0.elapsed_time(w1) / steps
    from mla_absorbed_decode_absorb_gb300 import ops
    if ops.mla_get_device_status() != ops.MLA_OK:
        raise RuntimeError(f"device status set during the {name} pass")
    t_roof, bound = A.roofline_seconds(kv_list, wl.n_q, peaks["hbm_gbs"], peaks["bf16_tflops"])
    if bound == "hbm":
        achieved, peak, unit = step_bytes / (attn_ms * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s"
    else:
        achieved, peak, unit = step_flops / (attn_ms * 1e-3) / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    out = {"B": wl.batch, "n_q": wl.n_q, "kv_tokens": int(sum(kv_list)), "split_pages": s.split_pages,
           "num_splits": s.num_splits, "us_per_step": step_ms * 1e3, "attn_us": attn_ms * 1e3,
           "stage_us": {k: v * 1e3 for k, v in stage_ms.items()},
           "us_per_step_warm_l2": warm_ms * 1e3, "us_per_step_graph_warm_l2": graph_ms * 1e3,
           "algorithmic_bytes": step_bytes, "algorithmic_flops": step_flops,
           "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
                        "roofline_us": t_roof * 1e6},
           "steps": steps}
    del g, s
    torch.cuda.empty_cache()
    return out


def run_ours(args, wl):
    import torch.distributed as dist

    from mla_absorbed_decode_absorb_gb300 import ops
    from mla_absorbed_decode_absorb_gb300.runtime import DecodeSession, LayerSession

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    ops.mla_set_launch_overlap(args.launch_overlap)
    layer = wl.d_model > 0
    if layer:
        li = W.generate_layer(wl, seed=rank)
        inp = li.base
        s = LayerSession(li, device=dev, split_pages=args.split_pages, fold=wl.fold)
    else:
        inp = W.generate(wl, seed=rank)
        s = DecodeSession(inp, device=dev, split_pages=args.split_pages)
    stream = torch.cuda.current_stream()
    flush_w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    flush_r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_sink = torch.empty((), dtype=torch.float32, device=dev)

    def flush_l2():
        # Write a buffer larger than L2, then read another one: L2 ends up
        # holding clean lines of neither the step's inputs nor the written
        # buffer, so the step pays neither reuse nor the flush's write-backs.
        flush_w.zero_()
        torch.sum(flush_r, dim=0, out=flush_sink)
    kv_list = inp.kv_lens.tolist()
    prefill = s.path == "non_absorbed"
    fp8 = wl.cache_format == "fp8"
    step_bytes = A.step_cache_bytes(kv_list, wl.cache_format)
    if prefill:  # the metric counts new tokens; the roofline rates the attention's FLOPs
        step_units = wl.batch * wl.n_q
        step_flops = A.prefill_attention_flops(kv_list, wl.n_q)
        decompress_flops = A.decompress_flops(kv_list)
    else:
        step_units = step_bytes + (A.layer_weight_bytes(wl.d_model, fold=wl.fold) if layer else 0)
        step_flops = A.step_attention_flops(kv_list, wl.n_q)

    for _ in range(max(args.warmup, 3)):
        flush_l2()
        s.step()
    torch.cuda.synchronize()
    if ops.mla_get_device_status() != ops.MLA_OK:
        raise RuntimeError("device status set during warm-up")

    # Timed region: whole steps, events only at step boundaries (so that each
    # kernel may overlap its predecessor's tail), L2 flushed before every step.
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    clocks = ClockSampler(local_rank) if rank == 0 else None
    if clocks:
        clocks.start()
    barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for k in range(K):
        flush_l2()
        ev[k][0].record(stream)
        s.step()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    barrier()
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop() if clocks else None
    step_ms = [a.elapsed_time(b) for a, b in ev]
    if ops.mla_get_device_status() != ops.MLA_OK:
        raise RuntimeError("device status set during the timed region")

    # Stage breakdown (separate pass, an event after every launch): per-kernel
    # durations, and the attention kernel's for the roofline.
    stages = s.stage_names()
    K3 = min(K, 100)
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)] for _ in range(K3)]
    for k in range(K3):
        flush_l2()
        e = sev[k]
        e[0].record(stream)
        for i, name in enumerate(stages):
            getattr(s, name)()
            e[i + 1].record(stream)
    torch.cuda.synchronize()
    per_stage = [[sev[k][i].elapsed_time(sev[k][i + 1]) for k in range(K3)] for i in range(len(stages))]
    attn_i = stages.index("prefill_attn" if prefill else "attend_partial")
    (mean_ms, attn_ms), total_bytes = reduce_over_ranks([sum(step_ms) / K, sum(per_stage[attn_i]) / K3],
                                                       step_units, dev)
    if ops.mla_get_device_status() != ops.MLA_OK:
        raise RuntimeError("device status set during the stage breakdown")

    # the same steps without the L2 flush (warm L2: small caches fit in it), back to back
    K4 = min(K, 100)
    ew = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    torch.cuda.synchronize()
    ew[0].record(stream)
    for _ in range(K4):
        s.step()
    ew[1].record(stream)
    torch.cuda.synchronize()
    warm_ms = ew[0].elapsed_time(ew[1]) / K4

    # the same, each step replayed from one CUDA graph (one host call per step)
    graph_ms = None
    if isinstance(s, DecodeSession):
        sg = s.capture()
        torch.cuda.synchronize()
        ew[0].record(stream)
        for _ in range(K4):
            sg.replay()  # launches on the current stream
        ew[1].record(stream)
        torch.cuda.synchronize()
        graph_ms = ew[0].elapsed_time(ew[1]) / K4

    # end to end: inputs from pinned host memory, output back to host, inside the timed region
    e2e = None
    if not args.no_e2e:
        host_in = s.host_step_buffer(pin=True)   # all of this step's inputs, one packed buffer
        host_out = torch.empty(s.out.shape, dtype=s.out.dtype).pin_memory()
        h2d = host_in.numel()
        d2h = host_out.numel() * host_out.element_size()
        K2 = min(K, 200)
        e2e_ms = []
        for k in range(K2 + 3):
            flush_l2()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            s.upload(host_in)
            s.step(host_out=host_out)
            b.record(stream)
            b.synchronize()
            if k >= 3:
                e2e_ms.append(a.elapsed_time(b))
        (m,), _ = reduce_over_ranks([sum(e2e_ms) / len(e2e_ms)], 0, dev)
        e2e = {"value": total_bytes / (m * 1e-3) / (1 if prefill else 1e9), "unit": "tokens/s" if prefill else "GB/s",
               "ms_per_step": m, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    # mla_decode_attn as the C ABI defines it (split attention, then the separate
    # log-sum-exp merge kernel), timed apart from the step in which the merge is
    # fused into the out-projection
    attn_combine_ms = None
    if isinstance(s, DecodeSession) and s.path == "absorbed":
        ea = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K3)]
        for k in range(K3):
            flush_l2()
            ea[k][0].record(stream)
            s.attend_partial()
            if s.num_splits > 1:
                s.combine()
            ea[k][1].record(stream)
        torch.cuda.synchronize()
        (attn_combine_ms,), _ = reduce_over_ranks([sum(a.elapsed_time(b) for a, b in ea) / K3], 0, dev)

    peaks, peak_src = load_peaks()
    split_info = {"split_pages": s.split_pages, "num_splits": s.num_splits}
    path_name, launches = s.path, s.launches_per_step() * K
    per_workload = None
    if (world == 1 and not args.no_per_workload and isinstance(s, DecodeSession) and s.path == "absorbed"
            and not fp8):
        del s
        torch.cuda.empty_cache()
        per_workload = {}
        for other in W.DECODE_REPORT_WORKLOADS:
            if other != wl.name:
                per_workload[other] = measure_decode_workload(other, dev, stream, flush_l2, args.per_workload_steps,
                                                              peaks)

    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return 0

    t_mem, bound = A.roofline_seconds(kv_list, wl.n_q, peaks["hbm_gbs"], peaks["bf16_tflops"])
    attn_s = attn_ms * 1e-3
    if prefill:
        t_mem, bound = (step_flops + decompress_flops) / (peaks["bf16_tflops"] * 1e12), "tensor"
        achieved, peak, unit = step_flops / attn_s / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    elif bound == "hbm":
        achieved, peak, unit = step_bytes / attn_s / 1e9, peaks["hbm_gbs"], "GB/s"
    else:
        achieved, peak, unit = step_flops / attn_s / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    roofline = {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
                "traffic": None if prefill else profiled_traffic(wl.name), "peak_source": peak_src,
                "kernel": PREFILL_KERNEL if prefill else (DOMINANT_KERNEL_FP8 if fp8 else DOMINANT_KERNEL),
                "algorithmic_bytes": step_bytes,
                "algorithmic_flops": step_flops}

    cpu = None
    cpu_absorbed = None
    if world == 1 and not args.no_cpu_baseline and prefill:
        ntok, secs, desc = oracle_prefill_sample(inp, args.cpu_seconds)
        cpu = {"value": ntok / secs, "unit": "tokens/s", **cpu_cores_info(), "kind": "oracle", "sample": desc}
    elif world == 1 and not args.no_cpu_baseline and layer:
        nseq, secs = oracle_layer_sample(li, args.cpu_seconds)
        cpu = {"value": step_units / (secs / nseq * inp.batch) / 1e9, "unit": "GB/s", **cpu_cores_info(),
               "kind": "oracle",
               "sample": f"{nseq} of {inp.batch} sequences through the fp64 layer ({secs:.1f} s), a step costing "
                         f"{inp.batch} sequences"}
    elif world == 1 and not args.no_cpu_baseline:
        nb, secs, nseq = oracle_sample(inp, args.cpu_seconds)
        cpu = {"value": nb / secs / 1e9, "unit": "GB/s", **cpu_cores_info(), "kind": "oracle",
               "sample": f"{nseq} of {inp.batch} sequences, all 128 heads, fp64 non-absorbed form ({secs:.1f} s)"}
        nb2, secs2, nseq2 = oracle_sample(inp, min(5.0, args.cpu_seconds), absorbed=True)
        cpu_absorbed = {"value": nb2 / secs2 / 1e9, "unit": "GB/s", **cpu_cores_info(), "kind": "oracle",
                        "sample": f"{nseq2} of {inp.batch} sequences, all 128 heads, fp64 absorbed form ({secs2:.1f} s)"}

    line = {
        "metric": METRIC_PREFILL if prefill else (METRIC_LAYER if layer else METRIC),
        "value": total_bytes / (mean_ms * 1e-3) / (1 if prefill else 1e9), "unit": "tokens/s" if prefill else "GB/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": mean_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16" if fp8 else "bf16",
        "cache_dtype": "e4m3 codes, one fp32 scale per token (the MMAs run on f16)" if fp8 else "bf16",
        "data": "synthetic",
        "config": workload_config(wl, inp, world, split_info),
        "us_per_step": mean_ms * 1e3,
        "attn_us": attn_ms * 1e3,
        "attn_tflops": step_flops / attn_s / 1e12,
        "attn_gbs": step_bytes / attn_s / 1e9,
        "path": path_name,
        "decompress_tflops": (decompress_flops / (1e-3 * sum(per_stage[stages.index("decompress")]) / K3) / 1e12
                              if prefill else None),
        "stage_us": {n: 1e3 * sum(v) / K3 for n, v in zip(stages, per_stage)},
        "launch_overlap": ops.mla_get_launch_overlap(),
        "roofline_time_us": t_mem * 1e6,
        "roofline": roofline,
        "decode_attn_with_combine": None if attn_combine_ms is None else {
            "us": attn_combine_ms * 1e3,
            "achieved_gbs": step_bytes / (attn_combine_ms * 1e-3) / 1e9,
            "frac_of_hbm": step_bytes / (attn_combine_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "what": "mla_decode_attn: split attention plus the separate log-sum-exp merge kernel (in the step "
                    "the merge runs fused into the out-projection)"},
        "per_workload": per_workload,
        "cpu_baseline": cpu,
        "cpu_baseline_absorbed": cpu_absorbed,
        "us_per_step_warm_l2": warm_ms * 1e3,
        "us_per_step_graph_warm_l2": None if graph_ms is None else graph_ms * 1e3,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clk,
        "wall_s_timed_region": t_wall,
    }
    print(json.dumps(line))
    return 0


def main(argv=None):
    args = parse_args(argv)
    wl = (W.WORKLOADS.get(args.workload) or W.PREFILL_WORKLOADS.get(args.workload)
          or W.FP8_WORKLOADS.get(args.workload) or W.LAYER_WORKLOADS[args.workload])
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
