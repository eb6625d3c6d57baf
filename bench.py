#!/usr/bin/env python3
"""Attention forward throughput on GB300: TFLOP/s, % of dense bf16 peak, tokens/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step is one attn_fwd call (the whole hot path: tile loads, QK^T, masking,
streaming softmax, PV, epilogue) over one batch of seeded synthetic inputs
already resident in HBM; for the MHA sublayer workload it is one mha_fwd call
(Q/K/V projections, attention, output projection with residual + LayerNorm).
The timed steps are one CUDA graph of those steps (no per-call host overhead;
--no-graph times eager calls instead). Default workload: long-sequence causal
self-attention, bf16, B=4 h=16 n=8192 d=128 (Q, K, V and O are 134 MB each, so
the 402 MB of inputs are larger than the 129 MB L2 and every step streams
them from HBM). The same run also measures the other configurations the metric
is quoted on (long causal d=64 h=32, encoder fp32, decoder causal, cross-attention
with key padding, the MHA sublayer) and reports each under "configs" with the
same fields; --configs none skips them.

FLOPs per step are the defined count 4*B*h*n_q*n_k*d, halved for causal (plus
2*M*N*K for each of the four projections of the MHA sublayer).
Timing: W untimed warm-up steps, then exactly K steps back to back on the
launching stream (one CUDA graph of the K steps) between two CUDA events,
bracketed by a barrier and a device synchronize; max over ranks. A separate pass
times every step on its own (one graph launch and one pair of events per step)
for the median, p10 and p90 of single steps. Inputs that fit in L2 are kept out of it by rotation: the steps cycle
through device copies of every input whose total is three times the L2, so each
step reads inputs last touched long enough ago to come from HBM. A sustained leg
then replays a graph of many
steps back to back for a few seconds while nvidia-smi samples the SM clock,
throttle reasons and power, so the clock under load is on record. The e2e leg
repeats the measurement with the host copies in the timed region: pinned host
Q/K/V -> device, attn_fwd, output -> pinned host. The CPU baseline is the fp64
oracle on a bounded sample of the same workload on this host's cores.

--impl reference times the fp64 CPU oracle itself (the only other
implementation of this method) on the same workload, metric and unit.

With N > 1 (torchrun, one rank per GPU) every rank runs the full workload on
its own GPU with no data-path collective (attention over (batch, head) is
embarrassingly parallel): weak scaling, value = all ranks' FLOPs / max time.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s and % of GB300 BF16 tensor peak (1 GPU); tokens/s"
PE_METRIC = "positional encoding GB/s (HBM-bound elementwise)"
BWD_METRIC = "attention backward TFLOP/s (2.5x the forward's FLOPs; 1 GPU)"


def metric_of(w):
    """(metric, unit) of a workload's bench line."""
    if w.kind == "pe":
        return (PE_METRIC, "GB/s")
    if w.kind == "bwd":
        return (BWD_METRIC, "TFLOP/s")
    return (METRIC, "TFLOP/s")
DEFAULT_WORKLOAD = "long_causal_d128"
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_HBM_GBS = 8000.0
L2_BYTES = 129e6
# Workloads whose inputs fit in L2 rotate over device copies of their inputs whose
# total is at least this much: a step's inputs were last touched after more than
# twice the L2's size of other data, so they come from HBM.
ROTATE_BYTES = 3 * L2_BYTES
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
FP32_FMA_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12  # SMs x fp32 lanes x 2 FLOP x max SM clock
MIN_CLOCK_SAMPLES = 5  # fewer samples inside a window say nothing about its clock
# The other configurations the metric is quoted on, measured in the same run as the
# default workload, each with its own roofline, per-step spread, e2e and clocks.
COMPANION_WORKLOADS = ("long_causal_d64", "enc_self_f32", "dec_causal_bf16", "cross_bf16",
                       "mha_bf16")
PROFILE_DIR = os.path.join(ROOT, "profiles")
# Sources of the persistent attention kernel; a profile summary may name others on
# a "kernel_sources:" line.
KERNEL_SOURCES = ("head_attention_gb300/csrc/attn_tc.cu", "head_attention_gb300/csrc/ptx.cuh",
                  "head_attention_gb300/csrc/row_softmax.cuh")


# ---------------------------------------------------------------- helpers

def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="hattn", choices=["hattn", "reference"])
    ap.add_argument("--cpu-budget-s", type=float, default=15.0,
                    help="CPU seconds of oracle work for the CPU baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="time eager calls instead of CUDA-graph replays of one step")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch size B (smaller cases for profiler "
                         "captures; the default keeps the named workload)")
    ap.add_argument("--configs", default="all", choices=["all", "none"],
                    help="with the default workload, also measure the other configurations "
                         "the metric is quoted on")
    ap.add_argument("--sustained-s", type=float, default=3.0,
                    help="seconds of back-to-back steps in the default workload's sustained leg")
    ap.add_argument("--companion-sustained-s", type=float, default=1.0,
                    help="seconds of the sustained leg of every other configuration")
    ap.add_argument("--no-sustained", action="store_true")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def reduce_max(value: float, world: int) -> float:
    """Max of a float over ranks (identity at world size 1)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(flops_per_rank_step: float, world: int, ms_per_step_max: float) -> float:
    """Whole-job throughput under weak scaling: every rank processes one step's
    FLOPs per step, and the job takes the slowest rank's time."""
    return flops_per_rank_step * world / (ms_per_step_max * 1e-3) / 1e12


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_sha(sources=KERNEL_SOURCES) -> str:
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the workload's attention kernel from a committed ncu
    summary (profiles/<kernel>_<workload>.md), if it was taken on the current source
    of that kernel (the files its "kernel_sources:" line names, by default the
    persistent kernel's); else None."""
    if not os.path.isdir(PROFILE_DIR):
        return None
    for name in sorted(os.listdir(PROFILE_DIR)):
        if not name.endswith(f"_{workload}.md") or name.startswith("launches_"):
            continue
        text = open(os.path.join(PROFILE_DIR, name), encoding="utf-8").read()
        sha = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", text)
        traffic = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
        if not sha or not traffic:
            continue
        srcs = re.search(r"kernel_sources:\s*(.+)", text)
        sources = tuple(srcs.group(1).split()) if srcs else KERNEL_SOURCES
        try:
            current = kernel_source_sha(sources)
        except OSError:
            continue
        if sha.group(1) == current:
            return float(traffic.group(1))
    return None


class ClockSampler:
    """nvidia-smi samples (every 100 ms) of SM clock, power and throttle reasons,
    taken for the whole run; summary(window) reduces the samples of one window."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 100

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.samples = []
        self.proc = None
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, window=None):
        """Median SM clock and power, max clock and the throttle reasons seen, over the
        samples taken inside window = (t0, t1) (wall clock; every sample if None)."""
        rows = list(self.samples)
        if window is not None:
            t0, t1 = window
            rows = [r for r in rows if t0 <= r[0] <= t1 + self.PERIOD_MS * 1e-3]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "samples": 0,
                    "reasons": ["no nvidia-smi samples inside the window"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        mhz, max_mhz, watts = [], [], []
        for _, v in rows:
            try:
                mhz.append(float(v[0]))
                max_mhz.append(float(v[1]))
                watts.append(float(v[2]))
            except (ValueError, IndexError):
                continue
            for name, flag in zip(names, v[4:8]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(mhz) if mhz else None,
                "sm_max_mhz": max(max_mhz) if max_mhz else None,
                "sm_mhz_min": min(mhz) if mhz else None,
                "power_w_median": statistics.median(watts) if watts else None,
                "power_w_max": max(watts) if watts else None,
                "samples": len(mhz), "reasons": sorted(reasons)}


def gpu_uuid(dev_index: int) -> str:
    import torch
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(dev_index).uuid)
    except Exception:
        return str(dev_index)


# ---------------------------------------------------------------- CPU oracle timing

def _head_arrays(inp, w, b, i):
    """fp64 copies of one (batch, head) slice, shaped [1, n, 1, d]."""
    from synth import inputs as synth
    out = []
    for name in ("q", "k", "v"):
        a = inp[name][b:b + 1, :, i:i + 1, :]
        out.append(synth.widen(a.copy(), w.dtype))
    return out


def _rows_flops(w, rows, kv_len):
    """Exact visible-pair FLOPs (4*d per visible (query, key) pair) of these query rows."""
    if w.mask_kind & 1:
        return float(sum(4 * w.d_k * min(t + 1, kv_len) for t in rows))
    return float(4 * w.d_k * kv_len * len(rows))


def oracle_sample_rate(w, inp, budget_s: float, sample_index: int = 0, threads: int = 0,
                       gpu_head=None, errs=None):
    """Times the oracle on whole (batch, head) units of the workload, one after
    another from unit `sample_index` on, until about budget_s seconds of work;
    returns (TFLOP/s, threads, description) counting the exact FLOPs of the
    visible (query, key) pairs the oracle computed. threads = 0: every host core.
    With gpu_head(b, i) (the GPU's output of that unit, fp64 [n_q, d_v]) and a dict
    errs, the largest and the summed absolute difference of the oracle's outputs
    from the GPU's are accumulated there (after the timing of each unit)."""
    import oracle
    threads = threads or os.cpu_count() or 1
    n_units = w.B * w.h
    done, flops, elapsed = [], 0.0, 0.0
    while elapsed < budget_s and len(done) < n_units:
        u = (sample_index + len(done)) % n_units
        b, i = u % w.B, u // w.B
        q, k, v = _head_arrays(inp, w, b, i)
        kv_len = int(inp["key_lens"][b]) if inp.get("key_lens") is not None else w.n_k
        kl = None if inp.get("key_lens") is None else inp["key_lens"][b:b + 1]
        t0 = time.perf_counter()
        ref = oracle.attn(q, k, v, w.scale, w.mask_kind, kl, nthreads=threads)
        elapsed += time.perf_counter() - t0
        flops += _rows_flops(w, range(w.n_q), kv_len)
        done.append((b, i))
        if gpu_head is not None and errs is not None:
            import numpy as np
            d = np.abs(gpu_head(b, i) - ref[0, :, 0, :])
            errs["max"] = max(errs.get("max", 0.0), float(d.max()))
            errs["sum"] = errs.get("sum", 0.0) + float(d.sum())
            errs["n"] = errs.get("n", 0) + d.size
    desc = (f"{len(done)} of {n_units} (batch, head) units, all {w.n_q} query rows each; "
            f"{flops / 1e9:.2f} GFLOP of visible (query, key) pairs in {elapsed:.2f} s")
    return flops / elapsed / 1e12, threads, desc


def oracle_mha_sample_rate(w, inp, budget_s: float, sample_index: int = 0):
    """Times the oracle's MHA sublayer on whole batch elements (all their query
    rows, their K/V projections included), one after another, until about
    budget_s seconds of work; returns (TFLOP/s, threads, description) counting
    the FLOPs the oracle performed."""
    import oracle
    from synth import inputs as synth
    threads = os.cpu_count() or 1
    wd = {n: synth.widen(inp[n], "bf16") for n in ("wq", "wk", "wv", "wo")}
    g64, b64 = inp["gamma"].astype("float64"), inp["beta"].astype("float64")
    hdk, hdv = w.h * w.d_k, w.h * w.d_v
    per_elem = (2.0 * w.n_k * w.d_model * (hdk + hdv)
                + w.n_q * (2.0 * w.d_model * hdk + 4.0 * w.n_k * w.h * w.d_k + 2.0 * hdv * w.d_model))
    done, elapsed = 0, 0.0
    while elapsed < budget_s and done < w.B:
        b = (sample_index + done) % w.B
        x_q = synth.widen(inp["x_q"][b:b + 1].copy(), "bf16")
        x_kv = synth.widen(inp["x_kv"][b:b + 1].copy(), "bf16")
        kl = None if inp["key_lens"] is None else inp["key_lens"][b:b + 1]
        t0 = time.perf_counter()
        oracle.mha(x_q, x_kv, wd["wq"], wd["wk"], wd["wv"], wd["wo"], g64, b64, inp["eps"], w.h,
                   w.mask_kind, kl, nthreads=threads)
        elapsed += time.perf_counter() - t0
        done += 1
    flops = per_elem * done
    desc = (f"{done} of {w.B} batch elements, whole sublayer (projections, attention, "
            f"output projection, LayerNorm); {flops / 1e9:.2f} GFLOP in {elapsed:.2f} s")
    return flops / elapsed / 1e12, threads, desc


def oracle_pe_sample_rate(w, inp, budget_s: float, sample_index: int = 0):
    """Times the oracle's positional encoding on whole batch elements until about
    budget_s seconds of work; returns (GB/s of algorithmic bytes: one read of the
    embeddings and one write of the result, at the kernel's element size,
    threads, description)."""
    import oracle
    from synth import inputs as synth
    done, elapsed, nbytes = 0, 0.0, 0.0
    while elapsed < budget_s and done < w.B:
        b = (sample_index + done) % w.B
        emb = synth.widen(inp["emb"][b:b + 1].copy(), "bf16")
        t0 = time.perf_counter()
        oracle.pos_encoding(1, w.n_q, w.d_model, emb, w.d_model ** 0.5)
        elapsed += time.perf_counter() - t0
        nbytes += 2.0 * w.n_q * w.d_model * 2
        done += 1
    desc = (f"{done} of {w.B} batch elements ({w.n_q} x {w.d_model} each), single-threaded; "
            f"{nbytes / 1e6:.1f} MB in {elapsed:.2f} s")
    return nbytes / elapsed / 1e9, 1, desc


def oracle_layer_sample_rate(w, inp, budget_s: float, sample_index: int = 0):
    """Times the oracle's encoder / decoder layer (its sublayers composed, each
    output rounded to bf16 as the API passes it on) on whole batch elements until
    about budget_s seconds of work; returns (TFLOP/s of the layer's defined FLOPs,
    threads, description)."""
    import oracle
    from synth import inputs as synth
    threads = os.cpu_count() or 1
    wd = lambda a: synth.widen(a, "bf16")
    rb = lambda a: synth.bf16_bits_to_f64(synth.round_to_bf16_bits(a))

    def mha(xq, xkv, m, mask, kl):
        return oracle.mha(xq, xkv, wd(m["wq"]), wd(m["wk"]), wd(m["wv"]), wd(m["wo"]),
                          m["gamma"].astype("float64"), m["beta"].astype("float64"), inp["eps"],
                          w.h, mask, kl, nthreads=threads)

    f = inp["ffn"]
    fw = (wd(f["w1"]), f["b1"].astype("float64"), wd(f["w2"]), f["b2"].astype("float64"),
          f["gamma"], f["beta"], f["eps"])
    per_elem = w.layer_flops() / w.B
    done, elapsed = 0, 0.0
    while elapsed < budget_s and done < w.B:
        b = (sample_index + done) % w.B
        kl = None if inp["key_lens"] is None else inp["key_lens"][b:b + 1]
        x = wd(inp["x"][b:b + 1].copy())
        t0 = time.perf_counter()
        if w.kind == "encoder":
            y1 = rb(mha(x, x, inp["self_attn"], 2 if kl is not None else 0, kl))
        else:
            y0 = rb(mha(x, x, inp["self_attn"], 1, None))
            y1 = rb(mha(y0, wd(inp["memory"][b:b + 1].copy()), inp["cross_attn"],
                        2 if kl is not None else 0, kl))
        oracle.ffn(y1, *fw, nthreads=threads)
        elapsed += time.perf_counter() - t0
        done += 1
    desc = (f"{done} of {w.B} batch elements (the whole layer for each); "
            f"{done * per_elem / 1e9:.2f} GFLOP in {elapsed:.2f} s")
    return done * per_elem / elapsed / 1e12, threads, desc


def oracle_bwd_sample_rate(w, inp, budget_s: float, sample_index: int = 0):
    """Times the oracle's attention backward on whole (batch, head) units until about
    budget_s seconds of work; returns (TFLOP/s at the backward's defined count of 2.5x
    the forward's visible-pair FLOPs, threads, description). The oracle runs one thread."""
    import oracle
    from synth import inputs as synth
    n_units = w.B * w.h
    done, flops, elapsed = 0, 0.0, 0.0
    while elapsed < budget_s and done < n_units:
        u = (sample_index + done) % n_units
        b, i = u % w.B, u // w.B
        q, k, v = _head_arrays(inp, w, b, i)
        g = synth.widen(inp["dout"][b:b + 1, :, i:i + 1].copy(), w.dtype)
        kl = None if inp.get("key_lens") is None else inp["key_lens"][b:b + 1]
        kv_len = int(kl[0]) if kl is not None else w.n_k
        t0 = time.perf_counter()
        oracle.attn_bwd(q, k, v, g, w.scale, w.mask_kind, kl)
        elapsed += time.perf_counter() - t0
        flops += 2.5 * _rows_flops(w, range(w.n_q), kv_len)
        done += 1
    desc = (f"{done} of {n_units} (batch, head) units, single-threaded; {flops / 1e9:.2f} GFLOP "
            f"(2.5x the forward's visible pairs) in {elapsed:.2f} s")
    return flops / elapsed / 1e12, 1, desc


def pe_inputs(w):
    from synth import inputs as synth
    return {"emb": synth.round_to_bf16_bits(synth.draw_normal(w.seed, 0, (w.B, w.n_q, w.d_model)))}


def workload_inputs(w):
    from synth import inputs as synth
    if w.kind == "pe":
        return pe_inputs(w)
    if w.kind in ("encoder", "decoder"):
        return synth.layer_inputs(w)
    if w.kind == "bwd":
        return synth.attn_bwd_inputs(w)
    return synth.mha_inputs(w) if w.kind == "mha" else synth.attn_inputs(w)


def load_workload(args):
    from synth import inputs as synth
    w = synth.workload(args.workload)
    if args.batch > 0:
        w = w.with_(B=args.batch)
    return w


def sample_rate(w, inp, budget_s: float, sample_index: int = 0):
    if w.kind == "pe":
        return oracle_pe_sample_rate(w, inp, budget_s, sample_index)
    if w.kind in ("encoder", "decoder"):
        return oracle_layer_sample_rate(w, inp, budget_s, sample_index)
    if w.kind == "bwd":
        return oracle_bwd_sample_rate(w, inp, budget_s, sample_index)
    if w.is_mha:
        return oracle_mha_sample_rate(w, inp, budget_s, sample_index)
    return oracle_sample_rate(w, inp, budget_s, sample_index)


# ---------------------------------------------------------------- GPU arm

def _device_array(a, dtype):
    import numpy as np
    import torch
    if dtype == "f32":
        return torch.from_numpy(a).cuda()
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def _setup_attention(w, inp):
    """Device tensors and a step closure for one attn_fwd call."""
    import torch

    import head_attention_gb300 as hattn
    q, k, v = (_device_array(inp[n], w.dtype) for n in ("q", "k", "v"))
    kl = None if inp["key_lens"] is None else torch.from_numpy(inp["key_lens"]).cuda()
    out = torch.empty((w.B, w.n_q, w.h, w.d_v), dtype=q.dtype, device="cuda")

    def bind(q, k, v, out):
        def step():
            hattn.attn_fwd(q, k, v, out=out, scale=w.scale, mask_kind=w.mask_kind, key_lens=kl)
        return step

    def rebind():
        """The same step on a second set of device buffers (for the pipelined e2e leg)."""
        q2, k2, v2, o2 = (torch.empty_like(t) for t in (q, k, v, out))
        return {"q": (inp["q"], q2), "k": (inp["k"], k2), "v": (inp["v"], v2)}, o2, bind(q2, k2, v2, o2)

    def clone():
        """The same step on device copies of every input (and a new output)."""
        kl_c = None if kl is None else kl.clone()
        q2, k2, v2 = (t.clone() for t in (q, k, v))
        o2 = torch.empty_like(out)

        def step():
            hattn.attn_fwd(q2, k2, v2, out=o2, scale=w.scale, mask_kind=w.mask_kind, key_lens=kl_c)
        return step

    host = {"inputs": {"q": (inp["q"], q), "k": (inp["k"], k), "v": (inp["v"], v)},
            "output": out, "rebind": rebind, "clone": clone}
    return bind(q, k, v, out), host, 1


def _setup_mha(w, inp):
    """Device tensors, workspace and a step closure for one mha_fwd call."""
    import torch

    import head_attention_gb300 as hattn
    dev = {n: _device_array(inp[n], "bf16") for n in ("x_q", "x_kv", "wq", "wk", "wv", "wo")}
    gamma = torch.from_numpy(inp["gamma"]).cuda()
    beta = torch.from_numpy(inp["beta"]).cuda()
    kl = None if inp["key_lens"] is None else torch.from_numpy(inp["key_lens"]).cuda()
    y = torch.empty_like(dev["x_q"])
    ws = torch.empty(hattn.mha_workspace_bytes(hattn.HATTN_BF16, w.B, w.n_q, w.n_k, w.d_model, w.h,
                                               w.d_k, w.d_v), dtype=torch.uint8, device="cuda")

    def make(dev, gamma, beta, kl, y, ws):
        def step():
            hattn.mha_fwd(dev["x_q"], dev["x_kv"], dev["wq"], dev["wk"], dev["wv"], dev["wo"],
                          gamma, beta, inp["eps"], w.h, y=y, mask_kind=w.mask_kind, key_lens=kl,
                          workspace=ws)
        return step

    def clone():
        """The same step on device copies of every input (and new output and workspace)."""
        return make({n: t.clone() for n, t in dev.items()}, gamma.clone(), beta.clone(),
                    None if kl is None else kl.clone(), torch.empty_like(y), torch.empty_like(ws))

    host = {"inputs": {"x_q": (inp["x_q"], dev["x_q"])}, "output": y, "clone": clone}
    return make(dev, gamma, beta, kl, y, ws), host, 3


def _setup_decode(w, inp):
    """Device tensors, workspace and a step closure for one attn_decode_fwd call."""
    import torch

    import head_attention_gb300 as hattn
    q, k, v = (_device_array(inp[n], "bf16") for n in ("q", "k", "v"))
    kl = torch.from_numpy(inp["key_lens"]).cuda()
    out = torch.empty_like(q)
    ws = torch.empty(hattn.attn_decode_workspace_bytes(w.B, w.h, w.n_k, w.d_k), dtype=torch.uint8,
                     device="cuda")

    def step():
        hattn.attn_decode_fwd(q, k, v, kl, out=out, scale=w.scale, workspace=ws)

    host = {"inputs": {"q": (inp["q"], q)}, "output": out}
    return step, host, 2


def _setup_pe(w, inp):
    """Embeddings on the device and a step closure for one pos_encoding_fwd call."""
    import torch

    import head_attention_gb300 as hattn
    emb = _device_array(inp["emb"], "bf16")
    out = torch.empty_like(emb)

    def step():
        hattn.pos_encoding_fwd(out, emb=emb, emb_scale=w.d_model ** 0.5)

    host = {"inputs": {"emb": (inp["emb"], emb)}, "output": out}
    return step, host, 1


def _setup_layer(w, inp):
    """Device tensors, workspace and a step closure for one encoder_layer_fwd /
    decoder_layer_fwd call (five or eight kernel launches)."""
    import torch

    import head_attention_gb300 as hattn
    dev = lambda a: _device_array(a, "bf16")
    f32 = lambda a: torch.from_numpy(a).cuda()

    def mha_w(m):
        return {**{k: dev(m[k]) for k in ("wq", "wk", "wv", "wo")},
                "gamma": f32(m["gamma"]), "beta": f32(m["beta"])}

    f = inp["ffn"]
    ffn = {"w1": dev(f["w1"]), "w2": dev(f["w2"]), "b1": f32(f["b1"]), "b2": f32(f["b2"]),
           "gamma": f32(f["gamma"]), "beta": f32(f["beta"])}
    x = dev(inp["x"])
    y = torch.empty_like(x)
    kl = None if inp["key_lens"] is None else f32(inp["key_lens"])
    host_inputs = {"x": (inp["x"], x)}
    cl = lambda d: {n: t.clone() for n, t in d.items()}
    if w.kind == "encoder":
        sa = mha_w(inp["self_attn"])
        ws = torch.empty(hattn.encoder_layer_workspace_bytes(hattn.HATTN_BF16, w.B, w.n_q,
                                                             w.d_model, w.h, w.d_k, w.d_ff),
                         dtype=torch.uint8, device="cuda")

        def make(x, sa, ffn, kl, y, ws):
            def step():
                hattn.encoder_layer_fwd(x, sa, ffn, inp["eps"], w.h, key_lens=kl, y=y, workspace=ws)
            return step

        def clone():
            return make(x.clone(), cl(sa), cl(ffn), None if kl is None else kl.clone(),
                        torch.empty_like(y), torch.empty_like(ws))
        step = make(x, sa, ffn, kl, y, ws)
        launches = 5
    else:
        sa, ca = mha_w(inp["self_attn"]), mha_w(inp["cross_attn"])
        mem = dev(inp["memory"])
        host_inputs["memory"] = (inp["memory"], mem)
        ws = torch.empty(hattn.decoder_layer_workspace_bytes(hattn.HATTN_BF16, w.B, w.n_q, w.n_k,
                                                             w.d_model, w.h, w.d_k, w.d_ff),
                         dtype=torch.uint8, device="cuda")

        def make(x, mem, sa, ca, ffn, kl, y, ws):
            def step():
                hattn.decoder_layer_fwd(x, mem, sa, ca, ffn, inp["eps"], w.h, src_lens=kl, y=y,
                                        workspace=ws)
            return step

        def clone():
            return make(x.clone(), mem.clone(), cl(sa), cl(ca), cl(ffn),
                        None if kl is None else kl.clone(), torch.empty_like(y), torch.empty_like(ws))
        step = make(x, mem, sa, ca, ffn, kl, y, ws)
        launches = 8
    return step, {"inputs": host_inputs, "output": y, "clone": clone}, launches


def _setup_bwd(w, inp):
    """Device tensors, the forward's output and log-sum-exp, workspace and a step closure
    for one attn_bwd call (three kernel launches)."""
    import torch

    import head_attention_gb300 as hattn
    q, k, v, g = (_device_array(inp[n], w.dtype) for n in ("q", "k", "v", "dout"))
    kl = None if inp["key_lens"] is None else torch.from_numpy(inp["key_lens"]).cuda()
    out, lse = hattn.attn_fwd_lse(q, k, v, scale=w.scale, mask_kind=w.mask_kind, key_lens=kl)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(hattn.attn_bwd_workspace_bytes(w.B, w.h, w.n_q), dtype=torch.uint8,
                     device="cuda")

    def make(q, k, v, out, g, lse, kl, dq, dk, dv, ws):
        def step():
            hattn.attn_bwd(q, k, v, out, g, lse, scale=w.scale, mask_kind=w.mask_kind, key_lens=kl,
                           dq=dq, dk=dk, dv=dv, workspace=ws)
        return step

    def clone():
        """The same step on device copies of every input (new gradients and workspace)."""
        return make(*(t.clone() for t in (q, k, v, out, g, lse)), None if kl is None else kl.clone(),
                    *(torch.empty_like(t) for t in (dq, dk, dv, ws)))

    host = {"inputs": {"dout": (inp["dout"], g)}, "output": dq, "clone": clone}
    return make(q, k, v, out, g, lse, kl, dq, dk, dv, ws), host, 3


def io_bytes(w, inp):
    """(resident input bytes, algorithmic bytes) of one step. Resident bytes are every
    input tensor as it sits in HBM (they decide whether the step fits in L2);
    algorithmic bytes are the inputs the method must read once plus the output written
    once. With key padding only the first key_lens[b] rows of K and V are read."""
    esize = 4 if w.dtype == "f32" else 2
    if w.kind == "mha":
        bytes_in = (2 * w.B * w.n_q * w.d_model + 4 * w.d_model * w.h * w.d_k) * esize
        bytes_alg = bytes_in + w.B * w.n_q * w.d_model * esize
    elif w.kind in ("encoder", "decoder"):
        n_mha = 1 if w.kind == "encoder" else 2
        weights = n_mha * 4 * w.d_model * w.h * w.d_k + 2 * w.d_model * w.d_ff
        acts = w.B * w.n_q * w.d_model + (w.B * w.n_k * w.d_model if w.kind == "decoder" else 0)
        bytes_in = (acts + weights) * esize
        bytes_alg = bytes_in + w.B * w.n_q * w.d_model * esize
    elif w.kind == "bwd":
        qkv = w.B * (w.n_q * w.h * w.d_k + w.n_k * w.h * (w.d_k + w.d_v))
        bytes_in = (qkv + 2 * w.B * w.n_q * w.h * w.d_v) * esize + 4 * w.B * w.h * w.n_q
        bytes_alg = bytes_in + qkv * esize
    elif w.kind == "decode":
        bytes_in = (w.B * w.n_k * w.h * (w.d_k + w.d_v) + w.B * w.h * w.d_k) * esize
        bytes_alg = ((float(inp["key_lens"].sum()) * w.h * (w.d_k + w.d_v) + w.B * w.h * w.d_k)
                     * esize + w.B * w.h * w.d_v * esize)
    elif w.kind == "pe":
        bytes_in = w.B * w.n_q * w.d_model * esize
        bytes_alg = 2 * bytes_in
    else:
        q_o = w.B * w.n_q * w.h * (w.d_k + w.d_v) * esize
        bytes_in = (w.B * w.n_q * w.h * w.d_k + w.B * w.n_k * w.h * (w.d_k + w.d_v)) * esize
        kv_rows = w.B * w.n_k
        if inp is not None and inp.get("key_lens") is not None:
            kv_rows = int(inp["key_lens"].astype("int64").sum())
        bytes_alg = q_o + kv_rows * w.h * (w.d_k + w.d_v) * esize
    return bytes_in, bytes_alg


def visible_pair_flops(w, inp):
    """4*d FLOPs per visible (query, key) pair: the count the method performs (the
    metric's defined count differs only under key padding, where it stays dense)."""
    if w.kind != "attn":
        return None
    if inp is not None and inp.get("key_lens") is not None and w.mask_kind & 2:
        lens = inp["key_lens"].astype("float64")
        if w.mask_kind & 1:
            n = w.n_q
            pairs = sum(min(L, n) * (min(L, n) + 1) / 2 for L in lens)
        else:
            pairs = float(lens.sum()) * w.n_q
        return 4.0 * w.h * w.d_k * pairs
    if w.mask_kind & 1:
        return 4.0 * w.B * w.h * w.d_k * w.n_q * (w.n_q + 1) / 2
    return 4.0 * w.B * w.h * w.d_k * w.n_q * w.n_k


def setup_workload(w):
    """(inputs, step closure, host buffers for the e2e leg, launches per step,
    defined FLOPs per step) of one workload, its inputs already on the device."""
    from synth import inputs as synth
    if w.kind == "mha":
        inp = synth.mha_inputs(w)
        step, host, launches = _setup_mha(w, inp)
        flops = w.attn_flops() + w.proj_flops()
    elif w.kind == "decode":
        inp = synth.attn_inputs(w)
        step, host, launches = _setup_decode(w, inp)
        flops = 4.0 * w.h * w.d_k * float(inp["key_lens"].sum())  # visible (query, key) pairs
    elif w.kind == "bwd":
        inp = synth.attn_bwd_inputs(w)
        step, host, launches = _setup_bwd(w, inp)
        flops = 2.5 * w.attn_flops()  # five n_q x n_k x d contractions against the forward's two
    elif w.kind in ("encoder", "decoder"):
        inp = synth.layer_inputs(w)
        step, host, launches = _setup_layer(w, inp)
        flops = w.layer_flops()
    elif w.kind == "pe":
        inp = pe_inputs(w)
        step, host, launches = _setup_pe(w, inp)
        flops = 0.0
    else:
        inp = synth.attn_inputs(w)
        step, host, launches = _setup_attention(w, inp)
        flops = w.attn_flops()
    return inp, step, host, launches, flops


def percentiles(xs):
    """(p10, median, p90) of a list of per-step times, by linear interpolation."""
    s = sorted(xs)
    if not s:
        return None, None, None

    def q(f):
        pos = f * (len(s) - 1)
        lo = int(math.floor(pos))
        hi = min(lo + 1, len(s) - 1)
        return s[lo] + (s[hi] - s[lo]) * (pos - lo)
    return q(0.1), q(0.5), q(0.9)


def time_steps(run, stream, steps):
    """Device time of exactly `steps` consecutive steps between two CUDA events on the
    launching stream: step i runs run[i % len(run)] (input copies in rotation, or
    one). Returns (total ms, wall-clock window)."""
    import torch
    torch.cuda.synchronize()
    t0 = time.time()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(steps):
        run[i % len(run)]()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b), (t0, time.time())


def step_latencies(run, stream, steps):
    """Per-step device times (ms) of `steps` steps, each between its own pair of CUDA
    events (so each includes the gap its own launch leaves): the spread of single
    steps, next to the throughput of the back-to-back timed steps."""
    import torch
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    torch.cuda.synchronize()
    ev[0].record(stream)
    for i in range(steps):
        run[i % len(run)]()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    return [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]


def sustained_leg(fns, stream, flops, bytes_alg, seconds, peaks, hbm_bound, l2_note):
    """Back-to-back replays of a CUDA graph of many steps (cycling through the input
    copies) for about `seconds`, with the SM clock and board power sampled
    throughout: the throughput a long run sees and the clock it ran at (time x median
    MHz compares runs at different clocks)."""
    import torch
    step_ms = _probe_step_ms(fns, stream)
    per_graph = max(len(fns), min(4096, int(math.ceil(50.0 / max(step_ms, 1e-3)))))
    per_graph -= per_graph % len(fns)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(per_graph):
            fns[i % len(fns)]()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    graph.replay()
    end.record(stream)
    torch.cuda.synchronize()
    replay_ms = start.elapsed_time(end)
    replays = max(2, int(math.ceil(seconds * 1e3 / max(replay_ms, 1e-3))))
    torch.cuda.synchronize()
    t0 = time.time()
    start.record(stream)
    for _ in range(replays):
        graph.replay()
    end.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    del graph
    steps = replays * per_graph
    ms = start.elapsed_time(end) / steps
    rec = {"seconds": round(steps * ms * 1e-3, 3), "steps": steps, "ms_per_step": round(ms, 5),
           "_clock_window": (t0, t1), "l2": l2_note}
    if hbm_bound:
        gbs = bytes_alg / (ms * 1e-3) / 1e9
        rec.update({"gbs_at_algorithmic_bytes": round(gbs, 1),
                    "frac_of_measured_hbm": round(gbs / peaks["hbm_gbs"], 4)})
    if flops:
        tf = flops / (ms * 1e-3) / 1e12
        rec.update({"value": round(tf, 2), "unit": "TFLOP/s",
                    "frac_of_sustained_bf16": round(tf / peaks["bf16_tflops_sustained"], 4),
                    "bf16_tflops_sustained": peaks["bf16_tflops_sustained"]})
    return rec


def _probe_step_ms(fns, stream):
    """A rough per-step time (a few eager steps) to size the sustained graph."""
    import torch
    fns[0]()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(5):
        fns[i % len(fns)]()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / 5


def roofline_of(w, kernel, flops, alg_flops, bytes_alg, step_ms, peaks, peak_src):
    """The roofline record of one workload's step: the bound is the larger of the two
    roofline times (FLOPs at the tensor (bf16) or fp32 FMA peak, algorithmic bytes at
    the measured HBM bandwidth); achieved and frac are taken against that bound."""
    alg = alg_flops if alg_flops is not None else flops
    gbs = bytes_alg / (step_ms * 1e-3) / 1e9
    tf = alg / (step_ms * 1e-3) / 1e12
    tensor_path = w.dtype == "bf16" and w.kind != "pe" and (
        w.kind != "bwd" or (w.d_k == w.d_v and w.d_k in (64, 128)))
    if w.kind in ("decode", "pe") or alg == 0:
        bound = "hbm"
    else:
        flop_peak = peaks["bf16_tflops"] if tensor_path else FP32_FMA_TFLOPS
        t_flop = alg / (flop_peak * 1e12)
        t_hbm = bytes_alg / (peaks["hbm_gbs"] * 1e9)
        bound = ("tensor" if tensor_path else "alu") if t_flop >= t_hbm else "hbm"
    rec = {"kernel": kernel, "bound": bound}
    if bound == "hbm":
        rec.update({"achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": round(gbs / peaks["hbm_gbs"], 4),
                    "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)",
                    "frac_of_nominal_8000": round(gbs / NOMINAL_HBM_GBS, 4)})
    elif bound == "tensor":
        rec.update({"achieved": round(tf, 2), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": round(tf / peaks["bf16_tflops"], 4),
                    "peak_source": f"{peak_src} (burst, MEASURED_PEAKS.json bf16_tflops)",
                    "frac_of_sustained": round(tf / peaks["bf16_tflops_sustained"], 4),
                    "frac_of_nominal_2250": round(tf / NOMINAL_BF16_TFLOPS, 4)})
    else:
        rec.update({"achieved": round(tf, 3), "peak": round(FP32_FMA_TFLOPS, 1), "unit": "TFLOP/s",
                    "frac": round(tf / FP32_FMA_TFLOPS, 4),
                    "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 FLOP x 2070 MHz (fp32 FMA)"})
    rec.update({"algorithmic_flops_per_launch": alg, "defined_flops_per_launch": flops,
                "algorithmic_bytes_per_launch": bytes_alg,
                "hbm_gbs_at_algorithmic_bytes": round(gbs, 1),
                "hbm_frac_at_algorithmic_bytes": round(gbs / peaks["hbm_gbs"], 4),
                "traffic": profiled_traffic(w.name)})
    if bound != "tensor" and tensor_path and alg:
        rec["frac_of_bf16_tensor_peak"] = round(tf / peaks["bf16_tflops"], 4)
    return rec


def kernel_name(w):
    tc_attn = w.dtype == "bf16" and w.d_k == w.d_v and w.d_k in (64, 128)
    short = tc_attn and w.n_q <= 128 and w.n_k <= (256 if w.d_k == 64 else 128)
    attn = (f"attn_short_kernel<{w.d_k}, {1 if w.n_k <= 128 else 2}>" if short else
            f"attn_tc_kernel<{w.d_k}>" if tc_attn else "attn_simt_kernel")
    return {"mha": "mha sublayer: proj_gemm + attn_tc_kernel + outproj_ln (one step)",
            "encoder": "encoder layer: MHA (proj_gemm, attn_tc_kernel, outproj_ln) + FFN "
                       "(proj_gemm with bias+ReLU, outproj_ln with bias) (one step)",
            "decoder": "decoder layer: two MHA sublayers + FFN (eight launches, one step)",
            "bwd": ("attention backward on tensor cores: row_dot + grads_tc (one step)" if tc_attn
                    else "attention backward on CUDA cores: row_dot + key_grads + query_grads"),
            "decode": f"decode_split_kernel<{w.d_k}> + decode_combine_kernel (one step)",
            "pe": "pos_encoding_kernel"}.get(w.kind, attn)


def measure(args, w, world, peaks, peak_src, sustained_s, with_e2e=True):
    """Everything the bench line reports about one workload except the CPU baseline:
    defined-FLOP throughput over exactly args.steps timed steps (one CUDA graph of
    those steps, or eager calls with --no-graph), per-step median / p10 / p90, the
    roofline of the step, a sustained leg with its clock record, and the e2e leg."""
    import torch

    import head_attention_gb300 as hattn
    inp, step, host, launches_per_step, flops = setup_workload(w)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if hattn.check_device_error(stream) != 0:
        raise RuntimeError(f"{w.name}: device error during warm-up")
    # Inputs that fit in the 129 MB L2 would be served from it after the first step:
    # then the steps rotate over device copies of every input, together more than
    # ROTATE_BYTES, so each step's inputs come from HBM.
    bytes_in, bytes_alg = io_bytes(w, inp)
    copies = 1 if bytes_in > L2_BYTES else int(math.ceil(ROTATE_BYTES / bytes_in))
    fns = [step] + [host["clone"]() for _ in range(copies - 1)]
    for fn in fns[1:]:
        fn()
    torch.cuda.synchronize()
    # The timed steps: one CUDA graph of exactly args.steps steps (input copies in
    # rotation), so no per-launch host or graph overhead sits between steps; the
    # per-step spread comes from a second pass with one graph launch per step.
    graphs, timed, timed_warm = [], None, None
    run = fns
    if not args.no_graph:
        for fn in fns:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            g.replay()
            graphs.append(g)
        timed = torch.cuda.CUDAGraph()
        with torch.cuda.graph(timed):
            for i in range(args.steps):
                fns[i % copies]()
        timed.replay()
        if copies > 1:
            # The same number of steps on one copy of the inputs, in one graph as well:
            # the hot-L2 time beside the cold one, with the same launch structure.
            timed_warm = torch.cuda.CUDAGraph()
            with torch.cuda.graph(timed_warm):
                for i in range(args.steps):
                    fns[0]()
            timed_warm.replay()
        torch.cuda.synchronize()
        run = [g.replay for g in graphs]
    l2_note = (f"inputs {bytes_in / 1e6:.0f} MB > 129 MB L2: streamed from HBM every step"
               if copies == 1 else
               f"inputs {bytes_in / 1e6:.2f} MB fit in L2: steps run back to back over {copies} "
               f"device copies of every input ({copies * bytes_in / 1e6:.0f} MB, "
               f"{copies * bytes_in / L2_BYTES:.1f}x the L2), so a step's inputs were last "
               f"touched {copies - 1} steps earlier and come from HBM")
    per_step = step_latencies(run, stream, args.steps)
    barrier(world)
    ms_local, window = time_steps([timed.replay] if timed is not None else run, stream,
                                  1 if timed is not None else args.steps)
    barrier(world)
    if hattn.check_device_error(stream) != 0:
        raise RuntimeError(f"{w.name}: device error during the timed region")
    ms_step = reduce_max(ms_local, world) / args.steps
    step_ms_local = ms_local / args.steps
    warm_ms = None
    if copies > 1:
        # The same steps on one copy of the inputs, which then stay in L2: the hot-L2
        # time next to the cold one.
        warm_total, _ = time_steps([timed_warm.replay] if timed_warm is not None else fns[:1], stream,
                                   1 if timed_warm is not None else args.steps)
        warm_ms = warm_total / args.steps
    hbm_bound_kind = w.kind in ("decode", "pe")
    alg_flops = visible_pair_flops(w, inp)
    p10, p50, p90 = percentiles(per_step)
    rec = {
        "workload": w.name,
        "description": w.description,
        "value": round(aggregate_tflops(flops, world, ms_step), 2) if w.kind != "pe"
        else round(bytes_alg * world / (ms_step * 1e-3) / 1e9, 1),
        "unit": metric_of(w)[1],
        "ms_per_step": round(ms_step, 5),
        "step_ms": {"p10": round(p10, 5), "median": round(p50, 5), "p90": round(p90, 5),
                    "min": round(min(per_step), 5), "max": round(max(per_step), 5),
                    "how": "each step its own graph launch between its own pair of events "
                           "(launch gap included); ms_per_step is the back-to-back time"},
        "tokens_per_s": round(w.tokens() * world / (ms_step * 1e-3), 1),
        "dtype": w.dtype,
        "l2": l2_note,
        "input_copies": copies,
        "warm_l2_ms_per_step": None if warm_ms is None else round(warm_ms, 5),
        "roofline": roofline_of(w, kernel_name(w), flops, alg_flops, bytes_alg, step_ms_local,
                                peaks, peak_src),
        "_clock_window": window,
        "gpu_launches": args.steps * launches_per_step,
    }
    if w.kind != "pe":
        rec["pct_of_measured_bf16_peak"] = round(100 * flops / (ms_step * 1e-3) / 1e12
                                                 / peaks["bf16_tflops"], 2)
        rec["pct_of_nominal_bf16_peak"] = round(100 * flops / (ms_step * 1e-3) / 1e12
                                                / NOMINAL_BF16_TFLOPS, 2)
    del graphs, run, timed
    if sustained_s > 0:
        rec["sustained"] = sustained_leg(fns, stream, flops if w.kind != "pe" else 0.0, bytes_alg,
                                         sustained_s, peaks,
                                         hbm_bound_kind or rec["roofline"]["bound"] == "hbm",
                                         l2_note)
        rec["gpu_launches_sustained"] = rec["sustained"]["steps"] * launches_per_step
    if with_e2e and w.kind != "pe":
        rec["e2e"] = e2e_leg(args, w, host, step, flops, world)
        rec["gpu_launches"] += rec["e2e"].pop("launches") * launches_per_step
    rec["_inp"] = inp
    rec["_out"] = host["output"]
    return rec


def finalize_clocks(rec, sampler, steps):
    """Fills in a workload record's clock records once sampling has stopped: the
    sustained leg's own, and the one the line reports for the timed steps. That is
    the samples inside the timed steps when there are at least MIN_CLOCK_SAMPLES of
    them, else (a timed region shorter than a few sampling periods) the sustained
    leg's, which runs right after the timed steps, with the source said."""
    timed = sampler.summary(rec.pop("_clock_window"))
    sus = rec.get("sustained")
    if sus is not None:
        sus["clocks"] = sampler.summary(sus.pop("_clock_window"))
        if sus["clocks"].get("sm_mhz"):
            sus["ms_x_median_mhz"] = round(sus["ms_per_step"] * sus["clocks"]["sm_mhz"], 2)
    if timed.get("samples", 0) >= MIN_CLOCK_SAMPLES or sus is None:
        rec["clocks"] = dict(timed, source="timed steps")
        return
    rec["clocks"] = dict(
        sus["clocks"],
        source=(f"sustained leg ({sus['seconds']} s of back-to-back steps right after the "
                f"timed steps); the {steps} timed steps ({rec['ms_per_step'] * steps:.3g} ms "
                f"of device time) held {timed.get('samples', 0)} samples"),
        timed_region_samples=timed.get("samples", 0),
        timed_region_reasons=timed.get("reasons", []))


def torch_int16():
    import torch
    return torch.int16


def config_of(w, world):
    """The workload as the bench line names it (the same for both arms)."""
    cfg = {"workload": w.name, "description": w.description, "B": w.B, "h": w.h,
           "n_q": w.n_q, "n_k": w.n_k, "d": w.d_k,
           "mask": {0: "none", 1: "causal", 2: "key_padding", 3: "causal+key_padding"}[w.mask_kind],
           "parallelism": f"replicas x{world} (independent (batch, head) work per GPU)"}
    if w.is_mha or w.kind in ("encoder", "decoder"):
        cfg["d_model"] = w.d_model
    if w.kind in ("encoder", "decoder"):
        cfg["d_ff"] = w.d_ff
    return cfg


def run_gpu(args, rank, world, local):
    import torch

    import head_attention_gb300 as hattn

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    hattn.build()
    hattn.load()
    peaks, peak_src = load_peaks()
    w = load_workload(args)
    companions = []
    if args.configs == "all" and w.name == DEFAULT_WORKLOAD and args.batch == 0:
        from synth import inputs as synth
        companions = [synth.workload(n) for n in COMPANION_WORKLOADS]

    sampler = ClockSampler(gpu_uuid(local))
    with sampler:
        time.sleep(0.3)  # let the sampler start
        head = measure(args, w, world, peaks, peak_src,
                       0.0 if args.no_sustained else args.sustained_s, with_e2e=not args.no_e2e)
        others = {}
        for cw in companions:
            rec = measure(args, cw, world, peaks, peak_src,
                          0.0 if args.no_sustained else args.companion_sustained_s,
                          with_e2e=not args.no_e2e)
            rec.pop("_inp")
            rec.pop("_out")
            others[cw.name] = rec
        time.sleep(0.25)  # the last samples of the last window
    inp = head.pop("_inp")
    out = head.pop("_out")
    for rec in [head, *others.values()]:
        finalize_clocks(rec, sampler, args.steps)

    result = {
        "metric": metric_of(w)[0],
        "value": head["value"],
        "unit": metric_of(w)[1],
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": head["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic: seeded Philox N(0,1) inputs rounded to the kernel dtype (no dataset)",
        "config": config_of(w, world),
        "timing": {"steps": (f"one CUDA graph of the {args.steps} timed steps" if not args.no_graph
                             else "eager calls"),
                   "l2": head["l2"]},
        "tokens_per_s": head["tokens_per_s"],
        "step_ms": head["step_ms"],
        "roofline": head["roofline"],
        "gpu_launches": head["gpu_launches"],
        "clocks": head["clocks"],
    }
    for key in ("pct_of_measured_bf16_peak", "pct_of_nominal_bf16_peak", "input_copies",
                "warm_l2_ms_per_step", "sustained", "e2e"):
        if key in head:
            result[key] = head[key]
    if others:
        result["configs"] = others
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        if w.kind == "attn":
            # The sampled units' oracle outputs are also compared with the GPU's output of
            # the timed workload (the parity of the bench's own run, on those units).
            import numpy as np
            from synth import inputs as synth

            def gpu_head(b, i):
                t = out[b, :, i, :].contiguous().cpu()
                if w.dtype == "f32":
                    return t.numpy().astype(np.float64)
                return synth.bf16_bits_to_f64(t.view(torch_int16()).numpy().view(np.uint16))
            errs = {}
            rate, threads, desc = oracle_sample_rate(w, inp, args.cpu_budget_s, gpu_head=gpu_head,
                                                     errs=errs)
            rate1, _, desc1 = oracle_sample_rate(w, inp, args.cpu_budget_s / 5, sample_index=7,
                                                 threads=1)
        else:
            errs = {}
            rate, threads, desc = sample_rate(w, inp, args.cpu_budget_s)
            rate1 = desc1 = None
        result["cpu_baseline"] = {"value": round(rate, 6), "unit": metric_of(w)[1], "cores": threads,
                                  "kind": "oracle", "sample": desc}
        if rate1 is not None:
            result["cpu_baseline"]["single_thread"] = {"value": round(rate1, 6), "sample": desc1}
        if errs.get("n"):
            result["cpu_baseline"]["gpu_vs_oracle"] = {
                "max_abs_err": errs["max"], "mean_abs_err": errs["sum"] / errs["n"],
                "elements": errs["n"],
                "tolerance": {"max": 1e-5} if w.dtype == "f32" else {"max": 2e-2, "mean": 2e-3}}
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return result


def e2e_pipelined(args, w, host, step, flops, world, pinned):
    """The e2e leg with copies overlapped across steps: two sets of device
    buffers and three streams (host-to-device, compute, device-to-host). Step i
    still copies its own inputs in and its own result out; its compute runs
    while step i+1's inputs arrive and step i-1's result leaves."""
    import torch
    sets = []
    for k in range(2):
        if k == 0:
            inputs, out, fn = host["inputs"], host["output"], step
        else:
            inputs, out, fn = host["rebind"]()
        pairs = [(pinned(h), d) for h, d in inputs.values()]
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        sets.append((pairs, out, hout, fn))
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = [{n: torch.cuda.Event() for n in ("in", "run", "out")} for _ in range(2)]
    for e in ev:  # every buffer starts free
        for n in ("run", "out"):
            e[n].record(torch.cuda.current_stream())

    def e2e_step(i):
        pairs, out, hout, fn = sets[i % 2]
        e = ev[i % 2]
        with torch.cuda.stream(s_in):
            s_in.wait_event(e["run"])   # the previous compute on these buffers is done
            for h, d in pairs:
                d.copy_(h, non_blocking=True)
            e["in"].record(s_in)
        with torch.cuda.stream(s_run):
            s_run.wait_event(e["in"])
            s_run.wait_event(e["out"])  # the previous result left this output buffer
            fn()
            e["run"].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(e["run"])
            hout.copy_(out, non_blocking=True)
            e["out"].record(s_out)

    steps = max(1, min(args.steps, 100))
    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    main = torch.cuda.current_stream()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(main)
    for s in (s_in, s_run, s_out):
        s.wait_event(start)
    for i in range(steps):
        e2e_step(i)
    for s in (s_in, s_run, s_out):
        main.wait_stream(s)
    end.record(main)
    torch.cuda.synchronize()
    barrier(world)
    ms = reduce_max(start.elapsed_time(end), world) / steps
    h2d = sum(h.numel() * h.element_size() for h, _ in sets[0][0])
    d2h = sets[0][2].numel() * sets[0][2].element_size()
    return {"value": round(flops * world / (ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 4), "steps": steps, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "launches": steps,
            "pipeline": "2 buffer sets; host-to-device / compute / device-to-host streams"}


def e2e_leg(args, w, host, step, flops, world):
    """Same metric through the public API with host buffers: every step copies
    the step's inputs from pinned host memory to the device, runs the eager
    call, and copies the result back to pinned host memory (overlapped across
    steps where the workload can bind its step to a second buffer set)."""
    import numpy as np
    import torch

    def pinned(a):
        t = torch.from_numpy(np.ascontiguousarray(a) if w.dtype == "f32"
                             else np.ascontiguousarray(a).view(np.int16))
        t = t.pin_memory()
        return t if w.dtype == "f32" else t.view(torch.bfloat16)

    in_bytes = sum(np.asarray(h).nbytes for h, _ in host["inputs"].values())
    if "rebind" in host and in_bytes >= (8 << 20):  # small steps: stream overhead would dominate
        return e2e_pipelined(args, w, host, step, flops, world, pinned)
    pairs = [(pinned(h), d) for h, d in host["inputs"].values()]
    out = host["output"]
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    stream = torch.cuda.current_stream()
    steps = max(1, min(args.steps, 100))

    def e2e_step():
        for h, d in pairs:
            d.copy_(h, non_blocking=True)
        step()
        hout.copy_(out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        e2e_step()
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = reduce_max(start.elapsed_time(end), world) / steps
    h2d = sum(h.numel() * h.element_size() for h, _ in pairs)
    d2h = hout.numel() * hout.element_size()
    return {"value": round(flops * world / (ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 4), "steps": steps, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "launches": steps}


# ---------------------------------------------------------------- reference arm

def run_reference(args, rank, world):
    from synth import inputs as synth
    if rank != 0:
        return None
    w = load_workload(args)
    inp = workload_inputs(w)
    total_budget_s = 150.0
    per_step = max(0.5, total_budget_s / max(1, args.steps + args.warmup))
    for i in range(args.warmup):
        sample_rate(w, inp, per_step, sample_index=i)
    rates = []
    descs = []
    t0 = time.perf_counter()
    threads = os.cpu_count() or 1
    for i in range(args.steps):
        rate, threads, desc = sample_rate(w, inp, per_step, sample_index=args.warmup + i)
        rates.append(rate)
        descs.append(desc)
    elapsed = time.perf_counter() - t0
    value = statistics.median(rates)
    return {
        "impl": "reference",
        "metric": metric_of(w)[0],
        "value": round(value, 6),
        "unit": metric_of(w)[1],
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * elapsed / max(1, args.steps), 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic: seeded Philox N(0,1) inputs rounded to bf16 (no dataset)",
        "config": config_of(w, world),
        "cpu_baseline": {"value": round(value, 6), "unit": metric_of(w)[1], "cores": threads,
                         "kind": "oracle",
                         "sample": f"each step: {descs[0] if descs else ''} (median over steps)"},
        "e2e": {"value": round(value, 6), "unit": metric_of(w)[1], "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.gpus != world and world > 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    if args.impl == "reference":
        result = run_reference(args, rank, world)
    else:
        result = run_gpu(args, rank, world, local)
    if rank == 0 and result is not None:
        print(json.dumps(result), flush=True)


if __name__ == "__main__":
    main()
