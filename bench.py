"""Benchmark of the absorbed-path MLA decode on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload ragged] [--impl ours|reference]

One step = one decode of the whole workload: the split-KV decode kernel plus
the LSE combine (mla_decode_splitkv + mla_combine through the C ABI), inputs
resident in HBM, L2 flushed before every step.  The scheduler metadata is
computed once per step outside the timed region (it is reused by every layer
of a decode step); the end-to-end leg (`e2e`) includes it together with the
host<->device copies.

Printed: one JSON line (rank 0).  `value` is the decode throughput as a
percentage of one GB300's roofline, summed over GPUs: 100 * sum_r t_roof / T,
t_roof = max(algorithmic bytes / HBM peak, algorithmic FLOPs / bf16 peak), T =
the slowest rank's time per step.  Peaks come from MEASURED_PEAKS.json.

With --impl reference the fp64 CPU oracle is timed on the host cores over a
bounded sample of the same workload (the reference arm of this comparison).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MLA decode TFLOP/s and KV GB/s (B=64,H=128,ctx 4K–32K) as % of GB300 roofline"
WORKLOAD_INDEX = {"tiny": 0, "uniform4k": 1, "ragged": 2, "long": 3, "fp8_mtp2": 4}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# ------------------------------------------------------------------ FLOP / byte accounting
D_C, D_R = 512, 64


def pair_flops(H: int, d_c: int = D_C, d_r: int = D_R) -> int:
    """FLOPs of one (query token, key) pair on the absorbed path: QK over d_c+d_r dims and
    PV over d_c dims for every head ("MLA inference: two computation paths and FlashMLA",
    section "Which is faster: count new tokens and cached tokens", pair_absorb)."""
    return 2 * H * (d_c + d_r) + 2 * H * d_c


def causal_pairs(q: int, k: int) -> int:
    """(query, key) pairs of q new tokens after k cached ones, k counting the new tokens, causal."""
    return q * k - q * (q - 1) // 2


def algorithmic_flops(seqlens, s_q: int, H: int, causal: bool = True) -> int:
    pairs = sum(causal_pairs(s_q, int(L)) if causal else s_q * int(L) for L in seqlens)
    return pairs * pair_flops(H)


def algorithmic_bytes(seqlens, s_q: int, H: int, kv_row_bytes: int, out_elem_bytes: int) -> int:
    """Bytes the decode must move at least once: every visible cache row (only the L_b
    tokens, not the rest of the last page), the queries, outputs, LSE, used block-table
    entries and the lengths."""
    B = len(seqlens)
    kv = sum(int(L) for L in seqlens) * kv_row_bytes
    q = B * s_q * H * (D_C + D_R) * 2
    out = B * s_q * H * D_C * out_elem_bytes
    lse = B * s_q * H * 4
    bt = sum((int(L) + 63) // 64 for L in seqlens) * 4
    return kv + q + out + lse + bt + 4 * B


def kv_bytes(seqlens, kv_row_bytes: int) -> int:
    return sum(int(L) for L in seqlens) * kv_row_bytes


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return dict(FALLBACK_PEAKS, source="fallback")


def qk8_tensor_peak(peaks) -> float:
    """Tensor peak (TFLOP/s) of the FP8-QK decode's mix of MMAs: the latent part of QK (d_c of the
    d_c + d_r QK dims of every pair) on E4M3 codes at twice the measured bf16 rate (the nominal
    fp8 : bf16 ratio of the tensor cores), the RoPE part of QK and all of PV at the bf16 rate."""
    fp8, bf16 = 2 * D_C, 2 * D_R + 2 * D_C  # FLOPs per head and pair
    return peaks["bf16_tflops"] * (fp8 + bf16) / (fp8 / 2 + bf16)


def roofline_time_s(flops: int, nbytes: int, peaks, qk8: bool = False) -> tuple[float, str]:
    t_b = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_f = flops / ((qk8_tensor_peak(peaks) if qk8 else peaks["bf16_tflops"]) * 1e12)
    return (t_b, "hbm") if t_b >= t_f else (t_f, "tensor")


DECODE_SOURCES = ("common.cuh", "decode_kernel.cuh", "plan.h", "ptx.cuh")


def kernel_source_hash() -> str:
    """Hash of the sources the decode kernel is compiled from (its device code and the planner
    whose metadata it walks); DRAM counters taken with other sources are not reported."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "mla_absorbed_decode_02_gb300", "csrc")
    for name in DECODE_SOURCES:
        with open(os.path.join(d, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def committed_traffic(workload: str):
    """DRAM traffic per launch of the decode kernel from the committed ncu summary, if the
    kernel sources still match the ones the counters were taken with."""
    path = os.path.join(ROOT, "profiles", f"decode_kernel_{workload}_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    return d.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks sampling
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (FileNotFoundError, OSError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ distributed helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def reduce_max(value: float, dist, device=None) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value: float, dist, device=None) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle (baseline / reference arm)
def cpu_oracle_sample(w, budget_s: float, threads: int, rng_seed: int = 7):
    """Time the fp64 oracle on whole (sequence, token) rows of w (all heads) until about
    budget_s of wall time is spent; returns (seconds, pairs covered, rows done)."""
    import oracle
    P = oracle.from_workload(w)
    rng = np.random.default_rng(rng_seed)
    order = [(int(b), t) for b in rng.permutation(w.batch) for t in range(w.s_q)]
    done, pairs = [], 0
    t0 = time.perf_counter()
    lock = threading.Lock()
    idx = [0]

    def worker():
        nonlocal pairs
        while True:
            with lock:
                if idx[0] >= len(order) or time.perf_counter() - t0 > budget_s:
                    return
                item = order[idx[0]]
                idx[0] += 1
            b, t = item
            P.rows(b, t)
            with lock:
                done.append(item)
                pairs += P.visible_keys(b, t)

    ts = [threading.Thread(target=worker) for _ in range(threads)]
    for th in ts:
        th.start()
    for th in ts:
        th.join()
    return time.perf_counter() - t0, pairs, len(done)


def cpu_baseline(w, peaks, budget_s: float, threads: int):
    secs, pairs, rows = cpu_oracle_sample(w, budget_s, threads)
    H = w.num_heads
    flops = pairs * pair_flops(H)
    nbytes = pairs * (656 if w.kv_dtype == "fp8" else 1152)
    t_roof, _ = roofline_time_s(flops, nbytes, peaks)
    return {"value": 100.0 * t_roof / secs if secs > 0 else None, "unit": "% of GB300 roofline",
            "cores": threads, "kind": "oracle", "tflops": flops / secs / 1e12,
            "sample": f"{rows} of {w.batch * w.s_q} (sequence, token) rows, all {H} heads, "
                      f"{pairs} (query, key) pairs, {secs:.1f} s wall on {threads} host threads"}


# ------------------------------------------------------------------ our arm
def _device_inputs(w, dev):
    import torch
    host = {
        "q_nope": torch.from_numpy(w.q_nope.view(np.int16)).view(torch.bfloat16),
        "q_rope": torch.from_numpy(w.q_rope.view(np.int16)).view(torch.bfloat16),
        "kv": (torch.from_numpy(w.kv.view(np.int16)).view(torch.bfloat16) if w.kv_dtype == "bf16"
               else torch.from_numpy(w.kv)),
        "bt": torch.from_numpy(w.block_table),
        "seq": torch.from_numpy(w.seqlens),
    }
    return host, {k: v.to(dev) for k, v in host.items()}


def _params(w, token_group=0, qk_fp8=False):
    from mla_absorbed_decode_02_gb300 import (MlaDecodeParams, MLA_KV_BF16, MLA_KV_FP8_E4M3, MLA_OUT_BF16,
                                              MLA_OUT_F32)
    return MlaDecodeParams.make(w.batch, w.s_q, w.num_heads, w.num_pages, w.block_table.shape[1], causal=w.causal,
                                kv_dtype=MLA_KV_FP8_E4M3 if w.kv_dtype == "fp8" else MLA_KV_BF16,
                                out_dtype=MLA_OUT_F32 if w.out_dtype == "f32" else MLA_OUT_BF16,
                                token_group=token_group, qk_fp8=int(qk_fp8))


def _accounting(w, peaks, qk8=False):
    flops = algorithmic_flops(w.seqlens, w.s_q, w.num_heads, w.causal)
    row_bytes = 656 if w.kv_dtype == "fp8" else 1152
    nbytes = algorithmic_bytes(w.seqlens, w.s_q, w.num_heads, row_bytes, 4 if w.out_dtype == "f32" else 2)
    t_roof, bound = roofline_time_s(flops, nbytes, peaks, qk8)
    return flops, nbytes, row_bytes, t_roof, bound


def _roofline(w, name, peaks, t_dec, qk8=False):
    """Roofline object of the decode kernel: algorithmic bytes (or FLOPs) per launch over its event time."""
    flops, nbytes, _, _, bound = _accounting(w, peaks, qk8)
    if bound == "hbm":
        achieved = nbytes / t_dec / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "peak_source": f"{peaks['source']} (copy, burst)"}
    elif qk8:
        achieved, peak = flops / t_dec / 1e12, qk8_tensor_peak(peaks)
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": f"{peaks['source']} (cuBLAS bf16, burst; the QK latent part at 2x that rate)"}
    else:
        achieved = flops / t_dec / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"], "peak_source": f"{peaks['source']} (cuBLAS bf16, burst)"}
    roof["traffic"] = committed_traffic(name)
    roof["kernel"] = ("mla_decode_fp8qk_kernel" if qk8 else
                      "mla_decode_fp8_kernel" if w.kv_dtype == "fp8" else "mla_decode_bf16_kernel")
    roof["kernel_ms"] = t_dec * 1e3
    return roof


class _NoFlush:
    """Stands in for the flush buffer when the decode is timed without flushing L2."""

    def zero_(self):
        pass


def time_workload(w, name, peaks, steps, warmup, dev, flush, dist=None, token_group=0, qk_fp8=False):
    """Device timing of one workload, inputs resident in HBM, L2 flushed before every step.

    Pass 1 times whole steps (decode kernel + LSE combine, nothing between the two launches, so
    the combine starts as a programmatic dependent of the decode kernel); pass 2 times the decode
    kernel alone (an event right after it).  Both report the median over `steps` steps after
    `warmup` untimed ones.  qk_fp8: the FP8-QK decode, its query quantised on the device first
    (mla_quantize_q_fp8, counted in both passes)."""
    import torch
    from mla_absorbed_decode_02_gb300 import (Decoder, mla_combine, mla_decode_splitkv, mla_device_error,
                                              mla_get_scheduler_metadata, mla_quantize_q_fp8)
    host, d = _device_inputs(w, dev)
    p = _params(w, token_group, qk_fp8)
    dec = Decoder(p, dev)
    out, lse = dec.new_outputs()
    stream = torch.cuda.current_stream(dev)
    mla_get_scheduler_metadata(p, d["seq"], dec.sched, stream)
    rows = w.batch * w.s_q * w.num_heads
    q8 = torch.empty((rows, 656), dtype=torch.uint8, device=dev) if qk_fp8 else None

    def decode():
        if qk_fp8:
            mla_quantize_q_fp8(d["q_nope"], d["q_rope"], q8, rows, stream)
            mla_decode_splitkv(p, q8, None, d["kv"], d["bt"], d["seq"], w.scale, out, lse, dec.sched, dec.workspace,
                               stream)
            return
        mla_decode_splitkv(p, d["q_nope"], d["q_rope"], d["kv"], d["bt"], d["seq"], w.scale, out, lse, dec.sched,
                           dec.workspace, stream)

    def combine():
        mla_combine(p, out, lse, dec.sched, dec.workspace, stream)

    for _ in range(warmup):
        flush.zero_()
        decode()
        combine()
    torch.cuda.synchronize(dev)
    assert mla_device_error(clear=True) == 0, "device error during warm-up"

    def timed(kernel_only):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)
        for k in range(steps):
            flush.zero_()
            evs[k][0].record(stream)
            decode()
            if kernel_only:
                evs[k][1].record(stream)
                combine()
            else:
                combine()
                evs[k][1].record(stream)
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        return [a.elapsed_time(b) / 1e3 for a, b in evs]

    step_s = timed(False)
    dec_s = timed(True)
    err = mla_device_error(clear=True)
    assert err == 0, f"device error word {err}"
    res = {"t_step": statistics.median(step_s), "t_step_mean": sum(step_s) / len(step_s),
           "t_dec": statistics.median(dec_s), "host": host, "dev": d, "p": p, "dec": dec, "out": out, "lse": lse}
    return res


def time_projections(w, peaks, steps, warmup, dev, flush, d_nope=128, d_v=128):
    """Median time of mla_absorb_query and mla_project_output for the workload's B*s_q tokens, with
    their roofline (bytes: weights + activations in and out; FLOPs: 2*T*H*K*N)."""
    import torch
    from mla_absorbed_decode_02_gb300 import mla_absorb_query, mla_device_error, mla_project_output
    T, H = w.batch * w.s_q, w.num_heads
    g = torch.Generator(device=dev).manual_seed(5)
    q_n = torch.randn((T, H, d_nope), generator=g, device=dev).to(torch.bfloat16)
    w_uk = (torch.randn((H, d_nope, 512), generator=g, device=dev) / 512 ** 0.5).to(torch.bfloat16)
    w_uv = (torch.randn((H, 512, d_v), generator=g, device=dev) / 512 ** 0.5).to(torch.bfloat16)
    q_abs = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    o = torch.empty((T, H, d_v), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    out = {}
    for name, call, K, N in (("absorb", lambda: mla_absorb_query(q_n, w_uk, q_abs, stream), d_nope, 512),
                             ("project", lambda: mla_project_output(q_abs, w_uv, o, stream), 512, d_v)):
        for _ in range(warmup):
            flush.zero_()
            call()
        ts = []
        for _ in range(steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            torch.cuda.synchronize(dev)
            ts.append(a.elapsed_time(b) / 1e3)
        t = statistics.median(ts)
        nbytes = 2 * (H * K * N + T * H * (K + N))
        flops = 2 * T * H * K * N
        t_roof, bound = roofline_time_s(flops, nbytes, peaks)
        out[name] = {"us": t * 1e6, "tokens": T, "heads": H, "k": K, "n": N, "bytes": nbytes, "flops": flops,
                     "bound": bound, "roofline_frac": t_roof / t}
    assert mla_device_error(clear=True) == 0
    return out


def extend_flops(q: int, k: int, H: int, d_c: int = D_C, d_nope: int = 128, d_r: int = D_R, d_v: int = 128) -> int:
    """FLOPs of an extend by path one ("Which is faster: count new tokens and cached tokens"):
    expanding every cached row into H keys and values, 2*d_c*H*(d_nope + d_v) each, plus the
    causal (query, key) pairs at 2*H*(d_nope + d_r) + 2*H*d_v each."""
    return k * 2 * d_c * H * (d_nope + d_v) + causal_pairs(q, k) * (2 * H * (d_nope + d_r) + 2 * H * d_v)


def time_extend(peaks, steps, warmup, dev, flush, prefix=32768, s_q=512, H=128, chunk=4096):
    """Median time of mla_extend appending s_q tokens to a `prefix`-row cache (one sequence, the
    pages' "append 512 tokens after a 32K cached prefix"), with its tensor roofline."""
    import torch
    import mla_workloads as mw
    from mla_absorbed_decode_02_gb300 import MlaExtendParams, mla_device_error, mla_extend, mla_extend_workspace_size
    L = prefix + s_q
    x = mw.make_extend([L], s_q=s_q, num_heads=H, seed=11, nan_tail=False)
    c = x.cache
    dv = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)
    q_n, q_r, kv, w_uk, w_uv = dv(x.q_nope), dv(x.q_rope), dv(c.kv), dv(x.w_uk), dv(x.w_uv)
    bt, seq = torch.from_numpy(c.block_table).to(dev), torch.from_numpy(c.seqlens).to(dev)
    p = MlaExtendParams.make(1, s_q, H, c.kv.shape[0], c.block_table.shape[1], L, chunk)
    ws = torch.empty(mla_extend_workspace_size(p), dtype=torch.uint8, device=dev)
    out = torch.empty((1, s_q, H, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((1, s_q, H), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call():
        mla_extend(p, q_n, q_r, kv, bt, seq, w_uk, w_uv, x.scale, out, lse, ws, stream)

    for _ in range(warmup):
        flush.zero_()
        call()
    ts = []
    for _ in range(steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        call()
        b.record(stream)
        torch.cuda.synchronize(dev)
        ts.append(a.elapsed_time(b) / 1e3)
    assert mla_device_error(clear=True) == 0
    t = statistics.median(ts)
    flops = extend_flops(s_q, L, H)
    nbytes = L * 1152 + s_q * H * (128 + D_R) * 2 + 2 * H * 128 * D_C * 2 + s_q * H * (128 * 2 + 4)
    t_roof, bound = roofline_time_s(flops, nbytes, peaks)
    n_chunks = (L + chunk - 1) // chunk
    return {"workload": f"append {s_q} tokens after a {prefix}-row cache (B=1, H={H}, d_nope=d_v=128)",
            "chunk_tokens": chunk, "launches": 2 * n_chunks, "us": t * 1e6, "flops": flops, "bytes": nbytes,
            "tflops": flops / t / 1e12, "bound": bound, "roofline_frac": t_roof / t,
            "timing": f"median of {steps} calls after {warmup}, L2 flushed before each, CUDA events"}


def run_ours(args, w, peaks, world, rank, local):
    import torch
    import mla_workloads as mw
    from mla_absorbed_decode_02_gb300.build import build
    from mla_absorbed_decode_02_gb300 import (mla_decode, mla_device_error, mla_get_scheduler_metadata,
                                              mla_quantize_q_fp8)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        build()
    dist = init_dist(world, "nccl")
    if dist is not None:
        dist.barrier()
        build()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)  # > L2 (129 MB)
    # The decode's inputs (the cache: 151 MB to 845 MB) are larger than L2; --l2 none times the
    # decode steps without the flush.  The projections and the extend always flush (their weights
    # fit in L2).
    flush_dec = _NoFlush() if args.l2 == "none" else flush
    stream = torch.cuda.current_stream(dev)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    qk8 = bool(args.qk_fp8)
    name = args.workload + ("_qk_fp8" if qk8 else "")
    r = time_workload(w, args.workload, peaks, args.steps, args.warmup, dev, flush_dec, dist, args.token_group, qk8)
    clk = clocks.stop()
    t_step, t_dec = r["t_step"], r["t_dec"]
    t_max = reduce_max(t_step, dist, dev)

    # ---- end to end through the public API: pinned host inputs -> device, plan, decode, results -> host
    host, d, p, dec, out, lse = r["host"], r["dev"], r["p"], r["dec"], r["out"], r["lse"]
    units = dec.num_units
    hq, hr, hbt, hseq = (host[k].pin_memory() for k in ("q_nope", "q_rope", "bt", "seq"))
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hlse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hr, hbt, hseq))
    d2h = hout.numel() * hout.element_size() + hlse.numel() * hlse.element_size()

    # The plan needs only the lengths: it runs on a second stream while the queries and the block
    # table cross the host link (copies are link-bound, ~200 GB/s on this host).
    plan_stream = torch.cuda.Stream(dev)
    rows = w.batch * w.s_q * w.num_heads
    q8 = torch.empty((rows, 656), dtype=torch.uint8, device=dev) if qk8 else None

    def e2e_step():
        d["seq"].copy_(hseq, non_blocking=True)
        seq_ready = torch.cuda.Event()
        seq_ready.record(stream)
        plan_stream.wait_event(seq_ready)
        mla_get_scheduler_metadata(p, d["seq"], dec.sched, plan_stream)
        planned = torch.cuda.Event()
        planned.record(plan_stream)
        d["q_nope"].copy_(hq, non_blocking=True)
        d["q_rope"].copy_(hr, non_blocking=True)
        d["bt"].copy_(hbt, non_blocking=True)
        stream.wait_event(planned)
        if qk8:
            mla_quantize_q_fp8(d["q_nope"], d["q_rope"], q8, rows, stream)
            mla_decode(p, q8, None, d["kv"], d["bt"], d["seq"], w.scale, out, lse, dec.sched, dec.workspace, stream)
        else:
            mla_decode(p, d["q_nope"], d["q_rope"], d["kv"], d["bt"], d["seq"], w.scale, out, lse, dec.sched,
                       dec.workspace, stream)
        hout.copy_(out, non_blocking=True)
        hlse.copy_(lse, non_blocking=True)

    for _ in range(args.warmup):
        flush_dec.zero_()
        e2e_step()
    torch.cuda.synchronize(dev)
    e_ms = []
    for _ in range(args.steps):
        flush_dec.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        b.record(stream)
        b.synchronize()
        e_ms.append(a.elapsed_time(b))
    t_e2e = reduce_max(statistics.median(e_ms) / 1e3, dist, dev)
    assert mla_device_error(clear=True) == 0
    del r, host, d, dec, out, lse

    flops, nbytes, row_bytes, t_roof, bound = _accounting(w, peaks, qk8)
    n = world
    value = 100.0 * n * t_roof / t_max
    res = {
        "metric": METRIC, "value": value, "unit": "% of GB300 roofline (summed over GPUs)", "n_gpus": n,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_max * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": ("bf16" if w.kv_dtype == "bf16" else
                  "fp8-e4m3 cache and query, e4m3 QK mma, bf16 PV mma" if qk8 else "fp8-e4m3 cache, bf16 mma"),
        "data": "synthetic (seeded N(0,1) bf16 queries and cache, random page permutation)",
        "config": {"workload": args.workload + (f" (first {w.batch} sequences)" if args.batch else ""),
                   "batch": w.batch, "heads": w.num_heads, "s_q": w.s_q,
                   "seqlens": f"{int(w.seqlens.min())}..{int(w.seqlens.max())} (sum {int(w.seqlens.sum())})",
                   "kv_dtype": w.kv_dtype, "pages": w.num_pages, "units": units, "token_group": args.token_group or 1,
                   "l2": (f"not flushed: the cache ({kv_bytes(w.seqlens, row_bytes) / 1e6:.0f} MB) is larger than "
                          "L2 (129 MB)" if args.l2 == "none"
                          else "flushed before every step (256 MiB write)"), "parallelism": f"replicas x{n}",
                   "timing": f"median of {args.steps} steps after {args.warmup} warm-up steps, CUDA events"},
        "tflops": n * flops / t_max / 1e12, "kv_gbs": n * kv_bytes(w.seqlens, row_bytes) / t_max / 1e9,
        "roofline": _roofline(w, name, peaks, t_dec, qk8),
        "e2e": {"value": 100.0 * n * t_roof / t_e2e, "unit": "% of GB300 roofline (summed over GPUs)",
                "ms_per_step": t_e2e * 1e3, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "includes": "H2D q/q_rope/block_table/seqlens, scheduler metadata (second stream, "
                            "overlapping the query copies), decode, D2H out/lse"},
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
        "peaks": {k: peaks[k] for k in ("hbm_gbs", "bf16_tflops", "source")},
    }

    # ---- the projections around the decode for this batch (query absorption before it, the value
    # projection after it): random DeepSeek-V3-shaped W_UK / W_UV, L2 flushed before each call
    res["projections"] = time_projections(w, peaks, args.steps, args.warmup, dev, flush)

    # ---- the expand path for an extend (chunked prefix expansion with the LSE merge)
    if world == 1 and not args.no_extend:
        res["extend"] = time_extend(peaks, min(args.steps, 20), min(args.warmup, 5), dev, flush)

    # ---- the other benchmark workloads (one GPU: the driver's multi-GPU runs time the headline only)
    if world == 1 and not args.no_per_config:
        per = {}
        clocks = ClockSampler(local)
        clocks.start()
        time.sleep(0.3)
        # (fp8_mtp2 three times: one CTA pair per new token; both new tokens of a sequence on shared
        # pages, token group 2, which reads the cache once; and the opt-in FP8-QK decode)
        for name, grp, qk8 in (("uniform4k", 0, False), ("long", 0, False), ("fp8_mtp2", 0, False),
                               ("fp8_mtp2", 2, False), ("fp8_mtp2", 0, True)):
            if name == args.workload and grp == args.token_group and qk8 == bool(args.qk_fp8):
                continue
            wk = mw.make_workload(WORKLOAD_INDEX[name])
            rk = time_workload(wk, name, peaks, args.steps, args.warmup, dev, flush_dec, token_group=grp, qk_fp8=qk8)
            _, _, _, tr, _ = _accounting(wk, peaks, qk8)
            key = name + (f"_token_group{grp}" if grp else "") + ("_qk_fp8" if qk8 else "")
            per[key] = {
                "value": 100.0 * tr / rk["t_step"], "ms_per_step": rk["t_step"] * 1e3,
                "kernel_ms": rk["t_dec"] * 1e3,
                "roofline": _roofline(wk, key, peaks, rk["t_dec"], qk8),
                "config": {"batch": wk.batch, "s_q": wk.s_q, "kv_dtype": wk.kv_dtype, "units": rk["dec"].num_units,
                           "token_group": grp or 1, "qk": "e4m3 codes (tcgen05 kind::f8f6f4)" if qk8 else "bf16",
                           "seqlens": f"{int(wk.seqlens.min())}..{int(wk.seqlens.max())} "
                                      f"(sum {int(wk.seqlens.sum())})"}}
            del rk, wk
            torch.cuda.empty_cache()
        per_clk = clocks.stop()
        res["per_config"] = per
        res["per_config_clocks"] = per_clk
    return res, dist


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="ragged", choices=sorted(WORKLOAD_INDEX))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="time the chosen workload only")
    ap.add_argument("--no-extend", action="store_true", help="skip the extend (expand path) timing")
    ap.add_argument("--l2", default="flush", choices=["flush", "none"],
                    help="flush L2 before every decode step (256 MiB write), or not (the cache is larger than L2)")
    ap.add_argument("--qk-fp8", action="store_true",
                    help="FP8 cache only: the opt-in decode with QK on E4M3 codes (query quantised on the device)")
    ap.add_argument("--token-group", type=int, default=0,
                    help="new tokens per work block for the chosen workload (mla_decode_params.token_group)")
    ap.add_argument("--batch", type=int, default=0,
                    help="keep only the first B sequences of the workload (same recipe; for profiling small cases)")
    args = ap.parse_args()
    import mla_workloads as mw

    world, rank, local = dist_env()
    peaks = load_peaks()
    w = mw.make_workload(WORKLOAD_INDEX[args.workload])
    if args.qk_fp8 and (w.kv_dtype != "fp8" or args.token_group > 1):
        ap.error("--qk-fp8 needs an FP8-cache workload and no token group")
    if args.batch:
        w = mw.first_sequences(w, args.batch)
    threads = os.cpu_count() or 1

    if args.impl == "reference":
        if rank != 0:
            return 0
        secs_total, pairs_total, rows_total = 0.0, 0, 0
        per = max(2.0, min(args.cpu_budget, 60.0 / max(1, args.steps + args.warmup)))
        for _ in range(args.warmup):
            cpu_oracle_sample(w, per, threads)
        for k in range(args.steps):
            s, pr, rows = cpu_oracle_sample(w, per, threads, rng_seed=100 + k)
            secs_total += s
            pairs_total += pr
            rows_total += rows
        flops = pairs_total * pair_flops(w.num_heads)
        nbytes = pairs_total * (656 if w.kv_dtype == "fp8" else 1152)
        t_roof, _ = roofline_time_s(flops, nbytes, peaks)
        value = 100.0 * t_roof / secs_total
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "% of GB300 roofline (summed over GPUs)",
                "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": secs_total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": args.workload, "batch": w.batch, "heads": w.num_heads,
                           "sample": "each step: whole (sequence, token) rows for ~%.0f s" % per},
                "cpu_baseline": {"value": value, "unit": "% of GB300 roofline", "cores": threads, "kind": "oracle",
                                 "sample": f"{rows_total} rows, {pairs_total} (query, key) pairs, all heads, "
                                           f"{secs_total:.1f} s over {args.steps} steps"},
                "e2e": {"value": value, "unit": "% of GB300 roofline (summed over GPUs)", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    res, dist = run_ours(args, w, peaks, world, rank, local)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(w, peaks, args.cpu_budget, threads)
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
