#!/usr/bin/env python3
"""Benchmark of the relative-position attention forward on GB300.

One step = one forward (relpos_attn_fwd through the C ABI) over one batch of
the workload. Default workload: the largest configuration, Shaw clipped
relative keys and values (B=4, H=8, L=4096, d=64, bf16, k=16). Prints one
JSON line (rank 0): the headline workload's numbers at the top level, and a
block of the same form (value, roofline of its dominant kernel, e2e through
the C ABI with host buffers, the fp64 CPU oracle on a bounded sample, clocks)
for every other configuration under "workloads", each timed as long as the
headline, plus the T5 backward.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-others] [--seconds S]

Timing: W untimed steps, then K steps bracketed by a barrier and a device
synchronize, timed with CUDA events on the launching stream; the K steps are
replayed from CUDA graphs that captured the library calls' launches, so the
host's launch rate does not limit the measurement. Consecutive
steps rotate over several copies of the inputs whose total exceeds the L2
cache, so every step reads its operands from HBM. SM clocks and throttle
reasons are sampled with nvidia-smi while the steps run.

Multi-GPU (torchrun): every rank runs an independent replica of the workload
(the (batch, head) units are independent; there is no exchange step), the
barrier is the only collective, and the value is the units of all ranks
divided by the slowest rank's time (weak scaling).

--impl reference times the fp64 CPU oracle on the host cores over a bounded
sample of the same workload (the reference arm of this comparison).
"""
from __future__ import annotations

import argparse
import ctypes
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
sys.path.insert(0, ROOT)

from transformer_attention_relative_gb300.workloads import (MODE_ALIBI, MODE_DEBERTA, MODE_SHAW,  # noqa: E402
                                                            MODE_NAMES, MODE_T5, MODE_TXL,
                                                            WORKLOADS, make_grad_output,
                                                            make_inputs)

L2_BYTES = 129 * 1024 * 1024
METRIC = "rel-pos attention fwd TFLOP/s (bf16) and % of GB300 dense BF16 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------- helpers

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def _code_only(text):
    """C/C++ source without its comments and blank lines: what the compiler
    sees (the sources hold no string literal with comment markers)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


CSRC = os.path.join(ROOT, "transformer_attention_relative_gb300", "csrc")
# the library headers every kernel's translation unit includes, and each
# kernel's own source files
COMMON_HEADERS = ("ptx.cuh", "relpos_common.cuh", "relpos_internal.h")
KERNEL_SOURCES = {
    "relpos_fwd_kernel": ("attn_fwd.cu",),
    "deberta_band_kernel": ("deberta_band.cu",),
    "relpos_decode_partial_kernel": ("decode.cu",),
    "relpos_bwd_stats_kernel": ("attn_bwd.cu", "relpos_bwd.cuh"),
    "relpos_bwd_dkdv_kernel": ("attn_bwd.cu", "relpos_bwd.cuh"),
    "txl_prep_kernel": ("txl_prep.cu",),
}


def _read_csrc(name):
    with open(os.path.join(CSRC, name), encoding="utf-8") as fh:
        return fh.read()


def _hash_files(names, read=_read_csrc):
    h = hashlib.sha256()
    for f in sorted(names):
        h.update(f.encode())
        h.update(_code_only(read(f)).encode())
    return h.hexdigest()[:16]


def source_hash():
    """Hash of all CUDA sources' code (comments excluded)."""
    return _hash_files([f for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h"))])


def kernel_hash(kernel, read=_read_csrc):
    """Hash of the code (comments excluded) that the kernel's translation unit
    compiles -- its own source files and the library headers -- to tell
    whether stored ncu counters were taken on the code that runs."""
    return _hash_files(KERNEL_SOURCES[kernel] + COMMON_HEADERS, read)


def stored_traffic(kernel, workload):
    """dram bytes per launch from profiles/traffic.txt if taken on the code
    the kernel is compiled from now."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    want = kernel_hash(kernel)
    with open(p) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#"):
                k, w, hsh, b = parts[:4]
                if k == kernel and w == workload and hsh == want:
                    return float(b)
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling in the background."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.samples = []   # (t, sm, max, hw, hw_thermal, sw_thermal, power_cap)
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                self.samples.append((time.time(), float(f[1]), float(f[2]),
                                     f[5] == "Active", f[6] == "Active", f[7] == "Active",
                                     f[8] == "Active"))
            except ValueError:
                pass

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        win = [s for s in self.samples if t0 <= s[0] <= t1]
        if not win:
            return None
        reasons = set()
        for s in win:
            for flag, name in zip(s[3:], ("hw_slowdown", "hw_thermal_slowdown",
                                           "sw_thermal_slowdown", "sw_power_cap")):
                if flag:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(s[1] for s in win),
                "sm_max_mhz": max(s[2] for s in win), "reasons": sorted(reasons),
                "samples": len(win)}


def kernels_per_step(w, backward=False):
    """This library's kernels launched by one call (memsets not counted)."""
    if backward:
        # row statistics, dK / dV (with dQ and the T5 / ALiBi table gradient),
        # dQ conversion (Shaw: dQ with the a_K term and the table partials,
        # then their sum)
        # (DeBERTa: the band pre-pass, statistics, dK / dV, the far-sum fold
        # and the dQ, dK conversions; its table products run in cuBLAS)
        return 4 if w.mode == MODE_SHAW else 6 if w.mode == MODE_DEBERTA else 3
    decode = (w.mode == MODE_T5 and w.Lq <= 8) or (w.mode == MODE_ALIBI and w.cache_len > 0)
    n = 2 if decode else 1
    if w.mode in (MODE_DEBERTA, MODE_TXL):
        n += 1  # the band / operand pre-pass
    if w.dtype == "fp32":
        n += 3
    return n


def dominant_kernel(w, backward=False):
    if backward:
        return "relpos_bwd_dkdv_kernel", "tensor"
    if (w.mode == MODE_T5 and w.Lq <= 8) or (w.mode == MODE_ALIBI and w.cache_len > 0):
        return "relpos_decode_partial_kernel", "hbm"
    return "relpos_fwd_kernel", "tensor"


# ---------------------------------------------------------------- GPU arm

class GpuRun:
    def __init__(self, w, device, stream):
        import torch
        import transformer_attention_relative_gb300 as rp
        self.rp = rp
        self.w = w
        self.device = device
        self.stream = stream
        x = make_inputs(w)
        self.host = x
        set_bytes = sum(t.numel() * t.element_size() for t in x.values() if t is not None)
        out_bytes = x["Q"].numel() * x["Q"].element_size()
        self.set_bytes = set_bytes + out_bytes
        self.nsets = max(1, min(16, math.ceil(2.5 * L2_BYTES / self.set_bytes)))
        self.sets = []
        for _ in range(self.nsets):
            d = {k: (v.to(device) if v is not None else None) for k, v in x.items()}
            d["out"] = torch.empty_like(d["Q"])
            self.sets.append(d)
        torch.cuda.synchronize()
        self.sptr = ctypes.c_void_p(stream.cuda_stream)
        self.dtype = 1 if w.dtype == "fp32" else 0

    def _call(self, d, out=None):
        w = self.w
        p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
        if w.cache_len and w.mode == MODE_ALIBI:  # keys at explicit positions
            rc = self.rp.relpos_alibi_decode_positions(
                p(d["Q"]), p(d["K"]), p(d["V"]), p(d["table0"]), p(d["key_pos"]), w.B, w.H, w.Lq, w.Lk,
                int(w.causal), w.q_offset, p(out if out is not None else d["out"]), self.sptr)
            if rc != 0:
                raise RuntimeError(f"relpos_alibi_decode_positions failed: {rc}")
            return
        if w.cache_len:  # keys at explicit positions
            rc = self.rp.relpos_t5_decode_positions(
                p(d["Q"]), p(d["K"]), p(d["V"]), p(d["table0"]), p(d["key_pos"]), w.B, w.H, w.Lq,
                w.Lk, w.num_buckets, w.rel_param, int(w.causal), w.q_offset,
                p(out if out is not None else d["out"]), self.sptr)
            if rc != 0:
                raise RuntimeError(f"relpos_t5_decode_positions failed: {rc}")
            return
        rc = self.rp.relpos_attn_fwd(w.mode, self.dtype, p(d["Q"]), p(d["K"]), p(d["V"]),
                                     p(d["table0"]), p(d["table1"]), w.B, w.H, w.Lq, w.Lk, w.d,
                                     w.num_buckets, w.rel_param, int(w.causal), w.q_offset,
                                     p(out if out is not None else d["out"]), self.sptr)
        if rc != 0:
            raise RuntimeError(f"relpos_attn_fwd failed: {rc}")

    def step(self, i):
        self._call(self.sets[i % self.nsets])

    def _graph(self, n, first):
        """CUDA graph of n consecutive steps (steps first .. first + n - 1)."""
        import torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            for i in range(n):
                self.step(first + i)
        return g

    def timed(self, steps, warmup, barrier):
        """Time exactly `steps` steps. The steps are replayed from CUDA graphs
        (the launch sequence of the library calls, captured once), so the
        number measures the device, not the host's launch rate."""
        import torch
        for i in range(warmup):
            self.step(i)
        torch.cuda.synchronize()
        per = self.nsets * max(1, math.ceil(32 / self.nsets))
        per = min(per, steps)
        reps, rem = divmod(steps, per)
        g_main = self._graph(per, 0)
        g_rem = self._graph(rem, 0) if rem else None
        with torch.cuda.stream(self.stream):  # replay() launches on the current stream
            g_main.replay()
            if g_rem is not None:
                g_rem.replay()
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        t0 = time.time()
        with torch.cuda.stream(self.stream):
            e0.record(self.stream)
            for _ in range(reps):
                g_main.replay()
            if g_rem is not None:
                g_rem.replay()
            e1.record(self.stream)
        torch.cuda.synchronize()
        t1 = time.time()
        barrier()
        ms = e0.elapsed_time(e1)
        return ms, t0, t1

    def sustain(self, seconds):
        """Run steps back to back for about `seconds` (clock sampling window)."""
        import torch
        g = self._graph(self.nsets * max(1, math.ceil(32 / self.nsets)), 0)
        t0 = time.time()
        while time.time() - t0 < seconds:
            with torch.cuda.stream(self.stream):
                for _ in range(20):
                    g.replay()
            torch.cuda.synchronize()
        return t0, time.time()

    def e2e(self, steps, warmup):
        """Same metric through the public call with host buffers: every step
        copies its inputs from pinned host memory and reads its output back.
        Steps run as a serving loop would run them: copies in (one stream per
        device buffer set, two sets alternating), the call and the copy out on
        streams of their own, so that one step's copies overlap the
        neighbouring steps' copies and work."""
        import torch
        pinned = {k: (v.pin_memory() if v is not None else None) for k, v in self.host.items()}
        nbuf = 2
        outs_h = [torch.empty(self.host["Q"].shape, dtype=self.host["Q"].dtype).pin_memory()
                  for _ in range(nbuf)]
        dsets = [self.sets[b % self.nsets] for b in range(nbuf)]
        if self.nsets < nbuf:  # one resident set only (large inputs): add a second
            d = {k: (torch.empty_like(v) if v is not None else None) for k, v in self.sets[0].items()}
            for k, v in self.host.items():
                if v is not None:
                    d[k].copy_(v)
            if "dQ" in d:  # the backward reads dQ back
                d["out"] = d["dQ"]
            dsets[1] = d
        h2d = sum(v.numel() * v.element_size() for v in pinned.values() if v is not None)
        d2h = outs_h[0].numel() * outs_h[0].element_size()
        s_ins = [torch.cuda.Stream(self.device) for _ in range(nbuf)]
        s_out = torch.cuda.Stream(self.device)
        s_c = self.stream
        ev_in = [torch.cuda.Event() for _ in range(nbuf)]
        ev_c = [torch.cuda.Event() for _ in range(nbuf)]
        ev_out = [torch.cuda.Event() for _ in range(nbuf)]

        def one(i):
            b = i % nbuf
            d = dsets[b]
            s_in = s_ins[b]
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_c[b])  # the call two steps back has read this set
                for k, v in pinned.items():
                    if v is not None:
                        d[k].copy_(v, non_blocking=True)
                ev_in[b].record(s_in)
            s_c.wait_event(ev_in[b])
            s_c.wait_event(ev_out[b])  # its output has been read back
            self._call(d)
            ev_c[b].record(s_c)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_c[b])
                outs_h[b].copy_(d["out"], non_blocking=True)
                ev_out[b].record(s_out)

        for i in range(warmup):
            one(i)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s_c)
        for st in s_ins + [s_out]:
            st.wait_stream(s_c)  # the timed region starts at e0 on every stream
        for i in range(steps):
            one(warmup + i)
        for st in s_ins + [s_c]:
            s_out.wait_stream(st)
        e1.record(s_out)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1), h2d, d2h


class BwdRun(GpuRun):
    """The T5, ALiBi or Shaw backward on the same inputs plus a drawn output
    gradient dO: one step is one relpos_t5_attn_bwd (relpos_alibi_attn_bwd,
    relpos_shaw_attn_bwd) call: dQ, dK, dV and the table (slope) gradients.
    Its end-to-end steps copy dO in with the inputs and read dQ back."""

    def __init__(self, w, device, stream):
        import torch
        super().__init__(w, device, stream)
        dO = make_grad_output(w)
        extra = 4 * dO.numel() * dO.element_size()  # dO, dQ, dK, dV
        self.nsets = max(1, min(16, math.ceil(2.5 * L2_BYTES / (self.set_bytes + extra))))
        self.sets = self.sets[:self.nsets]
        self.host = dict(self.host, dO=dO)
        for d in self.sets:
            d["dO"] = dO.to(device)
            d["dQ"] = torch.empty_like(d["Q"])
            d["out"] = d["dQ"]
            d["dK"] = torch.empty_like(d["K"])
            d["dV"] = torch.empty_like(d["V"])
            d["dbias"] = torch.empty_like(d["table0"], dtype=torch.float32)
            if w.mode in (MODE_SHAW, MODE_DEBERTA):
                d["dtab1"] = torch.empty_like(d["table1"], dtype=torch.float32)
        torch.cuda.synchronize()

    def _call(self, d, out=None):
        w = self.w
        p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
        if w.mode == MODE_DEBERTA:
            rc = self.rp.relpos_deberta_attn_bwd(p(d["Q"]), p(d["K"]), p(d["V"]), p(d["dO"]),
                                                 p(d["table0"]), p(d["table1"]), w.B, w.H, w.Lq, w.Lk, w.d,
                                                 w.rel_param, int(w.causal), w.q_offset, p(d["dQ"]),
                                                 p(d["dK"]), p(d["dV"]), p(d["dbias"]), p(d["dtab1"]),
                                                 self.sptr)
        elif w.mode == MODE_SHAW:
            rc = self.rp.relpos_shaw_attn_bwd(p(d["Q"]), p(d["K"]), p(d["V"]), p(d["dO"]),
                                              p(d["table0"]), p(d["table1"]), w.B, w.H, w.Lq, w.Lk, w.d,
                                              w.rel_param, int(w.causal), w.q_offset, p(d["dQ"]),
                                              p(d["dK"]), p(d["dV"]), p(d["dbias"]), p(d["dtab1"]),
                                              self.sptr)
        elif w.mode == MODE_ALIBI:
            rc = self.rp.relpos_alibi_attn_bwd(p(d["Q"]), p(d["K"]), p(d["V"]), p(d["dO"]),
                                               p(d["table0"]), w.B, w.H, w.Lq, w.Lk, w.d,
                                               int(w.causal), w.q_offset, p(d["dQ"]), p(d["dK"]),
                                               p(d["dV"]), p(d["dbias"]), self.sptr)
        else:
            rc = self.rp.relpos_t5_attn_bwd(p(d["Q"]), p(d["K"]), p(d["V"]), p(d["dO"]),
                                            p(d["table0"]), w.B, w.H, w.Lq, w.Lk, w.d,
                                            w.num_buckets, w.rel_param, int(w.causal), w.q_offset,
                                            p(d["dQ"]), p(d["dK"]), p(d["dV"]), p(d["dbias"]),
                                            self.sptr)
        if rc != 0:
            raise RuntimeError(f"attention backward failed: {rc}")


def bwd_flops(w):
    """Algorithmic flops of the backward: twice the forward's products, i.e.
    the four gradient products (dV = P^T dO, dP = dO V^T, dQ = dS K,
    dK = dS^T Q) over the visible (query, key) pairs, plus for Shaw and
    DeBERTa the table terms' products; the kernels' extra recomputations of
    S and dP (and DeBERTa's band pre-pass) are not counted."""
    return 2.0 * w.flops()


def cpu_baseline(w, budget_s=12.0):
    """Time the fp64 oracle on the host cores over a bounded sample of the
    workload: whole (batch, head) units, as many as fit in about budget_s."""
    from oracle import relpos_oracle as orc
    x = make_inputs(w)
    Q, K, V = (x[k].double().numpy() for k in ("Q", "K", "V"))
    t0 = x["table0"].double().numpy()
    t1 = x["table1"].double().numpy() if x["table1"] is not None else None
    start = time.perf_counter()
    if w.mode == MODE_TXL:  # the oracle takes the projected encodings r(t) = W R(t)
        t0 = orc.txl_position_table(t0, w.Lq, w.Lk, w.q_offset)
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    done = 0
    for (b, h) in heads:
        if w.cache_len and w.mode == MODE_ALIBI:
            kp = x["key_pos"].numpy()
            orc.alibi_attention_key_positions(Q[b:b + 1, h:h + 1], K[b:b + 1, h:h + 1], V[b:b + 1, h:h + 1],
                                              t0[h:h + 1], kp[b:b + 1, h:h + 1], causal=w.causal,
                                              q_offset=w.q_offset)
        elif w.cache_len:
            kp = x["key_pos"].numpy()
            orc.t5_attention_key_positions(Q[b:b + 1, h:h + 1], K[b:b + 1, h:h + 1], V[b:b + 1, h:h + 1],
                                           t0[:, h:h + 1], kp[b:b + 1, h:h + 1],
                                           num_buckets=w.num_buckets, max_distance=w.rel_param,
                                           causal=w.causal, q_offset=w.q_offset)
        else:
            orc.attention(w.mode, Q, K, V, t0, t1, num_buckets=w.num_buckets, rel_param=w.rel_param,
                          causal=w.causal, q_offset=w.q_offset, heads=[(b, h)])
        done += 1
        if time.perf_counter() - start > budget_s:
            break
    el = time.perf_counter() - start
    frac = done / len(heads)
    hbm = dominant_kernel(w)[1] == "hbm"
    work = (w.min_bytes() if hbm else w.flops()) * frac
    threads = len(os.sched_getaffinity(0))
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        if info:
            threads = max(i.get("num_threads", 1) for i in info)
    except Exception:
        pass
    value = work / el / (1e9 if hbm else 1e12)
    return {"value": value, "unit": "GB/s" if hbm else "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{done} of {len(heads)} (batch, head) units of {w.name}, all rows, "
                      f"fp64 numpy, {el:.1f} s"}, el, work


# ---------------------------------------------------------------- main

def max_over_ranks(value, world):
    """The largest value over all ranks (for times: the slowest rank's)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    dev = (torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl"
           else torch.device("cpu"))
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(flops_per_step, steps, world, ms_max):
    """Whole-job TFLOP/s: every rank ran `steps` steps of the workload (weak
    scaling), the job took the slowest rank's time."""
    return flops_per_step * steps * world / (ms_max / 1e3) / 1e12


def metric_of(w, backward=False):
    """(metric, unit, work per step, scale to the unit) of a workload."""
    if backward:
        return ("rel-pos attention bwd TFLOP/s (bf16): dQ, dK, dV and the table gradient",
                "TFLOP/s", bwd_flops(w), 1e12)
    if dominant_kernel(w)[1] == "hbm":
        return ("rel-pos attention cached-decode GB/s (bf16) and % of GB300 HBM bandwidth",
                "GB/s", float(w.min_bytes()), 1e9)
    return METRIC, "TFLOP/s", w.flops(), 1e12


def measure_block(w, device, stream, peaks, peak_src, sampler, barrier, world, *, steps=None,
                  warmup=5, seconds=2.0, cpu_budget=0.0, backward=False):
    """Time one workload and return its block: value, ms_per_step, roofline
    of the dominant kernel, e2e through the C ABI with host buffers, clocks
    during the timed region and, with cpu_budget > 0, the CPU oracle."""
    import torch
    g = BwdRun(w, device, stream) if backward else GpuRun(w, device, stream)
    for i in range(max(3, warmup)):
        g.step(i)
    torch.cuda.synchronize()
    n_est = g.nsets * max(1, math.ceil(32 / g.nsets))
    ms_est, _, _ = g.timed(n_est, 1, lambda: None)
    t_est = ms_est / n_est / 1e3
    if steps is None:
        steps = max(20, min(200000, int(seconds / t_est)))
    warmup = max(3, warmup)
    ms, t0, t1 = g.timed(steps, warmup, barrier)
    clocks = sampler.summary(t0 - 0.05, t1 + 0.05)
    window = "timed region"
    if clocks is None:
        a, b = g.sustain(1.0)
        clocks = sampler.summary(a, b)
        window = "1 s of the same steps right after the timed region (timed region too short)"
    if clocks is not None:
        clocks["window"] = window
    ms_max = max_over_ranks(ms, world)
    metric, unit, work, scale = metric_of(w, backward)
    value = work * steps * world / (ms_max / 1e3) / scale
    kname, bound = dominant_kernel(w, backward)
    avg_s = ms / steps / 1e3
    achieved = work / avg_s / scale
    peak = peaks["bf16_tflops"] if bound == "tensor" else peaks["hbm_gbs"]
    roofline = {"bound": bound, "kernel": kname, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak, "traffic": stored_traffic(kname, w.name + ("_backward" if backward else "")),
                "kernel_hash": kernel_hash(kname),
                "peak_source": f"{peak_src} ({'bf16_tflops burst' if bound == 'tensor' else 'hbm_gbs'})",
                "algorithmic_per_launch": work,
                "timed_as": "whole step (every kernel of the call) / steps"}
    if kernels_per_step(w, backward) > 1:
        roofline["note"] = (f"{kernels_per_step(w, backward)} kernels per step: achieved divides by "
                            "the whole step's time, a lower bound for the dominant kernel alone")
    e2e_steps = max(3, min(steps, 50))
    e2e_ms, h2d, d2h = g.e2e(e2e_steps, 2)
    block = {"metric": metric, "value": value, "unit": unit, "steps": steps, "warmup": warmup,
             "ms_per_step": ms_max / steps, "higher_is_better": True,
             "config": config_of(w, world, g, backward), "roofline": roofline,
             "e2e": {"value": work * e2e_steps / (e2e_ms / 1e3) / scale, "unit": unit,
                     "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
             "gpu_launches": steps * kernels_per_step(w, backward), "clocks": clocks}
    if cpu_budget > 0 and not backward:
        block["cpu_baseline"], _, _ = cpu_baseline(w, budget_s=cpu_budget)
    del g
    torch.cuda.empty_cache()
    return block


def config_of(w, world, g, backward=False):
    c = {"workload": w.name + ("_backward" if backward else ""), "mode": MODE_NAMES[w.mode],
         "B": w.B, "H": w.H, "Lq": w.Lq, "Lk": w.Lk, "d": w.d, "causal": w.causal,
         "q_offset": w.q_offset, "parallelism": f"replicas x{world}",
         "l2": f"{g.nsets} rotating input sets of {g.set_bytes / 1e6:.1f} MB "
               f"(> 129 MB L2), no flush"}
    if w.mode == MODE_T5:
        c["num_buckets"] = w.num_buckets
    if w.rel_param:
        c["rel_param"] = w.rel_param
    if w.cache_len:
        c["cache_len"] = w.cache_len
    return c


# every configuration gets a block of its own in the bench line
BLOCK_WORKLOADS = ("t5_base_bidir", "t5_causal", "shaw", "deberta", "txl_mem", "t5_decode",
                   "t5_decode_evicted", "alibi_decode_evicted", "alibi_bidir", "alibi_causal", "alibi_d128",
                   "t5_d128", "t5_tiny_fp32")
BACKWARD_WORKLOADS = ("t5_base_bidir", "t5_causal", "alibi_causal", "shaw", "deberta")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="shaw", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-others", action="store_true",
                    help="time the headline workload only")
    ap.add_argument("--seconds", type=float, default=2.0,
                    help="timed region per workload when --steps is not given")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward of the workload (T5 or ALiBi) as the headline")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = WORKLOADS[args.workload]
    peaks, peak_src = load_peaks()

    if args.impl == "reference":
        if rank != 0:
            return
        steps = args.steps if args.steps is not None else 3
        warm = min(args.warmup, 1)
        for _ in range(warm):
            cpu_baseline(w, budget_s=2.0)
        tot_work, tot_s = 0.0, 0.0
        last = None
        for _ in range(steps):
            cb, el, work = cpu_baseline(w, budget_s=args.cpu_budget / max(1, steps))
            tot_work += work
            tot_s += el
            last = cb
        metric, unit, _, scale = metric_of(w)
        val = tot_work / tot_s / scale
        last["value"] = val
        line = {"impl": "reference", "metric": metric, "value": val, "unit": unit,
                "n_gpus": args.gpus, "steps": steps, "warmup": warm,
                "ms_per_step": 1e3 * tot_s / steps, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": w.name, "mode": MODE_NAMES[w.mode], "B": w.B, "H": w.H,
                           "Lq": w.Lq, "Lk": w.Lk, "d": w.d},
                "cpu_baseline": last,
                "e2e": {"value": val, "unit": unit, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        barrier = dist.barrier
    else:
        barrier = lambda: None  # noqa: E731
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    import transformer_attention_relative_gb300 as rp
    rp.load_library()
    stream = torch.cuda.Stream(device)
    phys = os.environ.get("CUDA_VISIBLE_DEVICES", str(local_rank)).split(",")[local_rank]

    sampler = ClockSampler(phys)
    sampler.start()
    time.sleep(0.3)

    cpu_on = rank == 0 and world == 1 and not args.no_cpu
    head = measure_block(w, device, stream, peaks, peak_src, sampler, barrier, world,
                         steps=args.steps, warmup=args.warmup, seconds=args.seconds,
                         cpu_budget=args.cpu_budget if cpu_on and not args.backward else 0.0,
                         backward=args.backward)
    blocks = {}
    if not args.no_others and rank == 0:
        for name in BLOCK_WORKLOADS:
            if name == w.name:
                continue
            try:
                blocks[name] = measure_block(WORKLOADS[name], device, stream, peaks, peak_src, sampler,
                                             lambda: None, 1, steps=args.steps, warmup=args.warmup,
                                             seconds=args.seconds,
                                             cpu_budget=min(5.0, args.cpu_budget) if cpu_on else 0.0)
            except Exception as e:  # a configuration this build does not run
                blocks[name] = {"unavailable": str(e)[:160]}
        for name in BACKWARD_WORKLOADS:
            try:
                blocks[name + "_backward"] = measure_block(
                    WORKLOADS[name], device, stream, peaks, peak_src, sampler, lambda: None, 1,
                    steps=args.steps, warmup=args.warmup, seconds=args.seconds, backward=True)
            except Exception as e:
                blocks[name + "_backward"] = {"unavailable": str(e)[:160]}
    sampler.stop()

    if rank == 0:
        line = {
            "metric": head["metric"], "value": head["value"], "unit": head["unit"], "n_gpus": world,
            "steps": head["steps"], "warmup": head["warmup"], "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": head["config"],
            "frac_of_peak": head["value"] / world / (peaks["bf16_tflops"] if head["unit"] == "TFLOP/s"
                                                      else peaks["hbm_gbs"]),
            "roofline": head["roofline"], "e2e": head["e2e"], "gpu_launches": head["gpu_launches"],
            "clocks": head["clocks"], "cpu_baseline": head.get("cpu_baseline"),
            "source_hash": source_hash(), "workloads": blocks,
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
