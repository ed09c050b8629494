#!/usr/bin/env python
"""Decode-attention benchmark: KV GB/s, fraction of the HBM roofline, and
decode tokens/s on GB300, through libkvd's C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload npuw|gqa|long|paged]
    python bench.py --impl reference ...     # the fp64 CPU oracle as the reference arm

A step is one decode step of the workload: for the static-buffer workloads,
every layer appends the step's K/V row and runs masked split-KV attention
(+ the log-sum-exp combine); for the paged workload, the paged gather and the
paged attention over the whole cache.  ``value`` is algorithmic bytes per
second (valid K/V rows, mask, q and out, appended rows; no padding and no
split scratch), whole job over all ranks.  Multi-GPU runs are independent
replicas (weak scaling, no data-path collective).

Besides the main line (the 1152-slot NPUW-default buffer by default), the
JSON carries the same measurement for the other workloads under "workloads"
(batched GQA, paged, long context), which are the ones the 75 % HBM gate is
stated on.
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024

# dram__bytes_read.sum + dram__bytes_write.sum per launch of the attention
# split kernel, from the ncu capture summarised in profiles/, keyed by the
# hash of the kernel sources it was taken on (reported only while they match).
NCU_TRAFFIC = {}


# ------------------------------------------------------------ byte accounting

def masked_attend_bytes(lengths, Hq, Hkv, C, D, elem):
    """Valid K and V rows of every kv head, the mask row, q and out."""
    B = len(lengths)
    return (sum(int(L) for L in lengths) * Hkv * D * 2 * elem + B * C + 2 * B * Hq * D * elem)


def append_bytes(B, Hkv, D, elem):
    """Read and write of the new K and V rows."""
    return 4 * B * Hkv * D * elem


def paged_attend_bytes(lengths, Hq, Hkv, D, elem, BS):
    """Valid K and V rows, the block-table entries the sequences use, the
    cumsum, q and out."""
    Q = len(lengths)
    rows = sum(int(L) for L in lengths)
    entries = sum((int(L) + BS - 1) // BS for L in lengths)
    return rows * Hkv * D * 2 * elem + entries * 4 + (Q + 1) * 4 + 2 * Q * Hq * D * elem


def gather_bytes(lengths, Hk, Dk, Hv, Dv, elem, BS):
    """Read + write of every gathered row, plus the indices used."""
    Q = len(lengths)
    T = sum(int(L) for L in lengths)
    entries = sum((int(L) + BS - 1) // BS for L in lengths)
    return 2 * T * (Hk * Dk + Hv * Dv) * elem + entries * 4 + (Q + 1) * 4


def attention_flops(lengths, Hq, D):
    return 4 * sum(int(L) for L in lengths) * Hq * D


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "decode_attention_kv_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the GPU is busy."""
    FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id=None, interval_ms=50):
        self.bus_id = bus_id
        self.interval_ms = interval_ms
        self.proc = None
        self.path = None
        self.error = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="kvd_clocks_", suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", str(self.interval_ms)]
            if self.bus_id:
                cmd += ["-i", self.bus_id]
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception as e:  # nvidia-smi missing
            self.error = f"nvidia-smi unavailable: {e}"
        return self

    def stop(self):
        if self.proc is None:
            return {"unavailable": self.error or "not started"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"unavailable": "no samples"}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "", 1).isdigit()]
        smax = [float(r[3]) for r in rows if r[3].replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows), "interval_ms": self.interval_ms}


def bus_id_of(torch, dev):
    try:
        p = torch.cuda.get_device_properties(dev)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        return None


# ---------------------------------------------------------------- workloads

class MaskedBench:
    """Static-buffer workload: per layer append + masked attention."""

    def __init__(self, name, torch, kvd, dev, W):
        import workloads
        self.torch, self.kvd, self.dev, self.name = torch, kvd, dev, name
        if name == "npuw":
            w = workloads.npuw(device=dev)
            self.cycle, self.prompt = 128, 1024
        elif name == "gqa":
            w = workloads.gqa(device=dev)
            self.cycle, self.prompt = 1, None
        elif name == "long":
            w = workloads.long(device=dev)
            self.cycle, self.prompt = 1, None
        else:
            raise ValueError(name)
        self.w = w
        lay0 = w.layers[0]
        self.B, self.Hq, self.Hkv, self.C, self.D = w.B, w.Hq, w.Hkv, w.C, w.D
        self.elem = 2
        base = lay0.pos.to(torch.int64)
        # append position of step i: base + (i mod cycle)
        self.pos_table = torch.stack([(base + i).to(torch.int32) for i in range(self.cycle)]).to(dev)
        need = kvd.attend_masked_workspace_bytes(self.B, self.Hq, self.Hkv, self.C, self.D)
        self.ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        self.splits = need > 0
        self.out = [torch.empty_like(l.q) for l in w.layers]
        self.status = kvd.status_tensor(dev)
        self.lengths0 = [int(x) for x in lay0.lengths]

    @property
    def layers(self):
        return len(self.w.layers)

    def lengths_at(self, i):
        return [L + (i % self.cycle) for L in self.lengths0]

    def reset_if_wrapped(self, i):
        if self.cycle > 1 and i % self.cycle == 0 and i > 0:
            for lay in self.w.layers:
                lay.mask[:, self.prompt:] = 0

    def step(self, i, events=None):
        kvd = self.kvd
        pos = self.pos_table[i % self.cycle]
        for li, lay in enumerate(self.w.layers):
            kvd.append(lay.k_cache, lay.v_cache, lay.k_new, lay.v_new, pos, lay.mask, self.status)
            if events is not None:
                events[li][0].record()
            kvd.attend_masked(lay.q, lay.k_cache, lay.v_cache, lay.mask, lay.scale,
                              out=self.out[li], workspace=self.ws, dev_status=self.status)
            if events is not None:
                events[li][1].record()

    def launches_per_step(self):
        return self.layers * (2 + (1 if self.splits else 0))

    def attend_bytes(self, i):
        return masked_attend_bytes(self.lengths_at(i), self.Hq, self.Hkv, self.C, self.D, self.elem)

    def step_bytes(self, i):
        return self.layers * (self.attend_bytes(i) + append_bytes(self.B, self.Hkv, self.D, self.elem))

    def tokens_per_step(self):
        return self.B

    def e2e_setup(self):
        torch = self.torch
        self.h_q = [torch.empty(l.q.shape, dtype=l.q.dtype, pin_memory=True).copy_(l.q.cpu())
                    for l in self.w.layers]
        self.h_kn = [torch.empty(l.k_new.shape, dtype=l.k_new.dtype, pin_memory=True).copy_(l.k_new.cpu())
                     for l in self.w.layers]
        self.h_vn = [torch.empty(l.v_new.shape, dtype=l.v_new.dtype, pin_memory=True).copy_(l.v_new.cpu())
                     for l in self.w.layers]
        self.h_pos = torch.empty(self.pos_table.shape, dtype=torch.int32, pin_memory=True).copy_(
            self.pos_table.cpu())
        self.h_out = [torch.empty(l.q.shape, dtype=l.q.dtype, pin_memory=True) for l in self.w.layers]
        self.d_pos = torch.empty(self.B, dtype=torch.int32, device=self.dev)
        h2d = sum(t.numel() * t.element_size() for t in self.h_q + self.h_kn + self.h_vn) + self.B * 4
        d2h = sum(t.numel() * t.element_size() for t in self.h_out)
        return h2d, d2h

    def e2e_step(self, i):
        kvd = self.kvd
        self.d_pos.copy_(self.h_pos[i % self.cycle], non_blocking=True)
        for li, lay in enumerate(self.w.layers):
            lay.q.copy_(self.h_q[li], non_blocking=True)
            lay.k_new.copy_(self.h_kn[li], non_blocking=True)
            lay.v_new.copy_(self.h_vn[li], non_blocking=True)
            kvd.append(lay.k_cache, lay.v_cache, lay.k_new, lay.v_new, self.d_pos, lay.mask,
                       self.status)
            kvd.attend_masked(lay.q, lay.k_cache, lay.v_cache, lay.mask, lay.scale,
                              out=self.out[li], workspace=self.ws, dev_status=self.status)
            self.h_out[li].copy_(self.out[li], non_blocking=True)

    def config(self):
        e = self.elem
        ws_bytes = self.layers * 2 * self.B * self.Hkv * self.C * self.D * e
        return {"workload": self.name, "batch": self.B, "q_heads": self.Hq, "kv_heads": self.Hkv,
                "head_dim": self.D, "capacity": self.C, "layers": self.layers,
                "valid_len_step0": (self.lengths0 if len(self.lengths0) <= 4 else
                                    {"min": min(self.lengths0), "max": max(self.lengths0),
                                     "mean": sum(self.lengths0) / len(self.lengths0)}),
                "l2": f"inputs larger than L2: {ws_bytes / 2**30:.2f} GiB of layer caches "
                      f"rotated per step vs {L2_BYTES // 2**20} MiB L2"}


class PagedBench:
    """Paged workload: gather_pa_kv_cache + paged attention over one cache."""

    def __init__(self, torch, kvd, dev, W):
        import workloads
        self.torch, self.kvd, self.dev, self.name = torch, kvd, dev, "paged"
        pw = workloads.paged(device=dev)
        self.pw = pw
        self.Q, self.Hq, self.D = pw.q.shape
        self.NB, self.BS, self.Hkv, _ = pw.key_cache.shape
        self.elem = 2
        self.lengths = [int(x) for x in pw.lengths]
        self.ko = torch.empty((pw.total_tokens, self.Hkv, self.D), dtype=torch.bfloat16, device=dev)
        self.vo = torch.empty_like(self.ko)
        self.out = torch.empty_like(pw.q)
        cols = pw.block_tables.shape[1]
        need = kvd.attend_paged_workspace_bytes(self.Q, self.Hq, self.Hkv, self.BS, cols, self.D)
        self.ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        self.splits = need > 0
        self.status = kvd.status_tensor(dev)
        self.layers = 1

    def step(self, i, events=None, gather_events=None):
        kvd, pw = self.kvd, self.pw
        if gather_events is not None:
            gather_events[0].record()
        kvd.gather_paged(pw.key_cache, pw.value_cache, pw.block_tables, pw.seq_lens, pw.seq_offset,
                         self.ko, self.vo, total_tokens=pw.total_tokens, dev_status=self.status)
        if gather_events is not None:
            gather_events[1].record()
        if events is not None:
            events[0][0].record()
        kvd.attend_paged(pw.q, pw.key_cache, pw.value_cache, pw.block_tables, pw.seq_lens,
                         pw.seq_offset, pw.scale, out=self.out, workspace=self.ws,
                         dev_status=self.status)
        if events is not None:
            events[0][1].record()

    def reset_if_wrapped(self, i):
        pass

    def launches_per_step(self):
        return 2 + (1 if self.splits else 0)

    def attend_bytes(self, i):
        return paged_attend_bytes(self.lengths, self.Hq, self.Hkv, self.D, self.elem, self.BS)

    def gather_bytes(self):
        return gather_bytes(self.lengths, self.Hkv, self.D, self.Hkv, self.D, self.elem, self.BS)

    def step_bytes(self, i):
        return self.attend_bytes(i) + self.gather_bytes()

    def tokens_per_step(self):
        return self.Q

    def e2e_setup(self):
        torch = self.torch
        self.h_q = torch.empty(self.pw.q.shape, dtype=self.pw.q.dtype, pin_memory=True).copy_(
            self.pw.q.cpu())
        self.h_out = torch.empty(self.pw.q.shape, dtype=self.pw.q.dtype, pin_memory=True)
        return self.h_q.numel() * 2, self.h_out.numel() * 2

    def e2e_step(self, i):
        self.pw.q.copy_(self.h_q, non_blocking=True)
        self.step(i)
        self.h_out.copy_(self.out, non_blocking=True)

    def config(self):
        return {"workload": "paged", "num_blocks": self.NB, "block_size": self.BS,
                "kv_heads": self.Hkv, "q_heads": self.Hq, "head_dim": self.D, "sequences": self.Q,
                "total_tokens": self.pw.total_tokens,
                "l2": f"inputs larger than L2: {2 * sum(self.lengths) * self.Hkv * self.D * 2 / 2**30:.2f}"
                      f" GiB of valid K/V rows per step vs {L2_BYTES // 2**20} MiB L2"}


def make_bench(name, torch, kvd, dev):
    if name == "paged":
        return PagedBench(torch, kvd, dev, None)
    return MaskedBench(name, torch, kvd, dev, None)


# ------------------------------------------------------------------- timing

def timed(torch, dist, fn, K, start=0):
    """Barrier + synchronize on both sides; CUDA events on the current stream."""
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(start, start + K):
        fn(i)
    e1.record()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    return e0.elapsed_time(e1)


def max_over_ranks(torch, dist, x):
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(torch, dist, x):
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def measure_workload(b, torch, dist, K, W, peak, main=False, clocks=None):
    """Warm-up, the timed K steps, a per-launch event pass for the attention
    kernel, and (main only) the end-to-end pass and the graph pass."""
    res = {}
    i = 0
    for _ in range(W):
        b.reset_if_wrapped(i)
        b.step(i)
        i += 1
    torch.cuda.synchronize()

    def run(j):
        b.reset_if_wrapped(j)
        b.step(j)

    if clocks is not None:
        clocks.start()
        soak_end = time.time() + 0.6  # fill a few sampling intervals before the timed steps
        while time.time() < soak_end:
            run(i)
            i += 1
            torch.cuda.synchronize()
    start = i
    ms = timed(torch, dist, run, K, start)
    if clocks is not None:
        res["clocks"] = clocks.stop()
    i += K
    step_bytes = sum(b.step_bytes(j) for j in range(start, start + K))
    ms = max_over_ranks(torch, dist, ms)
    total_bytes = sum_over_ranks(torch, dist, step_bytes)
    res["ms_per_step"] = ms / K
    res["gbs"] = total_bytes / (ms / 1e3) / 1e9
    res["tokens_per_s"] = sum_over_ranks(torch, dist, b.tokens_per_step() * K) / (ms / 1e3)

    # per-launch attention durations (CUDA events around each attention call)
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(b.layers)] for _ in range(K)]
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)] if isinstance(b, PagedBench) else None
    torch.cuda.synchronize()
    for k in range(K):
        b.reset_if_wrapped(i + k)
        if gev is not None:
            b.step(i + k, events=evs[k], gather_events=gev[k])
        else:
            b.step(i + k, events=evs[k])
    torch.cuda.synchronize()
    durs = [s.elapsed_time(e) for row in evs for (s, e) in row]
    attend_bytes = sum(b.attend_bytes(i + k) for k in range(K)) / K
    avg_ms = sum(durs) / len(durs)
    achieved = attend_bytes / (avg_ms / 1e3) / 1e9
    res["attend_ms_per_launch"] = avg_ms
    res["attend_gbs"] = achieved
    res["attend_frac"] = achieved / peak
    if gev is not None:
        gd = [s.elapsed_time(e) for (s, e) in gev]
        g_ms = sum(gd) / len(gd)
        res["gather_ms_per_launch"] = g_ms
        res["gather_gbs"] = b.gather_bytes() / (g_ms / 1e3) / 1e9
        res["gather_frac"] = res["gather_gbs"] / peak
    i += K
    res["_next_step"] = i
    return res


def measure_e2e(b, torch, dist, K, start):
    h2d, d2h = b.e2e_setup()
    for j in range(3):
        b.reset_if_wrapped(start + j)
        b.e2e_step(start + j)
    torch.cuda.synchronize()
    start += 3

    def run(j):
        b.reset_if_wrapped(j)
        b.e2e_step(j)

    ms = timed(torch, dist, run, K, start)
    ms = max_over_ranks(torch, dist, ms)
    total = sum_over_ranks(torch, dist, sum(b.step_bytes(j) for j in range(start, start + K)))
    return {"value": total / (ms / 1e3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms / K}, start + K


def measure_graph(b, torch, K, start):
    """The same steps captured once as a CUDA graph (launch overhead removed);
    the append position advances inside the graph."""
    if not isinstance(b, MaskedBench):
        return None
    pos = b.pos_table[0].clone()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for li, lay in enumerate(b.w.layers):
            b.kvd.append(lay.k_cache, lay.v_cache, lay.k_new, lay.v_new, pos, lay.mask, b.status)
            b.kvd.attend_masked(lay.q, lay.k_cache, lay.v_cache, lay.mask, lay.scale,
                                out=b.out[li], workspace=b.ws, dev_status=b.status)
        if b.cycle > 1:
            pos.add_(1)
    # restart the position cycle
    for lay in b.w.layers:
        if b.prompt is not None:
            lay.mask[:, b.prompt:] = 0
    pos.copy_(b.pos_table[0])
    n = min(K, b.cycle) if b.cycle > 1 else K
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    total = sum(b.step_bytes(j) for j in range(n))
    for lay in b.w.layers:
        if b.prompt is not None:
            lay.mask[:, b.prompt:] = 0
    return {"gbs": total / (ms / 1e3) / 1e9, "ms_per_step": ms / n,
            "tokens_per_s": b.tokens_per_step() * n / (ms / 1e3), "steps": n}


# -------------------------------------------------------------- CPU oracle

def oracle_rate(name, seconds, W_mod=None):
    """Time the fp64 oracle (append + attention, or gather + paged attention)
    on host copies of the workload, for about `seconds` of CPU work.
    Returns (GB/s of algorithmic bytes, cores, description of the sample)."""
    import torch

    import oracle
    import workloads
    oracle.build()
    if name == "paged":
        pw = workloads.paged(device="cpu")
        lengths = [int(x) for x in pw.lengths]
        kb = pw.key_cache.view(torch.int16).numpy()
        vb = pw.value_cache.view(torch.int16).numpy()
        done_bytes, t0, n = 0, time.perf_counter(), 0
        Q = len(lengths)
        while True:
            q = n % Q
            sl_q = torch.tensor([0, lengths[q]], dtype=torch.int32)
            bt_q = pw.block_tables[q:q + 1]
            oracle.gather_paged(kb, vb, bt_q, sl_q)
            oracle.attend_paged(pw.q[q:q + 1], pw.key_cache, pw.value_cache, bt_q, sl_q, None,
                                pw.scale)
            done_bytes += paged_attend_bytes([lengths[q]], 32, 8, 128, 2, 128) + \
                gather_bytes([lengths[q]], 8, 128, 8, 128, 2, 128)
            n += 1
            el = time.perf_counter() - t0
            if el >= seconds or n >= 4 * Q:
                break
        return done_bytes / el / 1e9, oracle.threads(), f"{n} sequences of the paged workload " \
            f"(gather + paged attention), {el:.1f} s"
    if name == "npuw":
        w = workloads.npuw(device="cpu", layers=4)
    elif name == "gqa":
        w = workloads.gqa(device="cpu", layers=1)
    else:
        w = workloads.long(device="cpu", layers=1)
    done_bytes, t0, n = 0, time.perf_counter(), 0
    caches = [(l.k_cache.view(torch.int16).numpy().copy(), l.v_cache.view(torch.int16).numpy().copy(),
               l.mask.numpy().copy()) for l in w.layers]
    while True:
        li = n % len(w.layers)
        lay = w.layers[li]
        kh, vh, mh = caches[li]
        oracle.append(kh, vh, lay.k_new, lay.v_new, lay.pos, mh)
        oracle.attend_masked(lay.q, torch.from_numpy(kh).view(torch.bfloat16),
                             torch.from_numpy(vh).view(torch.bfloat16), torch.from_numpy(mh),
                             lay.scale)
        L = [int(x) for x in lay.lengths]
        done_bytes += masked_attend_bytes(L, w.Hq, w.Hkv, w.C, w.D, 2) + append_bytes(w.B, w.Hkv, w.D, 2)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return done_bytes / el / 1e9, oracle.threads(), \
        f"{n} layer-steps (append + attention) of the {name} workload, {el:.1f} s"


# -------------------------------------------------------------------- main

METRIC = "decode-attention KV GB/s and % of GB300 HBM peak; decode tokens/sec at 1 GPU"


def reference_arm(args, rank, world):
    """The reference arm: the fp64 CPU oracle as it stands, on the host cores,
    each step a bounded sample of the workload."""
    if rank != 0:
        return 0
    per_step = max(0.5, min(5.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_rate(args.workload, per_step * 0.2)
    rates = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        r, cores, sample = oracle_rate(args.workload, per_step)
        rates.append(r)
    el = time.perf_counter() - t0
    value = statistics.mean(rates)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": f"per step: {sample}"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kvd", choices=["kvd", "reference"])
    ap.add_argument("--workload", default="npuw", choices=["npuw", "gqa", "long", "paged"])
    ap.add_argument("--no-others", action="store_true", help="skip the other workloads")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return reference_arm(args, rank, world)

    import torch
    dist = None
    if world > 1:
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl")
        dist = tdist
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    from decode_attention_kv_gb300 import _build, kvd
    if rank == 0 or world == 1:
        _build.build()
    if dist is not None:
        dist.barrier()
    kvd.load()
    peak, peak_src = measured_peak()

    b = make_bench(args.workload, torch, kvd, dev)
    clocks = ClockSampler(bus_id_of(torch, dev))
    res = measure_workload(b, torch, dist, args.steps, args.warmup, peak, main=True, clocks=clocks)
    e2e, nxt = measure_e2e(b, torch, dist, args.steps, res["_next_step"])
    graph = measure_graph(b, torch, args.steps, nxt) if world == 1 else None
    st = int(b.status.item())
    if st != 0:
        raise RuntimeError(f"device status {st} during the benchmark")

    traffic = None
    key = (args.workload, kernel_source_hash())
    if key in NCU_TRAFFIC:
        traffic = NCU_TRAFFIC[key]

    others = {}
    if not args.no_others:
        for name in ("gqa", "long", "paged", "npuw"):
            if name == args.workload:
                continue
            ob = make_bench(name, torch, kvd, dev)
            r = measure_workload(ob, torch, dist, max(5, min(args.steps, 20)), 3, peak)
            ent = {"gbs": r["gbs"], "frac_of_" + peak_src: r["gbs"] / peak,
                   "ms_per_step": r["ms_per_step"], "tokens_per_s": r["tokens_per_s"],
                   "attend_gbs": r["attend_gbs"], "attend_frac": r["attend_frac"],
                   "attend_ms_per_launch": r["attend_ms_per_launch"], "config": ob.config()}
            if "gather_gbs" in r:
                ent.update(gather_gbs=r["gather_gbs"], gather_frac=r["gather_frac"],
                           gather_ms_per_launch=r["gather_ms_per_launch"])
            others[name] = ent
            del ob
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1:
        try:
            v, cores, sample = oracle_rate(args.workload, args.cpu_seconds)
            cpu = {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample}
        except Exception as e:  # the oracle needs gcc on the host
            cpu = {"unavailable": f"{type(e).__name__}: {e}"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": res["gbs"], "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": b.config(),
            "frac_of_hbm_peak": res["gbs"] / peak, "peak_source": peak_src,
            "decode_tokens_per_s": res["tokens_per_s"],
            "roofline": {"bound": "hbm", "achieved": res["attend_gbs"], "peak": peak, "unit": "GB/s",
                         "frac": res["attend_frac"], "traffic": traffic,
                         "kernel": "attention (split-KV kernel + combine), per layer",
                         "ms_per_launch": res["attend_ms_per_launch"],
                         "peak_source": peak_src},
            "e2e": e2e, "gpu_launches": b.launches_per_step() * args.steps,
            "clocks": res.get("clocks"), "cuda_graph": graph, "cpu_baseline": cpu,
            "workloads": others, "kernel_hash": kernel_source_hash(),
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
