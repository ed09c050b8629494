#!/usr/bin/env python
"""Decode-attention benchmark: KV GB/s, fraction of the HBM roofline, and
decode tokens/s on GB300, through libkvd's C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W]
                    [--workload gqa|long|paged|paged_gather|npuw|indexed|window|gqa_fp8|gqa_fp4|
                                paged_fp8|paged_fp4]
    python bench.py --impl reference ...     # the fp64 CPU oracle as the reference arm

A step is one decode step of the workload: for the static-buffer workloads,
every layer appends the step's K/V row and runs masked split-KV attention
(+ the log-sum-exp combine); for the paged workload, the paged gather and the
paged attention over the whole cache.  ``value`` is algorithmic bytes per
second (valid K/V rows, mask, q and out, appended rows; no padding and no
split scratch), whole job over all ranks.  Multi-GPU runs are independent
replicas (weak scaling, no data-path collective).

The main line is the batched-GQA workload (16 sequences, 32/8 heads,
capacity 8192, 32 layers: the largest single-GPU configuration, one of the
two the 75 % HBM target is stated on).  The same measurement of every other
workload -- long context (the other target), the paged cache, the
1152-slot static buffer, top-k index lists, a sliding window and quantised
caches -- goes under "workloads", each with its own roofline, CPU baseline
and end-to-end figure.
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024

# dram__bytes_read.sum + dram__bytes_write.sum of one launch of each
# workload's attention kernel from an ncu capture, keyed by the hash of the
# kernel sources it was taken on: reported only while the sources still hash
# to that revision, else null.
NCU_TRAFFIC = {
    ("npuw", "f081e2091b51ce68"): 17892096,  # attend_small_kernel, tensor-core consumers, 1152-slot buffer
    ("gqa", "f081e2091b51ce68"): 212512000,  # attend_kernel, tensor-core consumers, batched GQA
    ("long", "f081e2091b51ce68"): 540379648,  # attend_kernel, CUDA-core consumers, 32768 slots
    ("paged", "f081e2091b51ce68"): 521817088,  # attend_kernel, paged mode
    ("indexed", "f081e2091b51ce68"): 122609408,  # attend_kernel, index-list mode, gather warp
    ("window", "f081e2091b51ce68"): 67960832,  # attend_kernel, window entry, 4096-slot window
    ("gqa_fp8", "f081e2091b51ce68"): 120547328,  # attend_kernel, E4M3 consumers
    ("gqa_fp4", "f081e2091b51ce68"): 66348288,  # attend_kernel, E2M1 consumers
    ("paged_fp8", "f081e2091b51ce68"): 308250880,  # attend_kernel, paged mode, E4M3 rows
    ("paged_fp4", "f081e2091b51ce68"): 167010816,  # attend_kernel, paged mode, E2M1 rows
}

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


def paged_quant_attend_bytes(lengths, Hq, Hkv, D, row, BS):
    """Valid quantised K and V rows (`row` bytes each), the block-table
    entries the sequences use, the cumsum, bf16 q and out."""
    Q = len(lengths)
    rows = sum(int(L) for L in lengths)
    entries = sum((int(L) + BS - 1) // BS for L in lengths)
    return rows * Hkv * row * 2 + entries * 4 + (Q + 1) * 4 + 2 * Q * Hq * D * 2


def gather_bytes(lengths, Hk, Dk, Hv, Dv, elem, BS):
    """Read + write of every gathered row, plus the indices used."""
    Q = len(lengths)
    T = sum(int(L) for L in lengths)
    entries = sum((int(L) + BS - 1) // BS for L in lengths)
    return 2 * T * (Hk * Dk + Hv * Dv) * elem + entries * 4 + (Q + 1) * 4


def quant_attend_bytes(lengths, Hq, Hkv, C, D, row):
    """Valid quantised K and V rows (codes + fp32 scale + zero pad, `row`
    bytes each: D + 16 for E4M3, D/2 + 16 for E2M1), the mask row, bf16 q
    and out."""
    B = len(lengths)
    return (sum(int(L) for L in lengths) * Hkv * row * 2 + B * C + 2 * B * Hq * D * 2)


def quant_append_bytes(B, Hkv, D, row):
    """bf16 new K and V rows read, their quantised rows written."""
    return 2 * B * Hkv * (D * 2 + row)


def indexed_attend_bytes(listed, topk, Hq, Hkv, D, elem):
    """The listed K and V rows of every kv head, the index lists (topk int32
    entries per query, padding included), q and out."""
    B = len(listed)
    return (sum(int(n) for n in listed) * Hkv * D * 2 * elem + B * topk * 4
            + 2 * B * Hq * D * elem)


def attention_flops(lengths, Hq, D):
    return 4 * sum(int(L) for L in lengths) * Hq * D


def kernel_source_hash():
    """Hash of the CUDA sources' code (comments and blank space left out, so
    that documentation edits keep a profile's counters attached)."""
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "decode_attention_kv_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name)) as f:
                code = f.read()
            code = re.sub(r"/\*.*?\*/", "", code, flags=re.S)
            code = re.sub(r"//[^\n]*", "", code)
            code = re.sub(r"\s+", " ", code)
            h.update(name.encode() + code.encode())
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

# Layer caches of each static-buffer workload (the workload generators' defaults).
LAYERS = {"npuw": 32, "gqa": 32, "long": 8, "window": 8, "gqa_fp8": 32, "gqa_fp4": 32,
          "indexed": 32}


def masked_config(name, w, layers, lengths0):
    """The config block of a static-buffer workload (both arms print it)."""
    elem = 2
    cache = layers * 2 * w.B * w.Hkv * w.C * w.D * elem
    L = lengths0
    c = {"workload": name, "batch": w.B, "q_heads": w.Hq, "kv_heads": w.Hkv,
         "head_dim": w.D, "capacity": w.C, "layers": layers, "dtype": "bf16",
         "valid_len_step0": (L if len(L) <= 4 else
                             {"min": min(L), "max": max(L), "mean": sum(L) / len(L)}),
         "l2": f"inputs larger than L2: {cache / 2**30:.2f} GiB of layer caches rotated "
               f"per step vs {L2_BYTES // 2**20} MiB L2"}
    if w.window:
        rows = layers * 2 * w.Hkv * sum(min(x, w.window) for x in L) * w.D * elem
        c.update({"window": w.window,
                  "attention": "kvd_append_attend_window (splits over each row's window)",
                  "l2": f"inputs larger than L2: the windows' K/V rows of the {layers} layers "
                        f"read per step are {rows / 2**20:.0f} MiB vs {L2_BYTES // 2**20} MiB L2"})
    if name == "indexed":
        listed = [min(IndexedBench.TOPK, x) for x in L]
        c.update({"topk": IndexedBench.TOPK,
                  "listed_per_entry": {"min": min(listed), "max": max(listed)}})
    if name in QUANT_FORMATS:
        fmt = QUANT_FORMATS[name]
        row = quant_row_bytes(name, w.D)
        cache = layers * 2 * w.B * w.Hkv * w.C * row
        c.update({"dtype": f"{fmt.lower()} K/V, bf16 q/out",
                  "kv_format": f"{fmt} codes + fp32 row scale, {row}-byte rows",
                  "l2": f"inputs larger than L2: {cache / 2**30:.2f} GiB of layer caches "
                        f"rotated per step vs {L2_BYTES // 2**20} MiB L2"})
    return c


def paged_config(pw, name="paged"):
    NB, BS, Hkv, RB = pw.key_cache.shape
    Q, Hq, D = pw.q.shape
    lengths = [int(x) for x in pw.lengths]
    row = pw.key_cache.element_size() * RB  # bytes of one K (or V) row of one kv head
    rows = 2 * sum(lengths) * Hkv * row
    cache = 2 * pw.key_cache.numel() * pw.key_cache.element_size()
    c = {"workload": name, "num_blocks": NB, "block_size": BS, "kv_heads": Hkv,
         "q_heads": Hq, "head_dim": D, "sequences": Q, "dtype": "bf16",
         "total_tokens": pw.total_tokens,
         "l2": f"inputs larger than L2: {rows / 2**30:.2f} GiB of valid K/V rows per step "
               f"(of a {cache / 2**30:.1f} GiB cache) vs {L2_BYTES // 2**20} MiB L2"}
    if name in PAGED_QUANT:
        fmt = PAGED_QUANT[name]
        c.update({"dtype": f"{fmt.lower()} K/V, bf16 q/out",
                  "kv_format": f"{fmt} codes + fp32 row scale, {row}-byte rows"})
    return c


def workload_config(name):
    """The config block of a workload, built from host copies of its inputs
    (the reference arm prints the same block as the GPU arm)."""
    import workloads
    if name in ("paged", "paged_gather"):
        return paged_config(workloads.paged(device="cpu"), name)
    if name in PAGED_QUANT:
        return paged_config(workloads.paged_quant(name[-3:], device="cpu"), name)
    gen = {"indexed": "gqa"}.get(name, name)
    w = getattr(workloads, gen)(device="cpu", layers=1)
    return masked_config(name, w, LAYERS[name], [int(x) for x in w.layers[0].lengths])


ROW_PAD = 16  # quantised rows: codes, fp32 scale, 12 zero bytes
QUANT_FORMATS = {"gqa_fp8": "E4M3", "gqa_fp4": "E2M1"}
# the paged workload over quantised rows
PAGED_QUANT = {"paged_fp8": "E4M3", "paged_fp4": "E2M1"}
KV_FORMATS = {**QUANT_FORMATS, **PAGED_QUANT}


def quant_row_bytes(name, D):
    """Bytes of one quantised K/V row: D E4M3 codes or D/2 bytes of E2M1
    code pairs, then the 16-byte scale field."""
    return (D if name == "gqa_fp8" else D // 2) + ROW_PAD


def attention_kernel_name(kind, plan, g, mode="masked", fused=False):
    """The kernel that runs a workload's attention, as the launch list names it."""
    if plan.splits == 0:
        return f"attend_small_kernel ({kind} consumers; one CTA per split, cluster merge)"
    tail = ", fused append" if fused else ""
    if plan.splits == 1:
        comb = ", rows written directly"
    else:
        comb = f", {plan.splits} splits, then combine_kernel"
    return f"attend_kernel ({kind} consumers, {mode} mode, g={g}{tail}{comb})"


class MaskedBench:
    """Static-buffer workload: every layer appends the step's K/V row and runs
    masked split-KV attention.  The 1152-slot buffer advances its append slot
    each step (1024, 1025, ... 1151, then the response part is cleared and the
    cycle restarts); the other workloads re-append at the last valid slot."""

    def __init__(self, name, torch, kvd, dev, layers=None):
        import workloads
        self.torch, self.kvd, self.dev, self.name = torch, kvd, dev, name
        kw = {} if layers is None else {"layers": layers}
        if name == "npuw":
            w = workloads.npuw(device=dev, **kw)
            self.cycle, self.prompt = 128, 1024
        elif name == "gqa":
            w = workloads.gqa(device=dev, **kw)
            self.cycle, self.prompt = 1, None
        elif name == "long":
            w = workloads.long(device=dev, **kw)
            self.cycle, self.prompt = 1, None
        elif name == "window":
            w = workloads.window(device=dev, **kw)
            self.cycle, self.prompt = 1, None
        elif name in ("gqa_fp8", "gqa_fp4"):
            w = getattr(workloads, name)(device=dev, **kw)
            self.cycle, self.prompt = 1, None
        else:
            raise ValueError(name)
        self.w = w
        lay0 = w.layers[0]
        self.B, self.Hq, self.Hkv, self.C, self.D = w.B, w.Hq, w.Hkv, w.C, w.D
        self.elem = 2
        self.layers = len(w.layers)
        base = lay0.pos.to(torch.int64)
        # append slot of step j: base + (j mod cycle)
        self.pos_table = torch.stack([(base + i).to(torch.int32) for i in range(self.cycle)]).to(dev)
        self.gpos = self.pos_table[0].clone()
        # the sliding window runs through the window entries (splits over each
        # row's window only)
        self.win = w.window
        if self.win:
            need = kvd.attend_window_workspace_bytes(self.B, self.Hq, self.Hkv, self.C, self.D,
                                                     self.win)
        else:
            need = kvd.attend_masked_workspace_bytes(self.B, self.Hq, self.Hkv, self.C, self.D)
        self.ws = kvd.workspace(need, dev)
        self.out = [torch.empty_like(l.q) for l in w.layers]
        self.status = kvd.status_tensor(dev)
        self.lengths0 = [int(x) for x in lay0.lengths]
        self.graph = None

    def reset_cycle(self):
        if self.prompt is not None:
            for lay in self.w.layers:
                lay.mask[:, self.prompt:] = 0
        self.gpos.copy_(self.pos_table[0])

    def _wrap(self, j):
        if self.cycle > 1 and j > 0 and j % self.cycle == 0:
            self.reset_cycle()

    def _layer(self, li, lay, pos):
        """The layer's decode step: append + attention in one call (one
        launch and the combine)."""
        if self.win:
            self.kvd.append_attend_window(lay.q, lay.k_cache, lay.v_cache, lay.mask, lay.k_new,
                                          lay.v_new, pos, self.win, lay.scale, out=self.out[li],
                                          workspace=self.ws, dev_status=self.status)
            return
        self.kvd.append_attend_masked(lay.q, lay.k_cache, lay.v_cache, lay.mask, lay.k_new,
                                      lay.v_new, pos, lay.scale, out=self.out[li],
                                      workspace=self.ws, dev_status=self.status)

    def eager_run(self, j, timing=False):
        """One step, one binding call per layer; with timing, CUDA events
        around each call."""
        torch = self.torch
        self._wrap(j)
        pos = self.pos_table[j % self.cycle]
        evs = []
        for li, lay in enumerate(self.w.layers):
            if timing:
                e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
                e[0].record()
            self._layer(li, lay, pos)
            if timing:
                e[1].record()
                evs.append(("attend", e[0], e[1]))
        return evs

    def capture(self):
        """The whole step as one CUDA graph; the append slot lives in a device
        word that the graph itself advances."""
        torch = self.torch
        self.reset_cycle()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for li, lay in enumerate(self.w.layers):
                self._layer(li, lay, self.gpos)
            if self.cycle > 1:
                self.gpos.add_(1)
        self.graph = g
        self.reset_cycle()

    def graph_run(self, j):
        self._wrap(j)
        self.graph.replay()

    def copy_setup(self):
        """copy_kvcache inputs for the static-buffer workload with a prompt:
        prefill caches of capacity `prompt` holding the decode caches' prompt
        rows, so that the hand-over rewrites identical rows and the prefix
        mask of the prompt (the state reset_cycle leaves)."""
        if self.prompt is None:
            return False
        torch = self.torch
        self.pk = [l.k_cache[:, :, :self.prompt].contiguous() for l in self.w.layers]
        self.pv = [l.v_cache[:, :, :self.prompt].contiguous() for l in self.w.layers]
        self.cn = torch.full((self.B,), self.prompt, dtype=torch.int32, device=self.dev)
        ws = self.w.layers
        self.pcopy = self.kvd.PrefixCopy(self.pk, self.pv, [l.k_cache for l in ws],
                                         [l.v_cache for l in ws], [l.mask for l in ws])
        return True

    def copy_run(self):
        self.pcopy.run(self.cn, self.status)

    def copy_bytes(self):
        """Read + write of every copied K and V row of every layer."""
        return 4 * self.layers * self.B * self.Hkv * self.prompt * self.D * self.elem

    def launches_per_step(self):
        """One fused append + attention call per layer: one launch (the
        small-launch kernel) or two (the split kernel and the combine)."""
        if self.win:
            return self.layers * self.attention_plan().launches
        return self.layers * self.kvd.attend_masked_launches(self.B, self.Hq, self.Hkv, self.C,
                                                             self.D)

    def lengths_at(self, j):
        return [L + (j % self.cycle) for L in self.lengths0]

    def rows_at(self, j):
        """Rows each batch entry attends to (the window's, if it has one)."""
        L = self.lengths_at(j)
        return [min(x, self.w.window) for x in L] if self.w.window else L

    def attend_bytes(self, j):
        return masked_attend_bytes(self.rows_at(j), self.Hq, self.Hkv, self.C, self.D, self.elem)

    def step_bytes(self, j):
        return self.layers * (self.attend_bytes(j) + append_bytes(self.B, self.Hkv, self.D, self.elem))

    def tokens_per_step(self):
        return self.B

    def flops_per_step(self):
        """Attention FLOPs of one step (reported, not bounding): 4 per query
        head, attended slot and dim."""
        return self.layers * attention_flops(self.rows_at(0), self.Hq, self.D)

    def e2e_setup(self):
        """End to end as a caller runs the step: every layer's q and new K/V
        rows live in one device staging buffer filled by one host-to-device
        copy per step (plus the step's positions), the step's kernels run as
        one CUDA graph of the binding's calls, and every layer's output comes
        back in one device-to-host copy."""
        torch = self.torch
        L = self.w.layers
        ins = [l.q for l in L] + [l.k_new for l in L] + [l.v_new for l in L]
        self.d_in = torch.empty(sum(t.numel() for t in ins), dtype=ins[0].dtype, device=self.dev)
        views, off = [], 0
        for t in ins:
            n = t.numel()
            self.d_in[off:off + n].copy_(t.reshape(-1))
            views.append(self.d_in[off:off + n].view(t.shape))
            off += n
        nl = len(L)
        for li, lay in enumerate(L):
            lay.q, lay.k_new, lay.v_new = views[li], views[nl + li], views[2 * nl + li]
        self.d_out = torch.empty(sum(o.numel() for o in self.out), dtype=self.out[0].dtype,
                                 device=self.dev)
        self.out = [self.d_out[i * o.numel():(i + 1) * o.numel()].view(o.shape)
                    for i, o in enumerate(self.out)]
        self.h_in = torch.empty(self.d_in.shape, dtype=self.d_in.dtype, pin_memory=True)
        self.h_in.copy_(self.d_in.cpu())
        self.h_out = torch.empty(self.d_out.shape, dtype=self.d_out.dtype, pin_memory=True)
        self.h_pos = torch.empty(self.pos_table.shape, dtype=torch.int32, pin_memory=True)
        self.h_pos.copy_(self.pos_table.cpu())
        self.capture()  # the graph now reads the staging views and writes d_out
        h2d = self.h_in.numel() * self.h_in.element_size() + self.B * 4
        d2h = self.h_out.numel() * self.h_out.element_size()
        return h2d, d2h

    def e2e_step(self, j):
        """Host buffers in, the step, host buffers out."""
        self._wrap(j)
        self.gpos.copy_(self.h_pos[j % self.cycle], non_blocking=True)
        self.d_in.copy_(self.h_in, non_blocking=True)
        self.graph.replay()
        self.h_out.copy_(self.d_out, non_blocking=True)

    def attention_plan(self):
        if self.win:
            return self.kvd.attend_window_plan(self.B, self.Hq, self.Hkv, self.C, self.D, self.win)
        return self.kvd.attend_masked_plan(self.B, self.Hq, self.Hkv, self.C, self.D)

    def kernel_name(self):
        g = self.Hq // self.Hkv
        plan = self.attention_plan()
        # the one-launch kernel takes the tensor-core consumers for every bf16
        # group width, the split kernel from 4 query heads per kv head
        kind = "tensor-core" if (g >= 4 or plan.splits == 0) else "CUDA-core"
        return attention_kernel_name(kind, plan, g, mode="window" if self.win else "masked",
                                     fused=True)

    def aux_ops(self):
        """The step's launches other than the attention kernel, per layer:
        the combine, when the plan splits rows (the append runs inside the
        attention launch)."""
        plan = self.attention_plan()
        part = self.kvd.workspace_partials(self.ws, plan, self.B * self.Hq, self.D)
        if part is None or plan.launches < 2:
            return {}
        po, pl = part
        return {"combine": lambda li: self.kvd.combine(po, pl, out=self.out[li].view(-1, self.D))}

    def config(self):
        return masked_config(self.name, self.w, self.layers, self.lengths0)


class PagedBench:
    """Paged workload over the whole 8192-block cache, in one of two steps:
    ``paged`` = one paged decode step (every sequence appends its new token
    into its block, then its query attends over its blocks through the block
    tables), ``paged_gather`` = gather_pa_kv_cache into contiguous rows.  The two are separate steps: a decode step reads the
    paged cache directly; the gather serves consumers of the contiguous layout
    (and, run right before the attention, would leave it a cache full of the
    gather's dirty lines to write back)."""

    def __init__(self, torch, kvd, dev, mode="paged"):
        import workloads
        self.torch, self.kvd, self.dev, self.name = torch, kvd, dev, mode
        self.gather_mode = mode == "paged_gather"
        pw = workloads.paged(device=dev)
        self.pw = pw
        self.Q, self.Hq, self.D = pw.q.shape
        self.NB, self.BS, self.Hkv, _ = pw.key_cache.shape
        self.elem = 2
        self.layers = 1
        self.lengths = [int(x) for x in pw.lengths]
        if self.gather_mode:
            self.ko = torch.empty((pw.total_tokens, self.Hkv, self.D), dtype=torch.bfloat16,
                                  device=dev)
            self.vo = torch.empty_like(self.ko)
        self.out = torch.empty_like(pw.q)
        cols = pw.block_tables.shape[1]
        need = kvd.attend_paged_workspace_bytes(self.Q, self.Hq, self.Hkv, self.BS, cols, self.D)
        self.ws = kvd.workspace(need, dev)
        self.status = kvd.status_tensor(dev)
        self.graph = None

    def reset_cycle(self):
        pass

    def _gather(self):
        pw = self.pw
        self.kvd.gather_paged(pw.key_cache, pw.value_cache, pw.block_tables, pw.seq_lens,
                              pw.seq_offset, self.ko, self.vo, total_tokens=pw.total_tokens,
                              dev_status=self.status)

    def _attend(self):
        pw = self.pw
        self.kvd.attend_paged(pw.q, pw.key_cache, pw.value_cache, pw.block_tables, pw.seq_lens,
                              pw.seq_offset, pw.scale, out=self.out, workspace=self.ws,
                              dev_status=self.status)

    def _append(self):
        pw = self.pw
        self.kvd.append_paged(pw.key_cache, pw.value_cache, pw.block_tables, pw.seq_offset,
                              pw.k_new, pw.v_new, pw.pos, dev_status=self.status)

    def _step(self):
        if self.gather_mode:
            self._gather()
        else:
            self._append()
            self._attend()

    def eager_run(self, j, timing=False):
        """One step; with timing, CUDA events around the call (its main
        kernel: the attention, or the gather)."""
        torch = self.torch
        if not timing:
            self._step()
            return []
        if self.gather_mode:
            e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            e[0].record()
            self._gather()
            e[1].record()
            return [("attend", e[0], e[1])]
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record()
        self._append()
        e[1].record()
        self._attend()
        e[2].record()
        return [("append", e[0], e[1]), ("attend", e[1], e[2])]

    def capture(self):
        torch = self.torch
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self._step()
        self.graph = g

    def graph_run(self, j):
        self.graph.replay()

    def launches_per_step(self):
        return 1 if self.gather_mode else 1 + self.attention_plan().launches

    def attend_bytes(self, j):
        """Algorithmic bytes of the step's main kernel."""
        if self.gather_mode:
            return self.gather_bytes()
        return paged_attend_bytes(self.lengths, self.Hq, self.Hkv, self.D, self.elem, self.BS)

    def gather_bytes(self):
        return gather_bytes(self.lengths, self.Hkv, self.D, self.Hkv, self.D, self.elem, self.BS)

    def step_bytes(self, j):
        if self.gather_mode:
            return self.attend_bytes(j)
        return self.attend_bytes(j) + append_bytes(self.Q, self.Hkv, self.D, self.elem)

    def tokens_per_step(self):
        return 0 if self.gather_mode else self.Q

    def flops_per_step(self):
        return 0 if self.gather_mode else attention_flops(self.lengths, self.Hq, self.D)

    def e2e_setup(self):
        """Attention: the step's queries in from pinned host memory, the
        outputs back.  Gather: the step's block tables, cumsum lengths and
        offsets in, the device status word back (the gathered rows stay on
        the device for their consumer)."""
        torch = self.torch
        pw = self.pw
        if self.gather_mode:
            self.h_in = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t.cpu())
                         for t in (pw.block_tables, pw.seq_lens, pw.seq_offset)]
            self.h_st = torch.empty(1, dtype=torch.int32, pin_memory=True)
            return sum(t.numel() * 4 for t in self.h_in), 4
        self.h_in = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t.cpu())
                     for t in (pw.q, pw.k_new, pw.v_new, pw.pos)]
        self.h_out = torch.empty(pw.q.shape, dtype=pw.q.dtype, pin_memory=True)
        return (sum(t.numel() * t.element_size() for t in self.h_in),
                self.h_out.numel() * self.h_out.element_size())

    def e2e_step(self, j):
        pw = self.pw
        if self.gather_mode:
            for d, h in zip((pw.block_tables, pw.seq_lens, pw.seq_offset), self.h_in):
                d.copy_(h, non_blocking=True)
            self._gather()
            self.h_st.copy_(self.status, non_blocking=True)
            return
        for d, h in zip((pw.q, pw.k_new, pw.v_new, pw.pos), self.h_in):
            d.copy_(h, non_blocking=True)
        self._append()
        self._attend()
        self.h_out.copy_(self.out, non_blocking=True)

    def attention_plan(self):
        cols = self.pw.block_tables.shape[1]
        return self.kvd.attend_paged_plan(self.Q, self.Hq, self.Hkv, self.BS, cols, self.D)

    def kernel_name(self):
        if self.gather_mode:
            return "gather_kernel (16-byte vectors, block-table indirection)"
        return attention_kernel_name("tensor-core", self.attention_plan(), self.Hq // self.Hkv,
                                     mode="paged")

    def aux_ops(self):
        """The paged append and the combine around the paged attention (the
        gather step is one launch)."""
        if self.gather_mode:
            return {}
        ops = {"append": lambda li: self._append()}
        plan = self.attention_plan()
        part = self.kvd.workspace_partials(self.ws, plan, self.Q * self.Hq, self.D)
        if part is not None and plan.launches > 1:
            po, pl = part
            ops["combine"] = lambda li: self.kvd.combine(po, pl, out=self.out.view(-1, self.D))
        return ops

    def config(self):
        return paged_config(self.pw, self.name)


class PagedQuantBench(PagedBench):
    """The paged decode step over quantised caches: every sequence's new K/V
    row quantised into its block (kvd_append_paged_fp8 / _fp4), then the
    paged attention over the quantised rows (kvd_attend_paged_fp8 / _fp4);
    the paged workload's sequences and tables."""

    def __init__(self, name, torch, kvd, dev):
        import workloads
        self.torch, self.kvd, self.dev, self.name = torch, kvd, dev, name
        self.fmt = name[-3:]
        self.gather_mode = False
        pw = workloads.paged_quant(self.fmt, device=dev)
        self.pw = pw
        self.Q, self.Hq, self.D = pw.q.shape
        self.NB, self.BS, self.Hkv, self.row = pw.key_cache.shape
        self.elem = 2
        self.layers = 1
        self.lengths = [int(x) for x in pw.lengths]
        self.out = torch.empty_like(pw.q)
        cols = pw.block_tables.shape[1]
        need = kvd.attend_paged_quant_workspace_bytes(self.fmt, self.Q, self.Hq, self.Hkv,
                                                      self.BS, cols, self.D)
        self.ws = kvd.workspace(need, dev)
        self.status = kvd.status_tensor(dev)
        self.graph = None

    def _attend(self):
        pw = self.pw
        self.kvd.attend_paged_quant(self.fmt, pw.q, pw.key_cache, pw.value_cache, pw.block_tables,
                                    pw.seq_lens, pw.seq_offset, pw.scale, out=self.out,
                                    workspace=self.ws, dev_status=self.status)

    def _append(self):
        pw = self.pw
        append = self.kvd.append_paged_fp8 if self.fmt == "fp8" else self.kvd.append_paged_fp4
        append(pw.key_cache, pw.value_cache, pw.block_tables, pw.seq_offset, pw.k_new, pw.v_new,
               pw.pos, dev_status=self.status)

    def attend_bytes(self, j):
        return paged_quant_attend_bytes(self.lengths, self.Hq, self.Hkv, self.D, self.row, self.BS)

    def step_bytes(self, j):
        return self.attend_bytes(j) + quant_append_bytes(self.Q, self.Hkv, self.D, self.row)

    def attention_plan(self):
        cols = self.pw.block_tables.shape[1]
        return self.kvd.attend_paged_quant_plan(self.fmt, self.Q, self.Hq, self.Hkv, self.BS,
                                                cols, self.D)

    def kernel_name(self):
        return attention_kernel_name(f"{PAGED_QUANT[self.name]} tensor-core", self.attention_plan(),
                                     self.Hq // self.Hkv, mode="paged")


class IndexedBench(MaskedBench):
    """Top-k sparse decode on the batched-GQA caches: every layer appends the
    step's K/V row, then attends over 2048 slots per batch entry drawn once
    (seeded, unique, from the entry's valid prefix; -1 pads a shorter
    prefix) -- the index-list attention of sparse (top-k) attention."""

    TOPK = 2048

    def __init__(self, torch, kvd, dev, layers=None):
        import workloads
        super().__init__("gqa", torch, kvd, dev, layers)
        self.name = "indexed"
        self.indices = workloads.index_lists(self.lengths0, self.TOPK).to(dev)
        self.listed = [min(self.TOPK, L) for L in self.lengths0]
        need = kvd.attend_indexed_workspace_bytes(self.B, self.Hq, self.Hkv, self.TOPK, self.D)
        self.ws = kvd.workspace(need, dev)

    def _layer(self, li, lay, pos):
        self.kvd.append(lay.k_cache, lay.v_cache, lay.k_new, lay.v_new, pos, None, self.status)
        self.kvd.attend_indexed(lay.q, lay.k_cache, lay.v_cache, self.indices, lay.scale,
                                out=self.out[li], workspace=self.ws, dev_status=self.status)

    def eager_run(self, j, timing=False):
        torch, kvd = self.torch, self.kvd
        pos = self.pos_table[j % self.cycle]
        evs = []
        for li, lay in enumerate(self.w.layers):
            if timing:
                e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                e[0].record()
            kvd.append(lay.k_cache, lay.v_cache, lay.k_new, lay.v_new, pos, None, self.status)
            if timing:
                e[1].record()
            kvd.attend_indexed(lay.q, lay.k_cache, lay.v_cache, self.indices, lay.scale,
                               out=self.out[li], workspace=self.ws, dev_status=self.status)
            if timing:
                e[2].record()
                evs += [("append", e[0], e[1]), ("attend", e[1], e[2])]
        return evs

    def launches_per_step(self):
        return self.layers * (1 + self.attention_plan().launches)  # append, attention (+ combine)

    def flops_per_step(self):
        return self.layers * attention_flops(self.listed, self.Hq, self.D)

    def attend_bytes(self, j):
        return indexed_attend_bytes(self.listed, self.TOPK, self.Hq, self.Hkv, self.D, self.elem)

    def copy_setup(self):
        return False

    def attention_plan(self):
        return self.kvd.attend_indexed_plan(self.B, self.Hq, self.Hkv, self.TOPK, self.D)

    def kernel_name(self):
        return attention_kernel_name("tensor-core", self.attention_plan(), self.Hq // self.Hkv,
                                     mode="index-list")

    def aux_ops(self):
        """The append kernel and the combine."""
        lays = self.w.layers
        ops = {"append": lambda li: self.kvd.append(lays[li].k_cache, lays[li].v_cache,
                                                    lays[li].k_new, lays[li].v_new, self.gpos,
                                                    None, self.status)}
        plan = self.attention_plan()
        part = self.kvd.workspace_partials(self.ws, plan, self.B * self.Hq, self.D)
        if part is not None and plan.launches > 1:
            po, pl = part
            ops["combine"] = lambda li: self.kvd.combine(po, pl, out=self.out[li].view(-1, self.D))
        return ops

    def config(self):
        return masked_config("indexed", self.w, self.layers, self.lengths0)


class QuantBench(MaskedBench):
    """The batched-GQA step over quantised caches (rows of 128 E4M3 codes, or
    64 bytes of E2M1 code pairs, + fp32 scale + 12 zero bytes): every layer
    quantises and appends the step's bf16 K/V rows, then attends over the
    quantised rows."""

    def __init__(self, name, torch, kvd, dev, layers=None):
        super().__init__(name, torch, kvd, dev, layers)
        self.fmt = "fp8" if name == "gqa_fp8" else "fp4"
        self.row = quant_row_bytes(name, self.D)
        self.append_fn = getattr(kvd, f"append_{self.fmt}")
        self.attend_fn = getattr(kvd, f"attend_masked_{self.fmt}")
        need = getattr(kvd, f"attend_masked_{self.fmt}_workspace_bytes")(
            self.B, self.Hq, self.Hkv, self.C, self.D)
        self.ws = kvd.workspace(need, dev)

    def _layer(self, li, lay, pos):
        self.append_fn(lay.k_cache, lay.v_cache, lay.k_new, lay.v_new, pos, lay.mask, self.status)
        self.attend_fn(lay.q, lay.k_cache, lay.v_cache, lay.mask, lay.scale, out=self.out[li],
                       workspace=self.ws, dev_status=self.status)

    def eager_run(self, j, timing=False):
        torch = self.torch
        pos = self.pos_table[j % self.cycle]
        evs = []
        for li, lay in enumerate(self.w.layers):
            if timing:
                e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                e[0].record()
            self.append_fn(lay.k_cache, lay.v_cache, lay.k_new, lay.v_new, pos, lay.mask,
                           self.status)
            if timing:
                e[1].record()
            self.attend_fn(lay.q, lay.k_cache, lay.v_cache, lay.mask, lay.scale,
                           out=self.out[li], workspace=self.ws, dev_status=self.status)
            if timing:
                e[2].record()
                evs += [("append", e[0], e[1]), ("attend", e[1], e[2])]
        return evs

    def launches_per_step(self):
        return self.layers * (1 + self.attention_plan().launches)  # append, attention (+ combine)

    def attend_bytes(self, j):
        return quant_attend_bytes(self.lengths_at(j), self.Hq, self.Hkv, self.C, self.D, self.row)

    def step_bytes(self, j):
        """Attention plus the append of the step's rows."""
        app = quant_append_bytes(self.B, self.Hkv, self.D, self.row)
        return self.layers * (self.attend_bytes(j) + app)

    def copy_setup(self):
        return False

    def attention_plan(self):
        return getattr(self.kvd, f"attend_masked_{self.fmt}_plan")(self.B, self.Hq, self.Hkv,
                                                                   self.C, self.D)

    def kernel_name(self):
        return attention_kernel_name(f"{QUANT_FORMATS[self.name]} tensor-core",
                                     self.attention_plan(), self.Hq // self.Hkv)

    def aux_ops(self):
        """The quantising append kernel and the combine."""
        lays = self.w.layers
        ops = {"append": lambda li: self.append_fn(lays[li].k_cache, lays[li].v_cache,
                                                   lays[li].k_new, lays[li].v_new, self.gpos,
                                                   lays[li].mask, self.status)}
        plan = self.attention_plan()
        part = self.kvd.workspace_partials(self.ws, plan, self.B * self.Hq, self.D)
        if part is not None and plan.launches > 1:
            po, pl = part
            ops["combine"] = lambda li: self.kvd.combine(po, pl, out=self.out[li].view(-1, self.D))
        return ops

    def config(self):
        return masked_config(self.name, self.w, self.layers, self.lengths0)


def make_bench(name, torch, kvd, dev, layers=None):
    if name in ("paged", "paged_gather"):
        return PagedBench(torch, kvd, dev, name)
    if name in PAGED_QUANT:
        return PagedQuantBench(name, torch, kvd, dev)
    if name in QUANT_FORMATS:
        return QuantBench(name, torch, kvd, dev, layers)
    if name == "indexed":
        return IndexedBench(torch, kvd, dev, layers)
    return MaskedBench(name, torch, kvd, dev, layers)


# ------------------------------------------------------------------- timing

_T0 = time.time()


def log(msg):
    print(f"[bench {time.time() - _T0:7.1f}s] {msg}", file=sys.stderr, flush=True)


def timed(torch, dist, fn, K):
    """Barrier + synchronize on both sides; CUDA events on the current stream."""
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for j in range(K):
        fn(j)
    e1.record()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    return e0.elapsed_time(e1)


def cpu_model():
    """The host CPU as /proc/cpuinfo names it (model name, else the Arm
    implementer / part codes), with the machine type."""
    import platform
    try:
        info = open("/proc/cpuinfo").read()
    except OSError:
        info = ""
    m = re.search(r"^model name\s*:\s*(.+)$", info, re.M)
    if m:
        return m.group(1).strip()
    imp = re.search(r"^CPU implementer\s*:\s*(\S+)", info, re.M)
    part = re.search(r"^CPU part\s*:\s*(\S+)", info, re.M)
    if imp and part:
        return f"{platform.machine()} implementer {imp.group(1)} part {part.group(1)}"
    return platform.machine()


def roofline_entry(b, res, peak, peak_src, traffic):
    """The attention kernel against the HBM roofline.  Its duration comes from
    the timed steps: the step time minus the step's other launches (the
    combine, a separate append, the gather), each kind timed on its own as a
    CUDA graph of its launches for every layer of the step, per layer."""
    ach = res["attend_gbs_in_step"]
    return {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
            "traffic": traffic, "bytes_per_launch": res["attend_bytes"],
            "kernel": b.kernel_name(), "ms_per_launch": res["attend_ms_in_step"],
            "duration_from": "timed steps minus the graph-timed other launches of the step",
            "other_launches_ms_per_step": res["aux_ms_per_step"],
            "attention_op": {"what": "attention + combine per layer inside the timed steps",
                             "ms_per_layer": res["op_ms_in_step"],
                             "achieved": res["op_gbs_in_step"],
                             "frac": res["op_gbs_in_step"] / peak},
            "per_launch_pass": {"what": "each attention call (attention + combine) between CUDA "
                                        "events, launches queued behind a spinning kernel",
                                "achieved": res["attend_gbs"], "frac": res["attend_frac"],
                                "ms_per_launch": res["attend_ms_per_launch"]},
            "peak_source": peak_src}


def step_quantiles(torch, b, K, flush):
    """p10 / p50 / p90 of K single graph replays, each between its own CUDA
    events; with ``flush``, a buffer of twice the L2 is written (untimed)
    before each step."""
    evs = []
    for j in range(K):
        if flush is not None:
            flush.fill_(float(j))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        b.graph_run(j)
        e1.record()
        evs.append((e0, e1))
    torch.cuda.synchronize()
    d = sorted(a.elapsed_time(c) for a, c in evs)
    q = lambda f: d[min(len(d) - 1, int(f * (len(d) - 1) + 0.5))]  # noqa: E731
    return {"p10": q(0.1), "p50": q(0.5), "p90": q(0.9), "n": len(d)}


def _reduce(torch, dist, x, op):
    if dist is None:
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=op)
    return float(t.item())


def max_over_ranks(torch, dist, x):
    return _reduce(torch, dist, x, None if dist is None else dist.ReduceOp.MAX)


def sum_over_ranks(torch, dist, x):
    return _reduce(torch, dist, x, None if dist is None else dist.ReduceOp.SUM)


def whole_job_rate(torch, dist, ms, nbytes):
    """Weak scaling: every rank processes its own workload; the job's rate is
    the bytes all ranks moved over the slowest rank's time (GB/s, ms)."""
    ms_max = max_over_ranks(torch, dist, ms)
    total = sum_over_ranks(torch, dist, nbytes)
    return total / (ms_max / 1e3) / 1e9, ms_max


def gate_stream(torch, ms=10):
    """Hold the stream with a spinning kernel so that the launches queued
    behind it run back to back, without host gaps between them."""
    torch.cuda._sleep(int(ms * 1e-3 * 2.0e9))


def measure_aux(b, torch, K):
    """Each kind of the step's non-attention launches timed on its own: a CUDA
    graph of that kind's launch for every layer, replayed K times between CUDA
    events.  Returns ms per step by kind."""
    out = {}
    for kind, op in b.aux_ops().items():
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for li in range(b.layers):
                op(li)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(K):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        out[kind] = e0.elapsed_time(e1) / K
        del g
    return out


def measure_workload(b, torch, dist, K, W, peak, clocks=None, min_timed_ms=None):
    """Warm-up; the timed K steps (the step captured once as a CUDA graph and
    replayed K times); CUDA events around every kernel call of K more steps
    queued behind a spinning kernel (per-launch durations); K eager steps
    through the binding (host launch overhead included).  With
    `min_timed_ms`, K grows until the timed steps span at least that long
    (short steps: one slow step would otherwise weigh on the mean), after
    0.2 s of untimed replays."""
    res = {}
    b.reset_cycle()
    for j in range(W):
        b.eager_run(j)
    torch.cuda.synchronize()
    log(f"  warm-up done (status {int(b.status.item())}); capturing the step")
    b.capture()
    for j in range(3):
        b.graph_run(j)
    torch.cuda.synchronize()
    log(f"  graph replays done (status {int(b.status.item())})")
    b.reset_cycle()
    if clocks is not None:
        clocks.start()
    if clocks is not None or min_timed_ms:
        # a few sampling intervals before the timed steps
        soak_end, j = time.time() + (0.6 if clocks is not None else 0.2), 0
        while time.time() < soak_end:
            b.graph_run(j)
            j += 1
            torch.cuda.synchronize()
        b.reset_cycle()
    if min_timed_ms:
        est = timed(torch, None, b.graph_run, 3) / 3
        K = max(K, int(math.ceil(min_timed_ms / max(est, 1e-3))))
        b.reset_cycle()
    res["steps"] = K
    ms = timed(torch, dist, b.graph_run, K)
    if clocks is not None:
        res["clocks"] = clocks.stop()
    res["gbs"], ms = whole_job_rate(torch, dist, ms, sum(b.step_bytes(j) for j in range(K)))
    res["ms_per_step"] = ms / K
    res["tokens_per_s"] = sum_over_ranks(torch, dist, b.tokens_per_step() * K) / (ms / 1e3)
    res["attention_tflops"] = b.flops_per_step() / (ms / K / 1e3) / 1e12
    # the distribution of single steps, and the same with L2 flushed before each
    b.reset_cycle()
    res["step_ms"] = step_quantiles(torch, b, K, None)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=b.dev)
    b.reset_cycle()
    res["step_ms_l2_flushed"] = step_quantiles(torch, b, K, flush)
    del flush

    log(f"  timed steps done: {ms / K:.3f} ms/step; per-launch pass")
    b.reset_cycle()
    ev = []
    for j in range(K):  # one step per gate: its launches fit in the launch queue
        torch.cuda.synchronize()
        gate_stream(torch)
        ev.append(b.eager_run(j, timing=True))
    torch.cuda.synchronize()
    for kind in ("attend", "append", "gather"):
        d = [s.elapsed_time(e) for row in ev for (k2, s, e) in row if k2 == kind]
        if d:
            res[kind + "_ms_per_launch"] = sum(d) / len(d)
    a_bytes = sum(b.attend_bytes(j) for j in range(K)) / K
    res["attend_bytes"] = a_bytes
    res["attend_gbs_per_launch"] = a_bytes / (res["attend_ms_per_launch"] / 1e3) / 1e9
    res["attend_gbs"] = res["attend_gbs_per_launch"]
    res["attend_frac"] = res["attend_gbs"] / peak
    # the attention kernel's duration inside the timed steps: the step time
    # minus the step's other launches, each kind timed alone as a graph
    layers = getattr(b, "layers", 1)
    aux = measure_aux(b, torch, K)
    res["aux_ms_per_step"] = aux
    attn_step = max(res["ms_per_step"] - sum(aux.values()), 1e-6)
    res["attend_ms_in_step"] = attn_step / layers
    res["attend_gbs_in_step"] = a_bytes / (res["attend_ms_in_step"] / 1e3) / 1e9
    # the attention operation (kernel + combine) per layer inside the steps
    op_step = max(res["ms_per_step"] - sum(v for k, v in aux.items() if k != "combine"), 1e-6)
    res["op_ms_in_step"] = op_step / layers
    res["op_gbs_in_step"] = a_bytes / (res["op_ms_in_step"] / 1e3) / 1e9
    if "gather_ms_per_launch" in res:
        res["gather_gbs"] = b.gather_bytes() / (res["gather_ms_per_launch"] / 1e3) / 1e9
        res["gather_frac"] = res["gather_gbs"] / peak
    if "gather" in aux:
        res["gather_gbs_graph"] = b.gather_bytes() / (aux["gather"] / 1e3) / 1e9

    b.reset_cycle()
    gbs_e, ms_e = whole_job_rate(torch, dist, timed(torch, dist, b.eager_run, K),
                                 sum(b.step_bytes(j) for j in range(K)))
    res["eager"] = {"gbs": gbs_e, "ms_per_step": ms_e / K}
    b.reset_cycle()
    return res


def measure_copy(b, torch, K):
    """kvd_copy_prefix over all layers (one launch), CUDA events around each
    launch queued behind a spinning kernel."""
    if not (hasattr(b, "copy_setup") and b.copy_setup()):
        return None
    for _ in range(3):
        b.copy_run()
    torch.cuda.synchronize()
    d = []
    for _ in range(K):
        gate_stream(torch)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        b.copy_run()
        e1.record()
        torch.cuda.synchronize()
        d.append(e0.elapsed_time(e1))
    b.reset_cycle()
    ms = sum(d) / len(d)
    return {"gbs": b.copy_bytes() / (ms / 1e3) / 1e9, "ms_per_launch": ms,
            "bytes": b.copy_bytes(), "layers": b.layers}


def measure_e2e(b, torch, dist, K):
    h2d, d2h = b.e2e_setup()
    b.reset_cycle()
    for j in range(3):
        b.e2e_step(j)
    torch.cuda.synchronize()
    b.reset_cycle()
    gbs, ms = whole_job_rate(torch, dist, timed(torch, dist, b.e2e_step, K),
                             sum(b.step_bytes(j) for j in range(K)))
    b.reset_cycle()
    return {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms / K}


# -------------------------------------------------------------- CPU oracle

def oracle_rate(name, seconds):
    """Time the fp64 oracle on host copies of the workload: whole layers
    (append + attention; for the paged workload gather + paged attention over
    all sequences), repeated for about ``seconds`` of CPU work and at least
    one layer.  Returns the cpu_baseline dict: GB/s of the same algorithmic
    bytes as the GPU line, per-layer milliseconds, cores, sample."""
    import torch

    import oracle
    import workloads
    oracle.build()

    def run(step, per_layer_bytes, what):
        done, t0, n = 0, time.perf_counter(), 0
        while True:
            step(n)
            done += per_layer_bytes
            n += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                break
        return {"value": done / el / 1e9, "unit": "GB/s", "cores": oracle.threads(),
                "kind": "oracle", "per_layer_ms": el / n * 1e3, "layers_timed": n,
                "sample": f"{n} whole layers of the {name} workload ({what}), {el:.1f} s",
                "cpu_model": cpu_model()}

    if name in ("paged", "paged_gather"):
        pw = workloads.paged(device="cpu")
        lengths = [int(x) for x in pw.lengths]
        if name == "paged_gather":
            kb = pw.key_cache.view(torch.int16).numpy()
            vb = pw.value_cache.view(torch.int16).numpy()

            def step(n):
                oracle.gather_paged(kb, vb, pw.block_tables, pw.seq_lens, pw.seq_offset)
            return run(step, gather_bytes(lengths, 8, 128, 8, 128, 2, 128),
                       "gather of all 64 sequences")

        kb = pw.key_cache.view(torch.int16).numpy()
        vb = pw.value_cache.view(torch.int16).numpy()

        def step(n):
            oracle.append_paged(kb, vb, pw.block_tables, pw.seq_offset, pw.k_new, pw.v_new, pw.pos)
            oracle.attend_paged(pw.q, pw.key_cache, pw.value_cache, pw.block_tables, pw.seq_lens,
                                pw.seq_offset, pw.scale)
        return run(step, paged_attend_bytes(lengths, 32, 8, 128, 2, 128) + append_bytes(64, 8, 128, 2),
                   "paged append + attention of all 64 sequences")
    if name in PAGED_QUANT:
        fmt = name[-3:]
        pw = workloads.paged_quant(fmt, device="cpu")
        lengths = [int(x) for x in pw.lengths]
        kb, vb = pw.key_cache.numpy(), pw.value_cache.numpy()
        row = kb.shape[-1]

        def step(n):
            oracle.append_paged_quant(kb, vb, pw.block_tables, pw.seq_offset, pw.k_new, pw.v_new,
                                      pw.pos, fmt)
            oracle.attend_paged_quant(pw.q, kb, vb, pw.block_tables, pw.seq_lens, pw.seq_offset,
                                      pw.scale, fmt)
        return run(step, paged_quant_attend_bytes(lengths, 32, 8, 128, row, 128)
                   + quant_append_bytes(64, 8, 128, row),
                   f"quantising paged append + {PAGED_QUANT[name]} paged attention of all 64 sequences")
    if name == "indexed":
        w = workloads.gqa(device="cpu", layers=1)
        lay = w.layers[0]
        topk = IndexedBench.TOPK
        L = [int(x) for x in lay.lengths]
        idx = workloads.index_lists(L, topk)
        per = (indexed_attend_bytes([min(topk, x) for x in L], topk, w.Hq, w.Hkv, w.D, 2)
               + append_bytes(w.B, w.Hkv, w.D, 2))
        kh, vh = lay.k_cache.view(torch.int16).numpy().copy(), lay.v_cache.view(torch.int16).numpy().copy()

        def step(n):
            oracle.append(kh, vh, lay.k_new, lay.v_new, lay.pos, None)
            oracle.attend_indexed(lay.q, torch.from_numpy(kh).view(torch.bfloat16),
                                  torch.from_numpy(vh).view(torch.bfloat16), idx, lay.scale)
        return run(step, per, f"append + index-list attention, top-{topk}")
    if name in QUANT_FORMATS:
        w = getattr(workloads, name)(device="cpu", layers=1)
        lay = w.layers[0]
        kh, vh, mh = lay.k_cache.numpy().copy(), lay.v_cache.numpy().copy(), lay.mask.numpy().copy()
        L = [int(x) for x in lay.lengths]
        row = quant_row_bytes(name, w.D)
        per = (quant_attend_bytes(L, w.Hq, w.Hkv, w.C, w.D, row)
               + quant_append_bytes(w.B, w.Hkv, w.D, row))
        fmt = "fp8" if name == "gqa_fp8" else "fp4"
        append, attend = getattr(oracle, f"append_{fmt}"), getattr(oracle, f"attend_masked_{fmt}")

        def step(n):
            append(kh, vh, lay.k_new, lay.v_new, lay.pos, mh)
            attend(lay.q, kh, vh, mh, lay.scale)
        return run(step, per, f"{QUANT_FORMATS[name]} quantising append + attention")
    w = getattr(workloads, name)(device="cpu", layers=4 if name == "npuw" else 1)
    caches = [(l.k_cache.view(torch.int16).numpy().copy(), l.v_cache.view(torch.int16).numpy().copy(),
               l.mask.numpy().copy()) for l in w.layers]
    lay0 = w.layers[0]
    L = [min(int(x), w.window) if w.window else int(x) for x in lay0.lengths]
    per = masked_attend_bytes(L, w.Hq, w.Hkv, w.C, w.D, 2) + append_bytes(w.B, w.Hkv, w.D, 2)

    def step(n):
        li = n % len(w.layers)
        lay = w.layers[li]
        kh, vh, mh = caches[li]
        oracle.append(kh, vh, lay.k_new, lay.v_new, lay.pos, mh)
        kr = torch.from_numpy(kh).view(torch.bfloat16)
        vr = torch.from_numpy(vh).view(torch.bfloat16)
        if w.window:
            oracle.attend_window(lay.q, kr, vr, torch.from_numpy(mh), lay.pos, w.window, lay.scale)
        else:
            oracle.attend_masked(lay.q, kr, vr, torch.from_numpy(mh), lay.scale)
    return run(step, per, "append + attention")


# -------------------------------------------------------------------- main

METRIC = "decode-attention KV GB/s and % of GB300 HBM peak; decode tokens/sec at 1 GPU"


def reference_arm(args, rank, world):
    """The reference arm: the fp64 CPU oracle as it stands, on the host cores,
    each step a bounded sample of whole layers of the workload."""
    if rank != 0:
        return 0
    per_step = max(0.5, min(5.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_rate(args.workload, per_step * 0.2)
    rates, cb = [], None
    t0 = time.perf_counter()
    for _ in range(args.steps):
        cb = oracle_rate(args.workload, per_step)
        rates.append(cb["value"])
    el = time.perf_counter() - t0
    value = statistics.mean(rates)
    cb = dict(cb, value=value, sample=f"per step: {cb['sample']}")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args.workload),
            "cpu_baseline": cb,
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
    ap.add_argument("--workload", default="gqa",
                    choices=["gqa", "long", "paged", "paged_gather", "npuw", "indexed", "window",
                             "gqa_fp8", "gqa_fp4", "paged_fp8", "paged_fp4"])
    ap.add_argument("--no-others", action="store_true", help="skip the other workloads")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="oracle seconds for the main workload's CPU baseline")
    ap.add_argument("--cpu-seconds-others", type=float, default=4.0,
                    help="oracle seconds for each other workload's CPU baseline")
    ap.add_argument("--profile", action="store_true",
                    help="no timing: run --warmup + --steps eager steps of --workload (for ncu)")
    ap.add_argument("--layers", type=int, default=None,
                    help="layer caches of the static-buffer workloads (default: the workload's)")
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

    if args.profile:
        b = make_bench(args.workload, torch, kvd, dev, args.layers)
        for j in range(args.warmup + args.steps):
            b.eager_run(j)
        torch.cuda.synchronize()
        st = int(b.status.item())
        log(f"profile run of {args.workload}: {args.warmup + args.steps} steps, status {st}")
        return 0 if st == 0 else 1

    khash = kernel_source_hash()
    want_cpu = rank == 0 and world == 1

    def cpu_leg(name, seconds):
        if not want_cpu:
            return None
        log(f"{name}: cpu baseline (oracle)")
        try:
            return oracle_rate(name, seconds)
        except Exception as e:  # the oracle needs gcc on the host
            return {"unavailable": f"{type(e).__name__}: {e}"}

    def entry(name, b, res, e2e, cpu, copy):
        """One workload's figures: the step rate, the attention kernel's
        roofline, the end-to-end rate, the oracle beside it."""
        ent = {"value": res["gbs"], "unit": "GB/s", "frac_of_hbm_peak": res["gbs"] / peak,
               "steps": res["steps"], "ms_per_step": res["ms_per_step"],
               "decode_tokens_per_s": res["tokens_per_s"],
               "decode_tokens_per_s_eager":
                   b.tokens_per_step() / (res["eager"]["ms_per_step"] / 1e3),
               "attend_frac": res["op_gbs_in_step"] / peak,
               "attend_frac_per_launch_pass": res["attend_frac"],
               "roofline": roofline_entry(b, res, peak, peak_src, NCU_TRAFFIC.get((name, khash))),
               "e2e": e2e, "cpu_baseline": cpu, "eager": res["eager"],
               "attention_tflops": res["attention_tflops"],
               "step_ms": res["step_ms"], "step_ms_l2_flushed": res["step_ms_l2_flushed"],
               "gpu_launches_per_step": b.launches_per_step(), "config": b.config()}
        for k in ("append_ms_per_launch", "gather_gbs", "gather_frac", "gather_ms_per_launch",
                  "gather_gbs_graph"):
            if k in res:
                ent[k] = res[k]
        if copy is not None:
            ent["copy_prefix"] = copy
        return ent

    log(f"workload {args.workload}: building inputs")
    b = make_bench(args.workload, torch, kvd, dev, args.layers)
    clocks = ClockSampler(bus_id_of(torch, dev))
    log("timed steps")
    res = measure_workload(b, torch, dist, args.steps, args.warmup, peak, clocks=clocks)
    log(f"{args.workload}: {res['ms_per_step']:.3f} ms/step, {res['gbs']:.0f} GB/s; "
        f"attention kernel {res['attend_ms_in_step'] * 1e3:.1f} us/layer in the step; e2e pass")
    e2e = measure_e2e(b, torch, dist, args.steps)
    copy = measure_copy(b, torch, min(args.steps, 10))
    if copy is not None:
        log(f"{args.workload}: copy_kvcache of {copy['layers']} layers {copy['gbs']:.0f} GB/s")
    st = int(b.status.item())
    if st != 0:
        raise RuntimeError(f"device status {st} during the benchmark")
    main_launches = b.launches_per_step()

    others = {}
    if not args.no_others:
        for name in ("long", "paged", "paged_gather", "npuw", "gqa", "indexed", "window",
                     "gqa_fp8", "gqa_fp4", "paged_fp8", "paged_fp4"):
            if name == args.workload:
                continue
            log(f"workload {name}")
            ob = make_bench(name, torch, kvd, dev)
            r = measure_workload(ob, torch, dist, max(5, min(args.steps, 20)), 3, peak,
                                 min_timed_ms=20.0)
            oe = measure_e2e(ob, torch, dist, max(5, min(args.steps, 20)))
            oc = measure_copy(ob, torch, 5)
            if int(ob.status.item()) != 0:
                raise RuntimeError(f"device status {int(ob.status.item())} in workload {name}")
            log(f"{name}: {r['gbs']:.0f} GB/s; attention kernel {r['attend_gbs_in_step']:.0f} GB/s "
                f"in the step, attention + combine {r['op_gbs_in_step']:.0f} GB/s")
            others[name] = entry(name, ob, r, oe, None, oc)
            del ob
            torch.cuda.empty_cache()

    cpu = cpu_leg(args.workload, args.cpu_seconds)
    for name, ent in others.items():
        ent["cpu_baseline"] = cpu_leg(name, args.cpu_seconds_others)

    if rank == 0:
        ent = entry(args.workload, b, res, e2e, cpu, copy)
        line = {
            "metric": METRIC, "value": res["gbs"], "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ("bf16" if args.workload not in KV_FORMATS
                      else f"{KV_FORMATS[args.workload].lower()} kv / bf16"),
            "data": "synthetic", "config": b.config(),
            "peak_source": peak_src,
            "timing": "each timed step is one CUDA-graph replay of the decode step "
                      "(all layers' kvd kernels); 'eager' = one binding call per kernel",
            "roofline": ent.pop("roofline"), "e2e": ent.pop("e2e"),
            "cpu_baseline": ent.pop("cpu_baseline"),
            "gpu_launches": main_launches * args.steps,
            "clocks": res.get("clocks"), "kernel_hash": khash,
        }
        ent.pop("config")
        for k, v in ent.items():
            if k not in line and k != "value":
                line[k] = v
        line["workloads"] = others
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
