#!/usr/bin/env python
"""Benchmark of the fused CSR edge-attention layer (forward + backward).

Default workload: the Graph Transformer layer on the largest graph, an R-MAT
graph with super nodes (N=2^20, 32.4M edges with self-loops, H=4, D=64, bf16,
forward + backward).  ``--config k`` runs one of the other synthetic
workloads (1: GT forward fp32 ER; 2: GATv2 Chung-Lu; 3: GT lognormal;
5: GT block-dense SBM; 6: min aggregation, lognormal graph, 512 features).

One step = forward + backward of the layer (forward only for workload 1) over
the whole graph, inputs resident on the device, L2 flushed (a write of twice
the L2 size) before every step and outside its timed interval.  The metric is
edge.heads per second (E counts self-loops) in units of 1e9.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle
instead (host cores, bounded row samples of the same workload).

Multi-GPU: the layer is one problem per graph; ``--gpus N`` under torchrun
runs N independent replicas (weak scaling), timed between barriers, max over
ranks.
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

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from sparse_graph_attention_csr_gb300 import synth  # noqa: E402

METRIC = "fused GT/GATv2 fwd+bwd edge·heads/sec (G/s)"
UNIT = "G edge·heads/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")

GT_KERNELS = ["gt_fwd", "gt_fwd_merge", "bsr_fwd", "bsr_bwd_delta", "gt_bwd_dq", "gt_bwd_dkdv",
              "gt_bwd_merge", "bsr_bwd_dq", "bsr_bwd_dkdv"]
AGG_KERNELS = ["agg_fwd", "agg_fwd_merge", "agg_bwd", "agg_bwd_merge"]
GATV2_KERNELS = ["gatv2_proj", "gatv2_fwd", "gatv2_fwd_merge", "gatv2_bwd_dst", "gatv2_bwd_src",
                 "gatv2_bwd_merge", "gatv2_bwd_dx", "gatv2_bwd_dw", "gatv2_bwd_reduce"]


# --------------------------------------------------------------------------- args

def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["native", "reference"], default="native")
    p.add_argument("--config", type=int, default=4, choices=[1, 2, 3, 4, 5, 6])
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0,
                   help="target CPU time of the oracle baseline sample")
    p.add_argument("--split-threshold", type=int, default=0)
    p.add_argument("--chunk-len", type=int, default=0)
    p.add_argument("--schedule", type=int, default=0, choices=[0, 1, 2],
                   help="Graph Transformer forward thread mapping: 0 edge stream, "
                        "1 feature-parallel, 2 edge-parallel scores + feature-parallel aggregation")
    p.add_argument("--reorder", choices=["none", "rcm", "degree"], default="none",
                   help="relabel the graph and node inputs once (outside the timed region) "
                        "with this ordering before planning")
    p.add_argument("--row-order", type=int, default=0, choices=[0, 1, 2],
                   help="walking order of the edge kernels: 0 default (= 1), 1 descending degree, "
                        "2 ascending id")
    p.add_argument("--tile-min-nnz", type=int, default=0,
                   help="> 0: block-sparse tensor-core forward (GT, bf16) with this tile threshold")
    p.add_argument("--nodes", type=int, default=0,
                   help="profiling case: the workload's recipe at this many nodes "
                        "(SBM, ER and Chung-Lu graphs; draws scale with N)")
    p.add_argument("--e2e-lanes", type=int, default=1,
                   help="streams per copy direction in the end-to-end run (each tensor cut into "
                        "this many row slices, one per stream)")
    p.add_argument("--json-out", default="")
    a = p.parse_args(argv)
    if a.e2e_lanes < 1:
        p.error("--e2e-lanes must be at least 1")
    return a


# ------------------------------------------------------------------ distributed

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- byte models

def algorithmic_bytes(kernel: str, N: int, E: int, H: int, D: int, F: int, s: int) -> int:
    """Compulsory bytes of one launch: index arrays, each node's own rows once,
    every gathered neighbour row once per edge, outputs once (fp32 lse/Delta)."""
    HD = H * D
    ptr, idx = 4 * (N + 1), 4 * E
    row = N * HD * s
    if kernel == "gt_fwd":
        return ptr + idx + row + E * 2 * HD * s + row + 4 * N * H
    if kernel == "gt_bwd_dq":
        return ptr + idx + 2 * row + 4 * N * H + E * 2 * HD * s + row + 4 * N * H
    if kernel == "gt_bwd_dkdv":
        return ptr + idx + 2 * row + E * (2 * HD * s + 8 * H) + 2 * row
    if kernel == "gatv2_fwd":
        return ptr + idx + row + E * HD * s + row + 4 * N * H
    if kernel == "gatv2_bwd_dst":
        return ptr + idx + 2 * row + 4 * N * H + E * HD * s + row + 4 * N * H
    if kernel == "gatv2_bwd_src":
        return ptr + idx + row + E * (2 * HD * s + 8 * H) + row
    if kernel == "agg_fwd":          # gathered rows; out and the win mask written
        return ptr + idx + E * HD * s + row + E * HD * s // 16
    if kernel == "agg_bwd":          # transposed CSR and edge map, win mask, each dOut row once, dX
        return ptr + 2 * idx + E * HD * s // 16 + row + row
    if kernel == "gatv2_proj":
        return N * F * s + F * HD * s + row
    if kernel == "gatv2_bwd_dx":
        return 2 * row + 2 * F * HD * s + N * F * s
    if kernel == "gatv2_bwd_dw":
        return N * F * s + row
    return 0


def bsr_bytes(kernel: str, N: int, H: int, D: int, s: int, n_tiles: int, n_entries: int) -> int:
    """Compulsory bytes of one block-sparse launch: each panel's own rows once,
    the 16 source rows of every kept tile once per head, 256 bytes of masks
    per tile, row statistics once; the dK/dV pass reads the 128 destination
    rows of every (row panel, column panel) entry."""
    HD = H * D
    row = N * HD * s
    tiles = n_tiles * (16 * 2 * HD * s + 256 + 4)
    if kernel == "bsr_fwd":          # Q; K, V per tile; out, lse read and written
        return row + tiles + 2 * row + 8 * N * H
    if kernel == "bsr_bwd_delta":    # Q, dOut, lse; K, V per tile; Delta_t written
        return 2 * row + 4 * N * H + tiles + 4 * N * H
    if kernel == "bsr_bwd_dq":       # as above + Delta read, dQ read and written
        return 2 * row + 8 * N * H + tiles + 2 * row
    if kernel == "bsr_bwd_dkdv":     # K, V; per entry Q, dOut, lse, Delta of 128 rows, 8 masks
        return 2 * row + n_entries * (128 * (2 * HD * s + 8 * H) + 8 * 256 + 36) + 4 * row
    return 0


def kernel_flops(kernel: str, N: int, H: int, D: int, F: int) -> int:
    HD = H * D
    if kernel == "gatv2_proj" or kernel == "gatv2_bwd_dw":
        return 2 * N * F * HD
    if kernel == "gatv2_bwd_dx":
        return 2 * 2 * N * HD * F
    return 0


def measured_peaks():
    try:
        with open(PEAKS_FILE) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


# the source files each kernel family is compiled from (its own kernels, the
# edge stream and the plan that orders its work); a traffic figure is kept
# only while these files are unchanged since the counters were taken
_COMMON = ["common.cuh", "plan.h", "plan.cu", "items.cuh", "stream.cuh"]
FAMILY_SOURCES = {
    "gt": _COMMON + ["gt.cuh", "gt_bf16.cu", "gt_f32.cu"],
    "gatv2": _COMMON + ["gatv2.cuh", "gatv2_bf16.cu", "gatv2_f32.cu", "gemm.cuh", "tc.cuh",
                        "tc_proj.cu", "tc_proj.cuh", "tc_dx.cu", "tc_dx.cuh"],
    "bsr": _COMMON + ["tc.cuh", "bsr.cu", "bsr_fwd.cu", "bsr_bwd.cu"],
    "agg": _COMMON + ["gt.cuh", "agg.cu"],
}


def kernel_family(kernel: str) -> str:
    for fam in ("gatv2", "bsr", "agg", "gt"):
        if kernel.startswith(fam):
            return fam
    return ""


def source_hash(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_graph_attention_csr_gb300", "csrc")
    files = FAMILY_SOURCES.get(kernel_family(kernel)) or sorted(os.listdir(csrc))
    for f in sorted(files):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def dram_rate(traffic, avg_ms: float, hbm_gbs: float) -> dict:
    """DRAM rate of a launch: its measured DRAM bytes (ncu, per launch) over its
    event-timed duration, and that rate as a fraction of the HBM peak.  Empty
    when no traffic figure is known for the current sources."""
    if not traffic or not avg_ms or avg_ms <= 0:
        return {}
    gbs = traffic / (avg_ms / 1e3) / 1e9
    return {"dram_gbs": gbs, "dram_frac": gbs / hbm_gbs}


def traffic_for(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, only if it was
    taken on the current sources of the kernel's family."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
    except Exception:
        return None
    e = t.get(workload, {}).get(kernel)
    if not e or e.get("source_hash") != source_hash(kernel):
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------- workload

class Workload:
    """Host inputs (pinned), device inputs, plan and step functions."""

    def __init__(self, key: int, device, split_threshold=0, chunk_len=0, tile_min_nnz=0, nodes=0,
                 schedule=0, reorder="none", row_order=0):
        import sparse_graph_attention_csr_gb300 as sga
        self.sga = sga
        self.w = synth.WORKLOADS[key]
        if nodes:
            w0 = self.w
            params = {k: int(v * nodes / w0.N) for k, v in w0.params.items() if k == "draws"}
            if w0.graph == "rmat":   # R-MAT draws node ids from 2^scale: nodes must be a power of two
                scale = int(nodes).bit_length() - 1
                if nodes != 1 << scale:
                    raise SystemExit("--nodes must be a power of two for the R-MAT workload")
                params["scale"] = scale
            self.w = w0.scaled(N=nodes, name=f"{w0.name}_at_n{nodes}", params=params)
        w = self.w
        self.device = device
        self.indptr, self.indices = synth.make_graph(w)
        if len(self.indptr) - 1 != w.N:
            raise SystemExit(f"graph has {len(self.indptr) - 1} nodes, the workload {w.N}")
        self.N, self.E = w.N, int(self.indptr[-1])
        self.units = self.E * w.H
        self.tdt = torch.float32 if w.dtype == "f32" else torch.bfloat16
        self.s = 4 if w.dtype == "f32" else 2
        if w.layer == "gt":
            x = synth.gt_inputs(w)
            if not w.backward:
                x["dOut"] = synth.round_to(synth.normal(w.seed, synth.STREAM_DOUT, (w.N, w.H, w.D)),
                                           w.dtype)
            self.in_names = ["Q", "K", "V"] + (["dOut"] if w.backward else [])
        elif w.layer.startswith("agg"):
            x = synth.agg_inputs(w)
            self.in_names = ["X", "dOut"]
        else:
            x = synth.gatv2_inputs(w)
            self.in_names = ["X", "W_l", "W_r", "a", "dOut"]
        self.reorder, self.reorder_ms = reorder, 0.0
        if reorder != "none":
            # relabel once: the graph on the device, node tensors on the host
            ip = torch.from_numpy(self.indptr).to(device)
            ix = torch.from_numpy(self.indices).to(device)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            perm = sga.reorder(ip, ix, reorder)
            ip, ix = sga.relabel_csr(ip, ix, perm)
            torch.cuda.synchronize()
            self.reorder_ms = (time.perf_counter() - t0) * 1e3
            self.indptr, self.indices = ip.cpu().numpy(), ix.cpu().numpy()
            pl = perm.long().cpu()
            node_keys = {"Q", "K", "V", "dOut", "X"}
            for k in list(x):
                if k in node_keys:
                    t, f64 = x[k]
                    t2 = torch.empty_like(t)
                    t2[pl] = t
                    f2 = np.empty_like(f64)
                    f2[pl.numpy()] = f64
                    x[k] = (t2, f2)
        self.host64 = {k: v[1] for k, v in x.items()}
        self.host = {k: x[k][0].pin_memory() if torch.cuda.is_available() else x[k][0]
                     for k in self.in_names}
        self.dev = {k: self.host[k].to(device) for k in self.in_names}
        self.ip = torch.from_numpy(self.indptr).to(device)
        self.ix = torch.from_numpy(self.indices).to(device)
        F = w.F if w.layer == "gatv2" else 0
        t0 = time.perf_counter()
        self.plan = sga.Plan(self.ip, self.ix, w.H, w.D, self.tdt, F=F,
                             split_threshold=split_threshold, chunk_len=chunk_len,
                             tile_min_nnz=tile_min_nnz,
                             layer=sga.SGA_LAYER_MINMAX if w.layer.startswith("agg")
                             else sga.SGA_LAYER_ATTENTION, schedule=schedule, row_order=row_order)
        self.row_order = row_order
        self.schedule = schedule
        torch.cuda.synchronize()
        self.plan_ms = (time.perf_counter() - t0) * 1e3
        self.tile_min_nnz = tile_min_nnz
        self.E_residual = self.plan.info()["E_residual"] if tile_min_nnz else self.E
        self.outputs = None

    @property
    def kernels(self):
        if self.w.layer.startswith("agg"):
            return AGG_KERNELS
        return GT_KERNELS if self.w.layer == "gt" else GATV2_KERNELS

    def forward(self, d):
        """The layer's forward on device tensors d: (outputs, saved tensors)."""
        sga, w = self.sga, self.w
        if w.layer == "gt":
            out, lse = sga.gt_attn_fwd(self.plan, d["Q"], d["K"], d["V"])
            return {"out": out, "lse": lse}, (out, lse)
        if w.layer.startswith("agg"):
            # the layer's outputs: the aggregate and the win mask its backward takes
            out, _, mask = sga.agg_minmax_fwd(self.plan, d["X"], w.layer[4:], arg=False)
            return {"out": out, "mask": mask}, mask
        FL, FR, out, lse = sga.gatv2_fwd(self.plan, d["X"], d["W_l"], d["W_r"], d["a"], 0.2)
        return {"out": out, "lse": lse}, (FL, FR, out, lse)

    def backward(self, d, saved):
        """The layer's backward: its gradients."""
        sga, w = self.sga, self.w
        if w.layer == "gt":
            out, lse = saved
            dQ, dK, dV = sga.gt_attn_bwd(self.plan, d["Q"], d["K"], d["V"], out, lse, d["dOut"])
            return {"dQ": dQ, "dK": dK, "dV": dV}
        if w.layer.startswith("agg"):
            return {"dX": sga.agg_minmax_bwd(self.plan, saved, d["dOut"])}
        FL, FR, out, lse = saved
        dX, dWl, dWr, da = sga.gatv2_bwd(self.plan, d["X"], d["W_l"], d["W_r"], d["a"], FL, FR,
                                         out, lse, d["dOut"], 0.2)
        return {"dX": dX, "dW_l": dWl, "dW_r": dWr, "da": da}

    def step(self, d=None):
        """One forward(+backward) pass on device tensors d; returns the outputs."""
        d = self.dev if d is None else d
        outs, saved = self.forward(d)
        if self.w.backward:
            outs.update(self.backward(d, saved))
        return outs

    def step_e2e(self, d_in, host_out, copy_stream):
        """One step from pinned host inputs to pinned host outputs, as a user
        overlaps it: the forward's inputs go up on the compute stream, the
        upstream gradient on a copy stream during the forward, the forward's
        outputs come down on the copy stream during the backward, the
        gradients on the compute stream after it."""
        main = torch.cuda.current_stream()
        bwd_only = [k for k in self.in_names if k == "dOut"]
        copy_stream.wait_stream(main)   # the previous step's reads of the input buffers are done
        for k in self.in_names:
            if k not in bwd_only:
                d_in[k].copy_(self.host[k], non_blocking=True)
        with torch.cuda.stream(copy_stream):
            for k in bwd_only:
                d_in[k].copy_(self.host[k], non_blocking=True)
        ev_in = copy_stream.record_event()
        outs, saved = self.forward(d_in)
        ev_fwd = main.record_event()
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(ev_fwd)
            for k, v in outs.items():
                host_out[k].copy_(v, non_blocking=True)
        ev_out = copy_stream.record_event()
        if self.w.backward:
            main.wait_event(ev_in)
            for k, v in self.backward(d_in, saved).items():
                host_out[k].copy_(v, non_blocking=True)
        main.wait_event(ev_out)

    def e2e_pipelined(self, steps, host_out, flush, lanes=1):
        """`steps` steps from pinned host inputs to pinned host outputs, the way a
        training loop overlaps its data movement: step k+1's inputs go up while
        step k computes (two device input buffers), step k's outputs come down
        while step k+1 computes.  Every step's inputs are copied up and all its
        outputs copied down inside the timed region, which runs from before the
        first upload to after the last download.  Each direction uses `lanes`
        streams: every tensor is cut into `lanes` row slices, slice i copied on
        stream i, so that copies can run on several copy engines at once.
        Returns milliseconds for all steps."""
        main = torch.cuda.current_stream()
        ups = [torch.cuda.Stream(self.device) for _ in range(lanes)]
        downs = [torch.cuda.Stream(self.device) for _ in range(lanes)]
        bufs = [{k: torch.empty_like(v) for k, v in self.dev.items()} for _ in range(2)]
        uploaded, consumed = [None, None], [None, None]
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)

        def slices(t):
            n = t.shape[0] if t.dim() else 1
            cut = [n * i // lanes for i in range(lanes + 1)]
            return [(cut[i], cut[i + 1]) for i in range(lanes)]

        def upload(b):
            done = []
            for i, st in enumerate(ups):
                with torch.cuda.stream(st):
                    if consumed[b] is not None:
                        st.wait_event(consumed[b])   # the step that read this buffer is done
                    for k in self.in_names:
                        dst, src = bufs[b][k], self.host[k]
                        if dst.dim() == 0:
                            if i == 0:
                                dst.copy_(src, non_blocking=True)
                            continue
                        lo, hi = slices(dst)[i]
                        if hi > lo:
                            dst[lo:hi].copy_(src[lo:hi], non_blocking=True)
                    done.append(st.record_event())
            uploaded[b] = done

        e0.record(main)
        for st in ups:
            st.wait_event(e0)
        upload(0)
        for k in range(steps):
            b = k % 2
            if k + 1 < steps:
                upload(1 - b)
            for ev in uploaded[b]:
                main.wait_event(ev)
            flush.zero_()   # L2 flushed before each step's compute, inside the region
            outs = self.step(bufs[b])
            consumed[b] = main.record_event()
            for i, st in enumerate(downs):
                with torch.cuda.stream(st):
                    st.wait_event(consumed[b])
                    for name, v in outs.items():
                        if v.dim() == 0:
                            if i == 0:
                                host_out[name].copy_(v, non_blocking=True)
                        else:
                            lo, hi = slices(v)[i]
                            if hi > lo:
                                host_out[name][lo:hi].copy_(v[lo:hi], non_blocking=True)
                        v.record_stream(st)   # the allocator keeps v until the copy is done
        for st in downs + ups:
            main.wait_stream(st)
        e1.record(main)
        e1.synchronize()
        return e0.elapsed_time(e1)


# --------------------------------------------------------------- CPU oracle leg

def row_sample(indptr, indices, n_rows, rng):
    """Random destination rows with their full edge lists, relabelled onto the
    nodes they touch.  Returns (indptr, indices, node_ids, n_rows)."""
    N = len(indptr) - 1
    rows = np.sort(rng.choice(N, size=min(n_rows, N), replace=False))
    deg = np.diff(indptr.astype(np.int64))[rows]
    srcs = np.concatenate([indices[indptr[r]:indptr[r + 1]] for r in rows]) if len(rows) else \
        np.zeros(0, np.int32)
    nodes = np.unique(np.concatenate([rows, srcs]))
    remap = {int(v): i for i, v in enumerate(nodes)}
    new_ptr = np.zeros(len(nodes) + 1, np.int64)
    row_pos = np.searchsorted(nodes, rows)
    counts = np.zeros(len(nodes), np.int64)
    counts[row_pos] = deg
    new_ptr[1:] = np.cumsum(counts)
    new_idx = np.empty(int(new_ptr[-1]), np.int32)
    for r, p in zip(rows, row_pos):
        seg = indices[indptr[r]:indptr[r + 1]]
        new_idx[new_ptr[p]:new_ptr[p + 1]] = np.searchsorted(nodes, seg)
    del remap
    return new_ptr.astype(np.int32), new_idx, nodes, len(rows)


def oracle_step(wl: synth.Workload, host64, ptr, idx, nodes):
    """The oracle's forward(+backward) of the workload's layer on a (sub)graph."""
    import oracle
    if wl.layer.startswith("agg"):
        _, arg = oracle.agg_fwd(ptr, idx, host64["X"][nodes], wl.layer[4:])
        if wl.backward:
            oracle.agg_bwd(arg, host64["dOut"][nodes])
        return
    if wl.layer == "gt":
        Q, K, V = (host64[k][nodes] for k in ("Q", "K", "V"))
        oracle.gt_fwd(ptr, idx, Q, K, V)
        if wl.backward:
            oracle.gt_bwd(ptr, idx, Q, K, V, host64["dOut"][nodes])
    else:
        X = host64["X"][nodes]
        store = wl.dtype
        oracle.gatv2_fwd(ptr, idx, X, host64["W_l"], host64["W_r"], host64["a"], 0.2, store=store)
        oracle.gatv2_bwd(ptr, idx, X, host64["W_l"], host64["W_r"], host64["a"],
                         host64["dOut"][nodes], 0.2, store=store)


def calibrate_sample(wl, host64, indptr, indices, target_s, rng):
    """Grow a row sample until one oracle step costs about target_s seconds."""
    N = len(indptr) - 1
    n = min(N, 2000)
    while True:
        ptr, idx, nodes, nr = row_sample(indptr, indices, n, rng)
        t0 = time.perf_counter()
        oracle_step(wl, host64, ptr, idx, nodes)
        dt = time.perf_counter() - t0
        if n >= N or dt >= 0.25 * target_s:
            scale = target_s / max(dt, 1e-3)
            n2 = int(min(N, max(n, n * scale)))
            if n2 <= n * 1.2 or n >= N:
                return ptr, idx, nodes, nr, dt
            n = n2
            ptr, idx, nodes, nr = row_sample(indptr, indices, n, rng)
            t0 = time.perf_counter()
            oracle_step(wl, host64, ptr, idx, nodes)
            return ptr, idx, nodes, nr, time.perf_counter() - t0
        n = min(N, n * 4)


def cpu_baseline(wl, host64, indptr, indices, target_s):
    import oracle
    rng = np.random.default_rng(1234)
    ptr, idx, nodes, nr, _ = calibrate_sample(wl, host64, indptr, indices, target_s / 2, rng)
    t0 = time.perf_counter()
    oracle_step(wl, host64, ptr, idx, nodes)
    dt = time.perf_counter() - t0
    units = int(ptr[-1]) * wl.H
    res = {"value": units / dt / 1e9, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
           "sample": f"{nr} random destination rows of {len(indptr) - 1} with their full edge "
                     f"lists ({int(ptr[-1])} of {int(indptr[-1])} edges), fp64 forward"
                     f"{'+backward' if wl.backward else ''}, one timed pass of {dt:.2f} s"}
    if wl.key in (1, 2):   # the two smallest workloads also on one core
        all_threads = oracle.threads()
        oracle.set_threads(1)
        try:
            ptr1, idx1, nodes1, nr1, _ = calibrate_sample(wl, host64, indptr, indices, target_s / 4,
                                                          np.random.default_rng(4321))
            t0 = time.perf_counter()
            oracle_step(wl, host64, ptr1, idx1, nodes1)
            dt1 = time.perf_counter() - t0
        finally:
            oracle.set_threads(all_threads)
        res["single_core"] = {"value": int(ptr1[-1]) * wl.H / dt1 / 1e9, "unit": UNIT, "cores": 1,
                              "sample": f"{nr1} random destination rows ({int(ptr1[-1])} edges), "
                                        f"one timed pass of {dt1:.2f} s"}
    return res


def run_reference(args, ws, rank):
    """Reference arm: the fp64 CPU oracle on bounded row samples."""
    if rank != 0:
        return
    import oracle
    wl = synth.WORKLOADS[args.config]
    indptr, indices = synth.make_graph(wl)
    x = (synth.gt_inputs(wl) if wl.layer == "gt" else
         synth.agg_inputs(wl) if wl.layer.startswith("agg") else synth.gatv2_inputs(wl))
    host64 = {k: v[1] for k, v in x.items()}
    if wl.layer == "gt" and not wl.backward:
        host64["dOut"] = np.zeros((wl.N, wl.H, wl.D))
    budget = 150.0
    per_step = budget / max(1, args.steps + args.warmup)
    rng = np.random.default_rng(99)
    ptr, idx, nodes, nr, _ = calibrate_sample(wl, host64, indptr, indices, per_step, rng)
    samples = []
    for s in range(args.warmup + args.steps):
        sp = row_sample(indptr, indices, nr, np.random.default_rng(1000 + s))
        samples.append(sp)
    for s in range(args.warmup):
        oracle_step(wl, host64, samples[s][0], samples[s][1], samples[s][2])
    t_total, units = 0.0, 0
    for s in range(args.warmup, args.warmup + args.steps):
        ptr, idx, nodes, _ = samples[s]
        t0 = time.perf_counter()
        oracle_step(wl, host64, ptr, idx, nodes)
        t_total += time.perf_counter() - t0
        units += int(ptr[-1]) * wl.H
    value = units / t_total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t_total / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "N": wl.N, "E": int(indptr[-1]), "H": wl.H, "D": wl.D,
                   "F": wl.F, "graph": wl.graph, "parallelism": "host cores (OpenMP)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
                         "sample": f"per step {nr} random destination rows with their full edge "
                                   f"lists (about {int(samples[0][0][-1])} edges)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- native arm

def run_native(args, ws, rank, local):
    import sparse_graph_attention_csr_gb300 as sga
    from sparse_graph_attention_csr_gb300 import build as sga_build
    sga_build.build()
    dev = torch.device("cuda", local)
    wl = Workload(args.config, dev, args.split_threshold, args.chunk_len, args.tile_min_nnz, args.nodes,
                  args.schedule, args.reorder, args.row_order)
    w = wl.w
    stream = torch.cuda.current_stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)

    # warm-up, then one profiled step per kernel kind to find the dominant one
    for _ in range(args.warmup):
        flush.zero_()
        wl.step()
    torch.cuda.synchronize()
    per_kernel = {}
    for k in wl.kernels:
        flush.zero_()
        sga.profile_start(k)
        wl.step()
        ms, n = sga.profile_stop()
        if n:
            per_kernel[k] = (ms, n)
    dominant = max(per_kernel, key=lambda k: per_kernel[k][0])

    # device memory of the layer: plan (transposed CSR, partitions), the
    # workspace it asks for, and the peak of torch allocations during one step
    # (outputs, saved tensors) above what was resident before it
    torch.cuda.synchronize()
    base_alloc = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    flush.zero_()
    wl.step()
    torch.cuda.synchronize()
    step_peak = torch.cuda.max_memory_allocated(dev) - base_alloc
    pinf = wl.plan.info()
    memory = {"plan_device_bytes": int(pinf["plan_device_bytes"]),
              "workspace_bytes": int(wl.plan.workspace.numel()),
              "inputs_bytes": int(sum(t.numel() * t.element_size() for t in wl.dev.values())),
              "step_peak_alloc_bytes": int(step_peak),
              "graph_bytes": int(4 * (wl.N + 1 + wl.E))}

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(ws)
    torch.cuda.synchronize()
    launches0 = sga.launch_count()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        wl.step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier(ws)
    launches = sga.launch_count() - launches0
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    # the dominant kernel, timed in a pass of its own (the same steps, L2
    # flushed before each) with events the library records around each of
    # its launches on the launching stream: the timed steps above carry no
    # extra event records
    sga.profile_start(dominant)
    for i in range(args.steps):
        flush.zero_()
        wl.step()
    torch.cuda.synchronize()
    dom_ms, dom_n = sga.profile_stop()
    # the same steps back to back without the L2 flush (labelled warm-L2; not the metric)
    ew0, ew1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ew0.record(stream)
    for i in range(args.steps):
        wl.step()
    ew1.record(stream)
    torch.cuda.synchronize()
    warm_ms = ew0.elapsed_time(ew1) / args.steps
    t_ms = max_over_ranks(sum(step_ms), ws, dev)
    value = ws * wl.units * args.steps / (t_ms / 1e3) / 1e9

    # roofline of the dominant kernel
    peaks, peak_kind = measured_peaks()
    F = w.F if w.layer == "gatv2" else 0
    avg_ms = dom_ms / max(dom_n, 1)
    flops = kernel_flops(dominant, wl.N, w.H, w.D, F)
    if flops and dominant in ("gatv2_proj", "gatv2_bwd_dx", "gatv2_bwd_dw"):
        ach = flops / (avg_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": ach / peaks["bf16_tflops"]}
    else:
        # on a block-sparse plan the CSR kernels see only the residual edges
        e_k = wl.E_residual if wl.tile_min_nnz else wl.E
        if dominant.startswith("bsr_"):
            inf = wl.plan.info()
            nbytes = bsr_bytes(dominant, wl.N, w.H, w.D, wl.s, inf["n_tiles"], inf["n_entries"])
        else:
            nbytes = algorithmic_bytes(dominant, wl.N, e_k, w.H, w.D, F, wl.s)
        ach = nbytes / (avg_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"], "algorithmic_bytes": nbytes}
    roof.update({"kernel": dominant, "launches": dom_n, "avg_launch_ms": avg_ms,
                 "peak_source": f"{peak_kind} ({'MEASURED_PEAKS.json' if peak_kind == 'measured' else '6.8 TB/s, 1.9 PFLOP/s'})",
                 # (block-sparse plans keep their own entries: their CSR passes see the residual)
                 "traffic": traffic_for(dominant, w.name + (f"_tiles{wl.tile_min_nnz}" if wl.tile_min_nnz else ""))})
    # what DRAM itself delivered during the launch (algorithmic bytes count
    # every gathered row, also those served from L2)
    roof.update(dram_rate(roof["traffic"], avg_ms, peaks["hbm_gbs"]))

    # block-sparse forward: tensor-core rate of the tile kernel (MMA work
    # issued, masked slots included) over one step
    bsr = None
    if wl.tile_min_nnz:
        inf = wl.plan.info()
        ms_b, n_b = per_kernel.get("bsr_fwd", (0.0, 0))
        mma = 2 * 2 * inf["n_tiles"] * w.H * 128 * 16 * w.D
        bsr = {"tile_min_nnz": wl.tile_min_nnz, "n_tiles": inf["n_tiles"], "n_entries": inf["n_entries"],
               "E_in_tiles": wl.E - inf["E_residual"], "E_residual": inf["E_residual"],
               "tile_fill": (wl.E - inf["E_residual"]) / max(1, inf["n_tiles"] * 128 * 16),
               "bsr_fwd_ms": ms_b, "mma_flop": mma}
        if ms_b > 0:
            t = mma / (ms_b / 1e3) / 1e12
            bsr.update({"mma_tflops": t, "frac_of_bf16_peak": t / peaks["bf16_tflops"]})

    # end to end: pinned host inputs -> device, layer, outputs -> pinned host
    e2e = None
    if not args.no_e2e:
        outs = wl.step()
        host_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in outs.items()}
        d_in = {k: torch.empty_like(v) for k, v in wl.dev.items()}
        h2d = sum(t.numel() * t.element_size() for t in wl.host.values())
        d2h = sum(t.numel() * t.element_size() for t in host_out.values())
        copy_stream = torch.cuda.Stream(dev)
        for _ in range(2):
            wl.step_e2e(d_in, host_out, copy_stream)
        torch.cuda.synchronize()
        barrier(ws)
        # one step at a time: each step's copies and compute in sequence
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e_ser = 0.0
        for _ in range(args.steps):
            flush.zero_()
            e0.record(stream)
            wl.step_e2e(d_in, host_out, copy_stream)
            e1.record(stream)
            e1.synchronize()
            e_ser += e0.elapsed_time(e1)
        e_ser = max_over_ranks(e_ser, ws, dev)
        # K steps as a loader pipelines them (the reported number)
        wl.e2e_pipelined(2, host_out, flush, args.e2e_lanes)
        torch.cuda.synchronize()
        barrier(ws)
        e_ms = max_over_ranks(wl.e2e_pipelined(args.steps, host_out, flush, args.e2e_lanes), ws, dev)
        e2e = {"value": ws * wl.units * args.steps / (e_ms / 1e3) / 1e9, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e_ms / args.steps,
               "overlap": "step k+1's inputs copied up and step k's outputs copied down while step k+1 "
                          "computes (two device input buffers); every step's copies inside the timed region",
               "copy_lanes": args.e2e_lanes,
               "serial_ms_per_step": e_ser / args.steps}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, wl.host64, wl.indptr, wl.indices, args.cpu_seconds)

    deg = synth.degree_summary(wl.indptr)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "layer": w.layer, "graph": w.graph, "N": wl.N, "E": wl.E,
                   "H": w.H, "D": w.D, "F": F, "max_degree": deg["max"],
                   "pass": "fwd+bwd" if w.backward else "fwd",
                   "l2": "flushed before every step (write of 2x L2), outside the timed interval",
                   "parallelism": f"replicas x{ws}",
                   "plan_build_ms": round(wl.plan_ms, 2),
                   "split_threshold": wl.plan.info()["split_threshold"],
                   "chunk_len": wl.plan.info()["chunk_len"],
                   "tile_min_nnz": wl.tile_min_nnz,
                   "schedule": ["stream", "feature", "bilevel"][wl.schedule],
                   "reorder": wl.reorder, "reorder_ms": round(wl.reorder_ms, 2),
                   "row_order": "ascending id" if wl.row_order == 2 else "descending degree"},
        "roofline": roof,
        "memory": memory,
        "block_sparse": bsr,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clk,
        "step_ms_p10_p50_p90": [float(np.percentile(step_ms, q)) for q in (10, 50, 90)],
        "warm_l2_ms_per_step": warm_ms,
        "kernel_ms_one_step": {k: round(v[0], 4) for k, v in per_kernel.items()},
        "wall_s": round(wall, 3),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
        if args.json_out:
            with open(args.json_out, "w") as f:
                json.dump(line, f, indent=1)


def main(argv=None):
    args = parse_args(argv)
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        run_native(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
