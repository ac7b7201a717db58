#!/usr/bin/env python
"""Decode-step benchmark of the CSA2 hot path on GB300.

One step = one decode step of a Full-mode CSA2 layer over the whole batch:
MXFP4 append of every sequence's new entry (main KV + indexer key) and FP8
append of its window entry, MXFP4 quantisation of the indexer query, the
full causal indexer scan with 8-position block maxima, block top-2048, pool
rescore + top-512, and sparse attention over 512 FP4 entries + the 128-entry
FP8 window (64 heads x 512, bf16 output).

Default workload: 8 sequences x 1,048,576 context entries, 1 query token
each (Full mode at 1M context). Other workloads: --workload 0..4, and
--workload 5, a chunked-prefill step (4096 new tokens of one sequence at
128K context through a Full layer, each token with its exact causal window;
reported in tokens/s).

Prints one JSON line (rank 0). `--impl reference` times the CPU oracle on
the same workload instead (a bounded sample, scaled to queries/s).
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
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode queries/s per CSA2 mode at context N; % of HBM roofline (1xGB300)"
METRIC_PREFILL = "chunked-prefill tokens/s of a CSA2 Full layer at context N; % of the scan's ALU roofline (1xGB300)"

# ncu DRAM traffic of the dominant kernel, per launch, with the hash of the
# sources it was measured on (reported as null once those sources change).
NCU_TRAFFIC = {
    # profiles/indexer_scan_b4_n1m.txt: 303.05 MB read + 4.91 MB written for 4 x 1M
    # positions; traffic grows with the positions scanned, so x2 for 8 x 1M.
    ("indexer_scan", 3): {"bytes_per_launch": 2 * (303.047424e6 + 4.906752e6),
                          "files": ['indexer.cu', 'sm103.cuh'], "hash": "e200950964d05106"},
}

def source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "sparse_attention_fp4_mxfp4_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm = [float(r[1]) for r in self.rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows if len(r) >= 9 for i in range(4)
                          if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(sm)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---- algorithmic bytes (reads the method must do) --------------------------------------

def scan_bytes(wl) -> int:
    """Full scan: 72 B per causal entry per sequence (all n_q tokens share
    the read; an entry is a token, or m tokens on the encoder side) + the FP4
    indexer query and head weights of each token."""
    return wl.B * (72 * (wl.N // wl.m) + wl.n_q * (32 * 72 + 32 * 4))


def causal_positions(wl) -> int:
    """Entries scored by the Full scan per step: sum over tokens of the
    entries each sees, floor((t + 1) / m)."""
    return wl.B * sum((wl.N - wl.n_q + j + 1) // wl.m for j in range(wl.n_q))


def scan_alu_ops(wl) -> int:
    """fp32 ALU operations the Full scan's score needs per step: for each
    causal (position, token) and each of 32 heads, a ReLU (max) and a
    weighted accumulation (fma)."""
    return causal_positions(wl) * 32 * 2


def alu_peak(dev) -> float:
    """fp32 lane operations per second: SMs x 128 lanes x the SM clock limit."""
    props = torch.cuda.get_device_properties(dev)
    mhz = None
    try:
        out = subprocess.run(["nvidia-smi", f"--id={dev.index or 0}", "--query-gpu=clocks.max.sm",
                              "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=20)
        mhz = float(out.stdout.strip().splitlines()[0])
    except (OSError, ValueError, IndexError, subprocess.TimeoutExpired):
        mhz = 2070.0
    return props.multi_processor_count * 128 * mhz * 1e6


def attn_bytes_per_query() -> int:
    # 512 FP4 entries x 288 B + 128 FP8 window entries x 512 B + q (64 x 512 bf16) + top-k.
    return 512 * 288 + 128 * 512 + 64 * 512 * 2 + 512 * 4


def stage_roofline(wl, kinds, stage_ms, peak) -> dict:
    """Per stage: the bytes the method must read in it per step, the rate its
    measured (eager, event-timed) duration gives, and that rate as a fraction
    of the measured HBM peak and of 8000 GB/s."""
    q = wl.B * wl.n_q
    n_full, n_reidx = kinds.count("full"), kinds.count("reindex")
    stage_bytes = {
        "scan": n_full * scan_bytes(wl),
        "blocktopk": n_full * q * 4 * ((wl.N // wl.m + 7) // 8),
        "rescore": (n_full + n_reidx) * q * (2048 * 576 + 32 * 72 + 32 * 4 + 2048 * 4),
        "attn": len(kinds) * q * attn_bytes_per_query(),
    }
    out = {}
    for name, ms in stage_ms.items():
        b = stage_bytes.get(name, 0)
        if not b or not ms:
            continue
        gbs = b / (ms * 1e-3) / 1e9
        out[name] = {"bytes_per_step": b, "gbs": gbs, "frac_measured": gbs / peak, "frac_8000": gbs / 8000.0}
    return out


def step_bytes(wl) -> int:
    """Reads the method must do per step, summed over the workload's layers."""
    q = wl.B * wl.n_q
    total = 0
    for kind in wl.layers:
        if kind == "full":
            total += scan_bytes(wl) + q * attn_bytes_per_query()
        elif kind == "reindex":
            total += q * (2048 * 576 + 32 * 72 + 32 * 4 + 2048 * 4 + attn_bytes_per_query())
        else:
            total += q * attn_bytes_per_query()
    return total


# ---- our arm ------------------------------------------------------------------------------------

def dominant_stage(wl, kinds):
    """The kernel whose HBM roofline the line reports: the scan when the step
    has a Full layer, else the pool rescore of a Reindex layer, else the
    attention; with its algorithmic bytes per launch and launches per step."""
    q = wl.B * wl.n_q
    if "full" in kinds:
        return "indexer_scan", scan_bytes(wl), "scan", 1
    if "reindex" in kinds:
        return ("indexer_rescore", q * (2048 * 576 + 32 * 72 + 32 * 4 + 2048 * 4), "rescore",
                kinds.count("reindex"))
    return "sparse_attn", q * attn_bytes_per_query(), "attn", len(kinds)


def measure(args, wl, dev, world, clocks=None):
    """Builds the workload, then times its step: the whole step as one CUDA
    graph (the headline), the same steps launched eagerly with events around
    every stage (per-kernel durations), and the end-to-end step through the
    public calls with host buffers. Returns the raw measurements."""
    import sparse_attention_fp4_mxfp4_gb300 as csa2
    from sparse_attention_fp4_mxfp4_gb300.step import Runner
    from sparse_attention_fp4_mxfp4_gb300.workload import build

    t_setup = time.time()
    S = build(wl, dev)
    R = Runner(S, prefill=wl.prefill)
    torch.cuda.synchronize()
    setup_s = time.time() - t_setup
    stream = torch.cuda.current_stream()
    ev = {}

    def mark(name):
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        ev.setdefault(name, []).append(e)

    for _ in range(args.warmup):
        R.step()
    torch.cuda.synchronize()
    st = csa2.csa2_check_device_status()
    if st != csa2.OK:
        raise RuntimeError("device status after warm-up: " + csa2.device_status_message())

    # The step's launches are captured once in a CUDA graph (a decode step has
    # the same shape every time); the graph is what the headline times.
    graph = None
    if not args.no_graph:
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            R.step()
        stream.wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            R.step()
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()
        st = csa2.csa2_check_device_status()
        if st != csa2.OK:
            raise RuntimeError("device status after graph warm-up: " + csa2.device_status_message())

    def timed(run_step, steps):
        barrier(world)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            run_step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return e0.elapsed_time(e1) / steps

    if clocks is not None:
        clocks.start()
    # Per-kernel durations: the same steps launched one by one with events
    # around every stage, back to back on the launching stream.
    stage_steps = args.steps if graph is None else max(3, min(args.steps, 500))
    ms_eager = timed(lambda: R.step(mark), stage_steps)
    ms = timed(graph.replay, args.steps) if graph is not None else ms_eager
    clk = clocks.stop() if clocks is not None else None
    stage_ms = {}
    for name in ("scan", "blocktopk", "rescore", "attn"):
        if name + "0" in ev:
            tt = [a.elapsed_time(b) for a, b in zip(ev[name + "0"], ev[name + "1"])]
            stage_ms[name] = sum(tt) / stage_steps  # per step (all layers)
    st = csa2.csa2_check_device_status()
    if st != csa2.OK:
        raise RuntimeError("device status after timing: " + csa2.device_status_message())
    e2e = None if args.no_e2e else run_e2e(args, wl, S, R, dev)
    out = {"ms": ms, "ms_eager": ms_eager, "stage_steps": stage_steps, "stage_ms": stage_ms, "e2e": e2e,
           "clocks": clk, "launches": R.launches, "setup_s": setup_s, "store_bytes": S.cache.nbytes(),
           "kinds": [L.kind for L in S.layers], "graph": graph is not None}
    del graph, R, S
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


# The decode modes the metric is quoted per, measured in the same run as the
# headline (which is the Full mode at 8 x 1M).
MODE_WORKLOADS = (1, 2, 4)


def mode_summary(args, wl, m, peak) -> dict:
    """One decode mode's device-timed queries/s, the HBM fraction of its
    dominant stage and its end-to-end queries/s."""
    kinds = m["kinds"]
    dom, dom_bytes, dom_stage, per_step = dominant_stage(wl, kinds)
    dms = m["stage_ms"].get(dom_stage)
    frac = dom_bytes / (dms / per_step * 1e-3) / 1e9 / peak if dms else None
    q = wl.B * wl.n_q
    return {"workload": wl.name, "mode": wl.mode, "layers": kinds, "batch": wl.B, "context": wl.N,
            "query_tokens": wl.n_q, "queries_per_step": q, "value": q / (m["ms"] * 1e-3), "unit": "queries/s",
            "ms_per_step": m["ms"], "steps": args.steps, "warmup": args.warmup,
            "hbm_fraction_step": (step_bytes(wl) / (m["ms"] * 1e-3) / 1e9) / peak,
            "dominant": {"kernel": dom, "frac_of_measured_hbm": frac, "algorithmic_bytes_per_launch": dom_bytes},
            "stage_ms": m["stage_ms"], "stage_roofline": stage_roofline(wl, kinds, m["stage_ms"], peak),
            "e2e": None if m["e2e"] is None else {k: m["e2e"][k] for k in ("value", "unit", "ms_per_step")},
            "clocks": m["clocks"], "gpu_launches": m["launches"] * args.steps}


def run_ours(args, wl, rank, world, local):
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    B, n_q, N = wl.B, wl.n_q, wl.N
    Q = B * n_q
    clocks = ClockSampler(local)
    m = measure(args, wl, dev, world, clocks)
    ms = m["ms"]
    ms_max = max_over_ranks(ms, world, dev)
    stage_ms = m["stage_ms"]
    peak, peak_kind = measured_peaks()
    kinds = m["kinds"]
    dom, dom_bytes, dom_stage, per_step = dominant_stage(wl, kinds)
    dom_ms = stage_ms.get(dom_stage)
    launch_ms = dom_ms / per_step if dom_ms else None
    achieved = dom_bytes / (launch_ms * 1e-3) / 1e9 if launch_ms else None
    traffic = None
    rec = NCU_TRAFFIC.get((dom, wl.index))
    if rec and rec["hash"] == source_hash(rec["files"]):
        traffic = rec["bytes_per_launch"]
    roof = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": (achieved / peak) if achieved else None, "traffic": traffic,
            "algorithmic_bytes_per_launch": dom_bytes, "peak_source": peak_kind}
    if wl.prefill:
        # A prefill chunk re-reads the same pages for every group of 8 tokens
        # (from L2): the scan is bound by the fp32 ALU work of its scores.
        ops = scan_alu_ops(wl)
        apk = alu_peak(dev)
        ach = ops / (launch_ms * 1e-3) / 1e12 if launch_ms else None
        roof = {"bound": "alu", "kernel": dom, "achieved": ach, "peak": apk / 1e12, "unit": "Top/s",
                "frac": (ach * 1e12 / apk) if ach else None, "traffic": traffic,
                "algorithmic_ops_per_launch": ops, "peak_source": "derived: SMs x 128 fp32 lanes x max SM clock",
                "tensor_flops_per_launch": causal_positions(wl) * 32 * 128 * 2}
    total_q = sum_over_ranks(float(Q), world, dev)
    value = total_q / (ms_max * 1e-3)
    sb = step_bytes(wl)
    line = {
        "metric": METRIC_PREFILL if wl.prefill else METRIC,
        "value": value,
        "unit": "tokens/s" if wl.prefill else "queries/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp4(e2m1)+e4m3 storage, f16 tensor-core operands, fp32 accumulate/softmax, bf16 out",
        "data": "synthetic (seeded generator; RMSNormed post-RoPE latents, N(0,1) indexer keys/queries)",
        "config": {"workload": wl.name, "mode": wl.mode, "layers": list(kinds), "batch": B, "context": N,
                   "query_tokens": n_q, "queries_per_step": Q, "prefill": wl.prefill, "tokens_per_entry": wl.m,
                   "l2": "inputs larger than L2 (store of %.1f GB; the step reads %.0f MB)" % (
                       m["store_bytes"] / 1e9, sb / 1e6),
                   "parallelism": f"replicas x{world} (independent sequences)", "setup_s": round(m["setup_s"], 1),
                   "launch": "CUDA graph of the whole step" if m["graph"] else "eager launches",
                   "ms_per_step_eager": m["ms_eager"], "stage_steps": m["stage_steps"]},
        "hbm_fraction_step": (sb / (ms_max * 1e-3) / 1e9) / peak,
        "stage_ms": stage_ms,
        "stage_roofline": stage_roofline(wl, kinds, stage_ms, peak),
        "roofline": roof,
        "clocks": m["clocks"],
        "gpu_launches": m["launches"] * args.steps,
        "e2e": m["e2e"],
    }
    # The other decode modes, same step and warm-up counts (replicas: every
    # rank runs them; rank 0 reports its own).
    if not args.no_modes and wl.index == 3 and not (args.B or args.N or args.nq):
        from synth.workloads import WORKLOADS
        modes = {}
        for idx in MODE_WORKLOADS:
            mwl = WORKLOADS[idx]
            modes[mwl.mode] = mode_summary(args, mwl, measure(args, mwl, dev, world, ClockSampler(local)), peak)
        line["modes"] = modes
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, budget_s=args.cpu_budget)
    return line


def run_e2e(args, wl, S, R, dev):
    """Same step through the public C-ABI with host inputs: every step copies
    its new entries and every layer's queries from pinned host memory, runs
    the layers with csa2_decode_group and reads every layer's output back."""
    import sparse_attention_fp4_mxfp4_gb300 as csa2
    from sparse_attention_fp4_mxfp4_gb300.step import append_layers
    from sparse_attention_fp4_mxfp4_gb300.workload import append_main
    c = S.cache
    host = {"latent": S.step_latent, "key": S.step_idx_key}
    if wl.m > 1:
        host["kv_gate"], host["idx_gate"] = S.step_kv_gate, S.step_idx_gate
    for li, L in enumerate(S.layers):
        host[f"swa{li}"] = S.step_swa[li]
        host[f"q{li}"] = L.q
        if L.q_idx is not None:
            host[f"qi{li}"] = L.q_idx
            host[f"w{li}"] = L.w
    # All of a step's inputs travel in one pinned buffer and one copy, all of
    # its outputs (every layer's out and lse) in one copy back.
    def pack(tensors):
        offs, total = {}, 0
        for k, t in tensors.items():
            offs[k] = total
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        return offs, total

    def view(buf, off, like):
        n = like.numel() * like.element_size()
        return buf[off:off + n].view(like.dtype).view(like.shape)

    in_offs, in_bytes = pack(host)
    host_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    for k, t in host.items():
        view(host_in, in_offs[k], t).copy_(t.cpu())
    outs_like = {f"o{li}": o for li, o in enumerate(R.out)}
    outs_like.update({f"l{li}": x for li, x in enumerate(R.lse)})
    out_offs, out_bytes = pack(outs_like)
    mode = {"full": csa2.MODE_FULL, "reindex": csa2.MODE_REINDEX, "reuse": csa2.MODE_REUSE}

    # Two sets of staging buffers: step k reads set k % 2 while the inputs of
    # step k + 1 arrive in the other set and the outputs of step k - 1 leave.
    sets = []
    for _ in range(2):
        din = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
        dout = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
        hout = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
        dev_in = {k: view(din, in_offs[k], t) for k, t in host.items()}
        outs_d = [view(dout, out_offs[f"o{li}"], o) for li, o in enumerate(R.out)]
        lses_d = [view(dout, out_offs[f"l{li}"], x) for li, x in enumerate(R.lse)]
        args_list = []
        for li, L in enumerate(S.layers):
            args_list.append(csa2.layer_args(
                mode[L.kind], B=wl.B, n_q=wl.n_q, max_ctx=wl.N, seq_len=S.seq_len, block_table=c.block_table,
                n_pages=c.n_pages, main_pages=c.main_pages, idx_pages=c.idx_pages, rings=c.rings,
                ring_idx=L.ring_idx, q=dev_in[f"q{li}"], out=outs_d[li], ws=R.ws, lse=lses_d[li],
                q_idx_codes=L.q_codes, q_idx_scales=L.q_scales, w=dev_in.get(f"w{li}"),
                pool=R.pool if L.kind == "full" else L.pool if L.kind == "reindex" else None,
                topk=R.topk if L.kind != "reuse" or li == 0 else None,
                swa_chunk=R.chunk[li] if wl.prefill else None, m=wl.m))
        ev = {k: torch.cuda.Event() for k in ("in_ready", "computed", "out_sent")}
        app = None
        if R.fused_appends:
            app = append_layers(S, swa=[dev_in[f"swa{li}"] for li in range(len(S.layers))],
                                q_idx=[dev_in.get(f"qi{li}") for li in range(len(S.layers))])
        sets.append(dict(din=din, dout=dout, hout=hout, dev_in=dev_in, args=args_list, app=app, ev=ev, used=False))
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(o.numel() * o.element_size() for o in R.out) + sum(x.numel() * 4 for x in R.lse)
    main = torch.cuda.current_stream()
    s_h2d, s_d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def compute(st):
        dev_in = st["dev_in"]
        if st["app"] is not None:
            csa2.csa2_decode_appends(dev_in["latent"], dev_in["key"], S.step_seq, S.step_pos, c.block_table,
                                     c.main_pages, c.idx_pages, st["app"])
        else:
            append_main(S, dev_in["latent"], dev_in["key"], dev_in.get("kv_gate"), dev_in.get("idx_gate"))
            for li, L in enumerate(S.layers):
                if wl.prefill:
                    csa2.csa2_quant_fp8_entries(dev_in[f"swa{li}"], R.chunk[li])
                else:
                    csa2.csa2_append_swa(dev_in[f"swa{li}"], S.step_ring_idx[li], S.step_pos, c.rings)
                if L.q_idx is not None:
                    csa2.csa2_quant_mxfp4(dev_in[f"qi{li}"], L.q_codes, L.q_scales)
        csa2.csa2_decode_group(st["args"])
        if wl.prefill:
            for li, L in enumerate(S.layers):
                csa2.csa2_ring_refill(R.chunk[li], S.seq_len, L.ring_idx, c.rings)

    def step_serial(k):
        """Copy in, compute, copy out, one after another on one stream."""
        st = sets[0]
        st["din"].copy_(host_in, non_blocking=True)
        compute(st)
        st["hout"].copy_(st["dout"], non_blocking=True)

    def step_pipelined(k):
        """Step k on staging set k % 2: its input copy waits until the step
        that last read the set has computed, its compute waits for its input
        and for the set's previous outputs to have left, its output copy waits
        for its compute."""
        st = sets[k % 2]
        ev = st["ev"]
        with torch.cuda.stream(s_h2d):
            if st["used"]:
                s_h2d.wait_event(ev["computed"])
            st["din"].copy_(host_in, non_blocking=True)
            ev["in_ready"].record(s_h2d)
        main.wait_event(ev["in_ready"])
        if st["used"]:
            main.wait_event(ev["out_sent"])
        if st.get("graph") is not None:
            st["graph"].replay()
        else:
            compute(st)
        ev["computed"].record(main)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(ev["computed"])
            st["hout"].copy_(st["dout"], non_blocking=True)
            ev["out_sent"].record(s_d2h)
        st["used"] = True

    steps = max(1, min(args.steps, 500))

    def timed(run):
        for k in range(max(3, args.warmup)):
            run(k)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(main)
        for k in range(steps):
            run(k)
        main.wait_stream(s_d2h)  # the last step's outputs are on the host
        e1.record(main)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    ms_serial = timed(step_serial)
    # Each staging set's calls (the same calls, its own buffers) recorded once
    # as a CUDA graph, replayed between the event waits of the copy streams.
    launch = "calls launched per step"
    if not args.no_graph:
        for st_ in sets:
            side = torch.cuda.Stream(device=dev)
            side.wait_stream(main)
            with torch.cuda.stream(side):
                compute(st_)
            main.wait_stream(side)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                compute(st_)
            st_["graph"] = g
        torch.cuda.synchronize()
        launch = "each step's calls replayed as a CUDA graph"
    ms_calls_only = None
    if sets[0].get("graph") is not None:
        # The same graph of public calls without any copy: separates the
        # copies' cost from the launch order of csa2_decode_group.
        g = sets[0]["graph"]
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(main)
        for _ in range(steps):
            g.replay()
        e1.record(main)
        torch.cuda.synchronize()
        ms_calls_only = e0.elapsed_time(e1) / steps
    ms = timed(step_pipelined)
    st = csa2.csa2_check_device_status()
    if st != csa2.OK:
        raise RuntimeError("device status after the end-to-end steps: " + csa2.device_status_message())
    return {"value": wl.B * wl.n_q / (ms * 1e-3), "unit": "tokens/s" if wl.prefill else "queries/s",
            "ms_per_step": ms, "steps": steps,
            "launch": launch + "; copies of steps k-1 and k+1 overlap the compute of step k "
                      "(two staging sets, copy streams)",
            "ms_per_step_serial": ms_serial, "ms_per_step_calls_only": ms_calls_only,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


# ---- the CPU oracle (baseline and reference arm) ------------------------------------------------

def oracle_query(wl, b=0, j=0, n_scan=None):
    """One query of the workload through the CPU oracle. Returns (seconds,
    scaled seconds for the whole query, description). n_scan limits the scan
    sample (positions 0..n_scan-1); its time is scaled to the full context."""
    import oracle
    import synth
    from sparse_attention_fp4_mxfp4_gb300.workload import n_blocks
    seed, N, n_q = wl.seed, wl.N, wl.n_q
    t = N - n_q + j
    li = 0
    q = synth.normal(seed, synth.Q + li, b, N - n_q + j, 1, 64 * 512).reshape(64, 512)
    desc = ""
    first = wl.layers[0]  # the layer whose query is timed (a group's first layer)
    if first in ("full", "reindex"):
        qi = synth.normal(seed, synth.IDXQ + li, b, t, 1, 32 * 128).reshape(32, 128)
        w = synth.uniform(seed, synth.W + li, b, t, 1, 32)[0]
    m = wl.m
    n_ent = (t + 1) // m  # entries the token sees
    if first == "full":
        n = n_ent if n_scan is None else min(n_ent, n_scan)
        t0 = time.perf_counter()
        if m == 1:
            keys = synth.normal(seed, synth.IDXKEY, b, 0, n, 128)
        else:  # the oracle compresses each entry's m tokens first
            x = synth.normal(seed, synth.IDXKEY, b, 0, n * m, 128).reshape(n, m, 128)
            z = synth.normal(seed, synth.IDXGATE, b, 0, n * m, 128).reshape(n, m, 128)
            keys = oracle.compress(x, z)
        r = oracle.full_indexer(qi, w, keys, n - 1, want_scores=False)
        t_idx = time.perf_counter() - t0
        scale = n_ent / n
        sel = r["topk"]
        desc = f"Full-mode query: oracle scan of {n} of {n_ent} entries" + (
            f", scan time scaled x{scale:.1f}" if scale > 1 else "") + (
            f" ({m} tokens per entry, compressed by the oracle)" if m > 1 else "")
    elif first == "reindex":
        assert m == 1, "the reference timing of a Reindex layer is written for one token per entry"
        keys = synth.normal(seed, synth.IDXKEY, b, 0, t + 1, 128)
        pool = synth.sample_sorted(seed, synth.POOL + li, b, t, n_blocks(t), 2048)
        t0 = time.perf_counter()
        r = oracle.reindex(qi, w, keys, t, pool)
        t_idx = time.perf_counter() - t0
        scale = 1.0
        sel = r["topk"]
        desc = "Reindex-mode query"
    else:
        sel = synth.sample_sorted(seed, synth.TOPK, b, t, n_ent, 512)
        t_idx, scale = 0.0, 1.0
        desc = "Reuse-mode query"
    sel = np.asarray(sel)
    sel = sel[sel >= 0].astype(np.int64)
    if m == 1:
        main = synth.latent_rows(seed, np.full(sel.size, b), sel)
    else:
        toks = (sel[:, None] * m + np.arange(m)).reshape(-1)
        x = synth.latent_rows(seed, np.full(toks.size, b), toks).reshape(sel.size, m, 512)
        z = synth.normal_rows(seed, synth.KVGATE, np.full(toks.size, b), toks, 512).reshape(sel.size, m, 512)
        main = oracle.compress(x, z)
    # A prefill token's window is exact: the decode window of a context ending at t.
    win = oracle.window_positions(t, t + 1 if wl.prefill else N, 128)
    wrows = synth.latent_rows(seed, np.full(win.size, b), win, tensor=synth.SWA + li)
    t0 = time.perf_counter()
    oracle.sparse_attention(q, main, wrows, 1.0 / math.sqrt(512))
    t_att = time.perf_counter() - t0
    return t_idx + t_att, t_idx * scale + t_att, desc + ", then oracle sparse attention over 512 + window keys"


def cpu_baseline(wl, budget_s=12.0):
    """The oracle on this host's cores, on the workload's own queries taken in
    order (sequence, token) until about budget_s seconds of oracle time."""
    import oracle
    done, spent, wall = 0, 0.0, time.perf_counter()
    desc = ""
    while spent < budget_s and done < 4 * wl.B * wl.n_q:
        b, j = divmod(done % (wl.B * wl.n_q), wl.n_q)
        _, s, desc = oracle_query(wl, b=b, j=j)
        spent += s
        done += 1
    unit = "tokens/s" if wl.prefill else "queries/s"
    return {"value": done / spent, "unit": unit, "cores": oracle.THREADS, "kind": "oracle",
            "sample": f"{done} queries of the workload in (sequence, token) order, each: " + desc,
            "oracle_s": round(spent, 2), "wall_s": round(time.perf_counter() - wall, 1)}


def run_reference(args, wl, rank, world):
    """--impl reference: the CPU oracle as it stands on this host's cores."""
    import oracle
    if rank != 0:
        return None
    n_total = args.steps + args.warmup
    # Bound the whole run to about two minutes: the scan sample per step shrinks with the step count.
    n_scan = None
    if wl.layers[0] == "full":
        probe_n = min(wl.N // wl.m, 65536)
        t0 = time.perf_counter()
        oracle_query(wl, n_scan=probe_n)
        per_pos = (time.perf_counter() - t0) / probe_n
        n_scan = int(max(4096, min(wl.N // wl.m, 100.0 / max(1, n_total) / max(per_pos, 1e-9))))
    for _ in range(args.warmup):
        oracle_query(wl, n_scan=n_scan)
    scaled = []
    desc = ""
    for _ in range(args.steps):
        _, s, desc = oracle_query(wl, n_scan=n_scan)
        scaled.append(s)
    sec = sum(scaled) / len(scaled)
    v = 1.0 / sec
    unit = "tokens/s" if wl.prefill else "queries/s"
    return {
        "impl": "reference", "metric": METRIC_PREFILL if wl.prefill else METRIC, "value": v, "unit": unit,
        "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (same seeded generator)",
        "config": {"workload": wl.name, "mode": wl.mode, "batch": wl.B, "context": wl.N, "query_tokens": wl.n_q},
        "cpu_baseline": {"value": v, "unit": unit, "cores": oracle.THREADS, "kind": "oracle",
                         "sample": desc + " (one query per step)"},
        "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=3)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="time eager launches instead of a CUDA graph")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-modes", action="store_true", help="skip the Reuse / Reindex / group modes of the default line")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--B", type=int, default=None, help="override the batch (profiling captures only)")
    ap.add_argument("--N", type=int, default=None, help="override the context (profiling captures only)")
    ap.add_argument("--nq", type=int, default=None, help="override the query tokens (profiling captures only)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    from synth.workloads import WORKLOADS
    wl = WORKLOADS[args.workload]
    if args.B or args.N or args.nq:
        from synth.workloads import Workload
        wl = Workload(wl.index, wl.name + f"_B{args.B or wl.B}_N{args.N or wl.N}_q{args.nq or wl.n_q}", wl.mode,
                      B=args.B or wl.B, N=args.N or wl.N, n_q=args.nq or wl.n_q, layers=wl.layers,
                      prefill=wl.prefill)
    rank, world, local = dist_env()
    if args.impl == "reference":
        line = run_reference(args, wl, rank, world)
    else:
        line = run_ours(args, wl, rank, world, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
