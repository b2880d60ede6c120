#!/usr/bin/env python
"""Benchmark of the DDTree verify step (tree build -> tree-verify MLA-absorb
attention -> greedy accept) on one GB300, against the CPU oracle.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload I] [--impl gb300|reference]

One JSON line on stdout (rank 0). A "step" is one ddt_verify_step over the
seeded synthetic batch of the chosen workload (default: the max-budget,
long-context workload, B=4 D=16 K=8 Q=65 H=64 T=32768, the largest one).
Inputs are resident in HBM; L2 is flushed (a 256 MiB write) before every timed
step and every timed attention call, outside the timed window. The step is
replayed from a CUDA graph and timed with CUDA events on its stream. The
other workloads with a 64-head target (single stream, small batch, wide
batch) are measured in the same run with the same protocol and reported
under "per_workload".

--impl reference times the CPU oracle (the plain float64 C code) on the
host's cores, on a bounded row sample of the same workload per step, scaled to
a full step. Under torchrun with N>1 each rank runs an independent replica
(the path does not shard across GPUs); rank 0 prints.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mla_tree_verify_ddt_gb300 import synth  # noqa: E402

METRIC = "verify steps/s and verify-attn TFLOP/s (% of roofline) at 1 GB300 vs CPU oracle"
UNIT = "verify steps/s"
FLOP_PER_ROW_KEY = 2 * 576 + 2 * 512  # QK^T over 576 dims + PV over 512 dims
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}
DEFAULT_WORKLOAD = 4          # max budget, long context: the largest workload
SIDE_WORKLOADS = (1, 2, 3)    # measured beside it, reported under per_workload
CPU_1CORE_WORKLOADS = (0, 1, 2)


# ------------------------------------------------------------------ helpers

def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def max_over_ranks(x: float, world: int) -> float:
    """Largest value over all replica ranks (host-side gloo collective; the
    timed path has no data exchange between GPUs)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return FALLBACK_PEAKS["hbm_gbs"], FALLBACK_PEAKS["bf16_tflops"], "fallback"


HOST_SIDE_MARK = b"// ---------------------------------------------------------------- host side"


def kernel_source_hash() -> str:
    """Hash of the attention kernel's device source: verify_attn.cu up to its
    host-side section, and the PTX helpers it includes."""
    h = hashlib.sha256()
    for f in ("verify_attn.cu", "ddt_ptx.cuh"):
        with open(os.path.join(ROOT, "mla_tree_verify_ddt_gb300", "csrc", f), "rb") as fh:
            data = fh.read()
        if HOST_SIDE_MARK in data:
            data = data[:data.index(HOST_SIDE_MARK)]
        h.update(data)
    return h.hexdigest()[:16]


def profiled_traffic(workload_name: str):
    """DRAM bytes per attention launch from the committed ncu summary, if it was
    taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", f"verify_attn_kernel_{workload_name}.txt")
    if not os.path.exists(p):
        return None
    vals = {}
    with open(p) as f:
        for line in f:
            if "=" in line and not line.startswith("#"):
                k, v = line.split("=", 1)
                vals[k.strip()] = v.strip()
    if vals.get("kernel_source_hash") != kernel_source_hash():
        return None
    try:
        return int(float(vals["dram_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        if not getattr(self, "out", ""):
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def algorithmic_work(depth: np.ndarray, n_nodes: np.ndarray, prefix_len: np.ndarray, H: int):
    """FLOP and HBM bytes one attention call must do: every valid (b, i, h)
    row sees T_b + depth_i + 1 keys; KV rows T_b + n_b are read once per
    sequence; Q rows in, fp32 out and lse written."""
    flop = 0
    byts = 0
    for b in range(depth.shape[0]):
        n = int(n_nodes[b])
        T = int(prefix_len[b])
        vis = (T + depth[b, :n].astype(np.int64) + 1).sum()
        flop += int(vis) * H * FLOP_PER_ROW_KEY
        byts += (T + n) * 1152 + n * H * (1152 + 2048 + 4)
    return flop, byts


def roofline(flop, algo_bytes, launch_ms, wl_name):
    hbm_gbs, bf16_tflops, peak_src = load_peaks()
    t_tensor = flop / (bf16_tflops * 1e12)
    t_hbm = algo_bytes / (hbm_gbs * 1e9)
    s = launch_ms / 1e3
    if t_tensor >= t_hbm:
        roof = {"bound": "tensor", "achieved": flop / s / 1e12, "peak": bf16_tflops, "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": algo_bytes / s / 1e9, "peak": hbm_gbs, "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = profiled_traffic(wl_name)
    roof["peak_source"] = (f"{peak_src} (MEASURED_PEAKS.json burst)" if peak_src == "measured"
                           else f"{peak_src} (profiling recipe)")
    roof["kernel"] = "verify_attn_kernel (+ merge_chunks_kernel when the key range is split)"
    roof["algorithmic_flop_per_launch"] = flop
    roof["algorithmic_bytes_per_launch"] = algo_bytes
    roof["launch_ms"] = launch_ms
    return roof


# ------------------------------------------------------------------ CPU oracle timing

def oracle_step_time(inp: synth.StepInputs, attn_budget_s: float, seed: int, n_threads: int):
    """Seconds for one full oracle step, measured on a bounded sample:
    the tree build and accept run in full; attention runs on a random sample
    of valid rows and is scaled to all rows by the per-row visible-key count.
    ``n_threads`` OpenMP threads run the attention rows (passed on every call:
    the oracle's thread count is sticky)."""
    import oracle
    wl = inp.wl
    t0 = time.perf_counter()
    ot = oracle.tree_build(inp.draft_tok, inp.draft_lp, inp.root_tok, wl.budget, wl.vocab)
    t_tree = time.perf_counter() - t0
    tg = synth.synth_target_argmax(ot.depth, ot.n_nodes, inp.draft_tok, inp.target_u,
                                   inp.target_alt, wl.p_match)
    t0 = time.perf_counter()
    oracle.tree_accept(ot, tg, wl.D)
    t_acc = time.perf_counter() - t0
    # all valid rows and their visible-key counts
    rows, work = [], []
    for b in range(wl.B):
        n = int(ot.n_nodes[b])
        for i in range(n):
            for h in range(wl.H):
                rows.append((b, i, h))
                work.append(int(inp.prefix_len[b]) + int(ot.depth[b, i]) + 1)
    rows = np.array(rows, np.int32)
    work = np.array(work, np.float64)
    rng = np.random.default_rng(seed)
    # calibrate: a small sample first, then a sample sized to the time budget
    pick = rng.choice(len(rows), min(len(rows), max(16, 4 * n_threads)), replace=False)
    t0 = time.perf_counter()
    _, _, cores = oracle.attn_rows(inp.q_lat, inp.q_rope, inp.c_kv, inp.k_rope, inp.prefix_len,
                                   ot.mask, ot.n_nodes, inp.scale, rows[pick], n_threads)
    t_cal = time.perf_counter() - t0
    per_key = t_cal / work[pick].sum()
    want = max(len(pick), min(len(rows), int(attn_budget_s / max(per_key * work.mean(), 1e-9))))
    if want > len(pick):
        pick = rng.choice(len(rows), want, replace=False)
        t0 = time.perf_counter()
        oracle.attn_rows(inp.q_lat, inp.q_rope, inp.c_kv, inp.k_rope, inp.prefix_len, ot.mask,
                         ot.n_nodes, inp.scale, rows[pick], n_threads)
        t_s = time.perf_counter() - t0
    else:
        t_s = t_cal
    t_attn = t_s * work.sum() / work[pick].sum()
    sample = (f"tree build + accept on all {wl.B} sequences; attention on {len(pick)} of "
              f"{len(rows)} valid (node, head) rows, scaled by visible keys")
    return t_tree + t_acc + t_attn, cores, sample


def oracle_median(inp, attn_budget_s, n_threads, runs=3):
    """Median over `runs` oracle steps (different row samples)."""
    ts, cores, sample = [], 1, ""
    for r in range(runs):
        t, cores, sample = oracle_step_time(inp, attn_budget_s, seed=1 + r, n_threads=n_threads)
        ts.append(t)
    return statistics.median(ts), cores, sample


def cpu_baseline(main_inp):
    """The oracle as it stands, timed on this host: the main workload on all
    cores, and the small workloads (tiny, single stream, small batch) on one
    core and on all cores; each a median of three bounded runs."""
    import oracle
    oracle.build()
    nproc = os.cpu_count() or 1
    t, cores, sample = oracle_median(main_inp, attn_budget_s=4.0, n_threads=nproc)
    out = {"value": 1.0 / t, "unit": UNIT, "cores": cores, "nproc": nproc, "kind": "oracle",
           "runs": 3, "statistic": "median",
           "sample": sample + " (median of 3 runs, each its own row sample)"}
    per = {}
    for idx in CPU_1CORE_WORKLOADS:
        inp = main_inp if synth.WORKLOADS[idx].name == main_inp.wl.name else synth.make_inputs(idx)
        entry = {}
        for label, n in (("1_core", 1), ("all_cores", nproc)):
            t, used, smp = oracle_median(inp, attn_budget_s=1.5, n_threads=n)
            entry[label] = {"value": 1.0 / t, "unit": UNIT, "ms_per_step": 1e3 * t, "cores": used,
                            "sample": smp}
        per[inp.wl.name] = entry
    out["per_workload"] = per
    return out


# ------------------------------------------------------------------ arms

def reference_arm(args, wl_idx, rank, world):
    if rank != 0:
        return
    import oracle
    oracle.build()
    inp = synth.make_inputs(wl_idx)
    wl = inp.wl
    nproc = os.cpu_count() or 1
    times = []
    cores = 1
    sample = ""
    for s in range(args.warmup + args.steps):
        t, cores, sample = oracle_step_time(inp, attn_budget_s=1.5, seed=s, n_threads=nproc)
        if s >= args.warmup:
            times.append(t)
    ms = 1000.0 * statistics.mean(times)
    value = 1000.0 / ms
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(wl, inp),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_dict(wl, inp):
    return {"workload": wl.name, "B": wl.B, "D": wl.D, "K": wl.K, "budget": wl.budget,
            "Q": wl.Qc, "H": wl.H, "T": list(wl.T) if isinstance(wl.T, tuple) else wl.T,
            "Tcap": inp.Tcap, "vocab": wl.vocab, "latent": 512, "rope": 64,
            "l2": "flushed before every timed step (256 MiB write)", "seed": synth.SEED_BASE}


class Bench:
    """Device, stream and L2-flush buffer shared by every measurement."""

    def __init__(self, torch, ddtree, dev):
        self.torch, self.ddtree, self.dev = torch, ddtree, dev
        self.s = torch.cuda.Stream(device=dev)
        self.flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def graph(self, fn):
        torch = self.torch
        with torch.cuda.stream(self.s):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.s):
            fn()
        return g

    def timed(self, graph, n, before=None):
        """n replays, each after an L2-evicting write and then `before`, if
        given, both outside its CUDA-event window; returns the event pairs."""
        torch, s = self.torch, self.s
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        with torch.cuda.stream(s):
            for e0, e1 in evs:
                self.flush.fill_(1)
                if before is not None:
                    before()
                e0.record(s)
                graph.replay()
                e1.record(s)
        return evs

    def mean_ms(self, graph, n, warm=3, before=None):
        self.timed(graph, warm, before)
        self.torch.cuda.synchronize()
        evs = self.timed(graph, n, before)
        self.torch.cuda.synchronize()
        return statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)


class Workload:
    """One workload's inputs on the device, its verify step as a CUDA graph
    and its attention call alone as another."""

    def __init__(self, bn: Bench, wl_idx: int):
        torch, ddtree, dev = bn.torch, bn.ddtree, bn.dev
        self.bn = bn
        inp = synth.make_inputs(wl_idx)
        self.inp, self.wl = inp, inp.wl
        wl = self.wl

        def bf16(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

        def i32(a):
            return torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)

        self.tok, self.lp, self.root = i32(inp.draft_tok), torch.from_numpy(inp.draft_lp).to(dev), i32(inp.root_tok)
        self.q_lat, self.q_rope = bf16(inp.q_lat), bf16(inp.q_rope)
        self.c_kv, self.k_rope = bf16(inp.c_kv), bf16(inp.k_rope)
        self.pl = i32(inp.prefix_len)
        # target argmax of the synthetic target model needs the tree: build it
        # once on the device, outside any timed region
        tree0 = ddtree.ddt_tree_build(self.tok, self.lp, self.root, wl.budget, wl.vocab)
        self.depth = tree0.depth.cpu().numpy()
        self.n_nodes = tree0.n_nodes.cpu().numpy()
        self.tg = i32(synth.synth_target_argmax(self.depth, self.n_nodes, inp.draft_tok, inp.target_u,
                                                inp.target_alt, wl.p_match))
        self.step = ddtree.VerifyStep(self.tok, self.lp, self.root, wl.vocab, wl.budget, self.q_lat, self.q_rope,
                                      self.c_kv, self.k_rope, self.pl, self.tg, inp.scale)
        self.nsplit = (self.step.ws_bytes // (wl.B * wl.Qc * wl.H * 513 * 4)) if self.step.ws_bytes else 1
        self.g_step = bn.graph(lambda: self.step.run(bn.s))
        self.attn_out = torch.empty_like(self.step.out)
        self.attn_lse = torch.empty_like(self.step.lse)
        self.g_attn = bn.graph(lambda: ddtree.ddt_verify_mla_attn(
            self.q_lat, self.q_rope, self.c_kv, self.k_rope, self.pl, self.step.tree, inp.scale,
            self.attn_out, self.attn_lse, self.step.workspace, stream=bn.s))
        self.flop, self.algo_bytes = algorithmic_work(self.depth, self.n_nodes, inp.prefix_len, wl.H)

    def attention_ms(self, n):
        return self.bn.mean_ms(self.g_attn, n)

    def e2e(self, steps, warmup, world):
        """The same metric end to end through the public API with host
        buffers: the step's inputs sit in one pinned host buffer laid out like
        one device buffer whose views are the step's input tensors (one copy
        in), the nodes' new KV rows go as below, and the accept result comes
        back in one copy (its four arrays are views of one device buffer). The whole step, copies included, is one CUDA
        graph replayed once a step; the host waits for the result every step."""
        torch, ddtree, dev, s = self.bn.torch, self.bn.ddtree, self.bn.dev, self.bn.s
        inp, wl = self.inp, self.wl
        D1 = wl.D + 1
        fields = [("tok", (wl.B, wl.D, wl.K), torch.int32, inp.draft_tok),
                  ("lp", (wl.B, wl.D, wl.K), torch.float32, inp.draft_lp), ("root", (wl.B,), torch.int32, inp.root_tok),
                  ("ql", (wl.B, wl.Qc, wl.H, 512), torch.int16, inp.q_lat.view(np.int16)),
                  ("qr", (wl.B, wl.Qc, wl.H, 64), torch.int16, inp.q_rope.view(np.int16)),
                  ("tg", (wl.B, wl.Qc), torch.int32, self.tg.cpu().numpy()),
                  ("pl", (wl.B,), torch.int32, inp.prefix_len)]
        # The nodes' new latent and rotary key rows: one host copy per tensor
        # straight into the cache for a single sequence; for several they
        # travel in the packed copy and two small kernels scatter them (fewer
        # operations than one copy per sequence and tensor; measured: B=4
        # 662 -> 682 steps/s, B=8 3736 -> 4176, B=1 21.9 k -> 18.9 k).
        scatter = wl.B > 1
        if scatter:
            fields += [("ckv_nodes", (wl.B, wl.Qc, 512), torch.int16,
                        np.stack([inp.c_kv[b, T:T + wl.Qc].view(np.int16) for b, T in enumerate(inp.prefix_len)])),
                       ("kr_nodes", (wl.B, wl.Qc, 64), torch.int16,
                        np.stack([inp.k_rope[b, T:T + wl.Qc].view(np.int16) for b, T in enumerate(inp.prefix_len)]))]

        def packed(specs, device, pin):
            offs, off = [], 0
            for _, shape, dt, _ in specs:
                offs.append(off)
                off += (int(np.prod(shape)) * torch.empty((), dtype=dt).element_size() + 255) // 256 * 256
            buf = torch.empty(off, dtype=torch.uint8, device=device)
            if pin:
                buf = buf.pin_memory()
            views = {}
            for (name, shape, dt, _), o in zip(specs, offs):
                n = int(np.prod(shape)) * torch.empty((), dtype=dt).element_size()
                views[name] = buf[o:o + n].view(dt).view(shape)
            return buf, views

        h_in, hv = packed(fields, "cpu", True)
        d_in, dv = packed(fields, dev, False)
        for name, _, _, arr in fields:
            hv[name].copy_(torch.from_numpy(np.ascontiguousarray(arr)))
        out_fields = [("accept_len", (wl.B,), torch.int32, None), ("accept_idx", (wl.B, D1), torch.int32, None),
                      ("commit_tok", (wl.B, D1), torch.int32, None), ("next_root", (wl.B,), torch.int32, None)]
        d_out, ov = packed(out_fields, dev, False)
        h_out = torch.empty(d_out.numel(), dtype=torch.uint8).pin_memory()
        step_e = ddtree.VerifyStep(dv["tok"], dv["lp"], dv["root"], wl.vocab, wl.budget,
                                   dv["ql"].view(torch.bfloat16), dv["qr"].view(torch.bfloat16), self.c_kv,
                                   self.k_rope, dv["pl"], dv["tg"], inp.scale,
                                   acc=ddtree.Accept(ov["accept_len"], ov["accept_idx"], ov["commit_tok"],
                                                     ov["next_root"]))
        # cache row of each node key: b * Tcap + T_b + m
        node_rows = torch.tensor([b * inp.Tcap + int(inp.prefix_len[b]) + m for b in range(wl.B) for m in range(wl.Qc)],
                                 dtype=torch.int64, device=dev)
        ckv_rows = self.c_kv.view(torch.int16).view(-1, 512)
        kr_rows = self.k_rope.view(torch.int16).view(-1, 64)
        T0 = int(inp.prefix_len[0])
        h_ckv0 = torch.from_numpy(np.ascontiguousarray(inp.c_kv[0, T0:T0 + wl.Qc].view(np.int16))).pin_memory()
        h_kr0 = torch.from_numpy(np.ascontiguousarray(inp.k_rope[0, T0:T0 + wl.Qc].view(np.int16))).pin_memory()
        h2d = h_in.numel() + (0 if scatter else h_ckv0.numel() * 2 + h_kr0.numel() * 2)
        d2h = h_out.numel()

        def e2e_step():
            d_in.copy_(h_in, non_blocking=True)
            if scatter:
                ckv_rows.index_copy_(0, node_rows, dv["ckv_nodes"].view(-1, 512))
                kr_rows.index_copy_(0, node_rows, dv["kr_nodes"].view(-1, 64))
            else:
                ckv_rows[T0:T0 + wl.Qc].copy_(h_ckv0, non_blocking=True)
                kr_rows[T0:T0 + wl.Qc].copy_(h_kr0, non_blocking=True)
            step_e.run(s)
            h_out.copy_(d_out, non_blocking=True)

        with torch.cuda.stream(s):
            for _ in range(warmup):
                e2e_step()
        torch.cuda.synchronize()
        g_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_e2e, stream=s):
            e2e_step()
        torch.cuda.synchronize()
        ms = []
        with torch.cuda.stream(s):
            g_e2e.replay()
            torch.cuda.synchronize()
            h_out.zero_()  # the timed steps must bring the result back themselves
            for _ in range(steps):
                self.bn.flush.fill_(1)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(s)
                g_e2e.replay()
                e1.record(s)
                e1.synchronize()  # the host needs the accept result before the next step
                ms.append(e0.elapsed_time(e1))
        # the result that came back is the device's
        assert np.array_equal(h_out[:wl.B * 4].view(torch.int32).numpy(), step_e.acc.accept_len.cpu().numpy())
        return {"value": world * 1000.0 / statistics.mean(ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "how": "one CUDA graph per step: copies in from pinned host memory, ddt_verify_step, "
                       "accept result copied out; host waits on it every step"}


def side_legs(bn: Bench, w: Workload, n, attn_ms, wl_idx):
    """bf16 output, paged cache, KV commit and temperature sampling on the
    main workload."""
    torch, ddtree, dev, s = bn.torch, bn.ddtree, bn.dev, bn.s
    inp, wl, flop = w.inp, w.wl, w.flop
    legs = {}
    # ---- the same attention with the latent output in bfloat16
    out16 = torch.empty(w.attn_out.shape, dtype=torch.bfloat16, device=dev)
    gb = bn.graph(lambda: ddtree.ddt_verify_mla_attn_bf16(
        w.q_lat, w.q_rope, w.c_kv, w.k_rope, w.pl, w.step.tree, inp.scale, out16, w.attn_lse,
        w.step.workspace, stream=s))
    bf16_ms = bn.mean_ms(gb, n)
    legs["bf16_out_attn"] = {"us": bf16_ms * 1e3, "tflops": flop / (bf16_ms / 1e3) / 1e12,
                             "vs_float32_out": attn_ms / bf16_ms, "out_bytes": int(out16.numel()) * 2}
    del out16, gb

    # ---- the same attention on a block-table (paged) cache: every key row in
    # a shuffled pool with junk rows, gathered by the kernel
    rng = np.random.default_rng(7)
    n_pool = wl.B * inp.Tcap + 1024
    perm = torch.from_numpy(rng.permutation(n_pool)[: wl.B * inp.Tcap].astype(np.int64)).to(dev)
    pool_kv = torch.zeros(n_pool, 512, dtype=torch.bfloat16, device=dev)
    pool_kr = torch.zeros(n_pool, 64, dtype=torch.bfloat16, device=dev)
    pool_kv[perm] = w.c_kv.reshape(-1, 512)
    pool_kr[perm] = w.k_rope.reshape(-1, 64)
    kv_index = perm.to(torch.int32).reshape(wl.B, inp.Tcap).contiguous()
    gp = bn.graph(lambda: ddtree.ddt_verify_mla_attn_paged(
        w.q_lat, w.q_rope, pool_kv, pool_kr, w.pl, kv_index, w.step.tree, inp.scale, w.attn_out, w.attn_lse,
        w.step.workspace, stream=s))
    paged_ms = bn.mean_ms(gp, n)
    legs["paged_attn"] = {"us": paged_ms * 1e3, "tflops": flop / (paged_ms / 1e3) / 1e12,
                          "vs_contiguous": attn_ms / paged_ms, "pool_rows": n_pool,
                          "note": "block table of page size 1 over a shuffled pool; two warps gather the rows "
                                  "with cp.async, reading the block table two tiles ahead"}
    del pool_kv, pool_kr, kv_index, perm, gp

    # ---- the KV commit after accept (the append of the accepted path's keys),
    # timed alone on scratch copies of the cache; the prefix lengths it
    # advances are reset before each call, outside the timed window
    kv_s, kr_s = w.c_kv.clone(), w.k_rope.clone()
    pl0 = w.pl.clone()
    pl_s, st_s = w.pl.clone(), torch.zeros_like(w.pl)
    gk = bn.graph(lambda: ddtree.ddt_kv_commit(w.step.acc, kv_s, kr_s, pl_s, st_s, stream=s))
    kv_commit_ms = bn.mean_ms(gk, n, before=lambda: pl_s.copy_(pl0))
    moved_rows = int((w.step.acc.accept_len.cpu().numpy().astype(np.int64) - 1).sum())
    legs["kv_commit"] = {"us": kv_commit_ms * 1e3, "moved_rows": moved_rows, "bytes_per_call": moved_rows * 1152 * 2,
                         "note": "latency-bound: one block per sequence, at most 16 rows of 1152 B moved"}
    del kv_s, kr_s, gk

    # ---- temperature sampling at every tree node (the sampling commit path)
    # on synthetic target logits [B,Qc,V] float32, then the accept walk on the
    # samples; the kernel streams the logits once, so it is HBM-bound. Timed
    # after writing the L2 flush buffer and then reading another buffer of
    # that size, so the kernel starts on a cold L2 that holds no dirty lines.
    lg, u = synth.sampling_inputs(wl_idx, w.depth, w.n_nodes, inp.draft_tok)
    logits = torch.from_numpy(lg).to(dev)
    u01 = torch.from_numpy(u).to(dev)
    del lg
    sample_tok = torch.empty(wl.B, wl.Qc, dtype=torch.int32, device=dev)
    node_p = torch.empty(wl.B, wl.Qc, dtype=torch.float32, device=dev)
    clean = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev).fill_(1.0)
    sink = torch.empty((), dtype=torch.float32, device=dev)
    hbm_gbs, _, peak_src = load_peaks()
    nbytes = logits.numel() * 4 + u01.numel() * 4 + sample_tok.numel() * 4 + node_p.numel() * 4
    smp = {"rows": wl.B * wl.Qc, "vocab": wl.vocab, "logits_bytes": logits.numel() * 4,
           "algorithmic_bytes_per_call": nbytes}
    for name, tau in (("temperature_1", 1.0), ("greedy", 0.0)):
        gs = bn.graph(lambda: ddtree.ddt_tree_sample(w.step.tree, logits, tau, u01, sample_tok, node_p, stream=s))
        ms = bn.mean_ms(gs, n, before=lambda: torch.sum(clean, dim=0, out=sink))
        gbs = nbytes / (ms / 1e3) / 1e9
        smp[name] = {"us": ms * 1e3, "achieved_gbs": gbs, "peak_gbs": hbm_gbs, "frac": gbs / hbm_gbs}
        del gs
    with torch.cuda.stream(s):
        ddtree.ddt_tree_sample(w.step.tree, logits, 1.0, u01, sample_tok, node_p, stream=s)
        acc = ddtree.ddt_tree_accept(w.step.tree, sample_tok, stream=s)
    torch.cuda.synchronize()
    smp["mean_accept_len_temperature_1"] = float(acc.accept_len.float().mean().item())
    smp["peak_source"] = f"{peak_src} HBM copy bandwidth"
    smp["bound"] = "hbm"
    legs["tree_sample"] = smp
    del logits, clean
    return legs


def gpu_arm(args, wl_idx, rank, world, local_rank):
    import torch

    from mla_tree_verify_ddt_gb300 import build as libbuild
    from mla_tree_verify_ddt_gb300 import ddtree

    libbuild.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")  # host-side barrier / max only
        pg = dist

    bn = Bench(torch, ddtree, dev)
    w = Workload(bn, wl_idx)
    wl, inp = w.wl, w.inp
    # tree build, attention, and the merge that also runs the accept (or the
    # accept alone when the key range is not split)
    launches_per_step = 3

    # warm-up
    bn.timed(w.g_step, args.warmup)
    torch.cuda.synchronize()

    # ---- timed region: K graph-replayed steps
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        evs = bn.timed(w.g_step, args.steps)
        torch.cuda.synchronize()
    if pg:
        pg.barrier()
    step_ms = [e0.elapsed_time(e1) for e0, e1 in evs]
    total_ms = max_over_ranks(sum(step_ms), world)
    ms_per_step = total_ms / args.steps
    value = world * 1000.0 / ms_per_step

    # ---- dominant kernel: attention alone, same protocol
    n_attn = max(args.steps, 10)
    attn_ms = w.attention_ms(n_attn)
    roof = roofline(w.flop, w.algo_bytes, attn_ms, wl.name)
    legs = side_legs(bn, w, n_attn, attn_ms, wl_idx)
    e2e = w.e2e(args.steps, args.warmup, world)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {**config_dict(wl, inp), "graph": True, "key_range_splits": w.nsplit,
                   "sequences_per_s": value * wl.B,
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "attn_tflops": w.flop / (attn_ms / 1e3) / 1e12,
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        **legs,
        "clocks": clk.summary(),
    }
    del w
    torch.cuda.empty_cache()

    # ---- the other 64-head workloads, same protocol, same run
    if not args.no_side_workloads:
        per = {}
        for idx in SIDE_WORKLOADS:
            if idx == wl_idx:
                continue
            sw = Workload(bn, idx)
            bn.timed(sw.g_step, args.warmup)
            torch.cuda.synchronize()
            with ClockSampler(local_rank) as sclk:
                sevs = bn.timed(sw.g_step, args.steps)
                torch.cuda.synchronize()
            sms = max_over_ranks(sum(e0.elapsed_time(e1) for e0, e1 in sevs), world) / args.steps
            sattn = sw.attention_ms(n_attn)
            per[sw.wl.name] = {
                "ms_per_step": sms, "value": world * 1000.0 / sms, "unit": UNIT,
                "sequences_per_s": world * 1000.0 / sms * sw.wl.B, "key_range_splits": sw.nsplit,
                "attn_launch_ms": sattn, "attn_tflops": sw.flop / (sattn / 1e3) / 1e12,
                "roofline": roofline(sw.flop, sw.algo_bytes, sattn, sw.wl.name),
                "e2e": sw.e2e(args.steps, args.warmup, world),
                "clocks": sclk.summary(),
            }
            del sw
            torch.cuda.empty_cache()
        line["per_workload"] = per
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD, help="index into synth.WORKLOADS")
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-side-workloads", action="store_true",
                    help="measure only the chosen workload (no per_workload entries)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        reference_arm(args, args.workload, rank, world)
    else:
        gpu_arm(args, args.workload, rank, world, local_rank)


if __name__ == "__main__":
    main()
