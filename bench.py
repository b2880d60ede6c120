#!/usr/bin/env python
"""Benchmark of the DDTree verify step (tree build -> tree-verify MLA-absorb
attention -> greedy accept) on one GB300, against the CPU oracle.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload I] [--impl gb300|reference]

One JSON line on stdout (rank 0). A "step" is one ddt_verify_step over the
seeded synthetic batch of the chosen workload (default: the single-stream
budget-8 workload, B=1 D=8 K=8 Q=9 H=64 T=4096). Inputs are resident in HBM;
L2 is flushed (a 256 MiB write) before every timed step and every timed
attention call, outside the timed window. The step is replayed from a CUDA
graph and timed with CUDA events on its stream.

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


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("verify_attn.cu", "ddt_ptx.cuh"):
        with open(os.path.join(ROOT, "mla_tree_verify_ddt_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
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


# ------------------------------------------------------------------ CPU oracle timing

def oracle_step_time(inp: synth.StepInputs, tree_fn, attn_budget_s: float, seed: int):
    """Seconds for one full oracle step, measured on a bounded sample:
    the tree build and accept run in full; attention runs on a random sample
    of valid rows and is scaled to all rows by the per-row visible-key count."""
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
    pick = rng.choice(len(rows), min(len(rows), 64), replace=False)
    t0 = time.perf_counter()
    _, _, cores = oracle.attn_rows(inp.q_lat, inp.q_rope, inp.c_kv, inp.k_rope, inp.prefix_len,
                                   ot.mask, ot.n_nodes, inp.scale, rows[pick])
    t_cal = time.perf_counter() - t0
    per_key = t_cal / work[pick].sum()
    want = max(64, min(len(rows), int(attn_budget_s / max(per_key * work.mean(), 1e-9))))
    if want > len(pick):
        pick = rng.choice(len(rows), want, replace=False)
        t0 = time.perf_counter()
        oracle.attn_rows(inp.q_lat, inp.q_rope, inp.c_kv, inp.k_rope, inp.prefix_len, ot.mask,
                         ot.n_nodes, inp.scale, rows[pick])
        t_s = time.perf_counter() - t0
    else:
        t_s = t_cal
    t_attn = t_s * work.sum() / work[pick].sum()
    sample = (f"tree build + accept on all {wl.B} sequences; attention on {len(pick)} of "
              f"{len(rows)} valid (node, head) rows, scaled by visible keys")
    return t_tree + t_acc + t_attn, cores, sample


# ------------------------------------------------------------------ arms

def reference_arm(args, wl_idx, rank, world):
    if rank != 0:
        return
    import oracle
    oracle.build()
    inp = synth.make_inputs(wl_idx)
    wl = inp.wl
    times = []
    cores = 1
    sample = ""
    for s in range(args.warmup + args.steps):
        t, cores, sample = oracle_step_time(inp, None, attn_budget_s=1.5, seed=s)
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


def sample_leg(ddtree, wl_idx, wl, inp, depth, n_nodes, tree, s, flush, dev, n, torch):
    """ddt_tree_sample at temperature 1 and in the greedy limit, each as a
    CUDA graph; per call: time, logits bytes / time against the measured HBM
    peak, and the acceptance the samples give."""
    lg, u = synth.sampling_inputs(wl_idx, depth, n_nodes, inp.draft_tok)
    logits = torch.from_numpy(lg).to(dev)
    u01 = torch.from_numpy(u).to(dev)
    del lg
    sample_tok = torch.empty(wl.B, wl.Qc, dtype=torch.int32, device=dev)
    node_p = torch.empty(wl.B, wl.Qc, dtype=torch.float32, device=dev)
    clean = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev).fill_(1.0)
    sink = torch.empty((), dtype=torch.float32, device=dev)
    hbm_gbs, _, peak_src = load_peaks()
    nbytes = logits.numel() * 4 + u01.numel() * 4 + sample_tok.numel() * 4 + node_p.numel() * 4
    out = {"rows": wl.B * wl.Qc, "vocab": wl.vocab, "logits_bytes": logits.numel() * 4,
           "algorithmic_bytes_per_call": nbytes}
    for name, tau in (("temperature_1", 1.0), ("greedy", 0.0)):
        with torch.cuda.stream(s):
            ddtree.ddt_tree_sample(tree, logits, tau, u01, sample_tok, node_p, stream=s)
        torch.cuda.synchronize()
        gs = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gs, stream=s):
            ddtree.ddt_tree_sample(tree, logits, tau, u01, sample_tok, node_p, stream=s)
        evs = []
        with torch.cuda.stream(s):
            for it in range(n + 3):
                flush.fill_(1)
                torch.sum(clean, dim=0, out=sink)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(s)
                gs.replay()
                e1.record(s)
                evs.append((e0, e1))
        torch.cuda.synchronize()
        ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs[3:])
        gbs = nbytes / (ms / 1e3) / 1e9
        out[name] = {"us": ms * 1e3, "achieved_gbs": gbs, "peak_gbs": hbm_gbs, "frac": gbs / hbm_gbs}
    # acceptance of the temperature-1 samples (the last timed calls were greedy)
    with torch.cuda.stream(s):
        ddtree.ddt_tree_sample(tree, logits, 1.0, u01, sample_tok, node_p, stream=s)
        acc = ddtree.ddt_tree_accept(tree, sample_tok, stream=s)
    torch.cuda.synchronize()
    out["mean_accept_len_temperature_1"] = float(acc.accept_len.float().mean().item())
    out["peak_source"] = f"{peak_src} HBM copy bandwidth"
    out["bound"] = "hbm"
    del logits, clean
    return out


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

    inp = synth.make_inputs(wl_idx)
    wl = inp.wl

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)

    tok, lp, root = i32(inp.draft_tok), torch.from_numpy(inp.draft_lp).to(dev), i32(inp.root_tok)
    q_lat, q_rope, c_kv, k_rope = bf16(inp.q_lat), bf16(inp.q_rope), bf16(inp.c_kv), bf16(inp.k_rope)
    pl = i32(inp.prefix_len)
    # target argmax of the synthetic target model needs the tree: build it
    # once on the device, outside any timed region
    tree0 = ddtree.ddt_tree_build(tok, lp, root, wl.budget, wl.vocab)
    depth = tree0.depth.cpu().numpy()
    n_nodes = tree0.n_nodes.cpu().numpy()
    tg = i32(synth.synth_target_argmax(depth, n_nodes, inp.draft_tok, inp.target_u,
                                       inp.target_alt, wl.p_match))
    step = ddtree.VerifyStep(tok, lp, root, wl.vocab, wl.budget, q_lat, q_rope, c_kv, k_rope, pl,
                             tg, inp.scale)
    plan_nsplit = step.ws_bytes and (step.ws_bytes // (wl.B * wl.Qc * wl.H * 513 * 4)) or 1
    # tree build, attention, and the merge that also runs the accept (or the
    # accept alone when the key range is not split)
    launches_per_step = 3

    s = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    with torch.cuda.stream(s):
        step.run(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step.run(s)
    # attention alone (the dominant kernel), also as a graph
    attn_out = torch.empty_like(step.out)
    attn_lse = torch.empty_like(step.lse)
    with torch.cuda.stream(s):
        ddtree.ddt_verify_mla_attn(q_lat, q_rope, c_kv, k_rope, pl, step.tree, inp.scale,
                                   attn_out, attn_lse, step.workspace, stream=s)
    torch.cuda.synchronize()
    ga = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ga, stream=s):
        ddtree.ddt_verify_mla_attn(q_lat, q_rope, c_kv, k_rope, pl, step.tree, inp.scale,
                                   attn_out, attn_lse, step.workspace, stream=s)

    def timed(graph, n):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        with torch.cuda.stream(s):
            for e0, e1 in evs:
                flush.fill_(1)          # evict L2, outside the timed window
                e0.record(s)
                graph.replay()
                e1.record(s)
        return evs

    # warm-up
    for e0, e1 in timed(g, args.warmup):
        pass
    torch.cuda.synchronize()

    # ---- timed region: K graph-replayed steps
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        evs = timed(g, args.steps)
        torch.cuda.synchronize()
    if pg:
        pg.barrier()
    step_ms = [e0.elapsed_time(e1) for e0, e1 in evs]
    total_ms = max_over_ranks(sum(step_ms), world)
    ms_per_step = total_ms / args.steps
    value = world * 1000.0 / ms_per_step

    # ---- dominant kernel: attention alone, same protocol
    for _ in timed(ga, 3):
        pass
    torch.cuda.synchronize()
    aevs = timed(ga, max(args.steps, 10))
    torch.cuda.synchronize()
    attn_ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in aevs)
    flop, algo_bytes = algorithmic_work(depth, n_nodes, inp.prefix_len, wl.H)
    hbm_gbs, bf16_tflops, peak_src = load_peaks()
    t_tensor = flop / (bf16_tflops * 1e12)
    t_hbm = algo_bytes / (hbm_gbs * 1e9)
    attn_s = attn_ms / 1e3
    if t_tensor >= t_hbm:
        roof = {"bound": "tensor", "achieved": flop / attn_s / 1e12, "peak": bf16_tflops,
                "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": algo_bytes / attn_s / 1e9, "peak": hbm_gbs,
                "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = profiled_traffic(wl.name)
    roof["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json burst)" if peak_src == "measured" else peak_src
    roof["kernel"] = "verify_attn_kernel (+ merge_chunks_kernel when the key range is split)"
    roof["algorithmic_flop_per_launch"] = flop
    roof["algorithmic_bytes_per_launch"] = algo_bytes
    roof["launch_ms"] = attn_ms

    # ---- the same attention with the latent output in bfloat16
    out16 = torch.empty(attn_out.shape, dtype=torch.bfloat16, device=dev)
    with torch.cuda.stream(s):
        ddtree.ddt_verify_mla_attn_bf16(q_lat, q_rope, c_kv, k_rope, pl, step.tree, inp.scale, out16, attn_lse,
                                        step.workspace, stream=s)
    torch.cuda.synchronize()
    gb = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gb, stream=s):
        ddtree.ddt_verify_mla_attn_bf16(q_lat, q_rope, c_kv, k_rope, pl, step.tree, inp.scale, out16, attn_lse,
                                        step.workspace, stream=s)
    for _ in timed(gb, 3):
        pass
    torch.cuda.synchronize()
    bevs = timed(gb, max(args.steps, 10))
    torch.cuda.synchronize()
    bf16_ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in bevs)
    bf16_out = {"us": bf16_ms * 1e3, "tflops": flop / (bf16_ms / 1e3) / 1e12, "vs_float32_out": attn_ms / bf16_ms,
                "out_bytes": int(out16.numel()) * 2}
    del out16

    # ---- the same attention on a block-table (paged) cache: every key row in
    # a shuffled pool with junk rows, gathered by the kernel
    rng = np.random.default_rng(7)
    n_pool = wl.B * inp.Tcap + 1024
    perm = torch.from_numpy(rng.permutation(n_pool)[: wl.B * inp.Tcap].astype(np.int64)).to(dev)
    pool_kv = torch.zeros(n_pool, 512, dtype=torch.bfloat16, device=dev)
    pool_kr = torch.zeros(n_pool, 64, dtype=torch.bfloat16, device=dev)
    pool_kv[perm] = c_kv.reshape(-1, 512)
    pool_kr[perm] = k_rope.reshape(-1, 64)
    kv_index = perm.to(torch.int32).reshape(wl.B, inp.Tcap).contiguous()
    with torch.cuda.stream(s):
        ddtree.ddt_verify_mla_attn_paged(q_lat, q_rope, pool_kv, pool_kr, pl, kv_index, step.tree, inp.scale,
                                         attn_out, attn_lse, step.workspace, stream=s)
    torch.cuda.synchronize()
    gp = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gp, stream=s):
        ddtree.ddt_verify_mla_attn_paged(q_lat, q_rope, pool_kv, pool_kr, pl, kv_index, step.tree, inp.scale,
                                         attn_out, attn_lse, step.workspace, stream=s)
    for _ in timed(gp, 3):
        pass
    torch.cuda.synchronize()
    pevs = timed(gp, max(args.steps, 10))
    torch.cuda.synchronize()
    paged_ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in pevs)
    paged = {"us": paged_ms * 1e3, "tflops": flop / (paged_ms / 1e3) / 1e12,
             "vs_contiguous": attn_ms / paged_ms, "pool_rows": n_pool,
             "note": "block table of page size 1 over a shuffled pool; the producer warp gathers rows with cp.async"}
    del pool_kv, pool_kr, kv_index, perm

    # ---- the KV commit after accept (the append of the accepted path's keys),
    # timed alone on scratch copies of the cache; the prefix lengths it
    # advances are reset before each call, outside the timed window
    kv_s, kr_s = c_kv.clone(), k_rope.clone()
    pl0 = pl.clone()
    pl_s, st_s = pl.clone(), torch.zeros_like(pl)
    with torch.cuda.stream(s):
        ddtree.ddt_kv_commit(step.acc, kv_s, kr_s, pl_s, st_s, stream=s)
    torch.cuda.synchronize()
    gk = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gk, stream=s):
        ddtree.ddt_kv_commit(step.acc, kv_s, kr_s, pl_s, st_s, stream=s)
    k_ms = []
    with torch.cuda.stream(s):
        for it in range(max(args.steps, 10) + 3):
            pl_s.copy_(pl0)
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            gk.replay()
            e1.record(s)
            k_ms.append((e0, e1))
    torch.cuda.synchronize()
    kv_commit_ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in k_ms[3:])
    moved_rows = int((step.acc.accept_len.cpu().numpy().astype(np.int64) - 1).sum())
    kv_commit = {"us": kv_commit_ms * 1e3, "moved_rows": moved_rows,
                 "bytes_per_call": moved_rows * 1152 * 2,
                 "note": "latency-bound: one block per sequence, at most 16 rows of 1152 B moved"}
    del kv_s, kr_s

    # ---- temperature sampling at every tree node (the sampling commit path)
    # on synthetic target logits [B,Qc,V] float32, then the accept walk on the
    # samples; the kernel streams the logits once, so it is HBM-bound. Timed
    # after writing the L2 flush buffer and then reading another buffer of
    # that size, so the kernel starts on a cold L2 that holds no dirty lines.
    sample = sample_leg(ddtree, wl_idx, wl, inp, depth, n_nodes, step.tree, s, flush, dev,
                        max(args.steps, 10), torch)

    # ---- end to end through the public API with host buffers: the step's
    # inputs sit in one pinned host buffer laid out like one device buffer
    # whose views are the step's input tensors (one copy in), the node KV rows
    # go one copy per sequence and tensor, and the accept result comes back in
    # one copy (its four arrays are views of one device buffer)
    D1 = wl.D + 1
    fields = [("tok", (wl.B, wl.D, wl.K), torch.int32, inp.draft_tok), ("lp", (wl.B, wl.D, wl.K), torch.float32,
              inp.draft_lp), ("root", (wl.B,), torch.int32, inp.root_tok),
              ("ql", (wl.B, wl.Qc, wl.H, 512), torch.int16, inp.q_lat.view(np.int16)),
              ("qr", (wl.B, wl.Qc, wl.H, 64), torch.int16, inp.q_rope.view(np.int16)),
              ("tg", (wl.B, wl.Qc), torch.int32, tg.cpu().numpy()), ("pl", (wl.B,), torch.int32, inp.prefix_len)]

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
    step_e = ddtree.VerifyStep(dv["tok"], dv["lp"], dv["root"], wl.vocab, wl.budget, dv["ql"].view(torch.bfloat16),
                               dv["qr"].view(torch.bfloat16), c_kv, k_rope, dv["pl"], dv["tg"], inp.scale,
                               acc=ddtree.Accept(ov["accept_len"], ov["accept_idx"], ov["commit_tok"],
                                                 ov["next_root"]))
    node_rows = [(b, int(inp.prefix_len[b])) for b in range(wl.B)]
    h_ckv_nodes = [torch.from_numpy(np.ascontiguousarray(inp.c_kv[b, T:T + wl.Qc].view(np.int16))).pin_memory()
                   for b, T in node_rows]
    h_kr_nodes = [torch.from_numpy(np.ascontiguousarray(inp.k_rope[b, T:T + wl.Qc].view(np.int16))).pin_memory()
                  for b, T in node_rows]
    ckv16, kr16 = c_kv.view(torch.int16), k_rope.view(torch.int16)
    h2d = h_in.numel() + sum(t.numel() * t.element_size() for t in [*h_ckv_nodes, *h_kr_nodes])
    d2h = h_out.numel()

    def e2e_step():
        d_in.copy_(h_in, non_blocking=True)
        for (b, T), hc, hk in zip(node_rows, h_ckv_nodes, h_kr_nodes):
            ckv16[b, T:T + wl.Qc].copy_(hc, non_blocking=True)
            kr16[b, T:T + wl.Qc].copy_(hk, non_blocking=True)
        step_e.run(s)
        h_out.copy_(d_out, non_blocking=True)

    with torch.cuda.stream(s):
        for _ in range(args.warmup):
            e2e_step()
    torch.cuda.synchronize()
    # the whole step, copies included, as one graph: one launch a step, as a
    # serving loop would replay it
    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_e2e, stream=s):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = []
    with torch.cuda.stream(s):
        g_e2e.replay()
        torch.cuda.synchronize()
        h_out.zero_()  # the timed steps must bring the result back themselves
        for _ in range(args.steps):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            g_e2e.replay()
            e1.record(s)
            e1.synchronize()  # the host needs the accept result before the next step
            e2e_ms.append(e0.elapsed_time(e1))
    e2e_value = world * 1000.0 / statistics.mean(e2e_ms)
    # the result that came back is the device's
    assert np.array_equal(h_out[:wl.B * 4].view(torch.int32).numpy(), step_e.acc.accept_len.cpu().numpy())

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {**config_dict(wl, inp), "graph": True, "key_range_splits": plan_nsplit,
                   "sequences_per_s": value * wl.B,
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "attn_tflops": flop / attn_s / 1e12,
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "how": "one CUDA graph per step: copies in from pinned host memory, ddt_verify_step, "
                       "accept result copied out; host waits on it every step"},
        "gpu_launches": launches_per_step * args.steps,
        "kv_commit": kv_commit,
        "paged_attn": paged,
        "bf16_out_attn": bf16_out,
        "tree_sample": sample,
        "clocks": clk.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        t, cores, sample = oracle_step_time(inp, None, attn_budget_s=12.0, seed=1)
        line["cpu_baseline"] = {"value": 1.0 / t, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=1, help="index into synth.WORKLOADS")
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--no-cpu-baseline", action="store_true")
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
