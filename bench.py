"""Benchmark: verified draft positions per second on GB300.

Default workload (one "step" = one call of the verification path over one
batch): chain verification with sampling, B=64 rows, K=8 draft tokens,
V=128256 (Llama-3-8B vocabulary), bf16 logits, temperature 0.7, per-row draft
noise. The step runs the rowscan pass (normalisers of all 1088 rows), the
acceptance decision and the residual / bonus draw.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload chain_batched|chain_single|chain_deep|greedy|tree|entropy|
                                warped|nucleus|kv_compact|merge|expand]

Under torchrun each rank verifies its own batch (seed + rank) on its own GPU:
rows are independent, so there is no collective in the data path (weak
scaling); a barrier brackets the timed region and the max time over ranks is
reported. ``--impl reference`` times the fp64 CPU oracle instead (rank 0).

Prints one JSON line.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified draft positions/sec & logit-read HBM GB/s (B=64,K=8,V=128256)"
L2_BYTES = 129 * 1024 * 1024


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_seed(seed: int, rank: int) -> int:
    """Each rank verifies its own batch: the generator seed is offset by the rank."""
    return seed + rank


def max_over_ranks(x: float, ws: int, device=None) -> float:
    """The slowest rank's time (all ranks get it); x itself when ws == 1."""
    if ws <= 1:
        return float(x)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput(units_per_step: float, steps: int, ws: int, total_ms: float) -> float:
    """Whole-job units per second: every rank does `steps` steps of
    `units_per_step` units within the slowest rank's time."""
    return units_per_step * steps * ws / (total_ms / 1e3)


# ------------------------------------------------------------- workloads --

def make_workload(name: str, seed: int):
    import gen

    if name == "chain_batched":
        c = gen.config_chain_batched(seed)
        return c, dict(workload="chain verify, batched serving: B=64 K=8 V=128256 bf16 T=0.7, draft noise "
                                "sigma_b~U(0.2,2)", B=64, K=8, V=128256, logits="bf16", temperature=0.7)
    if name == "chain_single":
        c = gen.config_chain_single(seed, T=1.0)
        return c, dict(workload="chain verify, single stream: B=1 K=5 V=128256 bf16 T=1", B=1, K=5, V=128256,
                       logits="bf16", temperature=1.0)
    if name == "chain_deep":
        c = gen.config_chain_deep(seed)
        return c, dict(workload="chain verify, deep drafts: B=256 K=16 V=152064 fp32 T=1", B=256, K=16, V=152064,
                       logits="f32", temperature=1.0)
    if name == "greedy":
        c = gen.chain_zipf(64, 8, 128256, __import__("torch").bfloat16, 0.0, 0.3, seed, name="greedy")
        return c, dict(workload="greedy chain verify: B=64 K=8 V=128256 bf16 T=0", B=64, K=8, V=128256,
                       logits="bf16", temperature=0.0)
    if name == "tree":
        t = gen.config_tree(seed)
        return t, dict(workload="merged-tree greedy verify + confidence routing: B=16 N=61 V=128256 bf16", B=16,
                       N=61, V=128256, logits="bf16")
    if name == "warped":
        c = gen.chain_zipf(64, 8, 128256, __import__("torch").bfloat16, 0.7, gen.workloads._sigma_spread, seed,
                           name="chain_batched", draft_top_k=50)
        c.top_k, c.top_p = 50, 0.9
        return c, dict(workload="chain verify with top-k 50 and top-p 0.9 on both models: B=64 K=8 V=128256 bf16 "
                                "T=0.7, draft noise sigma_b~U(0.2,2)", B=64, K=8, V=128256, logits="bf16",
                       temperature=0.7, top_k=50, top_p=0.9)
    if name == "nucleus":
        c = gen.chain_zipf(64, 8, 128256, __import__("torch").bfloat16, 0.7, gen.workloads._sigma_spread, seed,
                           name="chain_batched")
        c.top_k, c.top_p = 0, 0.95
        return c, dict(workload="chain verify with top-p 0.95 alone on both models (nuclei of thousands of tokens): "
                                "B=64 K=8 V=128256 bf16 T=0.7, draft noise sigma_b~U(0.2,2)", B=64, K=8, V=128256,
                       logits="bf16", temperature=0.7, top_k=0, top_p=0.95)
    if name == "entropy":
        t = gen.config_tree(seed)
        t.Ld = gen.tree_draft_logits(t, seed)
        return t, dict(workload="entropy routing of merged drafter trees: B=16 N=61 V=128256 bf16 drafter logits, T=1",
                       B=16, N=61, V=128256, logits="bf16", temperature=1.0)
    raise SystemExit(f"unknown workload {name}")


def units_per_step(name, w):
    if name in ("tree", "entropy"):
        return w.B * (w.N - 1)  # verified nodes
    return w.B * w.K  # verified draft positions


def algorithmic_bytes(name, w):
    """Logit bytes the dominant kernel (the rowscan pass) must read per
    launch: every row once."""
    es = w.Lt.element_size() if name in ("tree", "entropy") else w.Lp.element_size()
    if name in ("tree", "entropy"):
        return w.B * w.N * w.V * es
    if name == "greedy" or w.T == 0.0:
        return w.B * (w.K + 1) * w.V * es
    return w.B * (2 * w.K + 1) * w.V * es


# ---------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(gpu_index)], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        busy = [r for r in rows if r["power"] > 200.0] or rows
        reasons = set()
        for r in busy:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                              ("pcap", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in busy), "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(busy)}


# --------------------------------------------------------------- our arm --

def traffic_for(kernel_key: str):
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu
    summary, valid only while the kernel's source is unchanged."""
    import hashlib

    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
        ent = t[kernel_key]
        src = open(os.path.join(ROOT, ent["source"]), "rb").read()
        if hashlib.sha256(src).hexdigest()[:16] != ent["source_sha"]:
            return None
        return ent["bytes_per_launch"]
    except Exception:
        return None


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import speculative_decoding_verification_29_gb300 as sv

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=dev)
    w, cfg = make_workload(args.workload, rank_seed(args.seed, rank))
    name = args.workload
    stream = torch.cuda.current_stream()
    alg = algorithmic_bytes(name, w)
    # inputs smaller than twice L2 rotate over copies so that consecutive
    # steps never find their logits in L2
    n_sets = max(1, -(-2 * L2_BYTES // alg)) if alg < 2 * L2_BYTES else 1

    pass_only = None
    if name == "entropy":
        sets = [w.Ld.to(dev) for _ in range(n_sets)]
        ws_t = sv.alloc_workspace(sv.workspace_bytes(w.B, w.N, w.V, w.Ld.dtype), dev)
        out = sv.spec_tree_entropy(sets[0], w.n1, 1.0, workspace=ws_t)

        def step_dev(i):
            sv.spec_tree_entropy(sets[i % n_sets], w.n1, 1.0, out=out, workspace=ws_t)

        def step_split(i, ev):
            ev[0].record(stream)
            sv.spec_tree_entropy(sets[i % n_sets], w.n1, 1.0, out=out, workspace=ws_t)
            ev[1].record(stream)

        launches_per_step = 2
        timed_kernel = "rowscan_kernel (entropy) + tree_entropy_kernel (one call)"
        host = [w.Ld]
    elif name == "tree":
        sets = [tuple(t.to(dev) for t in (w.Lt, w.tok, w.R, w.mask, w.conf)) for _ in range(n_sets)]
        ws_t = sv.alloc_workspace(sv.workspace_bytes(w.B, w.N - 1, w.V, w.Lt.dtype), dev)
        out = sv.spec_verify_tree_greedy(*sets[0][:3], w.n1, tree_mask=sets[0][3], workspace=ws_t)
        cout = sv.spec_tree_confidence(sets[0][4], w.n1)

        def step_dev(i):
            Lt, tok, R, mask, conf = sets[i % n_sets]
            sv.spec_verify_tree_greedy(Lt, tok, R, w.n1, tree_mask=mask, out=out, workspace=ws_t)
            sv.spec_tree_confidence(conf, w.n1, out=cout)

        def step_split(i, ev):
            Lt, tok, R, mask, conf = sets[i % n_sets]
            ev[0].record(stream)
            sv.spec_verify_tree_greedy(Lt, tok, R, w.n1, tree_mask=mask, out=out, workspace=ws_t)
            ev[1].record(stream)
            sv.spec_tree_confidence(conf, w.n1, out=cout)

        launches_per_step = 3
        timed_kernel = "rowscan_kernel + tree_finish_kernel (one call)"
        host = [w.Lt, w.tok, w.R, w.mask, w.conf]
    else:
        sets = [tuple(t.to(dev) for t in (w.Lp, w.Lq, w.x, w.ua, w.ur)) for _ in range(n_sets)]
        T = w.T
        ws_t = sv.alloc_workspace(sv.workspace_bytes(w.B, w.K, w.V, w.Lp.dtype), dev)
        if T == 0.0:
            out = sv.spec_verify_chain_greedy(sets[0][0], sets[0][2], workspace=ws_t)

            def step_dev(i):
                Lp, Lq, x, ua, ur = sets[i % n_sets]
                sv.spec_verify_chain_greedy(Lp, x, out=out, workspace=ws_t)

            def step_split(i, ev):
                Lp, Lq, x, ua, ur = sets[i % n_sets]
                ev[0].record(stream)
                sv.spec_verify_chain_greedy(Lp, x, out=out, workspace=ws_t)
                ev[1].record(stream)

            timed_kernel = "rowscan_kernel + greedy_decide_kernel (one call)"
        elif name in ("warped", "nucleus"):
            ws_t = sv.alloc_workspace(sv.warped_workspace_bytes(w.B, w.K, w.V, w.Lp.dtype), dev)
            out = sv.spec_verify_chain_warped(*sets[0], T, w.top_k, w.top_p, workspace=ws_t)

            def step_dev(i):
                sv.spec_verify_chain_warped(*sets[i % n_sets], T, w.top_k, w.top_p, out=out, workspace=ws_t)

            def step_split(i, ev):
                ev[0].record(stream)
                sv.spec_verify_chain_warped(*sets[i % n_sets], T, w.top_k, w.top_p, out=out, workspace=ws_t)
                ev[1].record(stream)

            timed_kernel = ("rowscan_kernel + warp_select_kernel + chain_tail_kernel (one call)" if name == "warped"
                            else "rowscan_kernel + warp_select_kernel + topp_rows_kernel + chain_tail_kernel (one call)")
        else:
            out = sv.spec_verify_chain(*sets[0], T, workspace=ws_t)
            # one prepared call per rotating input set (the serving-loop form of the API)
            calls = [sv.prepare_verify_chain(*sets[j], T, out=out, workspace=ws_t) for j in range(n_sets)]

            def step_dev(i):
                calls[i % n_sets]()

            def step_split(i, ev):
                args_ = sets[i % n_sets]
                ev[0].record(stream)
                sv.spec_chain_scan(*args_, T, out, ws_t)
                ev[1].record(stream)
                sv.spec_chain_sample(*args_, T, out, ws_t)

            def pass_only(i):  # the streaming pass alone (its launches overlap as in a step)
                sv.spec_chain_scan(*sets[i % n_sets], T, out, ws_t)

            timed_kernel = "rowscan_kernel"
        # the nucleus workload: the warp path's probe, then the radix select of the rows it defers
        launches_per_step = {"warped": 3, "nucleus": 4}.get(name, 2)
        host = [w.Lp, w.Lq, w.x, w.ua, w.ur]

    # warm-up, then a short untimed soak so the clock sampler sees the load
    for i in range(max(args.warmup, 3)):
        step_dev(i)
    torch.cuda.synchronize()
    clocks = ClockSampler(local) if rank == 0 else None
    t_soak = time.time()
    while time.time() - t_soak < args.soak:
        for i in range(20):
            step_dev(i)
        torch.cuda.synchronize()

    # --graph: each step captured once as a CUDA graph (one per input copy)
    # and replayed. Eager launches through the API are the default: a graph
    # launch per step ends the programmatic overlap between consecutive
    # steps, which costs more than the host launches it saves here.
    graphs, launch_mode = None, "eager"
    if args.graph:
        try:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                for i in range(n_sets):
                    step_dev(i)
            torch.cuda.current_stream().wait_stream(side)
            torch.cuda.synchronize()
            graphs = []
            for i in range(n_sets):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    step_dev(i)
                graphs.append(g)
            launch_mode = "cuda_graph"
        except Exception as e:  # report and time the eager path instead
            graphs, launch_mode = None, f"eager (graph capture failed: {type(e).__name__})"
    run_step = (lambda i: graphs[i % n_sets].replay()) if graphs else step_dev
    for i in range(max(args.warmup, 3)):
        run_step(i)
    torch.cuda.synchronize()

    # timed region: K steps back to back, events only around the whole run
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(args.steps):
        run_step(i)
    end.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    total_ms = max_over_ranks(start.elapsed_time(end), ws, dev)

    # the dominant kernel: the same K steps again with events around the
    # streaming pass (an event between the two stages delays the second one,
    # so these steps are not the ones `value` is taken from)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    for i in range(args.steps):
        step_split(i, evs[i])
    torch.cuda.synchronize()
    k1_ms = [e[0].elapsed_time(e[1]) for e in evs]
    # the chain workloads' dominant kernel alone: K launches of the streaming
    # pass back to back, events around the run. The events around each pass
    # above keep it from launching while the tail before it drains (its
    # programmatic early launch), so they add that launch latency to it.
    k1_alone = None
    if pass_only is not None:
        pa, pb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for i in range(3):
            pass_only(i)
        torch.cuda.synchronize()
        pa.record(stream)
        for i in range(args.steps):
            pass_only(i)
        pb.record(stream)
        torch.cuda.synchronize()
        k1_alone = pa.elapsed_time(pb) / args.steps

    # end to end through the public API with pinned host buffers (the chain
    # paths through the host-buffer entry point: the library stages the
    # inputs, verifies and copies the outputs back in one call)
    pinned = [h.pin_memory() for h in host]
    h2d = sum(h.numel() * h.element_size() for h in pinned)
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    host_chain = name not in ("entropy", "tree", "warped", "nucleus")
    if host_chain and w.T == 0.0:  # greedy: only the target logits and the draft tokens are copied
        h2d = pinned[0].numel() * pinned[0].element_size() + pinned[2].numel() * pinned[2].element_size()
    if host_chain:
        hws = sv.alloc_workspace(sv.host_workspace_bytes(w.B, w.K, w.V, w.Lp.dtype), dev)
        hout = dict(accept_len=torch.empty(w.B, dtype=torch.int32).pin_memory(),
                    out_tokens=torch.empty(w.B, w.K + 1, dtype=torch.int32).pin_memory(),
                    row_status=torch.empty(w.B, dtype=torch.int32).pin_memory())
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    d2h = 0
    for _ in range(e2e_steps):
        if name == "entropy":
            o = sv.spec_tree_entropy(pinned[0], w.n1, 1.0, device=dev, node_entropy=False)
            res = [o["choice"].cpu(), o["scores"].cpu()]
        elif name == "tree":
            o = sv.spec_verify_tree_greedy(pinned[0], pinned[1], pinned[2], w.n1, tree_mask=pinned[3], device=dev)
            co = sv.spec_tree_confidence(pinned[4], w.n1, device=dev)
            res = [o["accept_len"].cpu(), o["out_tokens"].cpu(), co["choice"].cpu()]
        elif name in ("warped", "nucleus"):
            o = sv.spec_verify_chain_warped(*pinned, w.T, w.top_k, w.top_p, device=dev)
            res = [o["accept_len"].cpu(), o["out_tokens"].cpu()]
        else:  # sampling or greedy chain: host buffers in, host buffers out
            o = sv.spec_verify_chain_host(*pinned, w.T, out=hout, workspace=hws, device=dev)
            res = list(o.values())
        d2h = sum(r.numel() * r.element_size() for r in res)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, ws, dev)
    clk = clocks.stop() if clocks else None

    units = units_per_step(name, w)
    value = throughput(units, args.steps, ws, total_ms)
    e2e_value = throughput(units, e2e_steps, ws, e2e_s * 1e3)
    peak, peak_kind = _peaks()
    k1_in_step = float(np.mean(k1_ms))
    k1_mean = k1_alone if k1_alone is not None else k1_in_step
    achieved = alg / (k1_mean / 1e3) / 1e9
    kernel_key = {"tree": "rowscan_argmax_tree", "greedy": "rowscan_argmax_chain",
                  "entropy": "rowscan_entropy_tree"}.get(name, f"rowscan_stats_{name}")
    line = {
        "metric": METRIC if name == "chain_batched" else f"{'routed' if name == 'entropy' else 'verified'} "
                  f"{'nodes' if name in ('tree', 'entropy') else 'draft positions'}/sec ({name})",
        "value": value,
        "unit": "nodes/s" if name in ("tree", "entropy") else "positions/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded generator: peaked logits, Gumbel-max draft tokens)",
        "config": dict(cfg, parallelism=f"replicas x{ws} (independent batches, no data-path collective)",
                       launch=launch_mode,
                       l2=(f"logits {alg / 1e6:.0f} MB per step, {n_sets} rotating copies ({n_sets * alg / 1e6:.0f} MB) "
                          f">= 2 x L2 {L2_BYTES / 1e6:.0f} MB; no flush between steps")),
        "logit_read_gbs": alg / (total_ms / args.steps / 1e3) / 1e9,
        "roofline": {"bound": "hbm", "kernel": timed_kernel, "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic_for(kernel_key), "algorithmic_bytes": alg,
                     "kernel_ms_mean": k1_mean, "kernel_ms_in_step": k1_in_step,
                     "timing": ("the streaming pass alone, K launches back to back" if k1_alone is not None
                                else "events around each call")},
        "e2e": {"value": e2e_value, "unit": "nodes/s" if name in ("tree", "entropy") else "positions/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if name not in ("tree", "entropy"):
        al = out["accept_len"].cpu().numpy()
        line["accept_len_mean"] = float(al[al >= 0].mean())
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(name, w, args.cpu_seconds)
    if ws > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------- KV-cache compaction --

KV_PLANES, KV_S, KV_W, KV_SETS = 64, 2048, 1024, 16  # Llama-3-8B: 32 layers x K/V, 8 KV heads x 128


def kv_setup(seed: int, dev=None):
    """Merged-tree workload (config of the tree bench) and its accepted paths:
    the compaction that follows tree verification. On a device the paths come
    from the library's own tree verification, as a caller would chain the two
    calls; the reference arm (dev None) takes them from the oracle's."""
    import numpy as np

    import gen

    tb = gen.config_tree(seed)
    if dev is None:
        import oracle

        o = oracle.verify_tree_greedy(tb.Lt, tb.tok, tb.R, tb.n1, mask=tb.mask, threads=os.cpu_count() or 1)
        acc, path = o["accept_len"].astype(np.int32), o["path"].astype(np.int32)
    else:
        import torch

        import speculative_decoding_verification_29_gb300 as sv

        v = sv.spec_verify_tree_greedy(tb.Lt.to(dev), tb.tok.to(dev), tb.R.to(dev), tb.n1,
                                       tree_mask=tb.mask.to(dev))
        torch.cuda.synchronize()
        acc = v["accept_len"].cpu().numpy().astype(np.int32)
        path = v["path_nodes"].cpu().numpy().astype(np.int32)
    moved_rows = sum(int(np.sum(path[b, 1:acc[b] + 1] != np.arange(1, acc[b] + 1))) for b in range(tb.B) if acc[b] > 0)
    bases = [np.full(tb.B, 64 + 112 * j, np.int32) for j in range(KV_SETS)]
    cfg = dict(workload=f"KV-cache compaction after merged-tree verify: B={tb.B} N={tb.N}, cache {KV_PLANES} planes "
                        f"(32 layers x K/V) x S={KV_S} x {KV_W} bf16 (8 KV heads x 128)",
               B=tb.B, N=tb.N, planes=KV_PLANES, S=KV_S, W=KV_W, kv="bf16",
               accepted_tokens=int(acc[acc > 0].sum()), moved_rows_per_plane=moved_rows)
    bytes_per_step = moved_rows * KV_PLANES * KV_W * 2 * 2  # each moved row read once and written once
    return tb, acc, path, bases, bytes_per_step, cfg


def run_kv(args):
    import numpy as np
    import torch

    import speculative_decoding_verification_29_gb300 as sv

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    tb, acc, path, bases, bpstep, cfg = kv_setup(rank_seed(args.seed, rank), dev)
    B = tb.B
    kv = torch.empty(KV_PLANES, B, KV_S, KV_W, dtype=torch.int16, device=dev)
    for p in range(KV_PLANES):  # random bits, one plane at a time
        kv[p].random_(-(1 << 15), 1 << 15)
    kv = kv.view(torch.bfloat16)
    acc_d, path_d = torch.as_tensor(acc, device=dev), torch.as_tensor(path, device=dev)
    base_d = [torch.as_tensor(b_, device=dev) for b_ in bases]
    out = sv.spec_kv_compact(kv, base_d[0], acc_d, path_d)
    stream = torch.cuda.current_stream()

    def step_dev(i):  # each step compacts a different region: nothing of the last 15 steps is in L2
        sv.spec_kv_compact(kv, base_d[i % KV_SETS], acc_d, path_d, out=out)

    for i in range(max(args.warmup, 3)):
        step_dev(i)
    torch.cuda.synchronize()
    clocks = ClockSampler(local) if rank == 0 else None
    t_soak = time.time()
    while time.time() - t_soak < args.soak:
        for i in range(50):
            step_dev(i)
        torch.cuda.synchronize()
    # the K steps captured as one CUDA graph and replayed once: one call takes
    # a few microseconds on the GPU, less than a host launch through the API,
    # so eager launches would time the host
    launch = "cuda_graph (the K steps in one graph)"
    try:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step_dev(0)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(args.steps):
                step_dev(i)
        run = graph.replay
        run()
    except Exception as e:
        launch = f"eager (graph capture failed: {type(e).__name__})"

        def run():
            for i in range(args.steps):
                step_dev(i)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    run()
    end.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    total_ms = max_over_ranks(start.elapsed_time(end), ws, dev)
    k_ms = total_ms / args.steps  # one kernel per step: the step time bounds the kernel's duration
    # end to end: paths, lengths and bases from pinned host memory, lengths back
    host = [torch.as_tensor(bases[0]).pin_memory(), torch.as_tensor(acc).pin_memory(), torch.as_tensor(path).pin_memory()]
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        o = sv.spec_kv_compact(kv, host[0], host[1], host[2])
        res = [o["new_len"].cpu(), o["row_status"].cpu()]
    e2e_s = max_over_ranks(time.perf_counter() - t0, ws, dev)
    clk = clocks.stop() if clocks else None
    peak, peak_kind = _peaks()
    gb = bpstep / 1e9
    line = {
        "metric": "KV-cache compaction: cache bytes moved/sec (read + write)", "value": gb * args.steps * ws / (total_ms / 1e3),
        "unit": "GB/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (moved as bits)",
        "data": "synthetic (random cache bits; accepted paths from the oracle's verification of the merged trees)",
        "config": dict(cfg, parallelism=f"replicas x{ws}", launch=launch,
                       l2=f"{KV_SETS} cache regions in rotation, {bpstep / 1e6:.1f} MB moved per step; no flush"),
        "roofline": {"bound": "hbm", "kernel": "kv_compact_kernel", "achieved": gb / (k_ms / 1e3), "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": gb / (k_ms / 1e3) / peak, "traffic": None,
                     "algorithmic_bytes": bpstep, "kernel_ms_mean": k_ms},
        "e2e": {"value": gb * e2e_steps * ws / e2e_s, "unit": "GB/s",
                "h2d_bytes_per_step": sum(h.numel() * h.element_size() for h in host),
                "d2h_bytes_per_step": sum(r.numel() * r.element_size() for r in res), "steps": e2e_steps},
        "gpu_launches": args.steps, "clocks": clk,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = kv_cpu_baseline(tb, acc, path, bpstep, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)


def kv_cpu_baseline(tb, acc, path, bpstep, cpu_seconds, steps=None):
    """The oracle's compaction of the same paths on a host cache holding the
    touched positions (one thread)."""
    import numpy as np

    import oracle

    S = 64 + tb.N + 8
    kv = np.random.default_rng(0).integers(-(1 << 15), 1 << 15, (KV_PLANES, tb.B, S, KV_W)).astype(np.int16)
    base = np.full(tb.B, 64, np.int32)
    reps, t_tot = 0, 0.0
    while reps < (steps or 1) or (steps is None and t_tot < cpu_seconds / 4 and reps < 20):
        t0 = time.perf_counter()
        oracle.kv_compact(kv, KV_PLANES, tb.B, S, KV_W, (tb.B * S * KV_W, S * KV_W, KV_W), base, acc, path=path)
        t_tot += time.perf_counter() - t0
        reps += 1
    return {"value": bpstep / 1e9 * reps / t_tot, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{reps} compactions of a {S}-position host cache with the same paths (the oracle copies the "
                      f"whole cache each call: {t_tot:.1f} s)"}


# ------------------------------------------------------ oracle (CPU) arm --

def _oracle_step(name, w, rows, threads):
    import torch

    import oracle

    idx = torch.as_tensor(rows)
    if name == "entropy":
        oracle.tree_entropy(w.Ld[idx], w.n1)
    elif name == "tree":
        oracle.verify_tree_greedy(w.Lt[idx], w.tok[idx], w.R[idx], w.n1, mask=w.mask[idx], threads=threads)
        oracle.tree_confidence(w.conf[idx], w.n1)
    elif name in ("warped", "nucleus"):
        oracle.verify_chain_warped(w.Lp[idx], w.Lq[idx], w.x[idx], w.ua[idx], w.ur[idx], w.T, w.top_k, w.top_p,
                                   threads=threads)
    elif w.T == 0.0:
        oracle.verify_chain_greedy(w.Lp[idx], w.x[idx], threads=threads)
    else:
        oracle.verify_chain(w.Lp[idx], w.Lq[idx], w.x[idx], w.ua[idx], w.ur[idx], w.T, threads=threads)


def _sample_rows(name, w, threads, budget_s):
    """Rows per oracle step so that one step takes about budget_s seconds."""
    t0 = time.perf_counter()
    _oracle_step(name, w, [0], 1)
    one = max(time.perf_counter() - t0, 1e-4)
    n = int(budget_s * threads / one)
    return max(1, min(w.B, n)), one


def cpu_baseline(name, w, cpu_seconds):
    """The oracle timed on this host's cores over whole batches of the same
    workload, repeated until about `cpu_seconds` of CPU time were spent."""
    threads = os.cpu_count() or 1
    rows = list(range(w.B))
    reps, t_tot = 0, 0.0
    while reps < 1 or (t_tot * min(threads, w.B) < cpu_seconds and reps < 50):
        t0 = time.perf_counter()
        _oracle_step(name, w, rows, threads)
        t_tot += time.perf_counter() - t0
        reps += 1
    per_row_units = (w.N - 1) if name in ("tree", "entropy") else w.K
    cores = min(threads, w.B) if name != "entropy" else 1
    return {"value": w.B * per_row_units * reps / t_tot, "unit": "nodes/s" if name in ("tree", "entropy") else "positions/s",
            "cores": cores, "kind": "oracle",
            "sample": f"all {w.B} rows of the batch, {reps} repeats, fp64 C oracle on {cores} threads "
                      f"({t_tot:.1f} s wall, about {t_tot * cores:.0f} CPU-s)"}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import oracle

    oracle.build()
    w, cfg = make_workload(args.workload, args.seed)
    name = args.workload
    threads = os.cpu_count() or 1
    step_budget = max(0.2, min(2.0, 120.0 / max(1, args.steps + args.warmup)))
    n, _ = _sample_rows(name, w, threads, step_budget)
    rows = list(range(n))
    for _ in range(args.warmup):
        _oracle_step(name, w, rows, threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(name, w, rows, threads)
    dt = time.perf_counter() - t0
    per_row_units = (w.N - 1) if name in ("tree", "entropy") else w.K
    value = n * per_row_units * args.steps / dt
    unit = "nodes/s" if name in ("tree", "entropy") else "positions/s"
    line = {
        "impl": "reference",
        "metric": METRIC if name == "chain_batched" else f"verified positions/sec ({name})",
        "value": value, "unit": unit, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (same seeded generator)", "config": cfg,
        "cpu_baseline": {"value": value, "unit": unit, "cores": min(threads, n), "kind": "oracle",
                         "sample": f"each step verifies {n} of {w.B} rows of the batch on {min(threads, n)} threads"},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def merge_setup(seed: int):
    """Per-row drafter trees of the merged-tree workload (two 30-node trees per
    row, B=16), as the two drafters hand them over."""
    import numpy as np
    import torch

    import gen

    tb = gen.config_tree(seed)

    def batched(parents, toks):
        per = [gen.tree_from_parents(p) for p in parents]
        D = max(R.shape[1] for R, _, _ in per)
        Rn = max(R.shape[0] for R, _, _ in per)
        n = len(parents[0]) - 1
        R = torch.full((tb.B, Rn, D), -1, dtype=torch.int32)
        mask = torch.zeros(tb.B, n + 1, n + 1, dtype=torch.uint8)
        pos = torch.zeros(tb.B, n + 1, dtype=torch.int32)
        for b, (Rb, mb, pb) in enumerate(per):
            R[b, : Rb.shape[0], : Rb.shape[1]] = Rb
            mask[b], pos[b] = mb, pb
        return [torch.as_tensor(np.array(toks), dtype=torch.int32), mask, R, pos]

    t1 = batched(tb.parents1, tb.tok1)
    t2 = batched(tb.parents2, tb.tok2)
    cfg = dict(workload=f"batched merge of two drafter trees: B={tb.B}, {tb.n1} + {tb.N - 1 - tb.n1} non-root nodes",
               B=tb.B, N=tb.N)
    return tb, t1, t2, cfg


def run_merge(args):
    import torch

    import speculative_decoding_verification_29_gb300 as sv

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    tb, t1, t2, cfg = merge_setup(rank_seed(args.seed, rank))
    d1, d2 = [t.to(dev) for t in t1], [t.to(dev) for t in t2]
    out = sv.spec_merge_trees(*d1, *d2)
    stream = torch.cuda.current_stream()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        sv.spec_merge_trees(*d1, *d2)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        for _ in range(args.steps):
            sv.spec_merge_trees(*d1, *d2)
    graph.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(local) if rank == 0 else None
    t_soak = time.time()  # untimed replays so the clock sampler sees the load
    while time.time() - t_soak < max(args.soak, 0.5):
        graph.replay()
        torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    graph.replay()
    end.record(stream)
    torch.cuda.synchronize()
    total_ms = max_over_ranks(start.elapsed_time(end), ws, dev)
    host = [t.pin_memory() for t in t1 + t2]
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        o = sv.spec_merge_trees(*host, device=dev)
        res = [o["tokens"].cpu(), o["mask"].cpu(), o["retrieve"].cpu(), o["pos"].cpu()]
    e2e_s = time.perf_counter() - t0
    clk = clocks.stop() if clocks else None
    nbytes = sum(t.numel() * t.element_size() for t in d1 + d2) + sum(v.numel() * v.element_size()
                                                                     for k, v in out.items() if k != "n1")
    units = tb.B * (tb.N - 1)
    peak, peak_kind = _peaks()
    k_ms = total_ms / args.steps
    line = {"metric": "merged tree nodes/sec (batched merge of two drafter trees)",
            "value": throughput(units, args.steps, ws, total_ms), "unit": "nodes/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": k_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int32 / uint8", "data": "synthetic (the tree workload's drafter trees)",
            "config": dict(cfg, parallelism=f"replicas x{ws}", launch="cuda_graph (the K steps in one graph)"),
            "roofline": {"bound": "hbm", "kernel": "merge_trees_kernel", "achieved": nbytes / (k_ms / 1e3) / 1e9,
                         "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": nbytes / (k_ms / 1e3) / 1e9 / peak, "traffic": None, "algorithmic_bytes": nbytes,
                         "kernel_ms_mean": k_ms},
            "e2e": {"value": throughput(units, e2e_steps, ws, e2e_s * 1e3), "unit": "nodes/s",
                    "h2d_bytes_per_step": sum(h.numel() * h.element_size() for h in host),
                    "d2h_bytes_per_step": sum(r.numel() * r.element_size() for r in res), "steps": e2e_steps},
            "gpu_launches": args.steps, "clocks": clk}
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = merge_cpu_baseline(tb, t1, t2)
    if rank == 0:
        print(json.dumps(line), flush=True)


def merge_cpu_baseline(tb, t1, t2, reps=20):
    import oracle

    t0 = time.perf_counter()
    for _ in range(reps):
        for b in range(tb.B):
            oracle.merge_trees(t1[0][b:b + 1], t1[2][b], t1[1][b], t1[3][b], t2[0][b:b + 1], t2[2][b], t2[1][b],
                               t2[3][b])
    dt = time.perf_counter() - t0
    return {"value": tb.B * (tb.N - 1) * reps / dt, "unit": "nodes/s", "cores": 1, "kind": "oracle",
            "sample": f"{reps} merges of the {tb.B} tree pairs (numpy, one thread: {dt:.2f} s)"}


def run_merge_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    tb, t1, t2, cfg = merge_setup(args.seed)
    b = merge_cpu_baseline(tb, t1, t2, reps=max(1, min(args.steps, 50)))
    print(json.dumps({"impl": "reference", "metric": "merged tree nodes/sec (batched merge of two drafter trees)",
                      "value": b["value"], "unit": "nodes/s", "n_gpus": ws, "steps": args.steps,
                      "warmup": args.warmup, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                      "dtype": "int32 / uint8", "data": "synthetic", "config": cfg, "cpu_baseline": b,
                      "e2e": {"value": b["value"], "unit": "nodes/s", "h2d_bytes_per_step": 0,
                              "d2h_bytes_per_step": 0}}), flush=True)


EXP_B, EXP_F, EXP_M, EXP_V = 64, 10, 10, 128256
EXP_METRIC = "expanded frontier nodes/sec (drafter-tree expansion by cumulative probability)"


def expand_setup(seed: int):
    """One expansion step of 64 drafter trees: 10 frontier nodes per tree,
    the 10 best children kept, Llama-3 vocabulary, bf16 drafter logits."""
    import gen

    Ld, logc = gen.expand_frontier(EXP_B, EXP_F, EXP_V, seed=seed)
    cfg = dict(workload=f"drafter-tree expansion by cumulative probability: B={EXP_B} trees, F={EXP_F} frontier "
                        f"nodes, M={EXP_M} children kept, V={EXP_V} bf16 drafter logits, T=1",
               B=EXP_B, F=EXP_F, M=EXP_M, V=EXP_V)
    return Ld, logc, cfg


def run_expand(args):
    import torch

    import speculative_decoding_verification_29_gb300 as sv

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    Ld, logc, cfg = expand_setup(rank_seed(args.seed, rank))
    alg = Ld.numel() * Ld.element_size() + logc.numel() * 4 + EXP_B * EXP_M * 12
    n_sets = max(1, -(-2 * L2_BYTES // alg))  # consecutive steps never find their logits in L2
    sets = [(Ld.to(dev), logc.to(dev)) for _ in range(n_sets)]
    from speculative_decoding_verification_29_gb300 import _lib

    need = _lib.load().spec_expand_workspace_bytes(EXP_B, EXP_F, EXP_V, EXP_M, _lib.SPEC_BF16)
    ws_t = sv.alloc_workspace(need, dev)
    out = sv.spec_tree_expand(*sets[0], EXP_M, 1.0, workspace=ws_t)
    stream = torch.cuda.current_stream()

    def step_dev(i):
        sv.spec_tree_expand(*sets[i % n_sets], EXP_M, 1.0, out=out, workspace=ws_t)

    for i in range(max(args.warmup, 3)):
        step_dev(i)
    torch.cuda.synchronize()
    clocks = ClockSampler(local) if rank == 0 else None
    t_soak = time.time()
    while time.time() - t_soak < args.soak:
        for i in range(20):
            step_dev(i)
        torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(args.steps):
        step_dev(i)
    end.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    total_ms = max_over_ranks(start.elapsed_time(end), ws, dev)
    # per-call durations on the launching stream, for the roofline
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i, (a, b) in enumerate(evs):
        a.record(stream)
        step_dev(i)
        b.record(stream)
    torch.cuda.synchronize()
    k_ms = sum(a.elapsed_time(b) for a, b in evs) / len(evs)
    host = [Ld.pin_memory(), logc.pin_memory()]
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        o = sv.spec_tree_expand(host[0], host[1], EXP_M, 1.0, workspace=ws_t, device=dev)
        res = [o["parent"].cpu(), o["token"].cpu(), o["score"].cpu(), o["row_status"].cpu()]
    e2e_s = max_over_ranks(time.perf_counter() - t0, ws, dev)
    clk = clocks.stop() if clocks else None
    peak, peak_kind = _peaks()
    units = EXP_B * EXP_F
    line = {
        "metric": EXP_METRIC, "value": throughput(units, args.steps, ws, total_ms), "unit": "nodes/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 logits, f32 arithmetic",
        "data": "synthetic (peaked drafter logits, random path scores)",
        "config": dict(cfg, parallelism=f"replicas x{ws}", launch="eager",
                       l2=f"{n_sets} input copies in rotation ({alg / 1e6:.0f} MB each); no flush"),
        "roofline": {"bound": "hbm",
                     "kernel": "rowscan_kernel + expand_rows_kernel + expand_merge_kernel (one call)",
                     "achieved": alg / (k_ms / 1e3) / 1e9, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": alg / (k_ms / 1e3) / 1e9 / peak, "traffic": None, "algorithmic_bytes": alg,
                     "kernel_ms_mean": k_ms},
        "e2e": {"value": throughput(units, e2e_steps, ws, e2e_s * 1e3), "unit": "nodes/s",
                "h2d_bytes_per_step": sum(h.numel() * h.element_size() for h in host),
                "d2h_bytes_per_step": sum(r.numel() * r.element_size() for r in res), "steps": e2e_steps},
        "gpu_launches": 3 * args.steps, "clocks": clk,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = expand_cpu_baseline(Ld, logc, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)


def expand_cpu_baseline(Ld, logc, cpu_seconds, rows=None):
    """The oracle's expansion of whole trees (batch rows), one at a time, until
    the budget is spent (one thread)."""
    import oracle

    oracle.load()
    reps, t_tot, b = 0, 0.0, 0
    while (rows is None and t_tot < cpu_seconds) or (rows is not None and reps < rows):
        t0 = time.perf_counter()
        oracle.tree_expand(Ld[b:b + 1], logc[b:b + 1].double(), EXP_M)
        t_tot += time.perf_counter() - t0
        reps += 1
        b = (b + 1) % Ld.shape[0]
    return {"value": reps * EXP_F / t_tot, "unit": "nodes/s", "cores": 1, "kind": "oracle",
            "sample": f"{reps} trees of the batch expanded one at a time ({reps * EXP_F} frontier nodes, fp64 "
                      f"log-softmax and a full sort of the F*V children: {t_tot:.1f} s)"}


def run_expand_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    Ld, logc, cfg = expand_setup(args.seed)
    b = expand_cpu_baseline(Ld, logc, 0.0, rows=max(1, min(args.steps, 16)))
    print(json.dumps({"impl": "reference", "metric": EXP_METRIC, "value": b["value"], "unit": "nodes/s",
                      "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
                      "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
                      "cpu_baseline": b, "e2e": {"value": b["value"], "unit": "nodes/s", "h2d_bytes_per_step": 0,
                                                 "d2h_bytes_per_step": 0}}), flush=True)


def run_kv_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import oracle

    oracle.build()
    tb, acc, path, bases, bpstep, cfg = kv_setup(args.seed)
    b = kv_cpu_baseline(tb, acc, path, bpstep, 0.0, steps=max(1, min(args.steps, 20)))
    line = {"impl": "reference", "metric": "KV-cache compaction: cache bytes moved/sec (read + write)",
            "value": b["value"], "unit": "GB/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (moved as bits)",
            "data": "synthetic", "config": cfg, "cpu_baseline": b,
            "e2e": {"value": b["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="chain_batched",
                    choices=["chain_batched", "chain_single", "chain_deep", "greedy", "tree", "entropy", "kv_compact", "merge", "warped", "nucleus",
                             "expand"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--soak", type=float, default=1.0, help="untimed seconds of steps before timing (clock samples)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="CPU work budget of the oracle baseline")
    ap.add_argument("--graph", action="store_true", help="replay each step as a captured CUDA graph")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.workload == "expand":
        if args.impl == "reference":
            run_expand_reference(args)
        else:
            run_expand(args)
    elif args.workload == "merge":
        if args.impl == "reference":
            run_merge_reference(args)
        else:
            run_merge(args)
    elif args.workload == "kv_compact":
        if args.impl == "reference":
            run_kv_reference(args)
        else:
            run_kv(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
