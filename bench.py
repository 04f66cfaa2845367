"""Benchmark of wave-index tripartite decode attention on one B300 (or N
replicas, one per GPU, under torchrun).

One timed step = one decode query batch through every decode row of the hot
path (cluster scoring, top-r selection, steady + retrieval attention with the
estimation zone, log-sum-exp merge) against an index built on the GPU in the
same run.  The index build (segmented spherical k-means + finalize) is timed
in the same run and reported under "build"; "full_pass_ms" is one pass of
every row (build + decode) for one batch.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle
instead (the reference arm), on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import socket
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode attention queries/sec/layer at 128K ctx; achieved HBM GB/s vs 8 TB/s"
UNIT = "queries/s/layer"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="wi", choices=["wi", "reference"])
    ap.add_argument("--workload", default="llama3_8b_128k_b1")
    ap.add_argument("--budget-frac", type=float, default=None,
                    help="retrieval budget as a fraction of clusters (default: workload's)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sdpa", action="store_true",
                    help="skip the full-attention (torch SDPA) context timing")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-build-timing", action="store_true")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the 1M-context and batch-16 decode workloads")
    return ap.parse_args(argv)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=2)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=1)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------
# roofline bookkeeping
# ----------------------------------------------------------------------------
def kernel_source_hash():
    h = hashlib.sha256()
    for name in ("wi_decode.cu", "wi_device.cuh", "wi_internal.h", "wi_assign.cu", "wi_build.cu",
                 "wi_api.cu"):
        with open(os.path.join(ROOT, "cluster_indexed_sparse_wi_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, or None when the
    kernel sources changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    ent = rec.get(workload, {}).get(kernel)
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


def retrieved_unique_bytes(topk, size, G):
    """Bytes of K and V rows of the retrieved clusters, counted once per
    (sequence, KV head, cluster) over the query heads of a group."""
    import torch
    B, Hq, r = topk.shape
    Hkv = Hq // G
    ids = topk.view(B, Hkv, G * r).long()
    total = 0
    for b in range(B):
        for g in range(Hkv):
            u = torch.unique(ids[b, g])
            u = u[u >= 0]
            total += int(size[b, g][u].sum().item())
    return total * 128 * 2 * 2


# ----------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ----------------------------------------------------------------------------
def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        return max([i.get("num_threads", 1) for i in info] + [1])
    except Exception:
        return 1


def oracle_decode_sample(w, g_np, index_np, r, seconds, heads_of_group=0):
    """Times the oracle decode of the query heads of KV head `heads_of_group`
    of sequence 0, repeated until `seconds` of CPU work; returns
    (queries/s/layer, sample description, per-step seconds list)."""
    from oracle import wave_index as wi
    G = w.Hq // w.Hkv
    gsel = heads_of_group
    Kf = wi.bf16_bits_to_f64(g_np["K"][0, gsel])
    Vf = wi.bf16_bits_to_f64(g_np["V"][0, gsel])
    qf = wi.bf16_bits_to_f64(g_np["q"][0])
    hi = {k: index_np[k] for k in ("size", "centroid_key", "value_sum", "perm", "offset")}
    scale = 1.0 / math.sqrt(w.d)
    times = []
    t_end = time.perf_counter() + seconds
    while True:
        t0 = time.perf_counter()
        for h in range(gsel * G, gsel * G + G):
            wi.decode_head(qf[h], Kf, Vf, hi, w.sink, w.window, r, scale)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() > t_end:
            break
    per_query = statistics.mean(times) * (w.Hq / G)  # all Hq heads of one query
    desc = ("oracle decode of the %d query heads of KV head %d of one sequence (of %d), "
            "%d repetitions, scaled to all %d heads" % (G, gsel, w.Hq, len(times), w.Hq))
    return 1.0 / per_query, desc, times


def oracle_index_for_head(w, g_np, b=0, g=0):
    from oracle import wave_index as wi
    Kf = wi.bf16_bits_to_f64(g_np["K"][b, g])
    Vf = wi.bf16_bits_to_f64(g_np["V"][b, g])
    return wi.build_index_head(Kf, Vf, w.sink, w.window, w.seg_len, w.k_per_seg, w.iters)


def run_reference(args, w, r):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from workloads import generate
    t0 = time.perf_counter()
    g_np = generate(w, batches=[0])
    t_gen = time.perf_counter() - t0
    idx = oracle_index_for_head(w, g_np)  # setup, untimed
    from oracle import wave_index as wi
    G = w.Hq // w.Hkv
    Kf = wi.bf16_bits_to_f64(g_np["K"][0, 0])
    Vf = wi.bf16_bits_to_f64(g_np["V"][0, 0])
    qf = wi.bf16_bits_to_f64(g_np["q"][0])
    scale = 1.0 / math.sqrt(w.d)

    def step():
        for h in range(G):
            wi.decode_head(qf[h], Kf, Vf, idx, w.sink, w.window, r, scale)

    for _ in range(args.warmup):
        step()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    per_query = statistics.mean(times) * (w.Hq / G)
    value = 1.0 / per_query
    cores = blas_threads()
    sample = ("each step: oracle decode of the %d query heads of KV head 0 of sequence 0 "
              "(index of that head built by the oracle, untimed); value scaled to all %d heads"
              % (G, w.Hq))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.mean(times) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, r),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
        "setup_seconds": {"generate": t_gen},
    }
    print(json.dumps(line), flush=True)


def replica_workload(w, rank):
    """Rank `rank`'s replica of the workload: the same shapes over its own
    sequences (weak scaling; ranks share no data)."""
    return w if rank == 0 else w.replace(seeds=tuple(s + 100003 * rank for s in w.seeds))


def max_over_ranks(values, dist, device):
    """Element-wise maximum of per-rank timings (the only collective: timing)."""
    import torch
    t = torch.tensor(list(values), device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def workload_config(w, r):
    return {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N, "d": w.d,
            "clusters_per_head": w.n_clusters, "seg_len": w.seg_len, "k_per_seg": w.k_per_seg,
            "kmeans_iters": w.iters, "sink": w.sink, "window": w.window, "r": r,
            "l2": L2_HOW,
            "step": "decode (score + estimate of every cluster; select; attend + merge) over an "
                    "index built in the same run; build timed separately under 'build'"}


L2_HOW = ("flushed before every timed step, outside the events: a 256 MiB write, then a "
          "512 MiB read that evicts the lines the write left dirty, so that no input is "
          "L2-resident and the step does not pay the flush's write-back; the same steps "
          "after the write alone are reported as ms_per_step_write_flush")


class L2Flush:
    """Evicts every L2 line between timed steps: a 256 MiB write (the
    classic flush) followed by a 512 MiB read."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(128 << 20, dtype=torch.float32, device=dev)  # 512 MiB
        self.acc = torch.zeros((), dtype=torch.float32, device=dev)
        self.k = 0

    def write_only(self):
        self.k += 1
        self.w.fill_(self.k & 0xFF)

    def __call__(self):
        import torch
        self.write_only()
        torch.sum(self.r, dim=0, out=self.acc)


def decode_bytes(w, ix, topk, r, index_bytes=4):
    """Algorithmic bytes of one decode step: centroid keys and value sums
    (index_bytes per element: 4 for the f32 index, 2 for the bf16 one) with
    the sizes, once; steady K/V; retrieved K/V once per (sequence, KV head,
    cluster)."""
    C = w.n_clusters
    kbar = w.B * w.Hkv * C * (w.d * index_bytes + 4)
    vsum = w.B * w.Hkv * C * (w.d * index_bytes + 4)
    steady = w.B * w.Hkv * (w.sink + w.window) * w.d * 2 * 2
    retr = retrieved_unique_bytes(topk[..., :r].contiguous(), ix.size, w.Hq // w.Hkv) if r else 0
    return {"centroid_keys": kbar, "value_sums_sizes": vsum, "steady_kv": steady,
            "retrieved_kv_unique": retr}


def measure_variants(w, r, dev, args, pk, flush, ctx):
    """The decode options on the headline workload's index: attention-mass
    ranking, GQA-shared selection, the bf16 index (alone and with sharing),
    and speculative reuse (previous queries equal to the current ones, so
    every group takes its previous set).  Device time of the fused call per
    step, each with its own algorithmic bytes and roofline."""
    import torch
    import cluster_indexed_sparse_wi_b300 as wl
    K, V, q, ix = ctx["K"], ctx["V"], ctx["q"], ctx["ix"]
    stream = torch.cuda.current_stream()
    hbm_peak = float(pk["hbm_gbs"])
    out = []
    variants = (("rank=mass", dict(rank="mass"), {}),
                ("share=group", dict(share="group"), {}),
                ("index=bf16", dict(index_dtype="bf16"), {}),
                ("share=group,index=bf16", dict(share="group", index_dtype="bf16"), {}),
                ("reuse(tau=0.9)", {}, dict(tau=0.9)))
    for name, opts, call in variants:
        dec = wl.Decoder(ix, w.Hq, r, **opts)
        dec(q, K, V)
        torch.cuda.synchronize()
        if call:
            prev = dec.topk[..., :r].clone()
            fn = lambda: dec(q, K, V, with_topk=True, prev_q=q, prev_topk=prev, **call)
        else:
            fn = lambda: dec(q, K, V, with_topk=False)
        for _ in range(max(args.warmup, 3)):
            flush()
            fn()
        gr = wl.capture_graph(fn, dev)
        for _ in range(3):
            flush()
            gr.replay()
        step_ms = timed_steps(gr.replay, flush, args.steps, stream)
        assert dec.status() == 0
        dec(q, K, V, with_topk=True, **({} if not call else dict(prev_q=q, prev_topk=prev, **call)))
        torch.cuda.synchronize()
        by = decode_bytes(w, ix, dec.topk, r, index_bytes=2 if "bf16" in name else 4)
        ms = statistics.mean(step_ms)
        gbs = sum(by.values()) / (ms * 1e-3) / 1e9
        out.append({"variant": name, "ms_per_step": ms, "value": w.B / (ms * 1e-3), "unit": UNIT,
                    "roofline": {"kernel": "decode_kernel", "bound": "hbm", "achieved": gbs,
                                 "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
                                 "algorithmic_bytes_per_launch": sum(by.values())},
                    "bytes": by,
                    "reused_heads": int(dec.reused.sum()) if call else None})
        del dec, gr
    return out


def timed_steps(fn, flush, steps, stream):
    """Event time of `steps` calls of fn, each after flush() (outside the
    events); returns the per-step milliseconds."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        flush()
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def measure_workload(w, r, dev, args, pk, flush, rank=0, want_cpu=False, label=None):
    """Build the index of workload w on the GPU, then time the fused decode
    call (CUDA-graph replays) and its end-to-end host step; returns one
    result dict with its own roofline, clocks and e2e."""
    import torch
    import cluster_indexed_sparse_wi_b300 as wl
    from workloads import generate
    t0 = time.perf_counter()
    wr = replica_workload(w, rank)
    g_np = generate(wr)
    t_gen = time.perf_counter() - t0

    def up(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)

    K, V, q = up(g_np["K"]), up(g_np["V"]), up(g_np["q"])
    cfg = wl.IndexConfig(w.B, w.Hkv, w.N, w.sink, w.window, w.seg_len, w.k_per_seg, w.iters)
    ix = wl.WaveIndex(cfg, dev)
    ix.build(K, V)
    torch.cuda.synchronize()
    assert ix.status() == 0
    stream = torch.cuda.current_stream()
    dec = wl.Decoder(ix, w.Hq, r)
    for _ in range(max(args.warmup, 3)):
        flush()
        dec(q, K, V, with_topk=False)
    torch.cuda.synchronize()
    assert dec.status() == 0
    g_step = dec.capture(q, K, V)
    for _ in range(max(args.warmup, 3)):
        flush()
        g_step.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_uuid_str(dev))
    sampler.start()
    time.sleep(0.3)
    wall0 = time.perf_counter()
    step_ms = timed_steps(g_step.replay, flush, args.steps, stream)
    wall = time.perf_counter() - wall0
    wflush_ms = timed_steps(g_step.replay, flush.write_only, args.steps, stream)
    clocks = sampler.stop()
    assert dec.status() == 0
    # e2e through the public API with host buffers
    dstep = wl.DecodeStep(dec, K, V)
    q_src = q.cpu()
    e2e_ms = []
    for i in range(args.warmup + args.steps):
        flush()
        torch.cuda.synchronize()
        a0 = time.perf_counter()
        out_h, _ = dstep(q_src)
        a1 = time.perf_counter()
        if i >= args.warmup:
            e2e_ms.append((a1 - a0) * 1e3)
    assert torch.isfinite(out_h).all() and dec.status() == 0
    dec(q, K, V, with_topk=True)
    torch.cuda.synchronize()
    by = decode_bytes(w, ix, dec.topk, r)
    step_bytes = sum(by.values())
    ms = statistics.mean(step_ms)
    e2e_mean = statistics.mean(e2e_ms)
    hbm_peak = float(pk["hbm_gbs"])
    gbs = step_bytes / (ms * 1e-3) / 1e9
    res = {
        "workload": label or w.name, "r": r, "ms_per_step": ms,
        "ms_per_step_median": statistics.median(step_ms),
        "ms_per_step_write_flush": statistics.mean(wflush_ms),
        "value": w.B / (ms * 1e-3), "unit": UNIT,
        "roofline": {"kernel": "decode_kernel", "bound": "hbm", "achieved": gbs, "peak": hbm_peak,
                     "unit": "GB/s", "frac": gbs / hbm_peak,
                     "algorithmic_bytes_per_launch": step_bytes, "launch_ms": ms,
                     "frac_of_8tbs": gbs / NOMINAL_HBM_GBS},
        "bytes": by,
        "e2e": {"value": w.B / (e2e_mean * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": dstep.h2d_bytes, "d2h_bytes_per_step": dstep.d2h_bytes,
                "ms_per_step": e2e_mean, "ms_per_step_median": statistics.median(e2e_ms)},
        "clocks": clocks, "gpu_launches": args.steps, "wall_s_timed": wall,
        "setup_seconds": {"generate": t_gen},
    }
    if want_cpu and rank == 0 and not args.no_cpu_baseline:
        index_np = {
            "size": ix.size[0, 0].cpu().numpy().astype(np.int64),
            "centroid_key": ix.centroid_key[0, 0].double().cpu().numpy(),
            "value_sum": ix.value_sum[0, 0].double().cpu().numpy(),
            "perm": ix.perm[0, 0].cpu().numpy().astype(np.int64),
            "offset": ix.offset[0, 0].cpu().numpy().astype(np.int64),
        }
        val, desc, _ = oracle_decode_sample(w, g_np, index_np, r, args.cpu_seconds / 2)
        res["cpu_baseline"] = {"value": val, "unit": UNIT, "cores": blas_threads(),
                               "kind": "oracle", "sample": desc, "host_cpus": os.cpu_count()}
    ctx = {"w": w, "g_np": g_np, "K": K, "V": V, "q": q, "ix": ix, "dec": dec, "dstep": dstep,
           "step_ms": step_ms}
    return res, ctx


def gpu_uuid_str(dev):
    import torch
    u = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    return "GPU-" + str(u) if u else ""


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------
def relaunch_command(argv, n_gpus, port, python=None):
    """The torch.distributed.run command that starts this bench once per GPU
    (one process per GPU, rendezvous on 127.0.0.1) with the same arguments."""
    return [python or sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
            "--nproc-per-node", str(n_gpus), "--master-addr", "127.0.0.1",
            "--master-port", str(port), os.path.abspath(__file__)] + list(argv)


def maybe_relaunch(args, argv, run=subprocess.call):
    """`--gpus N` with N > 1 started as a single process: run the N ranks under
    torch.distributed.run and return its exit status; None when this process
    is already a rank (WORLD_SIZE set) or N == 1."""
    if args.gpus <= 1 or "WORLD_SIZE" in os.environ:
        return None
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return run(relaunch_command(argv, args.gpus, port))


def main():
    args = parse()
    rc = maybe_relaunch(args, sys.argv[1:])
    if rc is not None:
        return rc
    from workloads import WORKLOADS, generate, retrieval_budget
    w = WORKLOADS[args.workload]
    r = retrieval_budget(w, args.budget_frac) if args.budget_frac else w.r
    if args.impl == "reference":
        return run_reference(args, w, r)

    import torch
    import torch.distributed as dist
    import cluster_indexed_sparse_wi_b300 as wl

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pk, pk_kind = peaks()
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    # ---- the headline workload: decode (value), its stages, e2e, oracle
    res, ctx = measure_workload(w, r, dev, args, pk, flush, rank, want_cpu=False)
    K, V, q, ix, dec, g_np = ctx["K"], ctx["V"], ctx["q"], ctx["ix"], ctx["dec"], ctx["g_np"]
    C = w.n_clusters

    # ---- build (rows a1-a4), timed on its own
    build = None
    if not args.no_build_timing:
        bt = []
        for _ in range(3):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            ix.build(K, V)
            e1.record(stream)
            torch.cuda.synchronize()
            bt.append(e0.elapsed_time(e1))
        build_ms = statistics.median(bt)
        tokens = w.B * w.Hkv * w.N
        flops = 2.0 * w.B * w.Hkv * (w.N - w.sink - w.window) * w.k_per_seg * w.d * w.iters
        build = {"ms": build_ms, "tokens_indexed_per_s": tokens / (build_ms * 1e-3),
                 "assign_tflop": flops * 1e-12,
                 "assign_tflops_over_whole_build": flops / (build_ms * 1e-3) * 1e-12,
                 "launches": 2 + 3 * w.iters + 1}
        assert ix.status() == 0

    # ---- the same step as three stage-only launches (reported, not the value)
    names = ["score", "select", "attend"]
    g_stage = [wl.capture_graph(fn, dev) for fn in (
        lambda: dec.score(q), lambda: dec.select(), lambda: dec.attend(q, K, V))]
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for i in range(args.steps):
        flush()
        e = kev[i]
        e[0].record(stream)
        for j, gs in enumerate(g_stage):
            gs.replay()
            e[j + 1].record(stream)
    torch.cuda.synchronize()
    assert dec.status() == 0
    kern_ms = {n: statistics.mean(kev[i][j].elapsed_time(kev[i][j + 1])
                                  for i in range(args.steps)) for j, n in enumerate(names)}
    by = res["bytes"]
    kern_bytes = {"score": by["centroid_keys"] + by["value_sums_sizes"],
                  "select": w.B * w.Hq * C * 4,
                  "attend": by["steady_kv"] + by["retrieved_kv_unique"]}
    stage_gbs = {n: kern_bytes[n] / (kern_ms[n] * 1e-3) / 1e9 for n in names}

    # ---- context only: full-attention decode over the same K/V with torch SDPA
    sdpa = None
    if not args.no_sdpa:
        try:
            import torch.nn.functional as F
            q4 = q[:, :, None, :]
            for _ in range(3):
                F.scaled_dot_product_attention(q4, K, V, enable_gqa=True)
            ts = timed_steps(lambda: F.scaled_dot_product_attention(q4, K, V, enable_gqa=True),
                             flush, max(args.steps, 5), stream)
            sdpa_ms = statistics.median(ts)
            kv_bytes = 2 * K.numel() * K.element_size()
            sdpa = {"ms": sdpa_ms, "gbs": kv_bytes / (sdpa_ms * 1e-3) / 1e9, "bytes": kv_bytes,
                    "time_ratio_to_decode_step": sdpa_ms / res["ms_per_step"],
                    "how": "torch scaled_dot_product_attention (bf16, enable_gqa) of the step's "
                           "queries over all N keys; library kernel, context for the pages' "
                           "decode speed-up against full attention, not part of the value"}
        except Exception as e:  # context number only
            sdpa = {"unavailable": str(e)[:200]}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        index_np = {
            "size": ix.size[0, 0].cpu().numpy().astype(np.int64),
            "centroid_key": ix.centroid_key[0, 0].double().cpu().numpy(),
            "value_sum": ix.value_sum[0, 0].double().cpu().numpy(),
            "perm": ix.perm[0, 0].cpu().numpy().astype(np.int64),
            "offset": ix.offset[0, 0].cpu().numpy().astype(np.int64),
        }
        val, desc, _ = oracle_decode_sample(w, g_np, index_np, r, args.cpu_seconds)
        cpu = {"value": val, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
               "sample": desc, "host_cpus": os.cpu_count()}
    # ---- the decode options on the headline index
    variants = []
    if not args.no_sweep and ws == 1:
        try:
            variants = measure_variants(w, r, dev, args, pk, flush, ctx)
        except Exception as e:  # report, keep the headline
            variants = [{"error": str(e)[:300]}]

    del ctx, K, V, q, ix, dec, g_np
    torch.cuda.empty_cache()

    # ---- the other decode workloads (their own roofline, clocks, e2e)
    sweep = []
    if not args.no_sweep and ws == 1:
        for name, fracs, want_cpu in (("llama3_8b_1m_b1", (None,), True),
                                      ("llama3_8b_128k_b16", (0.01, 0.02, 0.03), False)):
            wx = WORKLOADS[name]
            for k, fr in enumerate(fracs):
                rx = retrieval_budget(wx, fr) if fr else wx.r
                label = name if fr is None else "%s@%g%%" % (name, fr * 100)
                try:
                    rx_res, cx = measure_workload(wx, rx, dev, args, pk, flush, rank,
                                                  want_cpu=want_cpu, label=label)
                    sweep.append(rx_res)
                    del cx
                    torch.cuda.empty_cache()
                except Exception as e:  # report, keep the headline
                    sweep.append({"workload": label, "error": str(e)[:300]})

    ms = res["ms_per_step"]
    e2e_mean = res["e2e"]["ms_per_step"]
    if ws > 1:
        ms, e2e_mean = max_over_ranks([ms, e2e_mean], dist, dev)
    queries = w.B * ws
    value = queries / (ms * 1e-3)
    roofline = dict(res["roofline"])
    roofline["traffic"] = recorded_traffic("decode_kernel", w.name)
    roofline["peak_source"] = (pk_kind + " (MEASURED_PEAKS.json hbm_gbs, burst copy)"
                               if pk_kind == "measured" else "fallback 6.4 TB/s")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(w, r),
        "roofline": roofline,
        "ms_per_step_write_flush": res["ms_per_step_write_flush"],
        "hbm": {"algorithmic_bytes_per_step": roofline["algorithmic_bytes_per_launch"],
                "achieved_gbs": roofline["achieved"], "frac_of_measured": roofline["frac"],
                "frac_of_8tbs": roofline["frac_of_8tbs"], "bytes": res["bytes"],
                "frac_of_measured_write_flush": roofline["algorithmic_bytes_per_launch"] /
                (res["ms_per_step_write_flush"] * 1e-3) / 1e9 / roofline["peak"]},
        "stage_launches": {"ms": kern_ms, "algorithmic_bytes": kern_bytes, "gbs": stage_gbs,
                           "how": "the step as three stage-only launches of decode_kernel "
                                  "(score + estimate; select; attend + merge), each a graph "
                                  "replay timed with CUDA events; not the value"},
        "cpu_baseline": cpu,
        "full_attention_sdpa": sdpa,
        "e2e": {"value": queries / (e2e_mean * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": res["e2e"]["h2d_bytes_per_step"],
                "d2h_bytes_per_step": res["e2e"]["d2h_bytes_per_step"],
                "ms_per_step": e2e_mean,
                "ms_per_step_median": res["e2e"]["ms_per_step_median"],
                "how": "DecodeStep graph: H2D q (pinned), decode_kernel, one D2H copy of out and "
                       "lse (pinned), host waits; wall clock per step (q copied into the pinned "
                       "buffer inside the timed region); value from the mean"},
        "gpu_launches": args.steps,
        "timing": "CUDA events around CUDA-graph replays of the decode call; L2 flushed "
                  "before every step outside the events",
        "clocks": res["clocks"],
        "build": build,
        "full_pass_ms": (build["ms"] + ms) if build else None,
        "sweep": sweep,
        "variants": variants,
        "wall_s_timed_region_1": res["wall_s_timed"],
        "setup_seconds": res["setup_seconds"],
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main() or 0)
