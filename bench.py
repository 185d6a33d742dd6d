"""Benchmark of the paged K/V attention hot path on GB300.

One step = one pass of the hot path over one batch of synthetic input:
``kv_scatter_slots`` of this step's new K/V rows, then ``paged_attention``
(split-KV decode kernel + split reduction).  The default workload is the GQA
decode batch (64 sequences, 32 query / 8 K/V heads, head_dim 128, 32-token
pages, cached lengths U[512, 8192], one new token each); the metric is the
K/V bytes the attention reads per second (paged decode KV GB/s), with
queries/s and the fraction of the measured HBM peak alongside.

Usage: ``python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]``.
Under torchrun every rank runs its own replica of the workload (seed + rank:
the sequences shard across GPUs with no collective on the data path; weak
scaling); rank 0 prints one JSON line.  ``--impl reference`` times the fp64
CPU oracle on a bounded sample of the same workload instead.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode KV GB/s"
# the sources of the timed decode launch; a committed DRAM-traffic figure is
# used only while their hash matches the one recorded beside it
DECODE_SOURCES = ["paged_kv_cache_189_gb300/csrc/decode.cu",
                  "paged_kv_cache_189_gb300/csrc/pkv_common.cuh",
                  "paged_kv_cache_189_gb300/csrc/pkv_api.cpp"]
UNIT = "GB/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gqa_decode", choices=["gqa_decode"])
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-seqs", type=int, default=64)
    return ap.parse_args()


# ----------------------------------------------------------------------------
# distributed plumbing (one process per GPU; no collective on the data path)
# ----------------------------------------------------------------------------
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, value, device):
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, value, device):
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------------------
# workload accounting (algorithmic bytes; no reading of device values)
# ----------------------------------------------------------------------------
def decode_bytes(case):
    """Algorithmic bytes of one decode attention launch and of its K/V alone."""
    kv_lens = case.kv_lens.numpy().astype(np.int64)
    Hq, Hkv, D = case.num_q_heads, case.num_kv_heads, case.head_dim
    rows = case.q.shape[0]
    kv = int(kv_lens.sum()) * Hkv * D * 2 * 2
    pages = int(((kv_lens + 31) // 32).sum())
    other = rows * Hq * D * 2 * 2 + rows * Hq * 4 + pages * 4 + case.batch * 4 * 3
    return kv + other, kv


def scatter_bytes(case):
    T = int((case.slots.numpy() >= 0).sum())
    return T * case.num_kv_heads * case.head_dim * 2 * 2 * 2 + T * 8


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self, t0, t1):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), parts[4:]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        sm = [r[0] for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for n, v in zip(names, r[2][1:]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "window": "nvidia-smi every 50 ms from before warm-up to after the timed steps"}


# ----------------------------------------------------------------------------
# the fp64 oracle as a CPU baseline / reference arm (process pool, spawn)
# ----------------------------------------------------------------------------
_W = {}


def _oracle_init(shm_names, shapes, meta):
    from multiprocessing import shared_memory
    for key, name in shm_names.items():
        shm = shared_memory.SharedMemory(name=name)
        _W[key + "_shm"] = shm
        _W[key] = np.ndarray(shapes[key], dtype=np.uint16, buffer=shm.buf)
    _W.update(meta)


def _oracle_seq(b):
    sys.path.insert(0, ROOT)
    from oracle import oracle as orc
    qi = _W["q_indptr"]
    kb, vb = _W["k"], _W["v"]
    # the step's scatter of this sequence's new rows (into a private copy of
    # the touched rows is not needed: attention reads the slot through the table)
    r0, r1 = int(qi[b]), int(qi[b + 1])
    slots = _W["slots"][r0:r1]
    P = kb.shape[1]
    k_local = {int(s): _W["new_k"][r0 + i] for i, s in enumerate(slots) if s >= 0}
    v_local = {int(s): _W["new_v"][r0 + i] for i, s in enumerate(slots) if s >= 0}
    table = _W["block_table"][b:b + 1]
    # materialise the touched pages with the scattered rows (oracle scatter on a
    # copy of just this sequence's pages keeps the shared pool read-only)
    pages = sorted({int(s) // P for s in k_local})
    kcopy = {p: kb[p].copy() for p in pages}
    vcopy = {p: vb[p].copy() for p in pages}
    for s, row in k_local.items():
        kcopy[s // P][s % P] = row
    for s, row in v_local.items():
        vcopy[s // P][s % P] = row
    # a small pool holding this sequence's pages, table remapped onto it
    used = [int(x) for x in table[0] if x >= 0][: -(-int(_W["kv_lens"][b]) // P)]
    kp = np.stack([kcopy.get(p, kb[p]) for p in used])
    vp = np.stack([vcopy.get(p, vb[p]) for p in used])
    t = np.arange(len(used), dtype=np.int32)[None, :]
    O, L = orc.paged_attention(_W["q"][r0:r1], kp, vp, t, _W["kv_lens"][b:b + 1],
                               np.array([0, r1 - r0]), _W["q_real"][b:b + 1], mask=_W["mask"],
                               causal_block=_W["causal_block"])
    return float(np.nansum(O))


class OraclePool:
    """Oracle over sequences of a case, one single-threaded worker per core."""

    def __init__(self, case, workers):
        import multiprocessing as mp
        from multiprocessing import shared_memory
        from oracle import oracle as orc
        self.shms = []
        names, shapes = {}, {}
        for key, t in (("k", case.k_pool), ("v", case.v_pool)):
            arr = orc.bf16_bits(t)
            shm = shared_memory.SharedMemory(create=True, size=arr.nbytes)
            np.ndarray(arr.shape, dtype=np.uint16, buffer=shm.buf)[...] = arr
            self.shms.append(shm)
            names[key], shapes[key] = shm.name, arr.shape
        meta = dict(q=orc.bf16_bits(case.q), new_k=orc.bf16_bits(case.new_k),
                    new_v=orc.bf16_bits(case.new_v), slots=case.slots.numpy(),
                    block_table=case.block_table.numpy(), kv_lens=case.kv_lens.numpy(),
                    q_indptr=case.q_indptr.numpy(), q_real=case.q_real.numpy(),
                    mask=case.mask, causal_block=case.causal_block)
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"
        ctx = mp.get_context("spawn")
        self.workers = workers
        self.pool = ctx.Pool(workers, initializer=_oracle_init, initargs=(names, shapes, meta))
        self.pool.map(_oracle_seq, [0] * workers)  # warm the workers

    def run(self, seqs):
        t0 = time.perf_counter()
        self.pool.map(_oracle_seq, list(seqs), chunksize=1)
        return time.perf_counter() - t0

    def close(self):
        self.pool.terminate()
        for s in self.shms:
            s.close()
            s.unlink()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def committed_traffic(workload, kernel_sources):
    """DRAM bytes per launch from a committed ncu summary, valid only while the
    kernel's sources are unchanged (hash recorded beside the figure)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f).get(workload)
    if not d:
        return None
    h = hashlib.sha256()
    for src in kernel_sources:
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    if d.get("sources_sha256") != h.hexdigest():
        return None
    return float(d["dram_bytes_per_launch"])


# ----------------------------------------------------------------------------
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from paged_kv_cache_189_gb300 import workloads as wl
    case = wl.gqa_decode(seed=1)
    _, kv_bytes_all = decode_bytes(case)
    workers = min(16, os.cpu_count() or 1)
    pool = OraclePool(case, workers)
    per_step = min(args.cpu_sample_seqs, 16)
    seqs_all = list(range(case.batch))
    kvl = case.kv_lens.numpy().astype(np.int64)
    times, bytes_done = [], []
    for i in range(args.warmup + args.steps):
        seqs = [seqs_all[(i * per_step + j) % case.batch] for j in range(per_step)]
        dt = pool.run(seqs)
        if i >= args.warmup:
            times.append(dt)
            bytes_done.append(int(kvl[seqs].sum()) * case.num_kv_heads * case.head_dim * 4)
    pool.close()
    total_t = sum(times)
    value = sum(bytes_done) / total_t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total_t / max(1, len(times)), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "gqa_decode", "batch": case.batch, "q_heads": 32,
                       "kv_heads": 8, "head_dim": 128, "page": 32,
                       "kv_len": "U[512,8192]+1", "sample_seqs_per_step": per_step},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": workers, "kind": "oracle",
                             "sample": f"{per_step} of the 64 sequences per step (rotating), "
                                       "decode attention incl. the step's scatter"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    from paged_kv_cache_189_gb300 import build as pkv_build
    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    if rank == 0:
        pkv_build.build()
    barrier(dist)
    from paged_kv_cache_189_gb300 import pkv, workloads as wl

    case = wl.gqa_decode(seed=1 + rank)
    attn_bytes, kv_bytes = decode_bytes(case)
    sc_bytes = scatter_bytes(case)
    Hq, Hkv, D = case.num_q_heads, case.num_kv_heads, case.head_dim
    rows = case.q.shape[0]
    max_kv = case.max_kv_len

    k_pool, v_pool = case.k_pool.to(dev), case.v_pool.to(dev)
    q = case.q.to(dev)
    new_k, new_v, slots = case.new_k.to(dev), case.new_v.to(dev), case.slots.to(dev)
    bt, kl, qi, qr = (case.block_table.to(dev), case.kv_lens.to(dev), case.q_indptr.to(dev),
                      case.q_real.to(dev))
    out = torch.empty(rows, Hq, D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(rows, Hq, dtype=torch.float32, device=dev)
    ws_bytes = pkv.paged_attention_workspace_size(case.batch, 1, Hq, Hkv, D, max_kv)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    launches_per_step = 1 + 1 + (1 if ws_bytes else 0)

    def attention():
        pkv.paged_attention(q, k_pool, v_pool, bt, kl, qi, out, q_real=qr, lse=lse,
                            max_q_rows=1, max_kv_len=max_kv, mask="causal", workspace=ws,
                            stream=stream)

    def step():
        pkv.kv_scatter_slots(new_k, new_v, slots, k_pool, v_pool, stream=stream)
        attention()

    clocks = ClockSampler(local)
    clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    wall0 = time.time()
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for i in range(args.steps):
            pkv.kv_scatter_slots(new_k, new_v, slots, k_pool, v_pool, stream=stream)
            ev[i][0].record(stream)
            attention()
            ev[i][1].record(stream)
        t_end.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    wall1 = time.time()
    clk = clocks.stop(wall0, wall1)
    ms_total = t_start.elapsed_time(t_end)
    attn_ms = [a.elapsed_time(b) for a, b in ev]
    ms_total_max = max_over_ranks(dist, ms_total, dev)
    kv_total = sum_over_ranks(dist, kv_bytes * args.steps, dev)
    queries_total = sum_over_ranks(dist, rows * args.steps, dev)
    value = kv_total / (ms_total_max * 1e-3) / 1e9

    # ---- end to end through the public API: pinned host inputs -> device,
    #      scatter + attention, result read back to the host, every step
    h_q = case.q.pin_memory()
    h_k, h_v, h_s = case.new_k.pin_memory(), case.new_v.pin_memory(), case.slots.pin_memory()
    h_kl, h_bt = case.kv_lens.pin_memory(), case.block_table.pin_memory()
    h_out = torch.empty(rows, Hq, D, dtype=torch.bfloat16).pin_memory()
    h_lse = torch.empty(rows, Hq, dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_k, h_v, h_s, h_kl, h_bt))
    d2h = h_out.numel() * 2 + h_lse.numel() * 4

    def e2e_step():
        with torch.cuda.stream(stream):
            q.copy_(h_q, non_blocking=True)
            new_k.copy_(h_k, non_blocking=True)
            new_v.copy_(h_v, non_blocking=True)
            slots.copy_(h_s, non_blocking=True)
            kl.copy_(h_kl, non_blocking=True)
            bt.copy_(h_bt, non_blocking=True)
            step()
            h_out.copy_(out, non_blocking=True)
            h_lse.copy_(lse, non_blocking=True)
        stream.synchronize()

    e2e_value = None
    if args.e2e_steps > 0:
        for _ in range(3):
            e2e_step()
        barrier(dist)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(dist, e0.elapsed_time(e1), dev)
        e2e_value = sum_over_ranks(dist, kv_bytes * args.e2e_steps, dev) / (e2e_ms * 1e-3) / 1e9

    if rank == 0:
        peak, peak_kind = measured_peaks()
        attn_avg_ms = statistics.mean(attn_ms)
        achieved = attn_bytes / (attn_avg_ms * 1e-3) / 1e9
        traffic = committed_traffic("gqa_decode", DECODE_SOURCES)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_total_max / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": "gqa_decode", "batch": case.batch, "q_heads": Hq,
                       "kv_heads": Hkv, "head_dim": D, "page": 32, "kv_len": "U[512,8192]+1",
                       "kv_bytes_per_step": kv_bytes, "queries_per_step": rows,
                       "l2": "inputs larger than L2 (1.14 GB of K/V read per step)",
                       "parallelism": f"replicas x{world} (sequences sharded by rank)"},
            "queries_per_s": queries_total / (ms_total_max * 1e-3),
            "hbm_frac": value / peak,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "kernel": "paged_attention: persistent split-KV decode kernel with the "
                                   "split merge fused in (plus a 2 KB counter memset); CUDA "
                                   "events around the call each timed step",
                         "bytes_per_launch": attn_bytes, "avg_launch_ms": attn_avg_ms,
                         "peak_source": f"{peak_kind} hbm_gbs"},
            "clocks": clk,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": args.e2e_steps},
            "gpu_launches": launches_per_step * args.steps,
            "scatter_bytes_per_step": sc_bytes,
        }
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(case, args)
        print(json.dumps(line), flush=True)
    barrier(dist)
    return 0


def cpu_baseline(case, args):
    workers = min(16, os.cpu_count() or 1)
    pool = OraclePool(case, workers)
    seqs = list(range(min(args.cpu_sample_seqs, case.batch)))
    dt = pool.run(seqs)
    pool.close()
    kvl = case.kv_lens.numpy().astype(np.int64)
    b = int(kvl[seqs].sum()) * case.num_kv_heads * case.head_dim * 4
    return {"value": b / dt / 1e9, "unit": UNIT, "cores": workers, "kind": "oracle",
            "sample": f"{len(seqs)} of {case.batch} sequences of the same step "
                      f"(scatter + decode attention, fp64), {dt:.2f} s"}


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
