"""Benchmark of the paged K/V attention hot path on GB300.

One step = one pass of the hot path over one batch of synthetic input:
``kv_scatter_slots`` of this step's new K/V rows, then ``paged_attention``
(and, per workload, the merge or the rotation of the rolling buffer).  The
headline workload is the GQA decode batch (64 sequences, 32 query / 8 K/V
heads, head_dim 128, 32-token pages, cached lengths U[512, 8192], one new
token each); the metric is the K/V bytes the attention reads per second
(paged decode KV GB/s), with queries/s and the fraction of the measured HBM
peak alongside.  The same JSON line carries, under ``workloads``, every other
workload measured the same way (chunked causal prefill and the block-causal
video step in prefill TFLOP/s; the shared-prefix step, its one-launch form and
the plain-decode ablation, multi-token decode and tiny decode in KV GB/s; the
exact-window denoising forward in prefill TFLOP/s), each with its roofline,
clocks, end-to-end figure and the fp64 oracle's time on the host cores.

Usage: ``python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
[--workload NAME] [--only]``.  ``--only`` measures just ``--workload``.
Under torchrun every rank runs its own independent replica of each workload
(seed + rank: weak scaling with no collective on the data path); rank 0 prints
one JSON line.  ``--impl reference`` times the fp64 CPU oracle on a bounded
sample of the same workload instead.
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
ATTN_TC_SOURCES = ["paged_kv_cache_189_gb300/csrc/attn_tc.cu",
                   "paged_kv_cache_189_gb300/csrc/pkv_common.cuh",
                   "paged_kv_cache_189_gb300/csrc/pkv_api.cpp"]
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
    ap.add_argument("--workload", default="gqa_decode",
                    choices=["gqa_decode", "chunked_prefill", "block_causal_video",
                             "shared_prefix", "shared_prefix_fused", "shared_prefix_verify",
                             "shared_prefix_plain_decode",
                             "tiny_decode", "multi_token_decode", "exact_window_video",
                             "exact_window_denoise"])
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", action="store_true",
                    help="measure only --workload (no 'workloads' object)")
    return ap.parse_args()


# the workloads measured besides the headline one, in the order they run
EXTRA_WORKLOADS = ("tiny_decode", "chunked_prefill", "shared_prefix", "shared_prefix_fused",
                   "shared_prefix_plain_decode", "block_causal_video", "multi_token_decode",
                   "exact_window_denoise", "exact_window_video")


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


def _local_pool(table_row, kv_len, scatter):
    """The pages of one row (logical order) as a small pool, with this step's
    scattered rows ``scatter`` ({slot: (k row, v row)}) applied to copies of
    the touched pages; the shared pools stay read-only."""
    kb, vb = _W["k"], _W["v"]
    P = kb.shape[1]
    used = [int(x) for x in table_row[: -(-int(kv_len) // P)]]
    kp = np.stack([kb[p] for p in used])
    vp = np.stack([vb[p] for p in used])
    where = {p: i for i, p in enumerate(used)}
    for s_, (kr, vr) in scatter.items():
        i = where.get(s_ // P)
        if i is not None:
            kp[i, s_ % P] = kr
            vp[i, s_ % P] = vr
    return kp, vp, np.arange(len(used), dtype=np.int32)[None, :]


def _scatter_rows(r0, r1):
    slots = _W["slots"][r0:r1]
    return {int(s_): (_W["new_k"][r0 + i], _W["new_v"][r0 + i]) for i, s_ in enumerate(slots) if s_ >= 0}


def _oracle_task(task):
    """One unit of the oracle's work on the step; returns a checksum so the
    work is not optimised away.

    ("seq", b, rows): sequence b's rows (absolute row indices; None = all),
      after the step's scatter of its new rows;
    ("group", g): a shared-prefix group: the prefix call over its samples'
      rows (mask none), each sample's tail call (causal), and the merge;
    ("window", rows): exact-window attention of the staged rows ``rows``
      over the long sequence (history from the pool, staged tokens new)."""
    sys.path.insert(0, ROOT)
    from oracle import oracle as orc
    kind = task[0]
    if kind == "seq":
        _, b, rows = task
        qi = _W["q_indptr"]
        r0, r1 = int(qi[b]), int(qi[b + 1])
        kp, vp, t = _local_pool(_W["block_table"][b], _W["kv_lens"][b], _scatter_rows(r0, r1))
        local = None if rows is None else [r - r0 for r in rows]
        O, _ = orc.paged_attention(_W["q"][r0:r1], kp, vp, t, _W["kv_lens"][b:b + 1],
                                   np.array([0, r1 - r0]), _W["q_real"][b:b + 1], mask=_W["mask"],
                                   causal_block=_W["causal_block"], rows=local)
        return float(np.nansum(O))
    if kind == "group":
        g = task[1]
        n, ql = _W["samples"], _W["q_len"]
        r0, r1 = g * n * ql, (g + 1) * n * ql
        kp, vp, t = _local_pool(_W["prefix_table"][g], _W["prefix_lens"][g], {})
        O_p, L_p = orc.paged_attention(_W["q"][r0:r1], kp, vp, t, _W["prefix_lens"][g:g + 1],
                                       np.array([0, r1 - r0]), None, mask="none")
        total = 0.0
        for r in range(g * n, (g + 1) * n):
            a0, a1 = r * ql, (r + 1) * ql
            kp, vp, t = _local_pool(_W["tail_table"][r], _W["tail_lens"][r], _scatter_rows(a0, a1))
            O_t, L_t = orc.paged_attention(_W["q"][a0:a1], kp, vp, t, _W["tail_lens"][r:r + 1],
                                           np.array([0, ql]), None, mask="causal")
            O, _ = orc.merge_attn_states(O_p[a0 - r0:a1 - r0], L_p[a0 - r0:a1 - r0], O_t, L_t)
            total += float(np.nansum(O))
        return total
    if kind == "window":
        rows = task[1]
        kb, vb = _W["k"], _W["v"]
        P = kb.shape[1]
        base = _W["pin"] + _W["committed"]
        pos = np.arange(base)
        pages = _W["table"][pos // P]
        k_seq = np.concatenate([kb[pages, pos % P], _W["new_k"]])
        v_seq = np.concatenate([vb[pages, pos % P], _W["new_v"]])
        O, _ = orc.exact_window_attention(_W["q"], k_seq, v_seq, _W["pin"], _W["committed"],
                                          _W["window"], _W["staged"], _W["block"], rows=rows)
        return float(np.nansum(O))
    raise ValueError(kind)


class OraclePool:
    """The oracle over tasks of one workload's step, one single-threaded
    worker process per core (spawned, so it is safe after CUDA is up)."""

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
                    new_v=orc.bf16_bits(case.new_v))
        if hasattr(case, "block_table"):
            meta.update(slots=case.slots.numpy(), block_table=case.block_table.numpy(),
                        kv_lens=case.kv_lens.numpy(), q_indptr=case.q_indptr.numpy(),
                        q_real=case.q_real.numpy(), mask=case.mask, causal_block=case.causal_block)
            e = case.extra
            if "prefix_table" in e:
                meta.update(samples=e["samples"], q_len=e["q_len"],
                            prefix_table=e["prefix_table"].numpy(), prefix_lens=e["prefix_lens"].numpy(),
                            tail_table=e["tail_table"].numpy(), tail_lens=e["tail_lens"].numpy())
        else:   # an exact-window forward
            meta.update(table=case.table.numpy(), pin=case.pin, committed=case.committed,
                        window=case.window, staged=case.staged, block=case.block)
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"
        ctx = mp.get_context("spawn")
        self.workers = workers
        self.pool = ctx.Pool(workers, initializer=_oracle_init, initargs=(names, shapes, meta))
        self.pool.map(abs, range(workers))  # wait for every worker to start

    def run(self, tasks):
        t0 = time.perf_counter()
        self.pool.map(_oracle_task, list(tasks), chunksize=1)
        return time.perf_counter() - t0

    def close(self):
        self.pool.terminate()
        self.pool.join()
        for s_ in self.shms:
            s_.close()
            s_.unlink()


def host_cores():
    return os.cpu_count() or 1


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def measured_tensor_peak():
    """Dense bf16 tensor peak: the burst figure.  The attention launches are
    timed one by one over runs of well under a second and hold the maximum SM
    clock (no power cap in the sampled clocks), while the sustained cuBLAS
    figure was taken at a power-capped clock."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


# End to end: steps that move at least this many bytes between host and device
# overlap their copies with the neighbouring steps (copy streams); smaller ones
# keep them on the compute stream.
PIPELINE_MIN_BYTES = 256 * 1024


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
# the oracle's bounded sample of each workload's step
# ----------------------------------------------------------------------------
def _oracle_warm(_):
    sys.path.insert(0, ROOT)
    from oracle import oracle  # noqa: F401  (import cost kept out of the timed run)
    return 0


def _chunks(seq, n):
    n = max(1, min(n, len(seq)))
    return [seq[i::n] for i in range(n)]


def oracle_sample(name, case, workers):
    """Tasks of the oracle's sample of one step of workload ``name``, the work
    they stand for in the workload metric's base unit (bytes or flops), and a
    one-line description."""
    if name == "exact_window_denoise" or name == "exact_window_video":
        Hq, D = case.num_q_heads, case.head_dim
        rows = list(range(0, case.staged, 8))
        from oracle import oracle as orc
        pairs = sum(len(orc.exact_window_keys(case.pin, case.committed, case.window, case.staged,
                                              case.block, r // case.block)) for r in rows)
        return ([("window", c) for c in _chunks(rows, workers)], 4.0 * D * Hq * pairs,
                f"{len(rows)} of {case.staged} query rows (every 8th), exact-window attention "
                "over the long sequence, fp64")
    Hq, Hkv, D = case.num_q_heads, case.num_kv_heads, case.head_dim
    tok = Hkv * D * 2 * 2
    kvl = case.kv_lens.numpy().astype(np.int64)
    qi = case.q_indptr.numpy()
    if name in ("gqa_decode", "multi_token_decode", "shared_prefix_plain_decode"):
        tasks = [("seq", b, None) for b in range(case.batch)]
        return (tasks, float(kvl.sum() * tok),
                f"all {case.batch} sequences of the step (scatter + attention over each "
                "sequence's whole row, fp64)")
    if name == "tiny_decode":
        reps = 500
        tasks = [("seq", b, None) for b in range(case.batch)] * reps
        return (tasks, float(kvl.sum() * tok * reps),
                f"the whole step (both sequences: scatter + decode attention, fp64) {reps} times")
    if name in ("shared_prefix", "shared_prefix_fused"):
        e = case.extra
        prefix = int(e["prefix_lens"][0])
        work = e["groups"] * prefix * tok + int(e["tail_lens"].sum()) * tok
        return ([("group", g) for g in range(e["groups"])], float(work),
                f"all {e['groups']} groups of the step: prefix call over each group's "
                f"{e['samples']} rows, every sample's tail call and the merge, fp64")
    if name in ("chunked_prefill", "block_causal_video"):
        from oracle import oracle as orc
        qr = case.q_real.numpy()
        stride = 8 if name == "chunked_prefill" else 4
        tasks, pairs, nrows = [], 0, 0
        for b in range(case.batch):
            rows = list(range(int(qi[b]), int(qi[b]) + int(qr[b]), stride))
            nrows += len(rows)
            pairs += sum(orc.visible_keys(r - int(qi[b]), int(qr[b]), int(kvl[b]), case.mask,
                                          case.causal_block) for r in rows)
            per_seq = max(1, workers // case.batch)
            tasks += [("seq", b, c) for c in _chunks(rows, per_seq)]
        return (tasks, 4.0 * D * Hq * pairs,
                f"{nrows} of {int(qr.sum())} real query rows (every {stride}th row of each "
                "sequence, after the step's scatter), fp64; the rotation is not included"
                if name == "block_causal_video" else
                f"{nrows} of {int(qr.sum())} real query rows (every {stride}th row of each "
                "sequence, after the step's scatter), fp64")
    return None


def time_oracle(name, case, workers, scale, unit, tasks=None):
    """Run the oracle's sample of one step on ``workers`` processes; returns
    (value in the metric's unit, seconds, description)."""
    sample = oracle_sample(name, case, workers)
    if sample is None:
        return None
    tk, work, desc = sample
    if tasks is not None:
        tk, work = tasks
    pool = OraclePool(case, workers)
    try:
        pool.pool.map(_oracle_warm, range(workers))
        dt = pool.run(tk)
    finally:
        pool.close()
    return work / dt / scale, dt, desc


def cpu_baseline_for(name, case, unit, scale):
    """The fp64 oracle, as it stands, on a bounded sample of the same step, on
    every host core (one single-threaded worker each); for the two decode
    workloads also on one core."""
    cores = host_cores()
    r = time_oracle(name, case, cores, scale, unit)
    if r is None:
        return None
    value, dt, desc = r
    out = {"value": value, "unit": unit, "cores": cores, "host_cores": cores, "kind": "oracle",
           "sample": f"{desc}; {dt:.2f} s on {cores} worker processes"}
    if name in ("gqa_decode", "tiny_decode"):
        Hkv, D = case.num_kv_heads, case.head_dim
        kvl = case.kv_lens.numpy().astype(np.int64)
        if name == "gqa_decode":
            seqs = list(range(16))
            tasks = ([("seq", b, None) for b in seqs], float(kvl[seqs].sum() * Hkv * D * 4))
            what = "16 of the 64 sequences of the step"
        else:
            tasks = ([("seq", b, None) for b in range(case.batch)] * 200, float(kvl.sum() * Hkv * D * 4 * 200))
            what = "the whole step 200 times"
        v1, dt1, _ = time_oracle(name, case, 1, scale, unit, tasks=tasks)
        out["one_thread"] = {"value": v1, "unit": unit, "cores": 1,
                             "sample": f"{what} (scatter + decode attention, fp64); {dt1:.2f} s on "
                                       "one worker process"}
    return out


# ----------------------------------------------------------------------------
def run_reference(args):
    """The reference arm: the fp64 oracle, as it stands, on the host cores, on
    a bounded sample of each step of the workload (rank 0 only)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from paged_kv_cache_189_gb300 import workloads as wl
    name = args.workload
    case = make_case(name, 0)
    meta = WORKLOAD_META[name]
    cores = host_cores()
    sample = oracle_sample(name, case, cores)
    if sample is None:
        print(json.dumps({"impl": "reference", "unavailable": f"no oracle sample for {name}"}))
        return 0
    tasks, work, desc = sample
    pool = OraclePool(case, cores)
    pool.pool.map(_oracle_warm, range(cores))
    times = []
    for i in range(args.warmup + args.steps):
        dt = pool.run(tasks)
        if i >= args.warmup:
            times.append(dt)
    pool.close()
    total_t = sum(times)
    value = work * len(times) / total_t / meta["scale"]
    line = {"impl": "reference", "metric": meta["metric"], "value": value, "unit": meta["unit"],
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total_t / max(1, len(times)), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": name, **meta["config"], "oracle_sample": desc},
            "cpu_baseline": {"value": value, "unit": meta["unit"], "cores": cores, "host_cores": cores,
                             "kind": "oracle", "sample": f"{desc}, each step"},
            "e2e": {"value": value, "unit": meta["unit"], "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# metric, unit and fixed configuration keys of each workload (as the bench
# line of our arm states them)
WORKLOAD_META = {
    "gqa_decode": dict(metric=METRIC, unit="GB/s", scale=1e9,
                       config=dict(batch=64, q_heads=32, kv_heads=8, head_dim=128, page=32,
                                   kv_len="U[512,8192]+1")),
    "tiny_decode": dict(metric=METRIC, unit="GB/s", scale=1e9,
                        config=dict(batch=2, q_heads=4, kv_heads=2, head_dim=64, page=32,
                                    kv_len="{37,100}")),
    "multi_token_decode": dict(metric="multi-token decode KV GB/s", unit="GB/s", scale=1e9,
                               config=dict(batch=64, q_heads=32, kv_heads=8, head_dim=128, page=32,
                                           q_len=4, kv_len="U[512,8192]+4")),
    "chunked_prefill": dict(metric="prefill TFLOP/s", unit="TFLOP/s", scale=1e12,
                            config=dict(batch=8, q_heads=32, kv_heads=8, head_dim=128, page=32,
                                        ctx="U[2048,16384]", chunk=512, mask="causal")),
    "block_causal_video": dict(metric="prefill TFLOP/s", unit="TFLOP/s", scale=1e12,
                               config=dict(batch=1, q_heads=40, kv_heads=40, head_dim=128, page=32,
                                           kv_len=7800, q_rows=1568, q_real=1560, causal_block=1560,
                                           mask="block_causal")),
    "shared_prefix": dict(metric="shared-prefix KV GB/s", unit="GB/s", scale=1e9,
                          config=dict(groups=16, samples=8, prefix=4096, tail="U[1,1024]", q_heads=32,
                                      kv_heads=8, head_dim=128, page=32)),
    "shared_prefix_fused": dict(metric="shared-prefix KV GB/s", unit="GB/s", scale=1e9,
                                config=dict(groups=16, samples=8, prefix=4096, tail="U[1,1024]",
                                            q_heads=32, kv_heads=8, head_dim=128, page=32)),
    "shared_prefix_plain_decode": dict(metric="shared-prefix KV GB/s", unit="GB/s", scale=1e9,
                                       config=dict(groups=16, samples=8, prefix=4096, tail="U[1,1024]",
                                                   q_heads=32, kv_heads=8, head_dim=128, page=32)),
    "exact_window_denoise": dict(metric="prefill TFLOP/s", unit="TFLOP/s", scale=1e12,
                                 config=dict(q_heads=32, kv_heads=8, head_dim=128, page=32,
                                             staged_tokens=1576, causal_block=1576)),
    "exact_window_video": dict(metric="prefill TFLOP/s", unit="TFLOP/s", scale=1e12,
                               config=dict(q_heads=32, kv_heads=8, head_dim=128, page=32,
                                           staged_tokens=1576, causal_block=394)),
}
WORKLOAD_SEED = {"gqa_decode": 1, "chunked_prefill": 2, "shared_prefix": 3, "block_causal_video": 4,
                 "shared_prefix_fused": 3, "shared_prefix_verify": 3, "shared_prefix_plain_decode": 3,
                 "tiny_decode": 0, "multi_token_decode": 5, "exact_window_video": 6,
                 "exact_window_denoise": 6}


def make_case(name, rank):
    """The seeded synthetic input of one workload for rank ``rank``."""
    from paged_kv_cache_189_gb300 import workloads as wl
    seed = WORKLOAD_SEED[name] + rank
    if name in ("exact_window_video", "exact_window_denoise"):
        return wl.exact_window_video(seed=seed, blocks_per_chunk=4 if name == "exact_window_video" else 1)
    return {"gqa_decode": wl.gqa_decode, "chunked_prefill": wl.chunked_prefill,
            "block_causal_video": wl.block_causal_video, "shared_prefix": wl.shared_prefix,
            "shared_prefix_fused": wl.shared_prefix, "shared_prefix_plain_decode": wl.shared_prefix,
            "shared_prefix_verify": lambda seed: wl.shared_prefix(seed, q_len=4),
            "tiny_decode": wl.tiny_decode, "multi_token_decode": wl.multi_token_decode}[name](seed=seed)


def visible_pairs(case):
    """(query row, visible key) pairs of a case's real rows, per query head."""
    kvl = case.kv_lens.numpy().astype(np.int64)
    qr = case.q_real.numpy().astype(np.int64)
    total = 0
    for b in range(case.batch):
        i = np.arange(qr[b])
        first_new = kvl[b] - qr[b]
        if case.mask == "none":
            vis = np.full(qr[b], kvl[b])
        elif case.mask == "causal":
            vis = first_new + i + 1
        else:
            cb = case.causal_block
            vis = first_new + np.minimum(qr[b], (i // cb + 1) * cb)
        total += int(vis.sum())
    return total


class StepPlan:
    """One workload step on the device: pre -> dominant -> post launches."""

    def __init__(self, **kw):
        self.__dict__.update(kw)


def build_exact_window_plan(name, rank, dev, stream):
    """A forward over exact windows: the commit (device layout + the committed
    private copies) runs once at set-up and is timed as an auxiliary call; a
    step is the forward of one layer: the staged K/V to their two slots, the
    earlier blocks' tokens to the later blocks' private pages, and one unmasked
    attention over all causal blocks."""
    import torch
    from paged_kv_cache_189_gb300 import pkv, workloads as wl

    case = make_case(name, rank)
    Hq, Hkv, D = case.num_q_heads, case.num_kv_heads, case.head_dim
    t = dict(k_pool=case.k_pool.to(dev), v_pool=case.v_pool.to(dev), q=case.q.to(dev),
             new_k=case.new_k.to(dev), new_v=case.new_v.to(dev), table=case.table.to(dev),
             priv=case.private_pages.to(dev),
             committed=torch.tensor([case.committed], dtype=torch.int64, device=dev))
    bufs = pkv.causal_layout_buffers(case.staged, case.block, case.row_stride, dev)

    def commit():
        pkv.causal_layout(t["table"], t["committed"], case.pin, case.window, case.staged, case.block,
                          t["priv"], bufs, stream=stream)
        pkv.copy_kv_slots(t["k_pool"], t["v_pool"], bufs["committed_src"], bufs["committed_dst"],
                          stream=stream)

    with torch.cuda.stream(stream):
        commit()
    torch.cuda.synchronize()

    def scatters():
        pkv.kv_scatter_slots(t["new_k"], t["new_v"], bufs["staged_slots"], t["k_pool"], t["v_pool"],
                             slots2=bufs["staged_slots2"], stream=stream)
        pkv.kv_scatter_slots(t["new_k"], t["new_v"], bufs["current_dst"], t["k_pool"], t["v_pool"],
                             src_idx=bufs["current_src_idx"], stream=stream)

    # key counts per block, closed form of the window (also what the device wrote)
    base = case.pin + case.committed
    kv_lens, ns = [], []
    for k in range(case.num_blocks):
        first = k * case.block
        n = min(case.block, case.staged - first)
        kv_lens.append(case.pin + min(case.window, base + first - case.pin) + n)
        ns.append(n)
    assert kv_lens == bufs["kv_lens"].tolist()
    pairs = sum(n * kl for n, kl in zip(ns, kv_lens))
    flops = 4.0 * D * Hq * pairs
    out = torch.empty(case.staged, Hq, D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(case.staged, Hq, dtype=torch.float32, device=dev)
    ws_b = pkv.paged_attention_workspace_size(case.num_blocks, case.block, Hq, Hkv, D, case.max_kv_len)
    ws = torch.empty(max(ws_b, 256), dtype=torch.uint8, device=dev)

    def attention():
        pkv.paged_attention(t["q"], t["k_pool"], t["v_pool"], bufs["rows"], bufs["kv_lens"],
                            bufs["q_indptr"], out, lse=lse, max_q_rows=case.block,
                            max_kv_len=case.max_kv_len, mask="none", workspace=ws, stream=stream)

    tok = Hkv * D * 2 * 2
    n_cur = int((bufs["current_dst"] >= 0).sum())
    n_com = int((bufs["committed_dst"] >= 0).sum())
    aux = {"scatter": (scatters, case.staged * tok * 3 + n_cur * tok * 2, "GB/s"),
           "commit": (commit, n_com * tok * 2, "GB/s")}
    peak_tc, tc_kind = measured_tensor_peak()
    cfg = {"workload": name, "pin_tokens": case.pin, "history_tokens": case.committed,
           "window_tokens": case.window, "staged_tokens": case.staged, "causal_block": case.block,
           "blocks": case.num_blocks, "kv_len_per_block": kv_lens, "q_heads": Hq, "kv_heads": Hkv,
           "head_dim": D, "page": 32, "mask": "none (exact-window rows)",
           "visible_pairs_per_head": pairs, "flops_per_step": flops,
           "l2": "K/V read per step larger than L2", "committed_private_copies": n_com,
           "current_private_copies": n_cur}
    return StepPlan(case=case, cfg=cfg, metric="prefill TFLOP/s", unit="TFLOP/s", work=flops, scale=1e12,
                    queries=case.staged, pre=[scatters], dominant=attention, post=[], aux=aux,
                    dom_label="paged_attention over the exact-window rows: tcgen05 tile kernel",
                    dom_work=flops / 1e12, bound="tensor", peak=peak_tc, peak_unit="TFLOP/s",
                    peak_src=f"{tc_kind} bf16_tflops (burst)",
                    h2d=([case.q, case.new_k, case.new_v], [t["q"], t["new_k"], t["new_v"]]),
                    # two scatters, the tile kernel, the split reduce (both
                    # exact-window workloads split their keys)
                    d2h=[out, lse], launches=4, traffic_sources=ATTN_TC_SOURCES)


def build_plan(name, rank, dev, stream):
    import torch
    from paged_kv_cache_189_gb300 import pkv, workloads as wl

    if name in ("exact_window_video", "exact_window_denoise"):
        return build_exact_window_plan(name, rank, dev, stream)
    case = make_case(name, rank)
    Hq, Hkv, D = case.num_q_heads, case.num_kv_heads, case.head_dim
    rows = case.q.shape[0]
    t = dict(k_pool=case.k_pool.to(dev), v_pool=case.v_pool.to(dev), q=case.q.to(dev),
             new_k=case.new_k.to(dev), new_v=case.new_v.to(dev), slots=case.slots.to(dev),
             bt=case.block_table.to(dev), kl=case.kv_lens.to(dev), qi=case.q_indptr.to(dev),
             qr=case.q_real.to(dev))
    out = torch.empty(rows, Hq, D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(rows, Hq, dtype=torch.float32, device=dev)
    kv_tok_bytes = Hkv * D * 2 * 2
    scatter = lambda: pkv.kv_scatter_slots(t["new_k"], t["new_v"], t["slots"], t["k_pool"],
                                           t["v_pool"], stream=stream)
    real_new = int((case.slots.numpy() >= 0).sum())
    aux = {"scatter": (scatter, real_new * kv_tok_bytes * 2 + real_new * 8, "GB/s")}
    cfg = {"workload": name, "batch": case.batch, "q_heads": Hq, "kv_heads": Hkv,
           "head_dim": D, "page": 32}
    peak_hbm, hbm_kind = measured_peaks()
    peak_tc, tc_kind = measured_tensor_peak()

    def attention_call(q, bt, kl, qi, qr, o, l, max_q_rows, max_kv_len, mask, cb=0, on=None):
        ws_b = pkv.paged_attention_workspace_size(int(kl.numel()), max_q_rows, Hq, Hkv, D, max_kv_len)
        ws = torch.empty(max(ws_b, 256), dtype=torch.uint8, device=dev)
        st = stream if on is None else on
        return lambda: pkv.paged_attention(q, t["k_pool"], t["v_pool"], bt, kl, qi, o, q_real=qr,
                                           lse=l, max_q_rows=max_q_rows, max_kv_len=max_kv_len,
                                           mask=mask, causal_block=cb, workspace=ws, stream=st)

    h2d_src = [case.q, case.new_k, case.new_v, case.slots, case.kv_lens, case.block_table]
    h2d_dst = [t["q"], t["new_k"], t["new_v"], t["slots"], t["kl"], t["bt"]]
    d2h_src = [out, lse]
    if name in ("gqa_decode", "tiny_decode"):
        attn_bytes, kv_bytes = decode_bytes(case)
        dom = attention_call(t["q"], t["bt"], t["kl"], t["qi"], t["qr"], out, lse, 1,
                             case.max_kv_len, "causal")
        cfg.update(kv_len="U[512,8192]+1" if name == "gqa_decode" else "{37,100}",
                   kv_bytes_per_step=kv_bytes, queries_per_step=rows,
                   l2="inputs larger than L2 (1.14 GB of K/V read per step)")
        return StepPlan(case=case, cfg=cfg, metric=METRIC, unit=UNIT, work=kv_bytes, scale=1e9,
                        queries=rows, pre=[scatter], dominant=dom, post=[], aux=aux,
                        dom_label="paged_attention: persistent split-KV decode kernel with the split "
                                  "merge fused in, behind a one-CTA launch that orders its work units",
                        dom_work=attn_bytes, bound="hbm", peak=peak_hbm, peak_unit="GB/s",
                        peak_src=f"{hbm_kind} hbm_gbs", h2d=(h2d_src, h2d_dst), d2h=d2h_src,
                        # scatter, the unit-order planner (only when the units outnumber
                        # the persistent CTAs; the tiny batch resets its counters with a
                        # memset node instead) and the decode kernel
                        launches=3 if name == "gqa_decode" else 2, traffic_sources=DECODE_SOURCES)
    if name == "multi_token_decode":
        attn_bytes, kv_bytes = decode_bytes(case)
        dom = attention_call(t["q"], t["bt"], t["kl"], t["qi"], t["qr"], out, lse, case.max_q_rows,
                             case.max_kv_len, "causal")
        cfg.update(kv_len="U[512,8192]+4", q_len=case.max_q_rows, kv_bytes_per_step=kv_bytes,
                   queries_per_step=rows, l2="inputs larger than L2")
        return StepPlan(case=case, cfg=cfg, metric="multi-token decode KV GB/s", unit=UNIT,
                        work=kv_bytes, scale=1e9, queries=rows, pre=[scatter], dominant=dom, post=[],
                        aux=aux, dom_label="paged_attention: tensor-core tile kernel, 4 tokens x 4 "
                                           "grouped heads = 16 of 128 tile rows",
                        dom_work=attn_bytes, bound="hbm", peak=peak_hbm, peak_unit="GB/s",
                        peak_src=f"{hbm_kind} hbm_gbs", h2d=(h2d_src, h2d_dst), d2h=d2h_src,
                        launches=2, traffic_sources=ATTN_TC_SOURCES)
    if name in ("chunked_prefill", "block_causal_video"):
        pairs = visible_pairs(case)
        flops = 4.0 * D * Hq * pairs
        dom = attention_call(t["q"], t["bt"], t["kl"], t["qi"], t["qr"], out, lse,
                             case.max_q_rows, case.max_kv_len, case.mask, case.causal_block)
        post = []
        launches = 2
        if name == "block_causal_video":
            e = case.extra
            tok = Hkv * D * 2
            n, sh, first = e["rotate_tokens"], e["rotate_shift_tokens"], e["rotate_first_token"]
            regions = [pool.view(torch.uint8).view(-1)[first * tok:(first + n) * tok]
                       for pool in (t["k_pool"], t["v_pool"])]

            def rotate():
                for reg in regions:
                    pkv.rotate_rows(reg, sh * tok // 16, rows=1, cols=n * tok // 16,
                                    row_stride=n * tok // 16, elem_size=16, stream=stream)
            post = [rotate]
            aux["rotate"] = (rotate, 2 * 2 * n * tok, "GB/s")
            launches = 4
            cfg.update(kv_len=int(case.kv_lens[0]), q_rows=rows, q_real=int(case.q_real[0]),
                       causal_block=case.causal_block)
        else:
            cfg.update(ctx="U[2048,16384]", chunk=512)
        cfg.update(mask=case.mask, visible_pairs_per_head=pairs, flops_per_step=flops,
                   l2="K/V read per step larger than L2")
        return StepPlan(case=case, cfg=cfg, metric="prefill TFLOP/s", unit="TFLOP/s", work=flops,
                        scale=1e12, queries=int(case.q_real.sum()), pre=[scatter], dominant=dom,
                        post=post, aux=aux,
                        dom_label="paged_attention: tcgen05 tile kernel (tensor memory, TMA)",
                        dom_work=flops / 1e12, bound="tensor", peak=peak_tc, peak_unit="TFLOP/s",
                        peak_src=f"{tc_kind} bf16_tflops (burst)", h2d=(h2d_src, h2d_dst),
                        d2h=d2h_src, launches=launches, traffic_sources=ATTN_TC_SOURCES)
    if name == "shared_prefix":
        e = case.extra
        Gn, n_s = e["groups"], e["samples"]
        pt = dict(pt=e["prefix_table"].to(dev), pl=e["prefix_lens"].to(dev),
                  pqi=e["prefix_q_indptr"].to(dev), pqr=e["prefix_q_real"].to(dev),
                  tt=e["tail_table"].to(dev), tl=e["tail_lens"].to(dev))
        o_p = torch.empty(rows, Hq, D, device=dev)
        l_p = torch.empty(rows, Hq, device=dev)
        o_t = torch.empty(rows, Hq, D, device=dev)
        l_t = torch.empty(rows, Hq, device=dev)
        prefix = int(e["prefix_lens"][0])
        dom = attention_call(t["q"], pt["pt"], pt["pl"], pt["pqi"], pt["pqr"], o_p, l_p, n_s,
                             prefix, "none")
        mt = int(e["tail_lens"].max())
        tail = attention_call(t["q"], pt["tt"], pt["tl"], t["qi"], t["qr"], o_t, l_t, 1, mt,
                              "causal")
        merge = lambda: pkv.merge_attn_states(o_p, l_p, o_t, l_t, out, lse, stream=stream)
        # the prefix and tail calls are independent: the tail call runs on a
        # second stream, forked after the scatter and joined before the merge
        side = torch.cuda.Stream(device=dev)
        ev_fork, ev_join = torch.cuda.Event(), torch.cuda.Event()
        tail_side = attention_call(t["q"], pt["tt"], pt["tl"], t["qi"], t["qr"], o_t, l_t, 1, mt, "causal",
                                   on=side)

        def fork_tail():
            ev_fork.record(stream)
            side.wait_event(ev_fork)
            tail_side()
            ev_join.record(side)

        def join_merge():
            stream.wait_event(ev_join)
            merge()
        prefix_bytes = Gn * prefix * kv_tok_bytes
        tail_bytes = int(e["tail_lens"].sum()) * kv_tok_bytes
        aux["tail_attention"] = (tail, tail_bytes, "GB/s")
        aux["merge"] = (merge, rows * Hq * (D * 4 * 2 + D * 2 + 12), "GB/s")
        cfg.update(groups=Gn, samples=n_s, prefix=prefix, tail="U[1,1024]",
                   kv_bytes_per_step=prefix_bytes + tail_bytes,
                   kv_bytes_without_sharing=rows * prefix * kv_tok_bytes + tail_bytes,
                   l2="prefix pages 16.8 MB per group; 537 MB of K/V per step")
        h2d_src = [case.q, case.new_k, case.new_v, case.slots, e["tail_lens"], e["tail_table"]]
        h2d_dst = [t["q"], t["new_k"], t["new_v"], t["slots"], pt["tl"], pt["tt"]]
        return StepPlan(case=case, cfg=cfg, metric="shared-prefix KV GB/s", unit="GB/s",
                        work=prefix_bytes + tail_bytes, scale=1e9, queries=rows, pre=[scatter, fork_tail],
                        dominant=dom, post=[join_merge], aux=aux,
                        dom_label="paged_attention, prefix call: tcgen05 tile kernel, 8 samples x 4 "
                                  "heads = 32 rows held 4 times, HBM-bound (the tail call runs "
                                  "concurrently on a second stream)",
                        dom_work=prefix_bytes, bound="hbm", peak=peak_hbm, peak_unit="GB/s",
                        peak_src=f"{hbm_kind} hbm_gbs", h2d=(h2d_src, h2d_dst), d2h=d2h_src,
                        # scatter, prefix tile, the tail call (unit-order planner +
                        # decode kernel), merge
                        launches=5, traffic_sources=ATTN_TC_SOURCES)
    if name in ("shared_prefix_fused", "shared_prefix_verify"):
        # the step plans the grouping on the device (plan_shared_prefix) and runs
        # every row's shared run + tail in one launch (shared_prefix_attention)
        e = case.extra
        Gn, n_s, q_len = e["groups"], e["samples"], e["q_len"]
        B = case.batch
        width = case.block_table.shape[1]
        stride = width * n_s                       # a group row: at most n_s full rows
        max_keys = stride * 32
        plan_out = pkv.plan_buffers(B, stride, dev)
        mgt = n_s * q_len                          # tokens of one group
        ws_b = pkv.shared_prefix_attention_workspace_size(B, q_len, mgt, max_keys, Hq, Hkv, D)
        ws = torch.empty(max(ws_b, 256), dtype=torch.uint8, device=dev)
        plan_call = lambda: pkv.plan_shared_prefix(t["bt"], t["kl"], t["qi"], plan_out, stream=stream)
        dom = lambda: pkv.shared_prefix_attention(t["q"], t["k_pool"], t["v_pool"], plan_out, t["qi"], out,
                                                  lse=lse, max_q_len=q_len, max_group_tokens=mgt,
                                                  max_group_keys=max_keys, workspace=ws, stream=stream)
        prefix = int(e["prefix_lens"][0])
        prefix_bytes = Gn * prefix * kv_tok_bytes
        tail_bytes = int(e["tail_lens"].sum()) * kv_tok_bytes
        io_bytes = rows * Hq * (D * 2 * 2 + 4)
        aux["plan"] = (plan_call, B * width * 4 * 2, "GB/s")
        cfg.update(groups=Gn, samples=n_s, q_len=q_len, prefix=prefix, tail="U[1,1024]",
                   kv_bytes_per_step=prefix_bytes + tail_bytes,
                   kv_bytes_without_sharing=B * prefix * kv_tok_bytes + tail_bytes,
                   l2="prefix pages 16.8 MB per group; 537 MB of K/V per step",
                   grouping="planned on the device every step")
        h2d_src = [case.q, case.new_k, case.new_v, case.slots, case.kv_lens, case.block_table]
        h2d_dst = [t["q"], t["new_k"], t["new_v"], t["slots"], t["kl"], t["bt"]]
        return StepPlan(case=case, cfg=cfg, metric="shared-prefix KV GB/s", unit="GB/s",
                        work=prefix_bytes + tail_bytes, scale=1e9, queries=rows, pre=[scatter, plan_call],
                        dominant=dom, post=[], aux=aux,
                        dom_label="shared_prefix_attention: one grouped tcgen05 tile launch (run + "
                                  "tails of a group per CTA), HBM-bound",
                        dom_work=prefix_bytes + tail_bytes + io_bytes, bound="hbm", peak=peak_hbm,
                        peak_unit="GB/s", peak_src=f"{hbm_kind} hbm_gbs", h2d=(h2d_src, h2d_dst),
                        # scatter, the planner's two kernels, the grouped tile kernel
                        d2h=d2h_src, launches=4, traffic_sources=ATTN_TC_SOURCES)
    if name == "shared_prefix_plain_decode":
        # the ablation: every sample's whole row (prefix ++ tail) through plain
        # decode, the prefix pages read once per sample instead of once per group
        e = case.extra
        Gn, n_s = e["groups"], e["samples"]
        prefix = int(e["prefix_lens"][0])
        prefix_bytes = Gn * prefix * kv_tok_bytes
        tail_bytes = int(e["tail_lens"].sum()) * kv_tok_bytes
        attn_bytes, kv_read = decode_bytes(case)
        dom = attention_call(t["q"], t["bt"], t["kl"], t["qi"], t["qr"], out, lse, 1, case.max_kv_len,
                             "causal")
        cfg.update(groups=Gn, samples=n_s, prefix=prefix, tail="U[1,1024]",
                   kv_bytes_per_step=prefix_bytes + tail_bytes, kv_bytes_read_per_step=kv_read,
                   l2="prefix pages 16.8 MB per group; 2.4 GB of K/V read per step",
                   note="value counts the shared prefix once per group, as the shared-prefix "
                        "entries do, so the three values compare step times; roofline counts "
                        "the bytes this path reads")
        return StepPlan(case=case, cfg=cfg, metric="shared-prefix KV GB/s", unit="GB/s",
                        work=prefix_bytes + tail_bytes, scale=1e9, queries=rows, pre=[scatter],
                        dominant=dom, post=[], aux=aux,
                        dom_label="paged_attention over each sample's whole row: persistent "
                                  "split-KV decode kernel behind its unit-order planner",
                        dom_work=attn_bytes, bound="hbm", peak=peak_hbm, peak_unit="GB/s",
                        peak_src=f"{hbm_kind} hbm_gbs", h2d=(h2d_src, h2d_dst), d2h=d2h_src,
                        # scatter, the unit-order planner, the decode kernel
                        launches=3, traffic_sources=DECODE_SOURCES)
    raise ValueError(name)


def measure(plan, name, args, rank, world, local, dev, stream, dist):
    """Time one workload: warm-up, then exactly ``args.steps`` steps between
    barriers and synchronisations (CUDA events on the launching stream, the
    dominant call bracketed by its own events every step), the auxiliary
    launches as CUDA-graph replays, then the end-to-end loop through the
    public API from pinned host memory.  Returns the JSON entry (every rank
    returns its copy; values aggregate over ranks)."""
    import torch

    def step():
        for f in plan.pre:
            f()
        plan.dominant()
        for f in plan.post:
            f()

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
            for f in plan.pre:
                f()
            ev[i][0].record(stream)
            plan.dominant()
            ev[i][1].record(stream)
            for f in plan.post:
                f()
        t_end.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    wall1 = time.time()
    clk = clocks.stop(wall0, wall1)
    ms_total = t_start.elapsed_time(t_end)
    dom_ms = [a.elapsed_time(b) for a, b in ev]
    ms_total_max = max_over_ranks(dist, ms_total, dev)
    work_total = sum_over_ranks(dist, plan.work * args.steps, dev)
    queries_total = sum_over_ranks(dist, plan.queries * args.steps, dev)
    value = work_total / (ms_total_max * 1e-3) / plan.scale

    # ---- auxiliary launches of the step, each timed alone: 20 calls captured
    #      in a CUDA graph and replayed, so host call overhead is not measured
    aux_out = {}
    for key, (fn, nbytes, unit) in plan.aux.items():
        reps = 20
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            fn()  # warm (first-call set-up happens outside the capture)
            torch.cuda.synchronize()
            with torch.cuda.graph(graph, stream=stream):
                for _ in range(reps):
                    fn()
            graph.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            graph.replay()
            b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / reps
        aux_out[key] = {"ms": ms, "bytes": nbytes, "GB/s": nbytes / (ms * 1e-3) / 1e9,
                        "timing": f"{reps} calls in one CUDA graph replay"}
        del graph

    # ---- end to end through the public API: pinned host inputs -> device,
    #      the whole step, result read back to the host, every step, as a
    #      pipelined serving loop.  A step's inputs travel as one copy (one
    #      pinned host buffer holds them all, each at a 256-byte aligned offset)
    #      into one of two device staging buffers on an input copy stream while
    #      the previous step runs; the step copies them on the device into the
    #      buffer its input tensors are views of, runs, and copies its results
    #      (output and LSE, likewise packed) into one of two device staging
    #      buffers, which an output copy stream brings to one of two pinned
    #      host buffers while the next step runs.  The host stays one step
    #      ahead: it waits for step i - 1's result on the host after enqueueing
    #      step i.  Every copy of every step lies inside the timed region.
    #      A step that moves under PIPELINE_MIN_BYTES keeps the copies on the
    #      compute stream instead: there the pipelined loop's extra host calls
    #      cost more than the copies it hides (the tiny decode step is
    #      host-bound).
    e2e_value = None
    srcs, dsts = plan.h2d
    d_in, in_offs = packed_device(dsts, dev)
    h_in = torch.empty(d_in.numel(), dtype=torch.uint8).pin_memory()
    for x, o in zip(srcs, in_offs):
        n = x.numel() * x.element_size()
        h_in[o:o + n].copy_(x.contiguous().view(-1).view(torch.uint8))
    d_out, _ = packed_device(plan.d2h, dev)
    h_out = [torch.empty(d_out.numel(), dtype=torch.uint8).pin_memory() for _ in range(2)]
    in_stage = [torch.empty_like(d_in) for _ in range(2)]
    out_stage = [torch.empty_like(d_out) for _ in range(2)]
    h2d = h_in.numel()
    d2h = d_out.numel()
    in_stream = torch.cuda.Stream(device=dev)
    out_stream = torch.cuda.Stream(device=dev)
    staged = [torch.cuda.Event() for _ in range(2)]     # inputs of a step are on the device
    consumed = [torch.cuda.Event() for _ in range(2)]   # a step took its inputs and left its results
    on_host = [torch.cuda.Event() for _ in range(2)]    # a step's results are on the host

    pipelined = h2d + d2h >= PIPELINE_MIN_BYTES
    # the step's launches (every call of the step through the public API, on
    # the compute stream and any side stream it forks) captured once as a CUDA
    # graph, as a serving loop replays a decode step: one host call per step
    # instead of one per launch.  A step that cannot be captured runs eagerly.
    graph = torch.cuda.CUDAGraph()
    try:
        if args.e2e_steps <= 0:
            raise RuntimeError("no end-to-end steps requested")
        with torch.cuda.stream(stream):
            step()
            torch.cuda.synchronize()
            with torch.cuda.graph(graph, stream=stream):
                step()
        torch.cuda.synchronize()
        run_step = graph.replay
    except Exception as exc:  # capture refused (or not needed): keep the eager step
        if args.e2e_steps > 0:
            print(f"bench: {name}: step not captured ({type(exc).__name__}: {exc}); eager end to end",
                  file=sys.stderr)
        torch.cuda.synchronize()
        run_step = step

    def e2e_serial(n, start=None):
        for i in range(n):
            with torch.cuda.stream(stream):
                d_in.copy_(h_in, non_blocking=True)
                run_step()
                h_out[i % 2].copy_(d_out, non_blocking=True)
                on_host[i % 2].record(stream)
            if i >= 1:
                on_host[(i - 1) % 2].synchronize()
        on_host[(n - 1) % 2].synchronize()

    def e2e_steps(n, start=None):
        if not pipelined:
            return e2e_serial(n, start)
        # copy stream order: inputs of steps 0 and 1, then results of step i
        # before inputs of step i + 2 (whose staging buffer step i frees)
        def bring_in(i):
            with torch.cuda.stream(in_stream):
                if i >= 2:
                    in_stream.wait_event(consumed[i % 2])
                in_stage[i % 2].copy_(h_in, non_blocking=True)
                staged[i % 2].record(in_stream)
        if start is not None:
            in_stream.wait_event(start)
            out_stream.wait_event(start)
        bring_in(0)
        if n > 1:
            bring_in(1)
        for i in range(n):
            with torch.cuda.stream(stream):
                stream.wait_event(staged[i % 2])
                d_in.copy_(in_stage[i % 2], non_blocking=True)
                run_step()
                if i >= 2:
                    stream.wait_event(on_host[i % 2])  # step i - 2's results have left
                out_stage[i % 2].copy_(d_out, non_blocking=True)
                consumed[i % 2].record(stream)
            with torch.cuda.stream(out_stream):
                out_stream.wait_event(consumed[i % 2])
                h_out[i % 2].copy_(out_stage[i % 2], non_blocking=True)
                on_host[i % 2].record(out_stream)
            if i + 2 < n:
                bring_in(i + 2)
            if i >= 1:
                on_host[(i - 1) % 2].synchronize()  # step i - 1's result is on the host
        on_host[(n - 1) % 2].synchronize()
        stream.wait_event(on_host[(n - 1) % 2])

    if args.e2e_steps > 0:
        e2e_steps(3)
        barrier(dist)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_steps(args.e2e_steps, start=e0)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(dist, e0.elapsed_time(e1), dev)
        e2e_value = sum_over_ranks(dist, plan.work * args.e2e_steps, dev) / (e2e_ms * 1e-3) / plan.scale

    dom_avg = statistics.mean(dom_ms)
    achieved = plan.dom_work / (dom_avg * 1e-3) / (1e9 if plan.bound == "hbm" else 1.0)
    traffic = committed_traffic(name, plan.traffic_sources)
    entry = {
        "metric": plan.metric, "value": value, "unit": plan.unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_total_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": dict(plan.cfg, parallelism=f"independent replicas x{world} (seed + rank), "
                                             "no collective"),
        "queries_per_s": queries_total / (ms_total_max * 1e-3),
        "roofline": {"bound": plan.bound, "achieved": achieved, "peak": plan.peak,
                     "unit": plan.peak_unit, "frac": achieved / plan.peak, "traffic": traffic,
                     "kernel": plan.dom_label + "; CUDA events around the call each timed step",
                     "work_per_launch": plan.dom_work, "avg_launch_ms": dom_avg,
                     "peak_source": plan.peak_src},
        "clocks": clk,
        "e2e": {"value": e2e_value, "unit": plan.unit, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
                "loop": ("pipelined: each step's inputs copied in (one pinned buffer, one copy) "
                         "while the previous step runs and its results copied out while the "
                         "next one runs, on two copy streams through double-buffered device "
                         "staging; the host waits for each step's result one step behind"
                         if pipelined else
                         "serial: each step's inputs copied in (one copy), the step, its results "
                         "copied out (one copy), all on the compute stream; the host waits for "
                         "each step's result one step behind")
                        + ("; the step's launches replayed as one captured CUDA graph"
                           if run_step is not step else "; the step's calls made eagerly")},
        "gpu_launches": plan.launches * args.steps,
        "aux": aux_out,
    }
    if plan.unit == "GB/s":
        entry["hbm_frac"] = value / plan.peak if plan.bound == "hbm" else None
    return entry


def run_ours(args):
    import gc
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
    stream = torch.cuda.Stream(device=dev)
    names = [args.workload]
    if not args.only and args.workload == "gqa_decode":
        names += list(EXTRA_WORKLOADS)
    line, extra = None, {}
    for name in names:
        plan = build_plan(name, rank, dev, stream)
        entry = measure(plan, name, args, rank, world, local, dev, stream, dist)
        case = plan.case
        del plan
        gc.collect()
        torch.cuda.empty_cache()
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            entry["cpu_baseline"] = cpu_baseline_for(name, case, entry["unit"], 1e9 if entry["unit"] == "GB/s"
                                                     else 1e12)
        del case
        if line is None:
            line = entry
        else:
            extra[name] = {k: v for k, v in entry.items()
                           if k not in ("n_gpus", "higher_is_better", "scaling", "vs_baseline", "data",
                                        "dtype", "warmup")}
    if rank == 0:
        if extra:
            line["workloads"] = extra
        print(json.dumps(line), flush=True)
    barrier(dist)
    return 0


def packed_device(tensors, dev):
    """One device byte buffer holding every tensor of ``tensors`` at a 256-byte
    aligned offset; each tensor is rebound in place to its view of the buffer
    (the step's callables keep working on the same tensor objects).  Returns
    ``(buffer, offsets)``.  The tensors' contents are not carried over."""
    import torch
    offs, total = [], 0
    for x in tensors:
        assert x.is_contiguous()
        offs.append(total)
        total += -(-x.numel() * x.element_size() // 256) * 256
    buf = torch.empty(max(total, 256), dtype=torch.uint8, device=dev)
    for x, o in zip(tensors, offs):
        x.set_(buf.untyped_storage(), o // x.element_size(), x.shape, x.stride())
    return buf, offs


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
