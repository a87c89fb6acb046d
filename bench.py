"""Benchmark of the paged decode path on GB300 (prints one JSON line).

Workload (default): one Llama-3-8B decode layer -- batch 32, 32 query / 8 KV
heads, head_dim 128, bf16, every context 8192 tokens in 16-token blocks,
block tables a random permutation of a 16384-block pool (1 GiB of K+V, more
than the 129 MB L2, so no flush is needed between steps). The default run
also measures the 128K-context 70B-GQA layer (batch 4, 64 q / 8 KV heads,
2 GiB of K+V) the same way and nests its figures under ``also``.

One step = the whole hot path for one decode token per sequence:
  pkv_copy_blocks (this workload shares no blocks: zero pairs, no launch)
  -> pkv_append (each sequence's new K/V at position 8191)
  -> pkv_decode_attention (one launch: split kernel with the merge fused).
value = KV bytes read per step / device time per step (decimal GB/s).

Beside the timed steps: a window of back-to-back decode calls (the kernel's
own duration, for the roofline), 50 single calls (percentiles), end-to-end
steps from pinned host memory, steps after an L2 scrub, and the append and
block-copy calls alone (microseconds per call). SM clocks are sampled with
nvidia-smi every 10 ms from warm-up to the end of the GPU work.

--workload prefix runs the shared-prefix call by default
(pkv_decode_attention_prefixed: every sequence in one group over the 256
shared blocks); --single-pass times pkv_decode_attention over the same tables.
There value counts the K/V bytes attended (logical); unique_kv_gbs counts each
stored byte once.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl pkv|reference]
                  [--workload NAME] [--also NAMES|none] [--single-pass]

--impl reference times the float64 CPU oracle (the only other code here) on
the host's cores, on a bounded sample of the same workload per step. Under
torchrun with N > 1 every rank runs its own replica of the workload on its
own GPU (weak scaling, no collective on the data path); timing is the max
over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

# Each oracle process runs one thread (BLAS included); the full-core baseline
# runs one such process per core.
for _var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ[_var] = "1"

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_209_gb300 import workloads as W  # noqa: E402

METRIC = "paged decode attention KV GB/s (% of GB300 HBM peak) and KV tokens/s, 1 GPU"
WORKLOAD = "llama8k"
ALSO_DEFAULT = {"llama8k": ["long128k"]}
FALLBACK_HBM_GBS = 6800.0
DECODE_WINDOW = 200       # back-to-back decode calls timed between two events (roofline)
SINGLE_CALLS = 50         # decode calls timed one by one (percentiles)
MOVE_WINDOW = 100         # append / block-copy calls timed back to back
COPY_PAIRS = (31, 1024)   # block-copy sizes timed: the copy-on-write prefix variant's 31 pairs, and 1024
HOST_SAMPLE_BYTES = 1 << 30   # K+V copied to the host for the CPU oracle baseline (at most, whole sequences)


WORKLOAD_NAMES = {
    "llama8k": "Llama-3-8B decode layer, every context 8192 tokens",
    "long128k": "70B-GQA decode layer, every context 131072 tokens",
    "mixed": "continuous-batching mix, contexts log-uniform on [16, 32768]",
    "prefix": "4096-token prefix shared by all sequences + private suffixes uniform in [1, 2048]",
    "spec4": "Llama-3-8B decode layer verifying 4 draft tokens per sequence (causal multi-query), context 8192",
    "llama8k_q8": "Llama-3-8B decode layer over an int8 KV cache (per-row float32 scales), every context 8192 tokens",
    "prefill512": "chunked prefill on the Llama-3-8B layer: 512 causal queries per sequence, context 8192",
}
L2_NOTE = {
    "llama8k": "inputs larger than L2 (1 GiB K+V per step)",
    "long128k": "inputs larger than L2 (2 GiB K+V per step)",
    "mixed": "inputs larger than L2 (4.65 GB K+V per step)",
    "prefix": "unique K+V (0.33 GB) larger than L2; the 16 MiB shared prefix is re-read from L2 by every "
              "sequence, so logical GB/s can exceed HBM bandwidth",
    "spec4": "inputs larger than L2 (1 GiB K+V per step, read once for the 4 queries of each sequence)",
    "llama8k_q8": "inputs larger than L2 (0.55 GB of K+V codes and scales per step)",
    "prefill512": "K+V 0.27 GB (larger than L2); the 16 query tiles of a sequence re-read its K/V, mostly from L2",
}


def workload_desc(name, cfg, lens):
    kind = "int8 K/V codes + float32 row scales, bf16 q" if cfg["dtype"] == "int8" else cfg["dtype"]
    return (f"{WORKLOAD_NAMES[name]}: batch {cfg['batch']}, {cfg['q_heads']} q / {cfg['kv_heads']} kv heads, "
            f"head_dim {cfg['head_dim']}, 16-token blocks, shuffled pool, {kind}, {int(lens.sum())} KV tokens")


def kv_bytes_per_token(cfg):
    """Bytes of one token's K and V over all KV heads (codes + scales for int8)."""
    if cfg["dtype"] == "int8":
        return 2 * cfg["kv_heads"] * (cfg["head_dim"] + 4)
    return 2 * cfg["kv_heads"] * cfg["head_dim"] * (4 if cfg["dtype"] == "f32" else 2)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ distributed plumbing
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, ws: int, device=None) -> float:
    if ws <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling (every 10 ms) of SM clocks and throttle reasons
    while the GPU work runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 10

    def __init__(self, gpu_id: str):
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"pkv_clocks_{os.getpid()}.csv")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", gpu_id, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.INTERVAL_MS)],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        # the GPU work starts once the sampler has written its first line (or after 5 s)
        t0 = time.time()
        while time.time() - t0 < 5.0 and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "sm_mhz_min": min(sm) if sm else None, "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm), "interval_ms": self.INTERVAL_MS,
                "span": "from the first warm-up step to the end of the GPU work of every workload in this line"}


# ------------------------------------------------------------------ peaks and profiles
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        return json.load(open(p))
    except Exception:
        return {}


def hbm_peak():
    peaks = measured_peaks()
    if "hbm_gbs" in peaks:
        return float(peaks["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_sha(files=("pkv_decode.cu",)):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "paged_kv_cache_209_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(summary, files=("pkv_decode.cu",)):
    """DRAM bytes per decode call from the committed ncu summary
    profiles/<summary>.md, if it was taken on the current kernel source
    (else None)."""
    p = os.path.join(ROOT, "profiles", f"{summary}.md")
    if not os.path.exists(p):
        return None
    text = open(p).read()
    m_sha = re.search(r"source_sha:\s*([0-9a-f]+)", text)
    m_tr = re.search(r"dram_bytes_per_call:\s*([0-9]+)", text)
    if not m_sha or not m_tr or m_sha.group(1) != kernel_source_sha(files):
        return None
    return int(m_tr.group(1))


# ------------------------------------------------------------------ CPU oracle baseline
# The oracle runs in worker processes (spawn start method: the workers never
# inherit a CUDA context), one thread each. Arrays reach them as .npy files
# in a temporary directory (shared memory where the host has /dev/shm),
# memory-mapped read-only.
_ARRAYS = {}


def _load(paths):
    out = []
    for p in paths:
        if p not in _ARRAYS:
            _ARRAYS[p] = np.load(p, mmap_mode="r")
        out.append(_ARRAYS[p])
    return out


def _oracle_task(task):
    """One unit of oracle work in a worker; returns the K/V bytes it attended."""
    kind, paths, args = task
    if kind == "warm":
        import oracle  # noqa: F401
        return 0
    if kind == "pair":          # decode: one (sequence, KV head)
        from oracle import attention as OA
        q, kp, vp, tables, lens = _load(paths)
        i, j, scale, kv_heads = args
        OA.decode_attention_pair(q, kp, vp, tables, lens, scale, i, j, kv_heads, "bf16")
        return int(lens[i]) * 2 * kp.shape[-1] * 2
    if kind == "mq":            # multi-query: the last `ns` of one sequence's nq queries, all KV heads
        from oracle import multiquery as OM
        q, kp, vp, tables, lens = _load(paths)
        i, scale, kv_heads, nq, ns = args
        OM.multiquery_attention(q[(i + 1) * nq - ns:(i + 1) * nq], kp, vp, tables[i:i + 1], lens[i:i + 1],
                                np.array([0, ns]), scale, kv_heads, "bf16")
        return int(lens[i]) * 2 * kv_heads * kp.shape[-1] * 2 * ns // nq
    if kind == "q8":            # int8 cache: one whole sequence, all KV heads
        from oracle import quant as OQ
        q, kc, vc, ks, vs, tables, lens = _load(paths)
        i, scale, kv_heads = args
        # the oracle dequantizes every block it is handed: hand it this sequence's blocks only
        nblk = (int(lens[i]) + 15) // 16
        sel = tables[i, :nblk]
        OQ.decode_attention_q8(q[i:i + 1], kc[sel], vc[sel], ks[sel], vs[sel],
                               np.arange(nblk, dtype=np.int32)[None, :], lens[i:i + 1], scale, kv_heads, "bf16")
        return int(lens[i]) * 2 * kv_heads * (kc.shape[-1] + 4)
    raise ValueError(kind)


class OracleRunner:
    """The float64 oracle over a host copy of (part of) a workload, timed on
    one core in this process or on all of the host's cores in a pool of
    single-threaded worker processes."""

    def __init__(self):
        self.dirs = []
        self.pool = None
        self.cores = host_cores()

    def start_pool(self):
        import multiprocessing as mp
        self.pool = mp.get_context("spawn").Pool(self.cores)
        self.pool.map(_oracle_task, [("warm", (), ())] * self.cores)

    def put(self, name, arr):
        """Writes ``arr`` where there is room for it (shared memory first)."""
        need = arr.nbytes + (1 << 20)
        for base in ("/dev/shm", tempfile.gettempdir()):
            if os.path.isdir(base) and shutil.disk_usage(base).free > 2 * need:
                break
        else:
            raise RuntimeError(f"no room for {need} bytes of oracle input")
        d = next((x for x in self.dirs if os.path.dirname(x) == base), None)
        if d is None:
            d = tempfile.mkdtemp(prefix="pkv_oracle_", dir=base)
            self.dirs.append(d)
        path = os.path.join(d, name + ".npy")
        np.save(path, np.ascontiguousarray(arr))
        return path

    def run(self, tasks, all_cores: bool, min_seconds: float = 0.0, max_seconds: float = 20.0):
        """Runs the tasks (repeated until ``min_seconds`` have passed, stopping
        early after ``max_seconds``); returns (bytes, seconds, tasks done)."""
        nbytes, done = 0, 0
        t0 = time.perf_counter()
        while True:
            if all_cores:
                for b in self.pool.imap_unordered(_oracle_task, tasks):
                    nbytes += b
                    done += 1
            else:
                for t in tasks:
                    nbytes += _oracle_task(t)
                    done += 1
                    if time.perf_counter() - t0 > max_seconds:
                        break
            el = time.perf_counter() - t0
            if el >= min_seconds or el > max_seconds:
                return nbytes, el, done

    def close(self):
        if self.pool is not None:
            self.pool.terminate()
            self.pool.join()
        _ARRAYS.clear()
        for d in self.dirs:
            shutil.rmtree(d, ignore_errors=True)


def oracle_tasks(runner, name, cfg, host):
    """Tasks covering the host copy ``host`` of a workload (every (sequence,
    KV head) pair for decode; every sequence for the int8 cache and for
    multi-query, chunked prefill on its last 8 queries)."""
    scale = 1.0 / np.sqrt(cfg["head_dim"])
    HKV = cfg["kv_heads"]
    nq = cfg.get("queries", 1)
    if cfg["dtype"] == "int8":
        paths = tuple(runner.put(k, host[k]) for k in ("q", "kc", "vc", "ks", "vs", "tables", "lens"))
        tasks = [("q8", paths, (i, scale, HKV)) for i in range(len(host["lens"]))]
        what = f"{len(tasks)} whole sequences (int8 cache, all KV heads)"
        return tasks, what
    paths = tuple(runner.put(k, host[k]) for k in ("q", "kp", "vp", "tables", "lens"))
    if nq > 1:
        ns = 8 if nq * cfg["q_heads"] // HKV > 32 else nq
        tasks = [("mq", paths, (i, scale, HKV, nq, ns)) for i in range(len(host["lens"]))]
        what = (f"the last {ns} of the {nq} queries of {len(tasks)} sequences (bytes credited in proportion)"
                if ns < nq else f"{len(tasks)} whole sequences ({nq} queries each)")
        return tasks, what
    tasks = [("pair", paths, (i, j, scale, HKV)) for i in range(len(host["lens"])) for j in range(HKV)]
    return tasks, f"{len(tasks)} (sequence, KV head) pairs"


# ------------------------------------------------------------------ reference arm
def run_reference(args, cfg):
    """--impl reference: the CPU oracle on all host cores, timed per step on a
    bounded sample of the workload: the longest sequence, all KV heads (two
    sequences for decode workloads, whose unit is one (sequence, KV head))."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import torch
    tables_all, lens_all, _ = W.workload_index(args.workload)
    order = np.argsort(-lens_all, kind="stable")
    nq = cfg.get("queries", 1)
    seqs = [int(order[0])] + ([int(order[1])] if nq == 1 and cfg["dtype"] != "int8" and len(order) > 1 else [])
    lens = lens_all[seqs].astype(np.int32)
    nbs = [(int(n) + 15) // 16 for n in lens]
    # Only the sampled sequences' blocks are materialised (on the host), renumbered 0 .. sum(nbs) - 1.
    tables = np.full((len(seqs), max(nbs)), -1, dtype=np.int32)
    off = 0
    for r, nb in enumerate(nbs):
        tables[r, :nb] = np.arange(off, off + nb)
        off += nb
    g = torch.Generator().manual_seed(cfg["seed"])
    shape = (off, cfg["kv_heads"], 16, cfg["head_dim"])
    q = torch.randn((len(seqs) * nq, cfg["q_heads"], cfg["head_dim"]), generator=g).to(torch.bfloat16)
    host = {"q": q.view(torch.int16).numpy().view(np.uint16), "tables": tables, "lens": lens}
    if cfg["dtype"] == "int8":
        rng = np.random.default_rng(cfg["seed"])
        host.update(kc=np.clip(np.rint(rng.standard_normal(shape) * 42), -127, 127).astype(np.int8),
                    vc=np.clip(np.rint(rng.standard_normal(shape) * 42), -127, 127).astype(np.int8),
                    ks=rng.uniform(0.02, 0.03, shape[:3]).astype(np.float32),
                    vs=rng.uniform(0.02, 0.03, shape[:3]).astype(np.float32))
    else:
        host.update(kp=torch.randn(shape, generator=g).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16),
                    vp=torch.randn(shape, generator=g).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    runner = OracleRunner()
    try:
        runner.start_pool()
        tasks, what = oracle_tasks(runner, args.workload, cfg, host)
        for _ in range(args.warmup):
            runner.run(tasks, all_cores=True)
        tot_b, tot_s = 0, 0.0
        for _ in range(args.steps):
            b, s_, _ = runner.run(tasks, all_cores=True)
            tot_b += b
            tot_s += s_
    finally:
        runner.close()
    gbs = tot_b / tot_s / 1e9
    sample = (f"{what} of the workload's longest sequence{'s' if len(seqs) > 1 else ''} per step "
              f"(lengths {[int(n) for n in lens]}), float64 NumPy oracle, {runner.cores} single-threaded processes")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_s / max(args.steps, 1) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(args.workload, cfg, lens_all), "sample": sample},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": runner.cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "kv_tokens_per_s": round(tot_b / kv_bytes_per_token(cfg) / tot_s, 1),
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm
def _events(torch, n):
    return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]


def measure_workload(name, args, ws, rank, device, single_pass=False, want_host=False):
    """Times one workload on this rank's GPU; returns its figures (and, with
    ``want_host``, the host copy of the workload for the CPU baseline)."""
    import torch
    from paged_kv_cache_209_gb300 import pkv
    cfg = dict(W.CONFIGS[name])
    w = W.device_workload(name, device, seed_offset=1000 * rank)
    B, HQ, HKV, D = cfg["batch"], cfg["q_heads"], cfg["kv_heads"], cfg["head_dim"]
    k_pool, v_pool, q, kn, vn = w["k_pool"], w["v_pool"], w["q"], w["k_new"], w["v_new"]
    tables, lens, slots, pairs = w["tables"], w["lens"], w["slots"], w["pairs"]
    tables_np, lens_np = w["tables_np"], w["lens_np"]
    MAXB = tables.shape[1]
    out = torch.empty_like(q)
    two_phase = name == "prefix" and not single_pass
    q8 = cfg["dtype"] == "int8"
    nq = w["queries"]
    qstart = w["query_start"]
    group, gblocks, mgb = w["prefix_group"], w["group_blocks"], w["max_group_blocks"]
    if q8:
        sc_pool = w["scales"]          # [blocks][heads][2][16]: K-row and V-row scales
        ws_bytes = pkv.pkv_decode_q8_workspace_size(B, HQ, MAXB, k_pool)
    elif two_phase:
        ws_bytes = pkv.pkv_decode_prefixed_workspace_size(B, HQ, MAXB, len(gblocks), mgb, k_pool)
    elif nq > 1:
        ws_bytes = pkv.pkv_multiquery_workspace_size(B, HQ, MAXB, nq, k_pool)
    else:
        ws_bytes = pkv.pkv_decode_workspace_size(B, HQ, MAXB, k_pool)
    workspace = torch.zeros(ws_bytes, dtype=torch.uint8, device=device)
    scale = w["scale"]
    stream = torch.cuda.current_stream()

    def decode():
        if q8:
            pkv.pkv_decode_attention_q8(q, k_pool, v_pool, sc_pool, tables, lens, scale, out=out,
                                        workspace=workspace, stream=stream)
        elif nq > 1:
            pkv.pkv_multiquery_attention(q, k_pool, v_pool, tables, lens, qstart, scale, nq, out=out,
                                         workspace=workspace, stream=stream)
        elif two_phase:
            pkv.pkv_decode_attention_prefixed(q, k_pool, v_pool, tables, lens, scale, group, gblocks, mgb, out=out,
                                              workspace=workspace, stream=stream)
        else:
            pkv.pkv_decode_attention(q, k_pool, v_pool, tables, lens, scale, out=out, workspace=workspace,
                                     stream=stream)

    def copy_blocks(p):
        if q8:
            pkv.pkv_copy_blocks_q8(p, k_pool, v_pool, sc_pool, stream=stream)
        else:
            pkv.pkv_copy_blocks(p, k_pool, v_pool, stream=stream)

    def append():
        if q8:
            pkv.pkv_append_q8(kn, vn, slots, k_pool, v_pool, sc_pool, stream=stream)
        else:
            pkv.pkv_append(kn, vn, slots, k_pool, v_pool, stream=stream)

    def step():
        copy_blocks(pairs)
        append()
        decode()

    # append + per 1024 sequences one decode launch (two with the shared-prefix pass)
    launches_per_step = 1 + (2 if two_phase else 1) * ((B + 1023) // 1024)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # -------- device-timed region: K whole steps, nothing else between the two events
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(args.steps):
        step()
    end.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    ms_total = max_over_ranks(start.elapsed_time(end), ws, device)
    status_bits = pkv.pkv_device_status(clear=False)

    # -------- the decode kernel's own duration: DECODE_WINDOW calls back to
    # back between two events on the launching stream (each call's launch and
    # prologue overlap the previous call's tail, as they overlap the append's
    # inside a step); then SINGLE_CALLS calls each between its own events.
    for _ in range(3):
        decode()
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    w0.record(stream)
    for _ in range(DECODE_WINDOW):
        decode()
    w1.record(stream)
    torch.cuda.synchronize()
    dec_avg_ms = max_over_ranks(w0.elapsed_time(w1) / DECODE_WINDOW, ws, device)
    evs = _events(torch, SINGLE_CALLS)
    for e0, e1 in evs:
        e0.record(stream)
        decode()
        e1.record(stream)
    torch.cuda.synchronize()
    single_ms = [e0.elapsed_time(e1) for e0, e1 in evs]

    # -------- end-to-end: per-step inputs from pinned host memory, result back to the host.
    # Every step's inputs live in one pinned host buffer and one device buffer
    # (256-byte aligned slices the kernels read in place), so a step costs one
    # host-to-device copy, the kernels and one device-to-host copy of its
    # result. Two sets of buffers alternate, as in a serving loop: on a second
    # stream the inputs of step k + 1 go in and the result of step k comes out
    # while the kernels of step k (or k + 1) run.
    names = ["q", "kn", "vn", "slots", "tables", "lens"] + (["group", "gblocks"] if two_phase else []) \
        + (["qstart"] if nq > 1 else [])
    srcs = {"q": q, "kn": kn, "vn": vn, "slots": slots, "tables": tables, "lens": lens, "group": group,
            "gblocks": gblocks, "qstart": qstart}
    offs, total = {}, 0
    for n in names:
        offs[n] = total
        total += (srcs[n].numel() * srcs[n].element_size() + 255) // 256 * 256
    pack_dev = [torch.zeros(total, dtype=torch.uint8, device=device) for _ in range(2)]
    pack_host = [torch.zeros(total, dtype=torch.uint8).pin_memory() for _ in range(2)]
    views = [{}, {}]
    for b in range(2):
        for n in names:
            t = srcs[n]
            nb = t.numel() * t.element_size()
            views[b][n] = pack_dev[b][offs[n]:offs[n] + nb].view(t.dtype).view(t.shape)
            views[b][n].copy_(t)
            pack_host[b][offs[n]:offs[n] + nb].copy_(t.reshape(-1).view(torch.uint8).cpu())
    q_dev_orig, tables_orig, lens_orig = q, tables, lens
    outs = [out, torch.empty_like(out)]
    out_pins = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    h2d = total
    d2h = out_pins[0].numel() * out_pins[0].element_size()

    def use(b):
        """Point the step's inputs and output at buffer set b."""
        nonlocal q, kn, vn, slots, tables, lens, group, gblocks, qstart, out
        v = views[b]
        q, kn, vn, slots, tables, lens = (v[n] for n in ["q", "kn", "vn", "slots", "tables", "lens"])
        if two_phase:
            group, gblocks = v["group"], v["gblocks"]
        if nq > 1:
            qstart = v["qstart"]
        out = outs[b]

    copy_stream = torch.cuda.Stream(device=device)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of set b are on the device
    ev_done = [torch.cuda.Event() for _ in range(2)]  # the step that used set b has finished
    ev_out = [torch.cuda.Event() for _ in range(2)]   # the result in outs[b] has reached the host

    def e2e_run(n_steps):
        with torch.cuda.stream(copy_stream):
            pack_dev[0].copy_(pack_host[0], non_blocking=True)
        ev_in[0].record(copy_stream)
        for k in range(n_steps):
            b = k & 1
            if k + 1 < n_steps:
                if k >= 1:
                    copy_stream.wait_event(ev_done[1 - b])   # step k - 1 has read set 1 - b
                with torch.cuda.stream(copy_stream):
                    pack_dev[1 - b].copy_(pack_host[1 - b], non_blocking=True)
                ev_in[1 - b].record(copy_stream)
            stream.wait_event(ev_in[b])
            if k >= 2:
                stream.wait_event(ev_out[b])                 # step k - 2's result has left outs[b]
            use(b)
            step()
            ev_done[b].record(stream)
            copy_stream.wait_event(ev_done[b])
            with torch.cuda.stream(copy_stream):
                out_pins[b].copy_(outs[b], non_blocking=True)
            ev_out[b].record(copy_stream)
        torch.cuda.synchronize()

    e2e_run(max(3, args.warmup))
    barrier(ws)
    t0 = time.perf_counter()
    e2e_run(args.steps)
    e2e_s = max_over_ranks(time.perf_counter() - t0, ws, device)
    barrier(ws)
    use(0)

    # -------- cold L2: a 256 MiB buffer (twice the L2) is written before each
    # step, and the step alone is event-timed (50 steps)
    scrub = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=device)
    cold = []
    for _ in range(50):
        scrub.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        cold.append((e0, e1))
    torch.cuda.synchronize()
    cold_ms = sorted(a0.elapsed_time(a1) for a0, a1 in cold)
    del scrub

    # -------- host copy for the CPU baseline (before the block-copy timing
    # overwrites blocks): the first sequences, in index order, up to 1 GiB of
    # K+V, with their blocks renumbered into a sub-pool
    host = None
    if want_host:
        per_seq = lens_np.astype(np.int64) * kv_bytes_per_token(cfg)
        n_seq = int(min(B, max(1, np.searchsorted(np.cumsum(per_seq), HOST_SAMPLE_BYTES) + 1)))
        t_s = tables_np[:n_seq]
        ids = np.unique(t_s[t_s >= 0])
        remap = -np.ones(w["num_blocks"], dtype=np.int64)
        remap[ids] = np.arange(len(ids))
        idx = torch.from_numpy(ids.astype(np.int64)).to(device)
        host = {"tables": np.where(t_s >= 0, remap[np.maximum(t_s, 0)], -1).astype(np.int32),
                "lens": lens_np[:n_seq],
                "q": q_dev_orig[:n_seq * nq].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)}
        if q8:
            host.update(kc=k_pool.index_select(0, idx).cpu().numpy(),
                        vc=np.ascontiguousarray(v_pool.index_select(0, idx).cpu().numpy().transpose(0, 1, 3, 2)),
                        ks=sc_pool[:, :, 0].index_select(0, idx).cpu().numpy(),
                        vs=sc_pool[:, :, 1].index_select(0, idx).cpu().numpy())
        else:
            host.update(kp=k_pool.index_select(0, idx).view(torch.int16).cpu().numpy().view(np.uint16),
                        vp=v_pool.index_select(0, idx).view(torch.int16).cpu().numpy().view(np.uint16))

    # -------- the append and the block copy alone: MOVE_WINDOW calls captured
    # in one CUDA graph and replayed between two events, so the figure is
    # device time per call (issued one by one from Python, these small calls
    # are bound by the host's launch rate instead)
    def window_us(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(MOVE_WINDOW):
                fn()
        graph.replay()
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        graph.replay()
        a1.record(stream)
        torch.cuda.synchronize()
        del graph
        return max_over_ranks(a0.elapsed_time(a1) * 1e3 / MOVE_WINDOW, ws, device)

    def append_cur():       # on the current stream (the capture stream while capturing)
        if q8:
            pkv.pkv_append_q8(kn, vn, slots, k_pool, v_pool, sc_pool)
        else:
            pkv.pkv_append(kn, vn, slots, k_pool, v_pool)

    def copy_cur(p):
        if q8:
            pkv.pkv_copy_blocks_q8(p, k_pool, v_pool, sc_pool)
        else:
            pkv.pkv_copy_blocks(p, k_pool, v_pool)

    append_us = window_us(append_cur)
    block_bytes = 2 * HKV * 16 * (D + 4 if q8 else D * (4 if cfg["dtype"] == "f32" else 2))   # K+V, one block
    copy_us = {}
    perm = np.random.default_rng(1234).permutation(w["num_blocks"])
    for n in COPY_PAIRS:
        if 2 * n > w["num_blocks"]:
            continue
        p = torch.from_numpy(np.stack([perm[:n], perm[n:2 * n]], axis=1).astype(np.int64)).to(device)
        us = window_us(lambda: copy_cur(p))
        copy_us[f"pairs_{n}"] = {"us_per_call": round(us, 2), "bytes_moved": 2 * n * block_bytes,
                                 "gbs": round(2 * n * block_bytes / (us * 1e-6) / 1e9, 1)}

    res = dict(name=name, cfg=cfg, lens_np=lens_np, B=B, HQ=HQ, HKV=HKV, D=D, q8=q8, nq=nq, two_phase=two_phase,
               mgb=mgb, pairs_n=int(pairs.shape[0]), ms_total=ms_total, dec_avg_ms=dec_avg_ms, single_ms=single_ms,
               e2e_s=e2e_s, h2d=h2d, d2h=d2h, cold_ms=cold_ms, status_bits=status_bits,
               launches_per_step=launches_per_step, append_us=append_us, copy_us=copy_us,
               q_bytes=q.numel() * q.element_size(), out_bytes=out.numel() * out.element_size())
    del w, k_pool, v_pool, workspace, pack_dev, q_dev_orig, tables_orig, lens_orig
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res, host


def summarize(res, args, ws):
    """The JSON figures of one measured workload."""
    name, cfg, lens_np = res["name"], res["cfg"], res["lens_np"]
    B, HQ, HKV, D, nq = res["B"], res["HQ"], res["HKV"], res["D"], res["nq"]
    q8, two_phase = res["q8"], res["two_phase"]
    kv_tokens = int(lens_np.sum())
    tok_bytes = kv_bytes_per_token(cfg)
    total_kv = kv_tokens * tok_bytes * ws
    ms_per_step = res["ms_total"] / args.steps
    value = total_kv / (ms_per_step * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()
    dec_avg_ms = res["dec_avg_ms"]
    # algorithmic bytes of one decode call: K+V of every live token read once,
    # q read, out written, block-table entries and lengths read. With the
    # shared-prefix pass the shared blocks count once (the bytes a perfect
    # kernel must move), not once per sequence.
    used_entries = int(((lens_np.astype(np.int64) + 15) // 16).sum())
    shared_tokens = int(res["mgb"]) * 16 * (B - 1) if two_phase else 0
    unique_kvb = (kv_tokens - shared_tokens) * tok_bytes
    alg_bytes = unique_kvb + res["q_bytes"] + res["out_bytes"] + used_entries * 4 + B * 4
    achieved = alg_bytes / (dec_avg_ms * 1e-3) / 1e9
    # chunked prefill (more than 32 query rows per KV head) runs on the
    # tensor-core tile kernel: a dense contraction, so its roofline is tensor
    # throughput. Algorithmic FLOPs: 4 D per (query row, visible token)
    # (2 D for q.k, 2 D for p.v), summed over the causal triangle.
    prefill = nq * (HQ // HKV) > 32
    if prefill:
        vis = sum(int(n) * nq - nq * (nq - 1) // 2 for n in lens_np)   # sum over t of (n - nq + t + 1)
        alg_flops = vis * HQ * D * 4
        tflops = alg_flops / (dec_avg_ms * 1e-3) / 1e12
        peaks = measured_peaks()
        t_peak = float(peaks.get("bf16_tflops", 1900.0))
        t_kind = "measured (cuBLAS bf16 burst)" if "bf16_tflops" in peaks else "fallback"
        traffic = profiled_traffic(f"decode_{name}", ("pkv_prefix.cu",))
    elif two_phase:
        traffic = profiled_traffic("decode_prefix_two_phase", ("pkv_decode.cu", "pkv_prefix.cu"))
    elif q8 or nq > 1:
        traffic = profiled_traffic(f"decode_{name}", ("pkv_multiquery.cu",))
    else:
        traffic = profiled_traffic(f"decode_{name}")
    window = (f"{DECODE_WINDOW} calls back to back between two CUDA events on the launching stream, after the "
              "timed steps (each call's launch and prologue overlap the previous call's tail)")
    if prefill:
        roof = {"bound": "tensor", "achieved": round(tflops, 2), "peak": t_peak, "peak_kind": t_kind,
                "unit": "TFLOP/s", "frac": round(tflops / t_peak, 4), "traffic": traffic,
                "kernel": "prefix_umma_kernel<128, prefill> (one launch per pkv_multiquery_attention call)",
                "avg_launch_ms": round(dec_avg_ms, 5), "launches_timed": DECODE_WINDOW, "timing": window,
                "algorithmic_flops": alg_flops, "algorithmic_bytes": alg_bytes}
    else:
        roof = {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "peak_kind": peak_kind,
                "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                "kernel": ("mq_tc_kernel<128, int8> (one launch per pkv_decode_attention_q8 call)" if q8
                           else "decode_tc_kernel<128> + prefix_umma_kernel<128> (one shared-prefix call)"
                           if two_phase else
                           "mq_tc_kernel<128> (one launch per pkv_multiquery_attention call)" if nq > 1 else
                           "decode_tc_kernel<128> (one launch per pkv_decode_attention call)"),
                "avg_launch_ms": round(dec_avg_ms, 5), "launches_timed": DECODE_WINDOW, "timing": window,
                "algorithmic_bytes": alg_bytes}
    single = res["single_ms"]
    cold_ms = res["cold_ms"]
    return {
        "value": round(value, 2), "ms_per_step": round(ms_per_step, 5),
        "hbm_frac": round(value / peak, 4),
        "unique_kv_gbs": round(unique_kvb * ws / (ms_per_step * 1e-3) / 1e9, 2),
        "kv_tokens_per_s": round(kv_tokens * ws / (ms_per_step * 1e-3), 1),
        "roofline": roof,
        "e2e": {"value": round(total_kv / (res["e2e_s"] / args.steps) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                "note": "wall time of K steps through the public API; every step copies its inputs from pinned "
                        "host memory and its result back; two buffer sets alternate so that those copies run "
                        "on a second stream beside the previous or next step's kernels"},
        "call_us": {"p10": round(1e3 * float(np.percentile(single, 10)), 2),
                    "p50": round(1e3 * float(np.percentile(single, 50)), 2),
                    "p90": round(1e3 * float(np.percentile(single, 90)), 2), "samples": len(single),
                    "note": "each call alone between its own events: includes the ramp that back-to-back calls "
                            "and the step's append hide"},
        "l2_scrubbed": {"step_us_p50": round(1e3 * cold_ms[len(cold_ms) // 2], 2),
                        "kv_gbs": round(total_kv / (cold_ms[len(cold_ms) // 2] * 1e-3) / 1e9, 2),
                        "unique_kv_gbs": round(unique_kvb * ws / (cold_ms[len(cold_ms) // 2] * 1e-3) / 1e9, 2),
                        "note": "256 MiB written before each of 50 event-timed steps"},
        "append_us": round(res["append_us"], 2),
        "copy_us": res["copy_us"],
        "gpu_launches": res["launches_per_step"] * args.steps,
        "device_status": res["status_bits"],
        "config": {"workload": workload_desc(name, cfg, lens_np), "l2": L2_NOTE[name],
                   "step": f"copy_blocks{'_q8' if q8 else ''} ({res['pairs_n']} pairs) + "
                           + f"{'quantizing append' if q8 else 'append'} ({B * nq} tokens) + "
                           + ("decode attention over the int8 cache" if q8
                              else "shared-prefix decode attention (two phases)" if two_phase
                              else f"causal multi-query attention ({nq} queries per sequence)" if nq > 1
                              else "decode attention"),
                   "kernel": ("tcgen05 tile kernel: 128 query rows per tile, S and O in tensor memory, the "
                              "context split over a thread-block cluster combined through distributed shared "
                              "memory" if prefill else
                              "tensor-core split-context kernel on int8 codes (exact in f16), per-row scales "
                              "applied to S and folded into P, merge fused" if q8 else
                              "tensor-core split-context kernel, merge fused"
                              + (", then the chunk-first pass over the shared blocks" if two_phase else ""))},
    }


def cpu_baselines(runner, name, cfg, host):
    """The oracle on one core (one pass over the workload, at most 20 s) and on
    all cores (repeated passes for at least 3 s)."""
    tasks, what = oracle_tasks(runner, name, cfg, host)
    b1, s1, d1 = runner.run(tasks, all_cores=False, max_seconds=20.0)
    one = {"value": round(b1 / s1 / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": f"{d1} of {what} of this workload (one pass, at most 20 s), float64 NumPy oracle, one thread"}
    bn, sn, dn = runner.run(tasks, all_cores=True, min_seconds=3.0)
    allc = {"value": round(bn / sn / 1e9, 4), "unit": "GB/s", "cores": runner.cores, "kind": "oracle",
            "sample": f"{what} of this workload, repeated for at least 3 s ({dn} tasks), float64 NumPy oracle, "
                      f"{runner.cores} single-threaded processes (one per core of os.sched_getaffinity)",
            "blas_threads_per_process": 1}
    return one, allc


def run_pkv(args, cfg):
    import torch
    ws, rank, local = dist_env()
    runner = None
    if rank == 0:
        runner = OracleRunner()
        runner.start_pool()            # spawned workers, before any CUDA call in this process
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    device = torch.device("cuda", torch.cuda.current_device())
    from paged_kv_cache_209_gb300 import pkv
    pkv.load_library()
    also = ALSO_DEFAULT.get(args.workload, []) if args.also is None else \
        [a for a in args.also.split(",") if a and a != "none"]
    gpu_id = str(torch.cuda.get_device_properties(device).uuid)
    gpu_id = gpu_id if gpu_id.startswith("GPU-") else "GPU-" + gpu_id
    sampler = ClockSampler(gpu_id) if rank == 0 else None
    try:
        head, host = measure_workload(args.workload, args, ws, rank, device, args.single_pass, want_host=rank == 0)
        extra = [measure_workload(a, args, ws, rank, device)[0] for a in also]
    finally:
        clocks = sampler.stop() if sampler else None
    if rank != 0:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    try:
        one, allc = cpu_baselines(runner, args.workload, cfg, host)
    finally:
        runner.close()
    s = summarize(head, args, ws)
    line = {
        "metric": METRIC, "value": s["value"], "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": s["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8" if head["q8"] else "bf16", "data": "synthetic",
        "config": s["config"],
    }
    line.update({k: v for k, v in s.items() if k not in ("value", "ms_per_step", "config")})
    line["cpu_baseline"] = one
    line["cpu_baseline_all_cores"] = allc
    line["step_overlap"] = ("ms_per_step can be shorter than call_us: inside a step the decode kernel's launch and "
                            "prologue overlap the append (programmatic dependent launch)")
    if extra:
        line["also"] = {}
        for r in extra:
            e = summarize(r, args, ws)
            line["also"][r["name"]] = {k: e[k] for k in ("value", "ms_per_step", "hbm_frac", "kv_tokens_per_s",
                                                         "roofline", "call_us", "e2e", "l2_scrubbed", "append_us",
                                                         "copy_us", "gpu_launches", "device_status", "config")}
    line["clocks"] = clocks
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["pkv", "reference"], default="pkv")
    ap.add_argument("--workload", choices=sorted(WORKLOAD_NAMES), default=WORKLOAD,
                    help="default: the 8K Llama-3-8B layer the headline metric is quoted on")
    ap.add_argument("--also", default=None,
                    help="comma-separated workloads measured after the main one and nested under 'also' "
                         "(default: long128k after llama8k; 'none' for none)")
    ap.add_argument("--single-pass", action="store_true",
                    help="prefix workload: plain decode over the full tables instead of the shared-prefix call")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    cfg = dict(W.CONFIGS[args.workload])
    if args.impl == "reference":
        run_reference(args, cfg)
    else:
        run_pkv(args, cfg)


if __name__ == "__main__":
    main()
