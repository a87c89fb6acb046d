"""Benchmark of the paged decode path on GB300 (prints one JSON line).

Workload (default): one Llama-3-8B decode layer -- batch 32, 32 query / 8 KV
heads, head_dim 128, bf16, every context 8192 tokens in 16-token blocks,
block tables a random permutation of a 16384-block pool (1 GiB of K+V, more
than the 129 MB L2, so no flush is needed between steps).

One step = the whole hot path for one decode token per sequence:
  pkv_copy_blocks (this workload shares no blocks: zero pairs, no launch)
  -> pkv_append (each sequence's new K/V at position 8191)
  -> pkv_decode_attention (one launch: split kernel with the merge fused).
value = KV bytes read per step / device time per step (decimal GB/s).

--workload prefix runs the shared-prefix call by default
(pkv_decode_attention_prefixed: every sequence in one group over the 256
shared blocks); --single-pass times pkv_decode_attention over the same tables.
There value counts the K/V bytes attended (logical); unique_kv_gbs counts each
stored byte once.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl pkv|reference]
                  [--workload NAME] [--single-pass]

--impl reference times the float64 CPU oracle (the only other code here),
on a bounded sample of the same workload per step. Under torchrun with
N > 1 every rank runs its own replica of the workload on its own GPU (weak
scaling, no collective on the data path); timing is the max over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

# The CPU oracle baseline runs on one thread (BLAS included), as its line states.
for _var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ[_var] = "1"

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_209_gb300 import workloads as W  # noqa: E402

METRIC = "paged decode attention KV GB/s (% of GB300 HBM peak) and KV tokens/s, 1 GPU"
WORKLOAD = "llama8k"
FALLBACK_HBM_GBS = 6800.0


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
    """nvidia-smi sampling of SM clocks and throttle reasons during a window."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.proc = None
        self.path = os.path.join("/tmp", f"pkv_clocks_{os.getpid()}.csv")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", gpu_id, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ peaks and profiles
def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        return float(json.load(open(p))["hbm_gbs"]), "measured"
    except Exception:
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
def oracle_sample_rate(q, kp, vp, tables, lens, scale, kv_heads, pairs, time_budget_s=None, nq=1, q_sample=None):
    """Run the float64 oracle on (seq, kv_head) pairs; returns (bytes, seconds, pairs done).
    With nq > 1 queries per sequence (rows i*nq .. i*nq+nq-1 of q), the
    multi-query oracle runs on whole sequences (all KV heads) instead; with
    q_sample, on the last q_sample queries of each (they see the same tokens as
    in the full call), credited with that fraction of the sequence's bytes."""
    from oracle import attention as OA
    from oracle import multiquery as OM
    done, nbytes = 0, 0
    t0 = time.perf_counter()
    for (i, j) in pairs:
        if nq > 1:
            if j:
                continue
            ns = nq if q_sample is None else min(q_sample, nq)
            OM.multiquery_attention(q[(i + 1) * nq - ns:(i + 1) * nq], kp, vp, tables[i:i + 1], lens[i:i + 1],
                                    np.array([0, ns]), scale, kv_heads, "bf16")
            nbytes += int(lens[i]) * 2 * kv_heads * kp.shape[-1] * 2 * ns // nq
        else:
            OA.decode_attention_pair(q, kp, vp, tables, lens, scale, i, j, kv_heads, "bf16")
            nbytes += int(lens[i]) * 2 * kp.shape[-1] * 2
        done += 1
        if time_budget_s is not None and time.perf_counter() - t0 > time_budget_s:
            break
    return nbytes, time.perf_counter() - t0, done


def oracle_sample_rate_q8(q, kc, vc, ks, vs, tables, lens, scale, kv_heads, time_budget_s=None):
    """The int8-cache oracle on whole sequences (all KV heads), one at a time;
    returns (bytes, seconds, sequences done). ``vc`` is in the oracle's
    token-row layout."""
    from oracle import quant as OQ
    done, nbytes = 0, 0
    t0 = time.perf_counter()
    for i in range(len(lens)):
        OQ.decode_attention_q8(q[i:i + 1], kc, vc, ks, vs, tables[i:i + 1], lens[i:i + 1], scale, kv_heads, "bf16")
        nbytes += int(lens[i]) * 2 * kv_heads * (kc.shape[-1] + 4)
        done += 1
        if time_budget_s is not None and time.perf_counter() - t0 > time_budget_s:
            break
    return nbytes, time.perf_counter() - t0, done


def cpu_sample_data_q8(w, q, tables_np, lens_np, seqs):
    """Host copies of the sampled sequences' int8 blocks (V codes turned to token rows)."""
    import torch
    ids = np.unique(tables_np[seqs].reshape(-1))
    ids = ids[ids >= 0]
    remap = -np.ones(w["k_pool"].shape[0], dtype=np.int64)
    remap[ids] = np.arange(len(ids))
    idx = torch.from_numpy(ids).to(q.device)
    kc = w["k_pool"].index_select(0, idx).cpu().numpy()
    vc = np.ascontiguousarray(w["v_pool"].index_select(0, idx).cpu().numpy().transpose(0, 1, 3, 2))
    ks = w["k_scales"].index_select(0, idx).cpu().numpy()
    vs = w["v_scales"].index_select(0, idx).cpu().numpy()
    qh = q[torch.tensor(seqs, device=q.device)].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    t = tables_np[seqs]
    t = np.where(t >= 0, remap[np.maximum(t, 0)], -1)
    return qh, kc, vc, ks, vs, t, lens_np[seqs]


def cpu_sample_data(k_pool, v_pool, q, tables_np, lens_np, seqs, nq=1):
    import torch
    ids = np.unique(tables_np[seqs].reshape(-1))
    ids = ids[ids >= 0]
    remap = -np.ones(k_pool.shape[0], dtype=np.int64)
    remap[ids] = np.arange(len(ids))
    idx = torch.from_numpy(ids).to(k_pool.device)
    kp = k_pool.index_select(0, idx).view(torch.int16).cpu().numpy().view(np.uint16)
    vp = v_pool.index_select(0, idx).view(torch.int16).cpu().numpy().view(np.uint16)
    rows = np.concatenate([np.arange(s * nq, (s + 1) * nq) for s in seqs])
    qh = q[torch.from_numpy(rows).to(q.device)].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    t = tables_np[seqs]
    t = np.where(t >= 0, remap[np.maximum(t, 0)], -1)
    return qh, kp, vp, t, lens_np[seqs]


def run_reference(args, cfg):
    """--impl reference: the CPU oracle, timed per step on a bounded sample:
    one (sequence, KV head) of the workload's longest sequence."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import torch
    tables_all, lens_all, _ = W.workload_index(args.workload)
    i0 = int(np.argmax(lens_all))
    lens = lens_all[i0:i0 + 1].astype(np.int32)
    n_used = int((lens[0] + 15) // 16)
    ids = tables_all[i0, :n_used]
    # Only the sampled sequence's blocks are materialised (on the host).
    g = torch.Generator().manual_seed(cfg["seed"])
    shape = (n_used, cfg["kv_heads"], 16, cfg["head_dim"])
    kp = torch.randn(shape, generator=g).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    vp = torch.randn(shape, generator=g).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    q = torch.randn((1, cfg["q_heads"], cfg["head_dim"]), generator=g).to(torch.bfloat16)
    q = q.view(torch.int16).numpy().view(np.uint16)
    t = np.arange(n_used, dtype=np.int64)[None, :]   # block j of the sample sits at index j of the sub-pool
    assert len(np.unique(ids)) == n_used
    scale = 1.0 / np.sqrt(cfg["head_dim"])
    pairs = [(0, 0)]
    if cfg["dtype"] == "int8":
        # int8 codes and float32 scales of the sampled sequence's blocks (token-row layout)
        rng = np.random.default_rng(cfg["seed"])
        qshape = shape[:3]
        kc = np.clip(np.rint(rng.standard_normal(shape) * 42), -127, 127).astype(np.int8)
        vc = np.clip(np.rint(rng.standard_normal(shape) * 42), -127, 127).astype(np.int8)
        ks = rng.uniform(0.02, 0.03, qshape).astype(np.float32)
        vs = rng.uniform(0.02, 0.03, qshape).astype(np.float32)

        def one_step():
            return oracle_sample_rate_q8(q, kc, vc, ks, vs, t, lens, scale, cfg["kv_heads"])[:2]
        what = f"1 sequence x {cfg['kv_heads']} KV heads ({int(lens[0])} tokens, int8 K+V codes, float32 scales)"
    else:
        def one_step():
            return oracle_sample_rate(q, kp, vp, t, lens, scale, cfg["kv_heads"], pairs)[:2]
        what = f"1 sequence x 1 KV head ({int(lens[0])} tokens, bf16 K+V)"
    for _ in range(args.warmup):
        one_step()
    tot_b, tot_s = 0, 0.0
    for _ in range(args.steps):
        b, s_ = one_step()
        tot_b += b
        tot_s += s_
    gbs = tot_b / tot_s / 1e9
    sample = f"{what} per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_s / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(args.workload, cfg, lens_all), "sample": sample},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "kv_tokens_per_s": round(tot_b / kv_bytes_per_token(cfg) / tot_s, 1),
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm
def run_pkv(args, cfg):
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    device = torch.device("cuda", torch.cuda.current_device())
    from paged_kv_cache_209_gb300 import pkv
    pkv.load_library()

    w = W.device_workload(args.workload, device, seed_offset=1000 * rank)
    B, HQ, HKV, D = cfg["batch"], cfg["q_heads"], cfg["kv_heads"], cfg["head_dim"]
    k_pool, v_pool, q, kn, vn = w["k_pool"], w["v_pool"], w["q"], w["k_new"], w["v_new"]
    tables, lens, slots, pairs = w["tables"], w["lens"], w["slots"], w["pairs"]
    tables_np, lens_np = w["tables_np"], w["lens_np"]
    MAXB = tables.shape[1]
    out = torch.empty_like(q)
    two_phase = args.workload == "prefix" and not args.single_pass
    q8 = cfg["dtype"] == "int8"
    nq = w["queries"]
    qstart = w["query_start"]
    group, gblocks, mgb = w["prefix_group"], w["group_blocks"], w["max_group_blocks"]
    if q8:
        ks_pool, vs_pool = w["k_scales"], w["v_scales"]
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
            pkv.pkv_decode_attention_q8(q, k_pool, v_pool, ks_pool, vs_pool, tables, lens, scale, out=out,
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

    def copy_and_append():
        if q8:
            pkv.pkv_copy_blocks_q8(pairs, k_pool, v_pool, ks_pool, vs_pool, stream=stream)
            pkv.pkv_append_q8(kn, vn, slots, k_pool, v_pool, ks_pool, vs_pool, stream=stream)
        else:
            pkv.pkv_copy_blocks(pairs, k_pool, v_pool, stream=stream)
            pkv.pkv_append(kn, vn, slots, k_pool, v_pool, stream=stream)

    def step():
        copy_and_append()
        decode()

    # append + per 1024 sequences one decode launch (two with the shared-prefix pass)
    launches_per_step = 1 + (2 if two_phase else 1) * ((B + 1023) // 1024)
    gpu_id = str(torch.cuda.get_device_properties(device).uuid)
    gpu_id = gpu_id if gpu_id.startswith("GPU-") else "GPU-" + gpu_id
    sampler = ClockSampler(gpu_id) if rank == 0 else None
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # -------- device-timed region: K whole steps. The decode call of every
    # 8th step is bracketed by events for the kernel's own duration (an event
    # between append and decode breaks their launch overlap, so only a sample
    # of the steps carries them).
    sample_every = 8
    sampled = list(range(0, args.steps, sample_every))
    ev_dec = {i: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for i in sampled}
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(args.steps):
        copy_and_append()
        ev = ev_dec.get(i)
        if ev:
            ev[0].record(stream)
        decode()
        if ev:
            ev[1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clocks = sampler.stop() if sampler else None
    ms_total = max_over_ranks(start.elapsed_time(end), ws, device)
    dec_ms = [e0.elapsed_time(e1) for e0, e1 in ev_dec.values()]
    dec_avg_ms = max_over_ranks(sum(dec_ms) / len(dec_ms), ws, device)
    status_bits = pkv.pkv_device_status(clear=False)

    # -------- end-to-end: per-step inputs from pinned host memory, result back to the host.
    # The step's inputs live in one pinned host buffer and one device buffer
    # (256-byte aligned slices), so a step costs one host-to-device copy, the
    # kernels (which read the device slices) and one device-to-host copy.
    names = ["q", "kn", "vn", "slots", "tables", "lens"] + (["group", "gblocks"] if two_phase else []) \
        + (["qstart"] if nq > 1 else [])
    srcs = {"q": q, "kn": kn, "vn": vn, "slots": slots, "tables": tables, "lens": lens, "group": group,
            "gblocks": gblocks, "qstart": qstart}
    offs, total = {}, 0
    for n in names:
        offs[n] = total
        total += (srcs[n].numel() * srcs[n].element_size() + 255) // 256 * 256
    pack_dev = torch.zeros(total, dtype=torch.uint8, device=device)
    pack_host = torch.zeros(total, dtype=torch.uint8).pin_memory()
    views = {}
    for n in names:
        t = srcs[n]
        nb = t.numel() * t.element_size()
        views[n] = pack_dev[offs[n]:offs[n] + nb].view(t.dtype).view(t.shape)
        views[n].copy_(t)
        pack_host[offs[n]:offs[n] + nb].copy_(t.reshape(-1).view(torch.uint8).cpu())
    q, kn, vn, slots, tables, lens = (views[n] for n in ["q", "kn", "vn", "slots", "tables", "lens"])
    if two_phase:
        group, gblocks = views["group"], views["gblocks"]
    if nq > 1:
        qstart = views["qstart"]
    out_pin = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = total
    d2h = out_pin.numel() * out_pin.element_size()

    def e2e_step():
        pack_dev.copy_(pack_host, non_blocking=True)
        step()
        out_pin.copy_(out, non_blocking=True)

    for _ in range(max(3, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    barrier(ws)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, ws, device)
    barrier(ws)

    # -------- cold L2: a 256 MiB buffer (twice the L2) is written before each
    # step, and the step alone is event-timed (50 steps)
    scrub = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=device)
    cold_ms = []
    for _ in range(50):
        scrub.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        cold_ms.append((e0, e1))
    torch.cuda.synchronize()
    cold_ms = sorted(a0.elapsed_time(a1) for a0, a1 in cold_ms)
    del scrub

    if rank != 0:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    kv_tokens = int(lens_np.sum())
    tok_bytes = kv_bytes_per_token(cfg)
    kvb = kv_tokens * tok_bytes
    total_kv = kvb * ws
    ms_per_step = ms_total / args.steps
    value = total_kv / (ms_per_step * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()
    # algorithmic bytes of one decode call: K+V of every live token read once,
    # q read, out written, block-table entries and lengths read. With the
    # shared-prefix pass the shared blocks count once (the bytes a perfect
    # kernel must move), not once per sequence.
    used_entries = int(((lens_np.astype(np.int64) + 15) // 16).sum())
    shared_tokens = int(mgb) * 16 * (B - 1) if two_phase else 0
    unique_kvb = (kv_tokens - shared_tokens) * tok_bytes
    alg_bytes = unique_kvb + q.numel() * q.element_size() + out.numel() * out.element_size() + used_entries * 4 + B * 4
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
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
            os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
        t_peak = float(peaks.get("bf16_tflops", 1900.0))
        t_kind = "measured (cuBLAS bf16 burst)" if "bf16_tflops" in peaks else "fallback"
    if prefill:
        traffic = profiled_traffic(f"decode_{args.workload}", ("pkv_prefix.cu",))
    elif two_phase:
        traffic = profiled_traffic("decode_prefix_two_phase", ("pkv_decode.cu", "pkv_prefix.cu"))
    elif q8 or nq > 1:
        traffic = profiled_traffic(f"decode_{args.workload}", ("pkv_multiquery.cu",))
    else:
        traffic = profiled_traffic(f"decode_{args.workload}")

    # -------- CPU oracle baseline on a bounded sample of the same workload
    order = np.argsort(-lens_np)
    sample_seqs = sorted({int(order[0]), int(order[len(order) // 2])})
    if q8:
        qh, kch, vch, ksh, vsh, th, lh = cpu_sample_data_q8(w, q, tables_np, lens_np, sample_seqs)
        cb, cs, cdone = oracle_sample_rate_q8(qh, kch, vch, ksh, vsh, th, lh, scale, HKV, time_budget_s=20.0)
        cpu_what = f"{cdone} whole sequences of {sample_seqs} (int8 cache, all KV heads), "
    else:
        qh, kph, vph, th, lh = cpu_sample_data(k_pool, v_pool, q, tables_np, lens_np, sample_seqs, nq)
        pairs_list = [(i, j) for i in range(len(sample_seqs)) for j in range(HKV)]
        qsamp = 8 if prefill else None
        cb, cs, cdone = oracle_sample_rate(qh, kph, vph, th, lh, scale, HKV, pairs_list, time_budget_s=20.0, nq=nq,
                                           q_sample=qsamp)
        cpu_what = (f"{cdone} (sequence, KV head) pairs of sequences {sample_seqs}, " if nq == 1
                    else f"the last {qsamp} of the {nq} queries of {cdone} sequences of {sample_seqs} "
                         "(bytes credited in proportion), " if prefill
                    else f"{cdone} whole sequences of {sample_seqs} ({nq} queries each), ")
    cpu_gbs = cb / cs / 1e9

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8" if q8 else "bf16",
        "data": "synthetic",
        "config": {"workload": workload_desc(args.workload, cfg, lens_np),
                   "l2": L2_NOTE[args.workload],
                   "step": f"copy_blocks{'_q8' if q8 else ''} ({int(pairs.shape[0])} pairs) + "
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
        "hbm_frac": round(value / peak, 4),
        "unique_kv_gbs": round(unique_kvb * ws / (ms_per_step * 1e-3) / 1e9, 2),
        "kv_tokens_per_s": round(kv_tokens * ws / (ms_per_step * 1e-3), 1),
        "roofline": ({"bound": "tensor", "achieved": round(tflops, 2), "peak": t_peak, "peak_kind": t_kind,
                      "unit": "TFLOP/s", "frac": round(tflops / t_peak, 4), "traffic": traffic,
                      "kernel": "prefix_umma_kernel<128, prefill> (one launch per pkv_multiquery_attention call)",
                      "avg_launch_ms": round(dec_avg_ms, 5), "launches_timed": len(dec_ms),
                      "algorithmic_flops": alg_flops, "algorithmic_bytes": alg_bytes} if prefill else
                     {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": ("mq_tc_kernel<128, int8> (one launch per pkv_decode_attention_q8 call)" if q8
                                else "decode_tc_kernel<128> + prefix_umma_kernel<128> (one shared-prefix call)"
                                if two_phase else
                                "mq_tc_kernel<128> (one launch per pkv_multiquery_attention call)" if nq > 1 else
                                "decode_tc_kernel<128> (one launch per pkv_decode_attention call)"),
                     "avg_launch_ms": round(dec_avg_ms, 5), "launches_timed": len(dec_ms),
                     "algorithmic_bytes": alg_bytes}),
        "cpu_baseline": {"value": round(cpu_gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": cpu_what + "float64 NumPy oracle, one thread"},
        "e2e": {"value": round(total_kv / (e2e_s / args.steps) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "call_us": {"p10": round(1e3 * float(np.percentile(dec_ms, 10)), 2),
                    "p50": round(1e3 * float(np.percentile(dec_ms, 50)), 2),
                    "p90": round(1e3 * float(np.percentile(dec_ms, 90)), 2), "samples": len(dec_ms)},
        "l2_scrubbed": {"step_us_p50": round(1e3 * cold_ms[len(cold_ms) // 2], 2),
                        "kv_gbs": round(total_kv / (cold_ms[len(cold_ms) // 2] * 1e-3) / 1e9, 2),
                        "unique_kv_gbs": round(unique_kvb * ws / (cold_ms[len(cold_ms) // 2] * 1e-3) / 1e9, 2),
                        "note": "256 MiB written before each of 50 event-timed steps"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "device_status": status_bits,
    }
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
