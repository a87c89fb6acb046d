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

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl pkv|reference]

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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_209_gb300 import workloads as W  # noqa: E402

METRIC = "paged decode attention KV GB/s (% of GB300 HBM peak) and KV tokens/s, 1 GPU"
WORKLOAD = "llama8k"
FALLBACK_HBM_GBS = 6800.0


def workload_desc(cfg):
    return (f"Llama-3-8B decode layer: batch {cfg['batch']}, {cfg['q_heads']} q / {cfg['kv_heads']} kv heads, "
            f"head_dim {cfg['head_dim']}, context {cfg['context']} tokens, 16-token blocks, "
            f"{cfg['num_blocks']}-block shuffled pool, bf16")


def kv_bytes_per_step(cfg):
    return cfg["batch"] * cfg["context"] * 2 * cfg["kv_heads"] * cfg["head_dim"] * 2


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


def kernel_source_sha():
    src = os.path.join(ROOT, "paged_kv_cache_209_gb300", "csrc", "pkv_decode.cu")
    return hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "decode_llama8k.md")
    if not os.path.exists(p):
        return None
    text = open(p).read()
    m_sha = re.search(r"source_sha:\s*([0-9a-f]+)", text)
    m_tr = re.search(r"dram_bytes_per_call:\s*([0-9]+)", text)
    if not m_sha or not m_tr or m_sha.group(1) != kernel_source_sha():
        return None
    return int(m_tr.group(1))


# ------------------------------------------------------------------ CPU oracle baseline
def oracle_sample_rate(q, kp, vp, tables, lens, scale, kv_heads, pairs, time_budget_s=None):
    """Run the float64 oracle on (seq, kv_head) pairs; returns (bytes, seconds, pairs done)."""
    from oracle import attention as OA
    done, nbytes = 0, 0
    t0 = time.perf_counter()
    for (i, j) in pairs:
        OA.decode_attention_pair(q, kp, vp, tables, lens, scale, i, j, kv_heads, "bf16")
        nbytes += int(lens[i]) * 2 * kp.shape[-1] * 2
        done += 1
        if time_budget_s is not None and time.perf_counter() - t0 > time_budget_s:
            break
    return nbytes, time.perf_counter() - t0, done


def cpu_sample_data(k_pool, v_pool, q, tables_np, lens_np, seqs):
    import torch
    ids = np.unique(tables_np[seqs].reshape(-1))
    ids = ids[ids >= 0]
    remap = -np.ones(k_pool.shape[0], dtype=np.int64)
    remap[ids] = np.arange(len(ids))
    idx = torch.from_numpy(ids).to(k_pool.device)
    kp = k_pool.index_select(0, idx).view(torch.int16).cpu().numpy().view(np.uint16)
    vp = v_pool.index_select(0, idx).view(torch.int16).cpu().numpy().view(np.uint16)
    qh = q[seqs].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    t = tables_np[seqs]
    t = np.where(t >= 0, remap[np.maximum(t, 0)], -1)
    return qh, kp, vp, t, lens_np[seqs]


def run_reference(args, cfg):
    """--impl reference: the CPU oracle, timed per step on a bounded sample."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import torch
    rng_seqs = [0]
    tables = W.permuted_tables(cfg["num_blocks"], cfg["batch"], cfg["context"] // 16, cfg["seed"])
    lens = np.full(cfg["batch"], cfg["context"], dtype=np.int32)
    # Only the sampled sequences' blocks are materialised (on the host).
    ids = np.unique(tables[rng_seqs].reshape(-1))
    remap = -np.ones(cfg["num_blocks"], dtype=np.int64)
    remap[ids] = np.arange(len(ids))
    g = torch.Generator().manual_seed(cfg["seed"])
    shape = (len(ids), cfg["kv_heads"], 16, cfg["head_dim"])
    kp = torch.randn(shape, generator=g).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    vp = torch.randn(shape, generator=g).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    q = torch.randn((1, cfg["q_heads"], cfg["head_dim"]), generator=g).to(torch.bfloat16)
    q = q.view(torch.int16).numpy().view(np.uint16)
    t = remap[tables[rng_seqs]]
    scale = 1.0 / np.sqrt(cfg["head_dim"])
    pairs = [(0, 0)]  # one (sequence, KV head): 8192 tokens, 4 MiB of K+V per step
    for _ in range(args.warmup):
        oracle_sample_rate(q, kp, vp, t, lens[:1], scale, cfg["kv_heads"], pairs)
    tot_b, tot_s = 0, 0.0
    for _ in range(args.steps):
        b, s, _ = oracle_sample_rate(q, kp, vp, t, lens[:1], scale, cfg["kv_heads"], pairs)
        tot_b += b
        tot_s += s
    gbs = tot_b / tot_s / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_s / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(cfg), "sample": "1 sequence x 1 KV head (8192 tokens) per step"},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": "1 sequence x 1 KV head (8192 tokens, 4 MiB of bf16 K+V) per step"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "kv_tokens_per_s": round(tot_b / (2 * cfg["kv_heads"] * cfg["head_dim"] * 2) / tot_s, 1),
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

    B, HQ, HKV, D = cfg["batch"], cfg["q_heads"], cfg["kv_heads"], cfg["head_dim"]
    NB, CTX = cfg["num_blocks"], cfg["context"]
    MAXB = CTX // 16
    seed = cfg["seed"] + 1000 * rank
    bf = torch.bfloat16
    k_pool = W.torch_normal((NB, HKV, 16, D), seed, bf, device)
    v_pool = W.torch_normal((NB, HKV, 16, D), seed + 1, bf, device)
    q_host = W.torch_normal((B, HQ, D), seed + 2, bf, "cpu")
    kn_host = W.torch_normal((B, HKV, D), seed + 3, bf, "cpu")
    vn_host = W.torch_normal((B, HKV, D), seed + 4, bf, "cpu")
    tables_np = W.permuted_tables(NB, B, MAXB, cfg["seed"])
    lens_np = np.full(B, CTX, dtype=np.int32)
    slots_np = W.slot_of(tables_np, lens_np.astype(np.int64) - 1)
    q = q_host.to(device)
    kn, vn = kn_host.to(device), vn_host.to(device)
    tables = torch.from_numpy(tables_np).to(device)
    lens = torch.from_numpy(lens_np).to(device)
    slots = torch.from_numpy(slots_np).to(device)
    pairs = torch.zeros((0, 2), dtype=torch.int64, device=device)
    out = torch.empty((B, HQ, D), dtype=bf, device=device)
    ws_bytes = pkv.pkv_decode_workspace_size(B, HQ, MAXB, k_pool)
    workspace = torch.zeros(ws_bytes, dtype=torch.uint8, device=device)
    scale = 1.0 / float(np.sqrt(D))
    stream = torch.cuda.current_stream()

    def step():
        pkv.pkv_copy_blocks(pairs, k_pool, v_pool, stream=stream)
        pkv.pkv_append(kn, vn, slots, k_pool, v_pool, stream=stream)
        pkv.pkv_decode_attention(q, k_pool, v_pool, tables, lens, scale, out=out, workspace=workspace,
                                 stream=stream)

    launches_per_step = 1 + (B + 1023) // 1024  # append + one decode launch per 1024 sequences
    gpu_id = str(torch.cuda.get_device_properties(device).uuid)
    gpu_id = gpu_id if gpu_id.startswith("GPU-") else "GPU-" + gpu_id
    sampler = ClockSampler(gpu_id) if rank == 0 else None
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # -------- device-timed region: K whole steps, events around each decode call
    ev_dec = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(args.steps):
        pkv.pkv_copy_blocks(pairs, k_pool, v_pool, stream=stream)
        pkv.pkv_append(kn, vn, slots, k_pool, v_pool, stream=stream)
        ev_dec[i][0].record(stream)
        pkv.pkv_decode_attention(q, k_pool, v_pool, tables, lens, scale, out=out, workspace=workspace,
                                 stream=stream)
        ev_dec[i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clocks = sampler.stop() if sampler else None
    ms_total = max_over_ranks(start.elapsed_time(end), ws, device)
    dec_ms = [a.elapsed_time(b) for a, b in ev_dec]
    dec_avg_ms = max_over_ranks(sum(dec_ms) / len(dec_ms), ws, device)
    status_bits = pkv.pkv_device_status(clear=False)

    # -------- end-to-end: per-step inputs from pinned host memory, result back to the host
    q_pin = q_host.pin_memory()
    kn_pin, vn_pin = kn_host.pin_memory(), vn_host.pin_memory()
    slots_pin = torch.from_numpy(slots_np).pin_memory()
    tables_pin = torch.from_numpy(tables_np).pin_memory()
    lens_pin = torch.from_numpy(lens_np).pin_memory()
    out_pin = torch.empty((B, HQ, D), dtype=bf).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (q_pin, kn_pin, vn_pin, slots_pin, tables_pin, lens_pin))
    d2h = out_pin.numel() * out_pin.element_size()

    def e2e_step():
        q.copy_(q_pin, non_blocking=True)
        kn.copy_(kn_pin, non_blocking=True)
        vn.copy_(vn_pin, non_blocking=True)
        slots.copy_(slots_pin, non_blocking=True)
        tables.copy_(tables_pin, non_blocking=True)
        lens.copy_(lens_pin, non_blocking=True)
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

    if rank != 0:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    kvb = kv_bytes_per_step(cfg)
    total_kv = kvb * ws
    ms_per_step = ms_total / args.steps
    value = total_kv / (ms_per_step * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()
    # algorithmic bytes of one decode call: K+V read, q read, out written,
    # block tables and lengths read, split pieces written and read back
    alg_bytes = kvb + q.numel() * 2 + out.numel() * 2 + tables.numel() * 4 + lens.numel() * 4
    achieved = alg_bytes / (dec_avg_ms * 1e-3) / 1e9
    traffic = profiled_traffic()

    # -------- CPU oracle baseline on a bounded sample of the same workload
    sample_seqs = [0, 1]
    qh, kph, vph, th, lh = cpu_sample_data(k_pool, v_pool, q, tables_np, lens_np, sample_seqs)
    pairs_list = [(i, j) for i in range(len(sample_seqs)) for j in range(HKV)]
    cb, cs, cdone = oracle_sample_rate(qh, kph, vph, th, lh, scale, HKV, pairs_list, time_budget_s=20.0)
    cpu_gbs = cb / cs / 1e9

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(cfg), "l2": "inputs larger than L2 (1 GiB K+V per step)",
                   "step": "copy_blocks (0 pairs) + append (32 tokens) + decode attention",
                   "kernel": "tensor-core split-context kernel, merge fused"},
        "hbm_frac": round(value / peak, 4),
        "kv_tokens_per_s": round(cfg["batch"] * cfg["context"] * ws / (ms_per_step * 1e-3), 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": "decode_tc_kernel<128> (one launch per pkv_decode_attention call)",
                     "avg_launch_ms": round(dec_avg_ms, 5), "algorithmic_bytes": alg_bytes},
        "cpu_baseline": {"value": round(cpu_gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{cdone} (sequence, KV head) pairs of 8192 tokens, float64 NumPy oracle"},
        "e2e": {"value": round(total_kv / (e2e_s / args.steps) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
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
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    cfg = dict(W.CONFIGS[WORKLOAD])
    if args.impl == "reference":
        run_reference(args, cfg)
    else:
        run_pkv(args, cfg)


if __name__ == "__main__":
    main()
