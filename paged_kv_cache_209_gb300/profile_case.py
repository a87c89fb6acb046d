"""Run decode steps of a named workload, for profiling under ncu.

    python -m paged_kv_cache_209_gb300.profile_case --workload llama8k --steps 5
    python -m paged_kv_cache_209_gb300.profile_case --workload prefix --two-phase --steps 5
    python -m paged_kv_cache_209_gb300.profile_case --workload spec4 --steps 5
    python -m paged_kv_cache_209_gb300.profile_case --workload llama8k_q8 --steps 5

One step is the hot path of the benchmark: block copy (no pairs in these
workloads), slot-mapped append, decode attention (with --two-phase, the
shared-prefix call with the workload's groups; spec4: the causal multi-query
call; llama8k_q8: the quantizing append and attention over the int8 cache).
No timing, no CPU oracle: this only drives the kernels so that a profiler
can capture them.
"""

import argparse

import torch

from paged_kv_cache_209_gb300 import pkv, workloads


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="llama8k", choices=sorted(workloads.CONFIGS))
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--kernel", type=int, default=0)
    ap.add_argument("--prefix-kernel", type=int, default=0)
    ap.add_argument("--two-phase", action="store_true", help="shared-prefix call (prefix workload)")
    args = ap.parse_args()
    torch.cuda.set_device(0)
    w = workloads.device_workload(args.workload, torch.device("cuda", 0))
    out = torch.empty_like(w["q"])
    B, HQ, MAXB = w["q"].shape[0], w["q"].shape[1], w["tables"].shape[1]
    q8 = w["cfg"]["dtype"] == "int8"
    nq = w["queries"]
    if q8:
        need = pkv.pkv_decode_q8_workspace_size(B, HQ, MAXB, w["k_pool"])
    elif nq > 1:
        need = pkv.pkv_multiquery_workspace_size(w["lens"].shape[0], HQ, MAXB, nq, w["k_pool"])
    elif args.two_phase:
        need = pkv.pkv_decode_prefixed_workspace_size(B, HQ, MAXB, len(w["group_blocks"]), w["max_group_blocks"],
                                                      w["k_pool"], kernel=args.kernel,
                                                      prefix_kernel=args.prefix_kernel)
    else:
        need = pkv.pkv_decode_workspace_size(B, HQ, MAXB, w["k_pool"], kernel=args.kernel)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for _ in range(args.steps):
        if q8:
            sc = w["scales"]
            pkv.pkv_copy_blocks_q8(w["pairs"], w["k_pool"], w["v_pool"], sc)
            pkv.pkv_append_q8(w["k_new"], w["v_new"], w["slots"], w["k_pool"], w["v_pool"], sc)
            pkv.pkv_decode_attention_q8(w["q"], w["k_pool"], w["v_pool"], sc, w["tables"], w["lens"], w["scale"],
                                        out=out, workspace=ws)
            continue
        pkv.pkv_copy_blocks(w["pairs"], w["k_pool"], w["v_pool"])
        pkv.pkv_append(w["k_new"], w["v_new"], w["slots"], w["k_pool"], w["v_pool"])
        if nq > 1:
            pkv.pkv_multiquery_attention(w["q"], w["k_pool"], w["v_pool"], w["tables"], w["lens"], w["query_start"],
                                         w["scale"], nq, out=out, workspace=ws)
        elif args.two_phase:
            pkv.pkv_decode_attention_prefixed(w["q"], w["k_pool"], w["v_pool"], w["tables"], w["lens"], w["scale"],
                                              w["prefix_group"], w["group_blocks"], w["max_group_blocks"], out=out,
                                              workspace=ws, kernel=args.kernel, prefix_kernel=args.prefix_kernel)
        else:
            pkv.pkv_decode_attention(w["q"], w["k_pool"], w["v_pool"], w["tables"], w["lens"], w["scale"], out=out,
                                     workspace=ws, kernel=args.kernel)
    torch.cuda.synchronize()
    bits = pkv.pkv_device_status()
    if bits:
        raise SystemExit(f"device status {bits}")
    print(f"{args.workload}: {args.steps} steps ok")


if __name__ == "__main__":
    main()
