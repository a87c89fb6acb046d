"""Full-size parity on the four bf16 workloads, in the benchmark's launch
configuration (default kernel choice and CTA count).

One decode step runs on the GPU (block copy, append, attention). The step's
slots and copy pairs come from the oracle's page pool, which rebuilds each
workload's state from its tables (and must reach exactly those tables). The
append is checked bit-exactly over both whole pools against the oracle's
append on a host copy; attention is checked over every output row against
the float64 oracle (max-abs and relative L2 over the whole output, and each
(sequence, KV head) pair within the max-abs bar), and again against the
independent CUDA-core kernel.
"""

import numpy as np
import pytest
import torch

import cases
from oracle import attention as OA
from oracle import kv_ops as OK
from oracle.paged_pool import PagedKVPool
from paged_kv_cache_209_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2 = 1e-2, 2e-3


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_209_gb300 import pkv as P
    P.load_library()
    return P


def run_step(pkv, w, kernel=0):
    pkv.pkv_copy_blocks(w["pairs"], w["k_pool"], w["v_pool"])
    pkv.pkv_append(w["k_new"], w["v_new"], w["slots"], w["k_pool"], w["v_pool"])
    return pkv.pkv_decode_attention(w["q"], w["k_pool"], w["v_pool"], w["tables"], w["lens"], w["scale"],
                                    kernel=kernel)


def oracle_step_indices(w):
    """Slots and copy pairs of the workload's step from the oracle's page pool;
    they must equal the ones the workload (and the benchmark) uses."""
    cfg = w["cfg"]
    slots, pairs = cases.simulate_workload_step(w["tables_np"], w["lens_np"], w["queries"], w["num_blocks"],
                                                cfg.get("prefix", 0) // 16)
    assert np.array_equal(slots, w["slots_np"]), "workload slots differ from the page pool's"
    assert np.array_equal(pairs, w["pairs"].cpu().numpy().reshape(-1, 2))
    return slots, pairs


def check_all_rows(name, out, want, rows_per_pair):
    """Every output row against the float64 oracle: max-abs and relative L2
    over the whole output, and max-abs per (row group) pair. Prints the worst."""
    got = out.detach().float().cpu().numpy().astype(np.float64)
    assert got.shape == want.shape
    ma, rl = cases.attention_errors(out, want)
    diff = np.abs(got - want).reshape(-1, rows_per_pair * want.shape[-1])
    worst_pair = float(diff.max(axis=1).max())
    print(f"{name}: {want.shape[0] * want.shape[1]} rows against the float64 oracle: max_abs={ma:.3e} "
          f"rel_l2={rl:.3e} worst pair max_abs={worst_pair:.3e}")
    assert ma <= MAX_ABS and rl <= REL_L2, (name, ma, rl)
    assert np.isfinite(got).all()


def check_workload(pkv, w, name, indices=None):
    kv_heads = w["cfg"]["kv_heads"]
    G = w["cfg"]["q_heads"] // kv_heads
    slots, pairs = indices if indices is not None else oracle_step_indices(w)
    hk, hv = cases.host_view(w["k_pool"]), cases.host_view(w["v_pool"])
    OK.copy_blocks(hk, hv, pairs)
    OK.append_tokens(hk, hv, cases.host_view(w["k_new"]), cases.host_view(w["v_new"]), slots)
    out = run_step(pkv, w)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status(clear=True) == 0
    assert np.array_equal(cases.host_view(w["k_pool"]), hk), "K pool differs after copy + append"
    assert np.array_equal(cases.host_view(w["v_pool"]), hv), "V pool differs after copy + append"
    want = OA.decode_attention(cases.host_view(w["q"]), hk, hv, w["tables_np"], w["lens_np"], w["scale"], kv_heads,
                               "bf16")
    check_all_rows(name, out, want, G)
    # every row against the CUDA-core kernel as well (a second implementation)
    ref = pkv.pkv_decode_attention(w["q"], w["k_pool"], w["v_pool"], w["tables"], w["lens"], w["scale"], kernel=1)
    d = (out.float() - ref.float())
    rel_all = (d.norm() / ref.float().norm()).item()
    assert rel_all <= 2e-3 and d.abs().max().item() <= 1e-2, rel_all


@pytest.mark.parametrize("name", ["llama8k", "long128k", "mixed", "prefix"])
def test_full_size_workload(pkv, name):
    w = W.device_workload(name, torch.device("cuda", 0))
    check_workload(pkv, w, name)
    del w
    torch.cuda.empty_cache()


def test_prefix_with_copy_on_write_pairs(pkv):
    """Prefix workload where odd sequence 2i+1 shares all of sequence 2i, so
    their partial last block is shared; the step's appends (index order)
    produce up to 32 copy-on-write pairs through the page-pool simulator."""
    cfg = W.CONFIGS["prefix"]
    suffix = W.uniform_suffixes(cfg["batch"], cfg["min_suffix"], cfg["max_suffix"], cfg["seed"])
    n_prefix_blocks = cfg["prefix"] // 16
    total = n_prefix_blocks + int(sum(W.blocks_needed(suffix[0::2]))) + cfg["batch"] + 8
    pool = PagedKVPool(total, 16, pop_order=np.random.default_rng(41).permutation(total))
    pool.create("root")
    pool.append("root", cfg["prefix"])
    for i in range(0, cfg["batch"], 2):
        pool.share_prefix("root", i, cfg["prefix"])
        pool.append(i, int(suffix[i]))
        pool.share_prefix(i, i + 1, pool.sequence_length(i))
    seqs = list(range(cfg["batch"]))
    slots = []
    for s in seqs:
        n = pool.sequence_length(s)
        pool.append(s, 1)
        slots.append(pool.slots(s, n, 1)[0])
    pairs = np.array(pool.take_copy_pairs(), dtype=np.int64).reshape(-1, 2)
    assert 16 <= len(pairs) <= 32
    tables = cases.padded_tables(pool, seqs)
    lens = np.array([pool.sequence_length(s) for s in seqs], dtype=np.int32)
    dev = torch.device("cuda", 0)
    HKV, D = cfg["kv_heads"], cfg["head_dim"]
    w = dict(cfg=cfg, k_pool=W.torch_normal((total, HKV, 16, D), 51, torch.bfloat16, dev),
             v_pool=W.torch_normal((total, HKV, 16, D), 52, torch.bfloat16, dev),
             q=W.torch_normal((cfg["batch"], cfg["q_heads"], D), 53, torch.bfloat16, dev),
             k_new=W.torch_normal((cfg["batch"], HKV, D), 54, torch.bfloat16, dev),
             v_new=W.torch_normal((cfg["batch"], HKV, D), 55, torch.bfloat16, dev),
             slots=torch.from_numpy(np.array(slots, np.int64)).to(dev), slots_np=np.array(slots, np.int64),
             pairs=torch.from_numpy(pairs).to(dev), tables=torch.from_numpy(tables).to(dev),
             lens=torch.from_numpy(lens).to(dev), tables_np=tables, lens_np=lens, scale=1.0 / np.sqrt(D))
    check_workload(pkv, w, "prefix with copy-on-write pairs", indices=(np.array(slots, np.int64), pairs))


def test_prefix_workload_two_phase(pkv):
    """The prefix workload through the shared-prefix call (all 64 sequences
    in one group over the 256 shared blocks), in the benchmark's launch
    configuration: every row against the single-pass float64 oracle, and
    against the plain decode."""
    w = W.device_workload("prefix", torch.device("cuda", 0))
    cfg = w["cfg"]
    kv_heads = cfg["kv_heads"]
    G = cfg["q_heads"] // kv_heads
    nb = cfg["prefix"] // 16
    slots, _ = oracle_step_indices(w)
    hk, hv = cases.host_view(w["k_pool"]), cases.host_view(w["v_pool"])
    OK.append_tokens(hk, hv, cases.host_view(w["k_new"]), cases.host_view(w["v_new"]), slots)
    pkv.pkv_copy_blocks(w["pairs"], w["k_pool"], w["v_pool"])
    pkv.pkv_append(w["k_new"], w["v_new"], w["slots"], w["k_pool"], w["v_pool"])
    group = torch.zeros(cfg["batch"], dtype=torch.int32, device="cuda")
    blocks = torch.tensor([nb], dtype=torch.int32, device="cuda")
    out = pkv.pkv_decode_attention_prefixed(w["q"], w["k_pool"], w["v_pool"], w["tables"], w["lens"], w["scale"],
                                            group, blocks, nb)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status(clear=True) == 0
    want = OA.decode_attention(cases.host_view(w["q"]), hk, hv, w["tables_np"], w["lens_np"], w["scale"], kv_heads,
                               "bf16")
    check_all_rows("prefix, two-phase call", out, want, G)
    ref = pkv.pkv_decode_attention(w["q"], w["k_pool"], w["v_pool"], w["tables"], w["lens"], w["scale"])
    d = out.float() - ref.float()
    assert (d.norm() / ref.float().norm()).item() <= 2e-3 and d.abs().max().item() <= 1e-2


def test_spec4_workload_multiquery(pkv):
    """The 8K Llama layer verifying 4 draft tokens per sequence: one append of
    128 new tokens and one multi-query call, as the benchmark runs them.
    Every row against the float64 causal oracle; every row also against the
    decode kernel run once per query position (query t of each sequence is a
    decode over the first 8192 - 4 + t + 1 tokens)."""
    from oracle import multiquery as OM
    w = W.device_workload("spec4", torch.device("cuda", 0))
    cfg, nq = w["cfg"], w["queries"]
    kv_heads = cfg["kv_heads"]
    G = cfg["q_heads"] // kv_heads
    slots, _ = oracle_step_indices(w)
    hk, hv = cases.host_view(w["k_pool"]), cases.host_view(w["v_pool"])
    OK.append_tokens(hk, hv, cases.host_view(w["k_new"]), cases.host_view(w["v_new"]), slots)
    pkv.pkv_append(w["k_new"], w["v_new"], w["slots"], w["k_pool"], w["v_pool"])
    out = pkv.pkv_multiquery_attention(w["q"], w["k_pool"], w["v_pool"], w["tables"], w["lens"], w["query_start"],
                                       w["scale"], nq)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status(clear=True) == 0
    assert np.array_equal(cases.host_view(w["k_pool"]), hk) and np.array_equal(cases.host_view(w["v_pool"]), hv)
    qs = np.arange(0, cfg["batch"] * nq + 1, nq)
    want = OM.multiquery_attention(cases.host_view(w["q"]), hk, hv, w["tables_np"], w["lens_np"], qs, w["scale"],
                                   kv_heads, "bf16")
    check_all_rows("spec4", out, want, G)
    for t in range(nq):
        ref = pkv.pkv_decode_attention(w["q"][t::nq].contiguous(), w["k_pool"], w["v_pool"], w["tables"],
                                       w["lens"] - (nq - 1 - t), w["scale"])
        d = out[t::nq].float() - ref.float()
        assert d.abs().max().item() <= 1e-2 and (d.norm() / ref.float().norm()).item() <= 2e-3, t


def test_llama8k_q8_workload(pkv):
    """The 8K Llama layer over an int8 cache, as the benchmark runs it: the
    quantizing append of the step's 32 tokens (whole pools bit-exact against
    the oracle's append) and one decode call; every row against the float64
    oracle over the values the cache stands for."""
    from oracle import quant as OQ
    w = W.device_workload("llama8k_q8", torch.device("cuda", 0))
    cfg = w["cfg"]
    kv_heads = cfg["kv_heads"]
    G = cfg["q_heads"] // kv_heads
    slots, _ = oracle_step_indices(w)
    hkc, hvc = w["k_pool"].cpu().numpy(), w["v_pool"].cpu().numpy()
    hks, hvs = w["k_scales"].cpu().numpy(), w["v_scales"].cpu().numpy()
    kn = OA.bf16_bits_to_f64(cases.host_view(w["k_new"]))
    vn = OA.bf16_bits_to_f64(cases.host_view(w["v_new"]))
    # the V pool is stored [block][head][d][16]; the oracle writes token rows through a transposed view
    OQ.append_tokens_q8(hkc, hvc.transpose(0, 1, 3, 2), hks, hvs, kn, vn, slots)
    pkv.pkv_append_q8(w["k_new"], w["v_new"], w["slots"], w["k_pool"], w["v_pool"], w["scales"])
    out = pkv.pkv_decode_attention_q8(w["q"], w["k_pool"], w["v_pool"], w["scales"], w["tables"],
                                      w["lens"], w["scale"])
    torch.cuda.synchronize()
    assert pkv.pkv_device_status(clear=True) == 0
    assert np.array_equal(w["k_pool"].cpu().numpy(), hkc) and np.array_equal(w["v_pool"].cpu().numpy(), hvc)
    assert np.array_equal(w["k_scales"].cpu().numpy(), hks) and np.array_equal(w["v_scales"].cpu().numpy(), hvs)
    want = OQ.decode_attention_q8(cases.host_view(w["q"]), hkc, hvc.transpose(0, 1, 3, 2), hks, hvs, w["tables_np"],
                                  w["lens_np"], w["scale"], kv_heads, "bf16")
    check_all_rows("llama8k_q8", out, want, G)


def test_prefill512_workload(pkv):
    """Chunked prefill on the 8K Llama layer (512 causal queries per sequence,
    the tensor-core tile path), as the benchmark runs it: the append of the
    chunk's 4096 tokens (pools bit-exact), then one multi-query call; every
    row against the float64 causal oracle."""
    from oracle import multiquery as OM
    w = W.device_workload("prefill512", torch.device("cuda", 0))
    cfg, nq = w["cfg"], w["queries"]
    kv_heads = cfg["kv_heads"]
    G = cfg["q_heads"] // kv_heads
    slots, _ = oracle_step_indices(w)
    hk, hv = cases.host_view(w["k_pool"]), cases.host_view(w["v_pool"])
    OK.append_tokens(hk, hv, cases.host_view(w["k_new"]), cases.host_view(w["v_new"]), slots)
    pkv.pkv_append(w["k_new"], w["v_new"], w["slots"], w["k_pool"], w["v_pool"])
    out = pkv.pkv_multiquery_attention(w["q"], w["k_pool"], w["v_pool"], w["tables"], w["lens"], w["query_start"],
                                       w["scale"], nq)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status(clear=True) == 0
    assert np.array_equal(cases.host_view(w["k_pool"]), hk) and np.array_equal(cases.host_view(w["v_pool"]), hv)
    qs = np.arange(0, cfg["batch"] * nq + 1, nq)
    want = OM.multiquery_attention(cases.host_view(w["q"]), hk, hv, w["tables_np"], w["lens_np"], qs, w["scale"],
                                   kv_heads, "bf16")
    check_all_rows("prefill512", out, want, G)


def test_prefill_at_the_query_limit(pkv):
    """The largest query count the multi-query call accepts: one sequence
    whose last 65536 tokens (max_query_len) are queries, after a 100-token
    prefix; 8 q / 2 KV heads, head_dim 64, i.e. 2048 tiles of 128 rows per KV
    head on the tensor-core path. Every output finite; the first, second,
    last and one middle query row against the float64 oracle."""
    from oracle import multiquery as OM
    nq, prefix = 65536, 100
    c = cases.random_case(71, [prefix + nq], 8, 2, 64, torch.bfloat16)
    q = torch.from_numpy(W.numpy_normal((nq, 8, 64), 72)).to(torch.bfloat16)
    dev = torch.device("cuda", 0)
    out = pkv.pkv_multiquery_attention(q.to(dev), c["k_pool"].to(dev), c["v_pool"].to(dev),
                                       torch.from_numpy(c["tables"]).to(dev), torch.from_numpy(c["lens"]).to(dev),
                                       torch.tensor([0, nq], dtype=torch.int32, device=dev), c["scale"], nq)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status(clear=True) == 0
    assert bool(torch.isfinite(out.float()).all())
    qh, hk, hv = cases.host_view(q), cases.host_view(c["k_pool"]), cases.host_view(c["v_pool"])
    for t in (0, 1, 40000, nq - 1):
        # query t sees tokens 0 .. prefix + t: the same as a one-query call on that many tokens
        want = OM.multiquery_attention(qh[t:t + 1], hk, hv, c["tables"], np.array([prefix + t + 1], dtype=np.int32),
                                       np.array([0, 1]), c["scale"], 2, "bf16")
        ma, rl = cases.attention_errors(out[t:t + 1], want)
        assert ma <= MAX_ABS and rl <= REL_L2, (t, ma, rl)
