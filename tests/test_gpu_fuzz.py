"""Seeded random shapes through every attention path, each against the float64
oracle (every output element, decode bars: max-abs 1e-2, relative L2 2e-3).

For each path 24 cases draw the batch, the context lengths (including empty
contexts and contexts inside one block), the query-head group size, head_dim
and, where the call takes them, forced CTA counts, query counts and prefix
groups; about half of the decode and multi-query cases hold K = NaN and
V = -inf in every slot no sequence holds. A failing case prints its seed, so
it can be rerun alone.
"""

import numpy as np
import pytest
import torch

import cases
from oracle import attention as OA
from oracle import multiquery as OM
from oracle import quant as OQ

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2 = 1e-2, 2e-3
N_CASES = 24


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_209_gb300 import pkv as P
    P.load_library()
    return P


def check(out, want, seed):
    ma, rl = cases.attention_errors(out, want)
    assert ma <= MAX_ABS and rl <= REL_L2, (seed, ma, rl)


def heads(rng, max_g=8):
    hkv = int(rng.choice([1, 2, 8]))
    g = int(rng.choice([g for g in (1, 2, 3, 4, 8) if g <= max_g]))
    return hkv * g, hkv


def lengths(rng, batch, hi):
    lens = rng.integers(0, hi, batch)
    lens[rng.random(batch) < 0.15] = 0                      # empty contexts
    lens[rng.random(batch) < 0.15] = rng.integers(1, 17)    # inside one block
    return lens


@pytest.mark.parametrize("seed", range(N_CASES))
def test_decode_random(pkv, seed):
    rng = np.random.default_rng(1000 + seed)
    hq, hkv = heads(rng)
    d = int(rng.choice([64, 128]))
    lens = lengths(rng, int(rng.integers(1, 40)), int(rng.choice([64, 700, 3000])))
    kw = {}
    if rng.random() < 0.5:
        kw["num_ctas"] = int(rng.integers(1, 400))          # cut segments at arbitrary places
    c = cases.random_case(1000 + seed, lens, hq, hkv, d, torch.bfloat16, poison=bool(rng.random() < 0.5))
    dev = torch.device("cuda", 0)
    out = pkv.pkv_decode_attention(c["q"].to(dev), c["k_pool"].to(dev), c["v_pool"].to(dev),
                                   torch.from_numpy(c["tables"]).to(dev), torch.from_numpy(c["lens"]).to(dev),
                                   c["scale"], **kw)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status(clear=True) == 0, seed
    want = OA.decode_attention(cases.host_view(c["q"]), cases.host_view(c["k_pool"]), cases.host_view(c["v_pool"]),
                               c["tables"], c["lens"], c["scale"], hkv, "bf16")
    check(out, want, seed)


@pytest.mark.parametrize("seed", range(N_CASES))
def test_multiquery_random(pkv, seed):
    """Both multi-query paths: query counts drawn so that about half the cases
    exceed 32 rows per (sequence, KV head) and run on the tile kernel."""
    rng = np.random.default_rng(2000 + seed)
    hq, hkv = heads(rng)
    G = hq // hkv
    d = int(rng.choice([64, 128]))
    lens = np.maximum(lengths(rng, int(rng.integers(1, 12)), int(rng.choice([40, 300, 1500]))), 1)
    mql = int(rng.choice([1, 2, 4, 8, 40, 130]))
    nqs = np.minimum(lens, rng.integers(0, mql + 1, len(lens)))
    c = cases.multiquery_case(2000 + seed, lens, nqs, hq, hkv, d, torch.bfloat16, poison=bool(rng.random() < 0.5))
    dev = torch.device("cuda", 0)
    out = pkv.pkv_multiquery_attention(c["q"].to(dev), c["k_pool"].to(dev), c["v_pool"].to(dev),
                                       torch.from_numpy(c["tables"]).to(dev), torch.from_numpy(c["lens"]).to(dev),
                                       torch.from_numpy(c["query_start"]).to(dev), c["scale"], mql)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status(clear=True) == 0, (seed, mql * G)
    want = OM.multiquery_attention(cases.host_view(c["q"]), cases.host_view(c["k_pool"]),
                                   cases.host_view(c["v_pool"]), c["tables"], c["lens"], c["query_start"], c["scale"],
                                   hkv, "bf16")
    check(out, want, (seed, mql * G))


@pytest.mark.parametrize("seed", range(N_CASES))
def test_prefixed_random(pkv, seed):
    """Shared-prefix groups of random sizes and prefix lengths (both chunk-first
    kernels), plus sequences in no group."""
    rng = np.random.default_rng(3000 + seed)
    hq, hkv = heads(rng)
    d = int(rng.choice([64, 128]))
    n = int(rng.integers(2, 30))
    ngroups = int(rng.integers(1, 4))
    member_of = rng.integers(-1, ngroups, n)
    group_blocks = rng.integers(0, 40, ngroups)
    suffix = rng.integers(0, 400, n)
    c = cases.grouped_case(3000 + seed, member_of, group_blocks, suffix, hq, hkv, d, torch.bfloat16)
    dev = torch.device("cuda", 0)
    mgb = int(c["group_blocks"].max())
    out = pkv.pkv_decode_attention_prefixed(
        c["q"].to(dev), c["k_pool"].to(dev), c["v_pool"].to(dev), torch.from_numpy(c["tables"]).to(dev),
        torch.from_numpy(c["lens"]).to(dev), c["scale"], torch.from_numpy(c["prefix_group"]).to(dev),
        torch.from_numpy(c["group_blocks"]).to(dev), mgb, prefix_kernel=int(rng.choice([1, 2])))
    torch.cuda.synchronize()
    assert pkv.pkv_device_status(clear=True) == 0, seed
    want = OA.decode_attention(cases.host_view(c["q"]), cases.host_view(c["k_pool"]), cases.host_view(c["v_pool"]),
                               c["tables"], c["lens"], c["scale"], hkv, "bf16")
    check(out, want, seed)


@pytest.mark.parametrize("seed", range(N_CASES))
def test_int8_random(pkv, seed):
    """Int8 cache: decode (no query offsets) or multi-query up to 32 rows."""
    rng = np.random.default_rng(4000 + seed)
    hq, hkv = heads(rng)
    G = hq // hkv
    lens = lengths(rng, int(rng.integers(1, 30)), int(rng.choice([64, 700, 2500])))
    multi = rng.random() < 0.5 and 32 // G >= 2
    if multi:
        lens = np.maximum(lens, 1)
        mql = int(rng.integers(2, 32 // G + 1))
        nqs = np.minimum(lens, rng.integers(0, mql + 1, len(lens)))
        c = cases.multiquery_case(4000 + seed, lens, nqs, hq, hkv, 128, torch.bfloat16)
    else:
        mql = 1
        c = cases.random_case(4000 + seed, lens, hq, hkv, 128, torch.bfloat16)
    kc, ks = OQ.quantize_rows(OA.bf16_bits_to_f64(cases.host_view(c["k_pool"])))
    vc, vs = OQ.quantize_rows(OA.bf16_bits_to_f64(cases.host_view(c["v_pool"])))
    dev = torch.device("cuda", 0)
    qs = torch.from_numpy(c["query_start"]).to(dev) if multi else None
    out = pkv.pkv_decode_attention_q8(
        c["q"].to(dev), torch.from_numpy(kc).to(dev),
        torch.from_numpy(np.ascontiguousarray(vc.transpose(0, 1, 3, 2))).to(dev),
        torch.from_numpy(np.stack([ks, vs], axis=2)).to(dev), torch.from_numpy(c["tables"]).to(dev), torch.from_numpy(c["lens"]).to(dev),
        c["scale"], query_start=qs, max_query_len=mql)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status(clear=True) == 0, seed
    kd, vd = OQ.dequantize_rows(kc, ks), OQ.dequantize_rows(vc, vs)
    qf = OA.bf16_bits_to_f64(cases.host_view(c["q"]))
    if multi:
        want = OM.multiquery_attention(qf, kd, vd, c["tables"], c["lens"], c["query_start"], c["scale"], hkv, "f64")
    else:
        want = OA.decode_attention(qf, kd, vd, c["tables"], c["lens"], c["scale"], hkv, "f64")
    check(out, want, seed)
