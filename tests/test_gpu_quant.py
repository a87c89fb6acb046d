"""Low-bit (int8) paged KV through the C ABI against the oracle.

The quantizing append and the block copy must match the oracle byte for byte
(codes and float32 scales; the V code pool is stored coordinate-major, so it
is compared transposed). Attention over the int8 pools (decode and causal
multi-query) must match the float64 oracle over the values the cached rows
stand for, within the decode tolerance; cases cover group sizes 1-8, ragged
and empty contexts, cut segments, and malformed inputs.
"""

import numpy as np
import pytest
import torch

import cases
from oracle import attention as OA
from oracle import multiquery as OM
from oracle import quant as OQ
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


def empty_pools(nb, hkv, d=128, seed=0):
    """Pools holding arbitrary earlier contents (every byte set)."""
    g = torch.Generator().manual_seed(seed)
    kc = torch.randint(-127, 128, (nb, hkv, 16, d), generator=g, dtype=torch.int8)
    vc = torch.randint(-127, 128, (nb, hkv, d, 16), generator=g, dtype=torch.int8)
    ks = torch.rand((nb, hkv, 16), generator=g) * 0.05
    vs = torch.rand((nb, hkv, 16), generator=g) * 0.05
    return kc, vc, torch.stack([ks, vs], dim=2).contiguous()   # scale pool [nb][hkv][2][16]


def host(t):
    return t.detach().cpu().numpy()


def logical_v(vc):
    """[blocks][heads][d][16] -> the oracle's [blocks][heads][16][d]."""
    return np.ascontiguousarray(host(vc).transpose(0, 1, 3, 2))


@pytest.mark.parametrize("d", [128, 64])
def test_append_and_copy_bit_exact(pkv, d):
    nb, hkv, T = 24, 4, 40
    kc, vc, sc = empty_pools(nb, hkv, d)
    rng = np.random.default_rng(3)
    k = torch.from_numpy(W.numpy_normal((T, hkv, d), 31) * rng.uniform(0.01, 50, (T, hkv, 1)).astype(np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(W.numpy_normal((T, hkv, d), 32)).to(torch.bfloat16)
    k[3, 1] = 0.0                                             # a zero row: scale 1
    # exact ties: scale 1 (max 127) with half-integer values, scale 2 (max 254) with odd integers;
    # the oracle rounds half to even
    tie = rng.integers(-254, 255, (2, d)).astype(np.float32)
    k[7, 0] = torch.from_numpy(np.r_[127.0, tie[0, 1:] / 2]).to(torch.bfloat16)
    v[9, 2] = torch.from_numpy(np.r_[254.0, tie[1, 1:]]).to(torch.bfloat16)
    slots = rng.permutation(nb * 16)[:T].astype(np.int64)
    slots[[5, 17]] = -1                                       # skipped tokens
    hkc, hvc, hsc = host(kc).copy(), logical_v(vc), host(sc).copy()
    # the oracle keeps K and V scales apart: it writes through views of the record's two rows
    OQ.append_tokens_q8(hkc, hvc, hsc[:, :, 0], hsc[:, :, 1], OA.bf16_bits_to_f64(cases.bf16_bits(k)),
                        OA.bf16_bits_to_f64(cases.bf16_bits(v)), slots)
    dkc, dvc, dsc = kc.cuda(), vc.cuda(), sc.cuda()
    pkv.pkv_append_q8(k.cuda(), v.cuda(), torch.from_numpy(slots).cuda(), dkc, dvc, dsc)
    torch.cuda.synchronize()
    assert np.array_equal(host(dkc), hkc) and np.array_equal(logical_v(dvc), hvc)
    assert np.array_equal(host(dsc), hsc)
    # two written blocks copied onto blocks 0 and 1 (no pair reads a block another one writes)
    srcs = [b for b in dict.fromkeys(int(s) // 16 for s in slots if s >= 0) if b > 1][:2]
    pairs = np.array([[srcs[0], 0], [srcs[1], 1]], dtype=np.int64)
    for arr in (hkc, hvc, hsc):
        for src, dst in pairs:
            arr[dst] = arr[src]
    pkv.pkv_copy_blocks_q8(torch.from_numpy(pairs).cuda(), dkc, dvc, dsc)
    torch.cuda.synchronize()
    assert np.array_equal(host(dkc), hkc) and np.array_equal(logical_v(dvc), hvc)
    assert np.array_equal(host(dsc), hsc)
    assert pkv.pkv_device_status(clear=True) == 0


def q8_case(seed, lens, q_heads, kv_heads, nqs=None, d=128):
    """Random K/V quantized by the oracle into int8 pools; q bf16."""
    c = cases.random_case(seed, lens, q_heads, kv_heads, d, torch.bfloat16)
    kf = OA.bf16_bits_to_f64(cases.host_view(c["k_pool"]))
    vf = OA.bf16_bits_to_f64(cases.host_view(c["v_pool"]))
    kc, ks = OQ.quantize_rows(kf)
    vc, vs = OQ.quantize_rows(vf)
    c.update(kc=kc, vc=vc, ks=ks, vs=vs)
    if nqs is not None:
        qs = np.concatenate([[0], np.cumsum(nqs)]).astype(np.int32)
        c["q"] = torch.from_numpy(W.numpy_normal((int(qs[-1]), q_heads, d), seed * 7 + 9)).to(torch.bfloat16)
        c["query_start"] = qs
    return c


def run_q8(pkv, c, **kw):
    dev = torch.device("cuda", 0)
    kc = torch.from_numpy(c["kc"]).to(dev)
    vc = torch.from_numpy(np.ascontiguousarray(c["vc"].transpose(0, 1, 3, 2))).to(dev)   # coordinate-major
    sc = torch.from_numpy(np.stack([c["ks"], c["vs"]], axis=2)).to(dev)   # [blocks][heads][2][16]
    qs = torch.from_numpy(c["query_start"]).to(dev) if "query_start" in c else None
    out = pkv.pkv_decode_attention_q8(c["q"].to(dev), kc, vc, sc, torch.from_numpy(c["tables"]).to(dev),
                                      torch.from_numpy(c["lens"]).to(dev), c["scale"], query_start=qs, **kw)
    torch.cuda.synchronize()
    return out


def want_q8(c):
    kd = OQ.dequantize_rows(c["kc"], c["ks"])
    vd = OQ.dequantize_rows(c["vc"], c["vs"])
    qf = OA.bf16_bits_to_f64(cases.host_view(c["q"]))
    if "query_start" in c:
        return OM.multiquery_attention(qf, kd, vd, c["tables"], c["lens"], c["query_start"], c["scale"],
                                       c["kv_heads"], "f64")
    return OA.decode_attention(qf, kd, vd, c["tables"], c["lens"], c["scale"], c["kv_heads"], "f64")


def check(out, ref):
    ma, rl = cases.attention_errors(out, ref)
    assert ma <= MAX_ABS and rl <= REL_L2, (ma, rl)


@pytest.mark.parametrize("hq,hkv", [(32, 8), (64, 8), (8, 8), (24, 8)])
def test_decode_q8_matches_oracle(pkv, hq, hkv):
    c = q8_case(hq + hkv, [300, 1, 0, 17, 1000, 64, 5], hq, hkv)
    out = run_q8(pkv, c)
    assert pkv.pkv_device_status(clear=True) == 0
    check(out, want_q8(c))
    assert bool((out[2] == 0).all())                          # an empty context gives a zero row


@pytest.mark.parametrize("num_ctas", [3, 40, 5000])
def test_decode_q8_cut_segments(pkv, num_ctas):
    c = q8_case(5, [2000, 333, 40, 1500], 32, 8)
    out = run_q8(pkv, c, num_ctas=num_ctas)
    assert pkv.pkv_device_status(clear=True) == 0
    check(out, want_q8(c))


@pytest.mark.parametrize("nqs,hq,mql", [([4, 4, 4, 1], 32, 4), ([8, 3, 0, 5], 32, 8), ([2, 1, 2, 2], 64, 2)])
def test_multiquery_q8_matches_oracle(pkv, nqs, hq, mql):
    c = q8_case(sum(nqs) + hq, [700, 40, 129, 9], hq, 8, nqs=nqs)
    out = run_q8(pkv, c, max_query_len=mql)
    assert pkv.pkv_device_status(clear=True) == 0
    check(out, want_q8(c))


@pytest.mark.parametrize("multi", [False, True])
def test_poisoned_scales_of_unused_slots(pkv, multi):
    """Slots no sequence holds (the rest of each last block, spare blocks)
    carry NaN K scales and +inf V scales: a masked token must contribute
    nothing, not 0 * inf. Decode and 4 queries per sequence."""
    lens = [300, 17, 1001, 45, 130]
    c = q8_case(78 + multi, lens, 32, 8, nqs=[4] * len(lens) if multi else None)
    live = np.zeros(c["ks"].shape[0::2], dtype=bool)         # [blocks][slots]
    for i, n in enumerate(c["lens"]):
        for t in range(int(n)):
            live[c["tables"][i, t // 16], t % 16] = True
    c["ks"].transpose(0, 2, 1)[~live] = np.nan
    c["vs"].transpose(0, 2, 1)[~live] = np.inf
    out = run_q8(pkv, c, max_query_len=4 if multi else 1)
    assert pkv.pkv_device_status(clear=True) == 0
    assert bool(torch.isfinite(out).all())
    with np.errstate(invalid="ignore"):                      # the oracle dequantizes the poisoned rows too
        ref = want_q8(c)
    check(out, ref)


def test_wide_scales_and_large_queries(pkv):
    """Row scales spanning four orders of magnitude, and queries far outside
    the f16 range (the kernel rescales each query row by a power of two before
    the f16 product). The bf16 output rounds relative to its size, so the
    max-abs bar scales with the largest output."""
    c = q8_case(77, [90, 200, 33, 700], 32, 8)
    rng = np.random.default_rng(8)
    c["ks"] = (c["ks"] * rng.uniform(1e-3, 10, c["ks"].shape)).astype(np.float32)
    c["vs"] = (c["vs"] * rng.uniform(1e-2, 1e2, c["vs"].shape)).astype(np.float32)
    q = OA.bf16_bits_to_f64(cases.host_view(c["q"])).astype(np.float32)
    c["q"] = torch.from_numpy(q * 3e5).to(torch.bfloat16)
    c["scale"] = float(np.float32(1.0 / (3e5 * np.sqrt(128))))
    out = run_q8(pkv, c)
    assert pkv.pkv_device_status(clear=True) == 0
    ref = want_q8(c)
    ma, rl = cases.attention_errors(out, ref)
    assert ma <= MAX_ABS * max(1.0, float(np.abs(ref).max())) and rl <= REL_L2, (ma, rl)


@pytest.mark.parametrize("vmax", [4.0e4, 1.0e6, 1.0e20])
@pytest.mark.parametrize("multi", [False, True])
def test_v_rows_beyond_the_f16_range_of_p(pkv, vmax, multi):
    """V rows whose largest magnitude is above ~32 000 (a V scale above 255)
    would take P' = P * s_v past the f16 maximum. The kernel runs a block
    holding such a row on P' and O scaled down by a power of two and scales
    O back, so the output still matches the oracle (relative bars: the
    output is as large as V). Sequence 0 has only such rows; in the others a
    fifth of the rows are."""
    c = q8_case(79, [90, 200, 33, 700], 32, 8, nqs=[3, 1, 2, 4] if multi else None)
    rng = np.random.default_rng(9)
    big = rng.random(c["vs"].shape) < 0.2
    big[c["tables"][0, :6]] = True
    c["vs"] = np.where(big, np.float32(vmax / 127), c["vs"]).astype(np.float32)
    out = run_q8(pkv, c, max_query_len=4 if multi else 1)
    assert pkv.pkv_device_status(clear=True) == 0
    assert bool(torch.isfinite(out.float()).all())
    ref = want_q8(c)
    ma, rl = cases.attention_errors(out, ref)
    assert ma <= MAX_ABS * max(1.0, float(np.abs(ref).max())) and rl <= REL_L2, (ma, rl)


def test_host_rejections(pkv):
    c = q8_case(9, [30, 40], 32, 8)
    with pytest.raises(pkv.PkvError) as e:
        run_q8(pkv, c, max_query_len=2)                       # multi-query needs query offsets
    assert e.value.name == "PKV_ERR_SHAPE"
    c64 = q8_case(9, [30, 40], 16, 2, d=64)
    with pytest.raises(pkv.PkvError) as e:
        run_q8(pkv, c64)                                      # the attention is head_dim 128 only
    assert e.value.name == "PKV_ERR_SHAPE"


def test_bad_block_id_and_checked_mode(pkv):
    """A block id outside the pool is never loaded: the call sets
    PKV_DEVERR_RANGE and the rows of the other sequences stay right; checked
    mode rejects the call before anything is written."""
    c = q8_case(21, [60, 45, 100], 32, 8)
    nb = c["kc"].shape[0]
    bad = dict(c, tables=c["tables"].copy())
    bad["tables"][1, 1] = nb + 7                               # sequence 1, its second block
    out = run_q8(pkv, bad)
    assert pkv.pkv_device_status(clear=True) & 2
    ref = want_q8(c)
    check(out[[0, 2]], ref[[0, 2]])
    dev = torch.device("cuda", 0)
    out2 = torch.full((3, 32, 128), 5.0, dtype=torch.bfloat16, device=dev)
    with pytest.raises(pkv.PkvError) as e:
        run_q8(pkv, bad, out=out2, flags=pkv.PKV_FLAG_CHECKED)
    assert e.value.name == "PKV_ERR_RANGE"
    assert bool((out2 == 5.0).all())
    assert pkv.pkv_device_status(clear=True) == 0


def test_bounded_wait_runs_out_and_is_reported(pkv):
    """The stall hook on the int8 attention: every wait runs out, the status
    reports it, and the next call is right."""
    c = q8_case(66, [200, 33, 700], 32, 8)
    pkv.pkv_device_status(clear=True)
    run_q8(pkv, c, flags=pkv.PKV_FLAG_TEST_STALL)
    assert pkv.pkv_device_status(clear=True) & pkv.PKV_DEVERR_TIMEOUT
    out = run_q8(pkv, c)
    assert pkv.pkv_device_status(clear=True) == 0
    check(out, want_q8(c))


def test_batch_above_one_launch(pkv):
    """More than 1024 sequences: one launch per 1024, decode rows at their
    absolute positions."""
    rng = np.random.default_rng(67)
    lens = rng.integers(0, 80, 1030)
    c = q8_case(67, lens, 8, 2)
    out = run_q8(pkv, c)
    assert pkv.pkv_device_status(clear=True) == 0
    check(out, want_q8(c))
