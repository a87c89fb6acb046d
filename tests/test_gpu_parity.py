"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Append and block copy must be bit-exact over both whole pools (touched and
untouched blocks). Attention (fp32 accumulation) must meet max |err| <= 1e-2
and relative L2 <= 2e-3 against the float64 oracle; fp32 caches are held to
a tighter 2e-5 relative.
"""

import numpy as np
import pytest
import torch

import cases
from oracle import attention as OA
from oracle import kv_ops as OK

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2 = 1e-2, 2e-3


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_209_gb300 import pkv as P
    P.load_library()
    return P


def dev(x, dtype=None):
    t = torch.as_tensor(x)
    if dtype is not None:
        t = t.to(dtype)
    return t.contiguous().cuda()


def oracle_attention(case, tables, lens, q=None, k_pool=None, v_pool=None):
    q = case["q"] if q is None else q
    kp = case["k_pool"] if k_pool is None else k_pool
    vp = case["v_pool"] if v_pool is None else v_pool
    return OA.decode_attention(cases.host_view(q), cases.host_view(kp), cases.host_view(vp), tables, lens,
                               float(case["scale"]), case["kv_heads"], cases.dtype_name(q))


def run_attention(pkv, q, kp, vp, tables, lens, scale, **kw):
    return pkv.pkv_decode_attention(q, kp, vp, dev(tables, torch.int32), dev(lens, torch.int32), float(scale), **kw)


def check_close(got, want, rel=REL_L2, max_abs=MAX_ABS):
    ma, rl = cases.attention_errors(got, want)
    assert np.all(np.isfinite(got.float().cpu().numpy())), "non-finite output"
    assert ma <= max_abs and rl <= rel, f"max_abs={ma:.3e} rel_l2={rl:.3e}"
    return ma, rl


# ------------------------------------------------------------------ append / copy
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_tiny_step_copy_append_bit_exact(pkv, dtype):
    c = cases.tiny_case(dtype=dtype)
    kp, vp = dev(c["k_pool"]), dev(c["v_pool"])
    assert len(c["pairs"]) == 1
    pkv.pkv_copy_blocks(dev(c["pairs"]), kp, vp)
    pkv.pkv_append(dev(c["k_new"]), dev(c["v_new"]), dev(c["slots"]), kp, vp)
    hk, hv = cases.host_view(c["k_pool"]).copy(), cases.host_view(c["v_pool"]).copy()
    OK.copy_blocks(hk, hv, c["pairs"])
    OK.append_tokens(hk, hv, cases.host_view(c["k_new"]), cases.host_view(c["v_new"]), c["slots"])
    assert np.array_equal(cases.host_view(kp), hk)
    assert np.array_equal(cases.host_view(vp), hv)


@pytest.mark.parametrize("head_dim,kv_heads,dtype", [(128, 8, torch.bfloat16), (64, 3, torch.float32),
                                                     (128, 1, torch.float32)])
def test_append_many_tokens_with_padding_bit_exact(pkv, head_dim, kv_heads, dtype):
    rng = np.random.default_rng(5)
    nb = 300
    T = 777
    slots = rng.permutation(nb * 16)[:T].astype(np.int64)
    slots[rng.choice(T, 40, replace=False)] = -1
    kp = torch.randn(nb, kv_heads, 16, head_dim, generator=torch.Generator().manual_seed(1)).to(dtype)
    vp = torch.randn(nb, kv_heads, 16, head_dim, generator=torch.Generator().manual_seed(2)).to(dtype)
    kn = torch.randn(T, kv_heads, head_dim, generator=torch.Generator().manual_seed(3)).to(dtype)
    vn = torch.randn(T, kv_heads, head_dim, generator=torch.Generator().manual_seed(4)).to(dtype)
    dkp, dvp = dev(kp), dev(vp)
    pkv.pkv_append(dev(kn), dev(vn), dev(slots), dkp, dvp)
    hk, hv = cases.host_view(kp).copy(), cases.host_view(vp).copy()
    OK.append_tokens(hk, hv, cases.host_view(kn), cases.host_view(vn), slots)
    assert np.array_equal(cases.host_view(dkp), hk)
    assert np.array_equal(cases.host_view(dvp), hv)


def test_copy_many_pairs_bit_exact(pkv):
    rng = np.random.default_rng(6)
    nb = 200
    ids = rng.permutation(nb)
    pairs = np.stack([ids[:37], ids[37:74]], axis=1).astype(np.int64)
    kp = torch.randn(nb, 8, 16, 128, generator=torch.Generator().manual_seed(7)).to(torch.bfloat16)
    vp = torch.randn(nb, 8, 16, 128, generator=torch.Generator().manual_seed(8)).to(torch.bfloat16)
    dkp, dvp = dev(kp), dev(vp)
    pkv.pkv_copy_blocks(dev(pairs), dkp, dvp)
    hk, hv = cases.host_view(kp).copy(), cases.host_view(vp).copy()
    OK.copy_blocks(hk, hv, pairs)
    assert np.array_equal(cases.host_view(dkp), hk)
    assert np.array_equal(cases.host_view(dvp), hv)


def test_zero_tokens_and_zero_pairs_are_no_ops(pkv):
    kp = dev(torch.randn(4, 2, 16, 64))
    vp = dev(torch.randn(4, 2, 16, 64))
    k0, v0 = kp.clone(), vp.clone()
    pkv.pkv_append(None, None, torch.zeros(0, dtype=torch.int64, device="cuda"), kp, vp)
    pkv.pkv_copy_blocks(torch.zeros(0, 2, dtype=torch.int64, device="cuda"), kp, vp)
    torch.cuda.synchronize()
    assert torch.equal(kp, k0) and torch.equal(vp, v0)


# ------------------------------------------------------------------ attention, tiny
@pytest.mark.parametrize("poison", [False, True])
def test_tiny_fp32_attention_before_and_after_step(pkv, poison):
    c = cases.tiny_case(dtype=torch.float32, poison=poison)
    q, kp, vp = dev(c["q"]), dev(c["k_pool"]), dev(c["v_pool"])
    got = run_attention(pkv, q, kp, vp, c["tables_before"], c["lens_before"], c["scale"])
    want = oracle_attention(c, c["tables_before"], c["lens_before"])
    check_close(got, want, rel=2e-5, max_abs=1e-4)
    # the step: copy, append, attend at the grown lengths
    pkv.pkv_copy_blocks(dev(c["pairs"]), kp, vp)
    pkv.pkv_append(dev(c["k_new"]), dev(c["v_new"]), dev(c["slots"]), kp, vp)
    got = run_attention(pkv, q, kp, vp, c["tables_after"], c["lens_after"], c["scale"])
    hk, hv = cases.host_view(c["k_pool"]).copy(), cases.host_view(c["v_pool"]).copy()
    OK.copy_blocks(hk, hv, c["pairs"])
    OK.append_tokens(hk, hv, cases.host_view(c["k_new"]), cases.host_view(c["v_new"]), c["slots"])
    want = OA.decode_attention(cases.host_view(c["q"]), hk, hv, c["tables_after"], c["lens_after"],
                               float(c["scale"]), 2, "f32")
    check_close(got, want, rel=2e-5, max_abs=1e-4)


def test_tiny_step_matches_contiguous_logical_attention(pkv):
    """After copy + append the paged result equals attention over the logical
    token sequence built without any paging (the notebook's B17 check)."""
    c = cases.tiny_case(dtype=torch.float32)
    kp, vp = dev(c["k_pool"]), dev(c["v_pool"])
    pkv.pkv_copy_blocks(dev(c["pairs"]), kp, vp)
    pkv.pkv_append(dev(c["k_new"]), dev(c["v_new"]), dev(c["slots"]), kp, vp)
    got = run_attention(pkv, dev(c["q"]), kp, vp, c["tables_after"], c["lens_after"], c["scale"])
    hk0 = c["k_pool"].numpy().astype(np.float64)
    hv0 = c["v_pool"].numpy().astype(np.float64)
    q = c["q"].numpy().astype(np.float64)
    for i in range(3):
        n_old = int(c["lens_before"][i])
        old_tab = c["tables_before"][i]
        ks = np.stack([hk0[old_tab[t // 16], :, t % 16, :] for t in range(n_old)] + [c["k_new"][i].numpy()])
        vs = np.stack([hv0[old_tab[t // 16], :, t % 16, :] for t in range(n_old)] + [c["v_new"][i].numpy()])
        want = OA.contiguous_attention(q[i], ks.astype(np.float64), vs.astype(np.float64), float(c["scale"]), 2)
        ma, rl = cases.attention_errors(got[i], want)
        assert rl < 2e-5, (i, rl)


# ------------------------------------------------------------------ attention, bf16 tensor-core path
SHAPES = [  # (lens, q_heads, kv_heads, head_dim)
    ([1, 7, 16, 17, 40, 100, 333], 32, 8, 128),
    ([5, 129, 1000, 2], 64, 8, 128),
    ([23, 300, 64], 8, 8, 64),
    ([16, 31, 250, 777], 6, 2, 128),
    ([513, 48, 9], 2, 1, 64),
]


@pytest.mark.parametrize("kernel", [1, 2])
@pytest.mark.parametrize("shape", range(len(SHAPES)))
def test_bf16_attention_ragged(pkv, shape, kernel):
    lens, qh, kvh, d = SHAPES[shape]
    c = cases.random_case(10 + shape, lens, qh, kvh, d, torch.bfloat16, poison=True)
    got = run_attention(pkv, dev(c["q"]), dev(c["k_pool"]), dev(c["v_pool"]), c["tables"], c["lens"],
                        c["scale"], kernel=kernel)
    want = oracle_attention(c, c["tables"], c["lens"])
    check_close(got, want)


@pytest.mark.parametrize("num_ctas", [1, 3, 7, 64, 1000, 5000])
def test_split_count_invariance(pkv, num_ctas):
    """Any CTA count (forcing segments to be cut anywhere) gives the same
    result within fp32 reassociation, and matches the oracle."""
    c = cases.random_case(30, [1, 17, 200, 1024, 4097, 33], 32, 8, 128, torch.bfloat16)
    args = (dev(c["q"]), dev(c["k_pool"]), dev(c["v_pool"]), c["tables"], c["lens"], c["scale"])
    ref = run_attention(pkv, *args, num_ctas=1)
    got = run_attention(pkv, *args, num_ctas=num_ctas)
    check_close(got, oracle_attention(c, c["tables"], c["lens"]))
    diff = (got.float() - ref.float()).abs().max().item()
    assert diff <= 2 ** -7, diff   # one bf16 ulp of an O(1) value at most


@pytest.mark.parametrize("num_ctas", [2, 3, 7, 64, 1000, 5000])
def test_split_count_invariance_fp32(pkv, num_ctas):
    """fp32 caches and fp32 output (CUDA-core kernel): cutting the contexts
    at any CTA count changes the result only by fp32 reassociation of the
    pieces' log-sum-exp merge, ~1e-6 relative against the one-CTA run (no
    output rounding hides a merge error here)."""
    c = cases.random_case(32, [1, 17, 200, 1024, 4097, 33], 32, 8, 128, torch.float32)
    args = (dev(c["q"]), dev(c["k_pool"]), dev(c["v_pool"]), c["tables"], c["lens"], c["scale"])
    ref = run_attention(pkv, *args, kernel=1, num_ctas=1)
    got = run_attention(pkv, *args, kernel=1, num_ctas=num_ctas)
    check_close(got, oracle_attention(c, c["tables"], c["lens"]), rel=2e-5)
    rel = ((got - ref).norm() / ref.norm()).item()
    ma = (got - ref).abs().max().item()
    print(f"num_ctas={num_ctas}: relative L2 {rel:.2e}, max-abs {ma:.2e} against one CTA")
    assert rel <= 1e-6 and ma <= 1e-5, (rel, ma)


@pytest.mark.parametrize("kernel", [1, 2])
@pytest.mark.parametrize("num_ctas", [0, 5, 37, 300])
def test_many_short_segments_with_cost_placed_ranges(pkv, kernel, num_ctas):
    """CTA ranges are placed by cost (a segment shorter than 256 blocks costs
    more than its blocks), so a range may hold many whole short segments and
    few blocks, or a cut piece of a long one. 150 sequences of 1-40 tokens
    around three long ones, at several CTA counts and on both kernels: every
    row against the oracle, and the CTA counts agree with each other."""
    rng = np.random.default_rng(33)
    lens = rng.integers(1, 41, 150)
    lens[[7, 80, 149]] = [5000, 9000, 4200]
    c = cases.random_case(33, lens, 32, 8, 128, torch.bfloat16)
    args = (dev(c["q"]), dev(c["k_pool"]), dev(c["v_pool"]), c["tables"], c["lens"], c["scale"])
    got = run_attention(pkv, *args, kernel=kernel, num_ctas=num_ctas)
    assert pkv.pkv_device_status() == 0
    check_close(got, oracle_attention(c, c["tables"], c["lens"]))
    ref = run_attention(pkv, *args, kernel=kernel, num_ctas=1)
    assert (got.float() - ref.float()).abs().max().item() <= 2 ** -7


def test_block_relabelling_gives_identical_output(pkv):
    c = cases.random_case(31, [3, 18, 35, 700], 32, 8, 128, torch.bfloat16, extra_blocks=11)
    nb = c["k_pool"].shape[0]
    perm = np.random.default_rng(3).permutation(nb)
    kp2 = torch.empty_like(c["k_pool"])
    vp2 = torch.empty_like(c["v_pool"])
    kp2[torch.from_numpy(perm)] = c["k_pool"]
    vp2[torch.from_numpy(perm)] = c["v_pool"]
    t2 = np.where(c["tables"] >= 0, perm[np.maximum(c["tables"], 0)], -1).astype(np.int32)
    a = run_attention(pkv, dev(c["q"]), dev(c["k_pool"]), dev(c["v_pool"]), c["tables"], c["lens"], c["scale"])
    b = run_attention(pkv, dev(c["q"]), dev(kp2), dev(vp2), t2, c["lens"], c["scale"])
    assert torch.equal(a, b)


def test_closed_forms_on_gpu(pkv):
    # one token: out = v0 exactly (softmax weight 1)
    c = cases.random_case(32, [1, 1, 1], 32, 8, 128, torch.bfloat16)
    got = run_attention(pkv, dev(c["q"]), dev(c["k_pool"]), dev(c["v_pool"]), c["tables"], c["lens"], c["scale"])
    vp = c["v_pool"]
    for i in range(3):
        blk = int(c["tables"][i][0])
        want = vp[blk, :, 0, :].repeat_interleave(4, dim=0)
        assert torch.equal(got[i].cpu(), want)
    # equal keys: out = mean(V) of the live tokens
    c = cases.random_case(33, [37, 300], 16, 4, 128, torch.bfloat16)
    kp = c["k_pool"].clone()
    kp[:] = kp[0, 0, 0]
    got = run_attention(pkv, dev(c["q"]), dev(kp), dev(c["v_pool"]), c["tables"], c["lens"], c["scale"])
    want = oracle_attention(c, c["tables"], c["lens"], k_pool=kp)
    check_close(got, want)


def test_zero_length_context_gives_zero_rows(pkv):
    c = cases.random_case(34, [0, 50, 0, 3], 32, 8, 128, torch.bfloat16)
    out = torch.full((4, 32, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    got = run_attention(pkv, dev(c["q"]), dev(c["k_pool"]), dev(c["v_pool"]), c["tables"], c["lens"], c["scale"],
                        out=out)
    assert torch.all(got[0] == 0) and torch.all(got[2] == 0)
    check_close(got, oracle_attention(c, c["tables"], c["lens"]))


def test_large_batch_is_split_across_launches(pkv):
    lens = np.random.default_rng(35).integers(1, 60, size=2500)
    c = cases.random_case(35, lens, 8, 2, 64, torch.bfloat16)
    got = run_attention(pkv, dev(c["q"]), dev(c["k_pool"]), dev(c["v_pool"]), c["tables"], c["lens"], c["scale"])
    check_close(got, oracle_attention(c, c["tables"], c["lens"]))


# ------------------------------------------------------------------ errors
def test_checked_mode_rejects_without_writing(pkv):
    kp = dev(torch.randn(8, 2, 16, 64))
    vp = dev(torch.randn(8, 2, 16, 64))
    k0, v0 = kp.clone(), vp.clone()
    kn = dev(torch.randn(2, 2, 64))
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_append(kn, kn, dev(np.array([3, 8 * 16], np.int64)), kp, vp, flags=pkv.PKV_FLAG_CHECKED)
    assert e.value.name == "PKV_ERR_RANGE"
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_append(kn, kn, dev(np.array([5, 5], np.int64)), kp, vp, flags=pkv.PKV_FLAG_CHECKED)
    assert e.value.name == "PKV_ERR_OVERLAP"
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_copy_blocks(dev(np.array([[1, 2], [2, 3]], np.int64)), kp, vp, flags=pkv.PKV_FLAG_CHECKED)
    assert e.value.name == "PKV_ERR_OVERLAP"
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_copy_blocks(dev(np.array([[1, 9]], np.int64)), kp, vp, flags=pkv.PKV_FLAG_CHECKED)
    assert e.value.name == "PKV_ERR_RANGE"
    torch.cuda.synchronize()
    assert torch.equal(kp, k0) and torch.equal(vp, v0)
    # a valid checked call goes through
    pkv.pkv_append(kn, kn, dev(np.array([3, 4], np.int64)), kp, vp, flags=pkv.PKV_FLAG_CHECKED)
    assert torch.equal(kp[0, :, 3], kn[0])


def test_checked_decode_rejects_bad_tables_and_fast_mode_flags_them(pkv):
    c = cases.random_case(36, [20, 40], 4, 2, 64, torch.bfloat16)
    tables = c["tables"].copy()
    tables[1, 2] = 10 ** 6
    out = torch.full((2, 4, 64), 3.0, dtype=torch.bfloat16, device="cuda")
    args = (dev(c["q"]), dev(c["k_pool"]), dev(c["v_pool"]), tables, c["lens"], c["scale"])
    with pytest.raises(pkv.PkvError) as e:
        run_attention(pkv, *args, out=out, flags=pkv.PKV_FLAG_CHECKED)
    assert e.value.name == "PKV_ERR_RANGE"
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)
    pkv.pkv_device_status(clear=True)
    got = run_attention(pkv, *args)
    assert pkv.pkv_device_status(clear=True) & pkv.PKV_DEVERR_RANGE
    assert torch.all(torch.isfinite(got.float()))
    # the first sequence does not touch the bad entry and is still exact
    want = oracle_attention(c, c["tables"], c["lens"])
    ma, rl = cases.attention_errors(got[0], want[0])
    assert rl <= REL_L2


def test_host_side_rejections(pkv):
    c = cases.random_case(37, [20], 4, 2, 64, torch.bfloat16)
    q, kp, vp = dev(c["q"]), dev(c["k_pool"]), dev(c["v_pool"])
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_decode_attention(q, kp, vp, dev(c["tables"], torch.int32), dev(c["lens"], torch.int32), 0.1,
                                 workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.name == "PKV_ERR_WORKSPACE"
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_decode_attention(q, kp, vp, dev(c["tables"], torch.int32), dev(c["lens"], torch.int32),
                                 float("nan"))
    assert e.value.name == "PKV_ERR_SHAPE"
    with pytest.raises(pkv.PkvError) as e:   # the tensor-core kernel is bf16-only
        pkv.pkv_decode_attention(q.float(), kp.float(), vp.float(), dev(c["tables"], torch.int32),
                                 dev(c["lens"], torch.int32), 0.1, kernel=2)
    assert e.value.name == "PKV_ERR_UNSUPPORTED"


@pytest.mark.parametrize("num_ctas", [0, 37, 500])
def test_workspace_reuse_leaves_counters_zero(pkv, num_ctas):
    """The merge counters in the workspace are back at zero after every call,
    so one zero-filled workspace serves any number of calls identically."""
    c = cases.random_case(38, [100, 2000, 3, 517, 4096], 32, 8, 128, torch.bfloat16)
    q, kp, vp = dev(c["q"]), dev(c["k_pool"]), dev(c["v_pool"])
    tables, lens = dev(c["tables"], torch.int32), dev(c["lens"], torch.int32)
    need = pkv.pkv_decode_workspace_size(5, 32, c["tables"].shape[1], kp, num_ctas=num_ctas)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    outs = [pkv.pkv_decode_attention(q, kp, vp, tables, lens, c["scale"], workspace=ws, num_ctas=num_ctas)
            for _ in range(3)]
    torch.cuda.synchronize()
    counters = ws[256:256 + 5 * 8 * 4 * 4]
    assert torch.count_nonzero(counters).item() == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    check_close(outs[0], oracle_attention(c, c["tables"], c["lens"]))


@pytest.mark.parametrize("stages", [8, 12])
@pytest.mark.parametrize("shape", [0, 1, 2])
def test_ring_depths_agree(pkv, stages, shape):
    """Both ring depths of the tensor-core kernel give the oracle's result
    (the planner picks one; both must be correct)."""
    lens, qh, kvh, d = SHAPES[shape]
    c = cases.random_case(40 + shape, lens, qh, kvh, d, torch.bfloat16, poison=True)
    got = run_attention(pkv, dev(c["q"]), dev(c["k_pool"]), dev(c["v_pool"]), c["tables"], c["lens"],
                        c["scale"], kernel=2, stages=stages, num_ctas=37)
    check_close(got, oracle_attention(c, c["tables"], c["lens"]))


@pytest.mark.parametrize("kernel,q_heads,kv_heads,head_dim", [
    (1, 32, 2, 128),   # G = 16: a warp slice spans four heads
    (1, 12, 1, 64),    # G = 12
    (1, 6, 1, 128),    # G = 6: slices cut heads in half
    (2, 6, 1, 128),
    (2, 3, 1, 64),     # G = 3
    (2, 5, 1, 128),    # G = 5
])
def test_group_sizes_with_cut_segments(pkv, kernel, q_heads, kv_heads, head_dim):
    """Group sizes whose warp slices do not align with heads, with segments
    cut across many CTAs so that every piece goes through the merge."""
    c = cases.random_case(50 + q_heads, [700, 33, 2000, 1], q_heads, kv_heads, head_dim, torch.bfloat16,
                          poison=True)
    for num_ctas in (1, 23, 181):
        got = run_attention(pkv, dev(c["q"]), dev(c["k_pool"]), dev(c["v_pool"]), c["tables"], c["lens"],
                            c["scale"], kernel=kernel, num_ctas=num_ctas)
        check_close(got, oracle_attention(c, c["tables"], c["lens"]))


def test_bounded_wait_runs_out_and_is_reported(pkv):
    """Failure detection: with the stall hook the producer issues nothing, the
    consumers' bounded waits run out, the kernel returns and the sticky
    status says so; the context stays usable for the next call."""
    c = cases.random_case(71, [300, 40, 1000], 32, 8, 128, torch.bfloat16)
    args = (dev(c["q"]), dev(c["k_pool"]), dev(c["v_pool"]), c["tables"], c["lens"], c["scale"])
    pkv.pkv_device_status(clear=True)
    run_attention(pkv, *args, kernel=2, flags=pkv.PKV_FLAG_TEST_STALL)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status(clear=True) & pkv.PKV_DEVERR_TIMEOUT
    got = run_attention(pkv, *args, kernel=2)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status(clear=True) == 0
    check_close(got, oracle_attention(c, c["tables"], c["lens"]))
    with pytest.raises(pkv.PkvError) as e:      # the hook exists for the tensor-core kernel only
        run_attention(pkv, *args, kernel=1, flags=pkv.PKV_FLAG_TEST_STALL)
    assert e.value.name == "PKV_ERR_UNSUPPORTED"


def test_checked_decode_rejects_a_zero_length_context(pkv):
    """A context of length 0 is no decode query: checked mode rejects it with
    PKV_ERR_RANGE and writes nothing; the default mode writes a zero row."""
    c = cases.random_case(37, [20, 0, 40], 8, 2, 128, torch.bfloat16)
    args = (dev(c["q"]), dev(c["k_pool"]), dev(c["v_pool"]), c["tables"], c["lens"], c["scale"])
    out = torch.full((3, 8, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        run_attention(pkv, *args, out=out, flags=pkv.PKV_FLAG_CHECKED)
    assert e.value.name == "PKV_ERR_RANGE"
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)
    got = run_attention(pkv, *args, out=out)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status(clear=True) == 0
    assert torch.all(got[1] == 0)
    check_close(got, oracle_attention(c, c["tables"], c["lens"]))


def test_device_status_is_shared_by_streams_and_sticky(pkv):
    """The sticky status is one word per device: a bit set by a call on one
    stream is seen from another stream, no later call clears it (successful
    or not), and only an explicit clear resets it."""
    c = cases.random_case(38, [20, 40], 4, 2, 64, torch.bfloat16)
    bad = c["tables"].copy()
    bad[1, 2] = 10 ** 6
    a, b = torch.cuda.Stream(), torch.cuda.Stream()
    args = (dev(c["q"]), dev(c["k_pool"]), dev(c["v_pool"]))
    torch.cuda.synchronize()
    pkv.pkv_device_status(clear=True)
    with torch.cuda.stream(a):
        run_attention(pkv, *args, bad, c["lens"], c["scale"], stream=a)
    a.synchronize()
    with torch.cuda.stream(b):
        good = run_attention(pkv, *args, c["tables"], c["lens"], c["scale"], stream=b)
    assert pkv.pkv_device_status(clear=False, stream=b) & pkv.PKV_DEVERR_RANGE
    with torch.cuda.stream(b):
        run_attention(pkv, *args, c["tables"], c["lens"], c["scale"], stream=b)
    assert pkv.pkv_device_status(clear=False, stream=a) & pkv.PKV_DEVERR_RANGE
    assert pkv.pkv_device_status(clear=True, stream=b) & pkv.PKV_DEVERR_RANGE
    assert pkv.pkv_device_status(clear=False, stream=a) == 0
    check_close(good, oracle_attention(c, c["tables"], c["lens"]))
