"""Multi-query (causal) paged attention through the C ABI against the oracle.

Calls with up to 32 query rows per (sequence, KV head) run on the split
decode kernel; more rows (a chunked prefill) on the tensor-core tile kernel.

Every output row is compared with the float64 oracle (query t of a sequence
with n tokens and nq queries attends to tokens 0 .. n - nq + t). Cases cover
group sizes 1-8, head_dim 64 and 128, query counts 0 to max_query_len per
sequence, contexts that are all queries (a whole prompt), contexts inside
one block, ragged lengths, forced CTA counts that cut segments (their merge),
batches above one launch, workspace reuse, malformed query ranges (flagged,
other rows right) and checked mode; one query per sequence is also checked
against the decode kernel.
"""

import numpy as np
import pytest
import torch

import cases
from oracle import multiquery as OM

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2 = 1e-2, 2e-3


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_209_gb300 import pkv as P
    P.load_library()
    return P


def dev(c):
    d = torch.device("cuda", 0)
    return dict(q=c["q"].to(d), k=c["k_pool"].to(d), v=c["v_pool"].to(d),
                tables=torch.from_numpy(c["tables"]).to(d), lens=torch.from_numpy(c["lens"]).to(d),
                qs=torch.from_numpy(c["query_start"]).to(d))


def want(c):
    return OM.multiquery_attention(cases.host_view(c["q"]), cases.host_view(c["k_pool"]),
                                   cases.host_view(c["v_pool"]), c["tables"], c["lens"], c["query_start"],
                                   c["scale"], c["kv_heads"], "bf16")


def run(pkv, c, d, mql, **kw):
    out = pkv.pkv_multiquery_attention(d["q"], d["k"], d["v"], d["tables"], d["lens"], d["qs"], c["scale"], mql, **kw)
    torch.cuda.synchronize()
    return out


def check(out, ref):
    ma, rl = cases.attention_errors(out, ref)
    assert ma <= MAX_ABS and rl <= REL_L2, (ma, rl)


CASES = {
    # name: (lens, query counts, q_heads, kv_heads, head_dim, max_query_len)
    "spec4_llama": ([300, 17, 64, 1000, 5], [4, 4, 4, 4, 4], 32, 8, 128, 4),
    "ragged_counts_g4": ([40, 33, 16, 200, 7, 90], [0, 3, 8, 1, 7, 5], 8, 2, 128, 8),
    "g8_d64": ([129, 48, 500, 3], [2, 4, 3, 3], 16, 2, 64, 4),
    "g1_whole_prompts": ([20, 32, 31], [20, 32, 31], 2, 2, 64, 32),
    "g3": ([77, 64, 12, 400], [10, 1, 10, 6], 6, 2, 128, 10),
    "single_block_contexts": ([1, 2, 15, 16], [1, 2, 8, 8], 8, 2, 128, 8),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_multiquery_matches_oracle(pkv, name):
    lens, nqs, hq, hkv, d, mql = CASES[name]
    c = cases.multiquery_case(len(name), lens, nqs, hq, hkv, d, torch.bfloat16)
    out = run(pkv, c, dev(c), mql)
    assert pkv.pkv_device_status(clear=True) == 0
    check(out, want(c))


@pytest.mark.parametrize("num_ctas", [3, 40, 5000])
def test_cut_segments(pkv, num_ctas):
    """Forced CTA counts cut (sequence, KV head) segments across CTAs; every
    warp's pieces are merged by the last one to finish."""
    lens, nqs = [1200, 333, 40, 2048], [4, 2, 4, 3]
    c = cases.multiquery_case(9, lens, nqs, 32, 8, 128, torch.bfloat16)
    out = run(pkv, c, dev(c), 4, num_ctas=num_ctas)
    assert pkv.pkv_device_status(clear=True) == 0
    check(out, want(c))


def test_one_query_per_sequence_is_decode(pkv):
    c = cases.multiquery_case(10, [70, 1, 512, 33], [1, 1, 1, 1], 32, 8, 128, torch.bfloat16)
    d = dev(c)
    mq = run(pkv, c, d, 1)
    dec = pkv.pkv_decode_attention(d["q"], d["k"], d["v"], d["tables"], d["lens"], c["scale"])
    diff = (mq.float() - dec.float())
    assert diff.abs().max().item() <= 1e-2 and (diff.norm() / dec.float().norm()).item() <= 2e-3
    check(mq, want(c))


def test_batch_above_one_launch_and_reuse(pkv):
    rng = np.random.default_rng(11)
    lens = rng.integers(1, 120, 1100)
    nqs = np.minimum(lens, rng.integers(0, 5, 1100))
    c = cases.multiquery_case(12, lens, nqs, 8, 2, 64, torch.bfloat16)
    d = dev(c)
    need = pkv.pkv_multiquery_workspace_size(1100, 8, c["tables"].shape[1], 4, d["k"])
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    ref = want(c)
    for _ in range(2):
        out = run(pkv, c, d, 4, workspace=ws)
        assert pkv.pkv_device_status(clear=True) == 0
        check(out, ref)


def test_malformed_query_ranges(pkv):
    """A sequence asking for more queries than it has tokens (or than
    max_query_len) gets no rows and sets PKV_DEVERR_RANGE; the other rows are
    right. Checked mode rejects the call and writes nothing."""
    c = cases.multiquery_case(13, [30, 3, 50], [2, 4, 2], 8, 2, 128, torch.bfloat16)   # 4 > 3 tokens
    d = dev(c)
    out = torch.full_like(d["q"], 5.0)
    run(pkv, c, d, 4, out=out)
    assert pkv.pkv_device_status(clear=True) & 2
    good = np.r_[0:2, 6:8]
    ref = want(dict(c, lens=np.array([30, 3, 50]), query_start=np.array([0, 2, 2, 4]),
                    q=torch.cat([c["q"][0:2], c["q"][6:8]])))
    check(out[torch.from_numpy(good).cuda()], ref)
    out2 = torch.full_like(d["q"], 5.0)
    with pytest.raises(pkv.PkvError) as e:
        run(pkv, c, d, 4, out=out2, flags=pkv.PKV_FLAG_CHECKED)
    assert e.value.name == "PKV_ERR_RANGE"
    assert bool((out2 == 5.0).all())


def test_host_rejections(pkv):
    c = cases.multiquery_case(14, [30, 40], [2, 2], 32, 8, 128, torch.bfloat16)
    d = dev(c)
    with pytest.raises(pkv.PkvError) as e:
        run(pkv, c, d, 65537, workspace=torch.zeros(256, dtype=torch.uint8, device="cuda"))
    assert e.value.name == "PKV_ERR_UNSUPPORTED"
    cf = cases.multiquery_case(14, [30, 40], [2, 2], 8, 2, 64, torch.float32)
    with pytest.raises(pkv.PkvError) as e:
        run(pkv, cf, dev(cf), 2)
    assert e.value.name == "PKV_ERR_DTYPE"


PREFILL = {
    # name: (lens, query counts, q_heads, kv_heads, head_dim, max_query_len) -- more than 32 rows
    "llama_ragged": ([300, 129, 1000, 64], [40, 129, 300, 64], 32, 8, 128, 300),
    "g8_d64": ([500, 77], [200, 77], 16, 2, 64, 200),
    "g1_whole_prompts": ([90, 33, 1], [90, 33, 1], 8, 8, 128, 90),
    "zero_queries": ([256, 40, 700], [100, 0, 37], 32, 8, 128, 100),
    "long_context_two_tiles": ([4000, 2500], [64, 33], 32, 8, 128, 64),
}


@pytest.mark.parametrize("name", sorted(PREFILL))
def test_prefill_matches_oracle(pkv, name):
    """Chunked prefill (tensor-core tiles): every output row against the
    float64 oracle."""
    lens, nqs, hq, hkv, d, mql = PREFILL[name]
    c = cases.multiquery_case(len(name) + 50, lens, nqs, hq, hkv, d, torch.bfloat16)
    out = run(pkv, c, dev(c), mql)
    assert pkv.pkv_device_status(clear=True) == 0
    check(out, want(c))


@pytest.mark.parametrize("hq,hkv,mql", [(64, 2, 1), (64, 2, 3), (128, 1, 2)])
def test_large_query_groups(pkv, hq, hkv, mql):
    """32 and 128 query heads per KV head: 32 rows per (sequence, KV head)
    still run on the split kernel, more on the tile kernel, where one query's
    heads fill whole tiles."""
    c = cases.multiquery_case(90 + hq + mql, [300, 17, 900], [mql] * 3, hq, hkv, 128, torch.bfloat16, poison=True)
    out = run(pkv, c, dev(c), mql)
    assert pkv.pkv_device_status(clear=True) == 0
    check(out, want(c))


def test_prefill_path_agrees_with_split_kernel(pkv):
    """The same 16-row call through both paths: max_query_len 4 (16 rows,
    split decode kernel) and 9 (36 rows, tensor-core tiles)."""
    c = cases.multiquery_case(61, [700, 40, 129, 2000], [4, 4, 3, 4], 32, 8, 128, torch.bfloat16)
    d = dev(c)
    a = run(pkv, c, d, 4)
    b = run(pkv, c, d, 9)
    assert pkv.pkv_device_status(clear=True) == 0
    diff = a.float() - b.float()
    assert diff.abs().max().item() <= 1e-2 and (diff.norm() / a.float().norm()).item() <= 2e-3
    check(b, want(c))


@pytest.mark.parametrize("mql", [4, 40])
def test_poisoned_tail_slots(pkv, mql):
    """Slots past every context (the rest of each last block, spare blocks)
    hold K = NaN and V = -inf: a masked token must contribute nothing, not
    0 * NaN. 4 queries per sequence run on the split kernel, 40 on the tiles;
    no length is a multiple of 16."""
    lens = [300, 17, 1001, 45, 130]
    c = cases.multiquery_case(66 + mql, lens, [min(mql, n) for n in lens], 32, 8, 128, torch.bfloat16,
                              poison=True)
    out = run(pkv, c, dev(c), mql)
    assert pkv.pkv_device_status(clear=True) == 0
    assert bool(torch.isfinite(out).all())
    check(out, want(c))


def test_prefill_malformed_query_ranges(pkv):
    """A sequence asking for more queries than it has tokens gets no rows and
    sets PKV_DEVERR_RANGE; the other rows are right; checked mode rejects."""
    c = cases.multiquery_case(62, [80, 30, 90], [40, 50, 33], 8, 2, 128, torch.bfloat16)   # 50 > 30 tokens
    d = dev(c)
    out = torch.full_like(d["q"], 5.0)
    run(pkv, c, d, 50, out=out)
    assert pkv.pkv_device_status(clear=True) & 2
    keep = np.r_[0:40, 90:123]
    ref = want(dict(c, lens=np.array([80, 90]), query_start=np.array([0, 40, 73]),
                    q=torch.cat([c["q"][0:40], c["q"][90:123]]), tables=c["tables"][[0, 2]]))
    check(out[torch.from_numpy(keep).cuda()], ref)
    out2 = torch.full_like(d["q"], 5.0)
    with pytest.raises(pkv.PkvError) as e:
        run(pkv, c, d, 50, out=out2, flags=pkv.PKV_FLAG_CHECKED)
    assert e.value.name == "PKV_ERR_RANGE"
    assert bool((out2 == 5.0).all())


def test_prefill_batch_above_one_launch(pkv):
    """More than 1024 sequences on the tile path: the call runs one launch per
    1024 sequences, with absolute query rows."""
    rng = np.random.default_rng(63)
    lens = rng.integers(9, 60, 1030)
    nqs = np.minimum(lens, rng.integers(0, 10, 1030))
    c = cases.multiquery_case(64, lens, nqs, 8, 2, 64, torch.bfloat16)
    out = run(pkv, c, dev(c), 9)          # 9 queries x 4 heads = 36 rows: the tile path
    assert pkv.pkv_device_status(clear=True) == 0
    check(out, want(c))


def test_bounded_wait_runs_out_and_is_reported(pkv):
    """Failure detection in the split kernel: with the stall hook its producer
    issues nothing, every consumer wait runs out (20 ms), the kernel returns
    and the sticky status says so; the next call on the same context and
    workspace is right. The tile path has no hook and rejects the flag."""
    c = cases.multiquery_case(65, [300, 40, 900], [4, 4, 2], 32, 8, 128, torch.bfloat16)
    d = dev(c)
    ws = torch.zeros(pkv.pkv_multiquery_workspace_size(3, 32, c["tables"].shape[1], 4, d["k"]), dtype=torch.uint8,
                     device="cuda")
    pkv.pkv_device_status(clear=True)
    run(pkv, c, d, 4, workspace=ws, flags=pkv.PKV_FLAG_TEST_STALL)
    assert pkv.pkv_device_status(clear=True) & pkv.PKV_DEVERR_TIMEOUT
    out = run(pkv, c, d, 4, workspace=ws)
    assert pkv.pkv_device_status(clear=True) == 0
    check(out, want(c))
    with pytest.raises(pkv.PkvError) as e:
        run(pkv, c, d, 9, flags=pkv.PKV_FLAG_TEST_STALL)
    assert e.value.name == "PKV_ERR_UNSUPPORTED"


@pytest.mark.parametrize("slope", [10.0, 3.0])
def test_prefill_running_maximum_moves_every_step(pkv, slope):
    """Scores that climb along the context, so that the tile kernel's running
    maximum moves past its lazy-rescale threshold in (nearly) every 64-token
    step, at both positions of the issuer's step pairs: O and a waiting P are
    rescaled. slope: base-2 logit increase per 32 tokens."""
    c = cases.multiquery_case(81, [1100, 700], [40, 33], 8, 2, 128, torch.bfloat16)
    k = c["k_pool"].float()
    q = c["q"].float()
    scale = c["scale"]
    # dimension 0 of q is 20 everywhere; dimension 0 of the token at logical position t is
    # slope / (log2(e) * scale * 20) * (t // 32), so logit_t = slope * (t // 32) / log2(e) + noise
    q[:, :, 0] = 20.0
    step = slope / (1.4426950408889634 * scale * 20.0)
    for i, n in enumerate(c["lens"]):
        for t in range(int(n)):
            blk, off = int(c["tables"][i, t // 16]), t % 16
            k[blk, :, off, 0] = step * (t // 32)
    c["k_pool"] = k.to(torch.bfloat16)
    c["q"] = q.to(torch.bfloat16)
    d = dev(c)
    out = run(pkv, c, d, 40)
    assert pkv.pkv_device_status(clear=True) == 0
    check(out, want(c))


@pytest.mark.parametrize("scale", [-0.125, 0.0, 3.0])
@pytest.mark.parametrize("mql", [4, 40])
def test_scale_sign_and_zero(pkv, scale, mql):
    """A negative scale (the largest weight sits at the smallest raw score),
    a zero scale (every visible token weighs the same: the output is the mean
    of the visible V rows) and a large one, on the split kernel (4 queries per
    sequence) and on the tensor-core tiles (40): every row against the
    oracle with that scale. At scale 3 the weights are nearly one-hot, so an
    output row is close to a single V row (entries up to ~5.5): the bf16
    rounding of a value in [4, 8) alone is up to 0.0156, above 1e-2, so the
    max-abs bar is taken relative to the largest output, as for the int8
    cache's wide scales; the relative L2 bar is unchanged."""
    c = cases.multiquery_case(70 + mql, [300, 129, 1000, 64], [mql] * 4, 32, 8, 128, torch.bfloat16)
    c["scale"] = scale
    out = run(pkv, c, dev(c), mql)
    assert pkv.pkv_device_status(clear=True) == 0
    assert bool(torch.isfinite(out.float()).all())
    ref = want(c)
    ma, rl = cases.attention_errors(out, ref)
    assert ma <= MAX_ABS * max(1.0, float(np.abs(ref).max())) and rl <= REL_L2, (ma, rl)
