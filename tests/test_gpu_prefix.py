"""Shared-prefix (two-phase) decode through the C ABI against the oracle.

The prefixed call must give, for every row, what softmax attention over the
sequence's whole context gives (the float64 single-pass oracle), within the
decode tolerance; the oracle's own two-phase restatement is checked against
the same rows. Cases cover one and several groups, sequences in no group,
groups that share no blocks, members whose context is only the shared
blocks, group sizes whose query rows leave ragged 64-row tiles, shared runs
that split over several chunks and ones that fit in one, forced CTA counts
for the suffix pass (cut segments whose merge feeds the fold), batches above
one launch, malformed groups (flagged, results still right), checked mode,
and the calls that reduce to the plain decode.
"""

import numpy as np
import pytest
import torch

import cases
from oracle import attention as OA
from oracle import prefix as OP

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
                group=torch.from_numpy(c["prefix_group"]).to(d), blocks=torch.from_numpy(c["group_blocks"]).to(d))


def oracle_rows(c, dtype="bf16"):
    return OA.decode_attention(cases.host_view(c["q"]), cases.host_view(c["k_pool"]), cases.host_view(c["v_pool"]),
                               c["tables"], c["lens"], c["scale"], c["kv_heads"], dtype)


def run(pkv, c, d, max_group_blocks=None, **kw):
    mgb = int(c["group_blocks"].max()) if max_group_blocks is None and len(c["group_blocks"]) else (max_group_blocks or 0)
    out = pkv.pkv_decode_attention_prefixed(d["q"], d["k"], d["v"], d["tables"], d["lens"], c["scale"], d["group"],
                                            d["blocks"], mgb, **kw)
    torch.cuda.synchronize()
    return out


def check(out, want):
    ma, rl = cases.attention_errors(out, want)
    assert ma <= MAX_ABS and rl <= REL_L2, (ma, rl)


CASES = {
    # name: (member_of, group_blocks, suffix seed/max, q_heads, kv_heads, head_dim)
    "one_group_g4_d128": ([0] * 12, [40], 100, 32, 8, 128),
    "two_groups_and_plain_g8_d64": ([0, 1, -1, 0, 1, 1, -1, 0, 0], [9, 23], 70, 16, 2, 64),
    "g1_full_tile": ([0] * 70, [6], 40, 2, 2, 128),
    "g3_ragged_tiles": ([0] * 30 + [1] * 7, [17, 3], 50, 6, 2, 128),
    "g5": ([0] * 14, [11], 33, 10, 2, 64),
    "g6_two_groups": ([1, 0] * 9, [5, 12], 20, 12, 2, 128),
    "g7": ([0] * 10 + [-1] * 3, [8], 64, 7, 1, 64),
    "empty_suffixes": ([0] * 6, [20], 0, 8, 2, 128),
    "group_without_blocks": ([0, 1, 1, 0], [0, 4], 30, 8, 2, 128),
    "unused_group": ([2, 2, 2, -1], [7, 3, 5], 25, 32, 8, 128),
}


@pytest.mark.parametrize("prefix_kernel", [1, 2])
@pytest.mark.parametrize("name", sorted(CASES))
def test_prefixed_matches_oracle(pkv, name, prefix_kernel):
    member_of, gb, smax, hq, hkv, d = CASES[name]
    rng = np.random.default_rng(len(name))
    suffix = rng.integers(0, smax + 1, len(member_of)) if smax else np.zeros(len(member_of), dtype=np.int64)
    c = cases.grouped_case(len(name) * 3 + 1, member_of, gb, suffix, hq, hkv, d, torch.bfloat16)
    dv = dev(c)
    out = run(pkv, c, dv, prefix_kernel=prefix_kernel)
    assert pkv.pkv_device_status(clear=True) == 0
    want = oracle_rows(c)
    check(out, want)
    two = OP.decode_attention_two_phase(cases.host_view(c["q"]), cases.host_view(c["k_pool"]),
                                        cases.host_view(c["v_pool"]), c["tables"], c["lens"], c["scale"], hkv,
                                        "bf16", c["prefix_group"], c["group_blocks"])
    check(out, two)


@pytest.mark.parametrize("prefix_kernel", [1, 2])
@pytest.mark.parametrize("num_ctas", [3, 40, 5000])
@pytest.mark.parametrize("max_group_blocks", [None, 60, 80])
def test_split_counts_and_chunking(pkv, num_ctas, max_group_blocks, prefix_kernel):
    """Forced CTA counts cut the own-token segments across CTAs (their merge
    writes the fold); a looser bound on the shared blocks changes how they are
    chunked. Same rows every time."""
    member_of = [0] * 9 + [1] * 5 + [-1] * 2
    suffix = np.random.default_rng(5).integers(1, 300, len(member_of))
    c = cases.grouped_case(77, member_of, [45, 2], suffix, 32, 8, 128, torch.bfloat16, width=80)
    dv = dev(c)
    out = run(pkv, c, dv, max_group_blocks=max_group_blocks, num_ctas=num_ctas, prefix_kernel=prefix_kernel)
    assert pkv.pkv_device_status(clear=True) == 0
    check(out, oracle_rows(c))


def test_workspace_reuse(pkv):
    """Counters must be back at zero after each call: a second call on the
    same workspace with other inputs is still right."""
    member_of = [0] * 8 + [-1]
    c1 = cases.grouped_case(5, member_of, [30], np.full(9, 17), 32, 8, 128, torch.bfloat16)
    c2 = cases.grouped_case(6, member_of, [30], np.full(9, 40), 32, 8, 128, torch.bfloat16)
    d1, d2 = dev(c1), dev(c2)
    need = pkv.pkv_decode_prefixed_workspace_size(9, 32, c1["tables"].shape[1], 1, 30, d1["k"])
    need = max(need, pkv.pkv_decode_prefixed_workspace_size(9, 32, c2["tables"].shape[1], 1, 30, d2["k"]))
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        for c, d in ((c1, d1), (c2, d2)):
            check(run(pkv, c, d, workspace=ws), oracle_rows(c))


def test_batch_above_one_launch(pkv):
    """1100 sequences: the call splits at 1024; a group spans the split."""
    member_of = [0] * 600 + [1] * 300 + [-1] * 50 + [0] * 150
    suffix = np.random.default_rng(9).integers(0, 40, len(member_of))
    c = cases.grouped_case(31, member_of, [5, 3], suffix, 8, 2, 64, torch.bfloat16)
    out = run(pkv, c, dev(c))
    assert pkv.pkv_device_status(clear=True) == 0
    check(out, oracle_rows(c))


def test_malformed_groups_flag_and_stay_right(pkv):
    """A group id past num_groups, and a group longer than a member's
    context, make those sequences plain: PKV_DEVERR_RANGE is set and every
    row is still the single-pass result."""
    member_of = [0, 0, 0, 0]
    c = cases.grouped_case(12, member_of, [6], [5, 9, 0, 30], 8, 2, 128, torch.bfloat16)
    c["prefix_group"] = np.array([0, 3, 0, 0], dtype=np.int32)          # 3 >= num_groups
    c["lens"] = c["lens"].copy()
    c["lens"][2] = 80                                                   # 5 whole blocks < 6 shared
    out = run(pkv, c, dev(c))
    assert pkv.pkv_device_status(clear=True) & 2
    check(out, oracle_rows(c))


def test_checked_mode_rejects_and_writes_nothing(pkv):
    member_of = [0, 0, 0, -1]
    c = cases.grouped_case(13, member_of, [4], [3, 20, 7, 9], 8, 2, 128, torch.bfloat16)
    d = dev(c)
    assert run(pkv, c, d, flags=pkv.PKV_FLAG_CHECKED) is not None
    bad = c["tables"].copy()
    bad[2, 1] = bad[3, 0]                      # member 2 does not begin with the group's blocks
    d["tables"] = torch.from_numpy(bad).cuda()
    out = torch.full_like(d["q"], 7.0)
    with pytest.raises(pkv.PkvError) as e:
        run(pkv, c, d, out=out, flags=pkv.PKV_FLAG_CHECKED)
    assert e.value.name == "PKV_ERR_RANGE"
    assert bool((out == 7.0).all())
    d["tables"] = torch.from_numpy(c["tables"]).cuda()
    d["blocks"] = torch.tensor([5], dtype=torch.int32, device="cuda")  # above max_group_blocks
    with pytest.raises(pkv.PkvError) as e:
        run(pkv, c, d, max_group_blocks=4, out=out, flags=pkv.PKV_FLAG_CHECKED)
    assert e.value.name == "PKV_ERR_RANGE"
    assert bool((out == 7.0).all())


def test_reduces_to_plain_call(pkv):
    """No groups, or a cache only the CUDA-core kernel serves: the plain decode, bit for bit."""
    member_of = [0, 0, -1]
    c = cases.grouped_case(14, member_of, [3], [4, 30, 10], 8, 2, 64, torch.bfloat16)
    d = dev(c)
    plain = pkv.pkv_decode_attention(d["q"], d["k"], d["v"], d["tables"], d["lens"], c["scale"])
    none = pkv.pkv_decode_attention_prefixed(d["q"], d["k"], d["v"], d["tables"], d["lens"], c["scale"],
                                             d["group"], d["blocks"][:0], 0)
    assert torch.equal(plain, none)
    cf = cases.grouped_case(14, member_of, [3], [4, 30, 10], 8, 2, 64, torch.float32)
    df = dev(cf)
    plain = pkv.pkv_decode_attention(df["q"], df["k"], df["v"], df["tables"], df["lens"], cf["scale"])
    grp = run(pkv, cf, df)
    assert torch.equal(plain, grp)
    check(grp, oracle_rows(cf, "f32"))


def test_host_rejections(pkv):
    c = cases.grouped_case(15, [0, 0], [2], [1, 2], 8, 2, 128, torch.bfloat16)
    d = dev(c)
    with pytest.raises(pkv.PkvError) as e:
        run(pkv, c, d, max_group_blocks=c["tables"].shape[1] + 1)
    assert e.value.name == "PKV_ERR_SHAPE"
    many = torch.zeros(1025, dtype=torch.int32, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_decode_attention_prefixed(d["q"], d["k"], d["v"], d["tables"], d["lens"], c["scale"], d["group"],
                                          many, 2)
    assert e.value.name == "PKV_ERR_UNSUPPORTED"


@pytest.mark.parametrize("d,hq,hkv", [(128, 32, 8), (64, 16, 2)])
def test_two_chunk_first_kernels_agree(pkv, d, hq, hkv):
    """The tcgen05 and the mma.sync chunk-first kernels on the same rows:
    two implementations of one pass (many members, a long shared run)."""
    member_of = [0] * 40 + [1] * 9 + [-1] * 3
    suffix = np.random.default_rng(3).integers(0, 90, len(member_of))
    c = cases.grouped_case(91, member_of, [70, 13], suffix, hq, hkv, d, torch.bfloat16)
    dv = dev(c)
    a = run(pkv, c, dv, prefix_kernel=1)
    b = run(pkv, c, dv, prefix_kernel=2)
    assert pkv.pkv_device_status(clear=True) == 0
    diff = (a.float() - b.float())
    assert diff.abs().max().item() <= 1e-2 and (diff.norm() / a.float().norm()).item() <= 2e-3
    check(b, oracle_rows(c))
