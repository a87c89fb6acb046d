"""Pins of the two-phase (shared-prefix) decode oracle, and planted mistakes
that must fail one of them.

The two-phase result must equal single-pass softmax attention over each
sequence's whole context (the identity behind the ChunkAttention abstract's
two-phase partition: softmax over a union of token sets is the log-sum-exp
combination of the softmaxes over the parts). The single-pass oracle is
pinned separately (closed forms, SDPA, brute force); the partial and the
combination are pinned here by closed forms.
"""

import numpy as np
import pytest

import oracle.prefix as P
from oracle import attention as OA


def grouped_case(seed, batch=7, kv_heads=2, G=3, d=16, groups=((0, 3), (1, 0)), members=None,
                 suffix_max=40, dtype="f32"):
    """Random pools and tables where the members of each group share the
    group's first blocks. ``groups`` lists (group id, shared blocks)."""
    rng = np.random.default_rng(seed)
    nb_total = 64
    perm = list(rng.permutation(nb_total))
    shared_ids = {g: [perm.pop() for _ in range(nb)] for g, nb in groups}
    group_blocks = [nb for _, nb in sorted(groups)]
    if members is None:
        members = [int(x) for x in rng.integers(-1, len(groups), batch)]
    lens, tables = [], []
    width = 12
    for i in range(batch):
        g = members[i]
        head = shared_ids[g] if g >= 0 else []
        n = len(head) * 16 + int(rng.integers(0, suffix_max + 1))
        own = [perm.pop() for _ in range(-(-n // 16) - len(head))]
        row = head + own
        tables.append(row + [-1] * (width - len(row)))
        lens.append(n)
    q = rng.standard_normal((batch, kv_heads * G, d))
    kp = rng.standard_normal((nb_total, kv_heads, 16, d))
    vp = rng.standard_normal((nb_total, kv_heads, 16, d))
    if dtype == "f32":
        q, kp, vp = (x.astype(np.float32) for x in (q, kp, vp))
    return q, kp, vp, np.array(tables), np.array(lens), members, group_blocks


def pin_two_phase_equals_single_pass():
    for seed in range(6):
        q, kp, vp, tables, lens, members, gb = grouped_case(seed)
        a = P.decode_attention_two_phase(q, kp, vp, tables, lens, 0.3, 2, "f32", members, gb)
        b = OA.decode_attention(q, kp, vp, tables, lens, 0.3, 2, "f32")
        assert np.max(np.abs(a - b)) < 1e-12, seed


def pin_edge_groups():
    # every sequence in one group; one member with an empty suffix; a group with no shared blocks
    q, kp, vp, tables, lens, members, gb = grouped_case(11, batch=5, groups=((0, 2), (1, 0)),
                                                        members=[0, 0, 1, 0, 1], suffix_max=0)
    assert all(lens[i] == 32 for i in (0, 1, 3))
    a = P.decode_attention_two_phase(q, kp, vp, tables, lens, 0.5, 2, "f32", members, gb)
    b = OA.decode_attention(q, kp, vp, tables, lens, 0.5, 2, "f32")
    assert np.max(np.abs(a - b)) < 1e-12


def pin_partial_closed_form():
    s, a = 0.7, 1.3
    e1 = np.zeros(4)
    e1[0] = 1.0
    K = np.stack([e1, np.zeros(4), -e1])
    V = np.arange(12, dtype=np.float64).reshape(3, 4)
    o, lse = P.partial_attention(a * e1, K, V, s)
    z = np.exp(s * a) + 1.0 + np.exp(-s * a)
    assert abs(lse[0] - np.log(z)) < 1e-14
    want = (np.exp(s * a) * V[0] + V[1] + np.exp(-s * a) * V[2]) / z
    assert np.max(np.abs(o[0] - want)) < 1e-13
    o0, l0 = P.partial_attention(np.ones((2, 4)), K[:0], V[:0], s)
    assert np.all(o0 == 0) and np.all(l0 == -np.inf)


def pin_combine_closed_forms():
    o1, o2 = np.array([[1.0, 2.0]]), np.array([[3.0, 6.0]])
    assert np.allclose(P.combine_partials([(o1, np.array([0.4])), (o2, np.array([0.4]))]), [[2.0, 4.0]])
    assert np.allclose(P.combine_partials([(o1, np.array([-np.inf])), (o2, np.array([5.0]))]), o2)
    w = np.array([np.log(3.0)])            # weights 3 : 1
    assert np.allclose(P.combine_partials([(o1, w), (o2, np.array([0.0]))]), [[1.5, 3.0]])
    assert np.all(P.combine_partials([(o1, np.array([-np.inf])), (o2, np.array([-np.inf]))]) == 0)


def pin_member_permutation():
    q, kp, vp, tables, lens, members, gb = grouped_case(5, members=[0, 0, 0, -1, 1, 0, 1])
    a = P.decode_attention_two_phase(q, kp, vp, tables, lens, 0.3, 2, "f32", members, gb)
    order = [5, 1, 2, 3, 6, 0, 4]
    b = P.decode_attention_two_phase(q[order], kp, vp, tables[order], lens[order], 0.3, 2, "f32",
                                     [members[i] for i in order], gb)
    assert np.max(np.abs(a[order] - b)) < 1e-12


def pin_check_groups_rejects():
    q, kp, vp, tables, lens, members, gb = grouped_case(3, members=[0, 0, -1, 0, 1, 1, 0])
    P.check_groups(tables, lens, members, gb)
    bad = tables.copy()
    bad[3, 1] = bad[2, 0]
    with pytest.raises(ValueError):
        P.check_groups(bad, lens, members, gb)
    with pytest.raises(ValueError):
        P.check_groups(tables, lens, members, [gb[0] + 40, gb[1]])
    with pytest.raises(ValueError):
        P.check_groups(tables, lens, [5] + members[1:], gb)


PINS = [pin_two_phase_equals_single_pass, pin_edge_groups, pin_partial_closed_form,
        pin_combine_closed_forms, pin_member_permutation, pin_check_groups_rejects]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


# ------------------------------------------------------------------ mutants
_orig_partial = P.partial_attention
_orig_combine = P.combine_partials
_orig_range = P.tokens_range


def _lse_without_max(q, K, V, scale):
    o, lse = _orig_partial(q, K, V, scale)
    if K.shape[0] == 0:
        return o, lse
    mx = (scale * (np.atleast_2d(q) @ K.T)).max(axis=1)
    return o, lse - mx


def _lse_base2(q, K, V, scale):
    o, lse = _orig_partial(q, K, V, scale)
    return o, lse / np.log(2.0)


def _combine_unweighted(parts):
    live = [o for o, lse in parts if np.all(np.isfinite(lse))]
    return sum(live) / max(len(live), 1) if live else np.zeros_like(parts[0][0])


def _combine_first_only(parts):
    return parts[0][0]


def _suffix_one_block_late(pool, table, first, last, kv_head, block_size=16):
    if first > 0:
        first += block_size
    return _orig_range(pool, table, min(first, last), last, kv_head, block_size)


def _suffix_one_block_early(pool, table, first, last, kv_head, block_size=16):
    if first > 0:
        first -= block_size
    return _orig_range(pool, table, first, last, kv_head, block_size)


def _two_phase_first_query(q, kp, vp, tables, lens, scale, kv_heads, dtype, prefix_group, group_blocks,
                           block_size=16):
    q = np.array(q)
    for p in range(len(group_blocks)):
        m = P.group_members(prefix_group, p)
        for i in m[1:]:
            q[i] = q[m[0]]
    return _orig_two_phase(q, kp, vp, tables, lens, scale, kv_heads, dtype, prefix_group, group_blocks,
                           block_size)


_orig_two_phase = P.decode_attention_two_phase

MUTANTS = {
    "lse_without_max": ("partial_attention", _lse_without_max),
    "lse_in_base_2": ("partial_attention", _lse_base2),
    "combine_ignores_lse": ("combine_partials", _combine_unweighted),
    "combine_drops_shared_part": ("combine_partials", _combine_first_only),
    "suffix_starts_one_block_late": ("tokens_range", _suffix_one_block_late),
    "suffix_starts_one_block_early": ("tokens_range", _suffix_one_block_early),
    "members_share_first_query": ("decode_attention_two_phase", _two_phase_first_query),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_prefix_mutant_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(P, attr, fn)
    failed = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin()
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
