"""Pins of the multi-query (causal) oracle, and planted mistakes that must
fail one of them.

Pinned against: PyTorch's own float64 scaled_dot_product_attention with an
explicit causal boolean mask over contiguous K/V (a library routine, not the
oracle retyped); the single-query decode oracle (one query per sequence);
and the notebook's statement that prefill chunks together hold exactly the
causal pairs of the whole prompt (a prompt attended in one call and in two
chunks gives the same rows).
"""

import numpy as np
import pytest
import torch

import oracle.multiquery as M
from oracle import attention as OA


def paged_case(seed, lens, nqs, kv_heads=2, G=3, d=16, width=None):
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens)
    nb = -(-lens // 16)
    total_blocks = int(nb.sum()) + 3
    perm = rng.permutation(total_blocks)
    w = width or int(nb.max())
    tables = np.full((len(lens), w), -1, dtype=np.int64)
    off = 0
    for i, b in enumerate(nb):
        tables[i, :b] = perm[off:off + b]
        off += b
    kp = rng.standard_normal((total_blocks, kv_heads, 16, d)).astype(np.float32)
    vp = rng.standard_normal((total_blocks, kv_heads, 16, d)).astype(np.float32)
    qs = np.concatenate([[0], np.cumsum(nqs)])
    q = rng.standard_normal((int(qs[-1]), kv_heads * G, d)).astype(np.float32)
    return q, kp, vp, tables, lens, qs


def contiguous(pool, table, n, h):
    return np.concatenate([pool[b, h] for b in table[: -(-n // 16)]], axis=0)[:n].astype(np.float64)


def pin_sdpa_causal():
    q, kp, vp, tables, lens, qs = paged_case(1, [37, 16, 5, 50], [4, 3, 5, 1])
    kvh, G = 2, 3
    out = M.multiquery_attention(q, kp, vp, tables, lens, qs, 0.4, kvh, "f32")
    for i, n in enumerate(lens):
        nq = qs[i + 1] - qs[i]
        for h in range(kvh):
            K = torch.from_numpy(contiguous(kp, tables[i], n, h))
            V = torch.from_numpy(contiguous(vp, tables[i], n, h))
            Q = torch.from_numpy(q[qs[i]:qs[i + 1], h * G:(h + 1) * G].astype(np.float64)).transpose(0, 1)
            mask = torch.tensor([[p <= n - nq + t for p in range(n)] for t in range(nq)])
            ref = torch.nn.functional.scaled_dot_product_attention(
                Q, K.expand(G, -1, -1), V.expand(G, -1, -1), attn_mask=mask, scale=0.4)
            got = out[qs[i]:qs[i + 1], h * G:(h + 1) * G].transpose(1, 0, 2)
            assert np.max(np.abs(got - ref.numpy())) < 1e-12, (i, h)


def pin_single_query_is_decode():
    q, kp, vp, tables, lens, qs = paged_case(2, [9, 33, 64, 1], [1, 1, 1, 1])
    a = M.multiquery_attention(q, kp, vp, tables, lens, qs, 0.3, 2, "f32")
    b = OA.decode_attention(q, kp, vp, tables, lens, 0.3, 2, "f32")
    assert np.max(np.abs(a - b)) < 1e-15


def pin_chunks_hold_the_prompt():
    # one sequence of 40 tokens attended as a whole prompt and as chunks 24 + 16
    q, kp, vp, tables, lens, qs = paged_case(3, [40], [40])
    whole = M.multiquery_attention(q, kp, vp, tables, lens, qs, 0.5, 2, "f32")
    first = M.multiquery_attention(q[:24], kp, vp, tables, np.array([24]), np.array([0, 24]), 0.5, 2, "f32")
    second = M.multiquery_attention(q[24:], kp, vp, tables, np.array([40]), np.array([0, 16]), 0.5, 2, "f32")
    assert np.max(np.abs(whole - np.concatenate([first, second]))) < 1e-15
    # the first query of a whole prompt sees only token 0: its output is that token's V
    assert np.max(np.abs(whole[0, :3] - vp[tables[0, 0], 0, 0])) < 1e-15


PINS = [pin_sdpa_causal, pin_single_query_is_decode, pin_chunks_hold_the_prompt]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def test_rejects_more_queries_than_tokens():
    q, kp, vp, tables, lens, qs = paged_case(4, [3], [3])
    with pytest.raises(ValueError):
        M.multiquery_attention(q, kp, vp, tables, np.array([2]), qs, 0.5, 2, "f32")


# ------------------------------------------------------------------ mutants
def _variant(visible_of):
    def fn(q, k_pool, v_pool, block_tables, context_lens, query_start, scale, kv_heads, dtype, block_size=16):
        total, query_heads, d = q.shape
        G = query_heads // kv_heads
        out = np.zeros((total, query_heads, d))
        for i in range(len(context_lens)):
            q0, q1 = int(query_start[i]), int(query_start[i + 1])
            n, nq = int(context_lens[i]), q1 - q0
            for t in range(nq):
                vis = max(1, min(n, visible_of(n, nq, t)))
                for j in range(kv_heads):
                    K = M.to_f64(M.gather_tokens(k_pool, block_tables[i], vis, j, block_size), dtype)
                    V = M.to_f64(M.gather_tokens(v_pool, block_tables[i], vis, j, block_size), dtype)
                    out[q0 + t, j * G:(j + 1) * G] = M.softmax_attention(
                        M.to_f64(q[q0 + t, j * G:(j + 1) * G], dtype), K, V, scale)
        return out
    return fn


MUTANTS = {
    "no_causal_mask": _variant(lambda n, nq, t: n),
    "query_does_not_see_itself": _variant(lambda n, nq, t: n - nq + t),
    "queries_reversed": _variant(lambda n, nq, t: n - t),
    "mask_one_token_late": _variant(lambda n, nq, t: n - nq + t + 2),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_multiquery_mutant_is_caught(name, monkeypatch):
    monkeypatch.setattr(M, "multiquery_attention", MUTANTS[name])
    failed = []
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
