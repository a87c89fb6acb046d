"""Planted mistakes in the oracle must fail at least one pin.

Each mutant below is a plausible error in the oracle (a dropped term, a
wrong index, a transposed operand, a missing normalisation). The mutant is
planted in the oracle module on the CPU for the duration of one test; the
test passes only if some pin then fails.
"""

import numpy as np
import pytest

import oracle.attention as A
import oracle.kv_ops as K
import oracle_pins


def _softmax_no_scale(q, Kt, V, scale):
    return _orig_softmax(q, Kt, V, 1.0)


def _softmax_no_normalise(q, Kt, V, scale):
    q = np.atleast_2d(q)
    if Kt.shape[0] == 0:
        return np.zeros((q.shape[0], V.shape[1]))
    s = scale * (q @ Kt.T)
    w = np.exp(s - s.max(axis=1, keepdims=True))
    return w @ V


def _softmax_no_max(q, Kt, V, scale):
    q = np.atleast_2d(q)
    if Kt.shape[0] == 0:
        return np.zeros((q.shape[0], V.shape[1]))
    w = np.exp(scale * (q @ Kt.T))
    return (w / w.sum(axis=1, keepdims=True)) @ V


def _softmax_wrong_axis(q, Kt, V, scale):
    q = np.atleast_2d(q)
    if Kt.shape[0] == 0:
        return np.zeros((q.shape[0], V.shape[1]))
    s = scale * (q @ Kt.T)
    w = np.exp(s - s.max(axis=0, keepdims=True))
    return (w / w.sum(axis=0, keepdims=True)) @ V


def _softmax_kv_swapped(q, Kt, V, scale):
    return _orig_softmax(q, V, Kt, scale)


def _gather_off_by_one(pool, table, n, h, block_size=16):
    return _orig_gather(pool, table, max(n - 1, 0), h, block_size) if n > 1 else _orig_gather(pool, table, n, h, block_size)


def _gather_wrong_block_index(pool, table, n, h, block_size=16):
    nb = -(-n // block_size)
    ids = list(table)[:nb][::-1]
    if nb == 0:
        return pool[:0, h, 0, :]
    return np.concatenate([pool[b, h] for b in ids], axis=0)[:n]


def _pair_wrong_group(q, kp, vp, tables, lens, scale, seq, kv_head, kv_heads, dtype, block_size=16):
    G = q.shape[1] // kv_heads
    n = int(lens[seq])
    Kt = A.to_f64(A.gather_tokens(kp, tables[seq], n, kv_head, block_size), dtype)
    V = A.to_f64(A.gather_tokens(vp, tables[seq], n, kv_head, block_size), dtype)
    heads = [h for h in range(q.shape[1]) if h % kv_heads == kv_head]   # interleaved groups
    qg = A.to_f64(q[seq, heads], dtype)
    return A.softmax_attention(qg, Kt, V, scale)


def _copy_k_only(kp, vp, pairs):
    pairs = np.asarray(pairs, dtype=np.int64).reshape(-1, 2)
    for s, d in pairs:
        kp[d] = kp[s]


def _copy_sequential_wrong_direction(kp, vp, pairs):
    pairs = np.asarray(pairs, dtype=np.int64).reshape(-1, 2)
    for s, d in pairs:
        kp[s] = kp[d]
        vp[s] = vp[d]


def _append_heads_reversed(kp, vp, kn, vn, slots, block_size=16):
    for t, s in enumerate(np.asarray(slots).reshape(-1)):
        if s < 0:
            continue
        b, o = divmod(int(s), block_size)
        kp[b, :, o, :] = kn[t][::-1]
        vp[b, :, o, :] = vn[t][::-1]


def _append_offset_swapped(kp, vp, kn, vn, slots, block_size=16):
    for t, s in enumerate(np.asarray(slots).reshape(-1)):
        if s < 0:
            continue
        b, o = divmod(int(s), block_size)
        # block and offset exchanged
        kp[o % kp.shape[0], :, b % block_size, :] = kn[t]
        vp[o % vp.shape[0], :, b % block_size, :] = vn[t]


def _widen_truncating(bits):
    return np.asarray(bits, dtype=np.uint16).astype(np.float64)


_orig_softmax = A.softmax_attention
_orig_gather = A.gather_tokens

MUTANTS = {
    "no_scale": (A, "softmax_attention", _softmax_no_scale),
    "no_normalise": (A, "softmax_attention", _softmax_no_normalise),
    "no_max_subtraction": (A, "softmax_attention", _softmax_no_max),
    "softmax_wrong_axis": (A, "softmax_attention", _softmax_wrong_axis),
    "k_v_swapped": (A, "softmax_attention", _softmax_kv_swapped),
    "gather_drops_last_token": (A, "gather_tokens", _gather_off_by_one),
    "gather_blocks_reversed": (A, "gather_tokens", _gather_wrong_block_index),
    "interleaved_gqa_groups": (A, "decode_attention_pair", _pair_wrong_group),
    "copy_k_pool_only": (K, "copy_blocks", _copy_k_only),
    "copy_wrong_direction": (K, "copy_blocks", _copy_sequential_wrong_direction),
    "append_heads_reversed": (K, "append_tokens", _append_heads_reversed),
    "append_block_offset_swapped": (K, "append_tokens", _append_offset_swapped),
    "bf16_widening_wrong": (A, "bf16_bits_to_f64", _widen_truncating),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    module, attr, fn = MUTANTS[name]
    monkeypatch.setattr(module, attr, fn)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin()
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
