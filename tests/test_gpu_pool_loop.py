"""A decode loop driven entirely through the C ABI: the native block pool
decides slots, copy-on-write pairs and tables; the kernels move and attend.
Every step is checked against the oracle (its own page-pool simulator, byte
moves and float64 attention): pools bit-exact, attention within tolerance.
"""

import numpy as np
import pytest
import torch

import cases
from oracle import attention as OA
from oracle import kv_ops as OK
from oracle.paged_pool import PagedKVPool

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_209_gb300 import pkv as P
    P.load_library()
    return P


def test_serving_loop_with_sharing_cow_and_release(pkv):
    rng = np.random.default_rng(81)
    NB, HKV, HQ, D = 96, 2, 8, 128
    order = rng.permutation(NB)
    pool = pkv.BlockPool(NB, 16, pop_order=order)
    ora = PagedKVPool(NB, 16, pop_order=order)
    gen = torch.Generator().manual_seed(82)
    kp_h = torch.randn(NB, HKV, 16, D, generator=gen).to(torch.bfloat16)
    vp_h = torch.randn(NB, HKV, 16, D, generator=gen).to(torch.bfloat16)
    kp, vp = kp_h.cuda(), vp_h.cuda()
    hk, hv = cases.host_view(kp_h).copy(), cases.host_view(vp_h).copy()

    def write(slots, n):
        kn = torch.randn(n, HKV, D, generator=gen).to(torch.bfloat16)
        vn = torch.randn(n, HKV, D, generator=gen).to(torch.bfloat16)
        pkv.pkv_append(kn.cuda(), vn.cuda(), torch.from_numpy(np.asarray(slots, np.int64)).cuda(), kp, vp)
        OK.append_tokens(hk, hv, cases.host_view(kn), cases.host_view(vn), slots)

    # a root prompt, then children sharing prefixes of several lengths (some mid-block)
    pool.add_sequence(0)
    ora.create(0)
    slots, _ = pool.append(0, 100)
    ora.append(0, 100)
    assert list(slots) == ora.slots(0, 0, 100)
    write(slots, 100)
    active = []
    for child, prefix in zip(range(1, 6), (100, 77, 64, 33, 5)):
        pool.share_prefix(0, child, prefix)
        ora.share_prefix(0, child, prefix)
        active.append(child)
    pool.release(0)
    ora.release(0)
    next_id = 6
    for step in range(8):
        if step == 4:                       # a request finishes, a new one arrives on freed blocks
            pool.release(active[1])
            ora.release(active.pop(1))
            pool.add_sequence(next_id)
            ora.create(next_id)
            s, _ = pool.append(next_id, 40)
            ora.append(next_id, 40)
            assert list(s) == ora.slots(next_id, 0, 40)
            write(s, 40)
            active.append(next_id)
            next_id += 1
        starts = [ora.sequence_length(s) for s in active]
        slots, pairs = pool.append_batch(active, [1] * len(active))
        for s in active:
            ora.append(s, 1)
        want_pairs = ora.take_copy_pairs()
        assert [tuple(p) for p in pairs] == want_pairs
        assert list(slots) == [ora.slots(s, st, 1)[0] for s, st in zip(active, starts)]
        if len(pairs):
            pkv.pkv_copy_blocks(torch.from_numpy(pairs).cuda(), kp, vp)
            OK.copy_blocks(hk, hv, pairs)
        write(slots, len(active))
        width = 8
        tables, lens = pool.block_tables(active, width)
        q = torch.randn(len(active), HQ, D, generator=gen).to(torch.bfloat16)
        out = pkv.pkv_decode_attention(q.cuda(), kp, vp, torch.from_numpy(tables).cuda(),
                                       torch.from_numpy(lens).cuda(), 1 / np.sqrt(D))
        torch.cuda.synchronize()
        assert np.array_equal(cases.host_view(kp), hk) and np.array_equal(cases.host_view(vp), hv), step
        want = OA.decode_attention(cases.host_view(q), hk, hv, tables, lens, 1 / np.sqrt(D), HKV, "bf16")
        ma, rl = cases.attention_errors(out, want)
        assert ma <= 1e-2 and rl <= 2e-3, (step, ma, rl)
        pool.validate()
