"""pkv_decode_attention_noalloc against pkv_decode_attention and the oracle.

The no-allocation entry point is for callers that cannot hand the library a
device workspace: plugins inside a framework whose memory pool they do not
own, latency-critical code that cannot afford cudaMalloc's implicit
synchronisation, deployments whose device-memory budget is fixed at start-up.
It runs the same decode kernel on a fixed array inside the library, so with
the same kernel and CTA count its output must be bit-identical to the
workspace entry point's, and within the decode bars of the float64 oracle.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test. It passes both alone in a
fresh process (the first call on the device does the array's set-up) and
after the other tests (the array then holds the previous calls' leftovers).
"""

import pytest
import torch

import cases
from oracle import attention as OA

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


def oracle(c):
    return OA.decode_attention(cases.host_view(c["q"]), cases.host_view(c["k_pool"]), cases.host_view(c["v_pool"]),
                               c["tables"], c["lens"], float(c["scale"]), c["kv_heads"], cases.dtype_name(c["q"]))


@pytest.mark.parametrize("kernel,num_ctas", [(0, 0), (0, 97), (1, 0)])
def test_noalloc_matches_the_workspace_entry_point_twice(pkv, kernel, num_ctas):
    c = cases.random_case(61, [1, 40, 333, 2048, 17, 5000], 32, 8, 128, torch.bfloat16, poison=True)
    q, kp, vp = dev(c["q"]), dev(c["k_pool"]), dev(c["v_pool"])
    tables, lens = dev(c["tables"], torch.int32), dev(c["lens"], torch.int32)
    want = oracle(c)
    ref = pkv.pkv_decode_attention(q, kp, vp, tables, lens, c["scale"], kernel=kernel, num_ctas=num_ctas,
                                   out=torch.full_like(q, float("nan")))
    for _ in range(2):   # two calls in a row on the shared array
        got = pkv.pkv_decode_attention_noalloc(q, kp, vp, tables, lens, c["scale"], kernel=kernel,
                                               num_ctas=num_ctas, out=torch.full_like(q, float("nan")))
        torch.cuda.synchronize()
        assert torch.equal(got, ref), "noalloc output differs from pkv_decode_attention's"
        ma, rl = cases.attention_errors(got, want)
        assert ma <= MAX_ABS and rl <= REL_L2, (ma, rl)
    assert pkv.pkv_device_status() == 0


def test_noalloc_after_a_call_that_timed_out(pkv):
    """A call stopped by its bounded waits (test hook: the producer issues
    nothing) leaves merge counters in the shared array; the next call clears
    them first, so its output is again exact."""
    c = cases.random_case(63, [300, 40, 1000, 4097], 32, 8, 128, torch.bfloat16)
    q, kp, vp = dev(c["q"]), dev(c["k_pool"]), dev(c["v_pool"])
    tables, lens = dev(c["tables"], torch.int32), dev(c["lens"], torch.int32)
    ref = pkv.pkv_decode_attention(q, kp, vp, tables, lens, c["scale"], kernel=2, num_ctas=64)
    pkv.pkv_device_status(clear=True)
    pkv.pkv_decode_attention_noalloc(q, kp, vp, tables, lens, c["scale"], kernel=2, num_ctas=64,
                                     flags=pkv.PKV_FLAG_TEST_STALL)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status(clear=True) & pkv.PKV_DEVERR_TIMEOUT
    for _ in range(2):
        got = pkv.pkv_decode_attention_noalloc(q, kp, vp, tables, lens, c["scale"], kernel=2, num_ctas=64,
                                               out=torch.full_like(q, float("nan")))
        torch.cuda.synchronize()
        assert pkv.pkv_device_status(clear=True) == 0
        assert torch.equal(got, ref)
    ma, rl = cases.attention_errors(got, oracle(c))
    assert ma <= MAX_ABS and rl <= REL_L2, (ma, rl)


def test_noalloc_refuses_work_beyond_its_array(pkv):
    c = cases.random_case(62, [64, 64], 32, 8, 128, torch.bfloat16)
    q, kp, vp = dev(c["q"]), dev(c["k_pool"]), dev(c["v_pool"])
    out = torch.full_like(q, 5.0)
    need = pkv.pkv_decode_workspace_size(2, 32, c["tables"].shape[1], kp, num_ctas=20000)
    assert need > pkv.PKV_NOALLOC_SCRATCH_BYTES
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_decode_attention_noalloc(q, kp, vp, dev(c["tables"], torch.int32), dev(c["lens"], torch.int32),
                                         c["scale"], out=out, num_ctas=20000)
    assert e.value.name == "PKV_ERR_WORKSPACE"
    torch.cuda.synchronize()
    assert torch.all(out == 5.0)
