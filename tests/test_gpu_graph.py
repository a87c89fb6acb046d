"""The step's calls inside a CUDA graph: append + attention captured once and
replayed must give the bytes an eager run gives (the kernels' merge order does
not depend on timing), for the decode, multi-query (both paths) and int8
calls. Workspaces are reused across replays (the kernels leave their counters
at zero)."""

import numpy as np
import pytest
import torch

import cases
from oracle import attention as OA
from oracle import quant as OQ

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_209_gb300 import pkv as P
    P.load_library()
    return P


def step_inputs(seed, lens, hq, hkv, d=128, nq=1):
    """A paged case plus the step's new rows: the last nq tokens of every
    sequence are (re)written by the append before attention."""
    c = cases.random_case(seed, lens, hq, hkv, d, torch.bfloat16)
    rng = np.random.default_rng(seed)
    pos = np.concatenate([np.arange(n - nq, n) for n in c["lens"]])
    seq = np.repeat(np.arange(len(lens)), nq)
    slots = c["tables"][seq, pos // 16].astype(np.int64) * 16 + pos % 16
    kn = torch.from_numpy(rng.standard_normal((len(slots), hkv, d)).astype(np.float32)).to(torch.bfloat16)
    vn = torch.from_numpy(rng.standard_normal((len(slots), hkv, d)).astype(np.float32)).to(torch.bfloat16)
    q = torch.from_numpy(rng.standard_normal((len(slots), hq, d)).astype(np.float32)).to(torch.bfloat16)
    qs = np.arange(0, len(slots) + 1, nq).astype(np.int32)
    dev = torch.device("cuda", 0)
    return dict(k=c["k_pool"].to(dev), v=c["v_pool"].to(dev), tables=torch.from_numpy(c["tables"]).to(dev),
                lens=torch.from_numpy(c["lens"]).to(dev), slots=torch.from_numpy(slots).to(dev), kn=kn.to(dev),
                vn=vn.to(dev), q=q.to(dev), qs=torch.from_numpy(qs).to(dev), scale=c["scale"], host=c)


def eager_and_graph(step, reset):
    """Run `step` eagerly, reset the state, capture it, replay twice; returns
    the eager output and the two replayed ones (copies)."""
    out_e = step().clone()
    torch.cuda.synchronize()
    reset()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                                   # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    reset()
    with torch.cuda.graph(g):
        out = step()
    outs = []
    for _ in range(2):
        reset()
        g.replay()
        torch.cuda.synchronize()
        outs.append(out.clone())
    return out_e, outs


def test_decode_step_in_a_graph(pkv):
    w = step_inputs(81, [300, 17, 1000, 64, 5], 32, 8)
    k0, v0 = w["k"].clone(), w["v"].clone()
    out = torch.empty_like(w["q"])
    ws = torch.zeros(pkv.pkv_decode_workspace_size(5, 32, w["tables"].shape[1], w["k"]), dtype=torch.uint8,
                     device="cuda")

    def step():
        pkv.pkv_append(w["kn"], w["vn"], w["slots"], w["k"], w["v"])
        return pkv.pkv_decode_attention(w["q"], w["k"], w["v"], w["tables"], w["lens"], w["scale"], out=out,
                                        workspace=ws)

    def reset():
        w["k"].copy_(k0)
        w["v"].copy_(v0)

    out_e, outs = eager_and_graph(step, reset)
    assert pkv.pkv_device_status(clear=True) == 0
    for o in outs:
        assert torch.equal(o, out_e)
    hk, hv = cases.host_view(w["k"]), cases.host_view(w["v"])
    want = OA.decode_attention(cases.host_view(w["q"]), hk, hv, w["host"]["tables"], w["host"]["lens"], w["scale"],
                               8, "bf16")
    ma, rl = cases.attention_errors(out_e, want)
    assert ma <= 1e-2 and rl <= 2e-3


@pytest.mark.parametrize("nq", [4, 40])
def test_multiquery_step_in_a_graph(pkv, nq):
    """4 queries per sequence (split kernel) and 40 (tensor-core tile kernel)."""
    w = step_inputs(82 + nq, [300, 64, 900], 32, 8, nq=nq)
    k0, v0 = w["k"].clone(), w["v"].clone()
    out = torch.empty_like(w["q"])
    ws = torch.zeros(max(256, pkv.pkv_multiquery_workspace_size(3, 32, w["tables"].shape[1], nq, w["k"])),
                     dtype=torch.uint8, device="cuda")

    def step():
        pkv.pkv_append(w["kn"], w["vn"], w["slots"], w["k"], w["v"])
        return pkv.pkv_multiquery_attention(w["q"], w["k"], w["v"], w["tables"], w["lens"], w["qs"], w["scale"], nq,
                                            out=out, workspace=ws)

    def reset():
        w["k"].copy_(k0)
        w["v"].copy_(v0)

    out_e, outs = eager_and_graph(step, reset)
    assert pkv.pkv_device_status(clear=True) == 0
    for o in outs:
        assert torch.equal(o, out_e)


def test_int8_step_in_a_graph(pkv):
    w = step_inputs(85, [200, 33, 700, 1], 32, 8)
    kc, ks = OQ.quantize_rows(OA.bf16_bits_to_f64(cases.host_view(w["host"]["k_pool"])))
    vc, vs = OQ.quantize_rows(OA.bf16_bits_to_f64(cases.host_view(w["host"]["v_pool"])))
    dev = torch.device("cuda", 0)
    pools0 = [torch.from_numpy(kc).to(dev), torch.from_numpy(np.ascontiguousarray(vc.transpose(0, 1, 3, 2))).to(dev),
              torch.from_numpy(np.stack([ks, vs], axis=2)).to(dev)]
    pools = [p.clone() for p in pools0]
    out = torch.empty_like(w["q"])
    ws = torch.zeros(pkv.pkv_decode_q8_workspace_size(4, 32, w["tables"].shape[1], pools[0]), dtype=torch.uint8,
                     device="cuda")

    def step():
        pkv.pkv_append_q8(w["kn"], w["vn"], w["slots"], *pools)
        return pkv.pkv_decode_attention_q8(w["q"], *pools, w["tables"], w["lens"], w["scale"], out=out,
                                           workspace=ws)

    def reset():
        for p, p0 in zip(pools, pools0):
            p.copy_(p0)

    out_e, outs = eager_and_graph(step, reset)
    assert pkv.pkv_device_status(clear=True) == 0
    for o in outs:
        assert torch.equal(o, out_e)
