"""Pins of the byte accounting against the notebook's printed contract.

Sources: "Notebook 10. KV cache and serving: bytes, pages, and ceilings",
section 1 (geometry), section 2 (the KV/token ladder and the 70B GQA context
memory table), section 3 (decode KV bytes of the roofline scenarios and the
FLOP count), section 6 (page waste) and section 9 (negative tests). The
model dimensions below are the ones that section 1 declares for each model.
"""

import json
import math
import os

import pytest

from oracle import geometry as g

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "notebook10_contract.json")))

MODELS = {
    "70B MHA-equivalent (H=64)": g.KVGeometry(80, 64, 128, 2),
    "LLaMA-3.3-70B GQA": g.KVGeometry(80, 8, 128, 2),
    "Llama-3-8B GQA": g.KVGeometry(32, 8, 128, 2),
    "DeepSeek-V3 MLA (latent+RoPE)": g.LatentKVGeometry(61, 512, 64, 2),
}


def test_kv_ladder():
    for name, geom in MODELS.items():
        assert geom.bytes_per_token == GOLDEN["kv_ladder_bytes_per_token"][name]
        assert geom.bytes_per_token / g.KIB == GOLDEN["kv_ladder_kib_per_token"][name]


def test_llama_3_8b_is_131072_bytes_per_token():
    assert g.KVGeometry(32, 8, 128).bytes_per_token == 131072
    # One layer of the same model: the unit of the decode kernel's traffic.
    assert g.KVGeometry(1, 8, 128).bytes_per_token == 4096


def test_context_memory_70b_gqa():
    g70 = MODELS["LLaMA-3.3-70B GQA"]
    for tokens, want in GOLDEN["context_memory_70b_gqa_bytes"].items():
        assert g.kv_payload_bytes(g70, int(tokens)) == want
    for tokens, gib in GOLDEN["context_memory_70b_gqa_binary_gib"].items():
        assert g.kv_payload_bytes(g70, int(tokens)) / g.GIB == gib


def test_decode_kv_bytes_of_the_roofline_scenarios():
    g8 = MODELS["Llama-3-8B GQA"]
    for tokens, want in GOLDEN["decode_kv_bytes_batch1_32_layers"].items():
        assert g.kv_payload_bytes(g8, int(tokens)) == want
    # Per layer, summed over a batch: the decode call's KV bytes.
    assert g.decode_kv_bytes([8192] * 32, 8, 128, 2) == 1073741824
    assert g.decode_kv_bytes([131072] * 4, 8, 128, 2) == 2147483648


def test_page_waste_closed_forms():
    assert math.isclose(g.naive_preallocation_waste(32768, 2048), GOLDEN["naive_waste_fraction"], abs_tol=1e-12)
    assert math.isclose(g.expected_paged_waste(2048, 16), GOLDEN["expected_paged_waste_fraction"], abs_tol=1e-12)
    # Block size 1 wastes nothing in expectation.
    assert g.expected_paged_waste(100, 1) == 0.0


def test_flop_counts():
    # Section 3: QK and AV together cost 4 FLOPs per (layer, head, dim, pair).
    assert g.attention_flops(1, 1, 1, 1, 0) == 4
    assert g.attention_flops(32, 32, 128, 1, 8191) == 4 * 32 * 32 * 128 * 8192
    # Chunked prefill covers exactly the pairs of the full prefill (section 7).
    chunks = [g.attention_flops(32, 32, 128, 512, p) for p in range(0, 8192, 512)]
    assert sum(chunks) == g.attention_flops(32, 32, 128, 8192)
    assert g.decode_attention_flops([8192] * 32, 32, 128) == 4 * 32 * 128 * 8192 * 32


def test_negative_geometry_and_payload():
    with pytest.raises(ValueError):
        g.KVGeometry(0, 8, 128, 2)
    g8 = MODELS["Llama-3-8B GQA"]
    with pytest.raises(ValueError):
        g.kv_payload_bytes(g8, -1)
    with pytest.raises(ValueError):
        g.kv_payload_bytes(g8, 1, 1, 1 / 3)
    with pytest.raises(ValueError):
        g.attention_flops(32, 32, 128, -1)
    # 3-bit storage of 128 KiB/token is exactly 24 KiB/token (section 8).
    assert g.kv_payload_bytes(g8, 1, 1, 3 / 16) == 24 * g.KIB
