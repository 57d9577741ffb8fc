"""The roofline byte/FLOP model against the byte accounting the pages print."""
import json
import os

import torch

from mla_latent_kv_17_gb300 import inputs, metrics

G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "byte_accounting.json")))


def near(key, v):
    g = G[key]
    assert abs(v - g["value"]) <= g.get("tolerance", 0), (key, v, g["value"])


def test_page_figures():
    near("bf16_bytes_per_token_per_layer", metrics.cache_bytes_per_token("bf16"))
    near("mha_equivalent_bytes_per_token", metrics.mha_kv_bytes_per_token(128, 128, 2))
    near("compression_ratio_fp16",
         metrics.mha_kv_bytes_per_token() / metrics.cache_bytes_per_token("bf16"))
    per_tok = metrics.model_kv_bytes_per_token(64, metrics.cache_bytes_per_token("bf16"))
    near("model_kv_kb_per_token_64_layers", per_tok / 1000)
    near("mha_mb_per_token_64_layers_d7168", 2 * 64 * 7168 * 2 / 1e6)
    near("mla_gb_per_request_8k", 8192 * per_tok / 1e9)
    near("mla_gb_per_request_128k", 131072 * per_tok / 1e9)
    near("dsa_read_reduction_L32k_k1024", 1 - 1024 / 32768)


def test_case_counts():
    c = inputs.make_case(2, 16, [100, 0], seed=1)
    a = metrics.algorithmic(c)
    assert a["tokens"] == 100
    assert a["flops"] == 100 * 16 * 2 * (576 + 512)
    expect = 100 * 1152 + 2 * 16 * 576 * 2 + 2 * 16 * 512 * 4 + 2 * 16 * 4 + 4 * 2 + 4 * 2
    assert a["bytes"] == expect
    c.indices = torch.tensor([[0, 5, 70, -1], [-1, -1, -1, -1]], dtype=torch.int32)
    a = metrics.algorithmic(c)
    assert a["tokens"] == 3 and a["flops"] == 3 * 16 * 2 * 1088
