"""The Python binding only marshals: it rejects tensors of the wrong device, dtype, shape or
layout before any library call (CPU only; no GPU needed)."""
import pytest
import torch

from mla_latent_kv_17_gb300 import ops


def bf16(*shape):
    return torch.zeros(*shape, dtype=torch.bfloat16)


def test_absorb_and_project_reject_bad_tensors():
    with pytest.raises(ValueError):
        ops.absorb_query(bf16(2, 4, 128), bf16(4, 128, 512))            # CPU tensors
    with pytest.raises(ValueError):
        ops.absorb_query(torch.zeros(2, 4, 128), bf16(4, 128, 512))     # fp32 query
    with pytest.raises(ValueError):
        ops.project_output(bf16(2, 4, 512), bf16(4, 128, 512))          # bf16 latent output
    with pytest.raises(ValueError):
        ops.project_output(torch.zeros(2, 4, 256), bf16(4, 128, 512))   # wrong width


def test_topk_rejects_bad_tensors():
    with pytest.raises(ValueError):
        ops.topk_select(torch.zeros(2, 64), torch.zeros(2, dtype=torch.int32), 8)   # CPU
    with pytest.raises(ValueError):
        ops.topk_select(torch.zeros(2, 64, dtype=torch.float64), torch.zeros(2, dtype=torch.int32), 8)
    with pytest.raises(ValueError):
        ops.topk_select(torch.zeros(2, 64).t(), torch.zeros(64, dtype=torch.int32), 8)  # column stride


def test_prefill_and_append_reject_bad_tensors():
    with pytest.raises(ValueError):
        ops.prefill_decompress(bf16(16, 576), bf16(2, 128, 512), bf16(2, 128, 512))  # CPU
    with pytest.raises(ValueError):
        ops.prefill_decompress(bf16(16, 512), bf16(2, 128, 512), bf16(2, 128, 512))  # entries width
    with pytest.raises(ValueError):
        ops.prefill_attention(bf16(16, 2, 128), bf16(16, 2, 64), bf16(16, 576), bf16(2, 16, 128),
                              bf16(2, 16, 128), 0.07)                                 # CPU
    with pytest.raises(ValueError):
        ops.cache_append(bf16(4, 64, 576), torch.zeros(2, 2, dtype=torch.int32),
                         torch.zeros(2, dtype=torch.int32), bf16(2, 512), bf16(2, 64))  # CPU ints
