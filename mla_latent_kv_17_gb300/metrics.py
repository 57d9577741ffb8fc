"""Algorithmic FLOP and byte counts of absorbed MLA decode (the roofline model).

Per token the cache entry is the 512-d latent plus the 64-d RoPE key: (512 + 64) x 2 B =
1152 B in bf16 ("MLA & DSA 推理性能优化指南" §4.1; "MLA 在极长上下文下的显存带宽突围",
latent compression: 1152 B per layer, 73.7 KB per token over 64 layers).  This library's
FP8 record is 656 B (512 e4m3 codes + 4 fp32 scales + 64 bf16 RoPE values); the guide's
"~576 B" counts the codes of all 576 channels and no scales.

FLOPs per attended token and head: 2 x 576 for the score (q~ . c + q_R . k_R) and 2 x 512
for the probability-weighted latent sum.  Exponentials and rescaling are not counted.

Algorithmic bytes of one decode call: the cache rows attended, the queries, the outputs,
the block-table entries touched, seq_lens and (sparse) the index lists.  Split-KV partial
results and any re-reads are overhead, not algorithmic bytes.
"""
from __future__ import annotations

D_LATENT, D_ROPE, D_ENTRY = 512, 64, 576
BYTES_PER_TOKEN = {"bf16": D_ENTRY * 2, "fp8": 656}
FLOPS_PER_TOKEN_HEAD = 2 * (D_ENTRY + D_LATENT)


def cache_bytes_per_token(kv_dtype: str = "bf16") -> int:
    return BYTES_PER_TOKEN[kv_dtype]


def mha_kv_bytes_per_token(heads: int = 128, d_head: int = 128, elem_bytes: int = 2) -> int:
    """K and V of every head, the uncompressed equivalent."""
    return heads * d_head * 2 * elem_bytes


def model_kv_bytes_per_token(layers: int, per_layer: int) -> int:
    return layers * per_layer


def attended_tokens(case) -> list[int]:
    """Tokens each request attends: seq_len (dense) or its non-padding indices (sparse)."""
    if case.indices is None:
        return [max(0, int(x)) for x in case.seq_lens.cpu().tolist()]
    idx = case.indices.cpu()
    return [int((idx[b] >= 0).sum()) for b in range(case.B)]


def algorithmic(case) -> dict:
    """FLOPs and bytes of one decode call over `case` (an inputs.Case)."""
    toks = attended_tokens(case)
    H, B = case.H, case.B
    bpt = cache_bytes_per_token(case.kv_dtype)
    flops = sum(toks) * FLOPS_PER_TOKEN_HEAD * H
    q_bytes = B * H * D_ENTRY * 2
    out_bytes = B * H * D_LATENT * 4 + B * H * 4
    if case.indices is None:
        table = sum(4 * ((L + 63) // 64) for L in toks)
        idx_bytes = 0
    else:
        idx = case.indices.cpu()
        table = 0
        for b in range(B):
            v = idx[b][idx[b] >= 0]
            table += 4 * int((v // 64).unique().numel()) if v.numel() else 0
        idx_bytes = 4 * idx.numel()
    nbytes = sum(toks) * bpt + q_bytes + out_bytes + table + 4 * B + idx_bytes
    return dict(flops=flops, bytes=nbytes, tokens=sum(toks), cache_bytes=sum(toks) * bpt,
                ai=flops / nbytes if nbytes else 0.0)


def roofline_seconds(flops: float, nbytes: float, peak_tflops: float, peak_gbs: float) -> float:
    return max(flops / (peak_tflops * 1e12), nbytes / (peak_gbs * 1e9))


def max_over_ranks(value: float, dist=None, device="cpu") -> float:
    """The largest `value` over all ranks of the initialised process group `dist` (the
    torch.distributed module), or `value` itself when there is none: a multi-rank run is
    timed by its slowest rank."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world_size: int, seconds: float) -> float:
    """Units all ranks processed per second when every rank processes `units_per_rank`
    (weak scaling) and the slowest rank took `seconds`."""
    return units_per_rank * world_size / seconds
