"""Seeded synthetic inputs for absorbed MLA decode.

This module only draws random numbers and lays them out; it holds none of the decode
arithmetic.  Both the CUDA library's tests/benchmark and the CPU oracle read the same
buffers it returns.

Shapes follow the workloads the decode path is measured on: H query heads, each with a
512-d absorbed query and a 64-d RoPE query (bf16, N(0,1)); one shared paged cache whose
per-token entry is the 512-d latent c_KV followed by the 64-d RoPE key k_R
("MLA & DSA 推理性能优化指南" §1.1 and §4.1: (512 + 64) x 2 B = 1152 B per token in 16-bit
form); 64-token pages handed out as a random permutation of the physical page pool.

FP8 cache records (656 B per token): 512 e4m3 "fn" codes, 4 little-endian fp32 scales
(one per 128 latent channels, scale = max|x| / 448, 1.0 for an all-zero block), then the
64 bf16 RoPE values.  Codes are round-to-nearest-even of x / scale, clamped to +-448.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

PAGE = 64
D_LATENT = 512
D_ROPE = 64
D_ENTRY = D_LATENT + D_ROPE
FP8_RECORD = 656
SOFTMAX_SCALE = 1.0 / math.sqrt(192.0)  # 1/sqrt(d_head 128 + d_rope 64)


@dataclass
class Case:
    """One decode batch.  Tensors live on ``device``; bf16 values are torch.bfloat16."""

    B: int
    H: int
    seq_lens: torch.Tensor          # int32 [B]
    block_table: torch.Tensor       # int32 [B, max_pages]
    q_nope: torch.Tensor            # bf16 [B, H, 512]
    q_rope: torch.Tensor            # bf16 [B, H, 64]
    cache: torch.Tensor             # bf16 [num_pages, 64, 576] or uint8 [num_pages, 64, 656]
    kv_dtype: str = "bf16"          # "bf16" or "fp8"
    scale: float = SOFTMAX_SCALE
    indices: Optional[torch.Tensor] = None   # int32 [B, topk] for token-sparse decode
    meta: dict = field(default_factory=dict)

    @property
    def num_pages(self) -> int:
        return int(self.cache.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    def to(self, device) -> "Case":
        f = lambda t: None if t is None else t.to(device)
        return Case(self.B, self.H, f(self.seq_lens), f(self.block_table), f(self.q_nope),
                    f(self.q_rope), f(self.cache), self.kv_dtype, self.scale, f(self.indices),
                    dict(self.meta))


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def seq_lens_uniform(B: int, lo: int, hi: int, seed: int) -> torch.Tensor:
    """Integers uniform in [lo, hi] (inclusive)."""
    g = _gen(seed, "cpu")
    return torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)


def seq_lens_lognormal(B: int, median: int, sigma: float, lo: int, hi: int,
                       seed: int) -> torch.Tensor:
    """round(exp(ln(median) + sigma * Z)) clipped to [lo, hi]."""
    g = _gen(seed, "cpu")
    z = torch.randn((B,), generator=g, dtype=torch.float64)
    v = torch.exp(math.log(median) + sigma * z).round().clamp(lo, hi)
    return v.to(torch.int32)


def _block_table(seq_lens: torch.Tensor, extra_pages: int, g: torch.Generator):
    pages = [(int(L) + PAGE - 1) // PAGE for L in seq_lens.tolist()]
    total = sum(pages) + int(extra_pages)
    perm = torch.randperm(max(total, 1), generator=g)
    max_pages = max(1, max(pages) if pages else 1)
    bt = torch.zeros((len(pages), max_pages), dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages):
        if n:
            bt[b, :n] = perm[off:off + n].to(torch.int32)
        off += n
    return bt, max(total, 1)


def _poison_tails(cache_rows: torch.Tensor, seq_lens, block_table, value):
    """Fill rows past the end of each request's last page (never attended) with `value`."""
    for b, L in enumerate(seq_lens.tolist()):
        r = L % PAGE
        if L > 0 and r:
            p = int(block_table[b, (L - 1) // PAGE])
            cache_rows[p, r:] = value


def quantize_fp8_records(latent: torch.Tensor, rope: torch.Tensor) -> torch.Tensor:
    """[..., 512] float latent + [..., 64] bf16 rope -> uint8 records [..., 656]."""
    lead = latent.shape[:-1]
    x = latent.float().reshape(*lead, 4, 128)
    amax = x.abs().amax(dim=-1, keepdim=True)
    s = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (x / s).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    codes = q.reshape(*lead, 512).view(torch.uint8)
    sc = s.reshape(*lead, 4).contiguous().view(torch.uint8).reshape(*lead, 16)
    rp = rope.to(torch.bfloat16).contiguous().view(torch.uint8).reshape(*lead, 128)
    return torch.cat([codes, sc, rp], dim=-1).contiguous()


def make_case(B: int, H: int, seq_lens, *, seed: int, kv_dtype: str = "bf16",
              extra_pages: int = 0, poison_tail: bool = True, device="cpu",
              q_scale: float = 1.0) -> Case:
    """Dense decode batch: N(0,1) queries and cache, shuffled pages.

    ``seq_lens`` is a list or int32 tensor.  Rows beyond each request's length in its last
    page are filled with NaN (or NaN codes) so that any read of them shows in the result.
    Large caches can be drawn directly on a CUDA device (``device="cuda"``); the draws then
    come from that device's generator.
    """
    seq_lens = torch.as_tensor(seq_lens, dtype=torch.int32).reshape(B)
    g = _gen(seed, "cpu")
    bt, num_pages = _block_table(seq_lens, extra_pages, g)
    q_nope = (torch.randn((B, H, D_LATENT), generator=g) * q_scale).to(torch.bfloat16)
    q_rope = (torch.randn((B, H, D_ROPE), generator=g) * q_scale).to(torch.bfloat16)
    gd = g if str(device) == "cpu" else _gen(seed * 7919 + 1, device)
    if kv_dtype == "bf16":
        cache = torch.randn((num_pages, PAGE, D_ENTRY), generator=gd, device=device,
                            dtype=torch.float32).to(torch.bfloat16)
        if poison_tail:
            _poison_tails(cache, seq_lens, bt, float("nan"))
    elif kv_dtype == "fp8":
        cache = torch.empty((num_pages, PAGE, FP8_RECORD), dtype=torch.uint8, device=device)
        step = 1024  # pages per chunk, bounds temporary memory
        for p0 in range(0, num_pages, step):
            p1 = min(num_pages, p0 + step)
            lat = torch.randn((p1 - p0, PAGE, D_LATENT), generator=gd, device=device)
            rope = torch.randn((p1 - p0, PAGE, D_ROPE), generator=gd, device=device)
            cache[p0:p1] = quantize_fp8_records(lat, rope)
        if poison_tail:
            _poison_tails(cache, seq_lens, bt, 0xFF)
    else:
        raise ValueError(kv_dtype)
    c = Case(B, H, seq_lens, bt, q_nope, q_rope, cache, kv_dtype)
    return c.to(device)


def sparse_indices(seq_lens, topk: int, window: int, seed: int) -> torch.Tensor:
    """Per request: `topk - window` distinct sorted uniform draws from [0, L - window)
    followed by the last `window` positions; when L < topk, all L positions then -1."""
    g = _gen(seed, "cpu")
    rows = []
    for L in torch.as_tensor(seq_lens).tolist():
        L = int(L)
        if L < topk:
            r = torch.full((topk,), -1, dtype=torch.int32)
            r[:L] = torch.arange(L, dtype=torch.int32)
        else:
            n_draw = topk - window
            span = L - window
            pick = torch.randperm(span, generator=g)[:n_draw].sort().values
            r = torch.cat([pick, torch.arange(span, L)]).to(torch.int32)
        rows.append(r)
    return torch.stack(rows).contiguous()


# --------------------------------------------------------------------------------------
# The five measured workloads.  Seeds are 17 + the workload's position in this list.
# --------------------------------------------------------------------------------------
WORKLOADS = {
    "tiny_dense_b1_h16_l256": dict(index=0, B=1, H=16, kind="dense"),
    "dsv3_dense_b64_h128_l1k_8k": dict(index=1, B=64, H=128, kind="dense"),
    "long_dense_b4_h128_l128k": dict(index=2, B=4, H=128, kind="dense"),
    "fp8_ragged_b128_h128_lognormal": dict(index=3, B=128, H=128, kind="fp8"),
    "dsa_sparse_b64_h128_l64k_top2048": dict(index=4, B=64, H=128, kind="sparse"),
}


def workload_seq_lens(name: str) -> torch.Tensor:
    w = WORKLOADS[name]
    seed = 17 + w["index"]
    if w["index"] == 0:
        return torch.tensor([256], dtype=torch.int32)
    if w["index"] == 1:
        return seq_lens_uniform(64, 1024, 8192, seed)
    if w["index"] == 2:
        return torch.full((4,), 131072, dtype=torch.int32)
    if w["index"] == 3:
        return seq_lens_lognormal(128, 4096, 1.0, 64, 32768, seed)
    if w["index"] == 4:
        return torch.full((64,), 65536, dtype=torch.int32)
    raise KeyError(name)


def make_workload(name: str, device="cpu") -> Case:
    w = WORKLOADS[name]
    seed = 17 + w["index"]
    sl = workload_seq_lens(name)
    kv = "fp8" if w["kind"] == "fp8" else "bf16"
    c = make_case(w["B"], w["H"], sl, seed=seed, kv_dtype=kv, device=device)
    if w["kind"] == "sparse":
        c.indices = sparse_indices(sl, 2048, 512, seed + 1000).to(device)
    c.meta["workload"] = name
    return c


D_HEAD = 128  # per-head nope query / value width d_h ("MLA & DSA 推理性能优化指南" §5.1)


def projection_inputs(B: int, H: int, seed: int, device="cpu"):
    """Per-head nope queries q^C [B,H,128] ~ N(0,1) and the two up-projections W^UK, W^UV
    [H,128,512] with N(0, 1/fan_in) entries (fan_in 128 for W^UK, 512 for W^UV), all rounded
    to bf16, plus a latent output [B,H,512] fp32 ~ N(0,1) for the value projection."""
    g = _gen(seed, "cpu")
    q_c = torch.randn(B, H, D_HEAD, generator=g).to(torch.bfloat16)
    w_uk = (torch.randn(H, D_HEAD, D_LATENT, generator=g) / math.sqrt(D_HEAD)).to(torch.bfloat16)
    w_uv = (torch.randn(H, D_HEAD, D_LATENT, generator=g) / math.sqrt(D_LATENT)).to(torch.bfloat16)
    out = torch.randn(B, H, D_LATENT, generator=g)
    return q_c.to(device), w_uk.to(device), w_uv.to(device), out.to(device)
