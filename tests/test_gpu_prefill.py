"""GPU parity of the non-absorbed prefill (through the C ABI) against the CPU oracle:
decompressed keys and values elementwise (|x - ref| <= 1e-2 + 1e-2 |ref|), then the causal
attention's out (same bound) and lse (1e-3) against the oracle's prefill with keys and
values rounded to bf16 (the tensors the attention reads), over one query, ragged tiles,
several key tiles, and the bench's 4096-token size on sampled heads; and the attention
against the exact decompression (out within the same bound, lse within 1e-3 plus the bound
of the keys' bf16 rounding)."""
import numpy as np
import pytest
import torch

import oracle
from mla_latent_kv_17_gb300 import inputs, ops

pytestmark = pytest.mark.gpu

SCALE = inputs.SOFTMAX_SCALE


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mla_latent_kv_17_gb300 import build
    build.build()
    ops.lib()


def _f64(t):
    return t.detach().float().cpu().double().numpy()


def _close(got, ref, what, atol=1e-2, rtol=1e-2):
    err = np.abs(got - ref)
    bad = ~(err <= atol + rtol * np.abs(ref))
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: mismatch at {i}: got {got[i]} ref {ref[i]} ({bad.sum()} of {bad.size})")


def _inputs(L, H, seed):
    g = torch.Generator().manual_seed(seed)
    entries = torch.randn(L, 576, generator=g).to(torch.bfloat16)
    q_nope = torch.randn(L, H, 128, generator=g).to(torch.bfloat16)
    q_rope = torch.randn(L, H, 64, generator=g).to(torch.bfloat16)
    _, w_uk, w_uv, _ = inputs.projection_inputs(1, H, seed=seed + 1)
    return entries, q_nope, q_rope, w_uk, w_uv


@pytest.mark.parametrize("L,H", [(1, 4), (300, 3), (1024, 8)])
def test_decompress_matches_oracle(L, H):
    entries, _, _, w_uk, w_uv = _inputs(L, H, 90 + L)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    k, v = ops.prefill_decompress(entries.cuda(), w_uk.cuda(), w_uv.cuda(), device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    lat = np.broadcast_to(_f64(entries)[:, None, :512], (L, H, 512))
    for name, got, w in (("k", k, w_uk), ("v", v, w_uv)):
        ref = oracle.project(lat, _f64(w)).transpose(1, 0, 2)  # [H, L, 128]
        _close(_f64(got), ref, f"decompress {name} L={L} H={H}")


# (384, 10): three query tiles (a pair and a tile alone) over a group of eight heads and a
# remainder group of two, in the CTA order the kernel uses
@pytest.mark.parametrize("L,H", [(1, 2), (129, 3), (300, 2), (700, 4), (384, 10)])
def test_prefill_attention_matches_oracle(L, H):
    entries, q_nope, q_rope, w_uk, w_uv = _inputs(L, H, 100 + L)
    ref_out, ref_lse = oracle.prefill(_f64(entries), _f64(q_nope), _f64(q_rope), _f64(w_uk), _f64(w_uv), SCALE,
                                      kv_bf16=True)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    e = entries.cuda()
    k, v = ops.prefill_decompress(e, w_uk.cuda(), w_uv.cuda(), device_status=status)
    out, lse = ops.prefill_attention(q_nope.cuda(), q_rope.cuda(), e, k, v, SCALE, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _close(_f64(out), ref_out, f"prefill out L={L} H={H}")
    _close(_f64(lse), ref_lse, f"prefill lse L={L} H={H}", atol=1e-3, rtol=0.0)


def test_prefill_bench_size_sampled_heads():
    # the 4096-token, 128-head prefill the bench times; the oracle checks two heads
    L, H = 4096, 128
    entries, q_nope, q_rope, w_uk, w_uv = _inputs(L, H, 110)
    e = entries.cuda()
    k, v = ops.prefill_decompress(e, w_uk.cuda(), w_uv.cuda())
    out, lse = ops.prefill_attention(q_nope.cuda(), q_rope.cuda(), e, k, v, SCALE)
    torch.cuda.synchronize()
    hs = [5, 127]
    ref_out, ref_lse = oracle.prefill(_f64(entries), _f64(q_nope[:, hs]), _f64(q_rope[:, hs]), _f64(w_uk[hs]),
                                      _f64(w_uv[hs]), SCALE, kv_bf16=True)
    _close(_f64(out[:, hs]), ref_out, "prefill out, sampled heads")
    _close(_f64(lse[:, hs]), ref_lse, "prefill lse, sampled heads", atol=1e-3, rtol=0.0)


BF16_UNIT = 2.0 ** -8  # |bf16(x) - x| <= 2^-8 |x| (round to nearest, 8 significant bits)


def _key_rounding_bound(entries, q_nope, w_uk):
    """Largest score error the bf16 rounding of the decompressed keys can cause, per (query,
    head): k = c W^UK reaches the tensor core as bf16(k), so |ds_t| <= scale * sum_d |q_d|
    |k_td| 2^-8 over the 128 decompressed dimensions (the RoPE part and the query are exact),
    and the log-sum-exp over the causal keys t <= i moves by at most max_t |ds_t|."""
    L, H = q_nope.shape[0], q_nope.shape[1]
    lat = _f64(entries)[:, :512]
    k = np.abs(oracle.project(np.broadcast_to(lat[:, None, :], (L, H, 512)), _f64(w_uk)))  # [L, H, 128]
    q = np.abs(_f64(q_nope))                                                             # [L, H, 128]
    out = np.zeros((L, H))
    causal = np.tril(np.ones((L, L), dtype=bool))
    for h in range(H):
        m = q[:, h, :] @ k[:, h, :].T                                                    # [query, key]
        out[:, h] = SCALE * BF16_UNIT * np.where(causal, m, 0.0).max(axis=1)
    return out


@pytest.mark.parametrize("L,H", [(129, 3), (700, 4)])
def test_prefill_attention_matches_exact_oracle(L, H):
    # the same attention against the oracle's prefill with exact (unrounded) keys and values,
    # as the pages define the decompression: out within 1e-2 + 1e-2 |ref| everywhere; lse
    # within 1e-3, or, where the bf16 rounding of the keys alone can move it by more, within
    # 1e-3 plus that rounding's bound
    entries, q_nope, q_rope, w_uk, w_uv = _inputs(L, H, 100 + L)
    ref_out, ref_lse = oracle.prefill(_f64(entries), _f64(q_nope), _f64(q_rope), _f64(w_uk), _f64(w_uv), SCALE,
                                      kv_bf16=False)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    e = entries.cuda()
    k, v = ops.prefill_decompress(e, w_uk.cuda(), w_uv.cuda(), device_status=status)
    out, lse = ops.prefill_attention(q_nope.cuda(), q_rope.cuda(), e, k, v, SCALE, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _close(_f64(out), ref_out, f"prefill out (exact oracle) L={L} H={H}")
    bound = 1e-3 + _key_rounding_bound(entries, q_nope, w_uk)
    err = np.abs(_f64(lse) - ref_lse)
    bad = ~(err <= bound)
    assert not bad.any(), (f"prefill lse (exact oracle) L={L} H={H}: {bad.sum()} over the bound, "
                           f"max err {err.max():.3e}, bound there {bound[np.unravel_index(err.argmax(), err.shape)]:.3e}")
