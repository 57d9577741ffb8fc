"""GPU parity of the cache append (through the C ABI) against the CPU oracle: the written
bytes must be identical (byte work, and the FP8 codes are decided in binary32 on both
sides), other rows untouched; then a decode over the appended cache against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from mla_latent_kv_17_gb300 import inputs, ops
from oracle_ref import assert_close, oracle_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mla_latent_kv_17_gb300 import build
    build.build()
    ops.lib()


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _inputs(B, fp8, num_pages, max_pages, seed):
    g = torch.Generator().manual_seed(seed)
    row_bytes = 656 if fp8 else 1152
    raw = torch.randint(0, 256, (num_pages * 64 * row_bytes,), dtype=torch.uint8, generator=g)
    bt = torch.randperm(num_pages, generator=g)[:B * max_pages].reshape(B, max_pages).to(torch.int32)
    # channel blocks of very different magnitudes, one all zero, some exact ties for e4m3
    mag = torch.tensor([1.0, 1e-3, 300.0, 0.0]).repeat_interleave(128)
    lat = (torch.randn(B, 512, generator=g) * mag).to(torch.bfloat16)
    lat[0, :4] = torch.tensor([448.0, -448.0, 1.0625, -1.1875]).to(torch.bfloat16)
    rope = torch.randn(B, 64, generator=g).to(torch.bfloat16)
    return raw, bt, lat, rope


def _gpu_append(raw, fp8, bt, positions, lat, rope, status=None):
    num_pages = raw.numel() // (64 * (656 if fp8 else 1152))
    if fp8:
        cache = raw.reshape(num_pages, 64, 656).clone().cuda()
    else:
        cache = raw.view(torch.bfloat16).reshape(num_pages, 64, 576).clone().cuda()
    ops.cache_append(cache, bt.cuda(), positions.cuda(), lat.cuda(), rope.cuda(), device_status=status)
    torch.cuda.synchronize()
    return cache.cpu().contiguous().view(torch.uint8).reshape(-1).numpy()


@pytest.mark.parametrize("fp8", [False, True])
def test_append_bytes_equal_oracle(fp8):
    B, num_pages, max_pages = 6, 24, 3
    raw, bt, lat, rope = _inputs(B, fp8, num_pages, max_pages, seed=21)
    positions = torch.tensor([0, 63, 64, 191, -1, 130], dtype=torch.int32)
    got = _gpu_append(raw, fp8, bt, positions, lat, rope)
    ref, err = oracle.append(raw.numpy(), fp8, bt.numpy(), positions.numpy(), _bits(lat), _bits(rope))
    assert err == 0
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("fp8", [False, True])
def test_append_many_requests_bytes_equal_oracle(fp8):
    # 300 requests (several CTAs, a ragged last one), one distinct row each
    B, num_pages, max_pages = 300, 640, 2
    raw, bt, lat, rope = _inputs(B, fp8, num_pages, max_pages, seed=22)
    positions = torch.randint(0, 128, (B,), dtype=torch.int32, generator=torch.Generator().manual_seed(5))
    got = _gpu_append(raw, fp8, bt, positions, lat, rope)
    ref, err = oracle.append(raw.numpy(), fp8, bt.numpy(), positions.numpy(), _bits(lat), _bits(rope))
    assert err == 0
    assert np.array_equal(got, ref)


def test_append_out_of_range_is_reported_and_skipped():
    B, num_pages, max_pages = 4, 16, 3
    raw, bt, lat, rope = _inputs(B, True, num_pages, max_pages, seed=23)
    bt = bt.clone()
    bt[1, 0] = num_pages + 7                       # page id out of range
    positions = torch.tensor([5, 10, 3 * 64, 70], dtype=torch.int32)  # request 2: beyond the table
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _gpu_append(raw, True, bt, positions, lat, rope, status=status)
    assert int(status.item()) == 5  # MLA_ERR_INDEX
    ref, err = oracle.append(raw.numpy(), True, bt.numpy(), positions.numpy(), _bits(lat), _bits(rope))
    assert err == 2
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_decode_after_append(kv):
    # every request gains one token (in its last page's first free row); the decode over
    # seq_lens + 1 must match the oracle over the oracle-appended cache
    lens = [100, 1, 250, 63 + 64]
    c = inputs.make_case(len(lens), 128, lens, seed=31, kv_dtype=kv)
    g = torch.Generator().manual_seed(9)
    lat = torch.randn(c.B, 512, generator=g).to(torch.bfloat16)
    rope = torch.randn(c.B, 64, generator=g).to(torch.bfloat16)
    positions = c.seq_lens.clone().to(torch.int32)
    fp8 = kv == "fp8"
    raw = c.cache.contiguous().view(torch.uint8).reshape(-1)
    ref, err = oracle.append(raw.numpy(), fp8, c.block_table.numpy(), positions.numpy(), _bits(lat), _bits(rope))
    assert err == 0
    c = c.to("cuda")
    ops.cache_append(c.cache, c.block_table, positions.cuda(), lat.cuda(), rope.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(c.cache.cpu().contiguous().view(torch.uint8).reshape(-1).numpy(), ref)
    c.seq_lens = c.seq_lens + 1
    ws = ops.Workspace(c.B, c.H)
    ops.plan(ws, c.seq_lens)
    out, lse = ops.decode(ws, c.q_nope, c.q_rope, c.cache, c.block_table, c.seq_lens, c.scale)
    assert ops.status(ws) == 0
    ro, rl = oracle_for(c)
    assert_close(out, lse, ro, rl, f"decode after append ({kv})")
