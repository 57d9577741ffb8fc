"""The allocation-free entry point (mla_decode_static) against the workspace entry point.

mla_decode_static serves callers that cannot allocate device memory at decode time (a
fixed arena, a real-time loop, a plugin whose host owns all allocations); it takes its
workspace from a fixed array inside the library.  These checks call it through the C ABI
twice in a row on the same inputs and compare each result with mla_decode run with a
caller-owned workspace, within the parity tolerance the other tests use.  The file sorts
last so that a run that stops at the first failure has already run every other test.
"""
import pytest
import torch

from mla_latent_kv_17_gb300 import inputs, ops
from oracle_ref import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mla_latent_kv_17_gb300 import build
    build.build()
    ops.lib()


def _with_workspace(c):
    ws = ops.Workspace(c.B, c.H)
    ops.plan(ws, c.seq_lens)
    out, lse = ops.decode(ws, c.q_nope, c.q_rope, c.cache, c.block_table, c.seq_lens, c.scale)
    assert ops.status(ws) == 0
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


@pytest.mark.parametrize("name", ["dsv3_dense_b64_h128_l1k_8k", "tiny_dense_b1_h16_l256"])
def test_static_entry_matches_workspace_entry_twice(name):
    c = inputs.make_workload(name, device="cuda")
    ref_out, ref_lse = _with_workspace(c)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        out, lse = ops.decode_static(c.q_nope, c.q_rope, c.cache, c.block_table, c.seq_lens,
                                     c.scale, device_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert_close(out, lse, ref_out, ref_lse, f"static {name}")


def test_static_entry_split_requests():
    # long requests force split-KV partials into the fixed scratch
    c = inputs.make_case(3, 128, [20000, 3, 9000], seed=31).to("cuda")
    ref_out, ref_lse = _with_workspace(c)
    for _ in range(2):
        out, lse = ops.decode_static(c.q_nope, c.q_rope, c.cache, c.block_table, c.seq_lens,
                                     c.scale)
        assert_close(out, lse, ref_out, ref_lse, "static split")


def test_static_entry_fp8_records_twice():
    # a ragged batch over an FP8-record cache, with one request long enough to be split
    c = inputs.make_case(5, 128, [64, 700, 2500, 1, 9000], seed=33, kv_dtype="fp8").to("cuda")
    ref_out, ref_lse = _with_workspace(c)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        out, lse = ops.decode_static(c.q_nope, c.q_rope, c.cache, c.block_table, c.seq_lens,
                                     c.scale, device_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert_close(out, lse, ref_out, ref_lse, "static fp8")


def test_static_entry_rejects_batches_beyond_the_fixed_array():
    c = inputs.make_case(400, 128, [64] * 400, seed=2).to("cuda")
    with pytest.raises(ops.MlaError) as e:
        ops.decode_static(c.q_nope, c.q_rope, c.cache, c.block_table, c.seq_lens, c.scale)
    assert e.value.status == 3
