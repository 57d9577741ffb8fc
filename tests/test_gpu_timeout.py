"""The decode kernel's bounded waits: a wait that runs out is reported, and the device and
the workspace stay usable.

The injected stall (mla_decode_inject_stall) makes the kernel's tensor-core issuer wait on
a barrier that nothing completes; with the wait limit lowered to about ten milliseconds
that wait runs out, the call records MLA_ERR_TIMEOUT, every other role of the kernel sees
the abort and winds down, and the kernel frees its tensor memory and returns.  Nothing
faults or traps.  The next call on the same workspace, with the hook off and the default
limit back, must succeed and match the oracle.
"""
import pytest
import torch

from mla_latent_kv_17_gb300 import inputs, ops
from guards import Guarded, guarded_workspace
from oracle_ref import assert_close, assert_close_fp8, oracle_for

pytestmark = pytest.mark.gpu

STALL_LIMIT_CYCLES = 20_000_000   # ~10 ms at 2 GHz


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mla_latent_kv_17_gb300 import build
    build.build()
    ops.lib()
    yield
    ops.inject_stall(False)
    ops.set_wait_limit(0)


def _case(kind):
    if kind == "sparse":
        c = inputs.make_case(2, 128, [700, 3000], seed=61, extra_pages=2)
        c.indices = inputs.sparse_indices(c.seq_lens, 256, 64, 61)
        return c.to("cuda")
    return inputs.make_case(3, 128, [300, 2000, 65], seed=62, kv_dtype=kind).to("cuda")


def _decode(c, ws, out, lse):
    if c.indices is not None:
        ops.decode_sparse(ws, c.q_nope, c.q_rope, c.cache, c.block_table, c.seq_lens, c.indices,
                          c.scale, out=out, lse=lse)
    else:
        ops.decode(ws, c.q_nope, c.q_rope, c.cache, c.block_table, c.seq_lens, c.scale, out=out,
                   lse=lse)


@pytest.mark.parametrize("kind", ["bf16", "fp8", "sparse"])
def test_wait_that_runs_out_is_reported_and_the_next_call_is_clean(kind):
    c = _case(kind)
    ws = guarded_workspace(c.B, c.H)
    topk = c.indices.shape[1] if c.indices is not None else 0
    ops.plan(ws, c.seq_lens if topk == 0 else None, topk=topk, kv_dtype=c.kv_dtype)
    out_g, lse_g = Guarded(c.B * c.H * 512 * 4), Guarded(c.B * c.H * 4)
    out = out_g.inner.view(torch.float32).view(c.B, c.H, 512)
    lse = lse_g.inner.view(torch.float32).view(c.B, c.H)
    ops.set_wait_limit(STALL_LIMIT_CYCLES)
    ops.inject_stall(True)
    try:
        _decode(c, ws, out, lse)
        st = ops.status(ws)
    finally:
        ops.inject_stall(False)
        ops.set_wait_limit(0)
    assert st == 6, ops.STATUS_NAMES.get(st, st)           # MLA_ERR_TIMEOUT
    assert ops.status(ws) == 0                               # read once, then cleared
    # the same workspace and plan, default limit: a normal call
    _decode(c, ws, out, lse)
    st = ops.status(ws)
    assert st == 0, ops.STATUS_NAMES.get(st, st)
    for g, what in ((out_g, "out"), (lse_g, "lse"), (ws.guard, "workspace")):
        g.check(what)
    ref_out, ref_lse = oracle_for(c)
    if kind == "fp8":
        assert_close_fp8(out, lse, ref_out, ref_lse, c, "after timeout (fp8)")
    else:
        assert_close(out, lse, ref_out, ref_lse, f"after timeout ({kind})")
