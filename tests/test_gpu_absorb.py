"""GPU parity of the query absorption and the value projection (through the C ABI) against
the CPU oracle: elementwise within |x - ref| <= 1e-2 + 1e-2 |ref| (bf16 inputs, fp32
accumulation, bf16 rounding of q~ or of the latent output), bit-exact where the weights
only select entries, and the whole chain absorb -> decode -> project against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from mla_latent_kv_17_gb300 import inputs, ops

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-2, 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mla_latent_kv_17_gb300 import build
    build.build()
    ops.lib()


def _f64(t):
    return t.detach().float().cpu().double().numpy()


def _close(got, ref, what):
    err = np.abs(got - ref)
    bad = ~(err <= ATOL + RTOL * np.abs(ref))
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: mismatch at {i}: got {got[i]} ref {ref[i]} ({bad.sum()} of {bad.size})")


# request counts: one, a full tile of 64, ragged tails over two and four tiles
SIZES = [(1, 128), (64, 128), (130, 3), (200, 16)]


@pytest.mark.parametrize("B,H", SIZES)
def test_absorb_matches_oracle(B, H):
    q_c, w_uk, _, _ = inputs.projection_inputs(B, H, seed=40 + B)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = ops.absorb_query(q_c.cuda(), w_uk.cuda(), device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _close(_f64(got), oracle.absorb(_f64(q_c), _f64(w_uk)), f"absorb B={B} H={H}")


@pytest.mark.parametrize("B,H", SIZES)
def test_project_matches_oracle(B, H):
    _, _, w_uv, out = inputs.projection_inputs(B, H, seed=50 + B)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = ops.project_output(out.cuda(), w_uv.cuda(), device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _close(_f64(got), oracle.project(_f64(out), _f64(w_uv)), f"project B={B} H={H}")


def test_absorb_identity_block_is_exact():
    # W^UK of head h = identity onto latent columns 128 ((h + 1) % 4) ..: q~ equals q^C there
    # and is zero elsewhere, bit for bit (one nonzero term per sum)
    B, H = 70, 5
    q_c, _, _, _ = inputs.projection_inputs(B, H, seed=61)
    w = torch.zeros(H, 128, 512)
    for h in range(H):
        c0 = 128 * ((h + 1) % 4)
        w[h, torch.arange(128), c0 + torch.arange(128)] = 1.0
    ref = oracle.absorb(_f64(q_c), w.double().numpy())
    got = ops.absorb_query(q_c.cuda(), w.to(torch.bfloat16).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(_f64(got), ref)


def test_project_column_selection_is_exact():
    # W^UV row j of head h selects latent column perm_h[j]: y = bf16(out) at those columns
    B, H = 97, 4
    _, _, _, out = inputs.projection_inputs(B, H, seed=62)
    g = torch.Generator().manual_seed(63)
    w = torch.zeros(H, 128, 512)
    for h in range(H):
        w[h, torch.arange(128), torch.randperm(512, generator=g)[:128]] = 1.0
    out_b = out.to(torch.bfloat16).float()  # the MMA operand is the bf16 latent output
    ref = oracle.project(_f64(out_b), w.double().numpy())
    got = ops.project_output(out.cuda(), w.to(torch.bfloat16).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(_f64(got), ref)


def test_absorbed_decode_chain_matches_oracle():
    # absorb -> plan -> decode -> project on one stream against the oracle's chain (the
    # oracle's q~ rounded to bf16, the decode's input type)
    lens = [300, 64, 1000, 1]
    H = 128
    c = inputs.make_case(len(lens), H, lens, seed=64)
    q_c, w_uk, w_uv, _ = inputs.projection_inputs(c.B, H, seed=65)
    q_abs = torch.from_numpy(oracle.absorb(_f64(q_c), _f64(w_uk))).to(torch.bfloat16)
    c.q_nope = q_abs
    ro, _ = oracle.decode_dense(c.q_nope, c.q_rope, c.cache, c.block_table, c.seq_lens, c.scale)
    ref = oracle.project(ro, _f64(w_uv))

    c = c.to("cuda")
    ws = ops.Workspace(c.B, H)
    q_nope = ops.absorb_query(q_c.cuda(), w_uk.cuda())
    ops.plan(ws, c.seq_lens)
    out, _ = ops.decode(ws, q_nope, c.q_rope, c.cache, c.block_table, c.seq_lens, c.scale)
    y = ops.project_output(out, w_uv.cuda())
    torch.cuda.synchronize()
    assert ops.status(ws) == 0
    _close(_f64(y), ref, "absorb -> decode -> project")
