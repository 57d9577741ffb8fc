"""GPU parity of the DSA top-k selection (through the C ABI) against the CPU oracle: index
lists must be identical (integer work; both sides order fp32 scores exactly, ties to the
lower position), including tie-heavy scores, signed zeros and infinities, short and empty
requests, a padded row stride, the full 64 x 65536 top-2048 size, and a sparse decode
over the selected indices."""
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


def _run(scores, lens, k):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = ops.topk_select(scores.cuda() if not scores.is_cuda else scores,
                          torch.as_tensor(lens, dtype=torch.int32).cuda(), k, device_status=status)
    torch.cuda.synchronize()
    return got.cpu().numpy(), int(status.item())


def test_topk_random_scores_equal_oracle():
    g = torch.Generator().manual_seed(70)
    lens = [5000, 701, 700, 3, 0, 4097]
    s = torch.randn(len(lens), 5000 + 100, generator=g)
    got, st = _run(s, lens, 700)
    assert st == 0
    assert np.array_equal(got, oracle.topk_select(s.numpy(), lens, 700))


def test_topk_tie_heavy_scores_equal_oracle():
    g = torch.Generator().manual_seed(71)
    vals = torch.tensor([-2.0, -0.0, 0.0, 0.5, 1.0, 3.0, float("inf"), float("-inf"), 1e-42, -1e-42])
    B, Lmax = 16, 3000
    s = vals[torch.randint(0, vals.numel(), (B, Lmax), generator=g)]
    lens = torch.randint(0, Lmax + 1, (B,), generator=g).tolist()
    lens[0], lens[1] = Lmax, 1000
    for k in (1, 999, 1000, 2048):
        got, st = _run(s, lens, k)
        assert st == 0
        assert np.array_equal(got, oracle.topk_select(s.numpy(), lens, k)), k


def test_topk_padded_row_stride():
    g = torch.Generator().manual_seed(72)
    full = torch.randn(7, 2052, generator=g).cuda()
    view = full[:, :2049]  # Lmax 2049, row stride 2052
    lens = [2049, 2048, 17, 1500, 0, 2000, 1]
    got, st = _run(view, lens, 256)
    assert st == 0
    assert np.array_equal(got, oracle.topk_select(full.cpu().numpy()[:, :2049], lens, 256))


def test_topk_dsa_size_equals_oracle():
    # 64 requests x 65536 scored positions, top 2048 (the DSA decode workload's shape)
    g = torch.Generator().manual_seed(73)
    s = torch.randn(64, 65536, generator=g)
    lens = [65536] * 60 + [65535, 2049, 2048, 100]
    got, st = _run(s, lens, 2048)
    assert st == 0
    assert np.array_equal(got, oracle.topk_select(s.numpy(), lens, 2048))


def test_topk_long_requests_reread_scores():
    # longer than the shared-memory key cache (32,768 keys): the candidates at or above the
    # first pass's bin go to a list in shared memory (a block of ties above everything else
    # in the second request)
    g = torch.Generator().manual_seed(76)
    s = torch.randn(2, 150000, generator=g)
    s[1, 1000:3000] = 5.0  # a block of ties above everything else
    lens = [150000, 149999]
    got, st = _run(s, lens, 2048)
    assert st == 0
    assert np.array_equal(got, oracle.topk_select(s.numpy(), lens, 2048))


def test_topk_long_requests_with_too_many_candidates():
    # past the key cache, and more positions in the selected bin than the candidate list holds
    # (16,384): all equal, or a wide block of equal scores at the k-th best value, so the later
    # passes read the scores again
    g = torch.Generator().manual_seed(77)
    s = torch.randn(3, 40000, generator=g)
    s[0, :] = 1.0
    s[1, 5000:30000] = 4.0        # 25,000 ties above everything else
    s[2, :] = -0.0
    s[2, 39000:] = 0.0            # signed zeros share a key
    lens = [40000, 40000, 33000]
    got, st = _run(s, lens, 2048)
    assert st == 0
    assert np.array_equal(got, oracle.topk_select(s.numpy(), lens, 2048))


@pytest.mark.parametrize("width", [32768, 32772])
def test_topk_cache_boundary_lengths(width):
    # rows of 32,768 positions fit the key cache, rows of 32,772 do not (candidate list)
    g = torch.Generator().manual_seed(78)
    s = torch.randn(4, width, generator=g)
    lens = [width, width - 1, 32767, 20000]
    got, st = _run(s, lens, 1000)
    assert st == 0
    assert np.array_equal(got, oracle.topk_select(s.numpy(), lens, 1000))


def test_topk_bad_length_is_reported():
    s = torch.randn(3, 64)
    got, st = _run(s, [10, 65, -1], 8)
    assert st == 5  # MLA_ERR_INDEX
    assert got[0].tolist() == oracle.topk_select(s.numpy()[:1], [10], 8)[0].tolist()
    assert (got[1] == -1).all() and (got[2] == -1).all()


def test_sparse_decode_over_selected_indices():
    lens = [3000, 500, 2100]
    c = inputs.make_case(len(lens), 128, lens, seed=74)
    g = torch.Generator().manual_seed(75)
    s = torch.randn(c.B, 3000, generator=g)
    idx_ref = oracle.topk_select(s.numpy(), lens, 1024)
    c.indices = torch.from_numpy(idx_ref)
    ro, rl = oracle_for(c)
    c = c.to("cuda")
    idx = ops.topk_select(s.cuda(), c.seq_lens, 1024)
    assert np.array_equal(idx.cpu().numpy(), idx_ref)
    ws = ops.Workspace(c.B, c.H)
    ops.plan(ws, None, topk=1024)
    out, lse = ops.decode_sparse(ws, c.q_nope, c.q_rope, c.cache, c.block_table, c.seq_lens, idx, c.scale)
    assert ops.status(ws) == 0
    assert_close(out, lse, ro, rl, "sparse decode over selected indices")
