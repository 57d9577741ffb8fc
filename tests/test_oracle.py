"""Pins for the CPU oracle: each test checks it against something other than itself.

The pages print no worked attention example, so the oracle is pinned by closed-form
algebra (the absorption identity of "MLA 在极长上下文下的显存带宽突围", run-time matrix
absorption), textbook special cases, a library decoder for the FP8 format, brute force on
tiny inputs, and structural invariants (split + merge, sparse with every index = dense).
Each pin is chosen so that a plausible slip in the oracle (a dropped RoPE term, a wrong
scale, a transposed operand, an off-by-one page row, a wrong FP8 scale group) fails it.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from mla_latent_kv_17_gb300 import inputs

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")
SCALE = 1.0 / math.sqrt(192.0)


def _rng(seed):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------------------
# absorbed == non-absorbed (closed-form algebra; P4 run-time matrix absorption, P1 §1.1)
# --------------------------------------------------------------------------------------
@pytest.mark.parametrize("H,N", [(1, 1), (3, 7), (8, 129)])
def test_absorbed_equals_nonabsorbed(H, N):
    r = _rng(100 + H * N)
    d_h = 128
    qC = r.standard_normal((H, d_h))
    qR = r.standard_normal((H, 64))
    W_UK = r.standard_normal((H, d_h, 512)) / math.sqrt(512)
    W_UV = r.standard_normal((H, d_h, 512)) / math.sqrt(512)
    C = r.standard_normal((N, 512))
    KR = r.standard_normal((N, 64))

    # Non-absorbed (MHA mode): decompress per-head keys/values, standard attention with
    # the 192-wide key [K_h | k_R] and query [q^C_h | q^R_h].
    ref_out = np.zeros((H, d_h))
    ref_lse = np.zeros(H)
    for h in range(H):
        K = C @ W_UK[h].T               # [N, 128]
        V = C @ W_UV[h].T               # [N, 128]
        s = (K @ qC[h] + KR @ qR[h]) * SCALE
        m = s.max()
        p = np.exp(s - m)
        ref_out[h] = (p / p.sum()) @ V
        ref_lse[h] = m + math.log(p.sum())

    # Absorbed: q~ = q^C W^UK, attend in latent space, project the latent output with W^UV.
    q_abs = np.stack([qC[h] @ W_UK[h] for h in range(H)])      # [H, 512]
    out_lat, lse = oracle.attend_f64(q_abs, qR, C, KR, SCALE)
    proj = np.stack([W_UV[h] @ out_lat[h] for h in range(H)])
    np.testing.assert_allclose(proj, ref_out, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def _absorb_project_pins(absorb, project):
    """Pins of the absorption and output projection, as a list of (name, ok) over the pair.

    1. absorbed decode through absorb/project == non-absorbed attention over decompressed
       per-head keys and values (the two never share a product);
    2. W^UK = identity on a head-dependent block of 128 latent columns gives q~ = q^C there
       and zeros elsewhere; W^UV selecting a head-dependent permutation of latent columns
       gives y = those entries of out;
    3. adjoint: <absorb(q, W), X> == <q, project(X, W)> for any X (absorb and project use
       the same matrix, once as q W and once as W x)."""
    r = _rng(71)
    res = []
    B, H, N, d_h = 2, 3, 13, 128
    qC = r.standard_normal((B, H, d_h))
    qR = r.standard_normal((B, H, 64))
    W_UK = r.standard_normal((H, d_h, 512)) / math.sqrt(512)
    W_UV = r.standard_normal((H, d_h, 512)) / math.sqrt(512)
    C = r.standard_normal((N, 512))
    KR = r.standard_normal((N, 64))
    q_abs = absorb(qC, W_UK)
    lat = np.zeros((B, H, 512))
    ok = True
    for b in range(B):
        o, _ = oracle.attend_f64(q_abs[b], qR[b], C, KR, SCALE)
        lat[b] = o
    y = project(lat, W_UV)
    for b in range(B):
        for h in range(H):
            K, V = C @ W_UK[h].T, C @ W_UV[h].T
            sc = (K @ qC[b, h] + KR @ qR[b, h]) * SCALE
            pr = np.exp(sc - sc.max())
            ok &= np.allclose(y[b, h], (pr / pr.sum()) @ V, rtol=1e-9, atol=1e-12)
    res.append(("absorbed == non-absorbed", bool(ok)))

    E = np.zeros((H, d_h, 512))
    for h in range(H):
        c0 = 128 * ((h + 1) % 4)
        E[h, np.arange(d_h), c0 + np.arange(d_h)] = 1.0
    qa = absorb(qC, E)
    ok = True
    for h in range(H):
        c0 = 128 * ((h + 1) % 4)
        ok &= np.array_equal(qa[:, h, c0:c0 + d_h], qC[:, h])
        ok &= not np.any(np.delete(qa[:, h], np.s_[c0:c0 + d_h], axis=1))
    res.append(("identity block", bool(ok)))

    Pm = np.zeros((H, d_h, 512))
    perms = [r.permutation(512)[:d_h] for _ in range(H)]
    for h in range(H):
        Pm[h, np.arange(d_h), perms[h]] = 1.0
    X = r.standard_normal((B, H, 512))
    yp = project(X, Pm)
    ok = all(np.array_equal(yp[:, h], X[:, h][:, perms[h]]) for h in range(H))
    res.append(("column selection", bool(ok)))

    lhs = float(np.sum(absorb(qC, W_UK) * X))
    rhs = float(np.sum(qC * project(X, W_UK)))
    res.append(("adjoint", abs(lhs - rhs) <= 1e-10 * max(1.0, abs(lhs))))
    return res


def test_absorb_and_project_pins():
    bad = [n for n, ok in _absorb_project_pins(oracle.absorb, oracle.project) if not ok]
    assert not bad, bad


# --------------------------------------------------------------------------------------
# DSA top-k selection (guide §1.2: the k best-scored earlier tokens, "GPU partial sort")
# --------------------------------------------------------------------------------------
def _topk_brute(scores, L, k):
    """Position t is kept iff fewer than min(k, L) positions beat it: a higher score, or an
    equal score at a lower position (pure Python, O(L^2))."""
    K = min(k, L)
    keep = []
    for t in range(L):
        beat = sum(1 for u in range(L) if scores[u] > scores[t] or (scores[u] == scores[t] and u < t))
        if beat < K:
            keep.append(t)
    return keep + [-1] * (k - len(keep))


def test_topk_matches_brute_force_on_tiny_inputs():
    r = _rng(90)
    for trial in range(40):
        Lmax = int(r.integers(1, 40))
        k = int(r.integers(1, 45))
        B = 3
        # few distinct values, so ties are common; signed zeros included
        s = r.choice(np.array([-1.5, -0.0, 0.0, 0.25, 2.0, 7.0], dtype=np.float32), size=(B, Lmax))
        lens = r.integers(0, Lmax + 1, size=B)
        got = oracle.topk_select(s, lens, k)
        for b in range(B):
            assert got[b].tolist() == _topk_brute(s[b].tolist(), int(lens[b]), k)


def test_topk_special_cases():
    L, k = 100, 16
    eq = np.ones((1, L), np.float32)
    assert oracle.topk_select(eq, [L], k)[0].tolist() == list(range(k))          # all tied
    dec = -np.arange(L, dtype=np.float32)[None]
    assert oracle.topk_select(dec, [L], k)[0].tolist() == list(range(k))         # decreasing
    inc = np.arange(L, dtype=np.float32)[None]
    assert oracle.topk_select(inc, [L], k)[0].tolist() == list(range(L - k, L))  # increasing
    short = oracle.topk_select(inc, [5], k)[0].tolist()
    assert short == list(range(5)) + [-1] * (k - 5)                              # L < k
    assert oracle.topk_select(inc, [0], k)[0].tolist() == [-1] * k               # empty
    z = np.array([[0.0, -0.0, 0.0, -0.0]], np.float32)                           # -0 == +0
    assert oracle.topk_select(z, [4], 2)[0].tolist() == [0, 1]


def test_topk_invariants_on_random_scores():
    r = _rng(91)
    B, Lmax, k = 4, 5000, 700
    s = r.standard_normal((B, Lmax)).astype(np.float32)
    lens = np.array([5000, 701, 700, 3])
    got = oracle.topk_select(s, lens, k)
    for b in range(B):
        L = int(lens[b])
        sel = got[b][got[b] >= 0]
        assert sel.size == min(k, L) and np.all(np.diff(sel) > 0) and np.all(sel < L)
        rest = np.setdiff1d(np.arange(L), sel)
        if rest.size:
            assert s[b, sel].min() >= s[b, rest].max()


# --------------------------------------------------------------------------------------
# Non-absorbed causal prefill (guide §3.1; operator survey §4)
# --------------------------------------------------------------------------------------
def _prefill_inputs(L, H, seed):
    r = _rng(seed)
    E = r.standard_normal((L, 576))
    qn = r.standard_normal((L, H, 128))
    qr = r.standard_normal((L, H, 64))
    wk = r.standard_normal((H, 128, 512)) / math.sqrt(512)
    wv = r.standard_normal((H, 128, 512)) / math.sqrt(512)
    return E, qn, qr, wk, wv


def _prefill_pins(prefill):
    """(name, ok) pairs over a prefill function: rows equal the absorbed decode of the same
    query over tokens 0..i projected with W^UV (the identity that lets decode skip the
    decompression); row 0 sees one key (out = W^UV c_0, lse = its scaled score); zero
    queries give uniform weights over t <= i (mean of the values, lse = ln(i + 1))."""
    res = []
    L, H = 9, 3
    E, qn, qr, wk, wv = _prefill_inputs(L, H, 80)
    out, lse = prefill(E, qn, qr, wk, wv, SCALE)
    q_abs = oracle.absorb(qn, wk)
    ok = True
    for i in range(L):
        lat, l2 = oracle.attend_f64(q_abs[i], qr[i], E[:i + 1, :512], E[:i + 1, 512:], SCALE)
        y = oracle.project(lat[None], wv)[0]
        ok &= np.allclose(out[i], y, rtol=1e-9, atol=1e-12) and np.allclose(lse[i], l2, rtol=1e-12, atol=1e-12)
    res.append(("rows == absorbed decode", bool(ok)))
    ok = True
    for h in range(H):
        ok &= np.allclose(out[0, h], wv[h] @ E[0, :512], rtol=1e-12, atol=1e-12)
        s0 = SCALE * (qn[0, h] @ (wk[h] @ E[0, :512]) + qr[0, h] @ E[0, 512:])
        ok &= abs(lse[0, h] - s0) < 1e-12
    res.append(("row 0", bool(ok)))
    out0, lse0 = prefill(E, np.zeros_like(qn), np.zeros_like(qr), wk, wv, SCALE)
    ok = True
    for i in range(L):
        for h in range(H):
            ok &= np.allclose(out0[i, h], (wv[h] @ E[:i + 1, :512].T).mean(axis=1), rtol=1e-12, atol=1e-12)
            ok &= abs(lse0[i, h] - math.log(i + 1)) < 1e-12
    res.append(("uniform weights", bool(ok)))
    return res


def test_prefill_pins():
    bad = [n for n, ok in _prefill_pins(oracle.prefill) if not ok]
    assert not bad, bad


def test_prefill_bf16_keys_values():
    """kv_bf16 equals the exact prefill run on keys and values rounded to bf16 beforehand:
    with W^UK, W^UV the identity on the first 128 latent columns the decompressed K, V are
    those columns, so rounding the entries themselves to bf16 must give the same result."""
    L, H = 7, 2
    E, qn, qr, _, _ = _prefill_inputs(L, H, 82)
    I = np.zeros((H, 128, 512))
    I[:, np.arange(128), np.arange(128)] = 1.0
    got, gl = oracle.prefill(E, qn, qr, I, I, SCALE, kv_bf16=True)
    Eb = E.copy()
    f = E[:, :128].astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16                        # binary32 -> bf16, nearest even
    Eb[:, :128] = u.astype(np.uint32).view(np.float32).astype(np.float64)
    ref, rl = oracle.prefill(Eb, qn, qr, I, I, SCALE)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(gl, rl, rtol=1e-12, atol=1e-12)
    assert np.abs(got - oracle.prefill(E, qn, qr, I, I, SCALE)[0]).max() > 1e-6  # the rounding shows


def test_rope_term_and_scale_matter():
    """Changing only k_R or only the scale must change the result (guards dropped terms)."""
    r = _rng(5)
    q, qr = r.standard_normal((2, 512)), r.standard_normal((2, 64))
    C, K = r.standard_normal((9, 512)), r.standard_normal((9, 64))
    o1, l1 = oracle.attend_f64(q, qr, C, K, SCALE)
    o2, l2 = oracle.attend_f64(q, qr, C, K * 2.0, SCALE)
    o3, l3 = oracle.attend_f64(q, qr, C, K, SCALE * 0.5)
    assert np.abs(o1 - o2).max() > 1e-3 and np.abs(l1 - l2).max() > 1e-3
    assert np.abs(o1 - o3).max() > 1e-3


# --------------------------------------------------------------------------------------
# Textbook special cases
# --------------------------------------------------------------------------------------
def test_weights_sum_to_one():
    r = _rng(1)
    v = r.standard_normal(512)
    C = np.tile(v, (37, 1))
    out, _ = oracle.attend_f64(r.standard_normal((4, 512)) * 3, r.standard_normal((4, 64)), C,
                               r.standard_normal((37, 64)), SCALE)
    np.testing.assert_allclose(out, np.tile(v, (4, 1)), rtol=1e-12, atol=1e-12)


def test_output_in_convex_hull():
    r = _rng(2)
    C = r.standard_normal((50, 512))
    out, _ = oracle.attend_f64(r.standard_normal((6, 512)) * 4, r.standard_normal((6, 64)), C,
                               r.standard_normal((50, 64)), SCALE)
    assert np.all(out <= C.max(axis=0) + 1e-12) and np.all(out >= C.min(axis=0) - 1e-12)


def test_single_token():
    r = _rng(3)
    q, qr = r.standard_normal((5, 512)), r.standard_normal((5, 64))
    C, K = r.standard_normal((1, 512)), r.standard_normal((1, 64))
    out, lse = oracle.attend_f64(q, qr, C, K, SCALE)
    np.testing.assert_array_equal(out, np.tile(C[0], (5, 1)))
    s0 = np.array([SCALE * (np.dot(q[h], C[0]) + np.dot(qr[h], K[0])) for h in range(5)])
    np.testing.assert_allclose(lse, s0, rtol=1e-13, atol=1e-13)


def test_zero_query_gives_mean_and_log_n():
    r = _rng(4)
    N = 77
    C = r.standard_normal((N, 512))
    out, lse = oracle.attend_f64(np.zeros((3, 512)), np.zeros((3, 64)), C,
                                 r.standard_normal((N, 64)), SCALE)
    np.testing.assert_allclose(out, np.tile(C.mean(axis=0), (3, 1)), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, np.full(3, math.log(N)), rtol=1e-14)


def test_empty_token_list():
    out, lse = oracle.attend_f64(np.ones((2, 512)), np.ones((2, 64)), np.zeros((0, 512)),
                                 np.zeros((0, 64)), SCALE)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_bruteforce_tiny_paged():
    """Pure-Python softmax without the max shift, gathering rows through the block table."""
    for seed, (B, H, lens) in enumerate([(1, 1, [1]), (2, 3, [5, 8]), (2, 4, [8, 3])]):
        c = inputs.make_case(B, H, lens, seed=seed, extra_pages=3)
        c.cache[:] = c.cache.float().clamp(-2, 2).to(torch.bfloat16)  # tiny case: no NaN tail
        out, lse = oracle.decode_dense(c.q_nope, c.q_rope, c.cache, c.block_table, c.seq_lens,
                                       SCALE)
        qn, qr = c.q_nope.double().numpy(), c.q_rope.double().numpy()
        cache = c.cache.double().numpy()
        bt = c.block_table.numpy()
        for b in range(B):
            for h in range(H):
                ws, acc = [], [0.0] * 512
                for t in range(lens[b]):
                    row = cache[bt[b, t // 64], t % 64]
                    s = sum(qn[b, h, i] * row[i] for i in range(512))
                    s += sum(qr[b, h, i] * row[512 + i] for i in range(64))
                    ws.append(math.exp(SCALE * s))
                z = sum(ws)
                for t in range(lens[b]):
                    row = cache[bt[b, t // 64], t % 64]
                    for i in range(512):
                        acc[i] += ws[t] / z * row[i]
                np.testing.assert_allclose(out[b, h], acc, rtol=1e-10, atol=1e-12)
                assert abs(lse[b, h] - math.log(z)) < 1e-10


def test_one_hot_reads_the_mapped_row():
    """Row r of physical page p holds the code (p, r); a dominant score on one token makes
    the output equal that row, so the output names the row the oracle read."""
    B, H = 2, 2
    lens = [130, 70]
    c = inputs.make_case(B, H, lens, seed=9, extra_pages=5)
    P = c.cache.shape[0]
    cache = torch.zeros((P, 64, 576), dtype=torch.float32)
    for p in range(P):
        for r in range(64):
            cache[p, r, 0] = p
            cache[p, r, 1] = r
    qn = torch.zeros((B, H, 512))
    qr = torch.zeros((B, H, 64))
    targets = [[0, 129], [69, 3]]
    cache[:, :, 512:] = 0
    for b in range(B):
        for h in range(H):
            t = targets[b][h]
            p = int(c.block_table[b, t // 64])
            cache[p, t % 64, 512 + 8 * h + b] = 1.0   # unique marker key for (b, h)
            qr[b, h, 8 * h + b] = 1000.0   # exp(-1000) underflows to 0 in double
    out, lse = oracle.decode_dense(qn.to(torch.bfloat16), qr.to(torch.bfloat16),
                                   cache.to(torch.bfloat16), c.block_table, c.seq_lens, 1.0)
    for b in range(B):
        for h in range(H):
            t = targets[b][h]
            assert out[b, h, 0] == int(c.block_table[b, t // 64])
            assert out[b, h, 1] == t % 64


# --------------------------------------------------------------------------------------
# Structural invariants: split + merge, sparse with all indices, duplicates
# --------------------------------------------------------------------------------------
def _dense_case(B=2, H=4, lens=(200, 131), seed=11):
    return inputs.make_case(B, H, list(lens), seed=seed, extra_pages=2)


def test_sparse_all_indices_equals_dense():
    c = _dense_case()
    topk = int(c.seq_lens.max())
    idx = torch.full((c.B, topk), -1, dtype=torch.int32)
    perm_idx = idx.clone()
    g = torch.Generator().manual_seed(0)
    for b, L in enumerate(c.seq_lens.tolist()):
        idx[b, :L] = torch.arange(L)
        perm_idx[b, :L] = torch.randperm(L, generator=g).to(torch.int32)
    d_out, d_lse = oracle.decode_dense(c.q_nope, c.q_rope, c.cache, c.block_table, c.seq_lens, SCALE)
    for ix in (idx, perm_idx):
        s_out, s_lse = oracle.decode_sparse(c.q_nope, c.q_rope, c.cache, c.block_table,
                                            c.seq_lens, ix, SCALE)
        np.testing.assert_allclose(s_out, d_out, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(s_lse, d_lse, rtol=1e-13, atol=1e-13)


def test_split_and_merge_equals_single_pass():
    c = _dense_case(B=1, H=3, lens=(300,))
    L = 300
    d_out, d_lse = oracle.decode_dense(c.q_nope, c.q_rope, c.cache, c.block_table, c.seq_lens, SCALE)
    for cuts in ([0, 1, 2, 300], [0, 64, 128, 192, 256, 300], [0, 150, 300], [0, 299, 300]):
        parts_o, parts_l = [], []
        for a, e in zip(cuts[:-1], cuts[1:]):
            ix = torch.full((1, L), -1, dtype=torch.int32)
            ix[0, :e - a] = torch.arange(a, e)
            o, l = oracle.decode_sparse(c.q_nope, c.q_rope, c.cache, c.block_table, c.seq_lens,
                                        ix, SCALE)
            parts_o.append(o[0])
            parts_l.append(l[0])
        po, pl = np.stack(parts_o), np.stack(parts_l)   # [S, H, 512], [S, H]
        for h in range(3):
            o, l = oracle.combine(po[:, h], pl[:, h])
            np.testing.assert_allclose(o, d_out[0, h], rtol=1e-11, atol=1e-13)
            assert abs(l - d_lse[0, h]) < 1e-12


def test_combine_empty_chunks():
    o, l = oracle.combine(np.zeros((3, 8)), np.full(3, -np.inf))
    assert np.all(o == 0) and l == -np.inf
    x = np.arange(8.0)
    o, l = oracle.combine(np.stack([x, np.zeros(8)]), np.array([0.5, -np.inf]))
    np.testing.assert_array_equal(o, x)
    assert l == 0.5


def test_sparse_duplicate_counts_twice_and_padding_skipped():
    c = _dense_case(B=1, H=2, lens=(40,))
    ix = torch.tensor([[5, 5, -1, 17, -1]], dtype=torch.int32)
    out, lse = oracle.decode_sparse(c.q_nope, c.q_rope, c.cache, c.block_table, c.seq_lens, ix,
                                    SCALE)
    cache = c.cache.double().numpy()
    rows = [cache[int(c.block_table[0, t // 64]), t % 64] for t in (5, 5, 17)]
    C = np.stack([r[:512] for r in rows])
    K = np.stack([r[512:] for r in rows])
    ref_o, ref_l = oracle.attend_f64(c.q_nope[0].double().numpy(), c.q_rope[0].double().numpy(),
                                     C, K, SCALE)
    np.testing.assert_allclose(out[0], ref_o, rtol=1e-13)
    np.testing.assert_allclose(lse[0], ref_l, rtol=1e-13)


def test_all_padding_and_zero_length():
    c = inputs.make_case(2, 2, [0, 10], seed=3)
    out, lse = oracle.decode_dense(c.q_nope, c.q_rope, c.cache, c.block_table, c.seq_lens, SCALE)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0])) and np.all(np.isfinite(lse[1]))
    ix = torch.full((2, 4), -1, dtype=torch.int32)
    out, lse = oracle.decode_sparse(c.q_nope, c.q_rope, c.cache, c.block_table, c.seq_lens, ix, SCALE)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_nan_tail_rows_never_read():
    c = inputs.make_case(3, 2, [1, 63, 65], seed=4)
    assert torch.isnan(c.cache.float()).any()
    out, lse = oracle.decode_dense(c.q_nope, c.q_rope, c.cache, c.block_table, c.seq_lens, SCALE)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))


def test_out_of_range_index_rejected():
    c = _dense_case(B=1, H=1, lens=(10,))
    with pytest.raises(ValueError):
        oracle.decode_sparse(c.q_nope, c.q_rope, c.cache, c.block_table, c.seq_lens,
                             torch.tensor([[10]], dtype=torch.int32), SCALE)
    with pytest.raises(ValueError):
        oracle.decode_sparse(c.q_nope, c.q_rope, c.cache, c.block_table, c.seq_lens,
                             torch.tensor([[-2]], dtype=torch.int32), SCALE)


# --------------------------------------------------------------------------------------
# FP8 latent cache
# --------------------------------------------------------------------------------------
def test_e4m3_decoder_against_library_and_format_constants():
    lib = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double()
    for code in range(256):
        v = oracle.e4m3_to_float(code)
        ref = float(lib[code])
        if math.isnan(ref):
            assert math.isnan(v)
        else:
            assert v == ref, (code, v, ref)
    # OCP FP8 e4m3: max normal 448, min normal 2^-6, min subnormal 2^-9, 1.0 = 0x38.
    assert oracle.e4m3_to_float(0x7E) == 448.0
    assert oracle.e4m3_to_float(0x08) == 2.0 ** -6
    assert oracle.e4m3_to_float(0x01) == 2.0 ** -9
    assert oracle.e4m3_to_float(0x38) == 1.0 and oracle.e4m3_to_float(0xB8) == -1.0
    assert math.isnan(oracle.e4m3_to_float(0x7F)) and math.isnan(oracle.e4m3_to_float(0xFF))


def _fp8_scales():
    g = torch.Generator().manual_seed(3)
    return torch.cat([torch.tensor([1.0, 1.0 / 448, 3.7e-3]), torch.rand(5, generator=g) * 0.05 + 1e-4]).float()


def test_fp8_latent_exact_is_code_times_scale():
    # the definition (guide §5.3: an FP8 code and its block scale): every code against
    # torch's own e4m3 decode times the fp32 scale, both widened to double, where the
    # product of a 4-bit and a 24-bit significand is exact
    vals = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double()
    for sc in _fp8_scales():
        for code in range(256):
            v = oracle.fp8_latent(code, float(sc))
            r = float(vals[code]) * float(sc)
            assert (math.isnan(v) and math.isnan(r)) or v == r, (code, float(sc), v, r)
    # a scale whose product is not a bf16 value stays unrounded: 1.125 * (1 + 2^-20)
    assert oracle.fp8_latent(0x39, 1.0 + 2.0 ** -20) == 1.125 * (1.0 + 2.0 ** -20)


def test_fp8_latent_bf16_operand_is_fp32_product_rounded_once_to_bf16():
    # the secondary mode: every code against torch's own e4m3 decode, fp32 multiply and
    # round-to-nearest-even bf16 conversion, for scales with full fp32 mantissas (so the
    # bf16 rounding matters)
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).float()
    for sc in _fp8_scales():
        ref = (vals * sc).to(torch.bfloat16).double()
        for code in range(256):
            v = oracle.fp8_latent(code, float(sc), operand="bf16")
            r = float(ref[code])
            assert (math.isnan(v) and math.isnan(r)) or v == r, (code, float(sc), v, r)
    # scale 1: e4m3 values are exact in bf16
    assert oracle.fp8_latent(0x7E, 1.0, operand="bf16") == 448.0
    assert oracle.fp8_latent(0x01, 1.0, operand="bf16") == 2.0 ** -9
    assert oracle.fp8_latent(0x39, 1.0 + 2.0 ** -20, operand="bf16") == 1.125


@pytest.mark.parametrize("operand", ["exact", "bf16"])
def test_fp8_decode_equals_dense_on_dequantised_values(operand):
    B, H, lens = 2, 3, [97, 64]
    c = inputs.make_case(B, H, lens, seed=21, kv_dtype="fp8", extra_pages=1)
    out, lse = oracle.decode_fp8(c.q_nope, c.q_rope, c.cache, c.block_table, c.seq_lens, SCALE,
                                 operand=operand)
    rec = c.cache
    codes = rec[..., :512].contiguous().view(torch.float8_e4m3fn).double()     # library decode
    scales = rec[..., 512:528].contiguous().view(torch.float32).double()       # [P,64,4]
    rope = rec[..., 528:656].contiguous().view(torch.bfloat16).double()
    if operand == "exact":   # code x scale in double (exact)
        lat = codes * scales.repeat_interleave(128, dim=-1)
    else:                    # fp32 product of code and block scale, rounded once to bf16 (torch)
        lat = (codes.float() * scales.float().repeat_interleave(128, dim=-1)).to(torch.bfloat16).double()
    for b in range(B):
        rows = [(int(c.block_table[b, t // 64]), t % 64) for t in range(lens[b])]
        C = np.stack([lat[p, r].numpy() for p, r in rows])
        K = np.stack([rope[p, r].numpy() for p, r in rows])
        o, l = oracle.attend_f64(c.q_nope[b].double().numpy(), c.q_rope[b].double().numpy(), C, K,
                                 SCALE)
        np.testing.assert_allclose(out[b], o, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(lse[b], l, rtol=1e-13)


def test_fp8_quantisation_error_within_format_bound():
    """e4m3 has 3 mantissa bits: |x - x_hat| <= 2^-4 |x| for normals, and the block scale
    maps max|x| exactly onto 448."""
    r = torch.randn((8, 64, 512))
    rope = torch.randn((8, 64, 64))
    rec = inputs.quantize_fp8_records(r, rope)
    codes = rec[..., :512].contiguous().view(torch.float8_e4m3fn).float()
    s = rec[..., 512:528].contiguous().view(torch.float32)
    xh = codes * s.repeat_interleave(128, dim=-1)
    err = (xh - r).abs()
    sub = s.repeat_interleave(128, dim=-1) * 2.0 ** -6
    assert torch.all(err <= 2.0 ** -4 * r.abs() + sub)
    amax = r.reshape(8, 64, 4, 128).abs().amax(-1)
    torch.testing.assert_close(s * 448.0, amax, rtol=1e-6, atol=0)


# ------------------------------------------------------------------------------ cache append
def _e4m3_values():
    return np.array([oracle.e4m3_to_float(c) for c in range(0x7F)])


def test_e4m3_encode_round_trips_every_finite_code():
    for c in list(range(0x7F)) + list(range(0x80, 0xFF)):
        v = oracle.e4m3_to_float(c)
        assert oracle.e4m3_encode(v) == c, hex(c)


def test_e4m3_encode_matches_torch_float8_including_ties():
    # torch's float8_e4m3fn conversion (round to nearest, ties to even) is an independent
    # implementation; the values cover every binade, random points and the exact midpoints
    # between neighbouring codes (where only ties-to-even decides)
    vals = _e4m3_values()
    mids = (vals[:-1] + vals[1:]) / 2
    rng = np.random.default_rng(3)
    rnd = np.exp(rng.uniform(np.log(1e-4), np.log(448.0), 4000)) * rng.choice([-1.0, 1.0], 4000)
    xs = np.concatenate([mids, -mids, rnd, [0.0, 1e-12, 448.0, -448.0]]).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(x)) for x in xs], dtype=np.uint8)
    assert np.array_equal(got, ref)


def _append_case(fp8, B=5, seed=4):
    rng = np.random.default_rng(seed)
    max_pages, num_pages = 3, 16
    row_bytes = 656 if fp8 else 1152
    cache = rng.integers(0, 256, size=num_pages * 64 * row_bytes, dtype=np.uint8)
    bt = rng.permutation(num_pages)[:B * max_pages].reshape(B, max_pages).astype(np.int32)
    positions = np.array([0, 63, 64, 191, -1][:B], dtype=np.int32)
    lat = torch.randn(B, 512) * torch.tensor([1.0, 1e-3, 30.0, 0.0]).repeat_interleave(128)
    c_kv = lat.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    k_rope = torch.randn(B, 64).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return cache, bt, positions, c_kv, k_rope


@pytest.mark.parametrize("fp8", [False, True])
def test_append_writes_the_mapped_row_and_nothing_else(fp8):
    cache, bt, positions, c_kv, k_rope = _append_case(fp8)
    new, err = oracle.append(cache, fp8, bt, positions, c_kv, k_rope)
    assert err == 0
    row_bytes = 656 if fp8 else 1152
    rows = new.reshape(-1, row_bytes)
    old = cache.reshape(-1, row_bytes)
    written = set()
    for b, p in enumerate(positions):
        if p < 0:
            continue
        r = int(bt[b, p // 64]) * 64 + p % 64
        written.add(r)
        if not fp8:
            assert np.array_equal(rows[r, :1024].view(np.uint16), c_kv[b])
        assert np.array_equal(rows[r, row_bytes - 128:].view(np.uint16), k_rope[b])
    untouched = [r for r in range(rows.shape[0]) if r not in written]
    assert np.array_equal(rows[untouched], old[untouched])


def test_append_fp8_record_equals_the_generator_quantiser():
    # the workload generator quantises with torch (amax / 448 scale, float8_e4m3fn cast):
    # a second implementation of the same record
    cache, bt, positions, c_kv, k_rope = _append_case(True)
    new, _ = oracle.append(cache, True, bt, positions, c_kv, k_rope)
    rows = new.reshape(-1, 656)
    lat = torch.from_numpy(c_kv.view(np.int16)).view(torch.bfloat16)
    rope = torch.from_numpy(k_rope.view(np.int16)).view(torch.bfloat16)
    ref = inputs.quantize_fp8_records(lat.float(), rope).numpy()
    for b, p in enumerate(positions):
        if p >= 0:
            r = int(bt[b, p // 64]) * 64 + p % 64
            assert np.array_equal(rows[r], ref[b]), b
    # the all-zero block (channels 384..511) has scale 1 and zero codes (signed zeros keep
    # their sign bit)
    r0 = int(bt[0, 0]) * 64
    assert np.frombuffer(rows[r0, 512 + 12:512 + 16].tobytes(), dtype=np.float32)[0] == 1.0
    assert not (rows[r0, 384:512] & 0x7F).any()


def test_append_dequantises_within_the_format_bound():
    cache, bt, positions, c_kv, k_rope = _append_case(True)
    new, _ = oracle.append(cache, True, bt, positions, c_kv, k_rope)
    rows = new.reshape(-1, 656)
    x = torch.from_numpy(c_kv.view(np.int16)).view(torch.bfloat16).double().numpy()
    for b, p in enumerate(positions):
        if p < 0:
            continue
        r = int(bt[b, p // 64]) * 64 + p % 64
        scales = np.frombuffer(rows[r, 512:528].tobytes(), dtype=np.float32)
        back = np.array([oracle.e4m3_to_float(c) for c in rows[r, :512]]) * np.repeat(scales, 128)
        # e4m3 keeps 3 mantissa bits: relative error <= 2^-4 for normals, and an absolute
        # error <= half the subnormal step (2^-10) times the scale below them
        bound = np.maximum(np.abs(x[b]) * 2.0 ** -4, np.repeat(scales, 128) * 2.0 ** -10) * 1.0001
        assert np.all(np.abs(back - x[b]) <= bound)


def test_append_reports_out_of_range_and_writes_nothing_for_them():
    cache, bt, positions, c_kv, k_rope = _append_case(False)
    bt = bt.copy()
    bt[1, 0] = 10_000                    # page id out of range (position 63 -> page 0)
    positions = positions.copy()
    positions[2] = 3 * 64                # beyond the block table (3 pages)
    new, err = oracle.append(cache, False, bt, positions, c_kv, k_rope)
    assert err == 2
    rows, old = new.reshape(-1, 1152), cache.reshape(-1, 1152)
    changed = np.nonzero((rows != old).any(axis=1))[0]
    expect = sorted(int(bt[b, p // 64]) * 64 + p % 64 for b, p in [(0, 0), (3, 191)])
    assert changed.tolist() == expect
