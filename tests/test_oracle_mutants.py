"""The pins must be strong enough to catch plausible slips.

Each mutant is a copy of the oracle's C source with one deliberate mistake (planted here,
on the CPU, never in the product).  It is compiled to a temporary library and run through
the same closed-form checks the oracle passes; every mutant must fail at least one.
"""
import ctypes
import math
import os
import subprocess

import numpy as np
import pytest

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "mla_oracle.c")
SCALE = 1.0 / math.sqrt(192.0)

MUTANTS = {
    "drop_rope_term": ("dot += qr[(size_t)h * D_ROPE + r] * Kr[(size_t)t * D_ROPE + r];",
                       "(void)r;"),
    "scale_after_exp": ("s[t] = scale * dot;", "s[t] = dot;"),
    "no_normalise": ("o[c] /= l;", "(void)0;"),
    "lse_log2": ("lse[h] = m + log(l);", "lse[h] = m + log2(l);"),
    "rope_in_output": ("for (int c = 0; c < D_LATENT; ++c) o[c] += w * C[(size_t)t * D_LATENT + c];",
                       "for (int c = 0; c < D_LATENT; ++c) o[c] += w * (c < D_ROPE ? Kr[(size_t)t * D_ROPE + c] : C[(size_t)t * D_LATENT + c]);"),
    "transposed_query": ("dot += qn[(size_t)h * D_LATENT + c] * C[(size_t)t * D_LATENT + c];",
                         "dot += qn[(size_t)(c % H) * D_LATENT + (h * 7 + c) % D_LATENT] * C[(size_t)t * D_LATENT + c];"),
}


# slips in the absorption / projection (checked with test_oracle's absorb/project pins)
PROJ_MUTANTS = {
    "absorb_head0_weights": ("s += q[k] * w_uk[((int64_t)h * dh + k) * D_LATENT + c];",
                             "s += q[k] * w_uk[((int64_t)0 * dh + k) * D_LATENT + c];"),
    "absorb_transposed_w": ("s += q[k] * w_uk[((int64_t)h * dh + k) * D_LATENT + c];",
                            "s += q[k] * w_uk[(int64_t)h * dh * D_LATENT + ((int64_t)c * dh + k) % (dh * D_LATENT)];"),
    "project_drops_last": ("for (int c = 0; c < D_LATENT; ++c) s += w[c] * o[c];",
                           "for (int c = 0; c < D_LATENT - 1; ++c) s += w[c] * o[c];"),
    "project_wrong_head": ("const double *o = out + ((int64_t)b * H + h) * D_LATENT;\n            for (int j",
                           "const double *o = out + ((int64_t)b * H + (h + 1) % H) * D_LATENT;\n            for (int j"),
}


def _build(tmp_path, name, old, new):
    src = open(SRC).read()
    assert old in src, name
    mut = tmp_path / f"{name}.c"
    mut.write_text(src.replace(old, new))
    so = tmp_path / f"lib{name}.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", "-o",
                           str(so), str(mut), "-lm"])
    lib = ctypes.CDLL(str(so))
    P, I, I64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.mla_oracle_attend_f64.argtypes = [I, I64, P, P, P, P, D, P, P]
    return lib


def _attend(lib, qn, qr, C, K, scale):
    H, N = qn.shape[0], C.shape[0]
    out = np.zeros((H, 512))
    lse = np.zeros(H)
    arrs = [np.ascontiguousarray(a, dtype=np.float64) for a in (qn, qr, C, K)]
    P = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    lib.mla_oracle_attend_f64(H, N, *[P(a) for a in arrs], scale, P(out), P(lse))
    return out, lse


def _pins_hold(att):
    """The closed-form pins of test_oracle.py, as a yes/no over an attend function."""
    r = np.random.default_rng(7)
    H, N, d_h = 3, 11, 128
    qC, qR = r.standard_normal((H, d_h)), r.standard_normal((H, 64))
    W_UK = r.standard_normal((H, d_h, 512)) / math.sqrt(512)
    W_UV = r.standard_normal((H, d_h, 512)) / math.sqrt(512)
    C, KR = r.standard_normal((N, 512)), r.standard_normal((N, 64))
    ok = True
    q_abs = np.stack([qC[h] @ W_UK[h] for h in range(H)])
    out, lse = att(q_abs, qR, C, KR, SCALE)
    for h in range(H):
        K, V = C @ W_UK[h].T, C @ W_UV[h].T
        s = (K @ qC[h] + KR @ qR[h]) * SCALE
        p = np.exp(s - s.max())
        ok &= np.allclose(W_UV[h] @ out[h], (p / p.sum()) @ V, rtol=1e-9, atol=1e-12)
        ok &= abs(lse[h] - (s.max() + math.log(p.sum()))) < 1e-12
    out, lse = att(np.zeros((2, 512)), np.zeros((2, 64)), C, KR, SCALE)
    ok &= np.allclose(out, np.tile(C.mean(0), (2, 1)), atol=1e-12)
    ok &= np.allclose(lse, math.log(N), atol=1e-13)
    return bool(ok)


def test_real_oracle_passes_pins():
    assert _pins_hold(oracle.attend_f64)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    lib = _build(tmp_path, name, old, new)
    assert not _pins_hold(lambda *a: _attend(lib, *a)), f"pins missed mutant {name}"


def _proj_fns(lib):
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.mla_oracle_absorb.argtypes = [I, I, I, P, P, P]
    lib.mla_oracle_project.argtypes = [I, I, I, P, P, P]
    ptr = lambda a: a.ctypes.data_as(ctypes.c_void_p)

    def absorb(q, w):
        q = np.ascontiguousarray(q, dtype=np.float64)
        w = np.ascontiguousarray(w, dtype=np.float64)
        out = np.zeros(q.shape[:2] + (512,))
        lib.mla_oracle_absorb(q.shape[0], q.shape[1], q.shape[2], ptr(q), ptr(w), ptr(out))
        return out

    def project(o, w):
        o = np.ascontiguousarray(o, dtype=np.float64)
        w = np.ascontiguousarray(w, dtype=np.float64)
        y = np.zeros(o.shape[:2] + (w.shape[1],))
        lib.mla_oracle_project(o.shape[0], o.shape[1], w.shape[1], ptr(o), ptr(w), ptr(y))
        return y

    return absorb, project


@pytest.mark.parametrize("name", sorted(PROJ_MUTANTS))
def test_projection_mutant_is_caught(tmp_path, name):
    from test_oracle import _absorb_project_pins
    old, new = PROJ_MUTANTS[name]
    lib = _build(tmp_path, name, old, new)
    res = _absorb_project_pins(*_proj_fns(lib))
    assert not all(ok for _, ok in res), f"pins missed mutant {name}"


# slips in the top-k selection, planted in a copy of oracle.topk_select's source
TOPK_MUTANTS = {
    "unsorted_output": ("sel = np.sort(order[:min(k, L)])", "sel = order[:min(k, L)]"),
    "keeps_lowest": ("np.argsort(-s[b, :L]", "np.argsort(s[b, :L]"),
    "reads_past_length": ("s[b, :L]", "s[b, :L + 1]"),
    "ties_to_high_position": ("order = np.argsort(-s[b, :L], kind=\"stable\")",
                              "order = (L - 1 - np.argsort(-s[b, :L][::-1], kind=\"stable\"))"),
}


def _topk_pins_hold(fn):
    from test_oracle import _topk_brute
    r = np.random.default_rng(92)
    for _ in range(30):
        Lmax, k = int(r.integers(2, 30)), int(r.integers(1, 30))
        s = r.choice(np.array([-1.0, 0.0, 0.5, 3.0], dtype=np.float32), size=(2, Lmax))
        lens = r.integers(0, Lmax, size=2)
        got = fn(s, lens, k)
        for b in range(2):
            if got[b].tolist() != _topk_brute(s[b].tolist(), int(lens[b]), k):
                return False
    return True


def test_real_topk_passes_pins():
    assert _topk_pins_hold(oracle.topk_select)


@pytest.mark.parametrize("name", sorted(TOPK_MUTANTS))
def test_topk_mutant_is_caught(name):
    import inspect
    import textwrap
    old, new = TOPK_MUTANTS[name]
    src = textwrap.dedent(inspect.getsource(oracle.topk_select))
    assert old in src, name
    ns = {"np": np}
    exec(src.replace(old, new), ns)
    assert not _topk_pins_hold(ns["topk_select"]), f"pins missed mutant {name}"


# slips in the non-absorbed prefill, planted in copies of the C oracle
PREFILL_MUTANTS = {
    "causal_excludes_diagonal": ("for (int t = 0; t <= i; ++t) {\n                double dot",
                                 "for (int t = 0; t < (i > 0 ? i : 1); ++t) {\n                double dot"),
    "values_from_w_uk": ("const double *wv = w_uv + ((int64_t)h * dh + j) * D_LATENT;",
                         "const double *wv = w_uk + ((int64_t)h * dh + j) * D_LATENT;"),
    "drops_rope_key": ("for (int r = 0; r < D_ROPE; ++r) dot += qr[r] * entries[(int64_t)t * D_ENTRY + D_LATENT + r];",
                       "(void)qr;"),
    "rope_key_from_latent": ("dot += qr[r] * entries[(int64_t)t * D_ENTRY + D_LATENT + r];",
                             "dot += qr[r] * entries[(int64_t)t * D_ENTRY + r];"),
}


@pytest.mark.parametrize("name", sorted(PREFILL_MUTANTS))
def test_prefill_mutant_is_caught(tmp_path, name):
    from test_oracle import _prefill_pins
    old, new = PREFILL_MUTANTS[name]
    lib = _build(tmp_path, name, old, new)
    P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
    lib.mla_oracle_prefill.argtypes = [I, I, I, P, P, P, P, P, D, I, P, P]
    ptr = lambda a: a.ctypes.data_as(ctypes.c_void_p)

    def prefill(E, qn, qr, wk, wv, scale):
        arrs = [np.ascontiguousarray(a, dtype=np.float64) for a in (E, qn, qr, wk, wv)]
        L, H, dh = arrs[1].shape
        out = np.zeros((L, H, dh))
        lse = np.zeros((L, H))
        lib.mla_oracle_prefill(L, H, dh, *[ptr(a) for a in arrs], scale, 0, ptr(out), ptr(lse))
        return out, lse

    assert not all(ok for _, ok in _prefill_pins(prefill)), f"pins missed mutant {name}"


# slips in the cache append and its FP8 quantiser, planted in copies of the C oracle
APPEND_MUTANTS = {
    "row_from_page_index": ("const int64_t row = (int64_t)page * PAGE_ROWS + pos % PAGE_ROWS;",
                            "const int64_t row = (int64_t)page * PAGE_ROWS + (pos / PAGE_ROWS) % PAGE_ROWS;"),
    "one_scale_for_all_blocks": ("for (int i = 0; i < 128; ++i) {\n                const float x = (float)bf16_bits_to_double(c[blk * 128 + i]);",
                                 "for (int i = 0; i < 128; ++i) {\n                const float x = (float)bf16_bits_to_double(c[((blk + i) % 4) * 128 + i]);"),
    "ties_away_from_even": ("if (d < bestd || (d == bestd && (c & 1) == 0 && (best & 1) == 1)) {",
                            "if (d < bestd || (d == bestd && c > best)) {"),
    "rope_not_copied": ("memcpy(dst + D_LATENT + 16, kr, D_ROPE * 2);", "(void)kr;"),
}


def _append_pins_hold(lib):
    """The append pins of test_oracle.py that need no oracle internals: the record equals the
    input generator's quantiser (a second implementation of reading 7), and only the mapped
    row of each request changes."""
    import torch
    from mla_latent_kv_17_gb300 import inputs
    P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    lib.mla_oracle_append.argtypes = [P, I, I64, P, I, P, P, P, I]
    lib.mla_oracle_append.restype = I
    ptr = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    r = np.random.default_rng(11)
    B, num_pages, max_pages = 5, 12, 2
    for fp8 in (True, False):
        rb = 656 if fp8 else 1152
        cache = r.integers(0, 256, size=num_pages * 64 * rb, dtype=np.uint8)
        bt = r.permutation(num_pages)[:B * max_pages].reshape(B, max_pages).astype(np.int32)
        pos = np.array([0, 63, 64, 100, 127], dtype=np.int32)
        mag = np.repeat([1.0, 1e-3, 300.0, 0.5], 128)
        lat = torch.from_numpy(r.standard_normal((B, 512)) * mag).to(torch.bfloat16)
        lat[0, :4] = torch.tensor([448.0, -448.0, 1.0625, -1.1875]).to(torch.bfloat16)  # exact ties
        rope = torch.from_numpy(r.standard_normal((B, 64))).to(torch.bfloat16)
        ck = np.ascontiguousarray(lat.view(torch.int16).numpy().view(np.uint16))
        kr = np.ascontiguousarray(rope.view(torch.int16).numpy().view(np.uint16))
        new = cache.copy()
        if lib.mla_oracle_append(ptr(new), 1 if fp8 else 0, num_pages, ptr(bt), max_pages, ptr(pos), ptr(ck),
                                 ptr(kr), B) != 0:
            return False
        rows, old = new.reshape(-1, rb), cache.reshape(-1, rb)
        mapped = {int(bt[b, p // 64]) * 64 + p % 64: b for b, p in enumerate(pos)}
        for i in range(rows.shape[0]):
            if i not in mapped and not np.array_equal(rows[i], old[i]):
                return False
        if fp8:
            ref = inputs.quantize_fp8_records(lat.float(), rope).numpy()
            want = lambda b: ref[b]
        else:
            want = lambda b: np.concatenate([ck[b].view(np.uint8), kr[b].view(np.uint8)])
        for i, b in mapped.items():
            if not np.array_equal(rows[i], want(b)):
                return False
    return True


def test_real_oracle_passes_append_pins(tmp_path):
    lib = _build(tmp_path, "identity", "#include <math.h>", "#include <math.h>")
    assert _append_pins_hold(lib)


@pytest.mark.parametrize("name", sorted(APPEND_MUTANTS))
def test_append_mutant_is_caught(tmp_path, name):
    old, new = APPEND_MUTANTS[name]
    lib = _build(tmp_path, name, old, new)
    assert not _append_pins_hold(lib), f"pins missed mutant {name}"
