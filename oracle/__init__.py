"""CPU oracle for absorbed MLA decode (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  The product path (the CUDA library and its Python binding)
never imports it and never falls back to it.

The arithmetic lives in ``mla_oracle.c`` (plain C, IEEE double, two-pass softmax);
this module compiles it with gcc on first use and marshals numpy arrays through
ctypes.  It shares no code with the CUDA library.

Functions follow these passages (page title, section):

* ``decode_dense`` / ``attend_f64``: "MLA 在极长上下文下的显存带宽突围" (run-time
  matrix absorption: score = q~ c^T + q^R k_R^T over the 576-wide cache entry) and
  "MLA & DSA 推理性能优化指南" §1.1 (absorbed path computes in the latent space).
* ``decode_sparse``: same guide §1.2 / §4.2 (attend over the top-k selected tokens).
* ``decode_fp8`` / ``e4m3_to_float``: same guide §5.3 (FP8 latent cache).  The format
  (e4m3 "fn", one fp32 scale per 128 channels) is this library's reading; the pages
  name only "FP8".  The dequantized latent is code x scale, exact (the default); the
  ``operand="bf16"`` mode rounds it to bf16 as a bf16 tensor-core operand would, a
  tighter secondary check only.
* ``append`` / ``e4m3_encode``: the cache append after a decode step (same guide §4,
  the decode figure: the output token is appended to the cache) and the FP8 record it
  writes (§5.3; per-128-channel scale max|x|/448, nearest e4m3 code, ties to even).
* ``absorb`` / ``project``: the query absorption q~ = q^C W^UK ("MLA 在极长上下文下的显存
  带宽突围", run-time matrix absorption) and the value up-projection W^UV applied to the
  latent output afterwards ("MLA & DSA 推理性能优化指南" §1.1), one matrix per head.
* ``topk_select``: the DSA token selection ("MLA & DSA 推理性能优化指南" §1.2: an indexer scores
  every earlier token and only the top-k take part in the attention; "GPU partial sort").
  This library's reading: the k highest scores of positions [0, seq_len), equal scores in
  ascending position order (-0.0 equals +0.0), returned as ascending positions padded with -1.
* ``prefill``: the non-absorbed (MHA-mode) path of the same guide (§3.1, §1.1): latents
  decompressed into per-head keys and values with W^UK and W^UV, then causal attention with
  192-wide keys ([K_h | k_R]) and 128-wide values ("MLA 最佳算子全景调研" §4).
* ``combine``: merge of split-KV partial results through their log-sum-exp, the
  "Fused Reduction" the operator survey ("MLA 最佳算子全景调研" §3) pairs with
  weight-absorbed decode.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libmla_oracle.so")
_lock = threading.Lock()
_lib = None

D_LATENT = 512
D_ROPE = 64
D_ENTRY = 576
PAGE_ROWS = 64
FP8_RECORD_BYTES = 656


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libmla_oracle.so`` (gcc, -O2)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            I64 = ctypes.c_int64
            D = ctypes.c_double
            lib.mla_oracle_attend_f64.argtypes = [I, I64, P, P, P, P, D, P, P]
            lib.mla_oracle_attend_f64.restype = None
            lib.mla_oracle_combine_f64.argtypes = [I, I, P, P, P, P]
            lib.mla_oracle_combine_f64.restype = None
            lib.mla_oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.mla_oracle_e4m3_to_double.restype = D
            lib.mla_oracle_fp8_latent.argtypes = [ctypes.c_uint8, ctypes.c_float]
            lib.mla_oracle_fp8_latent.restype = D
            lib.mla_oracle_fp8_latent_exact.argtypes = [ctypes.c_uint8, ctypes.c_float]
            lib.mla_oracle_fp8_latent_exact.restype = D
            lib.mla_oracle_e4m3_encode.argtypes = [ctypes.c_float]
            lib.mla_oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.mla_oracle_append.argtypes = [P, I, I64, P, I, P, P, P, I]
            lib.mla_oracle_append.restype = I
            lib.mla_oracle_absorb.argtypes = [I, I, I, P, P, P]
            lib.mla_oracle_absorb.restype = None
            lib.mla_oracle_project.argtypes = [I, I, I, P, P, P]
            lib.mla_oracle_project.restype = None
            lib.mla_oracle_prefill.argtypes = [I, I, I, P, P, P, P, P, D, I, P, P]
            lib.mla_oracle_prefill.restype = None
            lib.mla_oracle_default_threads.argtypes = []
            lib.mla_oracle_default_threads.restype = I
            common = [I, I, P, P, P, I64, P, I, P]
            lib.mla_oracle_decode_dense.argtypes = common + [D, P, P, I]
            lib.mla_oracle_decode_dense.restype = I
            lib.mla_oracle_decode_fp8.argtypes = common + [I, D, P, P, I]
            lib.mla_oracle_decode_fp8.restype = I
            lib.mla_oracle_decode_sparse.argtypes = common + [P, I, D, P, P, I]
            lib.mla_oracle_decode_sparse.restype = I
            _lib = lib
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return int(_load().mla_oracle_default_threads())


def e4m3_to_float(code: int) -> float:
    """Value of one e4m3 "fn" code (bias 7, no infinities, 0x7F/0xFF NaN)."""
    return float(_load().mla_oracle_e4m3_to_double(int(code) & 0xFF))


def fp8_latent(code: int, scale: float, operand: str = "exact") -> float:
    """One dequantized FP8 latent value: e4m3(code) * scale exactly, or with
    operand="bf16" bf16_rne(fp32(e4m3(code)) * fp32(scale))."""
    if operand == "exact":
        return float(_load().mla_oracle_fp8_latent_exact(int(code) & 0xFF, float(scale)))
    if operand == "bf16":
        return float(_load().mla_oracle_fp8_latent(int(code) & 0xFF, float(scale)))
    raise ValueError(operand)


def e4m3_encode(v: float) -> int:
    """Nearest e4m3 "fn" code to the binary32 value v (|v| <= 448), ties to the even code."""
    return int(_load().mla_oracle_e4m3_encode(float(v)))


def append(cache, fp8: bool, block_table, positions, c_kv, k_rope):
    """Cache append: returns (a new cache array with each request's token written, error count).

    cache: uint8 bytes of [num_pages][64][576] bf16 or [num_pages][64][656] FP8 records;
    block_table int32 [B][max_pages]; positions int32 [B] (< 0: skip); c_kv, k_rope: bf16 bits
    (uint16) [B][512], [B][64]."""
    lib = _load()
    cache = np.ascontiguousarray(np.asarray(cache, dtype=np.uint8)).copy()
    row_bytes = FP8_RECORD_BYTES if fp8 else 2 * D_ENTRY
    num_pages = cache.size // (row_bytes * PAGE_ROWS)
    bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int32))
    ck = np.ascontiguousarray(np.asarray(c_kv, dtype=np.uint16))
    kr = np.ascontiguousarray(np.asarray(k_rope, dtype=np.uint16))
    B = pos.shape[0]
    assert bt.shape[0] == B and ck.shape == (B, D_LATENT) and kr.shape == (B, D_ROPE)
    vp = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    err = lib.mla_oracle_append(vp(cache), 1 if fp8 else 0, num_pages, vp(bt), bt.shape[1], vp(pos), vp(ck), vp(kr), B)
    return cache, int(err)


def absorb(q_c, w_uk):
    """Absorbed queries: q_c [B][H][dh], w_uk [H][dh][512] (float64) -> [B][H][512]."""
    qc, pq = _c(q_c, np.float64)
    w, pw = _c(w_uk, np.float64)
    B, H, dh = qc.shape
    assert w.shape == (H, dh, D_LATENT)
    out = np.zeros((B, H, D_LATENT), np.float64)
    _load().mla_oracle_absorb(B, H, dh, pq, pw, out.ctypes.data_as(ctypes.c_void_p))
    return out


def project(out_latent, w_uv):
    """Per-head value projection: out [B][H][512], w_uv [H][dh][512] (float64) -> [B][H][dh]."""
    o, po = _c(out_latent, np.float64)
    w, pw = _c(w_uv, np.float64)
    B, H, D = o.shape
    dh = w.shape[1]
    assert D == D_LATENT and w.shape == (H, dh, D_LATENT)
    y = np.zeros((B, H, dh), np.float64)
    _load().mla_oracle_project(B, H, dh, po, pw, y.ctypes.data_as(ctypes.c_void_p))
    return y


def topk_select(scores, seq_lens, k):
    """DSA indices: scores float32 [B][Lmax], seq_lens int [B], k -> int32 [B][k].

    Row b keeps the min(k, seq_lens[b]) positions of [0, seq_lens[b]) with the largest scores
    (a stable sort on the negated scores puts equal scores in ascending position order),
    listed in ascending position order and padded with -1."""
    s = np.asarray(scores, dtype=np.float32)
    B = s.shape[0]
    out = np.full((B, k), -1, dtype=np.int32)
    for b in range(B):
        L = int(seq_lens[b])
        order = np.argsort(-s[b, :L], kind="stable")
        sel = np.sort(order[:min(k, L)])
        out[b, :sel.size] = sel
    return out


def prefill(entries, q_nope, q_rope, w_uk, w_uv, scale, kv_bf16=False):
    """Non-absorbed causal prefill of one sequence (float64 arrays): entries [L][576],
    q_nope [L][H][dh], q_rope [L][H][64], w_uk / w_uv [H][dh][512] -> out [L][H][dh], lse [L][H].
    kv_bf16: the decompressed keys and values are rounded to bf16 (the attention's operands)."""
    e, pe = _c(entries, np.float64)
    qn, pqn = _c(q_nope, np.float64)
    qr, pqr = _c(q_rope, np.float64)
    wk, pwk = _c(w_uk, np.float64)
    wv, pwv = _c(w_uv, np.float64)
    L, H, dh = qn.shape
    assert e.shape == (L, D_ENTRY) and qr.shape == (L, H, D_ROPE)
    assert wk.shape == (H, dh, D_LATENT) and wv.shape == (H, dh, D_LATENT)
    out = np.zeros((L, H, dh), np.float64)
    lse = np.zeros((L, H), np.float64)
    _load().mla_oracle_prefill(L, H, dh, pe, pqn, pqr, pwk, pwv, float(scale), 1 if kv_bf16 else 0,
                               out.ctypes.data_as(ctypes.c_void_p), lse.ctypes.data_as(ctypes.c_void_p))
    return out, lse


def attend_f64(q_nope, q_rope, C, Kr, scale):
    """Definition of absorbed decode for one request in double precision.

    q_nope [H,512], q_rope [H,64], C [N,512], Kr [N,64] (float64) -> out [H,512], lse [H].
    """
    lib = _load()
    qn, pqn = _c(q_nope, np.float64)
    qr, pqr = _c(q_rope, np.float64)
    c, pc = _c(C, np.float64)
    k, pk = _c(Kr, np.float64)
    H = qn.shape[0]
    N = c.shape[0]
    assert qn.shape == (H, D_LATENT) and qr.shape == (H, D_ROPE)
    assert c.shape == (N, D_LATENT) and k.shape == (N, D_ROPE)
    out = np.zeros((H, D_LATENT), np.float64)
    lse = np.zeros((H,), np.float64)
    lib.mla_oracle_attend_f64(H, N, pqn, pqr, pc, pk, float(scale),
                              out.ctypes.data_as(ctypes.c_void_p),
                              lse.ctypes.data_as(ctypes.c_void_p))
    return out, lse


def combine(outs, lses):
    """Merge S partial results of one head: outs [S,D], lses [S] -> out [D], lse."""
    lib = _load()
    o, po = _c(outs, np.float64)
    l, pl = _c(lses, np.float64)
    S, D = o.shape
    out = np.zeros((D,), np.float64)
    lse = np.zeros((1,), np.float64)
    lib.mla_oracle_combine_f64(S, D, po, pl, out.ctypes.data_as(ctypes.c_void_p),
                               lse.ctypes.data_as(ctypes.c_void_p))
    return out, float(lse[0])


def _bits16(a):
    """bf16 storage (torch.bfloat16 tensor or uint16/int16 numpy array) -> uint16 numpy."""
    if hasattr(a, "detach"):
        import torch
        a = a.detach().cpu().contiguous().view(torch.int16).numpy()
    return np.ascontiguousarray(a).view(np.uint16)


def _np(a, dtype):
    if hasattr(a, "detach"):
        a = a.detach().cpu().contiguous().numpy()
    return np.ascontiguousarray(a, dtype=dtype)


def _run(fn_name, q_nope, q_rope, cache, block_table, seq_lens, scale, nthreads,
         extra=(), cache_kind="bf16"):
    lib = _load()
    qn = _bits16(q_nope)
    qr = _bits16(q_rope)
    B, H, _ = qn.shape
    if cache_kind == "bf16":
        cb = _bits16(cache)
        num_pages = cb.shape[0]
    else:
        cb = _np(cache, np.uint8)
        num_pages = cb.shape[0]
    bt = _np(block_table, np.int32)
    sl = _np(seq_lens, np.int32)
    assert bt.shape[0] == B and sl.shape == (B,)
    out = np.zeros((B, H, D_LATENT), np.float64)
    lse = np.zeros((B, H), np.float64)
    P = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    args = [B, H, P(qn), P(qr), P(cb), num_pages, P(bt), bt.shape[1], P(sl)]
    args += list(extra)
    args += [float(scale), P(out), P(lse), int(nthreads)]
    rc = getattr(lib, fn_name)(*args)
    if rc != 0:
        raise ValueError(f"{fn_name}: a page or token reference is out of range")
    return out, lse


def decode_dense(q_nope, q_rope, cache, block_table, seq_lens, scale, nthreads=0):
    """Dense decode over the paged bf16 cache [num_pages,64,576] -> (out [B,H,512], lse [B,H])."""
    return _run("mla_oracle_decode_dense", q_nope, q_rope, cache, block_table, seq_lens,
                scale, nthreads)


def decode_fp8(q_nope, q_rope, cache, block_table, seq_lens, scale, nthreads=0, operand="exact"):
    """Dense decode over the paged FP8 cache [num_pages,64,656] (bytes).  operand="exact":
    latent = code x scale exactly (the definition); "bf16": that value rounded to bf16."""
    if operand not in ("exact", "bf16"):
        raise ValueError(operand)
    return _run("mla_oracle_decode_fp8", q_nope, q_rope, cache, block_table, seq_lens,
                scale, nthreads, extra=(1 if operand == "exact" else 0,), cache_kind="fp8")


def decode_sparse(q_nope, q_rope, cache, block_table, seq_lens, indices, scale, nthreads=0):
    """Token-sparse decode: indices [B,topk] int32 logical positions, -1 = padding."""
    idx = _np(indices, np.int32)
    P = idx.ctypes.data_as(ctypes.c_void_p)
    return _run("mla_oracle_decode_sparse", q_nope, q_rope, cache, block_table, seq_lens,
                scale, nthreads, extra=(P, idx.shape[1]))
