"""Python binding of libmla_decode (argument marshalling only).

Every function here checks tensor dtypes/shapes, passes raw device pointers and sizes to
the C ABI declared in ``include/mla_decode.h`` and raises on a non-OK status.  All
computation happens in the library's CUDA kernels.  If the library has not been built,
the first call raises; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libmla_decode.so")

MLA_OK = 0
STATUS_NAMES = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED",
                3: "MLA_ERR_WORKSPACE", 4: "MLA_ERR_CUDA", 5: "MLA_ERR_INDEX",
                6: "MLA_ERR_TIMEOUT", 7: "MLA_ERR_RANGE"}
KV_BF16, KV_FP8 = 0, 1

_lock = threading.Lock()
_lib = None


class MlaError(RuntimeError):
    def __init__(self, fn, status, text):
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)} ({text})")
        self.status = status


def lib():
    """The loaded libmla_decode (ctypes.CDLL); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with `python -m mla_latent_kv_17_gb300.build`")
            L = ctypes.CDLL(LIB_PATH)
            P, I, I64, F, SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                ctypes.c_size_t)
            L.mla_decode_workspace_size.argtypes = [I, I, I]
            L.mla_decode_workspace_size.restype = SZ
            L.mla_decode_plan.argtypes = [P, I, I, I, I, I, P, SZ, P]
            L.mla_decode_plan.restype = I
            L.mla_decode_plan_host.argtypes = [P, I, I, I, I, I, P, SZ]
            L.mla_decode_plan_host.restype = I
            L.mla_decode.argtypes = [P, SZ, P, P, P, I, I64, P, I, P, I, I, F, P, P, P]
            L.mla_decode.restype = I
            L.mla_decode_sparse.argtypes = [P, SZ, P, P, P, I64, P, I, P, P, I, I, I, F, P, P, P]
            L.mla_decode_sparse.restype = I
            L.mla_decode_static.argtypes = [P, P, P, I, I64, P, I, P, I, I, F, P, P, P, P]
            L.mla_decode_static.restype = I
            L.mla_cache_append.argtypes = [P, I, I64, P, I, P, P, P, I, P, P]
            L.mla_cache_append.restype = I
            L.mla_prefill_decompress.argtypes = [P, I, P, P, I, P, P, P, P]
            L.mla_prefill_decompress.restype = I
            L.mla_prefill_attention.argtypes = [P, P, P, P, P, I, I, F, P, P, P, P]
            L.mla_prefill_attention.restype = I
            L.mla_topk_select.argtypes = [P, I64, I, P, I, I, P, P, P]
            L.mla_topk_select.restype = I
            L.mla_absorb_query.argtypes = [P, P, I, I, P, P, P]
            L.mla_absorb_query.restype = I
            L.mla_project_output.argtypes = [P, P, I, I, P, P, P]
            L.mla_project_output.restype = I
            L.mla_decode_status.argtypes = [P, SZ, P]
            L.mla_decode_status.restype = I
            L.mla_decode_inject_stall.argtypes = [I]
            L.mla_decode_inject_stall.restype = I
            L.mla_decode_set_wait_limit.argtypes = [I64]
            L.mla_decode_set_wait_limit.restype = I
            L.mla_status_string.argtypes = [I]
            L.mla_status_string.restype = ctypes.c_char_p
            _lib = L
    return _lib


def _check(fn, st):
    if st != MLA_OK:
        raise MlaError(fn, st, lib().mla_status_string(st).decode())


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def workspace_size(B: int, H: int, num_sms: int = 0) -> int:
    n = lib().mla_decode_workspace_size(int(B), int(H), int(num_sms))
    if n == 0:
        raise MlaError("mla_decode_workspace_size", 1, "invalid arguments")
    return int(n)


class Workspace:
    """Device workspace holding a plan, the split-KV partials and the status word."""

    def __init__(self, B: int, H: int, num_sms: int = 0, device=None):
        self.B, self.H = int(B), int(H)
        self.nbytes = workspace_size(B, H, num_sms)
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8,
                               device=device or torch.device("cuda", torch.cuda.current_device()))
        self.topk = None

    def ptr(self):
        return _ptr(self.buf)


def _i32(t, name):
    if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous int32 CUDA tensor")
    return t


def _kv_code(kv_dtype) -> int:
    if kv_dtype in ("bf16", KV_BF16):
        return KV_BF16
    if kv_dtype in ("fp8", KV_FP8):
        return KV_FP8
    raise ValueError(f"kv_dtype must be 'bf16' or 'fp8', not {kv_dtype!r}")


def plan(ws: Workspace, seq_lens=None, topk: int = 0, num_sms: int = 0, stream=None,
         kv_dtype="bf16") -> Workspace:
    """Build the split-KV plan for seq_lens (device int32 [B]) or for topk index slots;
    kv_dtype ('bf16' or 'fp8') is the cache layout the decode will read."""
    if seq_lens is not None:
        _i32(seq_lens, "seq_lens")
    st = lib().mla_decode_plan(_ptr(seq_lens), ws.B, ws.H, int(topk), _kv_code(kv_dtype), int(num_sms),
                               ws.ptr(), ws.nbytes, _stream(stream))
    _check("mla_decode_plan", st)
    ws.topk = int(topk)
    return ws


def _outputs(B, H, device, out, lse):
    if out is None:
        out = torch.empty((B, H, 512), dtype=torch.float32, device=device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=device)
    if out.dtype != torch.float32 or out.shape != (B, H, 512) or not out.is_contiguous():
        raise ValueError("out must be contiguous fp32 [B,H,512]")
    if lse.dtype != torch.float32 or lse.shape != (B, H) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 [B,H]")
    return out, lse


def _queries(q_nope, q_rope):
    B, H, d = q_nope.shape
    if d != 512 or q_nope.dtype != torch.bfloat16 or not q_nope.is_contiguous():
        raise ValueError("q_nope must be contiguous bf16 [B,H,512]")
    if q_rope.shape != (B, H, 64) or q_rope.dtype != torch.bfloat16 or not q_rope.is_contiguous():
        raise ValueError("q_rope must be contiguous bf16 [B,H,64]")
    return B, H


def decode(ws: Workspace, q_nope, q_rope, cache, block_table, seq_lens, softmax_scale: float,
           out=None, lse=None, stream=None):
    """Dense decode; the cache is bf16 [P,64,576] or uint8 FP8 records [P,64,656]."""
    B, H = _queries(q_nope, q_rope)
    _i32(block_table, "block_table")
    _i32(seq_lens, "seq_lens")
    if cache.dtype == torch.bfloat16 and cache.shape[1:] == (64, 576):
        kv = KV_BF16
    elif cache.dtype == torch.uint8 and cache.shape[1:] == (64, 656):
        kv = KV_FP8
    else:
        raise ValueError("cache must be bf16 [P,64,576] or uint8 [P,64,656]")
    if not cache.is_contiguous():
        raise ValueError("cache must be contiguous")
    out, lse = _outputs(B, H, q_nope.device, out, lse)
    st = lib().mla_decode(ws.ptr(), ws.nbytes, _ptr(q_nope), _ptr(q_rope), _ptr(cache), kv,
                          cache.shape[0], _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
                          B, H, float(softmax_scale), _ptr(out), _ptr(lse), _stream(stream))
    _check("mla_decode", st)
    return out, lse


def cache_append(cache, block_table, positions, c_kv, k_rope, device_status=None, stream=None):
    """Writes request b's new token (c_kv [B,512], k_rope [B,64], bf16) at position positions[b]
    (int32 [B], < 0 skips) of the paged cache: bf16 [P,64,576] or uint8 FP8 records [P,64,656]
    (quantised on the way in).  device_status: optional int32 [1] tensor for MLA_ERR_INDEX."""
    _i32(block_table, "block_table")
    _i32(positions, "positions")
    if cache.dtype == torch.bfloat16 and cache.shape[1:] == (64, 576):
        kv = KV_BF16
    elif cache.dtype == torch.uint8 and cache.shape[1:] == (64, 656):
        kv = KV_FP8
    else:
        raise ValueError("cache must be bf16 [P,64,576] or uint8 [P,64,656]")
    B = positions.shape[0]
    for t, n, d in ((c_kv, "c_kv", 512), (k_rope, "k_rope", 64)):
        if t.dtype != torch.bfloat16 or t.shape != (B, d) or not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"{n} must be contiguous CUDA bf16 [{B},{d}]")
    if not cache.is_contiguous():
        raise ValueError("cache must be contiguous")
    if device_status is not None:
        _i32(device_status, "device_status")
    st = lib().mla_cache_append(_ptr(cache), kv, cache.shape[0], _ptr(block_table), block_table.shape[1],
                                _ptr(positions), _ptr(c_kv), _ptr(k_rope), B, _ptr(device_status),
                                _stream(stream))
    _check("mla_cache_append", st)
    return cache


def topk_select(scores, seq_lens, k: int, indices=None, device_status=None, stream=None):
    """DSA indices int32 [B,k]: per request the k best-scored positions of [0, seq_len)
    (scores fp32 [B,Lmax], ties to the lower position), ascending, padded with -1."""
    if scores.dtype != torch.float32 or scores.dim() != 2 or not scores.is_cuda or scores.stride(1) != 1:
        raise ValueError("scores must be a CUDA fp32 [B,Lmax] tensor with unit column stride")
    _i32(seq_lens, "seq_lens")
    B, Lmax = scores.shape
    if indices is None:
        indices = torch.empty((B, k), dtype=torch.int32, device=scores.device)
    elif indices.dtype != torch.int32 or indices.shape != (B, k) or not indices.is_contiguous():
        raise ValueError(f"indices must be contiguous int32 [{B},{k}]")
    if device_status is not None:
        _i32(device_status, "device_status")
    st = lib().mla_topk_select(_ptr(scores), scores.stride(0), Lmax, _ptr(seq_lens), B, int(k), _ptr(indices),
                               _ptr(device_status), _stream(stream))
    _check("mla_topk_select", st)
    return indices


def _bf16(t, shape, name):
    if t.dtype != torch.bfloat16 or tuple(t.shape) != tuple(shape) or not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name} must be contiguous CUDA bf16 {list(shape)}")


def prefill_decompress(entries, w_uk, w_uv, k_nope=None, v=None, device_status=None, stream=None):
    """Per-head keys and values of a sequence: entries bf16 [L,576] (latent | RoPE key) ->
    k_nope, v bf16 [H,L,128] with k_nope[h,t] = w_uk[h] @ c_t and v[h,t] = w_uv[h] @ c_t."""
    if entries.dim() != 2:
        raise ValueError("entries must be [L,576]")
    L = entries.shape[0]
    H = w_uk.shape[0]
    _bf16(entries, (L, 576), "entries")
    _weights(w_uk, H, "w_uk")
    _weights(w_uv, H, "w_uv")
    if k_nope is None:
        k_nope = torch.empty((H, L, 128), dtype=torch.bfloat16, device=entries.device)
    if v is None:
        v = torch.empty((H, L, 128), dtype=torch.bfloat16, device=entries.device)
    _bf16(k_nope, (H, L, 128), "k_nope")
    _bf16(v, (H, L, 128), "v")
    if device_status is not None:
        _i32(device_status, "device_status")
    st = lib().mla_prefill_decompress(_ptr(entries), L, _ptr(w_uk), _ptr(w_uv), H, _ptr(k_nope), _ptr(v),
                                      _ptr(device_status), _stream(stream))
    _check("mla_prefill_decompress", st)
    return k_nope, v


def prefill_attention(q_nope, q_rope, entries, k_nope, v, softmax_scale: float, out=None, lse=None,
                      device_status=None, stream=None):
    """Causal prefill attention (non-absorbed): q_nope bf16 [L,H,128], q_rope bf16 [L,H,64],
    entries bf16 [L,576], k_nope / v bf16 [H,L,128] -> out fp32 [L,H,128], lse fp32 [L,H]."""
    if q_nope.dim() != 3:
        raise ValueError("q_nope must be [L,H,128]")
    L, H = q_nope.shape[0], q_nope.shape[1]
    _bf16(q_nope, (L, H, 128), "q_nope")
    _bf16(q_rope, (L, H, 64), "q_rope")
    _bf16(entries, (L, 576), "entries")
    _bf16(k_nope, (H, L, 128), "k_nope")
    _bf16(v, (H, L, 128), "v")
    if out is None:
        out = torch.empty((L, H, 128), dtype=torch.float32, device=q_nope.device)
    if lse is None:
        lse = torch.empty((L, H), dtype=torch.float32, device=q_nope.device)
    if device_status is not None:
        _i32(device_status, "device_status")
    st = lib().mla_prefill_attention(_ptr(q_nope), _ptr(q_rope), _ptr(entries), _ptr(k_nope), _ptr(v), L, H,
                                     float(softmax_scale), _ptr(out), _ptr(lse), _ptr(device_status),
                                     _stream(stream))
    _check("mla_prefill_attention", st)
    return out, lse


def _weights(w, H, name):
    if w.dtype != torch.bfloat16 or w.shape != (H, 128, 512) or not w.is_contiguous() or not w.is_cuda:
        raise ValueError(f"{name} must be contiguous CUDA bf16 [{H},128,512]")


def absorb_query(q_c, w_uk, q_nope=None, device_status=None, stream=None):
    """Absorbed decode query q_nope[b,h] = q_c[b,h] @ w_uk[h] (bf16 [B,H,128] x bf16 [H,128,512]
    -> bf16 [B,H,512], fp32 accumulation)."""
    if q_c.dtype != torch.bfloat16 or q_c.dim() != 3 or q_c.shape[2] != 128 or not q_c.is_contiguous() \
            or not q_c.is_cuda:
        raise ValueError("q_c must be contiguous CUDA bf16 [B,H,128]")
    B, H = q_c.shape[0], q_c.shape[1]
    _weights(w_uk, H, "w_uk")
    if q_nope is None:
        q_nope = torch.empty((B, H, 512), dtype=torch.bfloat16, device=q_c.device)
    elif q_nope.dtype != torch.bfloat16 or q_nope.shape != (B, H, 512) or not q_nope.is_contiguous():
        raise ValueError(f"q_nope must be contiguous bf16 [{B},{H},512]")
    if device_status is not None:
        _i32(device_status, "device_status")
    st = lib().mla_absorb_query(_ptr(q_c), _ptr(w_uk), B, H, _ptr(q_nope), _ptr(device_status), _stream(stream))
    _check("mla_absorb_query", st)
    return q_nope


def project_output(out, w_uv, y=None, device_status=None, stream=None):
    """Per-head value projection y[b,h] = w_uv[h] @ out[b,h] (fp32 [B,H,512], bf16 [H,128,512]
    -> fp32 [B,H,128]; the latent output enters the bf16 MMA rounded to bf16)."""
    if out.dtype != torch.float32 or out.dim() != 3 or out.shape[2] != 512 or not out.is_contiguous() \
            or not out.is_cuda:
        raise ValueError("out must be contiguous CUDA fp32 [B,H,512]")
    B, H = out.shape[0], out.shape[1]
    _weights(w_uv, H, "w_uv")
    if y is None:
        y = torch.empty((B, H, 128), dtype=torch.float32, device=out.device)
    elif y.dtype != torch.float32 or y.shape != (B, H, 128) or not y.is_contiguous():
        raise ValueError(f"y must be contiguous fp32 [{B},{H},128]")
    if device_status is not None:
        _i32(device_status, "device_status")
    st = lib().mla_project_output(_ptr(out), _ptr(w_uv), B, H, _ptr(y), _ptr(device_status), _stream(stream))
    _check("mla_project_output", st)
    return y


def decode_sparse(ws: Workspace, q_nope, q_rope, cache, block_table, seq_lens, indices,
                  softmax_scale: float, out=None, lse=None, stream=None):
    """Token-sparse decode over indices [B,topk] (int32, -1 = padding); bf16 cache."""
    B, H = _queries(q_nope, q_rope)
    _i32(block_table, "block_table")
    _i32(seq_lens, "seq_lens")
    _i32(indices, "indices")
    if cache.dtype != torch.bfloat16 or cache.shape[1:] != (64, 576) or not cache.is_contiguous():
        raise ValueError("cache must be contiguous bf16 [P,64,576]")
    out, lse = _outputs(B, H, q_nope.device, out, lse)
    st = lib().mla_decode_sparse(ws.ptr(), ws.nbytes, _ptr(q_nope), _ptr(q_rope), _ptr(cache),
                                 cache.shape[0], _ptr(block_table), block_table.shape[1],
                                 _ptr(seq_lens), _ptr(indices), indices.shape[1], B, H,
                                 float(softmax_scale), _ptr(out), _ptr(lse), _stream(stream))
    _check("mla_decode_sparse", st)
    return out, lse


def decode_static(q_nope, q_rope, cache, block_table, seq_lens, softmax_scale: float,
                  out=None, lse=None, device_status=None, stream=None):
    """Dense plan + decode + merge with the library's fixed device scratch: no workspace
    argument and no allocation inside the call.  device_status: optional int32 CUDA
    tensor [1] that receives the call's device-side status word."""
    B, H = _queries(q_nope, q_rope)
    _i32(block_table, "block_table")
    _i32(seq_lens, "seq_lens")
    if cache.dtype == torch.bfloat16 and cache.shape[1:] == (64, 576):
        kv = KV_BF16
    elif cache.dtype == torch.uint8 and cache.shape[1:] == (64, 656):
        kv = KV_FP8
    else:
        raise ValueError("cache must be bf16 [P,64,576] or uint8 [P,64,656]")
    if not cache.is_contiguous():
        raise ValueError("cache must be contiguous")
    out, lse = _outputs(B, H, q_nope.device, out, lse)
    if device_status is not None:
        _i32(device_status, "device_status")
    st = lib().mla_decode_static(_ptr(q_nope), _ptr(q_rope), _ptr(cache), kv, cache.shape[0],
                                 _ptr(block_table), block_table.shape[1], _ptr(seq_lens), B, H,
                                 float(softmax_scale), _ptr(out), _ptr(lse), _ptr(device_status),
                                 _stream(stream))
    _check("mla_decode_static", st)
    return out, lse


def set_wait_limit(cycles: int = 0) -> None:
    """Limit of every pipeline wait of the decode kernel, in SM clock cycles, for later calls
    (0 restores the default of about two seconds)."""
    _check("mla_decode_set_wait_limit", lib().mla_decode_set_wait_limit(int(cycles)))


def inject_stall(enable: bool) -> None:
    """Test hook: while enabled, decode calls make their MMA issuer wait on a barrier that
    nothing completes, so that the wait runs out (MLA_ERR_TIMEOUT) without any fault."""
    _check("mla_decode_inject_stall", lib().mla_decode_inject_stall(1 if enable else 0))


def status(ws: Workspace, stream=None) -> int:
    """Synchronise and return (and clear) the device-side status code of the workspace."""
    return int(lib().mla_decode_status(ws.ptr(), ws.nbytes, _stream(stream)))


def plan_host(seq_lens, B: int, H: int, topk: int = 0, num_sms: int = 148, kv_dtype="bf16"):
    """Host twin of the planner: returns the plan bytes (numpy uint8) for host seq_lens."""
    import numpy as np
    n = lib().mla_decode_workspace_size(int(B), int(H), int(num_sms))
    buf = np.zeros(n, dtype=np.uint8)
    sl = None
    if seq_lens is not None:
        sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    st = lib().mla_decode_plan_host(
        sl.ctypes.data_as(ctypes.c_void_p) if sl is not None else None, int(B), int(H),
        int(topk), _kv_code(kv_dtype), int(num_sms), buf.ctypes.data_as(ctypes.c_void_p), n)
    _check("mla_decode_plan_host", st)
    return buf
