"""CPU checks of the C ABI: the library builds and loads, exports every declared symbol,
and rejects bad arguments on the host before touching a GPU."""
import ctypes
import os
import re

import pytest

from mla_latent_kv_17_gb300 import build as mbuild
from mla_latent_kv_17_gb300 import ops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session")
def L():
    mbuild.build()
    return ops.lib()


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", h)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names += re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", txt)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("mla_decode_workspace_size", "mla_decode_plan", "mla_decode", "mla_decode_sparse",
                 "mla_decode_status", "mla_status_string", "mla_decode_plan_host",
                 "mla_cache_append", "mla_absorb_query", "mla_project_output", "mla_topk_select",
                 "mla_prefill_decompress", "mla_prefill_attention", "mla_decode_set_wait_limit",
                 "mla_decode_inject_stall", "mla_decode_static"):
        assert must in names


def test_header_is_plain_c():
    # the boundary carries no C++ or torch types: the header compiles as C99 on its own
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            r = subprocess.run([cc, "-fsyntax-only", "-std=c99", "-Wall", "-Werror", "-x", "c",
                                os.path.join(ROOT, "include", h)], capture_output=True, text=True)
            assert r.returncode == 0, r.stderr


def test_c_program_uses_the_abi_without_python(L, tmp_path):
    # a plain C program links the library and calls its host-side entry points
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(ops.LIB_PATH)
    exe = str(tmp_path / "abi_host")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        os.path.join(ROOT, "tests", "c", "abi_host.c"), "-L", libdir, "-lmla_decode",
                        f"-Wl,-rpath,{libdir}", "-o", exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert "c abi ok" in r.stdout


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in include/ but not exported"


def test_status_strings(L):
    for code in range(8):
        s = L.mla_status_string(code).decode()
        assert s and s != "unknown status"
    assert L.mla_status_string(99).decode() == "unknown status"


def test_workspace_size_validation(L):
    assert L.mla_decode_workspace_size(0, 128, 148) == 0
    assert L.mla_decode_workspace_size(4, 0, 148) == 0
    assert L.mla_decode_workspace_size(4, 129, 148) == 0
    n1 = L.mla_decode_workspace_size(64, 128, 148)
    n2 = L.mla_decode_workspace_size(64, 128, 152)
    assert n1 > 0 and n2 >= n1
    # partial results: (B + units) slots of H x 512 fp32 dominate
    assert n1 >= (64 + 74) * 128 * 512 * 4


def test_decode_rejects_bad_arguments_on_host(L):
    P = ctypes.c_void_p
    fake = P(4096)  # never dereferenced: argument checks run before any CUDA call
    args = dict(ws=fake, ws_bytes=1 << 30, qn=fake, qr=fake, cache=fake, kv=0, num_pages=10,
                bt=fake, max_pages=4, sl=fake, B=2, H=16, scale=0.07, out=fake, lse=fake)

    def call(**kw):
        a = dict(args, **kw)
        return L.mla_decode(a["ws"], a["ws_bytes"], a["qn"], a["qr"], a["cache"], a["kv"],
                            a["num_pages"], a["bt"], a["max_pages"], a["sl"], a["B"], a["H"],
                            ctypes.c_float(a["scale"]), a["out"], a["lse"], None)

    assert call(qn=None) == 1
    assert call(cache=None) == 1
    assert call(B=0) == 1
    assert call(H=0) == 1
    assert call(H=129) == 2
    assert call(max_pages=0) == 1
    assert call(num_pages=0) == 1
    assert call(scale=float("nan")) == 1
    assert call(scale=float("inf")) == 1
    assert call(scale=0.0) == 1
    assert call(scale=-0.07) == 1
    assert call(kv=7) == 1
    assert call(qn=P(4098)) == 1          # not 16-byte aligned
    assert call(cache=P(4104)) == 1
    assert call(ws_bytes=16) == 3


def test_sparse_rejects_bad_arguments_on_host(L):
    P = ctypes.c_void_p
    f = P(4096)
    st = L.mla_decode_sparse(f, 1 << 30, f, f, f, 10, f, 4, f, None, 2048, 2, 16,
                             ctypes.c_float(0.07), f, f, None)
    assert st == 1
    st = L.mla_decode_sparse(f, 1 << 30, f, f, f, 10, f, 4, f, f, 0, 2, 16,
                             ctypes.c_float(0.07), f, f, None)
    assert st == 1


def test_plan_rejects_bad_arguments_on_host(L):
    P = ctypes.c_void_p
    assert L.mla_decode_plan(None, 2, 16, 0, 0, 148, None, 1 << 20, None) == 1
    assert L.mla_decode_plan(None, 2, 16, 0, 0, 148, P(4096), 1 << 20, None) == 1  # no seq_lens, no topk
    assert L.mla_decode_plan(P(4096), 2, 200, 0, 0, 148, P(4096), 1 << 20, None) == 2
    assert L.mla_decode_plan(P(4096), 2, 16, 0, 0, 148, P(4096), 64, None) == 3
    assert L.mla_decode_plan(P(4096), 2, 16, 0, 7, 148, P(4096), 1 << 20, None) == 1   # unknown cache layout
    assert L.mla_decode_plan(None, 2, 16, 64, 1, 148, P(4096), 1 << 20, None) == 2     # top-k over FP8 records
    assert L.mla_decode_plan_host(None, 2, 16, 0, 0, 0, P(4096), 1 << 20) == 1


def test_absorb_project_append_reject_bad_arguments_on_host(L):
    P = ctypes.c_void_p
    f = P(4096)
    odd = P(4096 + 8)  # not 16-byte aligned
    assert L.mla_absorb_query(None, f, 4, 16, f, None, None) == 1
    assert L.mla_absorb_query(f, f, 0, 16, f, None, None) == 1
    assert L.mla_absorb_query(f, f, 4, 0, f, None, None) == 1
    assert L.mla_absorb_query(f, odd, 4, 16, f, None, None) == 1
    assert L.mla_project_output(f, None, 4, 16, f, None, None) == 1
    assert L.mla_project_output(f, f, -1, 16, f, None, None) == 1
    assert L.mla_project_output(odd, f, 4, 16, f, None, None) == 1
    assert L.mla_prefill_decompress(None, 64, f, f, 4, f, f, None, None) == 1
    assert L.mla_prefill_decompress(f, 0, f, f, 4, f, f, None, None) == 1
    assert L.mla_prefill_decompress(f, 64, f, odd, 4, f, f, None, None) == 1
    assert L.mla_prefill_attention(f, f, None, f, f, 64, 4, ctypes.c_float(0.07), f, f, None, None) == 1
    assert L.mla_prefill_attention(f, f, f, f, f, 0, 4, ctypes.c_float(0.07), f, f, None, None) == 1
    assert L.mla_prefill_attention(f, f, f, f, f, 64, 4, ctypes.c_float(0.0), f, f, None, None) == 1
    assert L.mla_prefill_attention(f, odd, f, f, f, 64, 4, ctypes.c_float(0.07), f, f, None, None) == 1
    assert L.mla_topk_select(None, 64, 64, f, 2, 8, f, None, None) == 1
    assert L.mla_topk_select(f, 62, 62, f, 2, 8, f, None, None) == 1     # stride not a multiple of 4
    assert L.mla_topk_select(f, 64, 65, f, 2, 8, f, None, None) == 1     # stride < Lmax
    assert L.mla_topk_select(f, 64, 64, f, 2, 0, f, None, None) == 1     # k < 1
    assert L.mla_topk_select(odd, 64, 64, f, 2, 8, f, None, None) == 1
    assert L.mla_cache_append(f, 0, 10, f, 4, f, f, f, 0, None, None) == 1
    assert L.mla_cache_append(f, 7, 10, f, 4, f, f, f, 2, None, None) == 1
    assert L.mla_cache_append(odd, 0, 10, f, 4, f, f, f, 2, None, None) == 1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(ops, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(ops, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        ops.lib()
