"""C-ABI checks that need no GPU: exports, struct layout, host-side validation."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    import exact_io_aware_tiled_gb300 as fa
    fa.build()
    return fa.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["fa_fwd", "fa_bwd", "fa_fwd_workspace_size", "fa_bwd_workspace_size", "fa_check_status",
              "fa_dropout_mask", "fa_status_string", "fa_version"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    nm = shutil.which("nm")
    from exact_io_aware_tiled_gb300 import LIB
    if nm:
        out = subprocess.run([nm, "-D", "--defined-only", str(LIB)], capture_output=True, text=True).stdout
        exported = set(re.findall(r"\bT (fa_[a-z0-9_]+)\b", out))
    else:  # pragma: no cover
        exported = {n for n in declared_functions() if hasattr(lib, n)}
    for n in declared_functions():
        assert n in exported, n
        assert getattr(lib, n) is not None


def test_params_struct_layout_matches_c(tmp_path):
    from exact_io_aware_tiled_gb300._lib import fa_params
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    fields = [f for f, _ in fa_params._fields_]
    prog = ['#include <stdio.h>', '#include <stddef.h>', '#include "fa.h"', 'int main(void){',
            'printf("%zu\\n", sizeof(fa_params));']
    prog += ['printf("%%zu\\n", offsetof(fa_params, %s));' % f for f in fields]
    prog += ['return 0;}']
    c = tmp_path / "layout.c"
    c.write_text("\n".join(prog))
    exe = tmp_path / "layout"
    subprocess.run([gcc, "-I", os.path.join(ROOT, "include"), str(c), "-o", str(exe)], check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(fa_params)
    for f, off in zip(fields, vals[1:]):
        assert getattr(fa_params, f).offset == off, f


def _params(**kw):
    from exact_io_aware_tiled_gb300._lib import fa_params
    p = fa_params()
    p.B, p.H, p.N, p.d, p.dtype = 2, 3, 200, 64, 2
    p.stride_n, p.stride_h, p.stride_b = 64, 200 * 64, 3 * 200 * 64
    p.block_size = 128
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def test_status_strings(lib):
    assert lib.fa_status_string(0) == b"FA_OK"
    assert lib.fa_status_string(6) == b"FA_ERR_TIMEOUT"
    assert lib.fa_version() >= 102


def test_workspace_sizes(lib):
    p = _params()
    f = lib.fa_fwd_workspace_size(ctypes.byref(p))
    b = lib.fa_bwd_workspace_size(ctypes.byref(p))
    assert f >= 4
    # bwd holds the float32 dQ accumulator and the padded LSE / D rows
    assert b >= 2 * 3 * 200 * 64 * 4 + 2 * 2 * 3 * 256 * 4
    p32 = _params(dtype=0)
    assert lib.fa_bwd_workspace_size(ctypes.byref(p32)) < b


FAKE = ctypes.c_void_p(1 << 20)   # aligned, never dereferenced: validation fails first


@pytest.mark.parametrize("mut,code", [
    (dict(d=96), 2),                  # only head dims 64 and 128 are built
    (dict(d=128, dtype=0), 2),        # d = 128 has no float32 path
    (dict(d=0), 1),
    (dict(N=0), 1),
    (dict(dtype=7), 1),
    (dict(stride_n=68), 3),           # 68 * 2 bytes is not a multiple of 16
    (dict(dropout_p=1.0), 1),
    (dict(dropout_p=-0.1), 1),
    (dict(block_mask=1 << 20, block_size=64), 2),
    (dict(H_kv=2), 1),                # 3 query heads cannot share 2 K/V heads
    (dict(H_kv=1), 1),                # fewer K/V heads need their own strides
    (dict(H_kv=1, kv_stride_b=200 * 64, kv_stride_h=200 * 64, kv_stride_n=68), 3),
    (dict(window=5), 2),              # a sliding window needs causal masking
    (dict(window=-1, causal=1), 1),
])
def test_host_validation_rejects_before_launch(lib, mut, code):
    p = _params(**mut)
    ws = ctypes.c_void_p(1 << 21)
    st = lib.fa_fwd(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, ws, 1 << 30, None)
    assert st == code


def test_null_and_misaligned_pointers_and_small_workspace(lib):
    p = _params()
    ws = ctypes.c_void_p(1 << 21)
    assert lib.fa_fwd(None, FAKE, FAKE, FAKE, FAKE, FAKE, ws, 1 << 30, None) == 1
    assert lib.fa_fwd(ctypes.byref(p), None, FAKE, FAKE, FAKE, FAKE, ws, 1 << 30, None) == 1
    assert lib.fa_fwd(ctypes.byref(p), ctypes.c_void_p((1 << 20) + 8), FAKE, FAKE, FAKE, FAKE, ws, 1 << 30,
                      None) == 3
    assert lib.fa_fwd(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, ws, 16, None) == 4
    assert lib.fa_fwd(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, None, 1 << 30, None) == 4
    assert lib.fa_bwd(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, ws, 1 << 30,
                      None) == 1
    assert lib.fa_bwd(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws, 16, None) == 4
    assert lib.fa_dropout_mask(ctypes.byref(p), 2, 0, 0, 1, FAKE, None) == 1      # b out of range
    assert lib.fa_dropout_mask(ctypes.byref(p), 0, 0, 190, 20, FAKE, None) == 1   # rows past N


def test_product_path_refuses_to_run_without_library(tmp_path, monkeypatch):
    import exact_io_aware_tiled_gb300._lib as L
    monkeypatch.setattr(L, "_lib", None)
    monkeypatch.setattr(L, "_LIB_PATH", tmp_path / "missing.so")
    with pytest.raises(RuntimeError, match="not built"):
        L.load()


def test_binding_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "exact_io_aware_tiled_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", src, flags=re.M), f
                assert "oracle." not in src or f.endswith((".cu", ".cuh", ".h")), f


# ---- FP8 forward (ABI 1.2) ---------------------------------------------------
def test_fp8_structs_match_c(tmp_path):
    from exact_io_aware_tiled_gb300._lib import fa_fp8_layout, fa_fp8_params
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    prog = ['#include <stdio.h>', '#include <stddef.h>', '#include "fa.h"', 'int main(void){']
    for st in (fa_fp8_params, fa_fp8_layout):
        prog.append('printf("%%zu\\n", sizeof(%s));' % st.__name__)
        prog += ['printf("%%zu\\n", offsetof(%s, %s));' % (st.__name__, f) for f, _ in st._fields_]
    prog += ['return 0;}']
    c = tmp_path / "fp8layout.c"
    c.write_text("\n".join(prog))
    exe = tmp_path / "fp8layout"
    subprocess.run([gcc, "-I", os.path.join(ROOT, "include"), str(c), "-o", str(exe)], check=True)
    vals = iter(int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True).stdout.split())
    for st in (fa_fp8_params, fa_fp8_layout):
        assert next(vals) == ctypes.sizeof(st)
        for f, _ in st._fields_:
            assert getattr(st, f).offset == next(vals), f


def test_fp8_buffer_layout(lib):
    from exact_io_aware_tiled_gb300._lib import fa_fp8_layout
    p = _params(H=4, H_kv=2, kv_stride_b=2 * 200 * 64, kv_stride_h=200 * 64, kv_stride_n=64)
    lay = fa_fp8_layout()
    assert lib.fa_fp8_buffer_layout(ctypes.byref(p), ctypes.byref(lay)) == 0
    parts = [lay.q8, lay.k8, lay.v8t, lay.sq, lay.sk, lay.sv, lay.amax, lay.total]
    assert parts == sorted(parts) and all(x % 256 == 0 for x in parts)
    assert lay.k8 - lay.q8 >= 2 * 4 * 200 * 64            # Q codes: one byte per element
    assert lay.sq - lay.v8t >= 2 * 2 * 64 * 256           # V^T codes: keys padded to 256
    assert lay.sk - lay.sq >= 2 * 4 * 2 * 4               # two 128-row tiles per head
    assert lib.fa_fp8_buffer_layout(None, ctypes.byref(lay)) == 1


@pytest.mark.parametrize("mut,fmut,code", [
    (dict(dtype=0), {}, 2),           # no float32 FP8 path
    (dict(d=96, stride_n=96, stride_h=200 * 96, stride_b=600 * 96), {}, 2),   # head dimensions 64 and 128 only
    (dict(dropout_p=0.1), {}, 2),     # no dropout in the FP8 forward
    ({}, dict(per_tensor=2), 1),
    ({}, dict(signs=(1 << 20) + 4), 3),
    (dict(window=5), {}, 2),
])
def test_fp8_host_validation(lib, mut, fmut, code):
    from exact_io_aware_tiled_gb300._lib import fa_fp8_params
    p = _params(**mut)
    f = fa_fp8_params()
    for k, v in fmut.items():
        setattr(f, k, v)
    ws = ctypes.c_void_p(1 << 21)
    assert lib.fa_fp8_quantize(ctypes.byref(p), ctypes.byref(f), FAKE, FAKE, FAKE, ws, 1 << 30, None) == code
    assert lib.fa_fwd_fp8(ctypes.byref(p), ctypes.byref(f), ws, 1 << 30, FAKE, FAKE, ws, 1 << 30, None) == code


def test_fp8_small_buffers_are_refused(lib):
    from exact_io_aware_tiled_gb300._lib import fa_fp8_params
    p = _params()
    f = fa_fp8_params()
    ws = ctypes.c_void_p(1 << 21)
    assert lib.fa_fp8_quantize(ctypes.byref(p), ctypes.byref(f), FAKE, FAKE, FAKE, ws, 256, None) == 4
    assert lib.fa_fwd_fp8(ctypes.byref(p), ctypes.byref(f), ws, 256, FAKE, FAKE, ws, 1 << 30, None) == 4
    assert lib.fa_fwd_fp8(ctypes.byref(p), ctypes.byref(f), ws, 1 << 30, FAKE, FAKE, ws, 16, None) == 4
    assert lib.fa_fwd_fp8(ctypes.byref(p), None, ws, 1 << 30, FAKE, FAKE, ws, 1 << 30, None) == 1


@pytest.mark.parametrize("d", [64, 128])
def test_fp8_views_follow_the_library_layout(lib, d):
    import torch
    import exact_io_aware_tiled_gb300 as fa
    q = torch.empty((2, 4, 300, d), dtype=torch.bfloat16)
    k = torch.empty((2, 2, 300, d), dtype=torch.bfloat16)
    p = fa.make_params(q, k=k)
    lay = fa.fp8_layout(p)
    buf = torch.zeros(lay["total"], dtype=torch.uint8)
    v = fa.fp8_views(buf, lay, 2, 4, 2, 300, d)
    nt, npad = 3, 384
    shapes = dict(q8=(2, 4, 300, d), k8=(2, 2, 300, d), v8t=(2, 2, d, npad), sq=(2, 4, nt), sk=(2, 2, nt),
                  sv=(2, 2, nt))
    base = buf.data_ptr()
    spans = []
    for name, shp in shapes.items():
        t = v[name]
        assert tuple(t.shape) == shp and t.is_contiguous(), name
        assert t.data_ptr() - base == lay[name], name
        spans.append((t.data_ptr() - base, t.data_ptr() - base + t.numel() * t.element_size()))
    spans.sort()
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))     # no overlap
    assert spans[-1][1] <= lay["amax"] < lay["total"]
