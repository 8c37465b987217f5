"""ctypes binding of the C ABI in include/fa.h (argument marshalling only).

Every step of the attention computation runs in the CUDA kernels of
``libfa_gb300.so``; this module only checks tensor shapes and devices, allocates
outputs and the workspace with torch, and passes raw pointers and the current
CUDA stream.  If the library has not been built it raises -- there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import math
from pathlib import Path
from typing import Optional

import torch

_LIB_PATH = Path(__file__).resolve().parent / "libfa_gb300.so"

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_MISALIGNED, FA_ERR_WORKSPACE, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(7)
DTYPE_CODE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}

EXPORTED = ["fa_fwd_workspace_size", "fa_bwd_workspace_size", "fa_fwd", "fa_bwd", "fa_bwd_noalloc",
            "fa_noalloc_check_status", "fa_noalloc_scratch",
            "fa_check_status", "fa_dropout_mask", "fa_selftest_wait_timeout", "fa_status_string", "fa_version",
            "fa_fp8_buffer_layout", "fa_fp8_quantize", "fa_fwd_fp8"]


class fa_params(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("N", ctypes.c_int32), ("d", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("stride_b", ctypes.c_int64), ("stride_h", ctypes.c_int64), ("stride_n", ctypes.c_int64),
        ("scale", ctypes.c_float),
        ("causal", ctypes.c_int32),
        ("seqlens_k", ctypes.c_void_p),
        ("dropout_p", ctypes.c_float),
        ("seed", ctypes.c_uint64), ("offset", ctypes.c_uint64),
        ("block_mask", ctypes.c_void_p),
        ("block_size", ctypes.c_int32),
        ("o_f32", ctypes.c_void_p),
        ("prof_start", ctypes.c_void_p), ("prof_stop", ctypes.c_void_p),
        ("H_kv", ctypes.c_int32),
        ("kv_stride_b", ctypes.c_int64), ("kv_stride_h", ctypes.c_int64), ("kv_stride_n", ctypes.c_int64),
        ("window", ctypes.c_int32),
        ("fwd_kernel", ctypes.c_int32),
    ]


class fa_fp8_params(ctypes.Structure):
    _fields_ = [("per_tensor", ctypes.c_int32), ("signs", ctypes.c_void_p)]


class fa_fp8_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("q8", "k8", "v8t", "sq", "sk", "sv", "amax", "total")]


class FAError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        super().__init__("%s: %s" % (what, status_string(code)))


_lib = None


def load():
    """Load libfa_gb300.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not _LIB_PATH.exists():
        raise RuntimeError("libfa_gb300.so is not built; run "
                           "`python -m exact_io_aware_tiled_gb300._build` (or __graft_entry__.build())")
    lib = ctypes.CDLL(str(_LIB_PATH))
    P = ctypes.POINTER(fa_params)
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    lib.fa_fwd_workspace_size.argtypes = [P]
    lib.fa_fwd_workspace_size.restype = sz
    lib.fa_bwd_workspace_size.argtypes = [P]
    lib.fa_bwd_workspace_size.restype = sz
    lib.fa_fwd.argtypes = [P, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.fa_fwd.restype = ctypes.c_int
    lib.fa_bwd.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.fa_bwd.restype = ctypes.c_int
    lib.fa_check_status.argtypes = [vp, vp]
    lib.fa_check_status.restype = ctypes.c_int
    lib.fa_dropout_mask.argtypes = [P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, vp, vp]
    lib.fa_dropout_mask.restype = ctypes.c_int
    lib.fa_status_string.argtypes = [ctypes.c_int]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_version.argtypes = []
    lib.fa_version.restype = ctypes.c_int32
    F = ctypes.POINTER(fa_fp8_params)
    lib.fa_fp8_buffer_layout.argtypes = [P, ctypes.POINTER(fa_fp8_layout)]
    lib.fa_fp8_buffer_layout.restype = ctypes.c_int
    lib.fa_fp8_quantize.argtypes = [P, F, vp, vp, vp, vp, sz, vp]
    lib.fa_fp8_quantize.restype = ctypes.c_int
    lib.fa_fwd_fp8.argtypes = [P, F, vp, sz, vp, vp, vp, sz, vp]
    lib.fa_fwd_fp8.restype = ctypes.c_int
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load().fa_status_string(int(code)).decode()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_params(q: torch.Tensor, *, k: Optional[torch.Tensor] = None, causal=False, seqlens_k=None, dropout_p=0.0,
                seed=0, offset=0, block_mask=None, scale=None, o_f32=None, prof=None, window=0,
                fwd_kernel=0) -> fa_params:
    B, H, N, d = q.shape
    p = fa_params()
    p.B, p.H, p.N, p.d = B, H, N, d
    p.dtype = DTYPE_CODE[q.dtype]
    p.stride_b, p.stride_h, p.stride_n = q.stride(0), q.stride(1), q.stride(2)
    if k is not None:   # K/V (and dK/dV) layout; fewer heads = grouped-query attention
        p.H_kv = k.shape[1]
        p.kv_stride_b, p.kv_stride_h, p.kv_stride_n = k.stride(0), k.stride(1), k.stride(2)
    p.window = int(window)
    p.fwd_kernel = int(fwd_kernel)
    p.scale = 0.0 if scale is None else float(scale)
    p.causal = 1 if causal else 0
    p.seqlens_k = None if seqlens_k is None else seqlens_k.data_ptr()
    p.dropout_p = float(dropout_p)
    p.seed = int(seed) & (2 ** 64 - 1)
    p.offset = int(offset) & (2 ** 64 - 1)
    p.block_mask = None if block_mask is None else block_mask.data_ptr()
    p.block_size = 128
    p.o_f32 = None if o_f32 is None else o_f32.data_ptr()
    if prof is not None:
        p.prof_start, p.prof_stop = prof
    return p


def _same_layout(ts):
    """Tensors of one group must share one stride set with a contiguous last dim.

    The C ABI takes one stride set per group (q, o, dO, dQ and k, v, dK, dV),
    so tensors that differ would need a copy.  No copy is made here: that
    would be hidden HBM traffic on every call.  A mismatch raises instead."""
    ref = ts[0]
    for t in ts:
        if t.shape != ref.shape or t.dtype != ref.dtype:
            raise ValueError("tensors of one group must share shape and dtype: %s %s vs %s %s"
                             % (tuple(t.shape), t.dtype, tuple(ref.shape), ref.dtype))
        if t.stride() != ref.stride():
            raise ValueError("tensors of one group must share their strides (%s vs %s); make them "
                             "alike, e.g. with .contiguous() on each" % (t.stride(), ref.stride()))
    if ref.stride(3) != 1:
        raise ValueError("the last dimension must be contiguous (stride 1), got strides %s" % (ref.stride(),))
    return ts


def _layouts(q_like, kv):
    """Q-side tensors ([B,H,N,d]) and K/V-side tensors ([B,H_kv,N,d], H % H_kv == 0)."""
    q_like = _same_layout(q_like)
    kv = _same_layout(kv)
    q, k = q_like[0], kv[0]
    if k.dim() != 4 or (k.shape[0], k.shape[2], k.shape[3]) != (q.shape[0], q.shape[2], q.shape[3]):
        raise ValueError("k, v must be [B, H_kv, N, d] with the B, N, d of q")
    if k.shape[1] < 1 or q.shape[1] % k.shape[1] != 0:
        raise ValueError("the number of query heads must be a multiple of the number of K/V heads")
    if k.dtype != q.dtype:
        raise ValueError("q, k, v must share one dtype")
    return q_like, kv


def _check(q, name="q"):
    if q.dim() != 4:
        raise ValueError("%s must be [B, H, N, d]" % name)
    if not q.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if q.dtype not in DTYPE_CODE:
        raise ValueError("unsupported dtype %s" % q.dtype)


def _aux(seqlens_k, block_mask, q):
    B, N = q.shape[0], q.shape[2]
    if seqlens_k is not None:
        if tuple(seqlens_k.shape) != (B,):
            raise ValueError("seqlens_k must have shape [B]")
        seqlens_k = seqlens_k.to(device=q.device, dtype=torch.int32).contiguous()
    if block_mask is not None:
        nb = -(-N // 128)
        if tuple(block_mask.shape) != (nb, nb):
            raise ValueError("block_mask must have shape [ceil(N/128), ceil(N/128)] = [%d, %d]" % (nb, nb))
        block_mask = block_mask.to(device=q.device, dtype=torch.uint8).contiguous()
    return seqlens_k, block_mask


def _outputs(out, likes):
    """Caller-provided output tensors (checked against the shapes, dtypes and
    devices the call would allocate), or fresh ones."""
    if out is None:
        return [torch.empty_like(t) if isinstance(t, torch.Tensor) else torch.empty(t[0], dtype=t[1], device=t[2])
                for t in likes]
    if len(out) != len(likes):
        raise ValueError("out must hold %d tensors" % len(likes))
    for o, t in zip(out, likes):
        shape, dtype, device = (t.shape, t.dtype, t.device) if isinstance(t, torch.Tensor) else t
        if tuple(o.shape) != tuple(shape) or o.dtype != dtype or o.device != torch.device(device) or \
                not o.is_contiguous():
            raise ValueError("out tensor %s %s does not match %s %s (contiguous)" % (tuple(o.shape), o.dtype,
                                                                                  tuple(shape), dtype))
    return list(out)


def _workspace(lib_size, workspace, device):
    """A caller-provided uint8 workspace of at least lib_size bytes, or a fresh one."""
    if workspace is None:
        return torch.empty(lib_size, device=device, dtype=torch.uint8)
    if workspace.dtype != torch.uint8 or workspace.numel() < lib_size or workspace.device != device:
        raise ValueError("workspace must be a uint8 tensor of >= %d bytes on %s" % (lib_size, device))
    return workspace


def fwd(q, k, v, *, causal=False, seqlens_k=None, dropout_p=0.0, seed=0, offset=0, block_mask=None,
        scale=None, return_o_f32=False, stream=None, prof=None, window=0, out=None, workspace=None, fwd_kernel=0):
    """O, LSE (and optionally the float32 O before rounding) via fa_fwd.

    k, v may have fewer heads than q (grouped-query attention); ``window`` > 0
    (with ``causal``) restricts query i to keys i - window < j <= i.  ``out``
    = (o, lse) and ``workspace`` (uint8, fa_fwd_workspace_size bytes) let a
    caller reuse its own buffers instead of allocating on every call.
    ``fwd_kernel`` (head dimension 64): 0 lets the library choose, 1 / 2
    force the one- / two-query-tile kernel."""
    _check(q)
    (q,), (k, v) = _layouts([q], [k, v])
    lib = load()
    seqlens_k, block_mask = _aux(seqlens_k, block_mask, q)
    B, H, N, d = q.shape
    if out is not None and not q.is_contiguous():
        raise ValueError("out= takes contiguous outputs, so q must be contiguous too (o shares q's strides)")
    o, lse = _outputs(out, [q, ((B, H, N), torch.float32, q.device)])
    o32 = torch.empty((B, H, N, d), device=q.device, dtype=torch.float32) if return_o_f32 else None
    p = make_params(q, k=k, causal=causal, seqlens_k=seqlens_k, dropout_p=dropout_p, seed=seed, offset=offset,
                    block_mask=block_mask, scale=scale, o_f32=o32, prof=prof, window=window, fwd_kernel=fwd_kernel)
    wsz = lib.fa_fwd_workspace_size(ctypes.byref(p))
    ws = _workspace(wsz, workspace, q.device)
    st = lib.fa_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(ws), wsz, _stream(stream))
    if st != FA_OK:
        raise FAError(st, "fa_fwd")
    fwd.last_workspace = ws
    return (o, lse, o32) if return_o_f32 else (o, lse)


def bwd(q, k, v, o, do, lse, *, causal=False, seqlens_k=None, dropout_p=0.0, seed=0, offset=0, block_mask=None,
        scale=None, stream=None, prof=None, window=0, out=None, workspace=None):
    """dQ, dK, dV via fa_bwd (dK, dV have the K/V heads of k, v).  ``out`` =
    (dq, dk, dv) and ``workspace`` (uint8, fa_bwd_workspace_size bytes) let a
    caller reuse its own buffers; the outputs must then share q's / k's
    (contiguous) layout."""
    _check(q)
    (q, o, do), (k, v) = _layouts([q, o, do], [k, v])
    if out is not None and (not q.is_contiguous() or not k.is_contiguous()):
        raise ValueError("out= takes contiguous outputs, so q, o, dO, k and v must be contiguous too")
    if not lse.is_contiguous():
        raise ValueError("lse must be the contiguous [B, H, N] float32 tensor fwd returns")
    lib = load()
    seqlens_k, block_mask = _aux(seqlens_k, block_mask, q)
    dq, dk, dv = _outputs(out, [q, k, v])
    p = make_params(q, k=k, causal=causal, seqlens_k=seqlens_k, dropout_p=dropout_p, seed=seed, offset=offset,
                    block_mask=block_mask, scale=scale, prof=prof, window=window)
    wsz = lib.fa_bwd_workspace_size(ctypes.byref(p))
    ws = _workspace(wsz, workspace, q.device)
    st = lib.fa_bwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk),
                    _ptr(dv), _ptr(ws), wsz, _stream(stream))
    if st != FA_OK:
        raise FAError(st, "fa_bwd")
    bwd.last_workspace = ws
    return dq, dk, dv


def check_status(ws: torch.Tensor, stream=None) -> int:
    """Synchronise and return the status word a previous call left in ``ws``."""
    return load().fa_check_status(_ptr(ws), _stream(stream))


def dropout_mask(B, H, N, b, h, row0, nrows, *, dropout_p, seed=0, offset=0, device="cuda", stream=None):
    """uint8 [nrows, N] keep-mask of rows row0.. of head (b, h) via fa_dropout_mask."""
    lib = load()
    p = fa_params()
    p.B, p.H, p.N, p.d = B, H, N, 64
    p.dropout_p = float(dropout_p)
    p.seed = int(seed) & (2 ** 64 - 1)
    p.offset = int(offset) & (2 ** 64 - 1)
    out = torch.empty((nrows, N), device=device, dtype=torch.uint8)
    st = lib.fa_dropout_mask(ctypes.byref(p), b, h, row0, nrows, _ptr(out), _stream(stream))
    if st != FA_OK:
        raise FAError(st, "fa_dropout_mask")
    return out


def selftest_wait_timeout(device="cuda", stream=None, ws_ptr=None):
    """Run fa_selftest_wait_timeout: returns (status, gave_up[2], waited_ns of the second warp).

    ws_ptr: a raw device address of at least 256 bytes to use as the
    workspace (e.g. the fixed array of ``noalloc_scratch``); default a fresh
    256-byte tensor."""
    lib = load()
    fn = lib.fa_selftest_wait_timeout
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    ws = torch.empty(256, device=device, dtype=torch.uint8) if ws_ptr is None else None
    wsp = _ptr(ws) if ws_ptr is None else ctypes.c_void_p(int(ws_ptr))
    out = torch.zeros(2, device=device, dtype=torch.int32)
    ns = torch.zeros(1, device=device, dtype=torch.int64)
    st = fn(wsp, _ptr(out), _ptr(ns), _stream(stream))
    if st != FA_OK:
        raise FAError(st, "fa_selftest_wait_timeout")
    status = lib.fa_check_status(wsp, _stream(stream))
    return status, out.cpu().tolist(), int(ns.item())


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


def bwd_noalloc(q, k, v, o, do, lse, *, causal=False, seqlens_k=None, dropout_p=0.0, seed=0, offset=0,
                block_mask=None, scale=None, stream=None, window=0):
    """dQ, dK, dV via fa_bwd_noalloc: the backward pass using the library's own
    fixed device scratch array instead of a caller-allocated workspace (for
    callers that cannot allocate device memory; problems needing more than
    64 MiB of scratch are refused)."""
    _check(q)
    (q, o, do), (k, v) = _layouts([q, o, do], [k, v])
    lib = load()
    fn = lib.fa_bwd_noalloc
    fn.argtypes = [ctypes.POINTER(fa_params)] + [ctypes.c_void_p] * 10
    fn.restype = ctypes.c_int
    seqlens_k, block_mask = _aux(seqlens_k, block_mask, q)
    if not lse.is_contiguous():
        raise ValueError("lse must be the contiguous [B, H, N] float32 tensor fwd returns")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    p = make_params(q, k=k, causal=causal, seqlens_k=seqlens_k, dropout_p=dropout_p, seed=seed, offset=offset,
                    block_mask=block_mask, scale=scale, window=window)
    st = fn(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
            _stream(stream))
    if st != FA_OK:
        raise FAError(st, "fa_bwd_noalloc")
    return dq, dk, dv


def noalloc_check_status(stream=None) -> int:
    """Synchronise and return the status word the last bwd_noalloc on the
    current device left in the library's fixed scratch array."""
    lib = load()
    fn = lib.fa_noalloc_check_status
    fn.argtypes = [ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn(_stream(stream))


def noalloc_scratch():
    """(device address, bytes) of the fixed scratch array on the current device."""
    lib = load()
    fn = lib.fa_noalloc_scratch
    fn.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_size_t)]
    fn.restype = ctypes.c_int
    a, n = ctypes.c_void_p(), ctypes.c_size_t()
    st = fn(ctypes.byref(a), ctypes.byref(n))
    if st != FA_OK:
        raise FAError(st, "fa_noalloc_scratch")
    return int(a.value), int(n.value)


def _fp8_args(q, signs, per_tensor):
    f = fa_fp8_params()
    f.per_tensor = 1 if per_tensor else 0
    sg = None
    if signs is not None:
        sg = torch.as_tensor(signs).to(device=q.device, dtype=torch.int8).contiguous()
        if sg.numel() != q.shape[3]:
            raise ValueError("signs must have d entries")
        f.signs = sg.data_ptr()
    return f, sg


def fp8_layout(p: fa_params) -> dict:
    """Byte offsets of the quantised buffer's parts (fa_fp8_buffer_layout)."""
    lay = fa_fp8_layout()
    st = load().fa_fp8_buffer_layout(ctypes.byref(p), ctypes.byref(lay))
    if st != FA_OK:
        raise FAError(st, "fa_fp8_buffer_layout")
    return {n: int(getattr(lay, n)) for n, _ in fa_fp8_layout._fields_}


def fp8_views(buf: torch.Tensor, lay: dict, B, H, H_kv, N, d=64) -> dict:
    """The quantised buffer's parts as tensors (views, no copies)."""
    nt = -(-N // 128)
    npad = nt * 128

    def u8(off, shape):
        n = math.prod(shape)
        return buf[off:off + n].view(shape)

    def f32(off, shape):
        n = math.prod(shape)
        return buf[off:off + 4 * n].view(torch.float32).view(shape)

    return dict(q8=u8(lay["q8"], (B, H, N, d)), k8=u8(lay["k8"], (B, H_kv, N, d)),
                v8t=u8(lay["v8t"], (B, H_kv, d, npad)), sq=f32(lay["sq"], (B, H, nt)),
                sk=f32(lay["sk"], (B, H_kv, nt)), sv=f32(lay["sv"], (B, H_kv, nt)))


def fp8_quantize(q, k, v, *, signs=None, per_tensor=False, stream=None, buf=None):
    """Quantise q, k, v to E4M3 (fa_fp8_quantize): returns (buffer, views)."""
    _check(q)
    (q,), (k, v) = _layouts([q], [k, v])
    lib = load()
    p = make_params(q, k=k)
    f, sg = _fp8_args(q, signs, per_tensor)
    lay = fp8_layout(p)
    if buf is None:
        buf = torch.empty(lay["total"], device=q.device, dtype=torch.uint8)
    st = lib.fa_fp8_quantize(ctypes.byref(p), ctypes.byref(f), _ptr(q), _ptr(k), _ptr(v), _ptr(buf), buf.numel(),
                             _stream(stream))
    if st != FA_OK:
        raise FAError(st, "fa_fp8_quantize")
    fp8_quantize.last_signs = sg       # keep the device copy alive until the stream has used it
    return buf, fp8_views(buf, lay, q.shape[0], q.shape[1], k.shape[1], q.shape[2], q.shape[3])


def fwd_fp8(q, k, v, *, signs=None, per_tensor=False, causal=False, seqlens_k=None, block_mask=None, scale=None,
            window=0, return_o_f32=False, return_quantized=False, stream=None, prof=None, buf=None, out=None,
            workspace=None):
    """FP8 forward (fa_fp8_quantize + fa_fwd_fp8): O (dtype of q), LSE, and
    optionally the float32 O before rounding and the quantised operands.
    ``buf`` (the quantised buffer), ``out`` = (o, lse) and ``workspace`` let a
    caller reuse its own buffers."""
    _check(q)
    (q,), (k, v) = _layouts([q], [k, v])
    if out is not None and not q.is_contiguous():
        raise ValueError("out= takes contiguous outputs, so q must be contiguous too (o shares q's strides)")
    lib = load()
    seqlens_k, block_mask = _aux(seqlens_k, block_mask, q)
    B, H, N, d = q.shape
    f, sg = _fp8_args(q, signs, per_tensor)
    buf, views = fp8_quantize(q, k, v, signs=sg, per_tensor=per_tensor, stream=stream, buf=buf)
    o, lse = _outputs(out, [q, ((B, H, N), torch.float32, q.device)])
    o32 = torch.empty((B, H, N, d), device=q.device, dtype=torch.float32) if return_o_f32 else None
    p = make_params(q, k=k, causal=causal, seqlens_k=seqlens_k, block_mask=block_mask, scale=scale, o_f32=o32,
                    prof=prof, window=window)
    wsz = lib.fa_fwd_workspace_size(ctypes.byref(p))
    ws = _workspace(wsz, workspace, q.device)
    st = lib.fa_fwd_fp8(ctypes.byref(p), ctypes.byref(f), _ptr(buf), buf.numel(), _ptr(o), _ptr(lse), _ptr(ws), wsz,
                        _stream(stream))
    if st != FA_OK:
        raise FAError(st, "fa_fwd_fp8")
    fwd_fp8.last_workspace = ws
    fwd_fp8.last_signs = sg
    out = (o, lse)
    if return_o_f32:
        out = out + (o32,)
    if return_quantized:
        out = out + (views,)
    return out
