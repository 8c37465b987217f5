"""Shared helpers of the GPU parity tests: run the CUDA path, run the oracle, compare.

Tolerances (written here once, used by every parity test):
  float32 inputs: max|dO| <= 1e-5 on O, |dLSE| <= 1e-5, relative Frobenius
                  error <= 1e-5 for dQ, dK, dV.
  16-bit inputs:  max|dO| <= 4e-3 on the kernel's float32 O (exported before
                  the final rounding); the stored 16-bit O within 4e-3 plus
                  half an ulp of the storage dtype at |O_ref|; |dLSE| <= 1e-3;
                  relative Frobenius error <= 1e-2 for dQ, dK, dV.
With dropout the 16-bit O bound widens by the first-order effect of rounding
the MMA input P~ = Z o P / (1 - p) to the storage dtype (unit roundoff u =
2^-8 for bf16, 2^-11 for fp16): |dO_ic| <= 4e-3 + u * sum_j P~_ij |V_jc|.
Without dropout the kernel normalises by the sum of the rounded P it fed to
the MMA, the rounding errors cancel to first order and the plain 4e-3 holds;
with dropout the dropped terms break that cancellation.
Relative Frobenius error is ||G - G_ref|| / ||G_ref||, with the plain norm
of the exact gradient as the denominator.  The one exception is a gradient
that vanishes identically in exact arithmetic: a query row with a single
visible key has dS_i = P_i (dP_i - D_i) = 0 exactly (P_ij = 1 and D_i =
dP_ij), so its dQ row is zero and it adds nothing to dK.  When EVERY checked
row is of that kind (for dQ), or every visible pair feeding the checked key
columns comes from such a row (for dK), the denominator is replaced by a
tenth of the magnitude the gradient would have without that cancellation:
  floor(dQ) = 0.1 tau ||dO||_F rms_j||V_j|| rms_j||K_j||,
  floor(dK) = 0.1 tau ||dO||_F rms_j||V_j|| rms_i||Q_i||,
and the check bounds the absolute error by 1e-2 (1e-5) of that.  Any other
set of rows or columns -- every ordinary head -- gets no floor.  dV never
needs one: dV = P~^T dO has no cancelling sum, and a column no row sees has
dV = 0, where the error itself (exactly zero on the GPU) is checked.
The report carries the plain ratio under ``<name>`` and, under
``<name>_floored``, 1.0 where the floor was the denominator (else 0.0).
For a K/V head shared by g query heads (grouped-query attention) dK and dV
sum over the group, and so do their floors, in quadrature.
"""
from __future__ import annotations

import numpy as np
import torch

from exact_io_aware_tiled_gb300 import workloads as W
import exact_io_aware_tiled_gb300 as fa
from oracle import attention as A

TOL = {
    "f32": dict(o=1e-5, lse=1e-5, grad=1e-5),
    "f16": dict(o=4e-3, lse=1e-3, grad=1e-2),
    "bf16": dict(o=4e-3, lse=1e-3, grad=1e-2),
}
MANT_BITS = {"f16": 10, "bf16": 7, "f32": 23}
UNIT_ROUNDOFF = {"f16": 2.0 ** -11, "bf16": 2.0 ** -8, "f32": 2.0 ** -24}


def half_ulp(x, dtype):
    x = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(x, 1e-30)))
    if dtype == "f16":
        e = np.maximum(e, -14)
    return 0.5 * np.exp2(e - MANT_BITS[dtype])


def spec_of(wl: W.Workload) -> A.Spec:
    return A.Spec(B=wl.B, H=wl.H, N=wl.N, d=wl.d, causal=wl.causal,
                  seqlens_k=None if wl.seqlens is None else np.asarray(wl.seqlens),
                  block_mask=None if wl.block_mask is None else wl.block_mask.astype(bool),
                  block_size=wl.block_size, dropout_p=wl.dropout_p, seed=wl.dropout_seed,
                  offset=wl.dropout_offset, H_kv=wl.H_kv, window=wl.window)


def kwargs_of(wl: W.Workload):
    return dict(causal=wl.causal,
                seqlens_k=None if wl.seqlens is None else torch.from_numpy(np.asarray(wl.seqlens, dtype=np.int32)),
                dropout_p=wl.dropout_p, seed=wl.dropout_seed, offset=wl.dropout_offset,
                block_mask=None if wl.block_mask is None else torch.from_numpy(wl.block_mask.astype(np.uint8)),
                window=wl.window)


def run_gpu(wl: W.Workload, inputs, layout="bhnd", want_o32=True, fwd_kernel=0):
    """fwd + bwd through the C ABI; returns numpy float64 copies of everything.

    fwd_kernel selects the head-dimension-64 forward kernel (0: the library's
    choice, 1: one query tile per CTA, 2: two query tiles per CTA)."""
    dev = torch.device("cuda:0")
    t = {k: v.to(dev) for k, v in inputs.items()}
    if layout == "bnhd":   # non-contiguous strides: [B, N, H, d] memory viewed as [B, H, N, d]
        t = {k: v.transpose(1, 2).contiguous().transpose(1, 2) for k, v in t.items()}
    kw = kwargs_of(wl)
    want_o32 = want_o32 and wl.dtype != "f32"
    out = fa.fwd(t["q"], t["k"], t["v"], return_o_f32=want_o32, fwd_kernel=fwd_kernel, **kw)
    o, lse = out[0], out[1]
    st = fa.check_status(fa.fwd.last_workspace)
    assert st == 0, "fa_fwd device status %d" % st
    res = dict(o=o, lse=lse, o32=out[2] if want_o32 else None)
    if "do" in t:
        dq, dk, dv = fa.bwd(t["q"], t["k"], t["v"], o, t["do"], lse, **kw)
        st = fa.check_status(fa.bwd.last_workspace)
        assert st == 0, "fa_bwd device status %d" % st
        res.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    return res


def _np(x):
    """float64 numpy copy of a (device or host) tensor slice."""
    if isinstance(x, np.ndarray):
        return x.astype(np.float64)
    return x.float().cpu().numpy().astype(np.float64)


def np64(t):
    return t.float().numpy().astype(np.float64)


def rel_frob(a, b, floor=0.0):
    den = max(float(np.linalg.norm(b)), floor)
    return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a - b))


def _rms_row(x):
    return float(np.sqrt(np.mean(np.sum(x * x, axis=1))))


def rows_all_single_key(spec, b, rows, chunk=1024):
    """True iff every query row in ``rows`` sees at most one key.

    Such rows have dS = 0 exactly, so their dQ rows vanish and they add
    nothing to dK.  Stops at the first row that sees two keys."""
    rows = np.asarray(rows, dtype=np.int64)
    allc = np.arange(spec.N)
    for s in range(0, rows.size, chunk):
        if (A.visible(spec, b, rows[s:s + chunk], allc).sum(axis=1) > 1).any():
            return False
    return True


def cols_fed_by_single_key_rows(spec, b, cols, chunk=1024):
    """True iff every query row that sees one of ``cols`` sees only one key,
    i.e. dK of those key columns vanishes in exact arithmetic."""
    cols = np.asarray(cols, dtype=np.int64)
    allr = np.arange(spec.N)
    for s in range(0, spec.N, chunk):
        r = allr[s:s + chunk]
        seen = A.visible(spec, b, r, cols).any(axis=1)
        if seen.any() and not rows_all_single_key(spec, b, r[seen]):
            return False
    return True


def grad_check(report, name, got, ref, floor, tol, vanishes):
    """Record the plain relative error of ``got``; assert it against ``tol``.

    ``vanishes`` says the exact gradient is identically zero; only then is
    the error measured against ``floor`` instead of ||ref||."""
    err = float(np.linalg.norm(got - ref))
    nref = float(np.linalg.norm(ref))
    report[name] = err / nref if nref > 0 else err
    report[name + "_floored"] = 1.0 if vanishes else 0.0
    ok = err <= tol * (max(floor, nref) if vanishes else nref)
    assert ok, (name, report)


def check_head(wl, inputs, got, b, h, rows=None, cols=None, do_grads=True):
    """Compare query head h of batch b (optionally sampled rows / cols) with the oracle.

    O, LSE and dQ are checked for head h.  dK and dV belong to K/V head
    h // g and sum over the g query heads of its group; they are checked when
    h is the last head of its group (every head when g = 1)."""
    spec = spec_of(wl)
    tol = TOL[wl.dtype]
    g = spec.group
    hk = h // g
    q = np64(inputs["q"][b, h])
    k, v = np64(inputs["k"][b, hk]), np64(inputs["v"][b, hk])
    rr = np.arange(wl.N) if rows is None else np.asarray(rows)
    cc = np.arange(wl.N) if cols is None else np.asarray(cols)
    O, L = A.head_forward(spec, b, h, q, k, v, rows=rr)
    report = {}
    rr_t = torch.as_tensor(rr, dtype=torch.long)
    cc_t = torch.as_tensor(cc, dtype=torch.long)
    sel = lambda name, idx: _np(got[name][b, h][idx.to(got[name].device)])
    lse_g = sel("lse", rr_t)
    fin = np.isfinite(L)
    assert np.array_equal(np.isfinite(lse_g), fin), "LSE finiteness differs"
    report["lse"] = float(np.max(np.abs(lse_g[fin] - L[fin]), initial=0.0))
    assert report["lse"] <= tol["lse"], report
    o_g = sel("o", rr_t)
    if wl.dtype == "f32":
        report["o"] = float(np.max(np.abs(o_g - O), initial=0.0))
        assert report["o"] <= tol["o"], report
    else:
        bound = np.full_like(O, tol["o"])
        if wl.dropout_p > 0:
            O_abs, _ = A.head_forward(spec, b, h, q, k, np.abs(v), rows=rr)   # sum_j P~_ij |V_jc|
            bound = bound + UNIT_ROUNDOFF[wl.dtype] * O_abs
        o32 = sel("o32", rr_t)
        report["o32"] = float(np.max(np.abs(o32 - O), initial=0.0))
        report["o32_excess"] = float(np.max(np.abs(o32 - O) - bound, initial=-1.0))
        assert report["o32_excess"] <= 0.0, report
        excess = np.abs(o_g - O) - (bound + half_ulp(O, wl.dtype))
        report["o_stored_excess"] = float(np.max(excess, initial=-1.0))
        assert report["o_stored_excess"] <= 0.0, report
    if do_grads and "dq" in got:
        do = np64(inputs["do"][b, h])
        gr = A.head_backward(spec, b, h, q, k, v, do, rows=rr, cols=cc)
        ndo = float(np.linalg.norm(do))
        fl = 0.1 * spec.tau * ndo * _rms_row(v) * _rms_row(k)
        grad_check(report, "dq", sel("dq", rr_t), gr["dq"], fl, tol["grad"],
                   rows_all_single_key(spec, b, rr))
        if h % g == g - 1:
            dk_ref, dv_ref = np.zeros((cc.size, spec.d)), np.zeros((cc.size, spec.d))
            fk2 = 0.0
            for hq in range(hk * g, hk * g + g):
                qh, doh = np64(inputs["q"][b, hq]), np64(inputs["do"][b, hq])
                gh = gr if hq == h else A.head_backward(spec, b, hq, qh, k, v, doh, rows=np.arange(0), cols=cc)
                dk_ref += gh["dk"]
                dv_ref += gh["dv"]
                nd = float(np.linalg.norm(doh))
                fk2 += (0.1 * spec.tau * nd * _rms_row(v) * _rms_row(qh)) ** 2
            sel_kv = lambda name: _np(got[name][b, hk][cc_t.to(got[name].device)])
            grad_check(report, "dk", sel_kv("dk"), dk_ref, fk2 ** 0.5, tol["grad"],
                       cols_fed_by_single_key_rows(spec, b, cc))
            grad_check(report, "dv", sel_kv("dv"), dv_ref, 0.0, tol["grad"], False)
    return report


def sample_rows(N, seed, extra=256):
    rng = np.random.default_rng(seed)
    s = set(range(min(128, N))) | set(range(max(0, N - 128), N))
    for t in range(128, N, 128):
        s |= {t - 1, t}
        if t + 1 < N:
            s.add(t + 1)
    s |= set(rng.integers(0, N, size=min(extra, N)).tolist())
    return np.array(sorted(s))
