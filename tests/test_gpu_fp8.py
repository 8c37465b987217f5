"""GPU parity of the FP8 forward (fa_fp8_quantize + fa_fwd_fp8) against oracle/fp8.py.

What is compared, and how closely:
  * the quantiser decides integer codes, in float32 and in the same order on
    both sides, so its E4M3 codes (Q, K and the transposed V) and its float32
    scales must be bit-identical to the oracle's;
  * the forward is compared with exact attention (float64) of the
    dequantised inputs, rotated back (``oracle.fp8.head_forward``).  The
    difference the kernel may add is that of rounding the probabilities to
    E4M3 (living-dl-book, section 10: both products run in FP8), bounded
    from the format alone (the oracle's reading R6): per element by
    sum_j b_ij |V'_jc| with b_ij = max(2^-4 P_ij, 2^-10 / l_i), and in
    root-mean-square over a head by sqrt(mean(sum_j b_ij^2 V'_jc^2 / 3)).
    On top of both, ACC_TOL / ACC_RMS cover float32 against float64
    arithmetic elsewhere (the tensor-core sums, the exponentials, the row
    sum, the rotation back).  The stored 16-bit O gets half an ulp of the
    storage type more; the logsumexp, computed from the unrounded
    probabilities, must agree within 1e-3 (the 16-bit path's bound);
  * the error study: block scales with the rotation must beat one scale per
    tensor on the kernel's own output, as the pages report (living-dl-book,
    section 10; marketmaker.cc, "FA3", item 3).
The oracle's model of the kernel's own scaling of P
(``scaled_p_model_forward``) is reported beside these numbers as a
diagnostic; no assertion uses it.
"""
import numpy as np
import pytest
import torch

import exact_io_aware_tiled_gb300 as fa
from exact_io_aware_tiled_gb300 import workloads as W
from oracle import attention as A
from oracle import fp8 as F
from tests.parity import half_ulp, kwargs_of, sample_rows, spec_of

pytestmark = pytest.mark.gpu

ACC_TOL = 1e-3
ACC_RMS = 1e-4
LSE_TOL = 1e-3


def run_fp8(wl, inp, signs, per_tensor=False, layout="bhnd"):
    dev = torch.device("cuda:0")
    t = {k: v.to(dev) for k, v in inp.items() if k in ("q", "k", "v")}
    if layout == "bnhd":
        t = {k: v.transpose(1, 2).contiguous().transpose(1, 2) for k, v in t.items()}
    kw = kwargs_of(wl)
    kw.pop("dropout_p"), kw.pop("seed"), kw.pop("offset")
    o, lse, o32, views = fa.fwd_fp8(t["q"], t["k"], t["v"], signs=signs, per_tensor=per_tensor,
                                    return_o_f32=True, return_quantized=True, **kw)
    st = fa.check_status(fa.fwd_fp8.last_workspace)
    assert st == 0, "fa_fwd_fp8 device status %d" % st
    torch.cuda.synchronize()
    return dict(o=o, lse=lse, o32=o32, **{k: v.cpu().numpy() for k, v in views.items()})


def oracle_quantized(inp, signs, per_tensor=False, heads=None):
    """The oracle's codes and scales of q, k, v (optionally of heads (b, h) only)."""
    out = {}
    for n in ("q", "k", "v"):
        x = inp[n].float().numpy()
        if heads is not None:
            x = x[heads[0]:heads[0] + 1, heads[1]:heads[1] + 1]
        out[n + "8"], out["s" + n] = F.quantize(x, signs, per_tensor)
    return out


def assert_codes_equal(got, ref, b=None, h=None, hk=None):
    sl = (lambda a, hh: a) if b is None else (lambda a, hh: a[b:b + 1, hh:hh + 1])
    assert np.array_equal(sl(got["q8"], h), ref["q8"]), "Q codes differ"
    assert np.array_equal(sl(got["k8"], hk), ref["k8"]), "K codes differ"
    assert np.array_equal(sl(got["v8t"], hk), F.transpose_v(ref["v8"])), "V codes differ"
    for n, hh in (("sq", h), ("sk", hk), ("sv", hk)):
        assert np.array_equal(sl(got[n], hh), ref[n]), n + " differs"


def check_fp8_head(wl, got, qz, b, h, signs, rows=None, qb=None):
    """O / LSE of query head (b, h) against exact attention of its dequantised inputs.

    qz holds the oracle's codes of the whole problem (indexed by b, head), or
    of this head only when qb = (b, h, hk) says which head it is."""
    spec = spec_of(wl)
    hk = h // spec.group
    ib, ih, ik = (b, h, hk) if qb is None else (0, 0, 0)
    rr = np.arange(wl.N) if rows is None else np.asarray(rows)
    args = (qz["q8"][ib, ih], qz["sq"][ib, ih], qz["k8"][ib, ik], qz["sk"][ib, ik], qz["v8"][ib, ik], qz["sv"][ib, ik])
    O, L, worst, var = F.head_forward(spec, b, h, *args, signs, rows=rr)
    idx = torch.as_tensor(rr, dtype=torch.long)
    sel = lambda name: got[name][b, h][idx.to(got[name].device)].float().cpu().numpy().astype(np.float64)
    lse = sel("lse")
    fin = np.isfinite(L)
    assert np.array_equal(np.isfinite(lse), fin), "LSE finiteness differs"
    rep = {"lse": float(np.max(np.abs(lse[fin] - L[fin]), initial=0.0))}
    assert rep["lse"] <= LSE_TOL, rep
    o32 = sel("o32")
    err = np.abs(o32 - O)
    rep["o32"] = float(np.max(err, initial=0.0))
    rep["o32_excess"] = float(np.max(err - (worst + ACC_TOL), initial=-1.0))
    assert rep["o32_excess"] <= 0.0, rep
    rep["rms"] = float(np.sqrt(np.mean(err ** 2))) if err.size else 0.0
    rep["rms_bound"] = float(np.sqrt(np.mean(var))) if var.size else 0.0
    assert rep["rms"] <= rep["rms_bound"] + ACC_RMS, rep
    o = sel("o")
    rep["o_stored_excess"] = float(np.max(np.abs(o - O) - (worst + ACC_TOL + half_ulp(O, wl.dtype)), initial=-1.0))
    assert rep["o_stored_excess"] <= 0.0, rep
    # diagnostic only: the model of the kernel's own scaling of P
    Om, _ = F.scaled_p_model_forward(spec, b, h, *args, signs, rows=rr)
    rep["model_p99"] = float(np.quantile(np.abs(o32 - Om), 0.99)) if Om.size else 0.0
    return rep


CASES = {
    "causal_bf16": dict(B=1, H=2, N=300, dtype="bf16", causal=True, seed=801),
    "dense_f16_ragged": dict(B=2, H=2, N=200, dtype="f16", seed=802),
    "padding_window": dict(B=2, H=2, N=520, dtype="bf16", causal=True, window=200, seqlen_range=(100, 520),
                           seed=803),
    "gqa_sparse": dict(B=1, H=4, H_kv=2, N=640, dtype="bf16", sparse_butterfly=True, seed=804),
    "single_tile": dict(B=1, H=1, N=64, dtype="bf16", causal=True, seed=805),
    # head dimension 128 (FlashAttention-3's FP8 setting)
    "d128_causal_bf16": dict(B=1, H=2, N=300, d=128, dtype="bf16", causal=True, seed=808),
    "d128_gqa_padding_f16": dict(B=2, H=4, H_kv=2, N=400, d=128, dtype="f16", seqlen_range=(150, 400), seed=809),
    "d128_window_sparse": dict(B=1, H=2, N=520, d=128, dtype="bf16", causal=True, window=300,
                               sparse_butterfly=True, seed=810),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("rotate", [True, False])
def test_fp8_forward_matches_oracle(name, rotate):
    wl = W.Workload(name, **CASES[name])
    inp = W.make_inputs(wl, grads=False)
    signs = W.rotation_signs(wl.d, wl.seed) if rotate else None
    got = run_fp8(wl, inp, signs)
    qz = oracle_quantized(inp, signs)
    assert_codes_equal(got, qz)
    reps = [check_fp8_head(wl, got, qz, b, h, signs) for b in range(wl.B) for h in range(wl.H)]
    print(name, rotate, [{k: ("%.2e" % v) for k, v in r.items()} for r in reps])


@pytest.mark.parametrize("rotate", [True, False])
def test_fp8_per_tensor_scales(rotate):
    wl = W.Workload("pt", B=2, H=2, N=384, dtype="bf16", causal=True, seed=806, outlier_rate=1e-3, outlier_sd=10.0)
    inp = W.make_inputs(wl, grads=False)
    signs = W.rotation_signs(64, wl.seed) if rotate else None
    got = run_fp8(wl, inp, signs, per_tensor=True)
    qz = oracle_quantized(inp, signs, per_tensor=True)
    assert_codes_equal(got, qz)
    for n in ("sq", "sk", "sv"):
        assert np.all(got[n] == got[n].flat[0])
    for b in range(wl.B):
        for h in range(wl.H):
            check_fp8_head(wl, got, qz, b, h, signs)


def test_fp8_non_contiguous_layout_and_zero_blocks():
    wl = W.Workload("nc", B=2, H=2, N=256, dtype="bf16", causal=True, seed=807)
    inp = W.make_inputs(wl, grads=False)
    inp["q"][1, 0, :128] = 0          # an all-zero Q tile: scale 0, every score 0
    inp["k"][0, 1, 128:] = 0          # an all-zero K tile
    inp["v"][1, 1] = 0                # a whole V head of zeros: SV = 0, O = 0
    signs = W.rotation_signs(64, wl.seed)
    got = run_fp8(wl, inp, signs, layout="bnhd")
    qz = oracle_quantized(inp, signs)
    assert_codes_equal(got, qz)
    assert got["sq"][1, 0, 0] == 0 and got["sv"][1, 1].max() == 0
    for b in range(wl.B):
        for h in range(wl.H):
            check_fp8_head(wl, got, qz, b, h, signs)
    assert not got["o"][1, 1].any()


def test_fp8_error_study_block_rotation_beats_per_tensor():
    wl = W.Workload("study", B=1, H=2, N=1024, dtype="bf16", seed=20270, outlier_rate=1e-3, outlier_sd=10.0)
    inp = W.make_inputs(wl, grads=False)
    q, k, v = (inp[n].float().numpy() for n in ("q", "k", "v"))
    spec = spec_of(wl)
    exact, _ = A.attention_fwd(spec, q, k, v)
    signs = W.rotation_signs(64, wl.seed)
    errs = {}
    for name, sg, pt in (("per_tensor", None, True), ("block_rotated", signs, False)):
        got = run_fp8(wl, inp, sg, per_tensor=pt)
        O_in, _, _, var, _ = F.attention_fwd(spec, q, k, v, signs=sg, per_tensor=pt)
        o32 = got["o32"].float().cpu().numpy()
        e_gpu = F.relative_error(o32, exact)
        # by the triangle inequality on RMS: |e_gpu - e_in| <= the P rounding
        # bound (relative) plus the float32 slack
        e_in = F.relative_error(O_in, exact)
        rms_exact = float(np.sqrt(np.mean(exact ** 2)))
        e_p = (float(np.sqrt(np.mean(var))) + ACC_RMS) / rms_exact
        assert abs(e_gpu - e_in) <= e_p, (name, e_gpu, e_in, e_p)
        e_model = F.relative_error(F.scaled_p_model_attention_fwd(spec, q, k, v, signs=sg, per_tensor=pt)[0], exact)
        print("error study %s: kernel %.4f, Q/K/V quantisation alone %.4f, P-rounding bound %.4f, model %.4f"
              % (name, e_gpu, e_in, e_p, e_model))
        errs[name] = e_gpu
    assert errs["per_tensor"] / errs["block_rotated"] > 1.3, errs


def test_fp8_gpt2_medium_causal_sampled():
    wl = W.CONFIGS["gpt2_medium_causal_fp8"]
    inp = W.make_inputs(wl, grads=False)
    signs = W.rotation_signs(64, wl.seed)
    got = run_fp8(wl, inp, signs)
    rows = sample_rows(wl.N, seed=8, extra=64)
    for b, h in ((0, 0), (wl.B - 1, wl.H - 1), (17, 5)):
        qz = oracle_quantized(inp, signs, heads=(b, h))
        assert_codes_equal(got, qz, b=b, h=h, hk=h)
        check_fp8_head(wl, got, qz, b, h, signs, rows=rows, qb=(b, h, h))


@pytest.mark.parametrize("name", ["gpt2_medium_d128_causal_fp8"])
def test_fp8_d128_full_size_sampled(name):
    wl = W.CONFIGS[name]
    inp = W.make_inputs(wl, grads=False)
    signs = W.rotation_signs(wl.d, wl.seed)
    got = run_fp8(wl, inp, signs)
    rows = sample_rows(wl.N, seed=9, extra=64)
    for b, h in ((0, 0), (wl.B - 1, wl.H - 1), (33, 3)):
        qz = oracle_quantized(inp, signs, heads=(b, h))
        assert_codes_equal(got, qz, b=b, h=h, hk=h)
        check_fp8_head(wl, got, qz, b, h, signs, rows=rows, qb=(b, h, h))


def test_fp8_refuses_float32_and_other_head_dims():
    q = torch.zeros((1, 1, 128, 64), device="cuda", dtype=torch.float32)
    with pytest.raises(fa.FAError) as e:
        fa.fwd_fp8(q, q, q)
    assert e.value.code == 2
    q = torch.zeros((1, 1, 128, 96), device="cuda", dtype=torch.bfloat16)
    with pytest.raises(fa.FAError) as e:
        fa.fwd_fp8(q, q, q)
    assert e.value.code == 2
