"""Pins of the FP8 forward oracle (oracle/fp8.py) against the E4M3 format,
torch's float8_e4m3fn, the Sylvester construction, exact attention and the
pages' claim that block scales with a random rotation beat one scale per
tensor (living-dl-book, section 10; marketmaker.cc, "FA3: Mecanica da
tremonha", item 3)."""
import numpy as np
import pytest
import torch

from exact_io_aware_tiled_gb300 import workloads as W
from oracle import attention as A
from oracle import fp8 as F


def _torch_encode(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_decode_matches_format_and_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = F.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ours)
    assert np.array_equal(ours[fin], ref[fin])
    assert np.isnan(ours[0x7F]) and np.isnan(ours[0xFF]) and np.isnan(ours).sum() == 2
    assert ours[0x7E] == 448.0 and ours[0xFE] == -448.0
    assert ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6 and ours[0x07] == 7 * 2.0 ** -9
    assert ours[0x38] == 1.0 and ours[0x00] == 0.0 and np.signbit(ours[0x80])


def test_e4m3_encode_matches_torch_cast():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(100_000) * np.exp2(rng.uniform(-14, 9, 100_000))).astype(np.float32)
    x = np.clip(x, -448, 448)
    assert np.array_equal(F.e4m3_encode(x), _torch_encode(x))
    # every midpoint between neighbouring finite values: ties go to the even code
    vals = np.unique(F.e4m3_decode(np.arange(0x7F, dtype=np.uint8)))
    mid = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    got = F.e4m3_encode(mid)
    assert np.array_equal(got, _torch_encode(mid))
    assert np.all(got % 2 == 0)
    assert np.array_equal(F.e4m3_encode(-mid), got | 0x80)
    # saturation at the largest finite value (the kernel's satfinite conversion)
    assert np.all(F.e4m3_encode(np.array([448.0, 460.0, 470.0, 1e4, 1e30])) == 0x7E)
    assert np.all(F.e4m3_encode(np.array([-470.0, -1e30])) == 0xFE)
    assert F.e4m3_encode(np.array([np.nan]))[0] & 0x7F == 0x7F


@pytest.mark.parametrize("d", [2, 8, 64, 128])
def test_fwht_equals_sylvester_product(d):
    scipy_linalg = pytest.importorskip("scipy.linalg")
    H = F.sylvester(d)
    assert np.array_equal(H, scipy_linalg.hadamard(d))
    rng = np.random.default_rng(d)
    xi = rng.integers(-50, 50, size=(7, d)).astype(np.float32)          # exact in float32
    assert np.array_equal(F.fwht_f32(xi).astype(np.float64), xi.astype(np.float64) @ H)
    x = rng.standard_normal((7, d)).astype(np.float32)
    err = np.abs(F.fwht_f32(x) - x.astype(np.float64) @ H).max()
    assert err < 1e-5 * np.sqrt(d) * np.abs(x).max()


def test_rotation_is_orthogonal_and_keeps_the_scores():
    s = W.rotation_signs(64, 5)
    assert set(np.unique(s)) <= {-1, 1}
    M = F.rotation_matrix(s)
    assert np.abs(M @ M.T - np.eye(64)).max() < 1e-14
    rng = np.random.default_rng(0)
    q, k = rng.standard_normal((2, 40, 64))
    assert np.abs((q @ M) @ (k @ M).T - q @ k.T).max() < 1e-12
    x = rng.standard_normal((9, 64)).astype(np.float32)
    assert np.abs(F.rotate_rows_f32(x, s) - x.astype(np.float64) @ M).max() < 1e-5
    assert np.abs(F.unrotate_rows(x.astype(np.float64) @ M, s) - x).max() < 1e-12


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("rotate", [False, True])
def test_quantize_block_properties(rotate, d):
    wl = W.Workload("q", B=2, H=3, N=300, d=d, seed=11)
    x = W.make_inputs(wl, grads=False)["q"].float().numpy()
    x[1, 2, 128:256] = 0.0                                              # an all-zero block
    s = W.rotation_signs(d, 1) if rotate else None
    codes, scale = F.quantize(x, s)
    assert codes.shape == x.shape and scale.shape == (2, 3, 3) and scale.dtype == np.float32
    assert scale[1, 2, 1] == 0 and not codes[1, 2, 128:256].any()
    xr = F.rotate_rows_f32(x, s) if rotate else x.astype(np.float32)
    dq = F.dequantize(codes, scale)
    for b in range(2):
        for h in range(3):
            for t in range(3):
                blk = codes[b, h, t * 128:(t + 1) * 128]
                if scale[b, h, t] == 0:
                    continue
                assert (blk & 0x7F).max() == 0x7E                       # the block max lands on 448
                ref = xr[b, h, t * 128:(t + 1) * 128].astype(np.float64)
                got = dq[b, h, t * 128:(t + 1) * 128]
                sc = float(scale[b, h, t])
                # half an ulp: 2^-4 relative in the normal range, 2^-10 * scale below it
                assert np.all(np.abs(got - ref) <= np.maximum(2.0 ** -4 * np.abs(ref), 2.0 ** -10 * sc) * (1 + 1e-6))
    c_t, s_t = F.quantize(x, s, per_tensor=True)
    assert np.all(s_t == s_t.flat[0]) and s_t.flat[0] == np.float32(np.abs(xr).max()) / np.float32(448)
    vt = F.transpose_v(codes)
    assert vt.shape == (2, 3, d, 384) and not vt[..., 300:].any()
    assert np.array_equal(vt[0, 1, :, :300], codes[0, 1].T)


def _spec(wl):
    return A.Spec(B=wl.B, H=wl.H, N=wl.N, d=wl.d, causal=wl.causal, window=wl.window, H_kv=wl.H_kv,
                  seqlens_k=wl.seqlens, block_mask=None if wl.block_mask is None else wl.block_mask.astype(bool))


@pytest.mark.parametrize("kw", [dict(causal=True), dict(causal=True, window=100, seqlen_range=(150, 300)),
                                dict(H_kv=1, sparse_butterfly=True)])
def test_gate_is_exact_attention_of_the_dequantised_inputs(kw):
    wl = W.Workload("u", B=2, H=2, N=300, seed=17, **kw)
    inp = W.make_inputs(wl, grads=False)
    q, k, v = (inp[n].float().numpy() for n in ("q", "k", "v"))
    s = W.rotation_signs(64, 2)
    spec = _spec(wl)
    O, L, worst, var, qz = F.attention_fwd(spec, q, k, v, signs=s)
    back = {n: F.unrotate_rows(F.dequantize(qz[n + "8"], qz["s" + n]), s) for n in ("q", "k", "v")}
    Oe, Le = A.attention_fwd(spec, back["q"], back["k"], back["v"])
    assert np.abs(O - Oe).max() < 1e-10
    fin = np.isfinite(Le)
    assert np.array_equal(fin, np.isfinite(L)) and np.abs(L[fin] - Le[fin]).max() < 1e-10
    assert (worst >= 0).all() and (var >= 0).all() and (var <= worst * worst / 3 + 1e-30).all()
    # the diagnostic model with its rounding switched off is the same attention
    Om, Lm, _ = F.scaled_p_model_attention_fwd(spec, q, k, v, signs=s, round_p=False)
    assert np.abs(Om - Oe).max() < 1e-10
    assert np.abs(Lm[fin] - Le[fin]).max() < 1e-10


def _round_p_simulation(spec, q8, sq, k8, sk, v8, sv, signs, running=False, mant_bits=3, scale_err=0.0,
                        unrotate=True):
    """An implementation written here, apart from the oracle: round
    exp(S - m) in (0, 1] to a float with ``mant_bits`` mantissa bits
    (torch's float8_e4m3fn cast for 3), m the final row max or the running
    max over 128-key tiles, normalise by the unrounded row sum."""
    N, d = q8.shape
    qd, kd, vd = F.dequantize(q8, sq), F.dequantize(k8, sk), F.dequantize(v8, sv)
    vis = A.visible(spec, 0, np.arange(N), np.arange(N))
    S = np.where(vis, spec.tau * (qd @ kd.T), -np.inf)
    if running:
        m = np.concatenate([np.maximum.accumulate(
            np.stack([S[:, t:t + 128].max(axis=1) for t in range(0, N, 128)], axis=1), axis=1)[:, t // 128:t // 128 + 1]
            .repeat(min(128, N - t), axis=1) for t in range(0, N, 128)], axis=1)
    else:
        m = S.max(axis=1, keepdims=True).repeat(N, axis=1)
    mf = S.max(axis=1, keepdims=True)
    E = np.exp(S - m)                                   # in (0, 1], 0 where masked
    if mant_bits == 3:
        Er = torch.from_numpy(E.astype(np.float32)).to(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    else:
        mant, ex = np.frexp(E)
        Er = np.ldexp(np.round(mant * 2.0 ** (mant_bits + 1)) / 2.0 ** (mant_bits + 1), ex)
    ell = np.exp(S - mf).sum(axis=1, keepdims=True)
    W_ = Er * np.exp(m - mf) / ell
    Orot = W_ @ vd * (1.0 + scale_err)
    return F.unrotate_rows(Orot, signs) if (signs is not None and unrotate) else Orot


@pytest.mark.parametrize("running", [False, True])
@pytest.mark.parametrize("rotate", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_independent_fp8_rounding_of_p_stays_inside_both_bounds(running, rotate, d):
    wl = W.Workload("b", B=1, H=1, N=640, d=d, seed=31 + d, causal=True)
    inp = W.make_inputs(wl, grads=False)
    s = W.rotation_signs(d, 4) if rotate else None
    qz = {n: F.quantize(inp[n].float().numpy(), s) for n in ("q", "k", "v")}
    args = (qz["q"][0][0, 0], qz["q"][1][0, 0], qz["k"][0][0, 0], qz["k"][1][0, 0], qz["v"][0][0, 0], qz["v"][1][0, 0])
    spec = _spec(wl)
    O, L, worst, var = F.head_forward(spec, 0, 0, *args, signs=s)
    Osim = _round_p_simulation(spec, *args, s, running=running)
    err = np.abs(Osim - O)
    assert (err <= worst * (1 + 1e-9) + 1e-12).all()
    rms, rms_bound = np.sqrt(np.mean(err ** 2)), np.sqrt(np.mean(var))
    assert rms <= rms_bound, (rms, rms_bound)
    assert rms > 0.3 * rms_bound                      # the bound is not vacuous
    # planted mistakes of an implementation: a coarser (2-bit) mantissa, a
    # 10 % scale error, a missing back-rotation -- each breaks a bound
    coarse = np.sqrt(np.mean((_round_p_simulation(spec, *args, s, running=running, mant_bits=2) - O) ** 2))
    assert coarse > rms_bound
    scaled = _round_p_simulation(spec, *args, s, running=running, scale_err=0.1)
    assert np.sqrt(np.mean((scaled - O) ** 2)) > rms_bound
    if rotate:
        assert (np.abs(_round_p_simulation(spec, *args, s, running=running, unrotate=False) - O) > worst).any()


def test_equal_scores_give_the_mean_of_the_dequantised_values():
    # Q = 0: every visible score is 0, every probability 1 (exact in E4M3),
    # so O_i is the mean of the visible dequantised V rows (causal: rows
    # 0..i) and the rounding bounds are only the subnormal floor's.  The
    # diagnostic model with one scale per tensor (c_t = 256 exactly) agrees.
    wl = W.Workload("e", B=1, H=1, N=300, seed=23, causal=True)
    inp = W.make_inputs(wl, grads=False)
    q = np.zeros((1, 1, 300, 64), dtype=np.float32)
    k, v = (inp[n].float().numpy() for n in ("k", "v"))
    s = W.rotation_signs(64, 3)
    spec = A.Spec(B=1, H=1, N=300, d=64, causal=True)
    O, L, worst, var, qz = F.attention_fwd(spec, q, k, v, signs=s, per_tensor=True)
    vhat = F.unrotate_rows(F.dequantize(qz["v8"], qz["sv"])[0, 0], s)
    mean = np.cumsum(vhat, axis=0) / np.arange(1, 301)[:, None]
    assert np.abs(O[0, 0] - mean).max() < 1e-12
    assert np.abs(L[0, 0] - np.log(np.arange(1, 301))).max() < 1e-12
    Om, Lm, _ = F.scaled_p_model_attention_fwd(spec, q, k, v, signs=s, per_tensor=True)
    assert np.abs(Om[0, 0] - mean).max() < 1e-12
    assert np.abs(Lm[0, 0] - np.log(np.arange(1, 301))).max() < 1e-12


def test_block_scales_with_rotation_beat_one_scale_per_tensor_with_outliers():
    wl = W.Workload("o", B=1, H=2, N=512, seed=20270, outlier_rate=1e-3, outlier_sd=10.0)
    inp = W.make_inputs(wl, grads=False)
    q, k, v = (inp[n].float().numpy() for n in ("q", "k", "v"))
    spec = A.Spec(B=1, H=2, N=512, d=64)
    exact, _ = A.attention_fwd(spec, q, k, v)
    s = W.rotation_signs(64, wl.seed)
    # the error of quantising Q, K and V alone (the gate) and with the
    # probabilities rounded too (the diagnostic model)
    e_tensor = F.relative_error(F.attention_fwd(spec, q, k, v, per_tensor=True)[0], exact)
    e_block_rot = F.relative_error(F.attention_fwd(spec, q, k, v, signs=s)[0], exact)
    assert e_tensor / e_block_rot > 1.3, (e_tensor, e_block_rot)
    m_tensor = F.relative_error(F.scaled_p_model_attention_fwd(spec, q, k, v, per_tensor=True)[0], exact)
    m_block_rot = F.relative_error(F.scaled_p_model_attention_fwd(spec, q, k, v, signs=s)[0], exact)
    assert m_tensor / m_block_rot > 1.3, (m_tensor, m_block_rot)
    assert m_block_rot < 0.1


def test_model_rounds_probabilities_against_the_running_max():
    # Row 0 sees key tile 0 with every score 0 and key tile 1 with every score
    # equal to 3 (no rotation, equal V block scales, so c_t = 256).  Against
    # the running max each tile's probabilities are exactly 1 when rounded,
    # so the diagnostic model equals exact attention of the dequantised
    # inputs; rounding against the final max would round exp(-3) * 256
    # inexactly.
    N, d = 256, 64
    q = np.zeros((1, 1, N, d), dtype=np.float32)
    k = np.zeros((1, 1, N, d), dtype=np.float32)
    q[0, 0, :, 0] = 24.0                  # tau * 24 * 1 = 3 with tau = 1/8
    k[0, 0, 128:, 0] = 1.0
    rng = np.random.default_rng(5)
    v = rng.standard_normal((1, 1, N, d)).astype(np.float32)
    v[0, 0, 0, 0] = v[0, 0, 128, 0] = 4.0  # both V blocks have amax 4: equal scales
    v = np.clip(v, -3.9, 3.9)
    v[0, 0, 0, 0] = v[0, 0, 128, 0] = 4.0
    spec = A.Spec(B=1, H=1, N=N, d=d)
    O, L, qz = F.scaled_p_model_attention_fwd(spec, q, k, v)
    assert qz["sv"][0, 0, 0] == qz["sv"][0, 0, 1]
    back = {n: F.dequantize(qz[n + "8"], qz["s" + n]) for n in ("q", "k", "v")}
    Oe, Le = A.attention_fwd(spec, back["q"], back["k"], back["v"])
    assert np.abs(O - Oe).max() < 1e-12
    assert np.abs(L - Le).max() < 1e-12
