"""FP8 forward attention with block quantisation and incoherent processing.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).

What the pages say (living-dl-book, "Atencao Eficiente em Escala", section
10 on FlashAttention-3; marketmaker.cc, "FA3: Mecanica da tremonha", item 3):
Q, K and V are quantised to FP8 block by block, one scale factor per tile,
after a randomised Hadamard-style orthogonal rotation of every vector that
spreads an outlying coordinate over all coordinates.  The rotation is
invertible and is undone after the matmul, so the result is exact up to the
FP8 rounding.  The pages report 2.6x less error than FP8 with one scale per
tensor.

The pages leave the details open; the readings taken here:

R1  FP8 is E4M3 in its finite ("fn") form: 1 sign bit, 4 exponent bits with
    bias 7, 3 mantissa bits, no infinities, S.1111.111 is NaN, largest
    finite 448, subnormals down to 2^-9.  Rounding is to nearest, ties to
    even, saturating at +-448 (``e4m3_encode``).
R2  The rotation is M = diag(s) H_d / sqrt(d): H_d the Sylvester Hadamard
    matrix (H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]]) and s a vector of
    random signs, which is an input.  Rows are rotated: x' = x M.
R3  Q, K and V are all rotated.  Q'K'^T = Q M M^T K^T = Q K^T, so the scores
    need no undo; the output is rotated back, O = O' M^T
    (= (O' H_d) o s / sqrt(d)).
R4  A block is 128 rows x d of one head (the kernel's tile).  Its scale is
    amax / 448 and its codes are E4M3(x' * (448 / amax)); an all-zero block
    has scale 0 and codes 0.
R5  The per-tensor baseline has one scale for a whole tensor ([B, H, N, d])
    and no rotation.
R6  P is quantised too, as FlashAttention-3 does for its second product;
    the pages do not say on which scale.  The plainest reading rounds the
    unnormalised probabilities exp(S - m) in (0, 1] (m a running row max
    no larger than the final one) to E4M3 directly: a relative error of at
    most 2^-4 (half of the 3-bit mantissa's spacing) in the normal range and
    at most 2^-10 absolute below 2^-6.  Normalised by the unrounded row sum
    l_i = sum_j exp(S_ij - m_i) >= 1, the weight of key j then errs by
        b_ij = max(2^-4 P_ij, 2^-10 / l_i).
    An implementation that rounds on a grid at least as fine (a larger
    scale before the rounding) stays inside the same bound.  The gate
    (``head_forward``) is therefore exact attention of the dequantised,
    rotated inputs, rotated back, with two bounds on the difference:
      worst case   |dO_ic| <= sum_j b_ij |V'_jc|;
      RMS          E[dO_ic^2] <= sum_j b_ij^2 V'_jc^2 / 3
                   (a rounding error with spacing s has variance s^2 / 12,
                   and s <= 2 b_ij);
    where V' is in the output's coordinates: the rows of the dequantised,
    rotated V multiplied back by M^T (an error in key j's weight moves the
    whole row, so this is exact under the rotation).  One particular scaling of
    P (the GPU kernel's) is written out in ``scaled_p_model_forward`` as a
    diagnostic only; no test gates on it.
R7  The quantiser decides integer codes from floating-point values, so it
    works in float32 in a fixed order, as the kernel does: the sign flip,
    the fast Walsh-Hadamard butterflies (stage h = 1, 2, ..., d/2 pairs
    i and i + h, giving a + b and a - b), one multiply by the float32 value
    of 1/sqrt(d), the block's amax, inv = 448 / amax (one float32 division),
    x' * inv (one float32 multiply), then E4M3 rounding.  Only the quantiser
    has this property: the attention that follows is compared by tolerance.

Pinned by tests/test_oracle_fp8.py: every E4M3 code decodes as the format
defines and agrees with torch's float8_e4m3fn; rounding agrees with torch's
cast on random values and on exact midpoints; the butterflies equal the
Sylvester matrix product; M is orthogonal and the scores survive the
rotation; each nonzero block's largest code is 448; the gate equals exact
attention (oracle.attention) of the dequantised inputs rotated back; an
independent simulation that rounds exp(S - m) to E4M3 (final or running
max) stays inside both bounds of R6, while a coarser rounding or a 1 %
scale error breaks them; equal scores return the mean of the dequantised
V; and with outliers in the inputs, block scales with the rotation give
less error than one scale per tensor.
"""
from __future__ import annotations

import numpy as np

from . import attention as _attn

E4M3_MAX = 448.0
TILE = 128


# ----------------------------------------------------------------------------
# E4M3 (R1)
# ----------------------------------------------------------------------------
def e4m3_decode(codes) -> np.ndarray:
    """float64 value of each E4M3 byte (NaN for S.1111.111)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def e4m3_encode(x) -> np.ndarray:
    """E4M3 byte of each value: round to nearest, ties to even, saturating to +-448."""
    x = np.asarray(x, dtype=np.float64)
    sign = np.where(np.signbit(x), 0x80, 0).astype(np.int64)
    a = np.abs(x)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, np.minimum(a, 2.0 * E4M3_MAX))
    # subnormal range (and zero): multiples of 2^-9 below 2^-6
    sub = a < 2.0 ** -6
    code_sub = np.rint(a * 2.0 ** 9).astype(np.int64)          # 0..8; 8 is 2^-6 (E=1, M=0)
    # normal range: a = 2^e (1 + f), e from the binary exponent
    mant, ex = np.frexp(np.where(sub, 1.0, a))                  # a = mant * 2^ex, mant in [0.5, 1)
    e = ex - 1
    mm = np.rint((mant * 2.0 - 1.0) * 8.0).astype(np.int64)     # 0..8, ties to even
    e = np.where(mm == 8, e + 1, e)
    mm = np.where(mm == 8, 0, mm)
    code_norm = ((e + 7) << 3) | mm
    code = np.where(sub, code_sub, code_norm)
    code = np.minimum(code, 0x7E)                               # saturate at 448 (0x7F is NaN)
    code = np.where(nan, 0x7F, code)
    return (code | sign).astype(np.uint8)


def e4m3_round(x) -> np.ndarray:
    return e4m3_decode(e4m3_encode(x))


# ----------------------------------------------------------------------------
# rotation (R2, R7)
# ----------------------------------------------------------------------------
def sylvester(d: int) -> np.ndarray:
    """H_d by the Sylvester recursion (d a power of two)."""
    H = np.ones((1, 1))
    while H.shape[0] < d:
        H = np.block([[H, H], [H, -H]])
    assert H.shape[0] == d, "d must be a power of two"
    return H


def rotation_matrix(signs) -> np.ndarray:
    """M = diag(s) H_d / sqrt(d) in float64."""
    s = np.asarray(signs, dtype=np.float64)
    d = s.size
    return (s[:, None] * sylvester(d)) / np.sqrt(d)


def fwht_f32(x) -> np.ndarray:
    """x H_d along the last axis by the butterfly stages, in float32 (R7)."""
    y = np.array(x, dtype=np.float32, copy=True)
    d = y.shape[-1]
    h = 1
    while h < d:
        z = y.reshape(y.shape[:-1] + (d // (2 * h), 2, h))
        a = z[..., 0, :].copy()
        b = z[..., 1, :].copy()
        z[..., 0, :] = a + b
        z[..., 1, :] = a - b
        y = z.reshape(y.shape)
        h *= 2
    return y


def inv_sqrt_f32(d: int) -> np.float32:
    return np.float32(1.0 / np.sqrt(d))


def rotate_rows_f32(x, signs) -> np.ndarray:
    """x M in float32 with the kernel's operation order (R7)."""
    s = np.asarray(signs, dtype=np.float32)
    y = np.asarray(x, dtype=np.float32) * s
    y = fwht_f32(y)
    return (y * inv_sqrt_f32(y.shape[-1])).astype(np.float32)


def unrotate_rows(x, signs) -> np.ndarray:
    """x M^T in float64."""
    return np.asarray(x, dtype=np.float64) @ rotation_matrix(signs).T


# ----------------------------------------------------------------------------
# quantiser (R4, R5, R7)
# ----------------------------------------------------------------------------
def quantize(x, signs=None, per_tensor=False, tile=TILE):
    """Codes and scales of a [B, Hx, N, d] tensor.

    x: values of the stored 16-bit inputs (any float dtype, exactly
    representable in float32).  signs: the rotation's sign vector, or None
    for no rotation.  Returns (codes uint8 [B, Hx, N, d], scales float32
    [B, Hx, ceil(N / tile)]).
    """
    x = np.asarray(x, dtype=np.float32)
    B, Hx, N, d = x.shape
    nt = -(-N // tile)
    xr = rotate_rows_f32(x, signs) if signs is not None else x
    absx = np.abs(xr)
    amax = np.zeros((B, Hx, nt), dtype=np.float32)
    for t in range(nt):
        amax[:, :, t] = absx[:, :, t * tile:(t + 1) * tile, :].max(axis=(2, 3))
    if per_tensor:
        amax[...] = amax.max()
    f448 = np.float32(E4M3_MAX)
    with np.errstate(divide="ignore"):
        inv = np.where(amax > 0, f448 / np.where(amax > 0, amax, np.float32(1)), np.float32(0)).astype(np.float32)
    scale = (amax / f448).astype(np.float32)
    inv_rows = np.repeat(inv, tile, axis=2)[:, :, :N, None]
    codes = e4m3_encode((xr * inv_rows).astype(np.float32))
    return codes, scale


def transpose_v(v_codes, tile=TILE) -> np.ndarray:
    """[B, H, N, d] codes -> [B, H, d, Npad] with Npad = N rounded up to a tile, zero padded."""
    B, H, N, d = v_codes.shape
    npad = -(-N // tile) * tile
    out = np.zeros((B, H, d, npad), dtype=np.uint8)
    out[:, :, :, :N] = np.swapaxes(v_codes, 2, 3)
    return out


def dequantize(codes, scale, tile=TILE) -> np.ndarray:
    """float64 values of codes [..., N, d] with per-tile scales [..., nt]."""
    N = codes.shape[-2]
    s = np.repeat(np.asarray(scale, dtype=np.float64), tile, axis=-1)[..., :N, None]
    return e4m3_decode(codes) * s


# ----------------------------------------------------------------------------
# FP8 forward: the gate (R3, R6)
# ----------------------------------------------------------------------------
def head_forward(spec, b, h, q8, sq, k8, sk, v8, sv, signs=None, rows=None):
    """Exact attention of one head's dequantised FP8 inputs, and the bounds of R6.

    q8 [N, d] codes and sq [nt] scales of query head h; k8, v8 [N, d] and
    sk, sv [nt] of its K/V head (row-major V codes).  signs: the rotation
    the quantiser applied (None for none); the output is rotated back with
    it.  Returns (O, LSE, worst, var) for query ``rows``: O [R, d] and LSE
    [R] in float64; worst [R, d] the worst-case bound and var [R, d] the
    variance bound of the error that rounding the probabilities to E4M3
    adds (R6).
    """
    N, d = q8.shape
    rows = np.arange(N) if rows is None else np.asarray(rows, dtype=np.int64)
    cols = np.arange(N)
    qd, kd = dequantize(q8, sq), dequantize(k8, sk)
    # V rows rotated back (x M^T): the error of key j's weight moves the
    # whole row V_j, so the bounds use the rows in the output's coordinates
    vb = dequantize(v8, sv)
    if signs is not None:
        vb = unrotate_rows(vb, signs)
    O = np.zeros((rows.size, d))
    worst = np.zeros((rows.size, d))
    var = np.zeros((rows.size, d))
    lse = np.zeros(rows.size)
    for s0 in range(0, rows.size, _attn.ROW_CHUNK):
        r = rows[s0:s0 + _attn.ROW_CHUNK]
        vis = _attn.visible(spec, b, r, cols)
        S = spec.tau * (qd[r] @ kd.T)
        P, lse[s0:s0 + r.size] = _attn._softmax_rows(S, vis)
        m = np.where(vis, S, -np.inf).max(axis=1, initial=-np.inf)
        fin = np.isfinite(m)
        ls, ms = np.where(fin, lse[s0:s0 + r.size], 0.0), np.where(fin, m, 0.0)
        ell = np.where(fin, np.exp(ls - ms), 1.0)                  # sum_j exp(S_ij - m_i)
        bnd = np.where(vis, np.maximum(2.0 ** -4 * P, 2.0 ** -10 / ell[:, None]), 0.0)
        O[s0:s0 + r.size] = P @ vb
        worst[s0:s0 + r.size] = bnd @ np.abs(vb)
        var[s0:s0 + r.size] = (bnd * bnd) @ (vb * vb) / 3.0
    return O, lse, worst, var


def attention_fwd(spec, q, k, v, signs=None, per_tensor=False):
    """Quantise the whole problem and run the gate on every head.

    q [B, H, N, d], k and v [B, H_kv, N, d] (stored-dtype values).  Returns
    (O, LSE, worst, var, quantised) where quantised holds the codes and
    scales of q, k and v.
    """
    q8, sq = quantize(q, signs, per_tensor)
    k8, sk = quantize(k, signs, per_tensor)
    v8, sv = quantize(v, signs, per_tensor)
    B, H, N, d = q8.shape
    g = spec.group
    out = [np.zeros((B, H, N, d)), np.zeros((B, H, N)), np.zeros((B, H, N, d)), np.zeros((B, H, N, d))]
    for b in range(B):
        for h in range(H):
            hk = h // g
            res = head_forward(spec, b, h, q8[b, h], sq[b, h], k8[b, hk], sk[b, hk], v8[b, hk], sv[b, hk], signs)
            for o, x in zip(out, res):
                o[b, h] = x
    return (*out, dict(q8=q8, sq=sq, k8=k8, sk=sk, v8=v8, sv=sv))


# ----------------------------------------------------------------------------
# one scaling of the rounded probabilities, written out as a diagnostic
# ----------------------------------------------------------------------------
P_SCALE = 256.0


def scaled_p_model_forward(spec, b, h, q8, sq, k8, sk, v8, sv, signs=None, rows=None, round_p=True):
    """O and LSE of one head when P is rounded on one particular scale (diagnostic).

    The pages leave the scale of the rounded probabilities open (R6).  This
    models one choice: the Q-outer online softmax over ascending 128-key
    tiles rounds exp(S - m) * c_t to E4M3, m the running row max after tile
    t, c_t = 256 sv_t / SV (sv_t the tile's V scale, SV the head's largest),
    so that one accumulator serves tiles with different V scales; the row
    sum uses the unrounded probabilities and O' = (SV / 256) sum_t alpha_t
    A_t V8_t / l.  It predicts what such a kernel returns; it is not a gate.
    """
    N, d = q8.shape
    tau = spec.tau
    rows = np.arange(N) if rows is None else np.asarray(rows, dtype=np.int64)
    cols = np.arange(N)
    qd = dequantize(q8, sq)
    kd = dequantize(k8, sk)
    v8d = e4m3_decode(v8)
    sv = np.asarray(sv, dtype=np.float64)
    SV = float(sv.max()) if sv.size else 0.0
    c = P_SCALE * sv / SV if SV > 0 else np.zeros_like(sv)
    tile_of = cols // TILE
    nt = sv.size
    O = np.zeros((rows.size, d))
    lse = np.zeros(rows.size)
    for s0 in range(0, rows.size, _attn.ROW_CHUNK):
        r = rows[s0:s0 + _attn.ROW_CHUNK]
        S = tau * (qd[r] @ kd.T)
        vis = _attn.visible(spec, b, r, cols)
        S = np.where(vis, S, -np.inf)
        # running max after each key tile (ascending), and the final max
        tmax = np.stack([S[:, t * TILE:(t + 1) * TILE].max(axis=1, initial=-np.inf) for t in range(nt)], axis=1)
        mrun = np.maximum.accumulate(tmax, axis=1)
        mfin = mrun[:, -1]
        empty = ~np.isfinite(mfin)
        mrun_safe = np.where(np.isfinite(mrun), mrun, 0.0)
        mfin_safe = np.where(empty, 0.0, mfin)
        mj = mrun_safe[:, tile_of]                                   # reference max when key j is used
        E = np.where(vis, np.exp(np.where(vis, S, 0.0) - mj), 0.0)   # in (0, 1]
        X = E * c[tile_of][None, :]
        A = e4m3_round(X) if round_p else X
        alpha = np.where(vis, np.exp(mj - mfin_safe[:, None]), 0.0)  # rescale from tile t to the end
        ell = np.where(vis, np.exp(np.where(vis, S, 0.0) - mfin_safe[:, None]), 0.0).sum(axis=1)
        ell_safe = np.where(empty, 1.0, ell)
        W = alpha * A * (SV / P_SCALE) / ell_safe[:, None]
        Orot = np.where(empty[:, None], 0.0, W @ v8d)
        Oc = unrotate_rows(Orot, signs) if signs is not None else Orot
        O[s0:s0 + r.size] = Oc
        lse[s0:s0 + r.size] = np.where(empty, -np.inf, mfin_safe + np.log(ell_safe))
    return O, lse


def scaled_p_model_attention_fwd(spec, q, k, v, signs=None, per_tensor=False, round_p=True):
    """``scaled_p_model_forward`` over the whole problem: (O, LSE, quantised)."""
    q8, sq = quantize(q, signs, per_tensor)
    k8, sk = quantize(k, signs, per_tensor)
    v8, sv = quantize(v, signs, per_tensor)
    B, H, N, d = q8.shape
    g = spec.group
    O = np.zeros((B, H, N, d))
    L = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            hk = h // g
            O[b, h], L[b, h] = scaled_p_model_forward(spec, b, h, q8[b, h], sq[b, h], k8[b, hk], sk[b, hk],
                                                      v8[b, hk], sv[b, hk], signs, round_p=round_p)
    return O, L, dict(q8=q8, sq=sq, k8=k8, sk=sk, v8=v8, sv=sv)


def relative_error(approx, exact) -> float:
    """Root-mean-square error of approx over the root-mean-square of exact."""
    a = np.asarray(approx, dtype=np.float64)
    e = np.asarray(exact, dtype=np.float64)
    return float(np.sqrt(np.mean((a - e) ** 2)) / np.sqrt(np.mean(e ** 2)))
