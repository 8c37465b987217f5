"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of ``oracle/`` on the CPU (a dropped
scale, a flipped sign, a transposed operand, a wrong mask boundary, ...) and
runs the pin tests against the copy in a subprocess; at least one pin must
fail.  Nothing here touches a GPU.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = [
    ("attention.py", "dk += tau * (dS.T @ q[r])", "dk += (dS.T @ q[r])"),
    ("attention.py", "dS = P * (dP - Dr[:, None])", "dS = P * (dP + Dr[:, None])"),
    ("attention.py", "dq[s:s + ROW_CHUNK] = tau * (dS @ k)", "dq[s:s + ROW_CHUNK] = tau * (dS @ q[r])"),
    ("attention.py", "dv += Pt.T @ do[r]", "dv += P.T @ do[r]"),
    ("attention.py", "dP = Z * dPt / (1.0 - spec.dropout_p)", "dP = dPt"),
    ("attention.py", "Pt = keep(spec, b, h, r, cols) * P / (1.0 - spec.dropout_p)",
     "Pt = keep(spec, b, h, r, cols) * P"),
    ("attention.py", "m_safe + np.log(", "m_safe + np.log1p("),
    ("masks.py", "m &= cols <= rows", "m &= cols < rows"),
    ("masks.py", "m &= cols < int(seqlen_k)", "m &= cols <= int(seqlen_k)"),
    ("tiled.py", "Oi = alpha[:, None] * Oi + P @ v[cj[0]:cj[1]]", "Oi = Oi + P @ v[cj[0]:cj[1]]"),
    ("tiled.py", "l_new = a_old * li + a_til * P_til.sum(axis=1)", "l_new = li + a_til * P_til.sum(axis=1)"),
    ("philox.py", "c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0",
     "c0, c1, c2, c3 = hi0 ^ c1 ^ k0, lo1, hi1 ^ c3 ^ k1, lo0"),
    ("philox.py", "return half >= np.uint64(T)", "return half > np.uint64(T)"),
    ("philox.py", "32: dict(M0=0xD2511F53, M1=0xCD9E8D57", "32: dict(M0=0xD2511F55, M1=0xCD9E8D57"),
    ("philox.py", "W0=0x9E3779B9, W1=0xBB67AE85", "W0=0x9E3779B9, W1=0xBB67AE86"),
    ("masks.py", "m &= cols > rows - int(window)", "m &= cols >= rows - int(window)"),
    ("attention.py", "dk[b, h // g] += r[\"dk\"]", "dk[b, h // g] = r[\"dk\"]"),
    ("attention.py", "O[b, h], L[b, h] = head_forward(spec, b, h, q[b, h], k[b, h // g], v[b, h // g])",
     "O[b, h], L[b, h] = head_forward(spec, b, h, q[b, h], k[b, h % spec.hkv], v[b, h % spec.hkv])"),
    # the FP8 forward (oracle/fp8.py)
    ("fp8.py", "mm = np.rint((mant * 2.0 - 1.0) * 8.0)", "mm = np.floor((mant * 2.0 - 1.0) * 8.0 + 0.5)"),
    ("fp8.py", "code = np.minimum(code, 0x7E)", "code = np.minimum(code, 0x7F)"),
    ("fp8.py", "sub = a < 2.0 ** -6", "sub = a < 2.0 ** -7"),
    ("fp8.py", "return (s[:, None] * sylvester(d)) / np.sqrt(d)", "return (s[:, None] * sylvester(d)) / d"),
    ("fp8.py", "z[..., 1, :] = a - b", "z[..., 1, :] = b - a"),
    ("fp8.py", "scale = (amax / f448).astype(np.float32)", "scale = (amax / np.float32(240)).astype(np.float32)"),
    ("fp8.py", "Oc = unrotate_rows(Orot, signs)", "Oc = Orot"),
    ("fp8.py", "np.maximum(2.0 ** -4 * P, 2.0 ** -10 / ell[:, None])",
     "np.maximum(2.0 ** -5 * P, 2.0 ** -10 / ell[:, None])"),
    ("fp8.py", "var[s0:s0 + r.size] = (bnd * bnd) @ (vb * vb) / 3.0",
     "var[s0:s0 + r.size] = (bnd * bnd) @ (vb * vb) / 12.0"),
    ("fp8.py", "        vb = unrotate_rows(vb, signs)\n", "        pass\n"),
    ("fp8.py", "O[s0:s0 + r.size] = P @ vb", "O[s0:s0 + r.size] = P @ vb * 1.001"),
    ("fp8.py", "c = P_SCALE * sv / SV if SV > 0 else np.zeros_like(sv)", "c = P_SCALE * np.ones_like(sv)"),
    ("fp8.py", "mrun = np.maximum.accumulate(tmax, axis=1)",
     "mrun = np.repeat(tmax.max(axis=1, keepdims=True), nt, axis=1)"),
    ("fp8.py", "alpha = np.where(vis, np.exp(mj - mfin_safe[:, None]), 0.0)",
     "alpha = np.where(vis, np.exp(mfin_safe[:, None] - mj), 0.0)"),
]


@pytest.mark.slow
@pytest.mark.parametrize("fname,old,new", MUTATIONS)
def test_pins_catch_planted_mistake(tmp_path, fname, old, new):
    dst = tmp_path / "r"
    shutil.copytree(os.path.join(ROOT, "oracle"), dst / "oracle")
    shutil.copytree(os.path.join(ROOT, "tests"), dst / "tests",
                    ignore=shutil.ignore_patterns("test_oracle_mutations.py", "__pycache__", "test_gpu*", "test_zz*"))
    # the seeded input generator (no attention arithmetic) for the FP8 pins
    shutil.copytree(os.path.join(ROOT, "exact_io_aware_tiled_gb300"), dst / "exact_io_aware_tiled_gb300",
                    ignore=shutil.ignore_patterns("csrc", "_build", "*.so", "__pycache__"))
    p = dst / "oracle" / fname
    src = p.read_text()
    assert src.count(old) == 1, "mutation anchor not found: " + old
    p.write_text(src.replace(old, new))
    tests = [str(dst / "tests" / t) for t in ("test_oracle_attention.py", "test_oracle_tiled.py",
                                             "test_oracle_philox.py", "test_oracle_traffic.py",
                                             "test_oracle_gqa_window.py", "test_oracle_fp8.py")]
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "-m", "not slow", *tests], cwd=dst, capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, "planted mistake survived every pin:\n" + r.stdout[-2000:]
