"""The oracle's pins must catch plausible slips in the oracle itself.

Each case plants one mistake (a wrong field offset, bit position, zero point,
scale index, row stride, sign, dropped term, transposed operand or layout, a
loosened acceptance bar) in a private copy of the oracle, rebuilds it, and runs
the pin module (tests/test_oracle_pins.py) against the copy in a subprocess:
the pins must fail. An unmodified copy must pass. CPU only; nothing here
touches the CUDA library, and the mistakes are planted in copies, never in
the oracle the other tests use.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
C = "oracle/qmm_oracle.c"
PY = "oracle/__init__.py"

# (name, file, original text (must occur exactly once), planted text)
MUTATIONS = [
    # IEEE half and bfloat16 decodes, byte order
    ("f16 exponent bias", C, "expo - 25);", "expo - 24);"),
    ("f16 subnormal scale", C, "ldexp((double)mant, -24);", "ldexp((double)mant, -25);"),
    ("f16 sign dropped", C, "return sign ? -v : v;", "return v;"),
    ("bf16 shift", C, "((uint32_t)h) << 16;", "((uint32_t)h) << 15;"),
    ("u16 read big-endian", C, "(p[0] | (p[1] << 8))", "(p[1] | (p[0] << 8))"),
    ("Q6_K row bytes", C, "(k / 256) * 210 : 0;", "(k / 256) * 208 : 0;"),
    # Q4_0
    ("Q4_0 zero point", C, "out[i] = (float)((q_lo - 8) * d);", "out[i] = (float)((q_lo - 7) * d);"),
    ("Q4_0 nibble halves swapped", C, "int q_lo = qs[i] & 0x0F;\n        int q_hi = qs[i] >> 4;",
     "int q_hi = qs[i] & 0x0F;\n        int q_lo = qs[i] >> 4;"),
    ("Q4_0 quant offset", C, "const uint8_t *qs = blk + 2;", "const uint8_t *qs = blk + 4;"),
    # Q4_K
    ("Q4_K sub-block scale index", C, "q4_k_scale_min(scales, 2 * c + 1, &sc1, &m1);",
     "q4_k_scale_min(scales, 2 * c, &sc1, &m1);"),
    ("Q4_K scale top bits from the min byte", C, "((scales[s - 4] >> 6) << 4)", "((scales[s] >> 6) << 4)"),
    ("Q4_K min nibble", C, "*m = (scales[s + 4] >> 4)", "*m = (scales[s + 4] & 0x0F)"),
    ("Q4_K min dropped", C, "(float)(d * sc0 * q_lo - dmin * m0);", "(float)(d * sc0 * q_lo);"),
    ("Q4_K min sign", C, "(float)(d * sc1 * q_hi - dmin * m1);", "(float)(d * sc1 * q_hi + dmin * m1);"),
    ("Q4_K quant offset", C, "const uint8_t *qs = blk + 16;", "const uint8_t *qs = blk + 12;"),
    # Q6_K
    ("Q6_K qh bit pair", C, "(((H[l] >> 2) & 3) << 4)", "(((H[l] >> 4) & 3) << 4)"),
    ("Q6_K low-bits byte", C, "q[1] = (L[l + 32] & 0x0F)", "q[1] = (L[l] & 0x0F)"),
    ("Q6_K scale group", C, "scales[e / 16]", "scales[e / 32]"),
    ("Q6_K zero point", C, "(q[r] - 32)", "(q[r] - 31)"),
    ("Q6_K d offset", C, "rd_u16(blk + 208)", "rd_u16(blk + 206)"),
    ("Q6_K unsigned scales", C, "const int8_t *scales = (const int8_t *)(blk + 192);",
     "const uint8_t *scales = (const uint8_t *)(blk + 192);"),
    # Q8_0, Q5_0
    ("Q8_0 unsigned codes", C, "int q = (int)(int8_t)blk[2 + i];", "int q = (int)blk[2 + i];"),
    ("Q8_0 code offset", C, "int q = (int)(int8_t)blk[2 + i];", "int q = (int)(int8_t)blk[1 + i];"),
    ("Q5_0 high half takes the low qh bits", C, "((qh >> (i + 16)) & 1u)", "((qh >> i) & 1u)"),
    ("Q5_0 zero point", C, "out[i] = (float)((q_lo - 16) * d);", "out[i] = (float)((q_lo - 15) * d);"),
    ("Q5_0 quant offset", C, "const uint8_t *qs = blk + 6;", "const uint8_t *qs = blk + 5;"),
    ("Q5_0 halves swapped", C,
     "out[i] = (float)((q_lo - 16) * d);\n        out[i + 16] = (float)((q_hi - 16) * d);",
     "out[i + 16] = (float)((q_lo - 16) * d);\n        out[i] = (float)((q_hi - 16) * d);"),
    # plain and sampled products
    ("product magnitude without abs", C,
     "                acc += p;\n                mag += fabs(p);", "                acc += p;\n                mag += p;"),
    ("product output transposed", C, "            y[t * n + j] = acc;\n            s[t * n + j] = mag;\n        }\n    }\n    return 0;\n}\n\n/* The same product for `count` chosen outputs (t_idx[c], j_idx[c]) only. */",
     "            y[j * n_tokens + t] = acc;\n            s[t * n + j] = mag;\n        }\n    }\n    return 0;\n}\n\n/* The same product for `count` chosen outputs (t_idx[c], j_idx[c]) only. */"),
    ("sampled product token row", C, "const float *xt = x + t * k;\n        double acc = 0.0, mag = 0.0;",
     "const float *xt = x + j % n_tokens * k;\n        double acc = 0.0, mag = 0.0;"),
    # backward with respect to the input
    ("back-input magnitude without abs", C, "            dx[i] += p;\n            s[i] += fabs(p);",
     "            dx[i] += p;\n            s[i] += p;"),
    ("back-input dy index", C, "double p = (double)dy[j] * (double)wrow_scratch[i];",
     "double p = (double)dy[j - j0] * (double)wrow_scratch[i];"),
    ("back-input range end", C, "for (int64_t j = j0; j < j1; ++j) {", "for (int64_t j = j0; j + 1 < j1; ++j) {"),
    # expert-indexed product
    ("experts slice stride", C, "const uint8_t *we = w + e * rb * n;", "const uint8_t *we = w + e * rb;"),
    ("experts x row by slot", C, "double v = (double)x[p * k + i] * (double)wrow_scratch[i];",
     "double v = (double)x[sl * k + i] * (double)wrow_scratch[i];"),
    ("experts output layout", C, "y[(p * top_k + sl) * n + j] = acc;", "y[(sl * n_pos + p) * n + j] = acc;"),
    # MLX-style affine rows
    ("affine code order", C, "(word >> (bits * (i % per_word)))", "(word >> (bits * (per_word - 1 - i % per_word)))"),
    ("affine bias dropped", C, "out[i] = (float)((double)q * scale + bias);", "out[i] = (float)((double)q * scale);"),
    ("affine group of 32", C, "rd_u16(srow + 2 * (i / 64))", "rd_u16(srow + 2 * (i / 32))"),
    ("affine scale read from the biases", C, "rd_u16(srow + 2 * (i / 64))", "rd_u16(brow + 2 * (i / 64))"),
    ("affine dequant row stride", C, "sc + j * (k / 32), bi + j * (k / 32), k,\n                                      out + j * k))",
     "sc + j * (k / 64), bi + j * (k / 64), k,\n                                      out + j * k))"),
    ("affine product row stride", C,
     "sc + j * (k / 32), bi + j * (k / 32), k,\n                                      wrow_scratch))\n            return -1;\n        for",
     "sc + j * (k / 64), bi + j * (k / 64), k,\n                                      wrow_scratch))\n            return -1;\n        for"),
    ("affine sampled row stride", C,
     "sc + j * (k / 32), bi + j * (k / 32), k,\n                                      wrow_scratch))\n            return -1;\n        double",
     "sc + j * (k / 64), bi + j * (k / 64), k,\n                                      wrow_scratch))\n            return -1;\n        double"),
    # gated pairs
    ("silu sign", C, "if (act == 0) return g / (1.0 + exp(-g));", "if (act == 0) return g / (1.0 + exp(g));"),
    ("gelu cubic coefficient", C, "const double z = c * (g + 0.044715 * g * g * g);\n    return",
     "const double z = c * (g + 0.04715 * g * g * g);\n    return"),
    ("gelu factor 2 dropped", C, "return g / (1.0 + exp(-2.0 * z));\n}", "return g / (1.0 + exp(-z));\n}"),
    ("silu derivative", C, "return sg * (1.0 + g * (1.0 - sg));", "return sg * (1.0 + g * sg);"),
    ("gelu derivative chain factor", C, "2.0 * c * (1.0 + 3.0 * 0.044715 * g * g)", "c * (1.0 + 3.0 * 0.044715 * g * g)"),
    ("gate and up matrices swapped", C, "(m ? wu : wg)", "(m ? wg : wu)"),
    ("activation applied to up", C,
     "const double a = oracle_act(act, gu[0]);\n            y[t * n + j] = a * gu[1];",
     "const double a = oracle_act(act, gu[1]);\n            y[t * n + j] = a * gu[0];"),
    ("gated error bar drops the up term", C, "* su[0] + fabs(a) * su[1];", "* su[0];"),
    ("gated error bar with a signed derivative", C, "fabs(oracle_act_deriv(act, gu[0]))", "oracle_act_deriv(act, gu[0])"),
    ("gated act selector ignored", C, "if (act == 0) return g / (1.0 + exp(-g));",
     "if (act >= 0) return g / (1.0 + exp(-g));"),
    # cosine
    ("cosine of zero vectors 0", PY, "    if na == 0.0 and nb == 0.0:\n        return 1.0", "    if na == 0.0 and nb == 0.0:\n        return 0.0"),
    ("cosine without the norm of b", PY, "np.dot(a, b) / (np.sqrt(na) * np.sqrt(nb))", "np.dot(a, b) / (np.sqrt(na) * np.sqrt(na))"),
    # numpy-product helpers and the tile rule of the wrapper
    ("blas product transposed weights", PY, "    return x64 @ deq.T, np.abs(x64) @ np.abs(deq).T\n\n\ndef matmul_sampled",
     "    return x64 @ deq.T[::-1], np.abs(x64) @ np.abs(deq).T\n\n\ndef matmul_sampled"),
    ("blas back-input magnitude without abs", PY, "    return d @ deq, np.abs(d) @ np.abs(deq)",
     "    return d @ deq, np.abs(d @ deq)"),
    ("blas back-input tile ignored", PY, "    d = np.asarray(dy, np.float64).reshape(-1)[j_start:j_end]",
     "    d = np.asarray(dy, np.float64).reshape(-1)[:j_end - j_start]"),
    ("affine blas without abs", PY, "    deq = dequant_affine(bits, w, scales, biases, k, n).astype(np.float64)\n    x64 = np.atleast_2d(np.asarray(x, np.float64))\n    return x64 @ deq.T, np.abs(x64) @ np.abs(deq).T",
     "    deq = dequant_affine(bits, w, scales, biases, k, n).astype(np.float64)\n    x64 = np.atleast_2d(np.asarray(x, np.float64))\n    return x64 @ deq.T, np.abs(x64 @ deq.T)"),
    ("tile bar without |y_in|", PY, "        s[:, sl] = s_ref[:, sl] + np.abs(np.asarray(y_in, np.float64)[:, sl])",
     "        s[:, sl] = s_ref[:, sl]"),
    ("tile accumulate overwrites", PY, "        y[:, sl] = y[:, sl] + y_ref[:, sl]", "        y[:, sl] = y_ref[:, sl]"),
    # acceptance check
    ("bar 1e-3 instead of 1e-4", PY, "TOL_REL = 1e-4", "TOL_REL = 1e-3"),
    ("cosine floor 0.999", PY, "COSINE_FLOOR = 0.9999", "COSINE_FLOOR = 0.999"),
    ("check ignores the cosine", PY, "ok = (not bad.any()) and cos >= COSINE_FLOOR", "ok = not bad.any()"),
    ("check ignores NaN mismatches", PY, "    bad |= nan_mismatch\n", "\n"),
    ("check bar ten times wider", PY, "bad = (err > bound) & finite", "bad = (err > 10 * bound) & finite"),
]


def _copy_tree(dst):
    """The oracle, the seeded generators and the pin module, nothing built."""
    ign = shutil.ignore_patterns("*.so", "*.tmp", "__pycache__")
    shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(dst, "oracle"), ignore=ign)
    os.makedirs(os.path.join(dst, "tests"))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(dst, "tests", "golden"))
    for f in ("tests/conftest.py", "tests/test_oracle_pins.py", "qmm_synth.py"):
        shutil.copy(os.path.join(ROOT, f), os.path.join(dst, f))


def _run_pins(dst):
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py"], cwd=dst, capture_output=True, text=True,
                       timeout=600)
    failed = [l for l in r.stdout.splitlines() if l.startswith("FAILED")]
    return r.returncode, (failed[0] if failed else r.stdout[-300:] + r.stderr[-300:])


def _plant(base, idx):
    name, rel, old, new = MUTATIONS[idx]
    dst = os.path.join(base, f"m{idx:02d}")
    _copy_tree(dst)
    path = os.path.join(dst, rel)
    with open(path) as f:
        src = f.read()
    assert src.count(old) == 1, f"{name}: the original text occurs {src.count(old)} times"
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    return _run_pins(dst)


def test_unmodified_copy_passes_its_pins(tmp_path):
    _copy_tree(str(tmp_path))
    rc, msg = _run_pins(str(tmp_path))
    assert rc == 0, msg


def test_every_planted_mistake_fails_a_pin(tmp_path):
    workers = max(1, min(8, os.cpu_count() or 1))
    with ThreadPoolExecutor(workers) as ex:
        results = list(ex.map(lambda i: _plant(str(tmp_path), i), range(len(MUTATIONS))))
    # exit status 1 = tests ran and one failed; anything else (a build or
    # collection error) would not show that a pin caught the mistake
    missed = [(MUTATIONS[i][0], rc, msg) for i, (rc, msg) in enumerate(results) if rc != 1]
    assert not missed, "\n".join(f"{n}: exit {rc}: {m}" for n, rc, m in missed)


@pytest.mark.parametrize("idx", range(len(MUTATIONS)), ids=[m[0] for m in MUTATIONS])
def test_planted_text_is_present_once(idx):
    name, rel, old, new = MUTATIONS[idx]
    with open(os.path.join(ROOT, rel)) as f:
        assert f.read().count(old) == 1
    assert old != new
