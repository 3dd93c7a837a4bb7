"""Pins for the oracle: facts fixed by the pages and by the mathematics, each
chosen so that a plausible slip in the oracle (a wrong field offset, swapped
nibbles, a dropped min term, a wrong scale index, a transposed operand)
fails at least one of them. CPU only."""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import qmm_synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_constants.txt")


def _golden():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- sizes ----

def test_row_bytes_closed_forms():
    # (k/32)*18, (k/256)*144, (k/256)*210, 2k bytes per row (rullama matmul.rs checks)
    for k in (0, 32, 64, 96, 256, 512, 2560, 4096):
        assert oracle.row_bytes("q4_0", k) == (k // 32) * 18
        assert oracle.row_bytes("bf16", k) == 2 * k
        assert oracle.row_bytes("f16", k) == 2 * k
    for k in (0, 256, 512, 1536, 2560, 4096, 6144):
        assert oracle.row_bytes("q4_k", k) == (k // 256) * 144
        assert oracle.row_bytes("q6_k", k) == (k // 256) * 210
    # shapes the formats reject
    assert oracle.row_bytes("q4_0", 48) == 0
    assert oracle.row_bytes("q4_k", 128) == 0
    assert oracle.row_bytes("q6_k", 300) == 0
    assert oracle.row_bytes("bf16", 3) == 0


def test_golden_page_constants():
    for row in _golden():
        kind = row[0]
        if kind == "f16":
            assert oracle.f16_value(int(row[1], 16)) == float(row[2])
        elif kind == "block":
            fmt, elems, nbytes = row[1], int(row[2]), int(row[3])
            assert oracle.row_bytes(fmt, elems) == nbytes
            assert oracle.row_bytes(fmt, 4 * elems) == 4 * nbytes
        elif kind == "rowbytes":
            assert oracle.row_bytes(row[1], int(row[2])) == int(row[3])
        elif kind == "offset":
            fmt, field, off = row[1], row[2], int(row[3])
            _check_offset(fmt, field, off)
        elif kind == "affine":
            bits, k, rb, groups = (int(v) for v in row[1:5])
            assert oracle.affine_row_bytes(bits, k) == rb
            # one scale and one bias per group: the oracle accepts exactly
            # [n, groups] of each
            w = np.zeros(rb, np.uint8)
            sb = np.zeros(groups, np.uint16)
            oracle.dequant_affine(bits, w, sb, sb, k, 1)
            with pytest.raises(ValueError):
                oracle.dequant_affine(bits, w, sb[:-1], sb[:-1], k, 1)
        elif kind == "floor":
            assert row[1] == "cosine" and oracle.COSINE_FLOOR == float(row[2])
        else:
            raise AssertionError(f"unknown golden kind {kind}")


def _check_offset(fmt, field, off):
    """Write f16(0.0625) at the page-given offset of a block built so that the
    element values are exactly +-that field; the decoded weights must show it."""
    if fmt == "q4_0":
        blk = np.zeros(18, np.uint8)
        blk[off:off + 2] = [0x00, 0x2C]
        blk[2:] = 0x99  # q = 9 -> (9-8)*d = d
        w = oracle.dequant("q4_0", blk, 32, 1)
        assert np.all(w == 0.0625)
    elif fmt == "q4_k":
        blk = np.zeros(144, np.uint8)
        blk[off:off + 2] = [0x00, 0x2C]
        if field == "d":  # scale 1, min 0, q = 1 -> d
            sc, m = [1] * 8, [0] * 8
            q = np.ones(256, np.int64)
        else:             # scale 0, min 1 -> -dmin
            sc, m = [0] * 8, [1] * 8
            q = np.zeros(256, np.int64)
        blk[4:16] = _pack_q4_k_scales(sc, m)
        blk[16:144] = _pack_q4_k_qs(q)
        w = oracle.dequant("q4_k", blk, 256, 1)
        assert np.all(w == (0.0625 if field == "d" else -0.0625))
    elif fmt == "q6_k":
        blk = np.zeros(210, np.uint8)
        blk[off:off + 2] = [0x00, 0x2C]
        blk[192:208] = 1                       # every scale = 1
        q = np.full(256, 33, np.int64)         # q - 32 = 1
        blk[0:192] = _pack_q6_k_q(q)
        w = oracle.dequant("q6_k", blk, 256, 1)
        assert np.all(w == 0.0625)
    else:
        raise AssertionError(fmt)


# ----------------------------------------------------------- f16 / bf16 ----

def test_f16_decoder_exhaustive_against_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_value(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.copysign(1.0, oracle.f16_value(0x8000)) == -1.0


def test_f16_special_values():
    assert oracle.f16_value(0x3C00) == 1.0
    assert oracle.f16_value(0x0001) == 2.0 ** -24          # smallest subnormal
    assert oracle.f16_value(0x03FF) == 1023 * 2.0 ** -24   # largest subnormal
    assert oracle.f16_value(0x0400) == 2.0 ** -14          # smallest normal
    assert oracle.f16_value(0x7BFF) == 65504.0
    assert oracle.f16_value(0x7C00) == float("inf")
    assert oracle.f16_value(0xFC00) == float("-inf")
    assert np.isnan(oracle.f16_value(0x7E00))


def test_bf16_is_upper_half_of_f32():
    rng = np.random.default_rng(0)
    f = rng.normal(0, 3, 4096).astype(np.float32)
    hi = (f.view(np.uint32) >> 16).astype(np.uint16)
    got = np.array([oracle.bf16_value(int(h)) for h in hi], np.float32)
    # the page's CPU round trip: bits & 0xFFFF0000
    assert np.array_equal(got.view(np.uint32), f.view(np.uint32) & 0xFFFF0000)


# ------------------------------------------------------- block packing ----
# Test-side inverses of the ggml layouts, used only to build blocks whose
# element values are known in closed form.

def _pack_q4_k_scales(sc, m):
    b = [0] * 12
    for s in range(4):
        b[s] = (sc[s] & 63) | ((sc[s + 4] >> 4) << 6)
        b[s + 4] = (m[s] & 63) | ((m[s + 4] >> 4) << 6)
    for s in range(4, 8):
        b[s + 4] = (sc[s] & 15) | ((m[s] & 15) << 4)
    return np.array(b, np.uint8)


def _pack_q4_k_qs(q):
    qs = np.zeros(128, np.uint8)
    for c in range(4):
        for l in range(32):
            qs[32 * c + l] = q[64 * c + l] | (q[64 * c + 32 + l] << 4)
    return qs


def _pack_q6_k_q(q):
    out = np.zeros(192, np.uint8)
    ql, qh = out[:128], out[128:]
    for h in range(2):
        for l in range(32):
            e = 128 * h + l
            ql[64 * h + l] = (q[e] & 15) | ((q[e + 64] & 15) << 4)
            ql[64 * h + 32 + l] = (q[e + 32] & 15) | ((q[e + 96] & 15) << 4)
            qh[32 * h + l] = ((q[e] >> 4) | ((q[e + 32] >> 4) << 2)
                              | ((q[e + 64] >> 4) << 4) | ((q[e + 96] >> 4) << 6))
    return out


def test_q4_0_hand_packed():
    blk = np.zeros(18, np.uint8)
    blk[0:2] = [0x00, 0x3C]  # d = 1.0
    for i in range(16):
        blk[2 + i] = i | ((15 - i) << 4)
    w = oracle.dequant("q4_0", blk, 32, 1)[0]
    assert list(w[:16]) == [i - 8 for i in range(16)]
    assert list(w[16:]) == [7 - i for i in range(16)]
    # negative d flips the sign exactly
    blk[0:2] = [0x00, 0xB8]  # d = -0.5
    w = oracle.dequant("q4_0", blk, 32, 1)[0]
    assert list(w[:16]) == [-(i - 8) * 0.5 for i in range(16)]


@pytest.mark.parametrize("variant", ["small", "top_bits"])
def test_q4_k_hand_packed(variant):
    if variant == "small":
        sc = [s + 1 for s in range(8)]
        m = [s for s in range(8)]
        d, dmin, dbits, dminbits = 1.0, 1.0, 0x3C00, 0x3C00
    else:  # exercise the two top bits of every 6-bit field
        sc = [63 - s for s in range(8)]
        m = [32 + s for s in range(8)]
        d, dmin, dbits, dminbits = 0.5, 0.25, 0x3800, 0x3400
    q = np.array([(7 * e + e // 32) % 16 for e in range(256)], np.int64)  # low/high nibbles differ
    blk = np.zeros(144, np.uint8)
    blk[0:2] = [dbits & 0xFF, dbits >> 8]
    blk[2:4] = [dminbits & 0xFF, dminbits >> 8]
    blk[4:16] = _pack_q4_k_scales(sc, m)
    blk[16:] = _pack_q4_k_qs(q)
    w = oracle.dequant("q4_k", blk, 256, 1)[0]
    expect = [d * sc[e // 32] * q[e] - dmin * m[e // 32] for e in range(256)]
    assert list(w) == [np.float32(v) for v in expect]


def test_q6_k_hand_packed():
    q = np.array([(5 * e + e // 64) % 64 for e in range(256)], np.int64)
    blk = np.zeros(210, np.uint8)
    blk[0:192] = _pack_q6_k_q(q)
    blk[192:208] = np.array([s - 8 for s in range(16)], np.int8).view(np.uint8)
    blk[208:210] = [0x00, 0x3C]  # d = 1.0 at the page-given offset
    w = oracle.dequant("q6_k", blk, 256, 1)[0]
    expect = [(e // 16 - 8) * (q[e] - 32) for e in range(256)]
    assert list(w) == expect


def test_block_order_within_row():
    """Row of 3 Q4_0 blocks with d = 1, 2, 4: block b scales elements 32b..32b+31."""
    k = 96  # row_bytes = 54, not a multiple of 4: accepted (no u32-row constraint)
    row = np.zeros(54, np.uint8)
    for b, dbits in enumerate((0x3C00, 0x4000, 0x4400)):
        row[18 * b:18 * b + 2] = [dbits & 0xFF, dbits >> 8]
        row[18 * b + 2:18 * b + 18] = 0x9A  # low nibble 10 (q-8=2), high 9 (q-8=1)
    w = oracle.dequant("q4_0", row, k, 1)[0]
    for b, d in enumerate((1.0, 2.0, 4.0)):
        assert np.all(w[32 * b:32 * b + 16] == 2 * d)
        assert np.all(w[32 * b + 16:32 * b + 32] == 1 * d)


# ------------------------------------------------ invariants on random ----

def test_random_block_invariants():
    rng = np.random.default_rng(11)
    # Q4_0: w / d is an integer in [-8, 7]
    w = qmm_synth.gen_weights("q4_0", 256, 8, rng)
    deq = oracle.dequant("q4_0", w, 256, 8).reshape(8, 8, 32)
    d = w.reshape(8, 8, 18)[..., 0:2].copy().view("<f2").astype(np.float64)
    r = deq / d  # d has shape [8, 8, 1]: broadcasts over the 32 elements
    assert np.all(r == np.round(r)) and r.min() >= -8 and r.max() <= 7
    # Q6_K: w / (d * scale) is an integer in [-32, 31]
    w = qmm_synth.gen_weights("q6_k", 512, 4, rng)
    deq = oracle.dequant("q6_k", w, 512, 4).reshape(4, 2, 16, 16).astype(np.float64)
    blk = w.reshape(4, 2, 210)
    d = blk[..., 208:210].copy().view("<f2").astype(np.float64)[..., 0]
    sc = blk[..., 192:208].view(np.int8).astype(np.float64)
    denom = d[..., None] * sc
    ok = denom != 0
    r = deq[ok] / np.broadcast_to(denom[..., None], deq.shape)[ok]
    assert np.all(r == np.round(r)) and r.min() >= -32 and r.max() <= 31
    assert np.all(deq[~np.broadcast_to(ok[..., None], deq.shape)] == 0)


def test_q4_k_single_rounding():
    """A Q4_K block whose exact values need more than 24 bits: each decoded
    weight is the f32 nearest the exact d*sc*q - dmin*m (rounded once)."""
    d = Fraction(1) + Fraction(1, 1024)              # f16 0x3C01
    dmin = Fraction(1, 2 ** 14) * (1 + Fraction(1, 1024))  # f16 0x0401
    sc = [63, 62, 61, 60, 59, 58, 57, 55]
    m = [1, 3, 5, 7, 63, 33, 17, 9]
    q = np.array([(3 * e + 1) % 16 for e in range(256)], np.int64)
    blk = np.zeros(144, np.uint8)
    blk[0:2] = [0x01, 0x3C]
    blk[2:4] = [0x01, 0x04]
    blk[4:16] = _pack_q4_k_scales(sc, m)
    blk[16:] = _pack_q4_k_qs(q)
    w = oracle.dequant("q4_k", blk, 256, 1)[0]
    rounded_somewhere = False
    for e in range(256):
        exact = d * sc[e // 32] * int(q[e]) - dmin * m[e // 32]
        want = np.float32(float(exact))  # exact value fits a double; one RNE to f32
        assert w[e] == want, e
        rounded_somewhere |= Fraction(float(want)) != exact
    assert rounded_somewhere


# -------------------------------------------------------------- matmul ----

def test_identity_f16_and_bf16():
    # rullama matmul.rs f16_matmul_3x4_eye, widened: identity W gives y = x exactly
    k = n = 8
    x = (np.arange(k, dtype=np.float32) + 1) * 0.25
    for fmt, one in (("f16", 0x3C00), ("bf16", 0x3F80)):
        wbits = np.zeros((n, k), np.uint16)
        for j in range(n):
            wbits[j, j] = one
        y, s = oracle.matmul(fmt, wbits.astype("<u2").view(np.uint8).reshape(-1), x, k, n)
        assert np.array_equal(y[0], x.astype(np.float64))
        assert np.array_equal(s[0], np.abs(x).astype(np.float64))


def test_one_hot_x_picks_weight_column():
    rng = np.random.default_rng(3)
    for fmt, k in (("q4_0", 64), ("q4_k", 256), ("q6_k", 256), ("bf16", 32), ("f16", 32)):
        n = 5
        w = qmm_synth.gen_weights(fmt, k, n, rng)
        deq = oracle.dequant(fmt, w, k, n)
        for i in (0, 1, k // 2 + 3, k - 1):
            x = np.zeros((1, k), np.float32)
            x[0, i] = 1.0
            y, _ = oracle.matmul(fmt, w, x, k, n)
            assert np.array_equal(y[0], deq[:, i].astype(np.float64))


def test_brute_force_tiny_q4_0():
    """Hand-listed sums for a 2-row, k=32 Q4_0 product (row 1 uses d = -0.25)."""
    w = np.zeros(36, np.uint8)
    w[0:2] = [0x00, 0x3C]                    # d = 1
    w[2:18] = [(i % 16) | (((i + 3) % 16) << 4) for i in range(16)]
    w[18:20] = [0x00, 0xB4]                  # d = -0.25
    w[20:36] = [15 - i for i in range(16)]   # high nibbles 0
    x = np.array([[(i % 5) - 2 for i in range(32)]], np.float32)
    y, s = oracle.matmul("q4_0", w, x, 32, 2)
    r0 = Fraction(0)
    r1 = Fraction(0)
    for i in range(16):
        r0 += (i - 8) * ((i % 5) - 2) + (((i + 3) % 16) - 8) * (((i + 16) % 5) - 2)
        r1 += Fraction(-1, 4) * ((15 - i - 8) * ((i % 5) - 2) + (0 - 8) * (((i + 16) % 5) - 2))
    assert y[0, 0] == float(r0) and y[0, 1] == float(r1)


def test_matmul_matches_numpy_product_of_dequantized():
    """Dequantize-then-dot equals numpy's f64 matmul of the oracle's own weights,
    checked on multi-token inputs (catches a transposed operand or token stride)."""
    rng = np.random.default_rng(5)
    for fmt, k, n, nt in (("q4_0", 96, 7, 3), ("q4_k", 512, 5, 4), ("q6_k", 256, 9, 2),
                          ("bf16", 40, 6, 3), ("f16", 24, 4, 5)):
        w = qmm_synth.gen_weights(fmt, k, n, rng)
        x = qmm_synth.gen_x(nt, k, rng)
        deq = oracle.dequant(fmt, w, k, n).astype(np.float64)
        y, s = oracle.matmul(fmt, w, x, k, n)
        ref = x.astype(np.float64) @ deq.T
        np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(s, np.abs(x.astype(np.float64)) @ np.abs(deq.T), rtol=1e-12)


def test_blas_variant_equals_loop_oracle():
    rng = np.random.default_rng(8)
    for fmt, k, n, nt in (("q4_k", 512, 9, 3), ("bf16", 64, 5, 2), ("q6_k", 256, 4, 5)):
        w = qmm_synth.gen_weights(fmt, k, n, rng)
        x = qmm_synth.gen_x(nt, k, rng)
        y, s = oracle.matmul(fmt, w, x, k, n)
        yb, sb = oracle.matmul_blas(fmt, w, x, k, n)
        np.testing.assert_allclose(yb, y, rtol=1e-12, atol=1e-12 * float(np.max(s)))
        np.testing.assert_allclose(sb, s, rtol=1e-12)


def test_sampled_equals_full():
    rng = np.random.default_rng(6)
    w = qmm_synth.gen_weights("q6_k", 512, 11, rng)
    x = qmm_synth.gen_x(3, 512, rng)
    y, s = oracle.matmul("q6_k", w, x, 512, 11)
    t = np.array([0, 2, 1, 2])
    j = np.array([10, 0, 5, 7])
    ys, ss = oracle.matmul_sampled("q6_k", w, x, 512, 11, t, j)
    assert np.array_equal(ys, y[t, j]) and np.array_equal(ss, s[t, j])


def test_k_zero_gives_zero():
    y, s = oracle.matmul("bf16", np.zeros(0, np.uint8), np.zeros((2, 0), np.float32), 0, 3)
    assert np.all(y == 0) and np.all(s == 0)


# ------------------------------------------------- acceptance checker ----

def test_checker_catches_a_dropped_term():
    """A mistake planted in the oracle's output (one product term dropped from
    one output) must fail the 1e-4 * sum|x w| bar at the configs' k."""
    rng = np.random.default_rng(7)
    k, n = 4096, 64
    w = qmm_synth.gen_weights("q4_k", k, n, rng)
    x = qmm_synth.gen_x(1, k, rng)
    y, s = oracle.matmul("q4_k", w, x, k, n)
    deq = oracle.dequant("q4_k", w, k, n)
    ok, _, _, _ = oracle.check(y, y, s)
    assert ok
    i = int(np.argmax(np.abs(x[0] * deq[3])))
    bad = y.copy()
    bad[0, 3] -= float(x[0, i]) * float(deq[3, i])
    ok, worst, _, _ = oracle.check(bad, y, s)
    assert not ok and worst > 1e-4


def test_checker_catches_plausible_kernel_mistakes():
    """Outputs a faulty kernel would plausibly produce, built from the oracle's
    own weights, must each fail the acceptance check at the configs' k: one
    32-weight unit skipped, output columns shifted by one, two tokens swapped,
    a ragged last tile left unwritten, sub-block 2 of every super-block read
    with scale sc + 1 (a decoder slip repeats in every row), and zero point 7
    instead of 8 in the Q4_0 blocks at one position of every row. A slip
    confined to one sub-block of one row is below the bar's resolution (it
    moves one output by about 1e-5 of S here): the bit-exact dequant tests are
    what see those."""
    rng = np.random.default_rng(17)
    k, n, nt = 4096, 64, 3
    w = qmm_synth.gen_weights("q4_k", k, n, rng)
    x = qmm_synth.gen_x(nt, k, rng).astype(np.float64)
    y, s = oracle.matmul("q4_k", w, x.astype(np.float32), k, n)
    deq = oracle.dequant("q4_k", w, k, n).astype(np.float64)
    assert oracle.check(y, y, s)[0]
    bad = []
    u = int(np.argmax(np.abs((x[0].reshape(-1, 32) * deq[5].reshape(-1, 32)).sum(1))))
    b = y.copy(); b[0, 5] -= x[0, 32 * u:32 * u + 32] @ deq[5, 32 * u:32 * u + 32]; bad.append(b)
    b = y.copy(); b[:, 1:] = y[:, :-1]; bad.append(b)
    b = y.copy(); b[[0, 1]] = y[[1, 0]]; bad.append(b)
    b = y.copy(); b[:, 60:] = 0.0; bad.append(b)
    # d * q of sub-block 2 (low nibbles of quant bytes 32..63, quant bytes at 16)
    blk = w.reshape(n, k // 256, 144)
    dsb = np.ascontiguousarray(blk[:, :, 0:2]).view("<f2")[..., 0].astype(np.float64)
    q2 = (blk[:, :, 16 + 32:16 + 64] & 15).astype(np.float64)
    d2 = deq.copy().reshape(n, k // 256, 256)
    d2[:, :, 64:96] += dsb[:, :, None] * q2                # sc read as sc + 1
    b = x @ d2.reshape(n, k).T; bad.append(b)
    for i, yb in enumerate(bad):
        ok, worst, cos, msg = oracle.check(yb, y, s)
        assert not ok, (i, msg)
    w0 = qmm_synth.gen_weights("q4_0", k, n, rng)
    y0, s0 = oracle.matmul("q4_0", w0, x.astype(np.float32), k, n)
    dq0 = oracle.dequant("q4_0", w0, k, n).astype(np.float64)
    dblk = np.ascontiguousarray(w0.reshape(n, -1, 18)[:, 10, 0:2]).view("<f2")[:, 0]
    d3 = dq0.copy(); d3[:, 320:352] += dblk.astype(np.float64)[:, None]  # (q - 7) d
    assert not oracle.check(x @ d3.T, y0, s0)[0]
    # the resolution limit stated above
    d4 = deq.copy(); d4[7, 64:96] *= 1.0 + 1.0 / 32.0
    b = y.copy(); b[:, 7] = x @ d4[7]
    assert oracle.check(b, y, s)[0]


def test_checker_catches_sign_flip_by_cosine():
    y = np.linspace(-1, 1, 101)[None, :]
    s = np.full_like(y, 1e9)  # elementwise bar loose: cosine must catch it
    ok, _, cos, _ = oracle.check(-y, y, s)
    assert not ok and cos < 0


def test_cosine_zero_vectors():
    z = np.zeros(5)
    assert oracle.cosine(z, z) == 1.0
    assert oracle.cosine(z, np.ones(5)) == 0.0


def test_checker_cosine_floor_between_0_999_and_0_9999():
    """Errors inside the elementwise bar (S large against y) still fail when
    the direction drifts: cosine 0.99953 is below the 0.9999 floor, cosine
    0.999950 above it (both in closed form: (1 + a) / sqrt(2 (1 + a^2)))."""
    y_ref = np.array([[1.0, 1.0]])
    s_ref = np.full_like(y_ref, 1e4)  # bar 1.0 per element
    for a, want_ok in ((1.063, False), (1.02, True)):
        cos_exact = (1 + a) / np.sqrt(2 * (1 + a * a))
        ok, _, cos, _ = oracle.check(np.array([[1.0, a]]), y_ref, s_ref)
        assert abs(cos - cos_exact) < 1e-12
        assert ok == want_ok, (a, cos)
    assert 0.999 < (1 + 1.063) / np.sqrt(2 * (1 + 1.063 ** 2)) < 0.9999


def test_checker_nan_positions_must_agree():
    """A NaN reference (a NaN weight) must come out NaN, at the same place."""
    y_ref = np.array([[np.nan, 1.0, 2.0]])
    s_ref = np.array([[1.0, 1.0, 2.0]])
    ok, *_ = oracle.check(np.array([[np.nan, 1.0, 2.0]]), y_ref, s_ref)
    assert ok
    ok, *_ = oracle.check(np.array([[0.0, 1.0, 2.0]]), y_ref, s_ref)
    assert not ok
    ok, *_ = oracle.check(np.array([[1.0, np.nan, 2.0]]), np.array([[1.0, 1.0, 2.0]]), s_ref)
    assert not ok


def test_tiled_semantics():
    y_ref = np.arange(12, dtype=np.float64).reshape(2, 6)
    s_ref = np.ones_like(y_ref)
    y_in = np.full((2, 6), 100.0)
    y, s = oracle.tiled(y_ref, s_ref, 2, 4, True, y_in)
    assert np.array_equal(y[:, 2:4], 100 + y_ref[:, 2:4])
    assert np.array_equal(y[:, :2], y_in[:, :2]) and np.array_equal(y[:, 4:], y_in[:, 4:])
    assert np.array_equal(s[:, 2:4], 101 * np.ones((2, 2)))
    y, s = oracle.tiled(y_ref, s_ref, 0, 6, False, y_in)
    assert np.array_equal(y, y_ref)


# ------------------------------------------------- backward w.r.t. input ----

def test_back_input_brute_force_tiny_q4_0():
    """Hand-listed dx for the 2-row Q4_0 weights of the forward brute-force pin:
    dx[i] = 3 * w0[i] - 2 * w1[i] (row 1 has d = -0.25 and zero high nibbles)."""
    w = np.zeros(36, np.uint8)
    w[0:2] = [0x00, 0x3C]                    # d = 1
    w[2:18] = [(i % 16) | (((i + 3) % 16) << 4) for i in range(16)]
    w[18:20] = [0x00, 0xB4]                  # d = -0.25
    w[20:36] = [15 - i for i in range(16)]
    dx, s = oracle.matmul_back_input("q4_0", w, np.array([3.0, -2.0], np.float32), 32, 2)
    want = []
    for i in range(32):
        w0 = (i - 8) if i < 16 else (((i - 16 + 3) % 16) - 8)
        w1 = Fraction(-1, 4) * ((15 - i - 8) if i < 16 else (0 - 8))
        want.append(3 * w0 - 2 * w1)
    assert [Fraction(v) for v in dx] == want
    assert s[0] == abs(3 * (0 - 8)) + abs(2 * Fraction(-1, 4) * (15 - 8))


@pytest.mark.parametrize("fmt,k,n", [("q4_0", 64, 7), ("q4_k", 512, 5), ("q6_k", 256, 6),
                                     ("bf16", 40, 9), ("f16", 24, 3)])
def test_back_input_one_hot_dy_picks_a_row(fmt, k, n):
    """dy = e_j gives dx = row j of the dequantized weights, exactly."""
    rng = np.random.default_rng(11)
    w = qmm_synth.gen_weights(fmt, k, n, rng)
    deq = oracle.dequant(fmt, w, k, n)
    for j in (0, n - 1, n // 2):
        dy = np.zeros(n, np.float32)
        dy[j] = 1.0
        dx, s = oracle.matmul_back_input(fmt, w, dy, k, n)
        assert np.array_equal(dx, deq[j].astype(np.float64))
        assert np.array_equal(s, np.abs(deq[j]).astype(np.float64))


@pytest.mark.parametrize("fmt,k,n", [("q4_k", 512, 33), ("q6_k", 512, 17), ("q4_0", 96, 20)])
def test_back_input_is_the_adjoint_of_the_forward(fmt, k, n):
    """dy . (W x) == x . (W^T dy): ties the transposed product to the pinned
    forward one (a swapped index or operand breaks it)."""
    rng = np.random.default_rng(5)
    w = qmm_synth.gen_weights(fmt, k, n, rng)
    x = rng.standard_normal(k).astype(np.float32)
    dy = rng.standard_normal(n).astype(np.float32)
    y, _ = oracle.matmul(fmt, w, x, k, n)
    dx, _ = oracle.matmul_back_input(fmt, w, dy, k, n)
    lhs = float(np.dot(dy.astype(np.float64), y[0]))
    rhs = float(np.dot(x.astype(np.float64), dx))
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, float(np.abs(dy) @ np.abs(y[0])))


def test_back_input_sum_axis_tiles_add_up():
    """Tiles [0, m) and [m, n) of the sum axis add to the whole; an empty tile
    is zero; the blas variant agrees with the loop oracle."""
    fmt, k, n = "q6_k", 256, 40
    rng = np.random.default_rng(9)
    w = qmm_synth.gen_weights(fmt, k, n, rng)
    dy = rng.standard_normal(n).astype(np.float32)
    full, sf = oracle.matmul_back_input(fmt, w, dy, k, n)
    a, sa = oracle.matmul_back_input(fmt, w, dy, k, n, 0, 13)
    b, sb = oracle.matmul_back_input(fmt, w, dy, k, n, 13, n)
    np.testing.assert_allclose(a + b, full, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(sa + sb, sf, rtol=1e-12, atol=1e-12)
    z, sz = oracle.matmul_back_input(fmt, w, dy, k, n, 7, 7)
    assert not z.any() and not sz.any()
    c, sc = oracle.matmul_back_input_blas(fmt, w, dy, k, n, 13, n)
    np.testing.assert_allclose(c, b, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(sc, sb, rtol=1e-12)
    with pytest.raises(ValueError):
        oracle.matmul_back_input(fmt, w, dy, k, n, 10, 5)


# ------------------------------------------------- Q8_0, Q5_0 and experts ----

def test_q8_0_and_q5_0_row_bytes():
    for k in (0, 32, 64, 2048):
        assert oracle.row_bytes("q8_0", k) == (k // 32) * 34
        assert oracle.row_bytes("q5_0", k) == (k // 32) * 22
    assert oracle.row_bytes("q8_0", 48) == 0 and oracle.row_bytes("q5_0", 16) == 0


def test_q8_0_hand_packed():
    """d = 0.5 (f16 0x3800) and codes -16 .. 15 as signed bytes."""
    blk = np.zeros(34, np.uint8)
    blk[0:2] = [0x00, 0x38]
    codes = np.arange(-16, 16, dtype=np.int64)
    blk[2:34] = codes.astype(np.int8).view(np.uint8)
    w = oracle.dequant("q8_0", blk, 32, 1)[0]
    assert list(w) == [0.5 * c for c in range(-16, 16)]
    blk[2] = 0x80  # -128
    assert oracle.dequant("q8_0", blk, 32, 1)[0][0] == -64.0


def _pack_q5_0(d_bytes, q):
    """Pack 32 five-bit codes: element i < 16 -> low nibble of byte i and bit i
    of the high-bit word; element i + 16 -> high nibble and bit i + 16."""
    blk = np.zeros(22, np.uint8)
    blk[0:2] = d_bytes
    qh = 0
    for i in range(32):
        qh |= ((int(q[i]) >> 4) & 1) << i
    blk[2:6] = [(qh >> (8 * b)) & 0xFF for b in range(4)]
    for i in range(16):
        blk[6 + i] = (int(q[i]) & 15) | ((int(q[i + 16]) & 15) << 4)
    return blk


def test_q5_0_hand_packed():
    """Every code 0..31 once (a permutation, so a wrong bit index or nibble
    order moves values), d = 1 then d = -0.25."""
    q = np.random.default_rng(0).permutation(32)
    w = oracle.dequant("q5_0", _pack_q5_0([0x00, 0x3C], q), 32, 1)[0]
    assert list(w) == [float(v - 16) for v in q]
    w = oracle.dequant("q5_0", _pack_q5_0([0x00, 0xB4], q), 32, 1)[0]
    assert list(w) == [-0.25 * (v - 16) for v in q]


@pytest.mark.parametrize("fmt", ["q8_0", "q5_0"])
def test_new_formats_product_matches_numpy(fmt):
    rng = np.random.default_rng(2)
    k, n = 96, 7
    w = qmm_synth.gen_weights(fmt, k, n, rng)
    x = rng.standard_normal((3, k)).astype(np.float32)
    y, s = oracle.matmul(fmt, w, x, k, n)
    deq = oracle.dequant(fmt, w, k, n).astype(np.float64)
    np.testing.assert_allclose(y, x.astype(np.float64) @ deq.T, rtol=1e-12, atol=1e-12)


def test_experts_product_selects_slices():
    """Row (p, s) of the expert product equals the plain product of x[p] with
    the slice ids[p, s] cut out of the stacked bytes by hand; a bad id is
    rejected."""
    fmt, k, n, n_exp = "q5_0", 64, 5, 6
    rng = np.random.default_rng(4)
    w = qmm_synth.gen_weights(fmt, k, n * n_exp, rng)
    x = rng.standard_normal((3, k)).astype(np.float32)
    ids = np.array([[4, 0], [5, 2], [1, 3]], np.int32)
    y, s = oracle.matmul_experts(fmt, w, x, k, n, n_exp, ids)
    sl = oracle.row_bytes(fmt, k) * n
    for p in range(3):
        for t in range(2):
            e = ids[p, t]
            ye, se = oracle.matmul(fmt, w[e * sl:(e + 1) * sl], x[p], k, n)
            assert np.array_equal(y[p * 2 + t], ye[0]) and np.array_equal(s[p * 2 + t], se[0])
    with pytest.raises(ValueError):
        oracle.matmul_experts(fmt, w, x, k, n, n_exp, np.array([[6, 0], [0, 0], [0, 0]], np.int32))



# ------------------------------------------------- MLX-style affine rows ----

BF16_ONE, BF16_MINUS_ONE, BF16_HALF, BF16_TWO = 0x3F80, 0xBF80, 0x3F00, 0x4000


def _words_le(words):
    return np.array(words, dtype="<u4").view(np.uint8)


def test_affine_row_bytes():
    for k in (64, 128, 4096):
        assert oracle.affine_row_bytes(4, k) == k // 2
        assert oracle.affine_row_bytes(8, k) == k
    assert oracle.affine_row_bytes(4, 32) < 0 and oracle.affine_row_bytes(3, 64) < 0


def test_affine4_hand_packed_code_order():
    """Words 0x76543210, 0xFEDCBA98: codes 0..15 in order (lowest nibble
    first); scale 1, bias -1 give q - 1 exactly."""
    w = _words_le([0x76543210, 0xFEDCBA98] * 4)
    got = oracle.dequant_affine(4, w, np.array([BF16_ONE], np.uint16),
                                np.array([BF16_MINUS_ONE], np.uint16), 64, 1)[0]
    assert list(got) == [float(q - 1) for q in list(range(16)) * 4]


def test_affine8_hand_packed_code_order():
    """Bytes 0..63 (four codes per word, lowest byte first); scale 2^-7 (bf16
    0x3C00), bias 0: value i / 128."""
    w = np.arange(64, dtype=np.uint8)
    got = oracle.dequant_affine(8, w, np.array([0x3C00], np.uint16), np.array([0], np.uint16), 64, 1)[0]
    assert list(got) == [i / 128 for i in range(64)]
    w = np.full(64, 255, np.uint8)
    got = oracle.dequant_affine(8, w, np.array([BF16_ONE], np.uint16), np.array([BF16_HALF], np.uint16), 64, 1)[0]
    assert np.all(got == 255.5)


def test_affine_group_index():
    """Two rows of two groups: each group of 64 takes its own scale and bias,
    row-major [n, k/64]."""
    k, n = 128, 2
    w = _words_le([0x11111111] * 32)            # every code 1
    scales = np.array([[BF16_ONE, BF16_TWO], [BF16_HALF, BF16_ONE]], np.uint16)
    biases = np.array([[0, BF16_HALF], [BF16_MINUS_ONE, BF16_TWO]], np.uint16)
    got = oracle.dequant_affine(4, w, scales, biases, k, n)
    assert np.all(got[0, :64] == 1.0) and np.all(got[0, 64:] == 2.5)
    assert np.all(got[1, :64] == -0.5) and np.all(got[1, 64:] == 3.0)


def test_affine_4bit_and_8bit_agree_on_small_codes():
    """The same codes (< 16) packed at 4 and at 8 bits decode alike."""
    rng = np.random.default_rng(8)
    k, n = 192, 3
    codes = rng.integers(0, 16, size=(n, k))
    w8 = codes.astype(np.uint8).reshape(-1)
    w4 = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8).reshape(-1)
    _, scales, biases = qmm_synth.gen_affine(4, k, n, rng)
    a = oracle.dequant_affine(4, w4, scales, biases, k, n)
    b = oracle.dequant_affine(8, w8, scales, biases, k, n)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_affine_value_rounds_once():
    """code 1, scale 1, bias 2^-24 + 2^-30: the exact value lies just above
    half an f32 ulp past 1 and must round up to 1 + 2^-23 (one rounding of
    the exact value); bias bf16 pattern 0x3382 = 2^-24 * (1 + 2^-6)."""
    w = _words_le([0x00000001] + [0] * 7)
    got = oracle.dequant_affine(4, w, np.array([BF16_ONE], np.uint16), np.array([0x3382], np.uint16), 64, 1)[0]
    exact = Fraction(1) + Fraction(1, 2 ** 24) + Fraction(1, 2 ** 30)
    assert oracle.bf16_value(0x3382) == float(Fraction(1, 2 ** 24) + Fraction(1, 2 ** 30))
    assert float(exact) != 1.0 + 2.0 ** -23
    assert got[0] == np.float32(1.0 + 2.0 ** -23)
    assert got[1] == np.float32(2.0 ** -24 + 2.0 ** -30)   # code 0: the bias alone


@pytest.mark.parametrize("bits", [4, 8])
def test_affine_product_closed_form(bits):
    """Every code c: y = sum_g (c s_g + b_g) sum_{i in g} x_i, in fractions."""
    k, n, c = 256, 2, (5 if bits == 4 else 200)
    per = 32 // bits
    word = sum(c << (bits * i) for i in range(per))
    w = _words_le([word] * (n * k * bits // 32))
    rng = np.random.default_rng(6)
    _, scales, biases = qmm_synth.gen_affine(bits, k, n, rng)
    x = rng.standard_normal((2, k)).astype(np.float32)
    y, s = oracle.matmul_affine(bits, w, scales, biases, x, k, n)
    for t in range(2):
        for j in range(n):
            tot = Fraction(0)
            for g in range(k // 64):
                sc = Fraction(float(oracle.bf16_value(scales[j, g])))
                bi = Fraction(float(oracle.bf16_value(biases[j, g])))
                v = Fraction(float(np.float32(float(c * sc + bi))))   # the weight, rounded once
                tot += v * sum(Fraction(float(xv)) for xv in x[t, 64 * g:64 * g + 64])
            assert abs(Fraction(y[t, j]) - tot) <= Fraction(1, 10 ** 9) * (1 + abs(tot))


def test_affine_product_matches_numpy_and_sampled():
    rng = np.random.default_rng(9)
    k, n = 192, 11
    w, scales, biases = qmm_synth.gen_affine(4, k, n, rng)
    x = rng.standard_normal((3, k)).astype(np.float32)
    y, s = oracle.matmul_affine(4, w, scales, biases, x, k, n)
    deq = oracle.dequant_affine(4, w, scales, biases, k, n).astype(np.float64)
    np.testing.assert_allclose(y, x.astype(np.float64) @ deq.T, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s, np.abs(x.astype(np.float64)) @ np.abs(deq).T, rtol=1e-12)
    ti, ji = np.array([0, 2, 1]), np.array([10, 0, 5])
    ys, ss = oracle.matmul_affine_sampled(4, w, scales, biases, x, k, n, ti, ji)
    assert np.array_equal(ys, y[ti, ji]) and np.array_equal(ss, s[ti, ji])
    # the library-product variant used for full-size checks gives the same (y, S)
    yb, sb = oracle.matmul_affine_blas(4, w, scales, biases, x, k, n)
    np.testing.assert_allclose(yb, y, rtol=1e-12, atol=1e-12 * float(np.max(s)))
    np.testing.assert_allclose(sb, s, rtol=1e-12)



# ------------------------------------------------------- gated products ----

def test_activation_odd_part_identity():
    """act(g) - act(-g) = g for both (sigmoid(g) + sigmoid(-g) = 1, and the
    same for the tanh form): a sign or constant slip breaks it."""
    for name in ("swiglu", "geglu"):
        for g in (0.0, 0.3, 1.0, 2.5, 7.0, 30.0):
            assert abs(oracle.act(name, g) - oracle.act(name, -g) - g) <= 1e-12 * max(1.0, g)


def test_silu_against_library_sigmoid():
    from scipy.special import expit
    for g in np.linspace(-40, 40, 161):
        assert abs(oracle.act("swiglu", g) - g * expit(g)) <= 1e-14 * max(1.0, abs(g))
    assert oracle.act("swiglu", 0.0) == 0.0


def test_gelu_tanh_form_against_erf_gelu_and_sigmoid_identity():
    """The tanh form stays within 5e-4 of the erf GELU everywhere, equals
    g * sigmoid(2 z) with z its tanh argument (0.5 (1 + tanh z) = sigmoid(2z)),
    and gelu(1) = 0.8411919906 (the published tanh-form value)."""
    from scipy.special import erf, expit
    c = np.sqrt(2.0 / np.pi)
    for g in np.linspace(-10, 10, 401):
        v = oracle.act("geglu", g)
        assert abs(v - 0.5 * g * (1 + erf(g / np.sqrt(2)))) <= 5e-4
        assert abs(v - g * expit(2 * c * (g + 0.044715 * g ** 3))) <= 1e-13 * max(1.0, abs(g))
    assert abs(oracle.act("geglu", 1.0) - 0.8411919906) < 1e-10


def test_gelu_stable_form_matches_the_literal_tanh_form():
    """Where 0.5 g (1 + tanh z) is still accurate in double (|z| < 3), it and
    the oracle's g / (1 + e^(-2z)) agree to rounding; far into the negative
    tail the oracle keeps relative precision (it equals g e^(2z) to first order)."""
    c = np.sqrt(2.0 / np.pi)
    for g in np.linspace(-2.5, 2.5, 101):
        z = c * (g + 0.044715 * g ** 3)
        assert abs(oracle.act("geglu", g) - 0.5 * g * (1 + np.tanh(z))) <= 1e-15
    for g in (-8.0, -12.0, -20.0):
        z = c * (g + 0.044715 * g ** 3)
        v = oracle.act("geglu", g)
        assert v < 0 and abs(v / (g * np.exp(2 * z)) - 1) < 1e-6


def test_checker_absolute_floor():
    y_ref = np.array([[1e-40, 1.0]])
    s_ref = np.array([[1e-41, 1.0]])
    ok, *_ = oracle.check(np.array([[0.0, 1.0]]), y_ref, s_ref)
    assert not ok
    ok, *_ = oracle.check(np.array([[0.0, 1.0]]), y_ref, s_ref, atol=oracle.FLT_MIN)
    assert ok
    ok, *_ = oracle.check(np.array([[0.0, 1.001]]), y_ref, s_ref, atol=oracle.FLT_MIN)
    assert not ok


def test_activation_derivatives_by_central_differences():
    for name in ("swiglu", "geglu"):
        for g in (-6.0, -1.3, -0.2, 0.0, 0.4, 1.7, 5.0):
            h = 1e-5
            fd = (oracle.act(name, g + h) - oracle.act(name, g - h)) / (2 * h)
            assert abs(oracle.act_deriv(name, g) - fd) < 1e-7


@pytest.mark.parametrize("name", ["swiglu", "geglu"])
def test_glu_product_composes_the_plain_products(name):
    rng = np.random.default_rng(31)
    fmt, k, n = "q4_k", 512, 9
    wg = qmm_synth.gen_weights(fmt, k, n, rng)
    wu = qmm_synth.gen_weights(fmt, k, n, rng)
    x = rng.standard_normal((2, k)).astype(np.float32)
    y, s = oracle.matmul_glu(name, fmt, wg, wu, x, k, n)
    g, sg = oracle.matmul(fmt, wg, x, k, n)
    u, su = oracle.matmul(fmt, wu, x, k, n)
    for t in range(2):
        for j in range(n):
            a = oracle.act(name, g[t, j])
            assert y[t, j] == a * u[t, j]
            exp_s = abs(oracle.act_deriv(name, g[t, j])) * abs(u[t, j]) * sg[t, j] + abs(a) * su[t, j]
            assert s[t, j] == exp_s
    # swapping gate and up changes the result (the gate is the activated one)
    y2, _ = oracle.matmul_glu(name, fmt, wu, wg, x, k, n)
    assert not np.allclose(y, y2)


# ------------------------------------- a second, per-element decoder ----

def _f16(lo, hi):
    return np.array([lo | (hi << 8)], np.uint16).view(np.float16).astype(np.float64)[0]


def _element_decoder(fmt, blk, e):
    """Weight e of one block, from an index formula per element (written
    independently of the oracle's block loops); f64, rounded to f32 once."""
    b = [int(v) for v in blk]
    if fmt == "q4_0":
        q = (b[2 + e % 16] >> (4 * (e // 16))) & 15
        return np.float32((q - 8) * _f16(b[0], b[1]))
    if fmt == "q8_0":
        q = b[2 + e] - 256 * (b[2 + e] >= 128)
        return np.float32(q * _f16(b[0], b[1]))
    if fmt == "q5_0":
        qh = b[2] | (b[3] << 8) | (b[4] << 16) | (b[5] << 24)
        q = ((b[6 + e % 16] >> (4 * (e // 16))) & 15) | (((qh >> e) & 1) << 4)
        return np.float32((q - 16) * _f16(b[0], b[1]))
    if fmt == "q4_k":
        s = e // 32
        sc_b = b[4:16]
        if s < 4:
            sc, m = sc_b[s] & 63, sc_b[s + 4] & 63
        else:
            sc = (sc_b[s + 4] & 15) | ((sc_b[s - 4] >> 6) << 4)
            m = (sc_b[s + 4] >> 4) | ((sc_b[s] >> 6) << 4)
        q = (b[16 + 32 * (e // 64) + e % 32] >> (4 * (s % 2))) & 15
        return np.float32(_f16(b[0], b[1]) * sc * q - _f16(b[2], b[3]) * m)
    if fmt == "q6_k":
        h, rem = e // 128, e % 128
        r, l = rem // 32, rem % 32
        lo = b[64 * h + l + 32 * (r % 2)]
        lo = (lo >> 4) if r >= 2 else (lo & 15)
        hi = (b[128 + 32 * h + l] >> (2 * r)) & 3
        q = lo | (hi << 4)
        sc = b[192 + e // 16] - 256 * (b[192 + e // 16] >= 128)
        return np.float32(_f16(b[208], b[209]) * sc * (q - 32))
    raise ValueError(fmt)


@pytest.mark.parametrize("fmt,elems,nbytes", [("q4_0", 32, 18), ("q8_0", 32, 34), ("q5_0", 32, 22),
                                              ("q4_k", 256, 144), ("q6_k", 256, 210)])
def test_per_element_decoder_agrees_bit_for_bit(fmt, elems, nbytes):
    """Random blocks (every byte uniform: NaN, Inf and subnormal scales
    included): the oracle's block decoder and the per-element index formula
    give the same bits for every weight."""
    rng = np.random.default_rng(elems + nbytes)
    nblk = 24
    w = rng.integers(0, 256, size=nblk * nbytes, dtype=np.uint8)
    got = oracle.dequant(fmt, w, elems * nblk, 1)[0]
    with np.errstate(invalid="ignore", over="ignore"):   # Inf * 0 scales give NaN on both sides
        want = np.array([_element_decoder(fmt, w[nbytes * (i // elems):nbytes * (i // elems + 1)],
                                          i % elems) for i in range(elems * nblk)], np.float32)
    na, nb = np.isnan(got), np.isnan(want)
    assert np.array_equal(na, nb)
    assert np.array_equal(got.view(np.uint32)[~na], want.view(np.uint32)[~na])
