"""The seeded inputs follow their stated recipes: shapes, seeds, value ranges
and distributions of every named workload. Fields are read back with numpy's
own f16 / bf16 views, independently of both the oracle and the CUDA path.
CPU only; shrunken row counts keep it fast (each recipe is per element, so a
few rows show the same distribution as the full matrix)."""
import numpy as np
import pytest

import qmm_synth as S

# name -> (fmt, k, n, n_tokens, seed, x distribution, output tiles)
RECIPES = {
    "q4_0_gemv": ("q4_0", 256, 512, 1, 1, "uniform", 1),
    "bf16_gemv": ("bf16", 4096, 4096, 1, 2, "normal", 1),
    "f16_gemv": ("f16", 4096, 4096, 1, 2, "normal", 1),
    "q4_k_gemv": ("q4_k", 4096, 14336, 1, 3, "normal", 1),
    "q6_k_head": ("q6_k", 2560, 262144, 1, 4, "normal", 8),
    "q4_k_prefill": ("q4_k", 4096, 14336, 512, 5, "normal", 1),
    "q8_0_gemv": ("q8_0", 4096, 14336, 1, 8, "normal", 1),
    "q5_0_gemv": ("q5_0", 4096, 14336, 1, 9, "normal", 1),
}
EXPERT_RECIPES = {  # (fmt, k, n, n_experts, top_k, n_pos, seed)
    "q8_0_experts": ("q8_0", 2048, 768, 64, 8, 1, 6),
    "q5_0_experts": ("q5_0", 2048, 768, 64, 8, 1, 7),
    "q4_k_experts": ("q4_k", 2048, 768, 64, 8, 1, 14),
}
AFFINE_RECIPES = {  # (bits, k, n, n_tokens, seed)
    "affine4_gemv": (4, 4096, 14336, 1, 10),
    "affine8_gemv": (8, 4096, 14336, 1, 11),
    "affine4_prefill": (4, 4096, 14336, 512, 12),
    "affine8_prefill": (8, 4096, 14336, 512, 13),
}
# the f16 fields of each block: (byte offset, lower, upper end of the uniform draw)
SCALE_FIELDS = {
    "q4_0": [(0, 0.005, 0.05)],
    "q4_k": [(0, 0.001, 0.02), (2, 0.001, 0.02)],
    "q6_k": [(208, 0.0005, 0.01)],
    "q8_0": [(0, 0.002, 0.02)],
    "q5_0": [(0, 0.005, 0.05)],
}
# bytes drawn uniformly from 0..255: (first, last + 1) within a block
UNIFORM_BYTES = {
    "q4_0": (2, 18), "q4_k": (4, 144), "q6_k": (0, 192), "q8_0": (2, 34), "q5_0": (2, 22),
}


def _chi2_uniform(values, n_bins):
    counts = np.bincount(values.ravel(), minlength=n_bins).astype(np.float64)
    e = values.size / n_bins
    return float(((counts - e) ** 2 / e).sum())


def test_workload_tables_match_the_recipes():
    assert S.WORKLOADS == RECIPES
    assert S.EXPERT_WORKLOADS == EXPERT_RECIPES
    assert S.AFFINE_WORKLOADS == AFFINE_RECIPES


@pytest.mark.parametrize("name", sorted(RECIPES))
def test_workload_shapes_and_seed(name):
    fmt, k, n, nt, seed, xdist, _ = RECIPES[name]
    n_small = 8
    f, kk, nn, w, x = S.workload(name, n=n_small, n_tokens=min(nt, 4))
    assert (f, kk, nn) == (fmt, k, n_small)
    assert w.dtype == np.uint8 and w.size == S.row_bytes(fmt, k) * n_small
    assert x.dtype == np.float32 and x.shape == (min(nt, 4), k)
    # seeded: the same call gives the same bytes; the draw is numpy's PCG64 stream
    w2 = S.workload(name, n=n_small, n_tokens=min(nt, 4))[3]
    assert np.array_equal(w, w2)
    rng = np.random.default_rng(seed)
    assert np.array_equal(w, S.gen_weights(fmt, k, n_small, rng))


@pytest.mark.parametrize("fmt", sorted(SCALE_FIELDS))
def test_block_scales_lie_in_their_ranges(fmt):
    k = 256 * 4 if fmt in ("q4_k", "q6_k") else 32 * 32
    rows = 64
    blk = S.gen_weights(fmt, k, rows, np.random.default_rng(99)).reshape(-1, S.BLOCK_BYTES[fmt])
    for off, lo, hi in SCALE_FIELDS[fmt]:
        v = np.ascontiguousarray(blk[:, off:off + 2]).view("<f2").astype(np.float64).ravel()
        ulp = 2.0 ** -10  # relative f16 rounding of a normal value, both ways
        assert v.min() >= lo * (1 - ulp) and v.max() <= hi * (1 + ulp)
        span = hi - lo  # the draw fills its range: uniform, not a point
        assert v.min() < lo + 0.02 * span and v.max() > hi - 0.02 * span
        assert abs(v.mean() - (lo + hi) / 2) < 0.03 * span


@pytest.mark.parametrize("fmt", sorted(UNIFORM_BYTES))
def test_code_bytes_are_uniform(fmt):
    k = 256 * 4 if fmt in ("q4_k", "q6_k") else 32 * 32
    blk = S.gen_weights(fmt, k, 64, np.random.default_rng(98)).reshape(-1, S.BLOCK_BYTES[fmt])
    a, b = UNIFORM_BYTES[fmt]
    codes = blk[:, a:b]
    # 255 degrees of freedom: mean 255, sd about 22.6; a skewed draw lands far above
    assert _chi2_uniform(codes, 256) < 400
    nib = np.concatenate([codes & 15, codes >> 4]).ravel()
    assert _chi2_uniform(nib, 16) < 60  # 15 degrees of freedom


def test_q6_k_scales_are_int8_in_minus_32_to_31():
    blk = S.gen_weights("q6_k", 256 * 4, 256, np.random.default_rng(97)).reshape(-1, 210)
    sc = blk[:, 192:208].view(np.int8).astype(np.int64)
    assert sc.min() == -32 and sc.max() == 31
    assert _chi2_uniform(sc + 32, 64) < 150  # 63 degrees of freedom


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_16_bit_weights_are_normal_0_02(fmt):
    w = S.gen_weights(fmt, 4096, 64, np.random.default_rng(96)).view("<u2")
    if fmt == "bf16":
        v = (w.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    else:
        v = w.view("<f2").astype(np.float64)
    assert abs(v.mean()) < 5 * 0.02 / np.sqrt(v.size)  # five standard errors
    assert abs(v.std() / 0.02 - 1) < 0.01
    # Gaussian tails: about 4.55 % beyond two standard deviations
    assert abs(np.mean(np.abs(v) > 0.04) - 0.0455) < 0.003


def test_bf16_rounding_is_to_nearest_even():
    vals = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -9, -1.0 - 2.0 ** -8],
                    np.float32)
    # ties go to the even neighbour; below half an ulp rounds down
    want = np.array([0x3F80, 0x3F82, 0x3F80, 0xBF80], np.uint16)
    assert np.array_equal(S._bf16_bits_rne(vals), want)


def test_activations():
    xn = S.gen_x(64, 4096, np.random.default_rng(95))
    assert xn.dtype == np.float32 and abs(xn.mean()) < 0.01 and abs(xn.std() - 1) < 0.01
    xu = S.gen_x(64, 4096, np.random.default_rng(95), "uniform")
    assert xu.min() >= -1 and xu.max() < 1 and abs(xu.std() - 1 / np.sqrt(3)) < 0.01


def test_expert_ids_are_distinct_per_position_and_in_range():
    for name, (fmt, k, n, n_exp, top_k, n_pos, seed) in EXPERT_RECIPES.items():
        f, kk, nn, ne, w, x, ids = S.expert_workload(name, n_pos=16)
        assert (f, kk, nn, ne) == (fmt, k, n, n_exp)
        assert w.size == S.row_bytes(fmt, k) * n * n_exp
        assert ids.shape == (16, top_k) and ids.dtype == np.int32
        assert ids.min() >= 0 and ids.max() < n_exp
        assert all(len(set(r)) == top_k for r in ids.tolist())


def test_affine_scales_biases_and_codes():
    w, sc, bi = S.gen_affine(4, 4096, 64, np.random.default_rng(94))
    assert w.size == 64 * 4096 // 2 and sc.shape == bi.shape == (64, 4096 // 64)
    s = (sc.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    b = (bi.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    # fp32 draws truncated to bf16 move toward zero by less than 2^-7 relative
    assert s.min() >= 0.01 * (1 - 2.0 ** -7) and s.max() < 0.06
    assert b.min() >= -0.1 and b.max() < 0.1
    assert s.min() < 0.0105 and s.max() > 0.0595 and b.min() < -0.099 and b.max() > 0.099
    assert _chi2_uniform(np.concatenate([w & 15, w >> 4]), 16) < 60
    with pytest.raises(ValueError):
        S.gen_affine(4, 96, 2, np.random.default_rng(0))
    for name, (bits, k, n, nt, seed) in AFFINE_RECIPES.items():
        bb, kk, nn, w, sc, bi, x = S.affine_workload(name, n_tokens=2, n=4)
        assert (bb, kk, nn) == (bits, k, 4) and w.size == 4 * k * bits // 8 and x.shape == (2, k)


@pytest.mark.parametrize("fmt", ["q4_0", "q8_0", "q6_k", "q4_k"])
def test_constant_rows_repeat_one_weight(fmt):
    """set_constant_rows: every weight of a chosen row is the same value (read
    through the oracle's decoder), other rows are untouched."""
    import oracle
    oracle.build()
    k, n = 512, 7
    rng = np.random.default_rng(17)
    w = S.gen_weights(fmt, k, n, rng)
    rows = [1, 4, 6]
    w2 = S.set_constant_rows(fmt, w, k, rows)
    f, f2 = oracle.dequant(fmt, w, k, n), oracle.dequant(fmt, w2, k, n)
    for j in range(n):
        if j in rows:
            assert np.unique(f2[j]).size == 1 and f2[j][0] != 0.0
        else:
            assert np.array_equal(f[j], f2[j])
