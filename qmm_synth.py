"""Seeded synthetic inputs for the fused dequantize-and-multiply ``y = x @ W``.

This module only draws random numbers and lays them out as GGUF/ggml block
bytes; it holds none of the dequantization or matmul arithmetic. Both the
oracle (under ``oracle/``) and the CUDA path are fed from here, so the two
sides always see identical bytes.

Workload recipes (sizes, value distributions, seeds) follow the synthetic
stand-ins for the real-model shapes that the rullama ``matmul.rs`` tests use
(Gemma-4 projections, the vocab-sized output head):

* ``q4_0_gemv``     Q4_0, k=256, n=512; per-block f16 scale d ~ U[0.005, 0.05],
                    16 uniform quant bytes (so every nibble is uniform 0..15);
                    x ~ U[-1, 1]; seed 1.
* ``bf16_gemv`` / ``f16_gemv``
                    k=n=4096, w ~ N(0, 0.02) rounded to bf16 / f16
                    (round-to-nearest-even); x ~ N(0, 1); seed 2.
* ``q4_k_gemv``     Q4_K, k=4096, n=14336; d, dmin f16 ~ U[0.001, 0.02];
                    12 uniform packed-scale bytes (every 6-bit scale/min
                    uniform 0..63); 128 uniform quant bytes; x ~ N(0, 1); seed 3.
* ``q6_k_head``     Q6_K, k=2560, n=262144; ql/qh uniform bytes; int8 scales
                    uniform in [-32, 31]; f16 d ~ U[0.0005, 0.01]; x ~ N(0, 1);
                    seed 4; run as 8 output tiles of 32768 columns.
* ``q4_k_prefill``  Q4_K with the q4_k_gemv value distribution, N=512 tokens,
                    k=4096, n=14336; X ~ N(0, 1) [N x k]; seed 5 (also N=1, 8, 64).
* ``q8_0_experts`` / ``q5_0_experts`` / ``q4_k_experts``
                    expert-indexed decode: 64 stacked experts of n=768 rows,
                    k=2048, top_k = 8 experts per position, 1 position (also 4
                    and 64); Q8_0 d ~ U[0.002, 0.02] with uniform int8 codes,
                    Q5_0 d ~ U[0.005, 0.05] with uniform high-bit words and
                    nibbles, Q4_K with the q4_k_gemv distribution; ids drawn
                    without repetition per position; x ~ N(0, 1); seeds 6, 7, 14.
* ``q8_0_gemv`` / ``q5_0_gemv``
                    k=4096, n=14336, one token; the expert workloads' value
                    distributions; x ~ N(0, 1); seeds 8, 9.
* ``affine4_gemv`` / ``affine8_gemv`` / ``affine4_prefill`` / ``affine8_prefill``
                    MLX-style affine matrices, k=4096, n=14336, 1 or 512 tokens:
                    uniform code words, bf16 scales U[0.01, 0.06) and biases
                    U[-0.1, 0.1) per 64 weights (fp32 draws truncated to bf16);
                    x ~ N(0, 1); seeds 10-13.

Byte layouts written here (little-endian): Q4_0 block = f16 d then 16 quant
bytes (18 B); Q8_0 block = f16 d then 32 code bytes (34 B); Q5_0 block = f16 d,
a 4-byte high-bit word, 16 nibble bytes (22 B); Q4_K super-block = f16 d, f16 dmin, 12 scale bytes, 128 quant
bytes (144 B); Q6_K super-block = 128 ql bytes, 64 qh bytes, 16 int8 scales,
f16 d (210 B). BF16/F16 rows are plain 16-bit little-endian values.
"""
from __future__ import annotations

import numpy as np

FORMATS = ("bf16", "f16", "q4_0", "q4_k", "q6_k", "q8_0", "q5_0")

# elements per block and bytes per block of each format
BLOCK_ELEMS = {"bf16": 1, "f16": 1, "q4_0": 32, "q4_k": 256, "q6_k": 256, "q8_0": 32, "q5_0": 32}
BLOCK_BYTES = {"bf16": 2, "f16": 2, "q4_0": 18, "q4_k": 144, "q6_k": 210, "q8_0": 34, "q5_0": 22}


def row_bytes(fmt: str, k: int) -> int:
    """Bytes of one packed row of k weights (k must be a multiple of the block)."""
    return (k // BLOCK_ELEMS[fmt]) * BLOCK_BYTES[fmt]


def _f16_bytes(values: np.ndarray) -> np.ndarray:
    """f16 (round-to-nearest-even via numpy) as little-endian byte pairs."""
    h = values.astype(np.float16).astype("<f2")
    return h.view(np.uint8).reshape(values.shape + (2,))


def _bf16_bits_rne(values: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of f32 values, round-to-nearest-even (finite inputs)."""
    bits = values.astype(np.float32).view(np.uint32).astype(np.uint64)
    rounded = (bits + 0x7FFF + ((bits >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def gen_weights(fmt: str, k: int, n: int, rng: np.random.Generator, **dist) -> np.ndarray:
    """Packed weight bytes, shape [n * row_bytes(fmt, k)] uint8, row-major (row j = column j of W).

    Structure options: ``nonneg=True`` (bf16 / f16) draws |N(0, std)|;
    ``dmin_zero=True`` (q4_k) stores dmin = +0, so every min term vanishes and
    every weight is >= 0 (d and the codes stay as drawn)."""
    if fmt in ("bf16", "f16"):
        std = dist.get("std", 0.02)
        w = rng.normal(0.0, std, size=(n, k)).astype(np.float32)
        if dist.get("nonneg"):
            w = np.abs(w)
        if fmt == "bf16":
            bits = _bf16_bits_rne(w).astype("<u2")
        else:
            bits = w.astype(np.float16).astype("<f2").view("<u2")
        return np.ascontiguousarray(bits).view(np.uint8).reshape(-1)
    if fmt == "q4_0":
        lo, hi = dist.get("d_range", (0.005, 0.05))
        nb = k // 32
        blk = np.empty((n, nb, 18), np.uint8)
        blk[..., 0:2] = _f16_bytes(rng.uniform(lo, hi, size=(n, nb)))
        blk[..., 2:18] = rng.integers(0, 256, size=(n, nb, 16), dtype=np.uint8)
        return blk.reshape(-1)
    if fmt == "q4_k":
        lo, hi = dist.get("d_range", (0.001, 0.02))
        nb = k // 256
        blk = np.empty((n, nb, 144), np.uint8)
        blk[..., 0:2] = _f16_bytes(rng.uniform(lo, hi, size=(n, nb)))
        blk[..., 2:4] = _f16_bytes(rng.uniform(lo, hi, size=(n, nb)))
        blk[..., 4:144] = rng.integers(0, 256, size=(n, nb, 140), dtype=np.uint8)
        if dist.get("dmin_zero"):
            blk[..., 2:4] = 0
        return blk.reshape(-1)
    if fmt == "q6_k":
        lo, hi = dist.get("d_range", (0.0005, 0.01))
        nb = k // 256
        blk = np.empty((n, nb, 210), np.uint8)
        blk[..., 0:192] = rng.integers(0, 256, size=(n, nb, 192), dtype=np.uint8)
        sc = rng.integers(-32, 32, size=(n, nb, 16), dtype=np.int64).astype(np.int8)
        blk[..., 192:208] = sc.view(np.uint8)
        blk[..., 208:210] = _f16_bytes(rng.uniform(lo, hi, size=(n, nb)))
        return blk.reshape(-1)
    if fmt == "q8_0":
        lo, hi = dist.get("d_range", (0.002, 0.02))
        nb = k // 32
        blk = np.empty((n, nb, 34), np.uint8)
        blk[..., 0:2] = _f16_bytes(rng.uniform(lo, hi, size=(n, nb)))
        blk[..., 2:34] = rng.integers(0, 256, size=(n, nb, 32), dtype=np.uint8)
        return blk.reshape(-1)
    if fmt == "q5_0":
        lo, hi = dist.get("d_range", (0.005, 0.05))
        nb = k // 32
        blk = np.empty((n, nb, 22), np.uint8)
        blk[..., 0:2] = _f16_bytes(rng.uniform(lo, hi, size=(n, nb)))
        blk[..., 2:22] = rng.integers(0, 256, size=(n, nb, 20), dtype=np.uint8)
        return blk.reshape(-1)
    raise ValueError(f"unknown format {fmt!r}")


# Byte values that put every code of a block at its format's zero point (the
# code whose weight is 0 whatever the block's scale): Q4_0 nibbles 8 (0x88
# bytes); Q8_0 codes 0; Q5_0 code 16 = nibble 0 with its fifth bit set (the
# 4-byte high-bit word all ones); Q6_K code 32 = low nibble 0 with high bits
# 0b10 (ql bytes 0x00, qh bytes 0xAA). Q4_K has no zero point (its codes are
# unsigned with a separate min): there, codes 0 with dmin = +0 give weights
# that are exactly 0 while d and the 6-bit scales stay nonzero.
# (byte range within the block, value) per format; bf16 / f16 rows become +0.
_ZERO_POINT_BYTES = {
    "q4_0": [((2, 18), 0x88)],
    "q8_0": [((2, 34), 0x00)],
    "q5_0": [((2, 6), 0xFF), ((6, 22), 0x00)],
    "q6_k": [((0, 128), 0x00), ((128, 192), 0xAA)],
    "q4_k": [((2, 4), 0x00), ((16, 144), 0x00)],
}


def set_zero_point_rows(fmt: str, w: np.ndarray, k: int, rows) -> np.ndarray:
    """Copy of packed weights w in which every code of the given rows sits at
    the zero point (see _ZERO_POINT_BYTES); the rows' scales keep their drawn,
    nonzero values, so those rows' weights are all exactly 0."""
    rb = row_bytes(fmt, k)
    out = np.array(w, dtype=np.uint8, copy=True).reshape(-1, rb)
    rows = np.asarray(rows, dtype=np.int64)
    if fmt in ("bf16", "f16"):
        out[rows] = 0
        return out.reshape(-1)
    nb = BLOCK_BYTES[fmt]
    blk = out.reshape(out.shape[0], -1, nb)
    for (b0, b1), v in _ZERO_POINT_BYTES[fmt]:
        blk[rows, :, b0:b1] = v
    return blk.reshape(-1)


# Rows whose weights all repeat one value: every block of the row becomes a
# copy of the row's first block (its drawn f16 scales kept) with the codes
# and sub-block scales below, so every weight of the row is the same number.
# (byte range within the block, value) per format; Q4_K's twelve scale bytes
# give every sub-block sc = 1 and m = 45 (with codes 0 every weight is
# -45 dmin); Q6_K's int8 scales are all 37.
_CONSTANT_BYTES = {
    "q4_0": [((2, 18), 0x33)],
    "q8_0": [((2, 34), 0x5B)],
    "q6_k": [((0, 128), 0x00), ((128, 192), 0x00), ((192, 208), 37)],
    "q4_k": [((4, 8), 0x01), ((8, 12), 0xAD), ((12, 16), 0xD1), ((16, 144), 0x00)],
}


def set_constant_rows(fmt: str, w: np.ndarray, k: int, rows, q4_k_code: int = 0) -> np.ndarray:
    """Copy of packed weights w in which every weight of the given rows has
    the same value (see _CONSTANT_BYTES). For Q4_K, q4_k_code (0..15) sets
    every code: 0 gives the weight -dmin m; a nonzero code gives
    d q - dmin m, two terms of the same order that partly cancel."""
    rb = row_bytes(fmt, k)
    out = np.array(w, dtype=np.uint8, copy=True).reshape(-1, rb)
    rows = np.asarray(rows, dtype=np.int64)
    nb = BLOCK_BYTES[fmt]
    blk = out.reshape(out.shape[0], -1, nb)
    blk[rows] = blk[rows, :1, :]
    for (b0, b1), v in _CONSTANT_BYTES[fmt]:
        blk[rows, :, b0:b1] = v
    if fmt == "q4_k":
        blk[rows, :, 16:144] = (q4_k_code & 15) * 0x11
    return blk.reshape(-1)


def set_affine_zero_rows(bits: int, w: np.ndarray, scales: np.ndarray, biases: np.ndarray,
                         k: int, rows):
    """Copies of an affine matrix's arrays in which the given rows are what an
    MLX-style quantizer stores for all-zero groups: codes 0, bias +0 and the
    floor scale -1e-7 (as bf16 bits). Returns (w, scales, biases)."""
    rows = np.asarray(rows, dtype=np.int64)
    w = np.array(w, dtype=np.uint8, copy=True).reshape(scales.shape[0], -1)
    sc = np.array(scales, dtype=np.uint16, copy=True)
    bi = np.array(biases, dtype=np.uint16, copy=True)
    w[rows] = 0
    sc[rows] = _bf16_trunc(np.float32(-1e-7))
    bi[rows] = 0
    return w.reshape(-1), sc, bi


def gen_ids(n_pos: int, top_k: int, n_experts: int, rng: np.random.Generator) -> np.ndarray:
    """Expert ids [n_pos, top_k] int32, distinct within a position."""
    return np.stack([rng.choice(n_experts, size=top_k, replace=False) for _ in range(n_pos)]
                    ).astype(np.int32)


# name -> (fmt, k, n, n_experts, top_k, n_pos, seed)
EXPERT_WORKLOADS = {
    "q8_0_experts": ("q8_0", 2048, 768, 64, 8, 1, 6),
    "q5_0_experts": ("q5_0", 2048, 768, 64, 8, 1, 7),
    "q4_k_experts": ("q4_k", 2048, 768, 64, 8, 1, 14),
}


def expert_workload(name: str, n_pos: int | None = None):
    """Seeded (fmt, k, n, n_experts, W bytes of all experts, X [n_pos, k], ids [n_pos, top_k])."""
    fmt, k, n, n_exp, top_k, pos_default, seed = EXPERT_WORKLOADS[name]
    npos = pos_default if n_pos is None else n_pos
    rng = np.random.default_rng(seed)
    w = gen_weights(fmt, k, n * n_exp, rng)
    x = gen_x(npos, k, rng)
    ids = gen_ids(npos, top_k, n_exp, rng)
    return fmt, k, n, n_exp, w, x, ids


def _bf16_trunc(v: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of fp32 values by dropping the low 16 bits."""
    return (np.asarray(v, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def gen_affine(bits: int, k: int, n: int, rng: np.random.Generator):
    """MLX-style affine matrix (group 64): code words [n, k*bits/8] bytes of
    uniform random u32 words (every code uniform), bf16 scales U[0.01, 0.06)
    and biases U[-0.1, 0.1) [n, k/64], each an fp32 draw truncated to bf16."""
    if bits not in (4, 8) or k % 64:
        raise ValueError("affine matrices take 4 or 8 bits and k % 64 == 0")
    w = rng.integers(0, 256, size=n * k * bits // 8, dtype=np.uint8)
    g = k // 64
    scales = _bf16_trunc(rng.random((n, g), dtype=np.float32) * 0.05 + 0.01)
    biases = _bf16_trunc(rng.random((n, g), dtype=np.float32) * 0.2 - 0.1)
    return w, scales, biases


# name -> (bits, k, n, n_tokens, seed)
AFFINE_WORKLOADS = {
    "affine4_gemv": (4, 4096, 14336, 1, 10),
    "affine8_gemv": (8, 4096, 14336, 1, 11),
    "affine4_prefill": (4, 4096, 14336, 512, 12),
    "affine8_prefill": (8, 4096, 14336, 512, 13),
}


def affine_workload(name: str, n_tokens: int | None = None, n: int | None = None):
    """Seeded (bits, k, n, W code bytes, scales, biases, X [n_tokens, k])."""
    bits, k, n_full, nt_default, seed = AFFINE_WORKLOADS[name]
    n = n_full if n is None else n
    nt = nt_default if n_tokens is None else n_tokens
    rng = np.random.default_rng(seed)
    w, scales, biases = gen_affine(bits, k, n, rng)
    x = gen_x(nt, k, rng)
    return bits, k, n, w, scales, biases, x


def gen_x(n_tokens: int, k: int, rng: np.random.Generator, dist: str = "normal",
          value: float = 0.1) -> np.ndarray:
    """Activations [n_tokens, k] fp32: "normal" N(0, 1), "uniform" U[-1, 1],
    "abs_normal" |N(0, 1)| (every element positive), "constant" (every
    element the fp32 nearest `value`), "constant_rows" (row t constant at
    the fp32 nearest value * (t + 1))."""
    if dist == "uniform":
        return rng.uniform(-1.0, 1.0, size=(n_tokens, k)).astype(np.float32)
    if dist == "abs_normal":
        return np.abs(rng.normal(0.0, 1.0, size=(n_tokens, k))).astype(np.float32)
    if dist == "constant":
        return np.full((n_tokens, k), value, dtype=np.float32)
    if dist == "constant_rows":
        return (np.arange(1, n_tokens + 1, dtype=np.float64)[:, None] * value
                * np.ones((1, k))).astype(np.float32)
    return rng.normal(0.0, 1.0, size=(n_tokens, k)).astype(np.float32)


# name -> (fmt, k, n, n_tokens, seed, x distribution, output tiles)
WORKLOADS = {
    "q4_0_gemv": ("q4_0", 256, 512, 1, 1, "uniform", 1),
    "bf16_gemv": ("bf16", 4096, 4096, 1, 2, "normal", 1),
    "f16_gemv": ("f16", 4096, 4096, 1, 2, "normal", 1),
    "q4_k_gemv": ("q4_k", 4096, 14336, 1, 3, "normal", 1),
    "q6_k_head": ("q6_k", 2560, 262144, 1, 4, "normal", 8),
    "q4_k_prefill": ("q4_k", 4096, 14336, 512, 5, "normal", 1),
    "q8_0_gemv": ("q8_0", 4096, 14336, 1, 8, "normal", 1),
    "q5_0_gemv": ("q5_0", 4096, 14336, 1, 9, "normal", 1),
}


def workload(name: str, n_tokens: int | None = None, n: int | None = None):
    """Seeded (fmt, k, n, W bytes, X) for a named workload.

    ``n`` may shrink the output axis (rows of W) for oracle-sized cases; the
    draws for the first rows do not change with n only for the byte formats'
    layout, so shrunken cases are separate seeded draws, not prefixes.
    """
    fmt, k, n_full, nt_default, seed, xdist, _tiles = WORKLOADS[name]
    n = n_full if n is None else n
    nt = nt_default if n_tokens is None else n_tokens
    rng = np.random.default_rng(seed)
    w = gen_weights(fmt, k, n, rng)
    x = gen_x(nt, k, rng, xdist)
    return fmt, k, n, w, x
