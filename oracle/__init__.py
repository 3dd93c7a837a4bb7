"""Oracle for ``y = x @ W`` over GGUF/ggml-packed weights (plain C, f64 sums).

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the
bench's ``cpu_baseline`` / reference leg may import this package; the CUDA
product path never does, and nothing here imports the product package.

The arithmetic lives in ``qmm_oracle.c`` (see its header for the passages it
follows). This wrapper only compiles it with gcc, marshals numpy arrays to
it, and holds the acceptance check:

* per output ``|y - y_ref| <= 1e-4 * S`` where ``S = sum_i |x_i * w_ij|``
  (plus ``|y_in|`` when accumulating into a prefilled y), the bar that the
  matmul is held to;
* cosine similarity over f64 sums, floor 0.9999, as moeflux
  tests/graph_diff_oracle.rs ``cosine_sim`` / ``COSINE_FLOOR`` define it;
  two all-zero vectors count as equal (that function returns 0 for them,
  which is read here as "no disagreement").

Every function here has parity pins in tests/test_oracle_pins.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CODES = {"bf16": 0, "f16": 1, "q4_0": 2, "q4_k": 3, "q6_k": 4, "q8_0": 5, "q5_0": 6}
TOL_REL = 1e-4
COSINE_FLOOR = 0.9999


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE arithmetic, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                               "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, p = ctypes.c_int64, ctypes.c_void_p
            lib.oracle_f16_value.restype = ctypes.c_double
            lib.oracle_f16_value.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_value.restype = ctypes.c_float
            lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
            lib.oracle_row_bytes.restype = i64
            lib.oracle_row_bytes.argtypes = [ctypes.c_int, i64]
            lib.oracle_dequant.restype = ctypes.c_int
            lib.oracle_dequant.argtypes = [ctypes.c_int, p, i64, i64, p]
            lib.oracle_matmul.restype = ctypes.c_int
            lib.oracle_matmul.argtypes = [ctypes.c_int, p, p, i64, i64, i64, p, p, p]
            lib.oracle_matmul_back_input.restype = ctypes.c_int
            lib.oracle_matmul_back_input.argtypes = [ctypes.c_int, p, p, i64, i64, i64, i64, p, p, p]
            lib.oracle_matmul_experts.restype = ctypes.c_int
            lib.oracle_matmul_experts.argtypes = [ctypes.c_int, p, p, i64, i64, i64, i64, i64, p, p,
                                                  p, p]
            lib.oracle_matmul_sampled.restype = ctypes.c_int
            lib.oracle_matmul_sampled.argtypes = [ctypes.c_int, p, p, i64, i64, i64, i64, p, p, p, p, p]
            lib.oracle_affine_row_bytes.restype = i64
            lib.oracle_affine_row_bytes.argtypes = [ctypes.c_int, i64]
            lib.oracle_dequant_affine.restype = ctypes.c_int
            lib.oracle_dequant_affine.argtypes = [ctypes.c_int, p, p, p, i64, i64, p]
            lib.oracle_matmul_affine.restype = ctypes.c_int
            lib.oracle_matmul_affine.argtypes = [ctypes.c_int, p, p, p, p, i64, i64, i64, p, p, p]
            lib.oracle_matmul_affine_sampled.restype = ctypes.c_int
            lib.oracle_matmul_affine_sampled.argtypes = [ctypes.c_int, p, p, p, p, i64, i64, i64,
                                                         i64, p, p, p, p, p]
            lib.oracle_act.restype = ctypes.c_double
            lib.oracle_act.argtypes = [ctypes.c_int, ctypes.c_double]
            lib.oracle_act_deriv.restype = ctypes.c_double
            lib.oracle_act_deriv.argtypes = [ctypes.c_int, ctypes.c_double]
            lib.oracle_matmul_glu.restype = ctypes.c_int
            lib.oracle_matmul_glu.argtypes = [ctypes.c_int, ctypes.c_int, p, p, p, i64, i64, i64, p,
                                              p, p]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def f16_value(h: int) -> float:
    return _load().oracle_f16_value(int(h) & 0xFFFF)


def bf16_value(h: int) -> float:
    return _load().oracle_bf16_value(int(h) & 0xFFFF)


def row_bytes(fmt: str, k: int) -> int:
    return int(_load().oracle_row_bytes(CODES[fmt], int(k)))


def dequant(fmt: str, w: np.ndarray, k: int, n: int) -> np.ndarray:
    """fp32 weights [n, k] from packed bytes."""
    w = np.ascontiguousarray(w, dtype=np.uint8)
    rb = row_bytes(fmt, k)
    if (rb == 0 and k != 0) or w.size != rb * n:
        raise ValueError("bad shape for oracle dequant")
    out = np.empty((n, k), np.float32)
    if _load().oracle_dequant(CODES[fmt], _ptr(w), k, n, _ptr(out)) != 0:
        raise ValueError("oracle dequant rejected its arguments")
    return out


def matmul(fmt: str, w: np.ndarray, x: np.ndarray, k: int, n: int):
    """(y, S): y[t, j] = sum_i x[t, i] w[j, i] and S = sum_i |x w|, both f64 [N, n]."""
    w = np.ascontiguousarray(w, dtype=np.uint8)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    nt = x.shape[0]
    if x.shape[1] != k:
        raise ValueError("x must be [N, k]")
    y = np.empty((nt, n), np.float64)
    s = np.empty((nt, n), np.float64)
    scratch = np.empty(max(k, 1), np.float32)
    if _load().oracle_matmul(CODES[fmt], _ptr(w), _ptr(x), k, n, nt, _ptr(y), _ptr(s), _ptr(scratch)) != 0:
        raise ValueError("oracle matmul rejected its arguments")
    return y, s


def matmul_blas(fmt: str, w: np.ndarray, x: np.ndarray, k: int, n: int):
    """Same (y, S) as matmul, with the dot products done by numpy's f64 matrix
    product over the oracle's own fp32 weights (for full-size checks)."""
    deq = dequant(fmt, w, k, n).astype(np.float64)
    x64 = np.atleast_2d(np.asarray(x, np.float64))
    return x64 @ deq.T, np.abs(x64) @ np.abs(deq).T


def matmul_sampled(fmt: str, w: np.ndarray, x: np.ndarray, k: int, n: int, t_idx, j_idx):
    """(y, S) for the outputs (t_idx[c], j_idx[c]) only."""
    w = np.ascontiguousarray(w, dtype=np.uint8)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    t_idx = np.ascontiguousarray(t_idx, dtype=np.int64)
    j_idx = np.ascontiguousarray(j_idx, dtype=np.int64)
    cnt = t_idx.size
    y = np.empty(cnt, np.float64)
    s = np.empty(cnt, np.float64)
    scratch = np.empty(max(k, 1), np.float32)
    rc = _load().oracle_matmul_sampled(CODES[fmt], _ptr(w), _ptr(x), k, n, x.shape[0], cnt,
                                       _ptr(t_idx), _ptr(j_idx), _ptr(y), _ptr(s), _ptr(scratch))
    if rc != 0:
        raise ValueError("oracle sampled matmul rejected its arguments")
    return y, s


def matmul_experts(fmt: str, w: np.ndarray, x: np.ndarray, k: int, n: int, n_experts: int,
                   ids: np.ndarray):
    """(y, S) of the expert-indexed product: x [n_pos, k], ids [n_pos, top_k]
    (int32) into n_experts stacked slices of n rows; y and S are f64
    [n_pos * top_k, n] (row p * top_k + s)."""
    w = np.ascontiguousarray(w, dtype=np.uint8)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    ids = np.ascontiguousarray(np.atleast_2d(ids), dtype=np.int32)
    n_pos, top_k = ids.shape
    if x.shape != (n_pos, k) or w.size != row_bytes(fmt, k) * n * n_experts:
        raise ValueError("bad shapes for the expert product")
    y = np.empty((n_pos * top_k, n), np.float64)
    s = np.empty((n_pos * top_k, n), np.float64)
    scratch = np.empty(max(k, 1), np.float32)
    if _load().oracle_matmul_experts(CODES[fmt], _ptr(w), _ptr(x), k, n, n_experts, n_pos, top_k,
                                     _ptr(ids), _ptr(y), _ptr(s), _ptr(scratch)) != 0:
        raise ValueError("oracle expert product rejected its arguments")
    return y, s


def matmul_back_input(fmt: str, w: np.ndarray, dy: np.ndarray, k: int, n: int,
                      j_start: int = 0, j_end: int | None = None):
    """(dx, S) of the backward with respect to the input over rows
    [j_start, j_end): dx[i] = sum_j dy[j] w[j, i], S = sum_j |dy[j] w[j, i]|,
    both f64 [k]."""
    w = np.ascontiguousarray(w, dtype=np.uint8)
    dy = np.ascontiguousarray(np.asarray(dy).reshape(-1), dtype=np.float32)
    if dy.size != n:
        raise ValueError("dy must have n entries")
    j_end = n if j_end is None else j_end
    dx = np.empty(k, np.float64)
    s = np.empty(k, np.float64)
    scratch = np.empty(max(k, 1), np.float32)
    if _load().oracle_matmul_back_input(CODES[fmt], _ptr(w), _ptr(dy), k, n, j_start, j_end,
                                        _ptr(dx), _ptr(s), _ptr(scratch)) != 0:
        raise ValueError("oracle backward-input rejected its arguments")
    return dx, s


def matmul_back_input_blas(fmt: str, w: np.ndarray, dy: np.ndarray, k: int, n: int,
                           j_start: int = 0, j_end: int | None = None):
    """Same (dx, S) as matmul_back_input, by numpy's f64 product over the
    oracle's own fp32 weights (for full-size checks)."""
    j_end = n if j_end is None else j_end
    deq = dequant(fmt, w, k, n)[j_start:j_end].astype(np.float64)
    d = np.asarray(dy, np.float64).reshape(-1)[j_start:j_end]
    return d @ deq, np.abs(d) @ np.abs(deq)


def tiled(y_ref: np.ndarray, s_ref: np.ndarray, j_start: int, j_end: int, accumulate: bool,
          y_in: np.ndarray):
    """Expected output of an output-axis tile: columns [j_start, j_end) of y
    become y_ref (or y_in + y_ref when accumulating); other columns keep y_in.
    Returns (y_expected, S) with |y_in| added to S where it is summed in."""
    y = np.array(y_in, dtype=np.float64, copy=True)
    s = np.zeros_like(y)
    sl = slice(j_start, j_end)
    if accumulate:
        y[:, sl] = y[:, sl] + y_ref[:, sl]
        s[:, sl] = s_ref[:, sl] + np.abs(np.asarray(y_in, np.float64)[:, sl])
    else:
        y[:, sl] = y_ref[:, sl]
        s[:, sl] = s_ref[:, sl]
    return y, s


def cosine(a: np.ndarray, b: np.ndarray) -> float:
    """Cosine similarity with f64 sums; 1.0 when both vectors are all zero."""
    a = np.asarray(a, np.float64).reshape(-1)
    b = np.asarray(b, np.float64).reshape(-1)
    na = float(np.dot(a, a))
    nb = float(np.dot(b, b))
    if na == 0.0 and nb == 0.0:
        return 1.0
    if na == 0.0 or nb == 0.0:
        return 0.0
    return float(np.dot(a, b) / (np.sqrt(na) * np.sqrt(nb)))


FLT_MIN = 2.0 ** -126   # smallest normal fp32


def check(y: np.ndarray, y_ref: np.ndarray, s_ref: np.ndarray, tol: float = TOL_REL,
          atol: float = 0.0):
    """Acceptance check. Returns (ok, worst_ratio, cosine, message).

    ``atol`` is an absolute floor under the bar: results whose true value
    lies below fp32's normal range (a saturated gate activation, for one)
    cannot carry relative accuracy, so errors up to ``atol`` (FLT_MIN for
    the gated products) pass."""
    y = np.asarray(y, np.float64)
    err = np.abs(y - y_ref)
    bound = np.maximum(tol * s_ref, atol)
    nan_mismatch = np.isnan(y) != np.isnan(y_ref)
    finite = ~np.isnan(y_ref)
    bad = (err > bound) & finite
    bad |= nan_mismatch
    # err / S, with S raised to the absolute floor's equivalent (atol / tol) so
    # that the worst ratio is comparable with tol whichever bound applies
    s_eff = np.maximum(s_ref, atol / tol) if atol > 0 else s_ref
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(s_eff > 0, err / np.where(s_eff > 0, s_eff, 1.0), np.where(err > 0, np.inf, 0.0))
    worst = float(np.nanmax(ratio[finite])) if finite.any() else 0.0
    cos = cosine(np.where(finite, y, 0.0), np.where(finite, y_ref, 0.0))
    ok = (not bad.any()) and cos >= COSINE_FLOOR
    msg = f"bad={int(bad.sum())}/{y.size} worst err/S={worst:.3e} cosine={cos:.9f}"
    if bad.any():
        idx = np.argwhere(bad)[0]
        msg += f" first bad at {tuple(int(i) for i in idx)}: y={y[tuple(idx)]!r} ref={y_ref[tuple(idx)]!r} S={s_ref[tuple(idx)]!r}"
    return ok, worst, cos, msg


# ------------------------------------------------- MLX-style affine rows ----
# bits = 4 or 8; w: [n, k*bits/8] bytes of little-endian u32 code words;
# scales, biases: bf16 bit patterns [n, k/64] (uint16).

def affine_row_bytes(bits: int, k: int) -> int:
    return int(_load().oracle_affine_row_bytes(int(bits), int(k)))


def _affine_args(bits, w, scales, biases, k, n):
    w = np.ascontiguousarray(w, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    biases = np.ascontiguousarray(biases, dtype=np.uint16)
    rb = affine_row_bytes(bits, k)
    if rb < 0 or w.size != rb * n or scales.size != n * (k // 64) or biases.size != scales.size:
        raise ValueError("bad shapes for an affine matrix")
    return w, scales, biases


def dequant_affine(bits: int, w, scales, biases, k: int, n: int) -> np.ndarray:
    """fp32 weights [n, k]: code * scale + bias, rounded once."""
    w, scales, biases = _affine_args(bits, w, scales, biases, k, n)
    out = np.empty((n, k), np.float32)
    if _load().oracle_dequant_affine(bits, _ptr(w), _ptr(scales), _ptr(biases), k, n,
                                     _ptr(out)) != 0:
        raise ValueError("oracle affine dequant rejected its arguments")
    return out


def matmul_affine(bits: int, w, scales, biases, x, k: int, n: int):
    """(y, S) of x [N, k] times the affine matrix, f64 [N, n]."""
    w, scales, biases = _affine_args(bits, w, scales, biases, k, n)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    if x.shape[1] != k:
        raise ValueError("x must be [N, k]")
    nt = x.shape[0]
    y = np.empty((nt, n), np.float64)
    s = np.empty((nt, n), np.float64)
    scratch = np.empty(max(k, 1), np.float32)
    if _load().oracle_matmul_affine(bits, _ptr(w), _ptr(scales), _ptr(biases), _ptr(x), k, n, nt,
                                    _ptr(y), _ptr(s), _ptr(scratch)) != 0:
        raise ValueError("oracle affine matmul rejected its arguments")
    return y, s


def matmul_affine_sampled(bits: int, w, scales, biases, x, k: int, n: int, t_idx, j_idx):
    """(y, S) for the outputs (t_idx[c], j_idx[c]) only."""
    w, scales, biases = _affine_args(bits, w, scales, biases, k, n)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    t_idx = np.ascontiguousarray(t_idx, dtype=np.int64)
    j_idx = np.ascontiguousarray(j_idx, dtype=np.int64)
    cnt = t_idx.size
    y = np.empty(cnt, np.float64)
    s = np.empty(cnt, np.float64)
    scratch = np.empty(max(k, 1), np.float32)
    rc = _load().oracle_matmul_affine_sampled(bits, _ptr(w), _ptr(scales), _ptr(biases), _ptr(x),
                                              k, n, x.shape[0], cnt, _ptr(t_idx), _ptr(j_idx),
                                              _ptr(y), _ptr(s), _ptr(scratch))
    if rc != 0:
        raise ValueError("oracle affine sampled matmul rejected its arguments")
    return y, s


def matmul_affine_blas(bits: int, w, scales, biases, x, k: int, n: int):
    """Same (y, S) as matmul_affine via numpy's f64 product over the oracle's
    own fp32 weights (for full-size checks)."""
    deq = dequant_affine(bits, w, scales, biases, k, n).astype(np.float64)
    x64 = np.atleast_2d(np.asarray(x, np.float64))
    return x64 @ deq.T, np.abs(x64) @ np.abs(deq).T


# ------------------------------------------------------- gated products ----
ACTS = {"swiglu": 0, "geglu": 1}


def act(name: str, g: float) -> float:
    """silu (swiglu) or tanh-form GELU (geglu) of one value, in double."""
    return _load().oracle_act(ACTS[name], float(g))


def act_deriv(name: str, g: float) -> float:
    return _load().oracle_act_deriv(ACTS[name], float(g))


def matmul_glu(name: str, fmt: str, wg, wu, x, k: int, n: int):
    """(y, S): y = act(x Wg) * (x Wu), S its propagated error scale, f64 [N, n]."""
    wg = np.ascontiguousarray(wg, dtype=np.uint8)
    wu = np.ascontiguousarray(wu, dtype=np.uint8)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    if x.shape[1] != k or wg.size != wu.size:
        raise ValueError("bad shapes for the gated product")
    nt = x.shape[0]
    y = np.empty((nt, n), np.float64)
    s = np.empty((nt, n), np.float64)
    scratch = np.empty(max(k, 1), np.float32)
    if _load().oracle_matmul_glu(ACTS[name], CODES[fmt], _ptr(wg), _ptr(wu), _ptr(x), k, n, nt,
                                 _ptr(y), _ptr(s), _ptr(scratch)) != 0:
        raise ValueError("oracle gated matmul rejected its arguments")
    return y, s
