"""Rows whose codes all sit at the zero point under a nonzero scale: every
weight of such a row is exactly 0, so its reference output and its error
scale S are both 0, and the bar |y - y_ref| <= 1e-4 * S demands exactly 0.
Quantizers write such rows (padded vocabulary rows, all-zero groups: an
MLX-style affine quantizer stores codes 0, bias 0 and its floor scale for
them). Checked through every entry point that decodes codes: the one-token
GEMV, the tensor-core path, the backward with respect to the input (over a
tile of such rows), the expert-indexed product and the gated pair; against
the oracle, whose check also holds every other row to the usual bar."""
import numpy as np
import pytest

import oracle
import qmm_synth

torch = pytest.importorskip("torch")
import quantized_weight_gguf_gb300 as q  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
FMTS = ["q4_0", "q8_0", "q5_0", "q6_k", "q4_k", "bf16"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from quantized_weight_gguf_gb300 import build_lib
    build_lib.build()
    q.load()
    oracle.build()
    yield
    q.qmm_device_status()


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _sync():
    torch.cuda.synchronize()
    q.qmm_device_status()


def _assert(y, y_ref, s_ref, what, atol=0.0):
    ok, worst, cos, msg = oracle.check(np.atleast_2d(y), np.atleast_2d(y_ref),
                                       np.atleast_2d(s_ref), atol=atol)
    assert ok, f"{what}: {msg}"


def _k_for(fmt):
    return 2560 if fmt == "q6_k" else 4096


def _mixed(fmt, k, n, seed):
    """Weights with every third row (and the last) at the zero point."""
    rng = np.random.default_rng(seed)
    w = qmm_synth.gen_weights(fmt, k, n, rng)
    rows = np.union1d(np.arange(0, n, 3), [n - 1])
    return qmm_synth.set_zero_point_rows(fmt, w, k, rows), rows, rng


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("xdist", ["normal", "constant"])
def test_gemv_zero_point_rows_are_exactly_zero(fmt, xdist):
    k, n = _k_for(fmt), 700
    w, rows, rng = _mixed(fmt, k, n, 5 + len(fmt))
    x = qmm_synth.gen_x(1, k, rng, xdist, 1.0 / 3.0)
    y = q.matmul(fmt, _dev(w), _dev(x), k, n, path=q.PATH_GEMV)
    _sync()
    y = y.cpu().numpy()
    y_ref, s_ref = oracle.matmul(fmt, w, x, k, n)
    assert (s_ref[0, rows] == 0).all() and (y_ref[0, rows] == 0).all()
    assert (y[0, rows] == 0).all(), f"{fmt}: nonzero output on a zero-point row"
    _assert(y, y_ref, s_ref, f"gemv {fmt} {xdist}")


@pytest.mark.parametrize("fmt", FMTS)
def test_tensor_core_zero_point_rows_are_exactly_zero(fmt):
    k, n, nt = _k_for(fmt), 400, 24
    w, rows, rng = _mixed(fmt, k, n, 50 + len(fmt))
    x = qmm_synth.gen_x(nt, k, rng)
    y = q.matmul(fmt, _dev(w), _dev(x), k, n, path=q.PATH_MMA)
    _sync()
    y = y.cpu().numpy()
    y_ref, s_ref = oracle.matmul_blas(fmt, w, x, k, n)
    assert (y[:, rows] == 0).all(), f"{fmt}: nonzero output on a zero-point row"
    _assert(y, y_ref, s_ref, f"mma {fmt}")


@pytest.mark.parametrize("fmt", ["q4_0", "q8_0", "q5_0", "q6_k", "q4_k", "bf16"])
def test_backward_input_over_zero_point_rows(fmt):
    """A sum-axis tile made only of zero-point rows gives dx = 0 exactly (S = 0
    for every entry); the next tile, of ordinary rows, then accumulates."""
    k, n = (2048 if fmt == "bf16" else _k_for(fmt)), 600   # 16-bit rows: k <= 2048 here
    rng = np.random.default_rng(70 + len(fmt))
    w = qmm_synth.gen_weights(fmt, k, n, rng)
    half = n // 2
    w = qmm_synth.set_zero_point_rows(fmt, w, k, np.arange(half))
    dy = qmm_synth.gen_x(1, n, rng)[0]
    dx = q.matmul_backward_input(fmt, _dev(w), _dev(dy), k, n, j_start=0, j_end=half)
    _sync()
    dx0 = dx.cpu().numpy()
    assert (dx0 == 0).all(), f"{fmt}: nonzero dx over zero-point rows"
    q.matmul_backward_input(fmt, _dev(w), _dev(dy), k, n, dx=dx, j_start=half, j_end=n,
                            accumulate=True)
    _sync()
    ref, s = oracle.matmul_back_input(fmt, w, dy, k, n)
    _assert(dx.cpu().numpy(), ref, s, f"backward {fmt}")


@pytest.mark.parametrize("fmt", ["q8_0", "q5_0", "q4_k"])
def test_experts_with_zero_point_slices(fmt):
    k, n, n_exp, top_k, n_pos = 2048, 256, 6, 3, 2
    rng = np.random.default_rng(90 + len(fmt))
    w = qmm_synth.gen_weights(fmt, k, n * n_exp, rng)
    # experts 1 and 4 entirely at the zero point, plus every 5th row of the rest
    dead = np.concatenate([np.arange(n, 2 * n), np.arange(4 * n, 5 * n),
                           np.arange(0, n * n_exp, 5)])
    w = qmm_synth.set_zero_point_rows(fmt, w, k, np.unique(dead))
    x = qmm_synth.gen_x(n_pos, k, rng)
    ids = np.array([[1, 0, 4], [2, 4, 5]], dtype=np.int32)
    y = q.matmul_experts(fmt, _dev(w), _dev(x), _dev(ids), k, n, n_exp)
    _sync()
    y = y.cpu().numpy()
    y_ref, s_ref = oracle.matmul_experts(fmt, w, x, k, n, n_exp, ids)
    assert (y[0] == 0).all() and (y[2] == 0).all() and (y[4] == 0).all()
    _assert(y, y_ref, s_ref, f"experts {fmt}")


@pytest.mark.parametrize("which", ["gate", "up"])
@pytest.mark.parametrize("fmt", ["q6_k", "q4_k", "q5_0"])
def test_gated_pair_with_zero_point_rows(fmt, which):
    """A zero-point row in the gate (act(0) = 0) or the up matrix gives 0."""
    k, n = _k_for(fmt), 500
    rng = np.random.default_rng(110 + len(fmt))
    wg = qmm_synth.gen_weights(fmt, k, n, rng)
    wu = qmm_synth.gen_weights(fmt, k, n, rng)
    rows = np.arange(0, n, 4)
    if which == "gate":
        wg = qmm_synth.set_zero_point_rows(fmt, wg, k, rows)
    else:
        wu = qmm_synth.set_zero_point_rows(fmt, wu, k, rows)
    for nt in (1, 16):
        x = qmm_synth.gen_x(nt, k, rng)
        y = q.matmul_glu("swiglu", fmt, _dev(wg), _dev(wu), _dev(x), k, n)
        _sync()
        y = y.cpu().numpy()
        y_ref, s_ref = oracle.matmul_glu("swiglu", fmt, wg, wu, x, k, n)
        assert (y[:, rows] == 0).all(), f"{fmt} {which} tokens={nt}: nonzero output"
        _assert(y, y_ref, s_ref, f"glu {fmt} {which} tokens={nt}", atol=oracle.FLT_MIN)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("nt", [1, 16])
def test_affine_zero_groups_as_an_mlx_quantizer_writes_them(bits, nt):
    """Rows of all-zero groups: codes 0, bias 0, scale -1e-7 (bf16)."""
    k, n = 4096, 600
    rng = np.random.default_rng(130 + bits + nt)
    w, sc, bi = qmm_synth.gen_affine(bits, k, n, rng)
    rows = np.arange(1, n, 3)
    w, sc, bi = qmm_synth.set_affine_zero_rows(bits, w, sc, bi, k, rows)
    x = qmm_synth.gen_x(nt, k, rng)
    y = q.matmul_affine(f"affine{bits}", _dev(w), _dev(sc.view(np.int16)), _dev(bi.view(np.int16)),
                        _dev(x), k, n)
    _sync()
    y = y.cpu().numpy()
    y_ref, s_ref = oracle.matmul_affine_blas(bits, w, sc, bi, x, k, n)
    assert (y[:, rows] == 0).all(), f"affine{bits} tokens={nt}: nonzero output"
    _assert(y, y_ref, s_ref, f"affine{bits} tokens={nt}")


@pytest.mark.parametrize("bits", [4, 8])
def test_affine_experts_with_zero_groups(bits):
    k, n, n_exp = 2048, 192, 4
    rng = np.random.default_rng(150 + bits)
    w, sc, bi = qmm_synth.gen_affine(bits, k, n * n_exp, rng)
    w, sc, bi = qmm_synth.set_affine_zero_rows(bits, w, sc, bi, k, np.arange(n, 2 * n))
    x = qmm_synth.gen_x(1, k, rng)
    ids = np.array([[1, 3]], dtype=np.int32)
    y = q.matmul_experts(f"affine{bits}", _dev(w), _dev(x), _dev(ids), k, n, n_exp,
                         scales=_dev(sc.view(np.int16)), biases=_dev(bi.view(np.int16)))
    _sync()
    y = y.cpu().numpy()
    assert (y[0] == 0).all()
    # reference: the selected slices through the plain affine oracle
    rb = w.size // (n * n_exp)
    for s, e in enumerate(ids[0]):
        ws = w[e * n * rb:(e + 1) * n * rb]
        y_ref, s_ref = oracle.matmul_affine(bits, ws, sc[e * n:(e + 1) * n], bi[e * n:(e + 1) * n],
                                            x, k, n)
        _assert(y[s:s + 1], y_ref, s_ref, f"affine{bits} expert slot {s}")
