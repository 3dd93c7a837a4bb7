"""GPU parity of gated pairs y = act(x Wg) * (x Wu) (SwiGLU, GeGLU) through
the C ABI against the oracle: per output |y - y_ref| <= 1e-4 * S with S the
error scale propagated from the two products' bars (|act'(g)| |u| Sg +
|act(g)| Su, plus |y_in| when accumulating) and an absolute floor of the
smallest normal fp32 (2^-126), cosine >= 0.9999. One token
runs the fused gated GEMV; several tokens the tensor-core products and the
elementwise combine."""
import numpy as np
import pytest

import oracle
import qmm_synth

torch = pytest.importorskip("torch")
import quantized_weight_gguf_gb300 as q  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


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


def _assert(y, y_ref, s_ref, what):
    # results below fp32's normal range carry no relative accuracy: FLT_MIN floor
    ok, worst, cos, msg = oracle.check(y, y_ref, s_ref, atol=oracle.FLT_MIN)
    assert ok, f"{what}: {msg}"


def _run(act, fmt, wg, wu, x, k, n, **kw):
    y0 = kw.pop("y0", None)
    y = _dev(y0.astype(np.float32)) if y0 is not None else None
    out = q.matmul_glu(act, fmt, _dev(wg), _dev(wu), _dev(x), k, n, y=y, **kw)
    torch.cuda.synchronize()
    q.qmm_device_status()
    return out.cpu().numpy()


@pytest.mark.parametrize("act", ["swiglu", "geglu"])
@pytest.mark.parametrize("fmt,k,n", [("q4_k", 4096, 1000), ("q4_0", 96, 333), ("q6_k", 2560, 257),
                                     ("bf16", 4096, 300), ("f16", 64, 77), ("q8_0", 2048, 1),
                                     ("q5_0", 1024, 500), ("q4_k", 256, 14336)])
def test_fused_gemv_parity(act, fmt, k, n):
    rng = np.random.default_rng(k + n + len(act))
    wg = qmm_synth.gen_weights(fmt, k, n, rng)
    wu = qmm_synth.gen_weights(fmt, k, n, rng)
    x = qmm_synth.gen_x(1, k, rng)
    y = _run(act, fmt, wg, wu, x, k, n)
    y_ref, s_ref = oracle.matmul_glu(act, fmt, wg, wu, x, k, n)
    _assert(y, y_ref, s_ref, f"fused {act} {fmt} k={k} n={n}")


@pytest.mark.parametrize("act", ["swiglu", "geglu"])
def test_saturating_gates(act):
    """Gate values far into both tails (x scaled up): silu -> g or 0,
    GELU -> g or 0."""
    rng = np.random.default_rng(5)
    fmt, k, n = "q8_0", 1024, 700
    wg = qmm_synth.gen_weights(fmt, k, n, rng)
    wu = qmm_synth.gen_weights(fmt, k, n, rng)
    x = (qmm_synth.gen_x(1, k, rng) * 40.0).astype(np.float32)
    y = _run(act, fmt, wg, wu, x, k, n)
    y_ref, s_ref = oracle.matmul_glu(act, fmt, wg, wu, x, k, n)
    g, _ = oracle.matmul(fmt, wg, x, k, n)
    assert np.abs(g).max() > 20.0
    _assert(y, y_ref, s_ref, f"saturating {act}")


@pytest.mark.parametrize("act", ["swiglu", "geglu"])
@pytest.mark.parametrize("j0,j1,acc", [(5, 301, False), (130, 131, True), (0, 700, True)])
def test_tiles_and_accumulate(act, j0, j1, acc):
    rng = np.random.default_rng(j0 + j1)
    fmt, k, n = "q4_k", 512, 700
    wg = qmm_synth.gen_weights(fmt, k, n, rng)
    wu = qmm_synth.gen_weights(fmt, k, n, rng)
    x = qmm_synth.gen_x(1, k, rng)
    y_in = rng.normal(0, 1, (1, n)).astype(np.float32)
    y = _run(act, fmt, wg, wu, x, k, n, y0=y_in, j_start=j0, j_end=j1, accumulate=acc)
    y_ref, s_ref = oracle.matmul_glu(act, fmt, wg, wu, x, k, n)
    y_exp, s_exp = oracle.tiled(y_ref, s_ref, j0, j1, acc, y_in)
    outside = np.ones(n, bool)
    outside[j0:j1] = False
    assert np.array_equal(y[:, outside].view(np.uint32), y_in[:, outside].view(np.uint32))
    _assert(y[:, j0:j1], y_exp[:, j0:j1], s_exp[:, j0:j1], f"{act} tile")


@pytest.mark.parametrize("act", ["swiglu", "geglu"])
@pytest.mark.parametrize("fmt,k,n,nt", [("q4_k", 4096, 300, 8), ("q6_k", 2560, 129, 64),
                                        ("q8_0", 2048, 256, 3)])
def test_several_tokens(act, fmt, k, n, nt):
    rng = np.random.default_rng(nt + n)
    wg = qmm_synth.gen_weights(fmt, k, n, rng)
    wu = qmm_synth.gen_weights(fmt, k, n, rng)
    x = qmm_synth.gen_x(nt, k, rng)
    y = _run(act, fmt, wg, wu, x, k, n)
    y_ref, s_ref = oracle.matmul_glu(act, fmt, wg, wu, x, k, n)
    _assert(y, y_ref, s_ref, f"{act} N={nt}")
    # accumulate into a tile on the several-token form too
    y_in = rng.normal(0, 1, (nt, n)).astype(np.float32)
    y = _run(act, fmt, wg, wu, x, k, n, y0=y_in, j_start=7, j_end=n - 3, accumulate=True)
    y_exp, s_exp = oracle.tiled(y_ref, s_ref, 7, n - 3, True, y_in)
    assert np.array_equal(y[:, :7].view(np.uint32), y_in[:, :7].view(np.uint32))
    _assert(y[:, 7:n - 3], y_exp[:, 7:n - 3], s_exp[:, 7:n - 3], f"{act} N={nt} tile")


def test_fused_equals_unfused_composition_within_rounding():
    """The fused GEMV's gate and up sums are the plain GEMV's (same kernel
    arithmetic): act(gate) * up from two plain calls matches to fp32 rounding
    of the activation."""
    rng = np.random.default_rng(9)
    fmt, k, n = "q4_k", 4096, 2000
    wg = qmm_synth.gen_weights(fmt, k, n, rng)
    wu = qmm_synth.gen_weights(fmt, k, n, rng)
    x = qmm_synth.gen_x(1, k, rng)
    y = _run("swiglu", fmt, wg, wu, x, k, n)
    g = q.matmul(fmt, _dev(wg), _dev(x), k, n).cpu().numpy().astype(np.float64)
    u = q.matmul(fmt, _dev(wu), _dev(x), k, n).cpu().numpy().astype(np.float64)
    with np.errstate(over="ignore"):
        comp = g / (1.0 + np.exp(-g)) * u
    np.testing.assert_allclose(y, comp, rtol=2e-6, atol=1e-30)


def test_k_zero_writes_zeros():
    y_in = np.full((1, 8), 3.0, np.float32)
    w = np.zeros(0, np.uint8)
    x = np.zeros((1, 0), np.float32)
    y = _run("swiglu", "q4_k", w, w, x, 0, 8, y0=y_in)
    assert np.all(y == 0.0)


@pytest.mark.parametrize("act", ["swiglu", "geglu"])
def test_several_tokens_constant_rows_with_split_w(act):
    """Gated pairs on the tensor cores with QMM_FLAG_SPLIT_W: both products
    carry W as two fp16 terms, so rows whose weights repeat one value (gate
    and up) hold the bar with activations of one sign."""
    fmt, k, n, nt = "q4_k", 4096, 256, 16
    rng = np.random.default_rng(77)
    rows = np.arange(0, n, 2)
    wg = qmm_synth.set_constant_rows(fmt, qmm_synth.gen_weights(fmt, k, n, rng), k, rows)
    wu = qmm_synth.set_constant_rows(fmt, qmm_synth.gen_weights(fmt, k, n, rng), k, rows)
    x = qmm_synth.gen_x(nt, k, rng, "abs_normal")
    y = _run(act, fmt, wg, wu, x, k, n, flags=q.FLAG_SPLIT_W)
    y_ref, s_ref = oracle.matmul_glu(act, fmt, wg, wu, x, k, n)
    _assert(y, y_ref, s_ref, f"{act} N={nt} split W")
