"""Chains of calls in one stream where each call consumes the output of the
call before it, with no synchronization between them.

The tensor-core product lets the next kernel in the stream launch while it
runs; the x conversion and the GEMV launched without QMM_FLAG_OVERLAP_PREV are
programmatic dependents that wait for the preceding kernel before they read
anything. The results must be those of plain stream order: every output that a
later call reads is filled with NaN before the chain starts, so a read before
the producing kernel finished shows up as NaN (or as a mismatch) downstream.
Each step is checked against the oracle on the inputs it actually received."""
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


def _nan(shape):
    return torch.full(shape, float("nan"), dtype=torch.float32, device=DEV)


def _check(fmt, w, x, y, k, n, what):
    x = np.atleast_2d(x)
    if x.shape[0] > 1:
        y_ref, s_ref = oracle.matmul_blas(fmt, w, x, k, n)
    else:
        y_ref, s_ref = oracle.matmul(fmt, w, x, k, n)
    ok, worst, cos, msg = oracle.check(np.atleast_2d(y), y_ref, s_ref)
    assert ok, f"{what}: {msg}"


# (first path, second path): the second call reads the first call's y as its x
CHAINS = [(q.PATH_MMA, q.PATH_MMA), (q.PATH_MMA, q.PATH_GEMV), (q.PATH_GEMV, q.PATH_MMA),
          (q.PATH_GEMV, q.PATH_GEMV)]


@pytest.mark.parametrize("p1,p2", CHAINS)
@pytest.mark.parametrize("fmt", ["q4_k", "bf16"])
def test_second_call_reads_the_first_calls_output(fmt, p1, p2):
    k1, n1, n2 = 1024, 2048, 768
    rng = np.random.default_rng(300 + 10 * p1 + p2 + len(fmt))
    w1 = qmm_synth.gen_weights(fmt, k1, n1, rng)
    w2 = qmm_synth.gen_weights(fmt, n1, n2, rng)
    nt1 = 16 if p1 == q.PATH_MMA else 1
    x = qmm_synth.gen_x(nt1, k1, rng)
    w1d, w2d, xd = _dev(w1), _dev(w2), _dev(x)
    for rep in range(3):
        y1 = _nan((nt1, n1))
        y2 = _nan((nt1 if p2 == q.PATH_MMA else 1, n2))
        q.matmul(fmt, w1d, xd, k1, n1, y=y1, path=p1)
        # the GEMV takes the last row of y1 (one token), the tensor cores all of it
        x2 = y1 if p2 == q.PATH_MMA else y1[-1:]
        q.matmul(fmt, w2d, x2, n1, n2, y=y2, path=p2)
        torch.cuda.synchronize()
        q.qmm_device_status()
        y1h, y2h = y1.cpu().numpy(), y2.cpu().numpy()
        assert np.isfinite(y2h).all(), f"rep {rep}: the second call read y1 before it was written"
        _check(fmt, w1, x, y1h, k1, n1, f"rep {rep} first call")
        x2h = y1h if p2 == q.PATH_MMA else y1h[-1:]
        _check(fmt, w2, x2h, y2h, n1, n2, f"rep {rep} second call")


def test_overlapping_gemv_after_tensor_core_waits_for_its_x():
    """QMM_FLAG_OVERLAP_PREV (W independent of the preceding kernel, x not):
    the GEMV streams W at once but reads x, the tensor-core call's y, only
    after that call has finished."""
    fmt, k1, n1, n2 = "q4_k", 1024, 2048, 768
    rng = np.random.default_rng(321)
    w1 = qmm_synth.gen_weights(fmt, k1, n1, rng)
    w2 = qmm_synth.gen_weights(fmt, n1, n2, rng)
    x = qmm_synth.gen_x(8, k1, rng)
    w1d, w2d, xd = _dev(w1), _dev(w2), _dev(x)
    y1 = _nan((8, n1))
    y2 = _nan((1, n2))
    q.matmul(fmt, w1d, xd, k1, n1, y=y1, path=q.PATH_MMA)
    q.matmul(fmt, w2d, y1[3:4], n1, n2, y=y2, path=q.PATH_GEMV, flags=q.FLAG_OVERLAP_PREV)
    torch.cuda.synchronize()
    q.qmm_device_status()
    y1h, y2h = y1.cpu().numpy(), y2.cpu().numpy()
    assert np.isfinite(y2h).all()
    _check(fmt, w2, y1h[3:4], y2h, n1, n2, "overlapping GEMV")


def test_gated_pair_chain():
    """Gate product, then the up product whose epilogue reads the gate values,
    then a GEMV over the gated output: three dependent launches in a row."""
    fmt, k, n, n2 = "q4_k", 1024, 1024, 512
    rng = np.random.default_rng(333)
    wg = qmm_synth.gen_weights(fmt, k, n, rng)
    wu = qmm_synth.gen_weights(fmt, k, n, rng)
    w2 = qmm_synth.gen_weights(fmt, n, n2, rng)
    x = qmm_synth.gen_x(16, k, rng)
    y = _nan((16, n))
    y2 = _nan((1, n2))
    q.matmul_glu("swiglu", fmt, _dev(wg), _dev(wu), _dev(x), k, n, y=y)
    q.matmul(fmt, _dev(w2), y[-1:], n, n2, y=y2, path=q.PATH_GEMV)
    torch.cuda.synchronize()
    q.qmm_device_status()
    yh, y2h = y.cpu().numpy(), y2.cpu().numpy()
    y_ref, s_ref = oracle.matmul_glu("swiglu", fmt, wg, wu, x, k, n)
    ok, worst, cos, msg = oracle.check(yh, y_ref, s_ref, atol=oracle.FLT_MIN)
    assert ok, msg
    assert np.isfinite(y2h).all()
    _check(fmt, w2, yh[-1:], y2h, n, n2, "GEMV over the gated output")
