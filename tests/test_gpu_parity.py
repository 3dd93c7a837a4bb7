"""GPU parity: the CUDA path (through the C ABI) against the oracle, element by
element, on seeded synthetic inputs. Dequantization must be bit-identical;
products must meet |y - y_ref| <= 1e-4 * sum_i |x_i w_ij| per output and
cosine >= 0.9999."""
import os

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


def run(fmt, w, x, k, n, **kw):
    y0 = kw.pop("y0", None)
    y = _dev(y0.astype(np.float32)) if y0 is not None else None
    out = q.matmul(fmt, _dev(w), _dev(x), k, n, y=y, **kw)
    torch.cuda.synchronize()
    q.qmm_device_status()
    return out.cpu().numpy()


def assert_parity(y, y_ref, s_ref, what=""):
    ok, worst, cos, msg = oracle.check(y, y_ref, s_ref)
    log = os.environ.get("QMM_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(f"{what}\t{'ok' if ok else 'FAIL'}\t{msg}\n")
    assert ok, f"{what}: {msg}"
    return worst


def _bits_equal(a, b):
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    na, nb = np.isnan(a), np.isnan(b)
    assert np.array_equal(na, nb)
    assert np.array_equal(a.view(np.uint32)[~na], b.view(np.uint32)[~na])


# --------------------------------------------------------------- dequant ----

DEQ_CASES = [("bf16", 98, 33), ("f16", 70, 19), ("q4_0", 96, 41), ("q4_k", 512, 23),
             ("q6_k", 768, 29), ("bf16", 4096, 8), ("q4_0", 256, 512)]


@pytest.mark.parametrize("fmt,k,n", DEQ_CASES)
def test_dequant_bit_exact_synthetic(fmt, k, n):
    rng = np.random.default_rng(100 + k + n)
    w = qmm_synth.gen_weights(fmt, k, n, rng)
    got = q.dequant(fmt, _dev(w), k, n).cpu().numpy()
    _bits_equal(got, oracle.dequant(fmt, w, k, n))


@pytest.mark.parametrize("fmt,k,n", DEQ_CASES)
def test_dequant_bit_exact_random_bytes(fmt, k, n):
    """Every byte uniform: f16 scales include subnormals, inf and NaN."""
    rng = np.random.default_rng(200 + k + n)
    w = rng.integers(0, 256, size=qmm_synth.row_bytes(fmt, k) * n, dtype=np.uint8)
    got = q.dequant(fmt, _dev(w), k, n).cpu().numpy()
    _bits_equal(got, oracle.dequant(fmt, w, k, n))


def test_dequant_full_size_sampled_rows():
    fmt, k, n, w, _ = qmm_synth.workload("q6_k_head")
    got = q.dequant(fmt, _dev(w), k, n)
    rows = np.array([0, 1, 2, 12345, 131071, 131072, 200001, n - 2, n - 1])
    rb = qmm_synth.row_bytes(fmt, k)
    for j in rows:
        ref = oracle.dequant(fmt, w[j * rb:(j + 1) * rb], k, 1)[0]
        _bits_equal(got[int(j)].cpu().numpy(), ref)


# ------------------------------------------------------------------ GEMV ----

GEMV_CASES = [("bf16", 4096, 1000), ("f16", 64, 777), ("q4_0", 96, 333), ("q4_0", 256, 512),
              ("q4_k", 4096, 1500), ("q4_k", 256, 70), ("q6_k", 2560, 1000), ("q6_k", 256, 65),
              ("bf16", 16384, 300), ("q6_k", 16384, 77), ("f16", 32, 5), ("q4_k", 16384, 40)]


@pytest.mark.parametrize("fmt,k,n", GEMV_CASES)
def test_gemv_parity(fmt, k, n):
    rng = np.random.default_rng(k * 7 + n)
    w = qmm_synth.gen_weights(fmt, k, n, rng)
    x = qmm_synth.gen_x(1, k, rng)
    y = run(fmt, w, x, k, n, path=q.PATH_GEMV)
    y_ref, s_ref = oracle.matmul(fmt, w, x, k, n)
    assert_parity(y, y_ref, s_ref, f"gemv {fmt} k={k} n={n}")


@pytest.mark.parametrize("name", ["q4_0_gemv", "bf16_gemv", "f16_gemv", "q4_k_gemv"])
def test_gemv_full_workloads(name):
    fmt, k, n, w, x = qmm_synth.workload(name)
    y = run(fmt, w, x, k, n)   # auto path: GEMV for one token
    y_ref, s_ref = oracle.matmul(fmt, w, x, k, n)
    worst = assert_parity(y, y_ref, s_ref, name)
    assert worst < 1e-5, worst   # fp32 accumulation only: far inside the bar


def test_gemv_deterministic():
    fmt, k, n, w, x = qmm_synth.workload("q4_k_gemv", n=3000)
    a = run(fmt, w, x, k, n)
    b = run(fmt, w, x, k, n)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_q6_k_head_tiled_and_accumulated():
    """Vocab-sized head: 8 output tiles of 32768 columns, first pass writes,
    second pass accumulates onto a prefilled y; plus the untiled call."""
    fmt, k, n, w, x = qmm_synth.workload("q6_k_head")
    y_ref, s_ref = oracle.matmul(fmt, w, x, k, n)
    wd, xd = _dev(w), _dev(x)
    y = torch.full((1, n), float("nan"), device=DEV)
    tile = n // 8
    for t in range(8):
        q.matmul(fmt, wd, xd, k, n, y=y, j_start=t * tile, j_end=(t + 1) * tile,
                 accumulate=False)
    torch.cuda.synchronize()
    assert_parity(y.cpu().numpy(), y_ref, s_ref, "q6_k tiled write")
    y_in = np.random.default_rng(9).normal(0, 1, (1, n)).astype(np.float32)
    y = _dev(y_in)
    for t in range(8):
        q.matmul(fmt, wd, xd, k, n, y=y, j_start=t * tile, j_end=(t + 1) * tile,
                 accumulate=True)
    torch.cuda.synchronize()
    y_exp, s_exp = oracle.tiled(y_ref, s_ref, 0, n, True, y_in)
    assert_parity(y.cpu().numpy(), y_exp, s_exp, "q6_k tiled accumulate")
    y = q.matmul(fmt, wd, xd, k, n)
    torch.cuda.synchronize()
    assert_parity(y.cpu().numpy(), y_ref, s_ref, "q6_k untiled")
    q.qmm_device_status()


@pytest.mark.parametrize("path", [q.PATH_GEMV, q.PATH_MMA])
@pytest.mark.parametrize("j0,j1,acc", [(5, 301, False), (130, 131, True), (0, 1, False),
                                      (257, 700, True), (256, 601, True), (0, 700, True),
                                      (128, 700, False)])
def test_partial_tile_leaves_other_columns(path, j0, j1, acc):
    rng = np.random.default_rng(j0 * 13 + j1)
    k, n, nt = 512, 700, (1 if path == q.PATH_GEMV else 5)
    w = qmm_synth.gen_weights("q4_k", k, n, rng)
    x = qmm_synth.gen_x(nt, k, rng)
    y_in = rng.normal(0, 1, (nt, n)).astype(np.float32)
    y = run("q4_k", w, x, k, n, y0=y_in, j_start=j0, j_end=j1, accumulate=acc, path=path)
    y_ref, s_ref = oracle.matmul("q4_k", w, x, k, n)
    y_exp, s_exp = oracle.tiled(y_ref, s_ref, j0, j1, acc, y_in)
    outside = np.ones(n, bool)
    outside[j0:j1] = False
    assert np.array_equal(y[:, outside].view(np.uint32), y_in[:, outside].view(np.uint32))
    assert_parity(y[:, j0:j1], y_exp[:, j0:j1], s_exp[:, j0:j1], "tile")


# ------------------------------------------------------ tensor-core path ----

@pytest.mark.parametrize("nt", [1, 3, 8, 16, 17, 64, 200, 256, 300])
def test_mma_q4_k_token_counts(nt):
    rng = np.random.default_rng(nt)
    k, n = 4096, 300   # 300 = 2 full 128-row tiles + a ragged one
    w = qmm_synth.gen_weights("q4_k", k, n, rng)
    x = qmm_synth.gen_x(nt, k, rng)
    y = run("q4_k", w, x, k, n, path=q.PATH_MMA)
    y_ref, s_ref = oracle.matmul("q4_k", w, x, k, n)
    assert_parity(y, y_ref, s_ref, f"mma q4_k N={nt}")


@pytest.mark.parametrize("fmt,k,n,nt", [("bf16", 98, 130, 5), ("f16", 4096, 200, 40),
                                        ("q4_0", 96, 257, 7), ("q4_0", 4096, 128, 33),
                                        ("q6_k", 2560, 129, 20), ("q6_k", 256, 64, 2),
                                        ("bf16", 4096, 256, 512), ("q4_k", 256, 1, 2)])
def test_mma_all_formats(fmt, k, n, nt):
    rng = np.random.default_rng(k + n + nt)
    w = qmm_synth.gen_weights(fmt, k, n, rng)
    x = qmm_synth.gen_x(nt, k, rng)
    y = run(fmt, w, x, k, n, path=q.PATH_MMA)
    y_ref, s_ref = oracle.matmul(fmt, w, x, k, n)
    assert_parity(y, y_ref, s_ref, f"mma {fmt} k={k} n={n} N={nt}")


def test_mma_large_and_tiny_activations():
    """Rows of x far outside fp16 range are scaled by a power of two per token."""
    rng = np.random.default_rng(77)
    k, n = 1024, 256
    w = qmm_synth.gen_weights("q4_k", k, n, rng)
    x = qmm_synth.gen_x(4, k, rng)
    x[0] *= 1e6
    x[1] *= 1e-9
    x[2] = 0.0
    y = run("q4_k", w, x, k, n, path=q.PATH_MMA)
    y_ref, s_ref = oracle.matmul("q4_k", w, x, k, n)
    assert np.all(y[2] == 0.0)
    assert_parity(y, y_ref, s_ref, "scaled activations")


def test_gemv_and_mma_agree_on_one_token():
    fmt, k, n, w, x = qmm_synth.workload("q4_k_gemv", n=1024)
    a = run(fmt, w, x, k, n, path=q.PATH_GEMV)
    b = run(fmt, w, x, k, n, path=q.PATH_MMA)
    y_ref, s_ref = oracle.matmul(fmt, w, x, k, n)
    assert_parity(a, y_ref, s_ref, "gemv")
    assert_parity(b, y_ref, s_ref, "mma")


@pytest.mark.parametrize("nt", [1, 8, 64, 512])
def test_q4_k_prefill_full_size_sampled(nt):
    """Full prefill shape (k=4096, n=14336) at the crossover token counts;
    outputs sampled for the oracle, every output checked finite."""
    fmt, k, n, w, x = qmm_synth.workload("q4_k_prefill", n_tokens=nt)
    y = run(fmt, w, x, k, n)
    assert np.all(np.isfinite(y))
    rng = np.random.default_rng(nt)
    cnt = 3000
    t_idx = rng.integers(0, nt, cnt)
    j_idx = rng.integers(0, n, cnt)
    # always include the corners of the tile grid
    t_idx[:4] = [0, nt - 1, 0, nt - 1]
    j_idx[:4] = [0, 0, n - 1, n - 1]
    y_ref, s_ref = oracle.matmul_sampled(fmt, w, x, k, n, t_idx, j_idx)
    assert_parity(y[t_idx, j_idx], y_ref, s_ref, f"prefill N={nt}")


@pytest.mark.parametrize("nt", [64, 512])
def test_q4_k_prefill_full_size_every_output(nt):
    """Every output of the full prefill shape against the oracle (dot products
    by a library f64 matrix product over the oracle's weights)."""
    fmt, k, n, w, x = qmm_synth.workload("q4_k_prefill", n_tokens=nt)
    y = run(fmt, w, x, k, n)
    y_ref, s_ref = oracle.matmul_blas(fmt, w, x, k, n)
    assert_parity(y, y_ref, s_ref, f"prefill all outputs N={nt}")


def test_mma_repeatable_bits():
    """The tensor-core path gives the same bits on every call, including the
    row tiles of the last round that run as two k-halves adding into zeros
    (0 + a + b rounds the same in either order); accumulate mode adds the same
    result onto y."""
    fmt, k, n, w, x = qmm_synth.workload("q4_k_prefill", n_tokens=512)
    wd, xd = _dev(w), _dev(x)
    ys = []
    for _ in range(3):
        ys.append(q.matmul(fmt, wd, xd, k, n).cpu().numpy())
    torch.cuda.synchronize()
    q.qmm_device_status()
    _bits_equal(ys[0], ys[1])
    _bits_equal(ys[0], ys[2])
    # accumulate computes every tile whole (no k-halves): same sum up to the
    # rounding order of the halves
    y0 = np.full((512, n), 0.5, np.float32)
    yacc = run(fmt, w, x, k, n, y0=y0, accumulate=True)
    scale = float(np.abs(ys[0]).max())
    np.testing.assert_allclose(yacc, ys[0] + np.float32(0.5), rtol=1e-5, atol=1e-5 * scale)


# ------------------------------------------- overlapped (PDL) launches ----

def test_overlap_chain_reads_previous_output():
    """y1 = W1 x, then y2 = W2 y1 with QMM_FLAG_OVERLAP_PREV: the second GEMV
    streams W2 early but must read x = y1 only after the first one finished."""
    rng = np.random.default_rng(41)
    k1, n1, n2 = 4096, 2048, 3000
    w1 = qmm_synth.gen_weights("bf16", k1, n1, rng)
    w2 = qmm_synth.gen_weights("q4_k", n1, n2, rng)
    x = qmm_synth.gen_x(1, k1, rng)
    w1d, w2d, xd = _dev(w1), _dev(w2), _dev(x)
    for rep in range(3):
        y1 = torch.full((1, n1), float("nan"), device=DEV)
        y2 = torch.full((1, n2), float("nan"), device=DEV)
        q.matmul("bf16", w1d, xd, k1, n1, y=y1, flags=q.FLAG_OVERLAP_PREV)
        q.matmul("q4_k", w2d, y1, n1, n2, y=y2, flags=q.FLAG_OVERLAP_PREV)
        torch.cuda.synchronize()
        q.qmm_device_status()
        y1h = y1.cpu().numpy()
        r1, s1 = oracle.matmul("bf16", w1, x, k1, n1)
        assert_parity(y1h, r1, s1, "chain stage 1")
        r2, s2 = oracle.matmul("q4_k", w2, y1h, n1, n2)
        assert_parity(y2.cpu().numpy(), r2, s2, "chain stage 2")


def test_overlap_x_ready_accumulates_after_previous_store():
    """y = W1 x, then y += W2 x with OVERLAP_PREV | X_READY on the same y: the
    second kernel computes early but must add to y only after the first stored it."""
    rng = np.random.default_rng(42)
    k, n = 4096, 5000
    w1 = qmm_synth.gen_weights("q6_k", k, n, rng)
    w2 = qmm_synth.gen_weights("f16", k, n, rng)
    x = qmm_synth.gen_x(1, k, rng)
    w1d, w2d, xd = _dev(w1), _dev(w2), _dev(x)
    r1, s1 = oracle.matmul("q6_k", w1, x, k, n)
    r2, s2 = oracle.matmul("f16", w2, x, k, n)
    fl = q.FLAG_OVERLAP_PREV | q.FLAG_X_READY
    for rep in range(3):
        y = torch.full((1, n), float("nan"), device=DEV)
        q.matmul("q6_k", w1d, xd, k, n, y=y, flags=fl)
        q.matmul("f16", w2d, xd, k, n, y=y, accumulate=True, flags=fl)
        torch.cuda.synchronize()
        q.qmm_device_status()
        assert_parity(y.cpu().numpy(), r1 + r2, s1 + s2, "x-ready accumulate")


# ------------------------------------------------------------ edge cases ----

def test_k_zero_and_empty():
    y_in = np.arange(12, dtype=np.float32).reshape(2, 6)
    w = np.zeros(0, np.uint8)   # k = 0: no weight bytes
    x = np.zeros((2, 0), np.float32)
    y = run("bf16", w, x, 0, 6, y0=y_in, j_start=1, j_end=4)
    assert np.all(y[:, 1:4] == 0) and np.array_equal(y[:, [0, 4, 5]], y_in[:, [0, 4, 5]])
    y = run("bf16", w, x, 0, 6, y0=y_in, accumulate=True)
    assert np.array_equal(y, y_in)
    y = run("q4_k", np.zeros(0, np.uint8), np.ones((1, 256), np.float32), 256, 0)
    assert y.shape == (1, 0)


def test_all_zero_point_q4_0_row_is_exactly_zero():
    k, n = 256, 3
    w = np.zeros((n, k // 32, 18), np.uint8)
    w[..., 0:2] = [0x00, 0x3C]
    w[..., 2:] = 0x88          # every code 8 -> weight 0
    w = w.reshape(-1)
    x = qmm_synth.gen_x(1, k, np.random.default_rng(1))
    for path in (q.PATH_GEMV, q.PATH_MMA):
        y = run("q4_0", w, x, k, n, path=path)
        assert np.all(y == 0.0), path


def test_plain_signature_and_host_variant():
    fmt, k, n, w, x = qmm_synth.workload("q4_0_gemv")
    lib = q.load()
    wd, xd = _dev(w), _dev(x)
    yd = torch.empty((1, n), device=DEV)
    q.qmm_set_stream(torch.cuda.current_stream())
    q.qmm_matmul(fmt, wd, xd, k, n, 1, yd)
    torch.cuda.synchronize()
    y_ref, s_ref = oracle.matmul(fmt, w, x, k, n)
    assert_parity(yd.cpu().numpy(), y_ref, s_ref, "qmm_matmul")
    # host buffers in, host y out
    wh = torch.from_numpy(w).pin_memory()
    xh = torch.from_numpy(x).pin_memory()
    yh = torch.zeros((1, n)).pin_memory()
    a = q.make_args(fmt, wh, xh, yh, k, n, 1)
    q.qmm_matmul_host(a, torch.empty_like(wd), torch.empty_like(xd), torch.empty_like(yd))
    torch.cuda.synchronize()
    assert_parity(yh.numpy(), y_ref, s_ref, "qmm_matmul_host")
    assert lib is q.load()


@pytest.mark.parametrize("fmt,k,n,nt", [("q4_k", 256, 384, 2048), ("q8_0", 512, 200, 1500),
                                        ("bf16", 256, 130, 777)])
def test_mma_many_token_tiles(fmt, k, n, nt):
    """Many token tiles (up to 8 of 256) over few row pairs, ragged rows and
    tokens: the persistent schedule walks several rounds."""
    rng = np.random.default_rng(nt + n)
    w = qmm_synth.gen_weights(fmt, k, n, rng)
    x = qmm_synth.gen_x(nt, k, rng)
    y = run(fmt, w, x, k, n, path=q.PATH_MMA)
    y_ref, s_ref = oracle.matmul(fmt, w, x, k, n)
    assert_parity(y, y_ref, s_ref, f"mma {fmt} k={k} n={n} N={nt}")


@pytest.mark.parametrize("fmt,k", [("bf16", 16384), ("f16", 16384), ("q4_0", 16384),
                                   ("q8_0", 16384), ("q5_0", 16384)])
def test_gemv_largest_k(fmt, k):
    """The largest k the one-token kernel takes for each unit width."""
    rng = np.random.default_rng(k // 7)
    n = 96
    w = qmm_synth.gen_weights(fmt, k, n, rng)
    x = qmm_synth.gen_x(1, k, rng)
    y = run(fmt, w, x, k, n, path=q.PATH_GEMV)
    y_ref, s_ref = oracle.matmul(fmt, w, x, k, n)
    assert_parity(y, y_ref, s_ref, f"gemv {fmt} k={k}")


def test_workspace_must_be_device_memory_of_this_gpu():
    """The tensor-core path reads its x tiles from the workspace with copies
    shared by a pair of CTAs: a caller workspace in host memory (pinned or
    pageable) is rejected on the host with QMM_ERR_UNSUPPORTED, nothing
    enqueued; device memory of the current GPU is taken."""
    import ctypes
    fmt, k, n, nt = "q4_k", 1024, 256, 8
    rng = np.random.default_rng(17)
    w = qmm_synth.gen_weights(fmt, k, n, rng)
    x = qmm_synth.gen_x(nt, k, rng)
    wd, xd = _dev(w), _dev(x)
    y = torch.zeros((nt, n), device=DEV)
    a = q.make_args(fmt, wd, xd, y, k, n, nt, path=q.PATH_MMA)
    need = q.qmm_workspace_bytes(a)
    pinned = torch.empty(need + 256, dtype=torch.uint8).pin_memory()
    pageable = np.empty(need + 256, np.uint8)
    for base in (pinned.data_ptr(), pageable.ctypes.data):
        a.workspace, a.workspace_bytes = (base + 255) // 256 * 256, need
        assert q.load().qmm_matmul_ex(ctypes.byref(a)) == 10
        assert "device memory" in q.qmm_last_error()
    torch.cuda.synchronize()
    assert (y == 0).all()
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    a.workspace, a.workspace_bytes = ws.data_ptr(), need
    q.qmm_matmul_ex(a)
    torch.cuda.synchronize()
    q.qmm_device_status()
    y_ref, s_ref = oracle.matmul(fmt, w, x, k, n)
    assert_parity(y.cpu().numpy(), y_ref, s_ref, "device workspace")
