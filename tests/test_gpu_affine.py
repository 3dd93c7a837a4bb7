"""GPU parity of the MLX-style affine 4- and 8-bit matrices (codes in u32
words, bf16 scale and bias per group of 64) through the C ABI, against the
oracle: dequantization bit-identical; products within the product bar
|y - y_ref| <= 1e-4 * sum_i |x_i w_ij| (plus |y_in| when accumulating) and
cosine >= 0.9999, on the one-token GEMV and the tensor-core path."""
import numpy as np
import pytest

import oracle
import qmm_synth

torch = pytest.importorskip("torch")
import quantized_weight_gguf_gb300 as q  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
FMT = {4: "affine4", 8: "affine8"}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from quantized_weight_gguf_gb300 import build_lib
    build_lib.build()
    q.load()
    oracle.build()
    yield
    q.qmm_device_status()


def _dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(DEV)


def _bits_equal(a, b):
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    na, nb = np.isnan(a), np.isnan(b)
    assert np.array_equal(na, nb)
    assert np.array_equal(a.view(np.uint32)[~na], b.view(np.uint32)[~na])


def _assert(y, y_ref, s_ref, what):
    ok, worst, cos, msg = oracle.check(y, y_ref, s_ref)
    assert ok, f"{what}: {msg}"
    return worst


def _run(bits, w, sc, bi, x, k, n, **kw):
    y0 = kw.pop("y0", None)
    y = _dev(y0.astype(np.float32)) if y0 is not None else None
    out = q.matmul_affine(FMT[bits], _dev(w), _dev(sc), _dev(bi), _dev(x), k, n, y=y, **kw)
    torch.cuda.synchronize()
    q.qmm_device_status()
    return out.cpu().numpy()


# ------------------------------------------------------------- dequant ----

@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("k,n", [(64, 7), (192, 41), (4096, 33)])
def test_dequant_bit_exact(bits, k, n):
    rng = np.random.default_rng(bits * 1000 + k + n)
    w, sc, bi = qmm_synth.gen_affine(bits, k, n, rng)
    got = q.dequant_affine(FMT[bits], _dev(w), _dev(sc), _dev(bi), k, n).cpu().numpy()
    _bits_equal(got, oracle.dequant_affine(bits, w, sc, bi, k, n))


@pytest.mark.parametrize("bits", [4, 8])
def test_dequant_random_bf16_patterns(bits):
    """Scales and biases with every bf16 pattern class (subnormals, huge
    exponents, infinities, NaN)."""
    rng = np.random.default_rng(50 + bits)
    k, n = 256, 64
    w = rng.integers(0, 256, size=n * k * bits // 8, dtype=np.uint8)
    sc = rng.integers(0, 65536, size=(n, k // 64), dtype=np.uint16)
    bi = rng.integers(0, 65536, size=(n, k // 64), dtype=np.uint16)
    got = q.dequant_affine(FMT[bits], _dev(w), _dev(sc), _dev(bi), k, n).cpu().numpy()
    _bits_equal(got, oracle.dequant_affine(bits, w, sc, bi, k, n))


# -------------------------------------------------------------- products ----

@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("k,n", [(64, 5), (128, 777), (4096, 1000), (16384, 300), (2048, 1)])
def test_gemv_parity(bits, k, n):
    rng = np.random.default_rng(bits * 7 + k + n)
    w, sc, bi = qmm_synth.gen_affine(bits, k, n, rng)
    x = qmm_synth.gen_x(1, k, rng)
    y = _run(bits, w, sc, bi, x, k, n, path=q.PATH_GEMV)
    y_ref, s_ref = oracle.matmul_affine(bits, w, sc, bi, x, k, n)
    _assert(y, y_ref, s_ref, f"gemv affine{bits} k={k} n={n}")


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("k,n,nt", [(128, 130, 5), (2048, 257, 17), (4096, 300, 64),
                                    (4096, 256, 512), (1024, 128, 2), (64, 1, 3)])
def test_mma_parity(bits, k, n, nt):
    rng = np.random.default_rng(bits * 11 + k + n + nt)
    w, sc, bi = qmm_synth.gen_affine(bits, k, n, rng)
    x = qmm_synth.gen_x(nt, k, rng)
    y = _run(bits, w, sc, bi, x, k, n, path=q.PATH_MMA)
    y_ref, s_ref = oracle.matmul_affine(bits, w, sc, bi, x, k, n)
    _assert(y, y_ref, s_ref, f"mma affine{bits} k={k} n={n} N={nt}")


@pytest.mark.parametrize("path", [q.PATH_GEMV, q.PATH_MMA])
@pytest.mark.parametrize("j0,j1,acc", [(5, 301, False), (130, 131, True), (0, 700, True),
                                      (257, 700, False)])
def test_tiles_and_accumulate(path, j0, j1, acc):
    rng = np.random.default_rng(j0 * 3 + j1)
    k, n, nt = 1024, 700, (1 if path == q.PATH_GEMV else 6)
    w, sc, bi = qmm_synth.gen_affine(4, k, n, rng)
    x = qmm_synth.gen_x(nt, k, rng)
    y_in = rng.normal(0, 1, (nt, n)).astype(np.float32)
    y = _run(4, w, sc, bi, x, k, n, y0=y_in, j_start=j0, j_end=j1, accumulate=acc, path=path)
    y_ref, s_ref = oracle.matmul_affine(4, w, sc, bi, x, k, n)
    y_exp, s_exp = oracle.tiled(y_ref, s_ref, j0, j1, acc, y_in)
    outside = np.ones(n, bool)
    outside[j0:j1] = False
    assert np.array_equal(y[:, outside].view(np.uint32), y_in[:, outside].view(np.uint32))
    _assert(y[:, j0:j1], y_exp[:, j0:j1], s_exp[:, j0:j1], "affine tile")


@pytest.mark.parametrize("name", ["affine4_gemv", "affine8_gemv"])
def test_full_size_gemv_every_output(name):
    bits, k, n, w, sc, bi, x = qmm_synth.affine_workload(name)
    y = _run(bits, w, sc, bi, x, k, n)   # one token: the GEMV
    y_ref, s_ref = oracle.matmul_affine_blas(bits, w, sc, bi, x, k, n)
    worst = _assert(y, y_ref, s_ref, name)
    assert worst < 1e-5, worst


def test_full_size_prefill_sampled():
    """N = 512 on the tensor-core path, 2048 outputs recomputed one by one."""
    bits, k, n, w, sc, bi, x = qmm_synth.affine_workload("affine4_prefill")
    y = _run(bits, w, sc, bi, x, k, n)
    rng = np.random.default_rng(3)
    ti = rng.integers(0, x.shape[0], 2048)
    ji = rng.integers(0, n, 2048)
    y_ref, s_ref = oracle.matmul_affine_sampled(bits, w, sc, bi, x, k, n, ti, ji)
    _assert(y[ti, ji][None, :], y_ref[None, :], s_ref[None, :], "affine4 prefill sampled")


def test_gemv_and_mma_agree_on_one_token():
    rng = np.random.default_rng(12)
    k, n = 4096, 512
    w, sc, bi = qmm_synth.gen_affine(8, k, n, rng)
    x = qmm_synth.gen_x(1, k, rng)
    a = _run(8, w, sc, bi, x, k, n, path=q.PATH_GEMV)
    b = _run(8, w, sc, bi, x, k, n, path=q.PATH_MMA)
    y_ref, s_ref = oracle.matmul_affine(8, w, sc, bi, x, k, n)
    _assert(a, y_ref, s_ref, "gemv")
    _assert(b, y_ref, s_ref, "mma")


def test_repeatable_bits():
    rng = np.random.default_rng(13)
    k, n = 4096, 3000
    w, sc, bi = qmm_synth.gen_affine(4, k, n, rng)
    x = qmm_synth.gen_x(1, k, rng)
    a = _run(4, w, sc, bi, x, k, n)
    b = _run(4, w, sc, bi, x, k, n)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("bits", [4, 8])
def test_tensor_core_path_repeatable_bits(bits):
    """N = 512 on the raw-tile path, several calls into poisoned outputs: every
    call gives the same bits (the raw-tile ring is refilled only after its
    readers are done)."""
    rng = np.random.default_rng(40 + bits)
    k, n, nt = 4096, 4096, 512
    w, sc, bi = qmm_synth.gen_affine(bits, k, n, rng)
    x = qmm_synth.gen_x(nt, k, rng)
    wd, scd, bid, xd = _dev(w), _dev(sc), _dev(bi), _dev(x)
    ref = None
    for it in range(8):
        y = torch.full((nt, n), float(it + 1), device=DEV)
        q.matmul_affine(FMT[bits], wd, scd, bid, xd, k, n, y=y)
        torch.cuda.synchronize()
        q.qmm_device_status()
        got = y.cpu().numpy()
        if ref is None:
            ref = got
        else:
            assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), f"call {it}"


@pytest.mark.parametrize("bits,k,n,n_exp,top_k,n_pos", [(4, 1024, 300, 6, 3, 2), (8, 4096, 768, 16, 4, 3),
                                                       (4, 64, 7, 3, 2, 1)])
def test_affine_experts(bits, k, n, n_exp, top_k, n_pos):
    """Expert-indexed affine product: row p * top_k + s equals the plain affine
    product of x[p] with the slice ids[p, s] of the stacked codes, scales and
    biases (cut by hand)."""
    rng = np.random.default_rng(bits * 100 + k + n)
    w, sc, bi = qmm_synth.gen_affine(bits, k, n * n_exp, rng)
    x = qmm_synth.gen_x(n_pos, k, rng)
    ids = qmm_synth.gen_ids(n_pos, top_k, n_exp, rng)
    y = q.matmul_experts(FMT[bits], _dev(w), _dev(x), _dev(ids), k, n, n_exp, scales=_dev(sc),
                         biases=_dev(bi))
    torch.cuda.synchronize()
    q.qmm_device_status()
    y = y.cpu().numpy()
    rb = k * bits // 8
    for p in range(n_pos):
        for s in range(top_k):
            e = int(ids[p, s])
            yr, sr = oracle.matmul_affine(bits, w[e * n * rb:(e + 1) * n * rb], sc[e * n:(e + 1) * n],
                                          bi[e * n:(e + 1) * n], x[p], k, n)
            _assert(y[p * top_k + s][None, :], yr, sr, f"affine{bits} expert {e} pos {p} slot {s}")


def test_affine_experts_tile_accumulate_and_bad_id():
    rng = np.random.default_rng(61)
    bits, k, n, n_exp = 4, 512, 400, 4
    w, sc, bi = qmm_synth.gen_affine(bits, k, n * n_exp, rng)
    x = qmm_synth.gen_x(2, k, rng)
    ids = np.array([[3, 0], [-1, 2]], np.int32)
    y_in = rng.normal(0, 1, (4, n)).astype(np.float32)
    j0, j1 = 33, 301
    y = q.matmul_experts(FMT[bits], _dev(w), _dev(x), _dev(ids), k, n, n_exp, scales=_dev(sc),
                         biases=_dev(bi), y=_dev(y_in), j_start=j0, j_end=j1, accumulate=True)
    torch.cuda.synchronize()
    with pytest.raises(q.QmmError) as ei:
        q.qmm_device_status()
    assert ei.value.status == 11
    y = y.cpu().numpy()
    assert np.array_equal(y[2].view(np.uint32), y_in[2].view(np.uint32))   # bad id: row untouched
    outside = np.ones(n, bool)
    outside[j0:j1] = False
    assert np.array_equal(y[:, outside].view(np.uint32), y_in[:, outside].view(np.uint32))
    rb = k * bits // 8
    for row, (p, e) in ((0, (0, 3)), (1, (0, 0)), (3, (1, 2))):
        yr, sr = oracle.matmul_affine(bits, w[e * n * rb:(e + 1) * n * rb], sc[e * n:(e + 1) * n],
                                      bi[e * n:(e + 1) * n], x[p], k, n)
        ye, se = oracle.tiled(yr, sr, j0, j1, True, y_in[row][None, :])
        _assert(y[row][None, j0:j1], ye[:, j0:j1], se[:, j0:j1], f"row {row}")
