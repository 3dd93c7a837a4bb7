"""GPU parity of the 32-weight block formats Q8_0 and Q5_0 on every path
(dequantization bit-identical; one-token GEMV, tensor-core product and the
backward with respect to the input within the product bar), and of the
expert-indexed product (each position and slot multiplies by the expert
slice its id selects) against the oracle, through the C ABI."""
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


def _bits_equal(a, b):
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    na, nb = np.isnan(a), np.isnan(b)
    assert np.array_equal(na, nb)
    assert np.array_equal(a.view(np.uint32)[~na], b.view(np.uint32)[~na])


def _assert(y, y_ref, s_ref, what):
    ok, worst, cos, msg = oracle.check(y, y_ref, s_ref)
    assert ok, f"{what}: {msg}"


BLOCK32 = ["q8_0", "q5_0"]


# ------------------------------------------------------------- dequant ----

@pytest.mark.parametrize("fmt", BLOCK32)
@pytest.mark.parametrize("k,n", [(32, 7), (96, 41), (4096, 33)])
def test_dequant_bit_exact(fmt, k, n):
    rng = np.random.default_rng(k + n)
    w = qmm_synth.gen_weights(fmt, k, n, rng)
    got = q.dequant(fmt, _dev(w), k, n).cpu().numpy()
    _bits_equal(got, oracle.dequant(fmt, w, k, n))


@pytest.mark.parametrize("fmt", BLOCK32)
def test_dequant_random_bytes(fmt):
    """Every byte uniform: the f16 scales include subnormals, infinities and NaN."""
    rng = np.random.default_rng(5)
    k, n = 256, 64
    w = rng.integers(0, 256, size=qmm_synth.row_bytes(fmt, k) * n, dtype=np.uint8)
    got = q.dequant(fmt, _dev(w), k, n).cpu().numpy()
    _bits_equal(got, oracle.dequant(fmt, w, k, n))


# -------------------------------------------------------------- products ----

@pytest.mark.parametrize("fmt", BLOCK32)
@pytest.mark.parametrize("k,n,nt,path", [(32, 5, 1, q.PATH_GEMV), (4096, 1000, 1, q.PATH_GEMV),
                                         (14336, 300, 1, q.PATH_GEMV), (96, 333, 4, q.PATH_GEMV),
                                         (2048, 257, 1, q.PATH_MMA), (4096, 300, 17, q.PATH_MMA),
                                         (96, 130, 64, q.PATH_MMA), (4096, 256, 512, q.PATH_MMA)])
def test_product_parity(fmt, k, n, nt, path):
    rng = np.random.default_rng(k * 3 + n + nt)
    w = qmm_synth.gen_weights(fmt, k, n, rng)
    x = qmm_synth.gen_x(nt, k, rng)
    y = q.matmul(fmt, _dev(w), _dev(x), k, n, path=path)
    torch.cuda.synchronize()
    q.qmm_device_status()
    y_ref, s_ref = oracle.matmul(fmt, w, x, k, n)
    _assert(y.cpu().numpy(), y_ref, s_ref, f"{fmt} k={k} n={n} N={nt} path={path}")


@pytest.mark.parametrize("fmt", BLOCK32)
@pytest.mark.parametrize("k,n,r0,r1,acc", [(4096, 1000, 0, 1000, False), (2048, 333, 64, 300, True),
                                           (32, 9, 0, 9, False)])
def test_backward_input_parity(fmt, k, n, r0, r1, acc):
    """dx (+)= sum over the rows j in [r0, r1) of dy_j w_j."""
    rng = np.random.default_rng(k + n + r0)
    w = qmm_synth.gen_weights(fmt, k, n, rng)
    dy = qmm_synth.gen_x(1, n, rng)[0]
    dx_in = rng.normal(0, 1, k).astype(np.float32)
    dx = q.matmul_backward_input(fmt, _dev(w), _dev(dy), k, n, dx=_dev(dx_in), j_start=r0,
                                 j_end=r1, accumulate=acc)
    torch.cuda.synchronize()
    q.qmm_device_status()
    ref, s = oracle.matmul_back_input(fmt, w, dy, k, n, r0, r1)
    if acc:
        ref, s = ref + dx_in, s + np.abs(dx_in)
    _assert(dx.cpu().numpy()[None, :], ref[None, :], s[None, :], f"backward {fmt} k={k} n={n}")


# ------------------------------------------------------- expert product ----

def _experts(fmt, w, x, ids, k, n, n_exp, **kw):
    y0 = kw.pop("y0", None)
    y = _dev(y0) if y0 is not None else None
    out = q.matmul_experts(fmt, _dev(w), _dev(x), _dev(ids), k, n, n_exp, y=y, **kw)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("name", sorted(qmm_synth.EXPERT_WORKLOADS))
@pytest.mark.parametrize("n_pos", [1, 4])
def test_experts_workloads(name, n_pos):
    fmt, k, n, n_exp, w, x, ids = qmm_synth.expert_workload(name, n_pos=n_pos)
    y = _experts(fmt, w, x, ids, k, n, n_exp)
    q.qmm_device_status()
    y_ref, s_ref = oracle.matmul_experts(fmt, w, x, k, n, n_exp, ids)
    _assert(y.cpu().numpy(), y_ref, s_ref, f"{name} n_pos={n_pos}")


@pytest.mark.parametrize("fmt,k,n,n_exp,top_k,n_pos", [
    ("q4_k", 512, 130, 5, 2, 3), ("q6_k", 256, 64, 3, 3, 2), ("bf16", 96, 77, 4, 1, 5),
    ("q4_0", 96, 33, 7, 7, 1), ("q8_0", 32, 1, 2, 2, 2), ("f16", 64, 300, 6, 4, 2)])
def test_experts_every_format(fmt, k, n, n_exp, top_k, n_pos):
    rng = np.random.default_rng(n_exp * 100 + k + n)
    w = qmm_synth.gen_weights(fmt, k, n * n_exp, rng)
    x = qmm_synth.gen_x(n_pos, k, rng)
    ids = qmm_synth.gen_ids(n_pos, top_k, n_exp, rng)
    y = _experts(fmt, w, x, ids, k, n, n_exp)
    q.qmm_device_status()
    y_ref, s_ref = oracle.matmul_experts(fmt, w, x, k, n, n_exp, ids)
    _assert(y.cpu().numpy(), y_ref, s_ref, f"experts {fmt}")


def test_experts_repeated_ids_tile_and_accumulate():
    """The same expert in several slots (ids need not be distinct across
    positions), a column tile, and accumulation onto a prefilled y."""
    fmt, k, n, n_exp = "q5_0", 1024, 500, 4
    rng = np.random.default_rng(77)
    w = qmm_synth.gen_weights(fmt, k, n * n_exp, rng)
    x = qmm_synth.gen_x(3, k, rng)
    ids = np.array([[3, 3], [0, 2], [3, 1]], np.int32)
    y_in = rng.normal(0, 1, (6, n)).astype(np.float32)
    j0, j1 = 37, 411
    y = _experts(fmt, w, x, ids, k, n, n_exp, y0=y_in, j_start=j0, j_end=j1,
                 accumulate=True).cpu().numpy()
    q.qmm_device_status()
    y_ref, s_ref = oracle.matmul_experts(fmt, w, x, k, n, n_exp, ids)
    y_exp, s_exp = oracle.tiled(y_ref, s_ref, j0, j1, True, y_in)
    outside = np.ones(n, bool)
    outside[j0:j1] = False
    assert np.array_equal(y[:, outside].view(np.uint32), y_in[:, outside].view(np.uint32))
    _assert(y[:, j0:j1], y_exp[:, j0:j1], s_exp[:, j0:j1], "experts tile accumulate")
    # the two slots of position 0 chose the same expert: identical rows
    y = _experts(fmt, w, x, ids, k, n, n_exp).cpu().numpy()
    assert np.array_equal(y[0].view(np.uint32), y[1].view(np.uint32))


def test_experts_one_expert_equals_plain_product():
    """n_experts = 1, top_k = 1: the expert product is the one-token GEMV, bit for bit."""
    fmt, k, n = "q8_0", 2048, 768
    rng = np.random.default_rng(3)
    w = qmm_synth.gen_weights(fmt, k, n, rng)
    x = qmm_synth.gen_x(1, k, rng)
    ids = np.zeros((1, 1), np.int32)
    y_e = _experts(fmt, w, x, ids, k, n, 1).cpu().numpy()
    y_p = q.matmul(fmt, _dev(w), _dev(x), k, n, path=q.PATH_GEMV)
    torch.cuda.synchronize()
    assert np.array_equal(y_e.view(np.uint32), y_p.cpu().numpy().view(np.uint32))


def test_experts_bad_id_reported_and_row_untouched():
    fmt, k, n, n_exp = "q8_0", 256, 100, 4
    rng = np.random.default_rng(11)
    w = qmm_synth.gen_weights(fmt, k, n * n_exp, rng)
    x = qmm_synth.gen_x(2, k, rng)
    ids = np.array([[1, 4], [-1, 2]], np.int32)
    y_in = np.full((4, n), 7.0, np.float32)
    y = _experts(fmt, w, x, ids, k, n, n_exp, y0=y_in).cpu().numpy()
    with pytest.raises(q.QmmError) as ei:
        q.qmm_device_status()
    assert ei.value.status == 11
    q.qmm_device_status()   # the flag was cleared
    assert np.all(y[1] == 7.0) and np.all(y[2] == 7.0)
    good = np.array([[1, 1], [2, 2]], np.int32)
    y_ref, s_ref = oracle.matmul_experts(fmt, w, x, k, n, n_exp, good)
    _assert(y[[0, 3]], y_ref[[0, 3]], s_ref[[0, 3]], "rows with valid ids")


def test_experts_k_zero_and_empty_tile():
    y_in = np.full((2, 8), 3.0, np.float32)
    ids = np.zeros((2, 1), np.int32)
    w = np.zeros(0, np.uint8)
    x = np.zeros((2, 0), np.float32)
    y = _experts("q8_0", w, x, ids, 0, 8, 1, y0=y_in).cpu().numpy()
    assert np.all(y == 0.0)
    y = _experts("q8_0", w, x, ids, 0, 8, 1, y0=y_in, j_start=4, j_end=4).cpu().numpy()
    assert np.all(y == 3.0)


def test_experts_overlapped_launches():
    """Under programmatic dependent launch: ids rewritten by the preceding
    kernel are read after it (OVERLAP_PREV alone), and a chain of accumulating
    calls with X_READY stores in order."""
    fmt, k, n, n_exp = "q8_0", 2048, 768, 16
    rng = np.random.default_rng(21)
    w = qmm_synth.gen_weights(fmt, k, n * n_exp, rng)
    x = qmm_synth.gen_x(2, k, rng)
    ids_a = qmm_synth.gen_ids(2, 4, n_exp, rng)
    ids_b = qmm_synth.gen_ids(2, 4, n_exp, rng)
    wd, xd = _dev(w), _dev(x)
    idd = _dev(ids_a)
    src = _dev(ids_b)
    y = torch.zeros((8, n), device=DEV)
    for _ in range(3):
        idd.copy_(_dev(ids_a))
        q.matmul_experts(fmt, wd, xd, idd, k, n, n_exp, y=y)
        idd.copy_(src)   # the preceding kernel writes the ids
        q.matmul_experts(fmt, wd, xd, idd, k, n, n_exp, y=y, flags=q.FLAG_OVERLAP_PREV)
    torch.cuda.synchronize()
    q.qmm_device_status()
    y_ref, s_ref = oracle.matmul_experts(fmt, w, x, k, n, n_exp, ids_b)
    _assert(y.cpu().numpy(), y_ref, s_ref, "ids written by the preceding kernel")
    y.zero_()
    for _ in range(4):
        q.matmul_experts(fmt, wd, xd, idd, k, n, n_exp, y=y, accumulate=True,
                         flags=q.FLAG_OVERLAP_PREV | q.FLAG_X_READY)
    torch.cuda.synchronize()
    q.qmm_device_status()
    _assert(y.cpu().numpy(), 4 * y_ref, 4 * s_ref, "accumulating chain")


def test_experts_many_pairs():
    """A prefill-sized routing (64 positions x top 8 = 512 pairs, each pair
    one CTA's GEMV over its slice), ids repeating across positions."""
    fmt, k, n, n_exp = "q4_k", 256, 64, 16
    rng = np.random.default_rng(91)
    w = qmm_synth.gen_weights(fmt, k, n * n_exp, rng)
    x = qmm_synth.gen_x(64, k, rng)
    ids = qmm_synth.gen_ids(64, 8, n_exp, rng)
    y = _experts(fmt, w, x, ids, k, n, n_exp)
    q.qmm_device_status()
    y_ref, s_ref = oracle.matmul_experts(fmt, w, x, k, n, n_exp, ids)
    _assert(y.cpu().numpy(), y_ref, s_ref, "512 pairs")
