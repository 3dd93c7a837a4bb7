"""GPU parity of the backward with respect to the input, dx = W^T dy over a
row range of the sum axis (through the C ABI), against the oracle: per entry
|dx - dx_ref| <= 1e-4 * sum_j |dy_j w_ji| (+ |dx_in| when accumulating) and
cosine >= 0.9999."""
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


def _run(fmt, w, dy, k, n, **kw):
    dx0 = kw.pop("dx0", None)
    dx = _dev(dx0.astype(np.float32)) if dx0 is not None else None
    out = q.matmul_backward_input(fmt, _dev(w), _dev(dy), k, n, dx=dx, **kw)
    torch.cuda.synchronize()
    q.qmm_device_status()
    return out.cpu().numpy()


def _assert(dx, ref, s, what):
    ok, worst, cos, msg = oracle.check(dx[None, :], ref[None, :], s[None, :])
    assert ok, f"{what}: {msg}"


def _random_block_bytes(fmt, k, n, seed):
    """Uniform random bytes with the f16 super-block scales clamped to small
    finite values (random f16 patterns can be NaN or Inf)."""
    rng = np.random.default_rng(seed)
    rb = oracle.row_bytes(fmt, k)
    w = rng.integers(0, 256, size=n * rb, dtype=np.uint8).reshape(n, rb)
    if fmt == "q4_0":
        for b in range(k // 32):
            w[:, 18 * b:18 * b + 2] = [0x00, 0x2C]          # d = 0.0625
    elif fmt == "q4_k":
        for b in range(k // 256):
            w[:, 144 * b:144 * b + 4] = [0x00, 0x2C, 0x00, 0x28]  # d, dmin
    elif fmt == "q6_k":
        for b in range(k // 256):
            w[:, 210 * b + 208:210 * b + 210] = [0x00, 0x28]   # d = 0.03125
    return w.reshape(-1)


@pytest.mark.parametrize("fmt,k,n", [("q4_0", 64, 16), ("q4_k", 256, 16), ("q6_k", 256, 16)])
def test_back_input_small_random_blocks(fmt, k, n):
    w = _random_block_bytes(fmt, k, n, seed=k + n)
    dy = np.array([(j - 8) * 0.25 for j in range(n)], np.float32)
    dx = _run(fmt, w, dy, k, n)
    ref, s = oracle.matmul_back_input(fmt, w, dy, k, n)
    _assert(dx, ref, s, f"{fmt} k={k} n={n}")


@pytest.mark.parametrize("fmt,k,n", [("q4_k", 4096, 1500), ("q6_k", 2560, 777), ("q4_0", 256, 1001),
                                     ("q4_k", 512, 3), ("q6_k", 8192, 40), ("bf16", 2048, 300),
                                     ("f16", 1000, 77), ("q4_0", 8192, 65)])
def test_back_input_synthetic(fmt, k, n):
    rng = np.random.default_rng(7)
    w = qmm_synth.gen_weights(fmt, k, n, rng)
    dy = rng.standard_normal(n).astype(np.float32)
    dx = _run(fmt, w, dy, k, n)
    ref, s = oracle.matmul_back_input(fmt, w, dy, k, n)
    _assert(dx, ref, s, f"{fmt} k={k} n={n}")


def test_back_input_sum_axis_tiles_and_accumulate():
    """Three tiles of the sum axis: the first writes, the others add; the
    result matches the whole-range oracle, and an empty tile writes zeros."""
    fmt, k, n = "q6_k", 2560, 4099
    rng = np.random.default_rng(3)
    w = qmm_synth.gen_weights(fmt, k, n, rng)
    dy = rng.standard_normal(n).astype(np.float32)
    wd, dyd = _dev(w), _dev(dy)
    dx = torch.full((k,), 7.0, device=DEV)
    for t, (a, b) in enumerate([(0, 1500), (1500, 1501), (1501, n)]):
        q.matmul_backward_input(fmt, wd, dyd, k, n, dx=dx, j_start=a, j_end=b, accumulate=t > 0)
    torch.cuda.synchronize()
    q.qmm_device_status()
    ref, s = oracle.matmul_back_input(fmt, w, dy, k, n)
    _assert(dx.cpu().numpy(), ref, s, "three tiles")
    # accumulate onto a prefilled dx
    dx0 = rng.standard_normal(k).astype(np.float32)
    got = _run(fmt, w, dy, k, n, dx0=dx0, j_start=100, j_end=2000, accumulate=True)
    ref2, s2 = oracle.matmul_back_input(fmt, w, dy, k, n, 100, 2000)
    _assert(got, ref2 + dx0, s2 + np.abs(dx0), "accumulate")
    # empty range: zeros
    got = _run(fmt, w, dy, k, n, dx0=dx0, j_start=9, j_end=9)
    assert not got.any()


def test_back_input_repeatable_bits():
    fmt, k, n = "q4_k", 4096, 14336
    rng = np.random.default_rng(1)
    w = qmm_synth.gen_weights(fmt, k, n, rng)
    dy = rng.standard_normal(n).astype(np.float32)
    wd, dyd = _dev(w), _dev(dy)
    a = q.matmul_backward_input(fmt, wd, dyd, k, n).cpu().numpy()
    b = q.matmul_backward_input(fmt, wd, dyd, k, n).cpu().numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    ref, s = oracle.matmul_back_input_blas(fmt, w, dy, k, n)
    _assert(a, ref, s, "q4_k ffn backward")


def test_back_input_q6_k_head_tiles_full_size():
    """The output head (k=2560, n=262144) in 8 sum-axis tiles of 32768 rows;
    the first and the last tile are checked alone against the oracle, and the
    tiled sum against the whole-range oracle over all rows."""
    fmt, k, n, w, _ = qmm_synth.workload("q6_k_head")
    rng = np.random.default_rng(4)
    dy = rng.standard_normal(n).astype(np.float32)
    wd, dyd = _dev(w), _dev(dy)
    step = 32768
    first = q.matmul_backward_input(fmt, wd, dyd, k, n, j_start=0, j_end=step).cpu().numpy()
    ref, s = oracle.matmul_back_input(fmt, w, dy, k, n, 0, step)
    _assert(first, ref, s, "head tile 0")
    last = q.matmul_backward_input(fmt, wd, dyd, k, n, j_start=n - step, j_end=n).cpu().numpy()
    ref, s = oracle.matmul_back_input(fmt, w, dy, k, n, n - step, n)
    _assert(last, ref, s, "head tile 7")
    dx = torch.empty(k, device=DEV)
    for t in range(8):
        q.matmul_backward_input(fmt, wd, dyd, k, n, dx=dx, j_start=t * step,
                                j_end=(t + 1) * step, accumulate=t > 0)
    torch.cuda.synchronize()
    q.qmm_device_status()
    ref, s = oracle.matmul_back_input(fmt, w, dy, k, n)
    _assert(dx.cpu().numpy(), ref, s, "head, 8 tiles")


def test_back_input_overlapped_tiles():
    """Sum-axis tiles under programmatic launch: with OVERLAP_PREV | X_READY
    (dy not written by the preceding kernels) and with OVERLAP_PREV alone
    after a kernel that rewrites dy, the result matches the whole-range
    oracle."""
    fmt, k, n = "q4_k", 4096, 14336
    rng = np.random.default_rng(8)
    w = qmm_synth.gen_weights(fmt, k, n, rng)
    dy = rng.standard_normal(n).astype(np.float32)
    ref, s = oracle.matmul_back_input(fmt, w, dy, k, n)
    wd, dyd = _dev(w), _dev(dy)
    tiles = [(0, 3000), (3000, 3001), (3001, 9000), (9000, n)]
    for flags in (q.FLAG_OVERLAP_PREV | q.FLAG_X_READY, q.FLAG_OVERLAP_PREV):
        dx = torch.full((k,), 5.0, device=DEV)
        src = torch.zeros(n, device=DEV)
        for t, (a, b) in enumerate(tiles):
            if flags == q.FLAG_OVERLAP_PREV:
                src.copy_(dyd)          # the preceding kernel writes dy
                dyt = src
            else:
                dyt = dyd
            q.matmul_backward_input(fmt, wd, dyt, k, n, dx=dx, j_start=a, j_end=b,
                                    accumulate=t > 0, flags=flags)
        torch.cuda.synchronize()
        q.qmm_device_status()
        _assert(dx.cpu().numpy(), ref, s, f"overlapped tiles flags={flags}")
