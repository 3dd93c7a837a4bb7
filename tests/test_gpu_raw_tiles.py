"""GPU parity of the tensor-core path for the formats whose W tiles are staged
raw (Q4_0, Q5_0, Q8_0 by TMA at k % 256 == 0, k >= 1024; Q6_K by per-row bulk
copies from 16-byte boundaries, the matrix's last bytes by plain loads),
against the oracle through the C ABI: row counts that leave a ragged last row tile (the
tile's rows past n are the map's zero fill), token counts that leave a
partial token tile, output-axis windows (the tile's first row is then j_start,
not a multiple of 128) written or accumulated, and the k % 256 != 0 shapes
that keep the per-thread path. Columns outside a window keep their bits."""
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


CASES = [  # (fmt, k, n, n_tokens)
    ("q8_0", 1024, 129, 3), ("q8_0", 4096, 1000, 37), ("q8_0", 2048, 257, 130),
    ("q5_0", 1024, 1, 9), ("q5_0", 4096, 383, 64), ("q5_0", 3072, 640, 200),
    ("q4_0", 2048, 127, 17), ("q4_0", 4096, 900, 129), ("q4_0", 1280, 256, 5),
    ("q6_k", 2560, 131, 7), ("q6_k", 4096, 1000, 64), ("q6_k", 1024, 1, 33),
    ("q6_k", 1536, 385, 130),
    ("bf16", 4096, 1000, 37), ("f16", 2048, 257, 130), ("bf16", 1000, 129, 9),
]


@pytest.mark.parametrize("fmt,k,n,nt", CASES)
def test_raw_tile_block_formats(fmt, k, n, nt):
    rng = np.random.default_rng(k + n + nt + len(fmt))
    w = qmm_synth.gen_weights(fmt, k, n, rng)
    x = qmm_synth.gen_x(nt, k, rng)
    y_ref, s_ref = oracle.matmul_blas(fmt, w, x, k, n)
    y = q.matmul(fmt, _dev(w), _dev(x), k, n, path=q.PATH_MMA)
    torch.cuda.synchronize()
    q.qmm_device_status()
    ok, worst, cos, msg = oracle.check(y.cpu().numpy(), y_ref, s_ref)
    assert ok, f"{fmt} k={k} n={n} N={nt}: {msg}"
    # an output window that starts off a 128-row boundary, accumulated into y
    if n > 8:
        j0, j1 = n // 3 + 1, n - 2
        y_in = rng.normal(0, 1, (nt, n)).astype(np.float32)
        yd = _dev(y_in)
        q.matmul(fmt, _dev(w), _dev(x), k, n, y=yd, j_start=j0, j_end=j1, accumulate=True,
                 path=q.PATH_MMA)
        torch.cuda.synchronize()
        q.qmm_device_status()
        yt = yd.cpu().numpy()
        y_exp, s_exp = oracle.tiled(y_ref, s_ref, j0, j1, True, y_in)
        for sl in (slice(0, j0), slice(j1, n)):
            assert np.array_equal(yt[:, sl].view(np.uint32), y_in[:, sl].view(np.uint32))
        ok, worst, cos, msg = oracle.check(yt[:, j0:j1], y_exp[:, j0:j1], s_exp[:, j0:j1])
        assert ok, f"{fmt} window [{j0}, {j1}) accumulated: {msg}"


@pytest.mark.parametrize("fmt", ["q8_0", "q5_0", "q4_0"])
def test_k_not_a_multiple_of_256_keeps_the_per_thread_path(fmt):
    """k = 1056 (a multiple of 32, not of 256): the W and x split mode on the
    per-thread path, at the same bar."""
    k, n, nt = 1056, 300, 24
    rng = np.random.default_rng(99 + len(fmt))
    w = qmm_synth.gen_weights(fmt, k, n, rng)
    x = qmm_synth.gen_x(nt, k, rng)
    y = q.matmul(fmt, _dev(w), _dev(x), k, n, path=q.PATH_MMA)
    torch.cuda.synchronize()
    q.qmm_device_status()
    y_ref, s_ref = oracle.matmul_blas(fmt, w, x, k, n)
    ok, worst, cos, msg = oracle.check(y.cpu().numpy(), y_ref, s_ref)
    assert ok, msg


@pytest.mark.parametrize("fmt", ["q8_0", "q6_k"])
def test_repeated_calls_give_the_same_bits(fmt):
    """The raw slot is released only after its last block is decoded: calls
    repeated into a poisoned output give identical bits."""
    k, n, nt = 4096, 2000, 256
    rng = np.random.default_rng(5)
    wd = _dev(qmm_synth.gen_weights(fmt, k, n, rng))
    xd = _dev(qmm_synth.gen_x(nt, k, rng))
    first = None
    for _ in range(5):
        y = torch.full((nt, n), float("nan"), dtype=torch.float32, device=DEV)
        q.matmul(fmt, wd, xd, k, n, y=y, path=q.PATH_MMA)
        torch.cuda.synchronize()
        q.qmm_device_status()
        yh = y.cpu().numpy()
        assert np.isfinite(yh).all()
        if first is None:
            first = yh
        else:
            assert np.array_equal(first.view(np.uint32), yh.view(np.uint32))


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
@pytest.mark.parametrize("k,n,nt", [(4096, 1000, 8), (2048, 257, 130), (1024, 129, 3)])
def test_16_bit_tiles_as_the_a_operand(fmt, k, n, nt):
    """16-bit W tiles go by TMA straight into shared memory as the MMA's A
    operand (k % 8 == 0); BF16 takes x as two bf16 terms."""
    rng = np.random.default_rng(k + n + nt + len(fmt))
    w = qmm_synth.gen_weights(fmt, k, n, rng)
    x = qmm_synth.gen_x(nt, k, rng)
    y = q.matmul(fmt, _dev(w), _dev(x), k, n, path=q.PATH_MMA)
    torch.cuda.synchronize()
    q.qmm_device_status()
    y_ref, s_ref = oracle.matmul_blas(fmt, w, x, k, n)
    ok, worst, cos, msg = oracle.check(y.cpu().numpy(), y_ref, s_ref)
    assert ok, f"{fmt} k={k} n={n} N={nt}: {msg}"


def test_bf16_weights_outside_the_fp16_range():
    """BF16 weights far above fp16's largest value and far below its normal
    range: bf16 operands carry them exactly (an fp16 copy would overflow or
    lose bits)."""
    k, n, nt = 4096, 256, 16
    rng = np.random.default_rng(7)
    vals = rng.normal(0, 1, (n, k)).astype(np.float32)
    vals[0::4] *= 1e5
    vals[1::4] *= 1e-6
    u = vals.view(np.uint32)
    w = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16).view(np.uint8).reshape(-1)
    x = qmm_synth.gen_x(nt, k, rng)
    y = q.matmul("bf16", _dev(w), _dev(x), k, n, path=q.PATH_MMA)
    torch.cuda.synchronize()
    q.qmm_device_status()
    y_ref, s_ref = oracle.matmul_blas("bf16", w, x, k, n)
    ok, worst, cos, msg = oracle.check(y.cpu().numpy(), y_ref, s_ref)
    assert ok, msg
