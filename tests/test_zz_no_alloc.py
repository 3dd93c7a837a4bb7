"""qmm_matmul_noalloc: the tensor-core product for callers that cannot
allocate device memory (no CUDA allocator of their own, or no allocating,
device-synchronizing calls allowed on their hot path). Its scratch is a fixed
16 MiB array inside libqmm. Checked through the C ABI against the ordinary
entry point (qmm_matmul_ex with a caller-allocated workspace) on two calls in
a row, so the second call runs over the scratch the first one left behind:
both run the same kernels on the same inputs, so their outputs must agree bit
for bit, and the allocation-free output must also meet the product bar
against the oracle."""
import ctypes

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


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _existing(fmt, wd, xd, k, n):
    """The ordinary entry point on the tensor-core path, caller-owned workspace."""
    nt = xd.shape[0]
    y = torch.empty((nt, n), device=DEV)
    a = q.make_args(fmt, wd, xd, y, k, n, nt, path=q.PATH_MMA)
    need = q.qmm_workspace_bytes(a)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    a.workspace, a.workspace_bytes = ws.data_ptr(), need
    q.qmm_matmul_ex(a)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def _noalloc(fmt, wd, xd, k, n):
    nt = xd.shape[0]
    y = torch.full((nt, n), float("nan"), device=DEV)
    a = q.make_args(fmt, wd, xd, y, k, n, nt)
    rc = q.load().qmm_matmul_noalloc(ctypes.byref(a))
    assert rc == 0, q.qmm_last_error()
    torch.cuda.synchronize()
    q.qmm_device_status()
    return y.cpu().numpy()


@pytest.mark.parametrize("fmt,k,n,nt", [("q4_k", 4096, 1000, 64),   # raw Q4_K tiles, x split
                                        ("bf16", 512, 300, 40)])     # 16-bit rows, x split
def test_noalloc_matches_existing_entry_point_twice(fmt, k, n, nt):
    rng = np.random.default_rng(31 + nt)
    w = qmm_synth.gen_weights(fmt, k, n, rng)
    wd = _dev(w)
    for call in range(2):
        x = qmm_synth.gen_x(nt, k, rng)
        xd = _dev(x)
        got = _noalloc(fmt, wd, xd, k, n)
        ref = _existing(fmt, wd, xd, k, n)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), \
            f"call {call}: allocation-free and ordinary outputs differ"
        y_ref, s_ref = oracle.matmul_blas(fmt, w, x, k, n)
        ok, worst, cos, msg = oracle.check(got, y_ref, s_ref)
        assert ok, f"call {call}: {msg}"


def test_noalloc_rejects_calls_beyond_the_scratch():
    k, n, nt = 4096, 8, 4096   # fp16 copy of x alone is 32 MiB > 16 MiB
    a = q.make_args("q4_k", 16 * 1000, 16 * 2000, 16 * 3000, k, n, nt, stream=0)
    rc = q.load().qmm_matmul_noalloc(ctypes.byref(a))
    assert rc == 9  # QMM_ERR_WORKSPACE, nothing enqueued
    assert "scratch" in q.qmm_last_error()
