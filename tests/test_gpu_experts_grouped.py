"""GPU parity of the grouped (tensor-core) form of the expert-indexed product,
through the C ABI, against the oracle: the (position, slot) pairs are routed
by expert on the device and each expert's rows go through one tensor-core
pass over its slice (rullama src/backend/dispatch/mod.rs, the batched expert
matmul and its test `moe_expert_matmul_batched_gpu_vs_cpu`). Per output
|y - y_ref| <= 1e-4 * sum_i |x_i w_ij| and cosine >= 0.9999."""
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
    yield
    q.qmm_device_status()


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _run(fmt, w, x, ids, k, n, n_exp, **kw):
    y0 = kw.pop("y0", None)
    y = _dev(y0.astype(np.float32)) if y0 is not None else None
    out = q.matmul_experts(fmt, _dev(w), _dev(x), _dev(ids), k, n, n_exp, y=y, **kw)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _assert(y, y_ref, s_ref, what):
    ok, worst, cos, msg = oracle.check(y, y_ref, s_ref)
    assert ok, f"{what}: {msg}"


def test_auto_policy_picks_the_grouped_form():
    k, n, n_exp, top_k = 2048, 256, 16, 4
    a = q.make_args("q4_k", 16, 16, 16, k, n, 64, stream=0)
    assert q.qmm_experts_workspace_bytes(a, n_exp, top_k) > 0     # 256 pairs >= 2 * 16
    a = q.make_args("q4_k", 16, 16, 16, k, n, 4, stream=0)
    assert q.qmm_experts_workspace_bytes(a, n_exp, top_k) == 0    # 16 pairs: one GEMV each
    a = q.make_args("q4_k", 16, 16, 16, 512, n, 64, stream=0)
    assert q.qmm_experts_workspace_bytes(a, n_exp, top_k) == 0    # k < 1024: GEMV form
    a = q.make_args("q4_k", 16, 16, 16, 512, n, 64, path=q.PATH_MMA, stream=0)
    assert q.load().qmm_matmul_experts(ctypes.byref(a), 16, n_exp, top_k) == 10
    # the other raw-tile formats group from two pairs per expert; Q6_K from three
    for fmt, n_pos, grouped in (("q8_0", 64, True), ("q5_0", 64, True), ("q4_0", 64, True),
                                ("q8_0", 8, True), ("q6_k", 64, True), ("q6_k", 12, True),
                                ("q6_k", 11, False), ("q6_k", 8, False)):
        a = q.make_args(fmt, 16, 16, 16, k, n, n_pos, stream=0)
        assert (q.qmm_experts_workspace_bytes(a, n_exp, top_k) > 0) == grouped, (fmt, n_pos)


@pytest.mark.parametrize("fmt,k", [("q4_k", 2048), ("q8_0", 2048), ("q5_0", 1024), ("q6_k", 1024),
                                   ("q4_0", 2048), ("bf16", 1024), ("f16", 1024)])
def test_grouped_matches_oracle(fmt, k):
    n, n_exp, top_k, n_pos = 300, 16, 4, 64   # 300 rows: a ragged row tile
    rng = np.random.default_rng(k + len(fmt))
    w = qmm_synth.gen_weights(fmt, k, n * n_exp, rng)
    x = qmm_synth.gen_x(n_pos, k, rng)
    ids = qmm_synth.gen_ids(n_pos, top_k, n_exp, rng)
    y = _run(fmt, w, x, ids, k, n, n_exp, path=q.PATH_MMA)
    q.qmm_device_status()
    y_ref, s_ref = oracle.matmul_experts(fmt, w, x, k, n, n_exp, ids)
    _assert(y, y_ref, s_ref, f"grouped {fmt} k={k}")


def test_moe_ffn_shape_64_positions_and_determinism():
    """The expert workload's shape (64 experts of 768 rows, k = 2048, top 8)
    at 64 positions: 512 pairs, 8 per expert on average."""
    for name in ("q4_k_experts", "q8_0_experts"):
        fmt, k, n, n_exp, w, x, ids = qmm_synth.expert_workload(name, n_pos=64)
        y = _run(fmt, w, x, ids, k, n, n_exp, path=q.PATH_MMA)
        q.qmm_device_status()
        y_ref, s_ref = oracle.matmul_experts(fmt, w, x, k, n, n_exp, ids)
        _assert(y, y_ref, s_ref, f"{name}, 64 positions")
        y2 = _run(fmt, w, x, ids, k, n, n_exp, path=q.PATH_MMA)
        assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))
        yg = _run(fmt, w, x, ids, k, n, n_exp, path=q.PATH_GEMV)   # the per-pair form agrees too
        _assert(yg, y_ref, s_ref, f"{name}, GEMV form")


def test_skewed_routing_tiles_and_accumulate():
    """Every pair of most positions on one expert (many token tiles for it),
    experts that get no rows, a column tile, then an accumulating tile."""
    fmt, k, n, n_exp, top_k, n_pos = "q4_k", 1024, 384, 8, 2, 150
    rng = np.random.default_rng(77)
    w = qmm_synth.gen_weights(fmt, k, n * n_exp, rng)
    x = qmm_synth.gen_x(n_pos, k, rng)
    ids = np.zeros((n_pos, top_k), np.int32)
    ids[:, 0] = 3
    ids[:, 1] = np.where(np.arange(n_pos) % 5 == 0, 6, 1)
    y0 = rng.normal(size=(n_pos * top_k, n)).astype(np.float32)
    y = _run(fmt, w, x, ids, k, n, n_exp, y0=y0, j_start=100, j_end=300, path=q.PATH_MMA)
    q.qmm_device_status()
    y_ref, s_ref = oracle.matmul_experts(fmt, w, x, k, n, n_exp, ids)
    exp, s_exp = oracle.tiled(y_ref, s_ref, 100, 300, False, y0)
    _assert(y, exp, s_exp, "skewed, tile [100, 300)")
    y1 = _run(fmt, w, x, ids, k, n, n_exp, y0=y, j_start=100, j_end=300, accumulate=True,
              path=q.PATH_MMA)
    q.qmm_device_status()
    exp2, s_exp2 = oracle.tiled(y_ref, s_ref, 100, 300, True, y)
    _assert(y1, exp2, s_exp2, "skewed, accumulated tile")


def test_bad_ids_leave_rows_untouched_and_are_reported():
    fmt, k, n, n_exp, top_k, n_pos = "q8_0", 1024, 200, 6, 2, 40
    rng = np.random.default_rng(5)
    w = qmm_synth.gen_weights(fmt, k, n * n_exp, rng)
    x = qmm_synth.gen_x(n_pos, k, rng)
    ids = qmm_synth.gen_ids(n_pos, top_k, n_exp, rng)
    ids[3, 1] = -1
    ids[17, 0] = n_exp
    y0 = np.full((n_pos * top_k, n), 7.0, np.float32)
    y = _run(fmt, w, x, ids, k, n, n_exp, y0=y0, path=q.PATH_MMA)
    with pytest.raises(q.QmmError) as ei:
        q.qmm_device_status()
    assert ei.value.status == 11
    assert (y[3 * top_k + 1] == 7.0).all() and (y[17 * top_k] == 7.0).all()
    good = np.ones(n_pos * top_k, bool)
    good[[3 * top_k + 1, 17 * top_k]] = False
    ids_ok = np.where(ids < 0, 0, np.where(ids >= n_exp, 0, ids)).astype(np.int32)
    y_ref, s_ref = oracle.matmul_experts(fmt, w, x, k, n, n_exp, ids_ok)
    _assert(y[good], y_ref[good], s_ref[good], "rows with valid ids")
