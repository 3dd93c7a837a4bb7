"""The calls are stream-ordered and allocation-free when the caller passes its
scratch, so a sequence of them can be captured in a CUDA graph and replayed:
the replay gives bit-identical outputs to the eager calls (programmatic
launches included)."""
import numpy as np
import pytest

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
    yield
    q.qmm_device_status()


def _dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(DEV)


def test_graph_capture_and_replay_bit_identical():
    rng = np.random.default_rng(17)
    k, n = 4096, 1536
    w1 = _dev(qmm_synth.gen_weights("q4_k", k, n, rng))
    w2 = _dev(qmm_synth.gen_weights("q4_k", k, n, rng))
    wa, sc, bi = qmm_synth.gen_affine(4, k, n, rng)
    wa, sc, bi = _dev(wa), _dev(sc), _dev(bi)
    x1 = _dev(qmm_synth.gen_x(1, k, rng))
    x64 = _dev(qmm_synth.gen_x(64, k, rng))
    s = torch.cuda.Stream(device=DEV)
    y1 = torch.empty((1, n), device=DEV)
    y2 = torch.empty((1, n), device=DEV)
    yg = torch.empty((1, n), device=DEV)
    ya = torch.empty((1, n), device=DEV)
    y64 = torch.empty((64, n), device=DEV)
    ov = q.FLAG_OVERLAP_PREV | q.FLAG_X_READY
    a1 = q.make_args("q4_k", w1, x1, y1, k, n, 1, stream=s)
    a2 = q.make_args("q4_k", w2, x1, y2, k, n, 1, stream=s, flags=ov)
    ag = q.make_args("q4_k", w1, x1, yg, k, n, 1, stream=s, flags=ov)
    aa = q.make_args("affine4", wa, x1, ya, k, n, 1, stream=s, flags=ov)
    am = q.make_args("q4_k", w2, x64, y64, k, n, 64, stream=s)
    need = q.qmm_workspace_bytes(am)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    am.workspace, am.workspace_bytes = ws.data_ptr(), need

    def seq():
        q.qmm_matmul_ex(a1)
        q.qmm_matmul_ex(a2)
        q.qmm_matmul_glu(ag, w2, q.ACT_SWIGLU)
        q.qmm_matmul_affine(aa, sc, bi)
        q.qmm_matmul_ex(am)

    outs = (y1, y2, yg, ya, y64)
    with torch.cuda.stream(s):
        seq()                       # eager (also sets kernel attributes once)
    s.synchronize()
    q.qmm_device_status(s)
    eager = [o.cpu().numpy().copy() for o in outs]
    for o in outs:
        o.fill_(float("nan"))
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        seq()
    for _ in range(3):
        for o in outs:
            o.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        q.qmm_device_status()
        for e, o in zip(eager, outs):
            got = o.cpu().numpy()
            assert np.array_equal(got.view(np.uint32), e.view(np.uint32))
