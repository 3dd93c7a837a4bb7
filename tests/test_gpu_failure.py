"""Failure detection without a GPU fault: a kernel whose barrier wait nothing
satisfies gives up after its limit, records the fault, and returns; the host
reads it through qmm_device_status (QMM_ERR_DEVICE_TIMEOUT, then cleared)
and the context stays usable for the next product."""
import time

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


def test_bounded_wait_gives_up_and_is_reported():
    torch.cuda.init()
    assert q.qmm_device_status() == 0
    t0 = time.monotonic()
    q.qmm_check_bounded_wait()
    with pytest.raises(q.QmmError) as ei:
        q.qmm_device_status()
    waited = time.monotonic() - t0
    assert ei.value.status == 8, q.qmm_last_error()
    assert 0.04 <= waited < 30.0, waited
    assert q.qmm_device_status() == 0          # the flag was cleared
    # the context is usable: a product right after is correct
    rng = np.random.default_rng(2)
    k, n = 512, 300
    w = qmm_synth.gen_weights("q4_k", k, n, rng)
    x = qmm_synth.gen_x(1, k, rng)
    y = q.matmul("q4_k", torch.from_numpy(w).to(DEV), torch.from_numpy(x).to(DEV), k, n)
    torch.cuda.synchronize()
    assert q.qmm_device_status() == 0
    y_ref, s_ref = oracle.matmul("q4_k", w, x, k, n)
    ok, worst, cos, msg = oracle.check(y.cpu().numpy(), y_ref, s_ref)
    assert ok, msg
