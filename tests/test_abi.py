"""C ABI checks that need no GPU: the library builds and loads, exports every
function include/qmm.h declares, sizes follow the closed forms, and invalid
calls are rejected on the host with the documented status before any CUDA
call is made."""
import ctypes
import os
import re

import pytest

import quantized_weight_gguf_gb300 as q
from quantized_weight_gguf_gb300 import build_lib

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "qmm.h")


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return q.load()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qmm_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 10
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(q.EXPORTS)


def test_version(lib):
    assert q.qmm_version() == 100


@pytest.mark.parametrize("fmt,k,n,expect", [
    ("bf16", 4096, 4096, 2 * 4096 * 4096),
    ("f16", 4096, 4096, 2 * 4096 * 4096),
    ("q4_0", 256, 512, 73728),
    ("q4_k", 4096, 14336, 33030144),
    ("q6_k", 2560, 262144, 550502400),
    ("q4_0", 96, 7, 54 * 7),
    ("q6_k", 1536, 1, 1260),
    ("q6_k", 6144, 1, 5040),
    ("q4_k", 128, 4, 0),     # k not a multiple of 256
    ("q4_0", 48, 4, 0),      # k not a multiple of 32
    ("bf16", 3, 4, 0),       # odd k
    ("bf16", -2, 4, 0),
    (9, 256, 4, 0),          # unknown format
])
def test_weight_bytes(lib, fmt, k, n, expect):
    assert q.qmm_weight_bytes(fmt, k, n) == expect


def _args(**kw):
    base = dict(fmt="q4_k", w=16 * 1000, x=16 * 2000, y=16 * 3000, k=512, n=8, n_tokens=1,
                stream=0)
    base.update(kw)
    fmt, w, x, y, k, n, nt = (base.pop(f) for f in ("fmt", "w", "x", "y", "k", "n", "n_tokens"))
    return q.make_args(fmt, w, x, y, k, n, nt, **base)


@pytest.mark.parametrize("kw,status", [
    (dict(fmt=9), 1),
    (dict(k=300), 2),
    (dict(fmt="q4_0", k=48), 2),
    (dict(fmt="bf16", k=7), 2),
    (dict(n_tokens=0), 2),
    (dict(n=-1), 2),
    (dict(w_len=10), 3),
    (dict(j_start=3, j_end=2), 4),
    (dict(j_start=0, j_end=9), 4),
    (dict(j_start=-1, j_end=4), 4),
    (dict(y=None), 5),
    (dict(w=None), 5),
    (dict(w=16 * 1000 + 8), 6),
    (dict(x=16 * 2000 + 2), 6),
    (dict(path=5), 2),
])
def test_invalid_calls_rejected_on_host(lib, kw, status):
    a = _args(**kw)
    rc = lib.qmm_matmul_ex(ctypes.byref(a))
    assert rc == status, (rc, q.qmm_last_error())
    assert q.qmm_last_error() != ""
    assert q.qmm_select_path(a) == (-1 if status in (1, 2, 3, 4) else q.qmm_select_path(a))


def test_error_message_names_the_problem(lib):
    a = _args(k=300)
    assert lib.qmm_matmul_ex(ctypes.byref(a)) == 2
    assert "multiple of 256" in q.qmm_last_error()
    a = _args(w_len=10)
    assert lib.qmm_matmul_ex(ctypes.byref(a)) == 3
    assert "W bytes" in q.qmm_last_error()


def test_row_alignment_constraint_dropped(lib):
    """Q4_0 with k=96 has 54-byte rows (not a multiple of 4); it is accepted."""
    a = _args(fmt="q4_0", k=96, w_len=54 * 8)
    assert q.qmm_select_path(a) in (q.PATH_GEMV, q.PATH_MMA)


def test_path_policy_and_workspace(lib):
    a = _args(k=4096, n=14336, n_tokens=1)
    assert q.qmm_select_path(a) == q.PATH_GEMV
    assert q.qmm_workspace_bytes(a) == 0
    # two tokens: two GEMVs (2 x 11.0 us) beat one tensor-core call (24.7 us)
    a = _args(k=4096, n=14336, n_tokens=2)
    assert q.qmm_select_path(a) == q.PATH_GEMV
    a = _args(k=4096, n=14336, n_tokens=3)
    assert q.qmm_select_path(a) == q.PATH_MMA
    a = _args(k=4096, n=14336, n_tokens=512)
    assert q.qmm_select_path(a) == q.PATH_MMA
    # x is always split into two fp16 terms (high part and remainder)
    assert q.qmm_workspace_bytes(a) == 2 * 512 * 4096 * 2 + 2048
    # 16-bit weights split x into two fp16 terms; k is padded to 64 in the copies
    a = _args(fmt="bf16", k=40, n=8, n_tokens=3)
    assert q.qmm_workspace_bytes(a) == 2 * ((3 * 64 * 2 + 255) // 256) * 256 + 256
    a = _args(k=512, n=8, n_tokens=3)              # small-k K-quant: split as well
    assert q.qmm_workspace_bytes(a) == 2 * 3 * 512 * 2 + 256
    a = _args(k=4096, n=14336, n_tokens=1, path=q.PATH_MMA)
    assert q.qmm_select_path(a) == q.PATH_MMA
    a = _args(k=4096, n=14336, n_tokens=64, path=q.PATH_GEMV)
    assert q.qmm_select_path(a) == q.PATH_GEMV
    assert q.qmm_workspace_bytes(a) == 0
    # W split into two fp16 terms as well: up to 8 tokens of a quantized
    # format take one exact GEMV each; 16-bit formats are unaffected
    for nt, path in ((8, q.PATH_GEMV), (9, q.PATH_MMA)):
        a = _args(k=4096, n=14336, n_tokens=nt, flags=q.FLAG_SPLIT_W)
        assert q.qmm_select_path(a) == path
    a = _args(fmt="bf16", k=4096, n=4096, n_tokens=3, w_len=0, flags=q.FLAG_SPLIT_W)
    assert q.qmm_select_path(a) == q.PATH_MMA
    a = _args(k=4096, n=14336, n_tokens=64, flags=q.FLAG_SPLIT_W)
    assert q.qmm_workspace_bytes(a) == 2 * 64 * 4096 * 2 + 256


def test_dequant_rejects_bad_args(lib):
    assert lib.qmm_dequant(9, 16, 256, 1, 16, None) == 1
    assert lib.qmm_dequant(3, 16, 100, 1, 16, None) == 2
    assert lib.qmm_dequant(3, None, 256, 1, 16, None) == 5
    assert lib.qmm_dequant(3, 24, 256, 1, 16, None) == 6


def test_host_variant_rejects_null_staging(lib):
    a = _args()
    assert lib.qmm_matmul_host(ctypes.byref(a), None, 16, 16) == 5


def test_empty_work_needs_no_device(lib):
    """n == 0 or an empty tile returns OK without touching CUDA."""
    assert lib.qmm_matmul_ex(ctypes.byref(_args(n=0))) == 0
    assert lib.qmm_matmul_ex(ctypes.byref(_args(j_start=3, j_end=3))) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(n_tokens=2), 2),                 # one dy vector only
    (dict(flags=8), 2),                    # unknown flag
    (dict(k=300), 2),
    (dict(fmt=9), 1),
    (dict(w_len=10), 3),
    (dict(j_start=5, j_end=3), 4),
    (dict(y=None), 5),
    (dict(k=16384), 10),                   # 512 units per row: beyond the kernel
    (dict(fmt="bf16", k=4096), 10),
])
def test_backward_input_rejected_on_host(lib, kw, status):
    a = _args(**kw)
    with pytest.raises(q.QmmError) as ei:
        q.qmm_matmul_backward_input(a)
    assert ei.value.status == status, q.qmm_last_error()
    assert q.qmm_backward_input_workspace_bytes(a) == 0


def test_backward_input_empty_work_needs_no_device(lib):
    # k == 0: nothing to write, no device touched
    assert q.qmm_matmul_backward_input(_args(k=0)) == 0


@pytest.mark.parametrize("kw,extra,status", [
    (dict(), dict(n_experts=0), 2),
    (dict(), dict(top_k=0), 2),
    (dict(flags=8), dict(), 2),
    (dict(path=q.PATH_MMA), dict(), 10),
    (dict(k=300), dict(), 2),
    (dict(fmt=9), dict(), 1),
    (dict(w_len=144 * 2 * 8), dict(n_experts=3), 3),   # two slices given, three claimed
    (dict(j_start=5, j_end=3), dict(), 4),
    (dict(n_tokens=300), dict(top_k=300), 2),           # more than 65535 GEMVs
    (dict(), dict(ids=None), 5),
    (dict(), dict(ids=16 * 500 + 2), 6),
    (dict(k=16384 * 4), dict(), 10),                    # beyond the one-token kernel
])
def test_experts_rejected_on_host(lib, kw, extra, status):
    a = _args(**kw)
    e = dict(ids=16 * 500, n_experts=4, top_k=2)
    e.update(extra)
    with pytest.raises(q.QmmError) as ei:
        q.qmm_matmul_experts(a, e["ids"], e["n_experts"], e["top_k"])
    assert ei.value.status == status, q.qmm_last_error()


def test_experts_empty_work_needs_no_device(lib):
    # an empty tile: nothing to write, no ids read, no device touched
    assert q.qmm_matmul_experts(_args(j_start=3, j_end=3), None, 4, 2) == 0
    # all slices given: w_len = n_experts * slice bytes is accepted
    assert q.qmm_matmul_experts(_args(w_len=144 * 2 * 8 * 3, j_start=2, j_end=2), 16, 3, 1) == 0


# ------------------------------------------------------- affine formats ----

def test_affine_sizes_and_policy(lib):
    assert q.qmm_weight_bytes("affine4", 128, 3) == 192
    assert q.qmm_weight_bytes("affine8", 128, 3) == 384
    assert q.qmm_weight_bytes("affine4", 100, 1) == 0
    a = _args(fmt="affine4", k=4096, n=14336, n_tokens=1)
    assert q.qmm_select_path(a) == q.PATH_GEMV and q.qmm_workspace_bytes(a) == 0
    a = _args(fmt="affine8", k=4096, n=14336, n_tokens=64)
    assert q.qmm_select_path(a) == q.PATH_MMA
    assert q.qmm_workspace_bytes(a) == 2 * 64 * 4096 * 2 + 256


@pytest.mark.parametrize("fn,kw,sb,status", [
    ("ex", dict(fmt="affine4", k=128), None, 1),          # needs its scales and biases
    ("aff", dict(fmt="q4_k"), (16 * 700, 16 * 800), 1),   # not an affine format
    ("aff", dict(fmt="affine4", k=100), (16 * 700, 16 * 800), 2),
    ("aff", dict(fmt="affine8", k=128), (None, 16 * 800), 5),
    ("aff", dict(fmt="affine8", k=128), (16 * 700 + 2, 16 * 800), 6),
    ("aff", dict(fmt="affine4", k=128, w_len=10), (16 * 700, 16 * 800), 3),
    ("experts", dict(fmt="affine4", k=128), None, 1),
    ("experts_aff", dict(fmt="q4_k"), (16 * 700, 16 * 800), 1),
    ("experts_aff", dict(fmt="affine4", k=128), (None, 16 * 800), 5),
    ("experts_aff", dict(fmt="affine4", k=128), (16 * 700 + 2, 16 * 800), 6),
    ("experts_aff", dict(fmt="affine8", k=128, w_len=128 * 8 * 3), (16 * 700, 16 * 800), 3),
    ("back", dict(fmt="affine4", k=128), None, 1),
])
def test_affine_rejected_on_host(lib, fn, kw, sb, status):
    a = _args(**kw)
    with pytest.raises(q.QmmError) as ei:
        if fn == "ex":
            q.qmm_matmul_ex(a)
        elif fn == "aff":
            q.qmm_matmul_affine(a, *sb)
        elif fn == "experts":
            q.qmm_matmul_experts(a, 16 * 500, 4, 2)
        elif fn == "experts_aff":
            q.qmm_matmul_experts_affine(a, 16 * 500, 4, 2, *sb)
        else:
            q.qmm_matmul_backward_input(a)
    assert ei.value.status == status, q.qmm_last_error()


def test_affine_dequant_rejected_on_host(lib):
    assert lib.qmm_dequant(7, 16, 128, 1, 16, None) == 1
    assert lib.qmm_dequant_affine(2, 16, 16, 16, 128, 1, 16, None) == 1
    assert lib.qmm_dequant_affine(7, 16, 16, 16, 100, 1, 16, None) == 2
    assert lib.qmm_dequant_affine(7, 16, None, 16, 128, 1, 16, None) == 5
    assert lib.qmm_dequant_affine(7, 24, 16, 16, 128, 1, 16, None) == 6
    assert lib.qmm_dequant_affine(7, 16, 17, 16, 128, 1, 16, None) == 6
    assert lib.qmm_dequant_affine(7, 16, 16, 16, 0, 1, 16, None) == 0   # nothing to do


def test_affine_empty_work_needs_no_device(lib):
    assert q.qmm_matmul_affine(_args(fmt="affine4", k=128, j_start=3, j_end=3), None, None) == 0


# ------------------------------------------------------------ gated pairs ----

@pytest.mark.parametrize("kw,wu,act,status", [
    (dict(), 16 * 900, 0, 1),                 # unknown activation
    (dict(), 16 * 900, 3, 1),
    (dict(fmt="affine4", k=128), 16 * 900, 1, 1),
    (dict(k=300), 16 * 900, 1, 2),
    (dict(w_len=10), 16 * 900, 2, 3),
    (dict(j_start=4, j_end=2), 16 * 900, 1, 4),
    (dict(), None, 1, 5),
    (dict(), 16 * 900 + 4, 2, 6),
    (dict(k=16384 * 4, path=q.PATH_GEMV), 16 * 900, 1, 10),
])
def test_glu_rejected_on_host(lib, kw, wu, act, status):
    with pytest.raises(q.QmmError) as ei:
        q.qmm_matmul_glu(_args(**kw), wu, act)
    assert ei.value.status == status, q.qmm_last_error()


def test_glu_workspace_and_empty_work(lib):
    assert q.qmm_glu_workspace_bytes(_args(k=4096, n=14336)) == 0          # fused GEMV
    a = _args(k=4096, n=1000, n_tokens=8)
    one = (8 * 1000 * 4 + 255) // 256 * 256
    assert q.qmm_glu_workspace_bytes(a) == one + 2 * 8 * 4096 * 2 + 256
    assert q.qmm_glu_workspace_bytes(_args(fmt="affine4", k=128)) == 0
    assert q.qmm_matmul_glu(_args(j_start=3, j_end=3), None, 1) == 0


def _fresh_python(code):
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    return subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True,
                          timeout=300)


def test_missing_library_fails_loudly():
    """No fallback: without libqmm.so the binding raises instead of computing
    anything another way."""
    r = _fresh_python("import quantized_weight_gguf_gb300 as q\n"
                      "try:\n"
                      "    q.load('no_such_dir/libqmm.so')\n"
                      "except RuntimeError as e:\n"
                      "    print('raised:', e)\n"
                      "else:\n"
                      "    raise SystemExit('loaded')\n")
    assert r.returncode == 0 and "raised: libqmm.so is not built" in r.stdout, r.stdout + r.stderr


def test_product_package_never_reaches_the_oracle(lib):
    """The package neither imports the oracle nor mentions it in code."""
    r = _fresh_python("import sys\n"
                      "import quantized_weight_gguf_gb300 as q\n"
                      "q.load()\n"
                      "print(sorted(m for m in sys.modules if m == 'oracle' or m.startswith('oracle.')))\n")
    assert r.returncode == 0 and r.stdout.strip() == "[]", r.stdout + r.stderr
    pkg = os.path.dirname(q.__file__)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", src, re.M), f
                assert "qmm_oracle" not in src and "liboracle" not in src, f
