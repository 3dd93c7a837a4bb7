"""Python binding of libqmm (include/qmm.h): fused dequantize-and-multiply
``y = x @ W`` over GGUF/ggml-packed weights on one GB300 GPU.

Argument marshalling only: every step of the product runs in the CUDA
kernels of ``libqmm.so``. PyTorch supplies device memory and streams. The
functions carry the C names (``qmm_matmul``, ``qmm_matmul_ex``,
``qmm_dequant`` ...) and take plain integers / device pointers or torch
tensors; ``matmul``, ``dequant``, ``matmul_backward_input``,
``matmul_experts``, ``matmul_affine``, ``dequant_affine`` and ``matmul_glu``
are tensor-level conveniences over them.
If ``libqmm.so`` has not been built, every call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqmm.so")

FORMATS = {"bf16": 0, "f16": 1, "q4_0": 2, "q4_k": 3, "q6_k": 4, "q8_0": 5, "q5_0": 6,
           "affine4": 7, "affine8": 8}
PATH_AUTO, PATH_GEMV, PATH_MMA = 0, 1, 2
FLAG_OVERLAP_PREV = 1
FLAG_X_READY = 2
FLAG_SPLIT_W = 4
STATUS = {0: "QMM_OK", 1: "QMM_ERR_FORMAT", 2: "QMM_ERR_SHAPE", 3: "QMM_ERR_SIZE",
          4: "QMM_ERR_RANGE", 5: "QMM_ERR_NULL", 6: "QMM_ERR_ALIGN", 7: "QMM_ERR_CUDA",
          8: "QMM_ERR_DEVICE_TIMEOUT", 9: "QMM_ERR_WORKSPACE", 10: "QMM_ERR_UNSUPPORTED",
          11: "QMM_ERR_BAD_ID"}
EXPORTS = ("qmm_weight_bytes", "qmm_matmul", "qmm_set_stream", "qmm_matmul_ex",
           "qmm_workspace_bytes", "qmm_select_path", "qmm_matmul_host", "qmm_dequant",
           "qmm_device_status", "qmm_last_error", "qmm_version", "qmm_matmul_noalloc",
           "qmm_matmul_backward_input", "qmm_backward_input_workspace_bytes",
           "qmm_matmul_experts", "qmm_matmul_affine", "qmm_dequant_affine", "qmm_matmul_glu",
           "qmm_glu_workspace_bytes", "qmm_check_bounded_wait", "qmm_matmul_experts_affine",
           "qmm_experts_workspace_bytes")


class QmmError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class qmm_args(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int), ("w", ctypes.c_void_p), ("w_len", ctypes.c_size_t),
                ("x", ctypes.c_void_p), ("y", ctypes.c_void_p), ("k", ctypes.c_int64),
                ("n", ctypes.c_int64), ("n_tokens", ctypes.c_int64), ("j_start", ctypes.c_int64),
                ("j_end", ctypes.c_int64), ("accumulate", ctypes.c_int), ("path", ctypes.c_int),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("stream", ctypes.c_void_p), ("flags", ctypes.c_int)]


_lib = None


def load(path: str = LIB_PATH):
    """Load libqmm.so (raises if it is missing) and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libqmm.so is not built ({path}); run __graft_entry__.build() "
                           "or python -m quantized_weight_gguf_gb300.build_lib")
    lib = ctypes.CDLL(path)
    i64, vp, sz, i = ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    pa = ctypes.POINTER(qmm_args)
    sig = {
        "qmm_weight_bytes": (sz, [i, i64, i64]),
        "qmm_matmul": (i, [i, vp, vp, i64, i64, i64, vp]),
        "qmm_set_stream": (None, [vp]),
        "qmm_matmul_ex": (i, [pa]),
        "qmm_workspace_bytes": (sz, [pa]),
        "qmm_select_path": (i, [pa]),
        "qmm_matmul_host": (i, [pa, vp, vp, vp]),
        "qmm_dequant": (i, [i, vp, i64, i64, vp, vp]),
        "qmm_device_status": (i, [vp]),
        "qmm_last_error": (ctypes.c_char_p, []),
        "qmm_version": (i, []),
        "qmm_matmul_noalloc": (i, [pa]),
        "qmm_matmul_backward_input": (i, [pa]),
        "qmm_backward_input_workspace_bytes": (sz, [pa]),
        "qmm_matmul_experts": (i, [pa, vp, i64, i64]),
        "qmm_experts_workspace_bytes": (sz, [pa, i64, i64]),
        "qmm_matmul_affine": (i, [pa, vp, vp]),
        "qmm_matmul_glu": (i, [pa, vp, i]),
        "qmm_glu_workspace_bytes": (sz, [pa]),
        "qmm_check_bounded_wait": (i, [vp]),
        "qmm_matmul_experts_affine": (i, [pa, vp, i64, i64, vp, vp]),
        "qmm_dequant_affine": (i, [i, vp, vp, vp, i64, i64, vp, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(v):
    if v is None:
        return None
    if isinstance(v, int):
        return v
    if hasattr(v, "data_ptr"):
        return v.data_ptr()
    if hasattr(v, "ctypes"):
        return v.ctypes.data
    raise TypeError(f"cannot take a pointer of {type(v)}")


def _fmt(f):
    return FORMATS[f] if isinstance(f, str) else int(f)


def _check(status: int):
    if status != 0:
        raise QmmError(status, load().qmm_last_error().decode())
    return status


def _keep_until_done(buf, stream):
    """A per-call scratch tensor allocated on torch's current stream but used
    by kernels on another stream: tell the caching allocator, so the memory
    is not handed out again before that stream's work is done."""
    if buf is None or stream is None or stream == 0:
        return
    import torch
    s = stream if isinstance(stream, torch.cuda.Stream) else torch.cuda.ExternalStream(
        int(getattr(stream, "cuda_stream", stream)), device=buf.device)
    if s.cuda_stream != torch.cuda.current_stream(buf.device).cuda_stream:
        buf.record_stream(s)


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return int(getattr(stream, "cuda_stream", stream))


# --------------------------------------------------------- C-named calls ----

def qmm_weight_bytes(fmt, k: int, n: int) -> int:
    return load().qmm_weight_bytes(_fmt(fmt), k, n)


def qmm_set_stream(stream) -> None:
    load().qmm_set_stream(_stream(stream))


def qmm_matmul(fmt, w, x, k: int, n: int, n_tokens: int, y) -> int:
    return _check(load().qmm_matmul(_fmt(fmt), _ptr(w), _ptr(x), k, n, n_tokens, _ptr(y)))


def make_args(fmt, w, x, y, k, n, n_tokens, *, w_len=0, j_start=0, j_end=0, accumulate=False,
              path=PATH_AUTO, workspace=None, workspace_bytes=0, stream=None, flags=0) -> qmm_args:
    return qmm_args(_fmt(fmt), _ptr(w), w_len, _ptr(x), _ptr(y), k, n, n_tokens, j_start, j_end,
                    int(bool(accumulate)), int(path), _ptr(workspace), workspace_bytes,
                    _stream(stream) if stream != 0 else 0, int(flags))


def qmm_matmul_ex(args: qmm_args) -> int:
    return _check(load().qmm_matmul_ex(ctypes.byref(args)))


def qmm_matmul_noalloc(args: qmm_args) -> int:
    return _check(load().qmm_matmul_noalloc(ctypes.byref(args)))


def qmm_matmul_backward_input(args: qmm_args) -> int:
    return _check(load().qmm_matmul_backward_input(ctypes.byref(args)))


ACT_SWIGLU, ACT_GEGLU = 1, 2
ACTS = {"swiglu": ACT_SWIGLU, "geglu": ACT_GEGLU}


def qmm_matmul_glu(args: qmm_args, w_up, act) -> int:
    act = ACTS[act] if isinstance(act, str) else int(act)
    return _check(load().qmm_matmul_glu(ctypes.byref(args), _ptr(w_up), act))


def qmm_glu_workspace_bytes(args: qmm_args) -> int:
    return load().qmm_glu_workspace_bytes(ctypes.byref(args))


def qmm_matmul_affine(args: qmm_args, scales, biases) -> int:
    return _check(load().qmm_matmul_affine(ctypes.byref(args), _ptr(scales), _ptr(biases)))


def qmm_dequant_affine(fmt, w, scales, biases, k: int, n: int, out, stream=None) -> int:
    return _check(load().qmm_dequant_affine(_fmt(fmt), _ptr(w), _ptr(scales), _ptr(biases), k, n,
                                            _ptr(out), _stream(stream)))


def qmm_matmul_experts_affine(args: qmm_args, ids, n_experts: int, top_k: int, scales,
                              biases) -> int:
    return _check(load().qmm_matmul_experts_affine(ctypes.byref(args), _ptr(ids), n_experts, top_k,
                                                   _ptr(scales), _ptr(biases)))


def qmm_matmul_experts(args: qmm_args, ids, n_experts: int, top_k: int) -> int:
    return _check(load().qmm_matmul_experts(ctypes.byref(args), _ptr(ids), n_experts, top_k))


def qmm_experts_workspace_bytes(args: qmm_args, n_experts: int, top_k: int) -> int:
    return load().qmm_experts_workspace_bytes(ctypes.byref(args), n_experts, top_k)


def qmm_backward_input_workspace_bytes(args: qmm_args) -> int:
    return load().qmm_backward_input_workspace_bytes(ctypes.byref(args))


def qmm_workspace_bytes(args: qmm_args) -> int:
    return load().qmm_workspace_bytes(ctypes.byref(args))


def qmm_select_path(args: qmm_args) -> int:
    return load().qmm_select_path(ctypes.byref(args))


def qmm_matmul_host(args: qmm_args, dev_w, dev_x, dev_y) -> int:
    return _check(load().qmm_matmul_host(ctypes.byref(args), _ptr(dev_w), _ptr(dev_x), _ptr(dev_y)))


def qmm_dequant(fmt, w, k: int, n: int, out, stream=None) -> int:
    return _check(load().qmm_dequant(_fmt(fmt), _ptr(w), k, n, _ptr(out), _stream(stream)))


def qmm_check_bounded_wait(stream=None) -> int:
    return _check(load().qmm_check_bounded_wait(_stream(stream)))


def qmm_device_status(stream=None) -> int:
    return _check(load().qmm_device_status(_stream(stream)))


def qmm_last_error() -> str:
    return load().qmm_last_error().decode()


def qmm_version() -> int:
    return load().qmm_version()


# ------------------------------------------------------ tensor helpers ----

def matmul(fmt, w, x, k: int, n: int, *, y=None, j_start=0, j_end=0, accumulate=False,
           path=PATH_AUTO, stream=None, flags=0):
    """y = x @ W for torch CUDA tensors: w uint8 packed bytes, x float32 [N, k].
    Returns y float32 [N, n] (the given y when passed). Scratch for the
    tensor-core path is a torch allocation on x's device."""
    import torch
    if x.dim() == 1:
        x = x.unsqueeze(0)
    nt = x.shape[0]
    if y is None:
        y = torch.empty((nt, n), dtype=torch.float32, device=x.device)
    a = make_args(fmt, w, x, y, k, n, nt, w_len=w.numel() * w.element_size(), j_start=j_start,
                  j_end=j_end, accumulate=accumulate, path=path, stream=stream, flags=flags)
    need = qmm_workspace_bytes(a)
    ws = None
    if need:
        ws = torch.empty(need, dtype=torch.uint8, device=x.device)
        a.workspace = ws.data_ptr()
        a.workspace_bytes = need
    qmm_matmul_ex(a)
    _keep_until_done(ws, stream)
    return y


def matmul_backward_input(fmt, w, dy, k: int, n: int, *, dx=None, j_start=0, j_end=0,
                          accumulate=False, stream=None, flags=0):
    """dx = W^T dy over the rows [j_start, j_end) for torch CUDA tensors: w
    uint8 packed bytes, dy float32 [n]. Returns dx float32 [k] (the given dx
    when passed). Scratch is the library's own buffer."""
    import torch
    if dx is None:
        dx = torch.empty(k, dtype=torch.float32, device=dy.device)
    a = make_args(fmt, w, dy, dx, k, n, 1, w_len=w.numel() * w.element_size(), j_start=j_start,
                  j_end=j_end, accumulate=accumulate, stream=stream, flags=flags)
    qmm_matmul_backward_input(a)
    return dx


def matmul_experts(fmt, w, x, ids, k: int, n: int, n_experts: int, *, y=None, j_start=0,
                   j_end=0, accumulate=False, path=PATH_AUTO, stream=None, flags=0, scales=None,
                   biases=None):
    """Expert-indexed product for torch CUDA tensors: w uint8 (n_experts
    stacked slices of n rows), x float32 [n_pos, k], ids int32 [n_pos, top_k]
    on the device. Returns y float32 [n_pos * top_k, n] (the given y when
    passed). Scratch of the grouped form is a torch allocation on x's device."""
    import torch
    if x.dim() == 1:
        x = x.unsqueeze(0)
    if ids.dim() == 1:
        ids = ids.unsqueeze(0)
    n_pos, top_k = ids.shape
    if y is None:
        y = torch.empty((n_pos * top_k, n), dtype=torch.float32, device=x.device)
    a = make_args(fmt, w, x, y, k, n, n_pos, w_len=w.numel() * w.element_size(), j_start=j_start,
                  j_end=j_end, accumulate=accumulate, path=path, stream=stream, flags=flags)
    if scales is not None or biases is not None:
        qmm_matmul_experts_affine(a, ids, n_experts, top_k, scales, biases)
        return y
    need = qmm_experts_workspace_bytes(a, n_experts, top_k)
    ws = None
    if need:
        ws = torch.empty(need, dtype=torch.uint8, device=x.device)
        a.workspace, a.workspace_bytes = ws.data_ptr(), need
    qmm_matmul_experts(a, ids, n_experts, top_k)
    _keep_until_done(ws, stream)
    return y


def dequant(fmt, w, k: int, n: int, stream=None):
    """fp32 [n, k] weights from packed bytes (torch CUDA uint8 tensor)."""
    import torch
    out = torch.empty((n, k), dtype=torch.float32, device=w.device)
    qmm_dequant(fmt, w, k, n, out, stream)
    return out


def matmul_affine(fmt, w, scales, biases, x, k: int, n: int, *, y=None, j_start=0, j_end=0,
                  accumulate=False, path=PATH_AUTO, workspace=None, workspace_bytes=0,
                  stream=None, flags=0):
    """y = x @ W for an affine matrix ("affine4" / "affine8") on torch CUDA
    tensors: w uint8 code words, scales / biases bf16 or int16 [n, k/64],
    x float32 [N, k]. Returns y float32 [N, n] (the given y when passed)."""
    import torch
    if x.dim() == 1:
        x = x.unsqueeze(0)
    nt = x.shape[0]
    if y is None:
        y = torch.empty((nt, n), dtype=torch.float32, device=x.device)
    a = make_args(fmt, w, x, y, k, n, nt, w_len=w.numel() * w.element_size(), j_start=j_start,
                  j_end=j_end, accumulate=accumulate, path=path, stream=stream, flags=flags)
    own = None
    if workspace is None:
        need = qmm_workspace_bytes(a)
        if need:
            own = workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
            workspace_bytes = need
    if workspace is not None:
        a.workspace, a.workspace_bytes = _ptr(workspace), workspace_bytes
    qmm_matmul_affine(a, scales, biases)
    _keep_until_done(own, stream)
    return y


def dequant_affine(fmt, w, scales, biases, k: int, n: int, stream=None):
    """fp32 [n, k] weights of an affine matrix (torch CUDA tensors)."""
    import torch
    out = torch.empty((n, k), dtype=torch.float32, device=w.device)
    qmm_dequant_affine(fmt, w, scales, biases, k, n, out, stream)
    return out


def matmul_glu(act, fmt, w_gate, w_up, x, k: int, n: int, *, y=None, j_start=0, j_end=0,
               accumulate=False, path=PATH_AUTO, stream=None, flags=0):
    """y = act(x Wg) * (x Wu) ("swiglu" / "geglu") for torch CUDA tensors; the
    scratch of the several-token form is a torch allocation on x's device."""
    import torch
    if x.dim() == 1:
        x = x.unsqueeze(0)
    nt = x.shape[0]
    if y is None:
        y = torch.empty((nt, n), dtype=torch.float32, device=x.device)
    a = make_args(fmt, w_gate, x, y, k, n, nt, w_len=w_gate.numel() * w_gate.element_size(),
                  j_start=j_start, j_end=j_end, accumulate=accumulate, path=path, stream=stream,
                  flags=flags)
    need = qmm_glu_workspace_bytes(a)
    ws = None
    if need:
        ws = torch.empty(need, dtype=torch.uint8, device=x.device)
        a.workspace, a.workspace_bytes = ws.data_ptr(), need
    qmm_matmul_glu(a, w_up, act)
    _keep_until_done(ws, stream)
    return y
