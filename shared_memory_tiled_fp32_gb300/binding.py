"""ctypes binding of libtg_sgemm.so (the C ABI in include/tg_sgemm.h).

Argument marshalling only: every step of the product runs in the library's
CUDA kernels.  There is no fallback of any kind; if the library is missing the
calls raise.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtg_sgemm.so")

TG_OK = 0
STATUS = {
    0: "TG_OK",
    1: "TG_ERR_INVALID_VALUE",
    2: "TG_ERR_UNSUPPORTED_DEVICE",
    3: "TG_ERR_OUT_OF_MEMORY",
    4: "TG_ERR_CUDA",
    5: "TG_ERR_TIMEOUT",
    6: "TG_ERR_WORKSPACE_TOO_SMALL",
}
PATHS = {"auto": 0, "ffma": 1, "tf32x3": 2, "tiled": 3, "tf32bf16": 4}
PATH_NAMES = {v: k for k, v in PATHS.items()}

# Every symbol the headers in include/ declare.
EXPORTS = (
    "tg_sgemm",
    "tg_sgemm_ex",
    "tg_sgemm_general",
    "tg_sgemm_plan",
    "tg_sgemm_plan_general",
    "tg_sgemm_workspace_bytes",
    "tg_sgemm_host",
    "tg_sgemm_host_blocks",
    "tg_sgemm_host_device_bytes",
    "tg_sgemm_noalloc",
    "tg_sgemm_sync_status",
    "tg_sgemm_error_site",
    "tg_selftest_wait_timeout",
    "tg_status_string",
    "tg_sgemm_version",
    "tg_probe_tf32_mma",
    "tg_probe_f16_mma",
    "tg_probe_ffma",
    "tg_transpose",
    "tg_reduce_sum",
    "tg_reduce_plan",
)


class TgError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}" if what else STATUS.get(status, str(status)))


class Opts(ctypes.Structure):
    _fields_ = [
        ("path", ctypes.c_int),
        ("split_k", ctypes.c_int),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("main_begin", ctypes.c_void_p),
        ("main_end", ctypes.c_void_p),
    ]


class HostBlocksInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("row_blocks", "col_blocks", "first_block_rows", "block_rows",
                                             "block_cols", "split_row_blocks", "defer_copies_out")] + [
        ("model_ms", ctypes.c_double)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class PlanInfo(ctypes.Structure):
    _fields_ = [
        ("path", ctypes.c_int),
        ("split_k", ctypes.c_int),
        ("block_m", ctypes.c_int),
        ("block_n", ctypes.c_int),
        ("block_k", ctypes.c_int),
        ("stages", ctypes.c_int),
        ("tiles_m", ctypes.c_int),
        ("tiles_n", ctypes.c_int),
        ("units", ctypes.c_longlong),
        ("grid", ctypes.c_int),
        ("prepass", ctypes.c_int),
        ("launches", ctypes.c_int),
        ("workspace_bytes", ctypes.c_size_t),
        ("pair", ctypes.c_int),
        ("tail_units", ctypes.c_longlong),
        ("tail_lanes", ctypes.c_int),
        ("tail_kx", ctypes.c_int),
        ("fused_split", ctypes.c_int),
    ]

    def as_dict(self) -> dict:
        d = {name: getattr(self, name) for name, _ in self._fields_}
        d["path"] = PATH_NAMES.get(d["path"], d["path"])
        return d


_lib = None


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing; build it with `python -c 'import __graft_entry__ as g; g.build()'`"
            )
        L = ctypes.CDLL(LIB_PATH)
        i, p, vp = ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p
        gemm = [i, i, i, p, i, p, i, p, i, vp]
        L.tg_sgemm.argtypes = gemm
        L.tg_sgemm.restype = i
        L.tg_sgemm_ex.argtypes = gemm + [ctypes.POINTER(Opts)]
        L.tg_sgemm_ex.restype = i
        L.tg_sgemm_host.argtypes = gemm + [ctypes.POINTER(Opts)]
        L.tg_sgemm_host.restype = i
        L.tg_sgemm_noalloc.argtypes = gemm
        L.tg_sgemm_noalloc.restype = i
        ip = ctypes.POINTER(ctypes.c_int)
        L.tg_sgemm_host_blocks.argtypes = [i, i, i, i, i, ctypes.POINTER(HostBlocksInfo)]
        L.tg_sgemm_host_device_bytes.argtypes = [i, i, i, i, i, i, ctypes.POINTER(ctypes.c_size_t),
                                                 ctypes.POINTER(ctypes.c_size_t)]
        L.tg_sgemm_host_device_bytes.restype = i
        L.tg_sgemm_host_blocks.restype = i
        L.tg_sgemm_plan.argtypes = [i, i, i, p, i, p, i, p, i, i, i, i, ctypes.POINTER(PlanInfo)]
        L.tg_sgemm_plan.restype = i
        f = ctypes.c_float
        L.tg_sgemm_general.argtypes = [i, i, i, i, i, f, p, i, p, i, f, p, i, vp, ctypes.POINTER(Opts)]
        L.tg_sgemm_general.restype = i
        L.tg_sgemm_plan_general.argtypes = [i, i, i, i, i, p, i, p, i, p, i, i, i, i, ctypes.POINTER(PlanInfo)]
        L.tg_sgemm_plan_general.restype = i
        L.tg_sgemm_workspace_bytes.argtypes = [i, i, i, p, i, p, i, p, i, i, i]
        L.tg_sgemm_workspace_bytes.restype = ctypes.c_size_t
        L.tg_sgemm_sync_status.argtypes = [vp]
        L.tg_sgemm_sync_status.restype = i
        L.tg_sgemm_error_site.argtypes = [vp]
        L.tg_sgemm_error_site.restype = ctypes.c_uint
        L.tg_selftest_wait_timeout.argtypes = [ctypes.c_uint, vp]
        L.tg_selftest_wait_timeout.restype = i
        L.tg_status_string.argtypes = [i]
        L.tg_status_string.restype = ctypes.c_char_p
        L.tg_sgemm_version.argtypes = []
        L.tg_sgemm_version.restype = i
        L.tg_probe_tf32_mma.argtypes = [i, i, vp, ctypes.POINTER(ctypes.c_double)]
        L.tg_probe_tf32_mma.restype = i
        L.tg_probe_f16_mma.argtypes = [i, vp, ctypes.POINTER(ctypes.c_double)]
        L.tg_probe_f16_mma.restype = i
        L.tg_probe_ffma.argtypes = [i, p, vp, ctypes.POINTER(ctypes.c_double)]
        L.tg_probe_ffma.restype = i
        L.tg_transpose.argtypes = [i, i, i, p, i, p, i, vp]
        L.tg_transpose.restype = i
        L.tg_reduce_sum.argtypes = [i, ctypes.c_longlong, p, p, vp]
        L.tg_reduce_sum.restype = i
        L.tg_reduce_plan.argtypes = [i, ctypes.c_longlong, i, ctypes.POINTER(ctypes.c_int),
                                     ctypes.POINTER(ctypes.c_longlong), ctypes.POINTER(ctypes.c_size_t)]
        L.tg_reduce_plan.restype = i
        _lib = L
    return _lib


def _check(status: int, what: str):
    if status != TG_OK:
        raise TgError(status, what)


def _stream_handle(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _event_handle(ev):
    if ev is None:
        return None
    h = getattr(ev, "cuda_event", 0)
    if not h:
        raise ValueError("pass torch.cuda.Event objects that have been recorded once (created)")
    return h


def _rowmajor_ld(t, name):
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D")
    if t.numel() == 0:  # nothing is read: any strides will do
        return max(t.shape[1], 1)
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must have unit stride along its last dimension")
    return max(t.stride(0) if t.shape[0] > 1 else t.shape[1], t.shape[1], 1)


def make_opts(path="auto", split_k=0, workspace=None, main_begin=None, main_end=None) -> Opts:
    o = Opts()
    o.path = PATHS[path] if isinstance(path, str) else int(path)
    o.split_k = int(split_k)
    if workspace is not None:
        o.workspace = workspace.data_ptr()
        o.workspace_bytes = workspace.numel() * workspace.element_size()
    o.main_begin = _event_handle(main_begin)
    o.main_end = _event_handle(main_end)
    return o


def matmul(A, B, out=None, *, path="auto", split_k=0, workspace=None, main_begin=None,
           main_end=None, stream=None):
    """C = A @ B for float32 CUDA tensors (row-major, any row stride).

    Enqueues on ``stream`` (default: the current stream) and returns ``out``.
    """
    import torch

    for name, t in (("A", A), ("B", B)):
        if t.dtype != torch.float32 or not t.is_cuda:
            raise TypeError(f"{name} must be a float32 CUDA tensor")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError(f"inner dimensions differ: {tuple(A.shape)} x {tuple(B.shape)}")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    if out.dtype != torch.float32 or not out.is_cuda or tuple(out.shape) != (M, N):
        raise ValueError("out must be an (M, N) float32 CUDA tensor")
    lda, ldb, ldc = _rowmajor_ld(A, "A"), _rowmajor_ld(B, "B"), _rowmajor_ld(out, "out")
    # default options go as NULL (the library's defaults); the call is made on
    # A's device, switching to it only when it is not already current (the
    # switch costs more host time than the rest of this function)
    default = (path == "auto" and not split_k and workspace is None and main_begin is None
               and main_end is None)
    opts = None if default else ctypes.byref(make_opts(path, split_k, workspace, main_begin, main_end))
    dev = A.device.index
    L = _lib if _lib is not None else lib()
    if dev == torch.cuda.current_device():
        handle = (stream if stream is not None else torch.cuda.current_stream()).cuda_stream
        st = L.tg_sgemm_ex(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, out.data_ptr(), ldc, handle, opts)
    else:
        with torch.cuda.device(dev):
            handle = (stream if stream is not None else torch.cuda.current_stream()).cuda_stream
            st = L.tg_sgemm_ex(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, out.data_ptr(), ldc, handle, opts)
    _check(st, "tg_sgemm_ex")
    return out


def matmul_general(A, B, C=None, *, trans_a=False, trans_b=False, alpha=1.0, beta=0.0, path="auto",
                   split_k=0, workspace=None, stream=None, main_begin=None, main_end=None):
    """C = alpha * op(A) @ op(B) + beta * C for float32 CUDA tensors, where
    op(X) is X.T when the trans_ flag is set (A and B are the stored
    matrices).  C is required when beta != 0; it is returned."""
    import torch

    for name, t in (("A", A), ("B", B)):
        if t.dtype != torch.float32 or not t.is_cuda:
            raise TypeError(f"{name} must be a float32 CUDA tensor")
    M, K = (A.shape[1], A.shape[0]) if trans_a else tuple(A.shape)
    Kb, N = (B.shape[1], B.shape[0]) if trans_b else tuple(B.shape)
    if Kb != K:
        raise ValueError("inner dimensions differ")
    if C is None:
        if beta != 0.0:
            raise ValueError("C is required when beta != 0")
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    if C.dtype != torch.float32 or not C.is_cuda or tuple(C.shape) != (M, N):
        raise ValueError("C must be an (M, N) float32 CUDA tensor")
    lda, ldb, ldc = _rowmajor_ld(A, "A"), _rowmajor_ld(B, "B"), _rowmajor_ld(C, "C")
    o = make_opts(path, split_k, workspace, main_begin, main_end)
    with torch.cuda.device(A.device):
        st = lib().tg_sgemm_general(int(trans_a), int(trans_b), M, N, K, float(alpha), A.data_ptr(), lda,
                                    B.data_ptr(), ldb, float(beta), C.data_ptr(), ldc, _stream_handle(stream),
                                    ctypes.byref(o))
    _check(st, "tg_sgemm_general")
    return C


TRANSPOSE_VARIANTS = {"direct": 0, "tile32": 1, "padded": 2, "swizzled": 3}


def transpose(X, out=None, *, variant="padded", stream=None):
    """X^T of a float32 CUDA matrix through tg_transpose (include/tg_transpose.h)."""
    import torch

    if X.dtype != torch.float32 or not X.is_cuda:
        raise TypeError("X must be a float32 CUDA tensor")
    rows, cols = X.shape
    if out is None:
        out = torch.empty((cols, rows), dtype=torch.float32, device=X.device)
    if tuple(out.shape) != (cols, rows):
        raise ValueError("out must be (cols, rows)")
    v = TRANSPOSE_VARIANTS[variant] if isinstance(variant, str) else int(variant)
    with torch.cuda.device(X.device):
        st = lib().tg_transpose(v, rows, cols, X.data_ptr(), _rowmajor_ld(X, "X"), out.data_ptr(),
                                _rowmajor_ld(out, "out"), _stream_handle(stream))
    _check(st, "tg_transpose")
    return out


REDUCE_VARIANTS = {"interleaved": 0, "sequential": 1, "shuffle": 2, "atomic": 3, "fast": 4}


def reduce_sum(x, out=None, *, variant="fast", stream=None):
    """Sum of a float32 CUDA tensor (flattened, contiguous) through
    tg_reduce_sum (include/tg_reduce.h); returns a 1-element CUDA tensor."""
    import torch

    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise TypeError("x must be a contiguous float32 CUDA tensor")
    if out is None:
        out = torch.empty(1, dtype=torch.float32, device=x.device)
    v = REDUCE_VARIANTS[variant] if isinstance(variant, str) else int(variant)
    with torch.cuda.device(x.device):
        st = lib().tg_reduce_sum(v, x.numel(), x.data_ptr() if x.numel() else None, out.data_ptr(),
                                 _stream_handle(stream))
    _check(st, "tg_reduce_sum")
    return out


def reduce_plan(variant, n, num_sms=0) -> dict:
    """Launches of one tg_reduce_sum call (host arithmetic)."""
    passes = ctypes.c_int()
    counts = (ctypes.c_longlong * 8)()
    ws = ctypes.c_size_t()
    v = REDUCE_VARIANTS[variant] if isinstance(variant, str) else int(variant)
    _check(lib().tg_reduce_plan(v, n, num_sms, ctypes.byref(passes), counts, ctypes.byref(ws)), "tg_reduce_plan")
    return {"passes": passes.value, "counts": [counts[i] for i in range(passes.value)],
            "workspace_bytes": ws.value}


def matmul_noalloc(A, B, out, *, stream=None):
    """C = A @ B through tg_sgemm_noalloc: 3xTF32 with the library's fixed
    device scratch array instead of any allocation (``out`` must be given)."""
    import torch

    M, K = A.shape
    _, N = B.shape
    lda, ldb, ldc = _rowmajor_ld(A, "A"), _rowmajor_ld(B, "B"), _rowmajor_ld(out, "out")
    with torch.cuda.device(A.device):
        st = lib().tg_sgemm_noalloc(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, out.data_ptr(), ldc,
                                    _stream_handle(stream))
    _check(st, "tg_sgemm_noalloc")
    return out


def sgemm_host(A, B, out, *, path="auto", split_k=0, stream=None):
    """C = A @ B for float32 CPU tensors (pinned memory for async copies).

    Copies in, computes on the current device, copies out and synchronises.
    """
    import torch

    M, K = A.shape
    _, N = B.shape
    lda, ldb, ldc = _rowmajor_ld(A, "A"), _rowmajor_ld(B, "B"), _rowmajor_ld(out, "out")
    o = make_opts(path, split_k)
    st = lib().tg_sgemm_host(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, out.data_ptr(), ldc,
                             _stream_handle(stream), ctypes.byref(o))
    _check(st, "tg_sgemm_host")
    return out


def host_blocks(M, N, K, *, path="auto", num_sms=0) -> dict:
    """The output blocks sgemm_host pipelines (host arithmetic): row blocks
    [0, split_row_blocks) are cut into col_blocks column blocks, the later ones
    are full width; see include/tg_sgemm.h."""
    info = HostBlocksInfo()
    st = lib().tg_sgemm_host_blocks(M, N, K, PATHS[path] if isinstance(path, str) else int(path), num_sms,
                                    ctypes.byref(info))
    _check(st, "tg_sgemm_host_blocks")
    return info.as_dict()


def host_device_bytes(M, N, K, *, path="auto", split_k=0, num_sms=0) -> dict:
    """Device memory one sgemm_host call allocates (host arithmetic): the total
    and the largest single-product workspace within it."""
    total, ws = ctypes.c_size_t(), ctypes.c_size_t()
    st = lib().tg_sgemm_host_device_bytes(M, N, K, PATHS[path] if isinstance(path, str) else int(path), split_k,
                                          num_sms, ctypes.byref(total), ctypes.byref(ws))
    _check(st, "tg_sgemm_host_device_bytes")
    return {"total": total.value, "product_workspace": ws.value}


def plan(M, N, K, lda=None, ldb=None, ldc=None, *, A=0, B=0, C=0, path="auto", split_k=0,
         num_sms=0) -> dict:
    """What one call would launch (host arithmetic; num_sms=0 queries the device)."""
    info = PlanInfo()
    lda = max(K, 1) if lda is None else lda
    ldb = max(N, 1) if ldb is None else ldb
    ldc = max(N, 1) if ldc is None else ldc
    st = lib().tg_sgemm_plan(M, N, K, A or None, lda, B or None, ldb, C or None, ldc,
                             PATHS[path] if isinstance(path, str) else int(path), split_k, num_sms,
                             ctypes.byref(info))
    _check(st, "tg_sgemm_plan")
    return info.as_dict()


def plan_general(trans_a, trans_b, M, N, K, lda, ldb, ldc, *, A=0, B=0, C=0, path="auto", split_k=0,
                 num_sms=0) -> dict:
    """What tg_sgemm_general would launch (stored-matrix leading dimensions)."""
    info = PlanInfo()
    st = lib().tg_sgemm_plan_general(int(trans_a), int(trans_b), M, N, K, A or None, lda, B or None, ldb,
                                     C or None, ldc, PATHS[path] if isinstance(path, str) else int(path),
                                     split_k, num_sms, ctypes.byref(info))
    _check(st, "tg_sgemm_plan_general")
    return info.as_dict()


def sync_status(stream=None) -> int:
    """Synchronise and return (then clear) the device error status code."""
    return int(lib().tg_sgemm_sync_status(_stream_handle(stream)))


def error_site(stream=None) -> int:
    return int(lib().tg_sgemm_error_site(_stream_handle(stream)))


def selftest_wait_timeout(timeout_us: int, stream=None) -> int:
    return int(lib().tg_selftest_wait_timeout(timeout_us, _stream_handle(stream)))


def status_string(status: int) -> str:
    return lib().tg_status_string(status).decode()


def _time_probe(launch):
    import torch

    stream = torch.cuda.current_stream()
    launch(stream)  # warm-up
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    flop = launch(stream)
    e1.record(stream)
    e1.synchronize()
    return flop / (e0.elapsed_time(e1) * 1e-3) / 1e12


def probe_tf32_mma_tflops(iters=100000, use_collector=True) -> float:
    """Tensor TFLOP/s of the 3xTF32 main loop's MMA issue pattern, operands
    resident in shared memory (see include/tg_probes.h)."""
    def launch(stream):
        f = ctypes.c_double()
        _check(lib().tg_probe_tf32_mma(iters, int(use_collector), _stream_handle(stream), ctypes.byref(f)),
               "tg_probe_tf32_mma")
        return f.value
    return _time_probe(launch)


def probe_f16_mma_tflops(iters=100000) -> float:
    """Tensor TFLOP/s of the same issue pattern with kind::f16 MMAs (K=16),
    for comparison only: no GEMM path uses fp16 operands."""
    def launch(stream):
        f = ctypes.c_double()
        _check(lib().tg_probe_f16_mma(iters, _stream_handle(stream), ctypes.byref(f)), "tg_probe_f16_mma")
        return f.value
    return _time_probe(launch)


def probe_ffma_tflops(iters=100000) -> float:
    """fp32 FMA TFLOP/s with 16 independent chains per thread."""
    import torch

    sink = torch.zeros(1, device="cuda")

    def launch(stream):
        f = ctypes.c_double()
        _check(lib().tg_probe_ffma(iters, sink.data_ptr(), _stream_handle(stream), ctypes.byref(f)),
               "tg_probe_ffma")
        return f.value
    return _time_probe(launch)
