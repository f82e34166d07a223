"""Python binding of the C ABI in include/densegemm.h (argument marshalling only).

Every function named like the C entry point takes the same arguments, with
pointers given as ints or as tensors (their ``data_ptr()``), and returns the
C status code. All arithmetic runs in libdensegemm.so; importing this module
fails loudly if the library has not been built (there is no other code path).

``Gemm`` wraps a handle for callers holding torch tensors: it derives sizes and
leading dimensions from the tensors and raises ``GemmError`` on a bad status.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

_LIB_PATH = _build.LIB_PATH
if not os.path.exists(_LIB_PATH):
    raise ImportError(
        f"libdensegemm.so is not built ({_LIB_PATH}); run "
        "`python -m dense_gemm_cluster_gb300.build` or __graft_entry__.build()")
_lib = ctypes.CDLL(_LIB_PATH)

GEMM_OK = 0
GEMM_ERR_INVALID_ARG = 1
GEMM_ERR_UNSUPPORTED = 2
GEMM_ERR_ALIGNMENT = 3
GEMM_ERR_CUDA = 4
GEMM_ERR_DEVICE_TIMEOUT = 5
GEMM_ERR_NOT_SM103 = 6

GEMM_ROW_MAJOR = 0
GEMM_COL_MAJOR = 1
GEMM_OUT_BF16 = 0
GEMM_OUT_F32 = 1
GEMM_MODE_UNICAST = 0
GEMM_MODE_MCAST = 1
GEMM_DEBUG_EXTRA_TX = 1


class gemm_options_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "mode", "mcast_a", "mcast_b", "cluster_m", "cluster_n", "cta_group", "layout_a", "layout_b",
        "layout_c", "out_type", "block_n", "block_k", "stages", "max_clusters", "group_m", "schedule")] + [
        ("wait_timeout_ns", ctypes.c_uint64), ("debug_flags", ctypes.c_int), ("host_parts", ctypes.c_int),
        ("clock_probe", ctypes.c_int)]


class gemm_plan_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "block_m", "block_n", "block_k", "stages", "smem_bytes", "cluster_m", "cluster_n", "cta_group",
        "group_a", "group_b", "transposed")] + [
        ("tiles", ctypes.c_int64), ("clusters", ctypes.c_int64), ("l2_to_sm_operand_bytes", ctypes.c_int64),
        ("stream_k_tiles", ctypes.c_int64), ("l2_hint_a", ctypes.c_int), ("l2_hint_b", ctypes.c_int),
        ("k_rotate", ctypes.c_int), ("k_serpentine", ctypes.c_int), ("prefetch_kb", ctypes.c_int)]


_i64, _i32, _f32, _vp = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_void_p
_OPT_P = ctypes.POINTER(gemm_options_t)

_lib.gemm_options_default.argtypes = [_OPT_P]
_lib.gemm_options_default.restype = None
_lib.gemm_create.argtypes = [ctypes.POINTER(_vp), _OPT_P, _i32]
_lib.gemm_create.restype = _i32
_lib.gemm_run.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _f32, _f32, _vp]
_lib.gemm_run.restype = _i32
_lib.gemm_run_strided_batched.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _i64,
                                          _vp, _i64, _i64, _i64, _f32, _f32, _vp]
_lib.gemm_run_strided_batched.restype = _i32
_lib.gemm_run_host.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _f32, _f32, _vp]
_lib.gemm_run_host.restype = _i32
_lib.gemm_run_strided_batched_host.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _i64, _vp, _i64,
                                               _i64, _i64, _f32, _f32, _vp]
_lib.gemm_run_strided_batched_host.restype = _i32
_lib.gemm_query_status.argtypes = [_vp, _vp]
_lib.gemm_query_status.restype = _i32
_lib.gemm_read_clock.argtypes = [_vp, _vp, ctypes.POINTER(ctypes.c_uint64)]
_lib.gemm_read_clock.restype = _i32
_lib.gemm_plan.argtypes = [_OPT_P, _i64, _i64, _i64, _i64, _i32, ctypes.POINTER(gemm_plan_t)]
_lib.gemm_plan.restype = _i32
_lib.gemm_status_string.argtypes = [_i32]
_lib.gemm_status_string.restype = ctypes.c_char_p
_lib.gemm_last_error.argtypes = [_vp]
_lib.gemm_last_error.restype = ctypes.c_char_p
_lib.gemm_launch_count.argtypes = [_vp]
_lib.gemm_launch_count.restype = _i64
_lib.gemm_destroy.argtypes = [_vp]
_lib.gemm_destroy.restype = _i32
_lib.gemm_run_noalloc.argtypes = [_OPT_P, _i32, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _f32, _f32, _vp,
                                  ctypes.POINTER(ctypes.c_uint32)]
_lib.gemm_run_noalloc.restype = _i32


class gemm_work_item_t(ctypes.Structure):
    _fields_ = [("tile", ctypes.c_int64), ("kb0", ctypes.c_int32), ("kb1", ctypes.c_int32),
                ("kind", ctypes.c_int32), ("contrib_first", ctypes.c_int32), ("contrib_count", ctypes.c_int32),
                ("last", ctypes.c_int32)]


_lib.gemm_schedule_work.argtypes = [_i64, _i64, _i32, _i64, _i64, ctypes.POINTER(gemm_work_item_t), _i64]
_lib.gemm_schedule_work.restype = _i64

WORK_WHOLE, WORK_PARTIAL, WORK_FINISHER = 0, 1, 2


def gemm_schedule_work(tiles, dp_tiles, num_kb, clusters, cluster):
    """The work units one cluster of a persistent launch walks (host-only), as a list of
    (tile, kb0, kb1, kind, contrib_first, contrib_count, last) tuples."""
    n = _lib.gemm_schedule_work(tiles, dp_tiles, num_kb, clusters, cluster, None, 0)
    if n < 0:
        raise ValueError("gemm_schedule_work: invalid arguments")
    buf = (gemm_work_item_t * max(1, n))()
    _lib.gemm_schedule_work(tiles, dp_tiles, num_kb, clusters, cluster, buf, n)
    return [(it.tile, it.kb0, it.kb1, it.kind, it.contrib_first, it.contrib_count, it.last) for it in buf[:n]]


def library_path() -> str:
    return _LIB_PATH


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):           # numpy array (host pointer)
        return x.ctypes.data
    raise TypeError(f"cannot take a pointer of {type(x).__name__}")


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream               # torch.cuda.Stream


# ---------------------------------------------------------------- C-ABI names
def gemm_options_default() -> gemm_options_t:
    o = gemm_options_t()
    _lib.gemm_options_default(ctypes.byref(o))
    return o


def gemm_create(opt: gemm_options_t, device: int = 0):
    """Returns (status, handle); handle is an opaque int (0 on failure)."""
    h = _vp()
    s = _lib.gemm_create(ctypes.byref(h), ctypes.byref(opt), device)
    return s, (h.value or 0)


def gemm_run(h, M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, stream=None) -> int:
    return _lib.gemm_run(h, M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc, alpha, beta, _stream(stream))


def gemm_run_strided_batched(h, M, N, K, A, lda, strideA, B, ldb, strideB, C, ldc, strideC, batch,
                             alpha, beta, stream=None) -> int:
    return _lib.gemm_run_strided_batched(h, M, N, K, _ptr(A), lda, strideA, _ptr(B), ldb, strideB, _ptr(C),
                                         ldc, strideC, batch, alpha, beta, _stream(stream))


def gemm_run_strided_batched_host(h, M, N, K, A, lda, sA, B, ldb, sB, C, ldc, sC, batch, alpha, beta,
                                  stream=None) -> int:
    return _lib.gemm_run_strided_batched_host(h, M, N, K, _ptr(A), lda, sA, _ptr(B), ldb, sB, _ptr(C), ldc, sC, batch,
                                              alpha, beta, _stream(stream))


def gemm_run_host(h, M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, stream=None) -> int:
    return _lib.gemm_run_host(h, M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc, alpha, beta,
                              _stream(stream))


def gemm_query_status(h, stream=None) -> int:
    return _lib.gemm_query_status(h, _stream(stream))


def gemm_read_clock(h, stream=None):
    """Returns (status, (cycles, nanoseconds, ctas)) of the handle's clock probe since the last
    read, and clears the counters."""
    out = (ctypes.c_uint64 * 3)()
    s = _lib.gemm_read_clock(h, _stream(stream), out)
    return s, (int(out[0]), int(out[1]), int(out[2]))


def gemm_plan(opt: gemm_options_t, M, N, K, batch=1, sm_count=152):
    """Returns (status, gemm_plan_t); sm_count defaults to GB300's 152 SMs."""
    p = gemm_plan_t()
    s = _lib.gemm_plan(ctypes.byref(opt), M, N, K, batch, sm_count, ctypes.byref(p))
    return s, p


def gemm_status_string(s: int) -> str:
    return _lib.gemm_status_string(s).decode()


def gemm_last_error(h=None) -> str:
    return (_lib.gemm_last_error(h) or b"").decode()


def gemm_launch_count(h) -> int:
    return int(_lib.gemm_launch_count(h))


def gemm_destroy(h) -> int:
    return _lib.gemm_destroy(h)


def gemm_run_noalloc(opt: gemm_options_t, device, M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, stream=None,
                     status_out=None) -> int:
    """The allocation-free variant of gemm_run (no handle). ``status_out``: None, or a
    ``(ctypes.c_uint32 * 4)`` array that receives the status record (the call then synchronizes)."""
    return _lib.gemm_run_noalloc(ctypes.byref(opt), device, M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc,
                                 alpha, beta, _stream(stream), status_out)


# ---------------------------------------------------------------- convenience
class GemmError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{gemm_status_string(status)}: {message}")
        self.status = status


def make_options(**kw) -> gemm_options_t:
    """gemm_options_default() with fields overridden by keyword (layouts as "row"/"col",
    out_type as "bf16"/"f32", mode as "unicast"/"mcast")."""
    o = gemm_options_default()
    names = {"row": GEMM_ROW_MAJOR, "col": GEMM_COL_MAJOR, "bf16": GEMM_OUT_BF16, "f32": GEMM_OUT_F32,
             "unicast": GEMM_MODE_UNICAST, "mcast": GEMM_MODE_MCAST, "auto": 0, "dp": 1, "stream_k": 2, "clc": 3}
    for k, v in kw.items():
        if not hasattr(o, k):
            raise TypeError(f"gemm_options_t has no field {k!r}")
        setattr(o, k, names.get(v, v) if isinstance(v, str) else int(v))
    return o


class Gemm:
    """A handle bound to one device and one set of options (the fields of gemm_options_t as
    keywords: mode, mcast_a, mcast_b, cluster_m, cluster_n, cta_group (1, 2, or 0 for the pair
    wherever the cluster's extent along M is even), layout_a/b/c ("row" or
    "col"), out_type ("bf16" or "f32"), block_n, block_k, stages, max_clusters, group_m,
    schedule ("auto", "dp", "stream_k", "clc"), wait_timeout_ns, host_parts, clock_probe).

    Buffers are torch tensors or integer addresses (numpy arrays for the host entry points);
    sizes, leading dimensions and strides are in elements; `stream` is a torch.cuda.Stream, a
    raw cudaStream_t as an int, or None for the legacy default stream. Every call raises
    GemmError on a non-OK status. Usable as a context manager (closes the handle).
    """

    def __init__(self, device: int = 0, **options):
        self.options = make_options(**options)
        s, self.handle = gemm_create(self.options, device)
        if s != GEMM_OK:
            raise GemmError(s, gemm_last_error(None))

    def check(self, status: int) -> None:
        if status != GEMM_OK:
            raise GemmError(status, gemm_last_error(self.handle))

    def run(self, M, N, K, A, lda, B, ldb, C, ldc, alpha=1.0, beta=0.0, stream=None) -> None:
        """C <- alpha * A.B + beta * C on device buffers, asynchronously on `stream`."""
        self.check(gemm_run(self.handle, M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, stream))

    def run_strided_batched(self, M, N, K, A, lda, sA, B, ldb, sB, C, ldc, sC, batch, alpha=1.0, beta=0.0,
                            stream=None) -> None:
        """`batch` GEMMs, operand i at base + i * stride (a stride of 0 shares one operand)."""
        self.check(gemm_run_strided_batched(self.handle, M, N, K, A, lda, sA, B, ldb, sB, C, ldc, sC, batch,
                                            alpha, beta, stream))

    def run_host(self, M, N, K, A, lda, B, ldb, C, ldc, alpha=1.0, beta=0.0, stream=None) -> None:
        """run() on host buffers (pinned for full speed): the copies in and out are pipelined
        with the GEMMs, and C holds the result when the call returns."""
        self.check(gemm_run_host(self.handle, M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, stream))

    def run_strided_batched_host(self, M, N, K, A, lda, sA, B, ldb, sB, C, ldc, sC, batch, alpha=1.0, beta=0.0,
                                 stream=None) -> None:
        """run_strided_batched() on host buffers, pipelined over the batch."""
        self.check(gemm_run_strided_batched_host(self.handle, M, N, K, A, lda, sA, B, ldb, sB, C, ldc, sC, batch,
                                                 alpha, beta, stream))

    def read_clock(self, stream=None) -> dict:
        """The clock probe (options clock_probe=1) since the last read: SM cycles, nanoseconds
        and CTAs summed over the kernel's CTAs, and their ratio, the mean SM clock in GHz.
        Synchronises `stream` and clears the counters."""
        s, (c, ns, n) = gemm_read_clock(self.handle, stream)
        self.check(s)
        return {"cycles": c, "ns": ns, "ctas": n, "ghz": c / ns if ns else None}

    def query_status(self, stream=None) -> int:
        """Synchronises `stream` and returns the status of the runs on it (a bounded in-kernel
        wait that expired reports GEMM_ERR_DEVICE_TIMEOUT)."""
        return gemm_query_status(self.handle, stream)

    @property
    def launches(self) -> int:
        return gemm_launch_count(self.handle)

    def close(self) -> None:
        if self.handle:
            gemm_destroy(self.handle)
            self.handle = 0

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
        return False

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ---------------------------------------------------------------- TMA microbenchmark (include/tma_bench.h)
TMA_BENCH_UNICAST = 0
TMA_BENCH_MULTICAST = 1
TMA_BENCH_MULTICAST_SLICED = 2


class tma_bench_options_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "mode", "cluster", "ctas", "box_rows", "stages", "iters", "warmup", "streaming_stride")] + [
        ("wait_timeout_ns", ctypes.c_uint64), ("landed", ctypes.c_void_p), ("origin", ctypes.c_void_p)]


_lib.tma_bench_run.argtypes = [ctypes.POINTER(tma_bench_options_t), _vp, _i64, _i64, _i64, _vp, _vp, _vp,
                               ctypes.POINTER(_i32), ctypes.POINTER(ctypes.c_double),
                               ctypes.POINTER(ctypes.c_double), _vp]
_lib.tma_bench_run.restype = _i32
_lib.tma_bench_query_status.argtypes = [_vp]
_lib.tma_bench_query_status.restype = _i32
_lib.tma_bench_last_error.argtypes = []
_lib.tma_bench_last_error.restype = ctypes.c_char_p


def tma_bench_run(opt: tma_bench_options_t, src, rows, cols, ld, cycles, ns, verify, stream=None):
    """Returns (status, ctas_used, delivered_bytes, issued_bytes)."""
    n = _i32(0)
    d = ctypes.c_double(0.0)
    i = ctypes.c_double(0.0)
    s = _lib.tma_bench_run(ctypes.byref(opt), _ptr(src), rows, cols, ld, _ptr(cycles), _ptr(ns), _ptr(verify),
                           ctypes.byref(n), ctypes.byref(d), ctypes.byref(i), _stream(stream))
    return s, n.value, d.value, i.value


def tma_bench_query_status(stream=None) -> int:
    return _lib.tma_bench_query_status(_stream(stream))


def tma_bench_last_error() -> str:
    return (_lib.tma_bench_last_error() or b"").decode()


# ---------------------------------------------------------------- cluster halo-exchange stencil (include/stencil.h)
STENCIL_TILE = 8192
_lib.stencil_1d_run.argtypes = [_vp, _vp, _i64, _i32, _vp]
_lib.stencil_1d_run.restype = _i32
_lib.stencil_1d_query_status.argtypes = [_vp]
_lib.stencil_1d_query_status.restype = _i32


def stencil_1d_run(x, y, n, cluster, stream=None) -> int:
    return _lib.stencil_1d_run(_ptr(x), _ptr(y), n, cluster, _stream(stream))


def stencil_1d_query_status(stream=None) -> int:
    return _lib.stencil_1d_query_status(_stream(stream))


# ---------------------------------------------------------------- fused attention forward (include/attention.h)
_lib.attention_forward_run.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _f32, _i32, _i32, _i32, _i32,
                                       _vp]
_lib.attention_forward_run.restype = _i32
_lib.attention_forward_query_status.argtypes = [_vp]
_lib.attention_forward_query_status.restype = _i32


def attention_forward_run(Q, K, V, O, lse, batch, sq, sk, d, scale=0.0, out_f32=0, cluster=1, cta_group=1,
                          causal=0, stream=None) -> int:
    return _lib.attention_forward_run(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(lse), batch, sq, sk, d, scale,
                                      out_f32, cluster, cta_group, 1 if causal else 0, _stream(stream))


def attention_forward_query_status(stream=None) -> int:
    return _lib.attention_forward_query_status(_stream(stream))


_lib.attention_forward_run_host.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _f32, _i32, _i32,
                                            _i32, _i32, _vp, ctypes.c_size_t, _vp]
_lib.attention_forward_run_host.restype = _i32
_lib.attention_forward_host_workspace_bytes.argtypes = [_i64, _i64, _i64, _i64, _i32]
_lib.attention_forward_host_workspace_bytes.restype = ctypes.c_size_t


def attention_forward_host_workspace_bytes(batch, sq, sk, d, out_f32=0) -> int:
    return _lib.attention_forward_host_workspace_bytes(batch, sq, sk, d, out_f32)


def attention_forward_run_host(Q, K, V, O, lse, batch, sq, sk, d, workspace, workspace_bytes, scale=0.0, out_f32=0,
                               cluster=1, cta_group=1, causal=0, stream=None) -> int:
    """Host Q, K, V, O, lse (numpy arrays or pinned CPU tensors); `workspace` is device memory."""
    return _lib.attention_forward_run_host(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(lse), batch, sq, sk, d, scale,
                                           out_f32, cluster, cta_group, 1 if causal else 0, _ptr(workspace),
                                           workspace_bytes, _stream(stream))
