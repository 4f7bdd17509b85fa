"""ctypes binding of libsgemm.so, with the entry-point names of include/sgemm.h.

Argument marshalling only: every step of C = alpha*A*B + beta*C runs in the
CUDA library.  Matrix arguments may be raw device addresses (int) or objects
with ``data_ptr()`` (torch tensors); streams may be an int handle, a
``torch.cuda.Stream`` or ``None`` (torch's current stream).  A non-zero
status raises ``SgemmError``.  If the library has not been built the first
call raises -- there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

OK = 0
ERR_NULL = 1
ERR_INVALID_VALUE = 2
ERR_ALIAS = 3
ERR_BAD_HANDLE = 4
ERR_UNSUPPORTED_DEVICE = 5
ERR_LAUNCH = 6
ERR_CUDA = 7
ERR_DEVICE_TIMEOUT = 8
ERR_WRONG_DEVICE = 9
ERR_SCRATCH_TOO_SMALL = 10
ERR_DEVICE_CHECK = 11

VARIANT_AUTO = 0
VARIANT_TMA_128x256 = 1
VARIANT_TMA_128x128 = 2
VARIANT_TMA_64x64 = 3
VARIANT_TMA_64x64_SPLITK = 4
VARIANT_GENERIC = 5
VARIANT_SCALE = 6
VARIANT_TC_3XTF32 = 7
VARIANT_TC_3XTF32_PAIR = 8
VARIANT_TC_F16_PAIR = 9
VARIANT_GENERIC_F16 = 10
VARIANT_TMA_256x128 = 11
VARIANT_COUNT = 12
MATH_FP32 = 0
MATH_3XTF32 = 1
IN_BF16 = 1
IN_F16 = 2
RELAYOUT_AUTO = 0
RELAYOUT_OFF = 1
RELAYOUT_ALWAYS = 2
# sgemm_sk_sums_t: how a stream-K tile's parts are added (test hook)
SK_SUMS_AUTO, SK_SUMS_LAST, SK_SUMS_DEFERRED, SK_SUMS_SHARED = 0, 1, 2, 3
GEMM_VARIANTS = (VARIANT_TMA_256x128, VARIANT_TMA_128x256, VARIANT_TMA_128x128, VARIANT_TMA_64x64,
                 VARIANT_TMA_64x64_SPLITK, VARIANT_GENERIC, VARIANT_TC_3XTF32, VARIANT_TC_3XTF32_PAIR)

#: Every exported entry point of include/sgemm.h.
EXPORTS = ("sgemm_create", "sgemm_run", "sgemm_check_args", "sgemm_destroy", "sgemm_set_variant",
           "sgemm_last_variant", "sgemm_get_device_status", "sgemm_debug_timeout_probe",
           "sgemm_debug_set_smem_override", "sgemm_status_string", "sgemm_variant_name",
           "sgemm_version", "sgemm_run_noalloc", "sgemm_set_math_mode", "sgemm_run_host",
           "sgemm_run_ex", "sgemm_check_args_ex", "sgemm_last_launches", "sgemm_run_mixed",
           "sgemm_check_args_mixed", "sgemm_debug_fma_probe", "sgemm_debug_bank_probe",
           "sgemm_set_relayout", "sgemm_last_relayout", "sgemm_relayout_capacity", "sgemm_debug_plan",
           "sgemm_debug_set_stream_k_sums", "sgemm_debug_set_cluster_split", "sgemm_debug_set_stream_k_ctas",
           "sgemm_debug_set_stream_k_gap", "sgemm_debug_leave_aborted_state", "sgemm_debug_tf32_probe",
           "sgemm_debug_set_workspace_limit")


class SgemmError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}" if where else status_string(status))


_lib = None
_calls = None          # the compiled marshalling module for sgemm_run / sgemm_run_ex, when built
_calls_tried = False


def library_path() -> str:
    """The library to load: the in-tree build, or the file named by the
    SGEMM_LIBRARY environment variable (a build of the same sources with
    other flags, such as the device-checked build)."""
    return os.environ.get("SGEMM_LIBRARY") or _build.LIB


def lib() -> ctypes.CDLL:
    """The loaded CUDA library (raises if it was never built)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it first (dense_fp32_matrix_09_gb300.build.build())")
        L = ctypes.CDLL(path)
        vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        L.sgemm_create.argtypes = [ctypes.POINTER(vp)]
        L.sgemm_run.argtypes = [vp, i32, i32, i32, f32, vp, i32, vp, i32, f32, vp, i32, vp]
        L.sgemm_check_args.argtypes = [i32, i32, i32, f32, vp, i32, vp, i32, f32, vp, i32]
        L.sgemm_destroy.argtypes = [vp]
        L.sgemm_set_variant.argtypes = [vp, i32]
        L.sgemm_last_variant.argtypes = [vp, ctypes.POINTER(i32)]
        L.sgemm_last_launches.argtypes = [vp]
        L.sgemm_set_relayout.argtypes = [vp, i32]
        L.sgemm_last_relayout.argtypes = [vp]
        L.sgemm_relayout_capacity.argtypes = [vp]
        L.sgemm_relayout_capacity.restype = ctypes.c_longlong
        L.sgemm_debug_plan.argtypes = [i32, ctypes.POINTER(i32), ctypes.c_longlong, i32, i32, i32, i32, i32, i32, i32,
                                       i32, f32, i32, ctypes.c_longlong, ctypes.c_longlong, i32, ctypes.POINTER(i32)]
        L.sgemm_debug_fma_probe.argtypes = [vp, i32, i32, vp, ctypes.POINTER(ctypes.c_longlong), vp]
        L.sgemm_debug_tf32_probe.argtypes = [vp, i32, i32, ctypes.POINTER(ctypes.c_longlong), vp]
        L.sgemm_debug_bank_probe.argtypes = [vp, i32, i32, i32, vp, vp]
        L.sgemm_run_mixed.argtypes = [vp, i32, i32, i32, i32, i32, i32, f32, vp, i32, vp, i32, f32, vp, i32, vp]
        L.sgemm_check_args_mixed.argtypes = [i32, i32, i32, i32, i32, i32, f32, vp, i32, vp, i32, f32, vp, i32]
        L.sgemm_get_device_status.argtypes = [vp]
        L.sgemm_debug_timeout_probe.argtypes = [vp, ctypes.c_longlong, vp]
        L.sgemm_debug_set_smem_override.argtypes = [vp, i32]
        L.sgemm_debug_set_stream_k_sums.argtypes = [vp, i32]
        L.sgemm_debug_set_cluster_split.argtypes = [vp, i32]
        L.sgemm_debug_set_stream_k_ctas.argtypes = [vp, i32]
        L.sgemm_debug_set_stream_k_gap.argtypes = [vp, i32]
        L.sgemm_debug_leave_aborted_state.argtypes = [vp]
        L.sgemm_debug_set_workspace_limit.argtypes = [vp, i32]
        L.sgemm_status_string.argtypes = [i32]
        L.sgemm_status_string.restype = ctypes.c_char_p
        L.sgemm_variant_name.argtypes = [i32]
        L.sgemm_variant_name.restype = ctypes.c_char_p
        L.sgemm_version.argtypes = []
        L.sgemm_set_math_mode.argtypes = [vp, i32]
        i64 = ctypes.c_longlong
        L.sgemm_run_ex.argtypes = [vp, i32, i32, i32, i32, i32, f32, vp, i32, i64, vp, i32, i64, f32, vp, i32, i64,
                                   i32, vp]
        L.sgemm_check_args_ex.argtypes = [i32, i32, i32, i32, i32, f32, vp, i32, i64, vp, i32, i64, f32, vp, i32,
                                          i64, i32]
        L.sgemm_run_host.argtypes = [vp, i32, i32, i32, f32, vp, i32, vp, i32, f32, vp, i32, vp, vp, vp, vp]
        L.sgemm_run_noalloc.argtypes = [i32, i32, i32, f32, vp, i32, vp, i32, f32, vp, i32, vp]
        _lib = L
    return _lib


def _current_stream_handle() -> int:
    import torch
    return int(torch.cuda.current_stream().cuda_stream)


def calls_module():
    """The CPython module that marshals sgemm_run / sgemm_run_ex arguments
    (built next to the library by build.py), bound to the loaded library; None
    when it was not built -- the two calls then go through ctypes."""
    global _calls, _calls_tried
    if not _calls_tried:
        _calls_tried = True
        path = _build.CALLS
        if os.path.exists(path):
            import importlib.util
            lib()  # the library is loaded first; the module binds the same instance by path
            try:
                spec = importlib.util.spec_from_file_location("_sgemm_calls", path)
                mod = importlib.util.module_from_spec(spec)
                spec.loader.exec_module(mod)
                mod.init(library_path(), _current_stream_handle)
                _calls = mod
            except (ImportError, OSError):
                _calls = None  # a module built for another interpreter or machine: ctypes serves
    return _calls


def _ptr(x) -> int | None:
    """Address of a buffer: an int, a torch tensor (data_ptr) or a numpy array."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    return int(x.__array_interface__["data"][0])


def _stream(s) -> int:
    if s is None:
        return _current_stream_handle()
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _check(rc: int, where: str) -> int:
    if rc != OK:
        raise SgemmError(rc, where)
    return rc


def status_string(status: int) -> str:
    return lib().sgemm_status_string(int(status)).decode()


def variant_name(variant: int) -> str:
    return lib().sgemm_variant_name(int(variant)).decode()


def sgemm_version() -> int:
    return lib().sgemm_version()


def sgemm_create() -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    _check(lib().sgemm_create(ctypes.byref(h)), "sgemm_create")
    return h


def sgemm_destroy(h) -> None:
    _check(lib().sgemm_destroy(h), "sgemm_destroy")


def sgemm_run(h, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> None:
    """C <- alpha*A*B + beta*C on device buffers (row-major, leading dims)."""
    calls = _calls if _calls is not None else calls_module()
    if calls is not None:
        rc = calls.run(h, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)
    else:
        rc = lib().sgemm_run(h, int(M), int(N), int(K), float(alpha), _ptr(A), int(lda), _ptr(B),
                             int(ldb), float(beta), _ptr(C), int(ldc), _stream(stream))
    if rc != OK:
        raise SgemmError(rc, "sgemm_run")


def sgemm_run_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> None:
    """C <- alpha*A*B + beta*C without allocating anything (no handle; fixed
    in-library scratch, at most 512 output tiles of 64 x 64).  For callers that
    cannot allocate GPU memory; see include/sgemm.h for the sharing rules."""
    _check(lib().sgemm_run_noalloc(int(M), int(N), int(K), float(alpha), _ptr(A), int(lda), _ptr(B),
                                   int(ldb), float(beta), _ptr(C), int(ldc), _stream(stream)),
           "sgemm_run_noalloc")


def sgemm_run_host(h, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dA, dB, dC, stream=None) -> None:
    """C <- alpha*A*B + beta*C with A, B, C in host memory (page-locked for
    overlap), through the device staging buffers dA, dB, dC; copies overlap
    the per-panel GEMMs.  C is complete once `stream` has reached the call."""
    _check(lib().sgemm_run_host(h, int(M), int(N), int(K), float(alpha), _ptr(A), int(lda), _ptr(B), int(ldb),
                                float(beta), _ptr(C), int(ldc), _ptr(dA), _ptr(dB), _ptr(dC), _stream(stream)),
           "sgemm_run_host")


def sgemm_run_ex(h, transA, transB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc, strideC,
                 batch=1, stream=None) -> None:
    """C_b <- alpha*op(A_b)*op(B_b) + beta*C_b, b = 0..batch-1 (see include/sgemm.h)."""
    calls = _calls if _calls is not None else calls_module()
    if calls is not None:
        rc = calls.run_ex(h, transA, transB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc,
                          strideC, batch, stream)
    else:
        rc = lib().sgemm_run_ex(h, int(transA), int(transB), int(M), int(N), int(K), float(alpha), _ptr(A),
                                int(lda), int(strideA), _ptr(B), int(ldb), int(strideB), float(beta), _ptr(C),
                                int(ldc), int(strideC), int(batch), _stream(stream))
    if rc != OK:
        raise SgemmError(rc, "sgemm_run_ex")


def sgemm_check_args_ex(transA, transB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc, strideC,
                        batch=1) -> int:
    return lib().sgemm_check_args_ex(int(transA), int(transB), int(M), int(N), int(K), float(alpha), _ptr(A),
                                     int(lda), int(strideA), _ptr(B), int(ldb), int(strideB), float(beta), _ptr(C),
                                     int(ldc), int(strideC), int(batch))


def sgemm_check_args(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc) -> int:
    """Host-only validation; returns the status sgemm_run would return for these arguments."""
    return lib().sgemm_check_args(int(M), int(N), int(K), float(alpha), _ptr(A), int(lda), _ptr(B),
                                  int(ldb), float(beta), _ptr(C), int(ldc))


def sgemm_set_variant(h, variant: int) -> None:
    _check(lib().sgemm_set_variant(h, int(variant)), "sgemm_set_variant")


def sgemm_set_math_mode(h, mode: int) -> None:
    _check(lib().sgemm_set_math_mode(h, int(mode)), "sgemm_set_math_mode")


def sgemm_last_variant(h) -> tuple[int, int]:
    splits = ctypes.c_int(0)
    v = lib().sgemm_last_variant(h, ctypes.byref(splits))
    return v, splits.value


def sgemm_run_mixed(h, in_type, transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> None:
    """C <- alpha*op(A)*op(B) + beta*C with 16-bit A, B and FP32 C (see include/sgemm.h)."""
    _check(lib().sgemm_run_mixed(h, int(in_type), int(transA), int(transB), int(M), int(N), int(K), float(alpha),
                                 _ptr(A), int(lda), _ptr(B), int(ldb), float(beta), _ptr(C), int(ldc),
                                 _stream(stream)), "sgemm_run_mixed")


def sgemm_check_args_mixed(in_type, transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc) -> int:
    return lib().sgemm_check_args_mixed(int(in_type), int(transA), int(transB), int(M), int(N), int(K),
                                        float(alpha), _ptr(A), int(lda), _ptr(B), int(ldb), float(beta), _ptr(C),
                                        int(ldc))


def sgemm_debug_fma_probe(h, sink, ctas=0, iters=4096, stream=None) -> int:
    """Enqueue the FP32 FMA-rate probe (sink: ctas*256 floats on the device);
    returns the FLOP it performs."""
    flops = ctypes.c_longlong(0)
    _check(lib().sgemm_debug_fma_probe(h, int(ctas), int(iters), _ptr(sink), ctypes.byref(flops), _stream(stream)),
           "sgemm_debug_fma_probe")
    return flops.value


def sgemm_debug_tf32_probe(h, clusters=0, iters=4096, stream=None) -> int:
    """Enqueue the TF32 tensor-pipe rate probe; returns the TF32 FLOP it performs."""
    flops = ctypes.c_longlong(0)
    _check(lib().sgemm_debug_tf32_probe(h, int(clusters), int(iters), ctypes.byref(flops), _stream(stream)),
           "sgemm_debug_tf32_probe")
    return flops.value


def sgemm_debug_bank_probe(h, padded, sink, ctas=0, iters=64, stream=None) -> None:
    """Enqueue the shared-memory bank probe (sink: ctas*32 floats on the device)."""
    _check(lib().sgemm_debug_bank_probe(h, int(padded), int(ctas), int(iters), _ptr(sink), _stream(stream)),
           "sgemm_debug_bank_probe")


def sgemm_last_launches(h) -> int:
    return lib().sgemm_last_launches(h)


def sgemm_set_relayout(h, mode: int) -> None:
    _check(lib().sgemm_set_relayout(h, int(mode)), "sgemm_set_relayout")


def sgemm_last_relayout(h) -> int:
    """Operands the last call copied transposed first: bit 0 A, bit 1 B."""
    return lib().sgemm_last_relayout(h)


def sgemm_relayout_capacity(h) -> int:
    return lib().sgemm_relayout_capacity(h)


PLAN_FIELDS = ("kind", "variant", "copies", "op", "dp_tiles", "sk_ctas", "tiles", "launches", "splits",
               "fixup", "ksplit", "tc_bk", "sk_gap")
# "fixup": how the stream-K tiles' parts are added (0 last CTA or no stream-K, 1 second kernel, 2 shared)
FIXUP_LAST, FIXUP_DEFERRED, FIXUP_SHARED = 0, 1, 2
PLAN_NOTHING, PLAN_SCALE, PLAN_TENSOR_CORE, PLAN_GENERIC, PLAN_TMA = 0, 1, 2, 3, 4


def sgemm_debug_plan(num_sms, ctas_per_sm, transA, transB, M, N, K, *, alpha=1.0, batch=1, strideA=0,
                     strideB=0, tma_ok=True, relayout_floats=2 * 8192 * 8192, relayout_mode=RELAYOUT_AUTO,
                     math_mode=MATH_FP32, pinned=VARIANT_AUTO) -> dict:
    """The plan sgemm_run_ex would follow, computed on the host (no GPU):
    a dict with the fields of PLAN_FIELDS (see include/sgemm.h).  ``tma_ok``:
    True (both operands TMA-readable as stored), False (neither), or the
    bitmask of those that are (bit 0 A, bit 1 B)."""
    aligned = 3 if tma_ok is True else 0 if tma_ok is False else int(tma_ok)
    occ = (ctypes.c_int * VARIANT_COUNT)(*ctas_per_sm)
    out = (ctypes.c_int * len(PLAN_FIELDS))()
    _check(lib().sgemm_debug_plan(int(num_sms), occ, int(relayout_floats), int(relayout_mode), int(math_mode),
                                  int(pinned), int(transA), int(transB), int(M), int(N), int(K), float(alpha),
                                  int(batch), int(strideA), int(strideB), aligned, out),
           "sgemm_debug_plan")
    return dict(zip(PLAN_FIELDS, list(out)))


def sgemm_get_device_status(h) -> int:
    return lib().sgemm_get_device_status(h)


def sgemm_debug_timeout_probe(h, limit_ns: int, stream=None) -> None:
    _check(lib().sgemm_debug_timeout_probe(h, int(limit_ns), _stream(stream)), "sgemm_debug_timeout_probe")


def sgemm_debug_set_smem_override(h, nbytes: int) -> None:
    _check(lib().sgemm_debug_set_smem_override(h, int(nbytes)), "sgemm_debug_set_smem_override")


def sgemm_debug_set_workspace_limit(h, tiles: int) -> None:
    _check(lib().sgemm_debug_set_workspace_limit(h, int(tiles)), "sgemm_debug_set_workspace_limit")


def sgemm_debug_leave_aborted_state(h) -> None:
    _check(lib().sgemm_debug_leave_aborted_state(h), "sgemm_debug_leave_aborted_state")


def sgemm_debug_set_stream_k_ctas(h, ctas: int) -> None:
    """Test hook: stream-K CTAs of later calls' stream-K plans (0: the library's choice)."""
    _check(lib().sgemm_debug_set_stream_k_ctas(h, int(ctas)), "sgemm_debug_set_stream_k_ctas")


def sgemm_debug_set_stream_k_gap(h, gap: int) -> None:
    """Test hook: boundary charge of later calls' stream-K splits, in
    sixteenths of a K step (-1: the library's choice; 0: the even split)."""
    _check(lib().sgemm_debug_set_stream_k_gap(h, int(gap)), "sgemm_debug_set_stream_k_gap")


def sgemm_debug_set_cluster_split(h, ksplit: int) -> None:
    """0: automatic; 1: no cluster split-K; 2..8: that many CTAs per tile."""
    _check(lib().sgemm_debug_set_cluster_split(h, int(ksplit)), "sgemm_debug_set_cluster_split")


def sgemm_debug_set_stream_k_sums(h, mode: int) -> None:
    """mode: one of SK_SUMS_AUTO, SK_SUMS_LAST, SK_SUMS_DEFERRED, SK_SUMS_SHARED."""
    _check(lib().sgemm_debug_set_stream_k_sums(h, int(mode)), "sgemm_debug_set_stream_k_sums")


class Sgemm:
    """A handle as a context manager: ``with Sgemm() as g: g.run(...)``."""

    def __init__(self, variant: int = VARIANT_AUTO):
        self.h = sgemm_create()
        if variant != VARIANT_AUTO:
            sgemm_set_variant(self.h, variant)

    def run(self, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None):
        sgemm_run(self.h, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)

    def matmul(self, A, B, C, alpha=1.0, beta=0.0, stream=None):
        """C <- alpha*A@B + beta*C for 2-D row-major torch tensors (unit column stride)."""
        M, K = A.shape
        K2, N = B.shape
        if K2 != K or tuple(C.shape) != (M, N):
            raise ValueError(f"shape mismatch: {tuple(A.shape)} @ {tuple(B.shape)} -> {tuple(C.shape)}")
        for t in (A, B, C):
            if t.dim() != 2 or (t.numel() and t.stride(1) != 1):
                raise ValueError("operands must be 2-D with unit column stride")
        sgemm_run(self.h, M, N, K, alpha, A, max(A.stride(0), 1), B, max(B.stride(0), 1), beta, C,
                  max(C.stride(0), 1), stream)
        return C

    @property
    def last_variant(self):
        return sgemm_last_variant(self.h)

    def set_variant(self, v):
        sgemm_set_variant(self.h, v)

    def set_relayout(self, mode):
        sgemm_set_relayout(self.h, mode)

    @property
    def last_relayout(self) -> int:
        return sgemm_last_relayout(self.h)

    def device_status(self) -> int:
        return sgemm_get_device_status(self.h)

    def close(self):
        if self.h is not None:
            sgemm_destroy(self.h)
            self.h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
