"""The C-ABI library on the CPU: it builds for sm_103a, exports every entry
point include/sgemm.h declares, and its host-only logic (argument checks,
handle checks, status strings) behaves as documented.  No compute call is
made here; those are the GPU tests."""
import ctypes
import os
import re

import pytest

from dense_fp32_matrix_09_gb300 import build, sgemm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sgemm.h")

OK, NULL_, INVALID, ALIAS = sgemm.OK, sgemm.ERR_NULL, sgemm.ERR_INVALID_VALUE, sgemm.ERR_ALIAS


@pytest.fixture(scope="module")
def lib():
    build.build()
    return sgemm.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(sgemm_\w+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 12, names
    assert set(names) == set(sgemm.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_built_for_sm103a_only():
    assert "arch=compute_103a,code=sm_103a" in build.GENCODE


def test_status_and_variant_strings(lib):
    for s in range(12):
        assert sgemm.status_string(s).startswith("SGEMM_")
    assert sgemm.status_string(99) == "SGEMM_ERR_UNKNOWN"
    assert sgemm.variant_name(sgemm.VARIANT_TMA_128x256) == "tma_128x256"
    assert sgemm.sgemm_version() == 10000


def header_enum_values():
    """NAME -> value for every `NAME = value` enumerator of include/sgemm.h."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return {m.group(1): int(m.group(2)) for m in re.finditer(r"\b(SGEMM_[A-Z0-9_x]+)\s*=\s*(\d+)", text)}


def test_binding_constants_match_the_header():
    """Every constant the Python binding mirrors has the header's value, and
    every variant name the library reports matches its enumerator."""
    values = header_enum_values()
    pairs = {"OK": "SGEMM_OK", "ERR_NULL": "SGEMM_ERR_NULL", "ERR_INVALID_VALUE": "SGEMM_ERR_INVALID_VALUE",
             "ERR_ALIAS": "SGEMM_ERR_ALIAS", "ERR_BAD_HANDLE": "SGEMM_ERR_BAD_HANDLE",
             "ERR_UNSUPPORTED_DEVICE": "SGEMM_ERR_UNSUPPORTED_DEVICE", "ERR_LAUNCH": "SGEMM_ERR_LAUNCH",
             "ERR_CUDA": "SGEMM_ERR_CUDA", "ERR_DEVICE_TIMEOUT": "SGEMM_ERR_DEVICE_TIMEOUT",
             "ERR_WRONG_DEVICE": "SGEMM_ERR_WRONG_DEVICE", "ERR_SCRATCH_TOO_SMALL": "SGEMM_ERR_SCRATCH_TOO_SMALL",
             "ERR_DEVICE_CHECK": "SGEMM_ERR_DEVICE_CHECK",
             "MATH_FP32": "SGEMM_MATH_FP32", "MATH_3XTF32": "SGEMM_MATH_3XTF32", "IN_BF16": "SGEMM_IN_BF16",
             "IN_F16": "SGEMM_IN_F16", "RELAYOUT_AUTO": "SGEMM_RELAYOUT_AUTO", "RELAYOUT_OFF": "SGEMM_RELAYOUT_OFF",
             "RELAYOUT_ALWAYS": "SGEMM_RELAYOUT_ALWAYS", "VARIANT_COUNT": "SGEMM_VARIANT_COUNT_"}
    for name in dir(sgemm):
        if (name.startswith("VARIANT_") and name != "VARIANT_COUNT") or name.startswith("SK_SUMS_"):
            pairs[name] = "SGEMM_" + name
    for py, c in pairs.items():
        assert getattr(sgemm, py) == values[c], (py, c)
    variants = {k: v for k, v in values.items() if k.startswith("SGEMM_VARIANT_") and not k.endswith("_")}
    assert len(variants) == values["SGEMM_VARIANT_COUNT_"]
    assert sorted(variants.values()) == list(range(values["SGEMM_VARIANT_COUNT_"]))


def test_variant_names_match_the_enumerators(lib):
    for c, v in header_enum_values().items():
        if c.startswith("SGEMM_VARIANT_") and not c.endswith("_"):
            assert sgemm.variant_name(v) == c[len("SGEMM_VARIANT_"):].lower(), c


# Fake, never-dereferenced device addresses (only compared by the checks).
A0, B0, C0 = 0x10000000, 0x20000000, 0x30000000


def chk(M, N, K, alpha=1.0, A=A0, lda=None, B=B0, ldb=None, beta=0.0, C=C0, ldc=None):
    lda = max(K, 1) if lda is None else lda
    ldb = max(N, 1) if ldb is None else ldb
    ldc = max(N, 1) if ldc is None else ldc
    return sgemm.sgemm_check_args(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc)


def test_check_args_sizes_and_leading_dims(lib):
    assert chk(4, 5, 6) == OK
    assert chk(-1, 5, 6) == INVALID
    assert chk(4, -5, 6) == INVALID
    assert chk(4, 5, -6) == INVALID
    assert chk(4, 5, 6, lda=5) == INVALID      # lda < K
    assert chk(4, 5, 6, ldb=4) == INVALID      # ldb < N
    assert chk(4, 5, 6, ldc=4) == INVALID      # ldc < N
    assert chk(4, 5, 0, lda=0) == INVALID      # lda < max(1, K)
    assert chk(4, 5, 6, lda=7, ldb=9, ldc=8) == OK
    assert chk(1000, 1500, 777, lda=780, ldb=1504, ldc=1504) == OK


def test_check_args_null_rules(lib):
    assert chk(0, 5, 6, A=None, B=None, C=None) == OK            # M == 0: nothing referenced
    assert chk(4, 0, 6, A=None, B=None, C=None) == OK
    assert chk(4, 5, 6, C=None) == NULL_
    assert chk(4, 5, 6, A=None) == NULL_
    assert chk(4, 5, 6, B=None) == NULL_
    assert chk(4, 5, 6, alpha=0.0, A=None, B=None, beta=2.0) == OK  # A, B not referenced
    assert chk(4, 5, 0, A=None, B=None) == OK


def test_check_args_alias(lib):
    M, N, K = 4, 5, 6
    # C starting inside A's window
    assert chk(M, N, K, C=A0 + 8) == ALIAS
    # C ending exactly where B starts: no overlap
    c_bytes = ((M - 1) * N + N) * 4
    assert chk(M, N, K, C=B0 - c_bytes) == OK
    assert chk(M, N, K, C=B0 - c_bytes + 4) == ALIAS
    # alpha == 0: A and B are not read, so no aliasing rule applies
    assert chk(M, N, K, alpha=0.0, C=A0) == OK


def chk_ex(tA, tB, M, N, K, alpha=1.0, A=A0, lda=None, sA=0, B=B0, ldb=None, sB=0, beta=0.0, C=C0, ldc=None,
           sC=0, batch=1):
    lda = max(M if tA else K, 1) if lda is None else lda
    ldb = max(K if tB else N, 1) if ldb is None else ldb
    ldc = max(N, 1) if ldc is None else ldc
    return sgemm.sgemm_check_args_ex(tA, tB, M, N, K, alpha, A, lda, sA, B, ldb, sB, beta, C, ldc, sC, batch)


def test_check_args_ex_leading_dims_follow_the_stored_shape(lib):
    # op(A) = A^T: A is stored K x M, so lda >= M (not K)
    assert chk_ex(1, 0, 4, 5, 6, lda=4) == OK
    assert chk_ex(1, 0, 4, 5, 6, lda=3) == INVALID
    assert chk_ex(0, 0, 4, 5, 6, lda=4) == INVALID
    # op(B) = B^T: B is stored N x K, so ldb >= K
    assert chk_ex(0, 1, 4, 5, 6, ldb=6) == OK
    assert chk_ex(0, 1, 4, 5, 6, ldb=5) == INVALID
    assert chk_ex(1, 1, 4, 5, 6) == OK
    assert chk_ex(2, 0, 4, 5, 6) == INVALID       # trans flags are 0 or 1
    assert chk_ex(0, -1, 4, 5, 6) == INVALID


def test_check_args_ex_batch_rules(lib):
    c_elems = 3 * 5 + 5                              # M=4, N=5, ldc=5: window of 20 cells
    assert chk_ex(0, 0, 4, 5, 6, batch=-1) == INVALID
    assert chk_ex(0, 0, 4, 5, 6, batch=0, A=None, B=None, C=None) == OK
    assert chk_ex(0, 0, 4, 5, 6, batch=2, sA=24, sB=30, sC=c_elems) == OK
    assert chk_ex(0, 0, 4, 5, 6, batch=2, sA=24, sB=30, sC=c_elems - 1) == INVALID   # outputs overlap
    assert chk_ex(0, 0, 4, 5, 6, batch=2, sA=0, sB=0, sC=c_elems) == OK             # shared A and B
    assert chk_ex(0, 0, 4, 5, 6, batch=2, sA=-1, sC=c_elems) == INVALID
    assert chk_ex(0, 0, 4, 5, 6, batch=1, sC=0) == OK                                 # stride unused
    # C of the second batch entry reaching into A's batch window
    assert chk_ex(0, 0, 4, 5, 6, batch=2, sA=24, C=A0 - 4 * c_elems, sC=c_elems) == ALIAS
    assert chk_ex(0, 0, 4, 5, 6, batch=2, sA=24, C=A0 - 8 * c_elems, sC=c_elems) == OK


def test_check_args_is_the_nn_batch1_case(lib):
    for args in [(4, 5, 6), (0, 5, 6), (4, 5, 0), (4, -5, 6)]:
        assert chk(*args) == chk_ex(0, 0, *args)
    assert chk(4, 5, 6, C=A0 + 8) == chk_ex(0, 0, 4, 5, 6, C=A0 + 8) == ALIAS


def chk_mixed(t, tA, tB, M, N, K, alpha=1.0, A=A0, lda=None, B=B0, ldb=None, beta=0.0, C=C0, ldc=None):
    lda = max(M if tA else K, 1) if lda is None else lda
    ldb = max(K if tB else N, 1) if ldb is None else ldb
    ldc = max(N, 1) if ldc is None else ldc
    return sgemm.sgemm_check_args_mixed(t, tA, tB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc)


def test_check_args_mixed(lib):
    for t in (sgemm.IN_BF16, sgemm.IN_F16):
        assert chk_mixed(t, 0, 0, 4, 5, 6) == OK
        assert chk_mixed(t, 1, 1, 4, 5, 6) == OK
        assert chk_mixed(t, 1, 0, 4, 5, 6, lda=3) == INVALID      # A stored K x M: lda >= M
        assert chk_mixed(t, 0, 1, 4, 5, 6, ldb=5) == INVALID      # B stored N x K: ldb >= K
        assert chk_mixed(t, 0, 0, 4, 5, 6, C=None) == NULL_
        assert chk_mixed(t, 0, 0, 4, 5, 6, alpha=0.0, A=None, B=None) == OK
        # 16-bit windows: A = 4 x 6 halves = 48 bytes; C just past it is fine, inside it aliases
        assert chk_mixed(t, 0, 0, 4, 5, 6, C=A0 + 48) == OK
        assert chk_mixed(t, 0, 0, 4, 5, 6, C=A0 + 46) == ALIAS
    assert chk_mixed(0, 0, 0, 4, 5, 6) == INVALID
    assert chk_mixed(3, 0, 0, 4, 5, 6) == INVALID


def test_bad_handles_are_rejected_without_dereference(lib):
    assert lib.sgemm_run(None, 1, 1, 1, 1.0, A0, 1, B0, 1, 0.0, C0, 1, None) == sgemm.ERR_BAD_HANDLE
    assert lib.sgemm_run(ctypes.c_void_p(0x1234), 1, 1, 1, 1.0, A0, 1, B0, 1, 0.0, C0, 1, None) == \
        sgemm.ERR_BAD_HANDLE
    assert lib.sgemm_destroy(None) == sgemm.ERR_BAD_HANDLE
    assert lib.sgemm_destroy(ctypes.c_void_p(0x1234)) == sgemm.ERR_BAD_HANDLE
    assert lib.sgemm_set_variant(None, 1) == sgemm.ERR_BAD_HANDLE
    assert lib.sgemm_last_variant(None, None) == -1
    assert lib.sgemm_get_device_status(None) == sgemm.ERR_BAD_HANDLE
    assert lib.sgemm_create(None) == sgemm.ERR_NULL
    for fake in (None, ctypes.c_void_p(0x1234)):
        assert lib.sgemm_set_math_mode(fake, sgemm.MATH_FP32) == sgemm.ERR_BAD_HANDLE
        assert lib.sgemm_set_relayout(fake, sgemm.RELAYOUT_AUTO) == sgemm.ERR_BAD_HANDLE
        assert lib.sgemm_debug_set_smem_override(fake, 0) == sgemm.ERR_BAD_HANDLE
        assert lib.sgemm_debug_set_stream_k_sums(fake, 0) == sgemm.ERR_BAD_HANDLE
        assert lib.sgemm_debug_set_cluster_split(fake, 0) == sgemm.ERR_BAD_HANDLE
        assert lib.sgemm_debug_set_stream_k_ctas(fake, 0) == sgemm.ERR_BAD_HANDLE
        assert lib.sgemm_debug_set_stream_k_gap(fake, 0) == sgemm.ERR_BAD_HANDLE
        assert lib.sgemm_debug_leave_aborted_state(fake) == sgemm.ERR_BAD_HANDLE
        assert lib.sgemm_debug_tf32_probe(fake, 0, 1, None, None) == sgemm.ERR_BAD_HANDLE
        assert lib.sgemm_debug_set_workspace_limit(fake, 0) == sgemm.ERR_BAD_HANDLE
        assert lib.sgemm_last_launches(fake) == -1
        assert lib.sgemm_last_relayout(fake) == -1
        assert lib.sgemm_relayout_capacity(fake) == -1


def test_create_without_gpu_reports_unsupported(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p(0xdead)
    assert lib.sgemm_create(ctypes.byref(h)) == sgemm.ERR_UNSUPPORTED_DEVICE
    assert h.value is None


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(sgemm, "_lib", None)
    monkeypatch.setattr(build, "LIB", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="missing"):
        sgemm.lib()


def test_marshalling_module_reaches_the_library(lib):
    """The compiled module that marshals sgemm_run / sgemm_run_ex arguments is
    built next to the library and binds the same library instance: a call with
    a handle that was never created comes back from the library as
    SGEMM_ERR_BAD_HANDLE, whatever form the buffers and the stream take (ints,
    objects with data_ptr(), numpy arrays, objects with cuda_stream)."""
    import numpy as np
    torch = pytest.importorskip("torch")
    calls = sgemm.calls_module()
    assert calls is not None, build.calls_build_error

    class Stream:
        cuda_stream = 0

    t = torch.empty(16)
    a = np.empty(16, dtype=np.float32)
    bogus = ctypes.c_void_p(0x1000)
    for buf in (t, a, 0x2000, None):
        assert calls.run(bogus, 8, 8, 8, 1.0, buf, 8, buf, 8, 0.0, t, 8, 0) == sgemm.ERR_BAD_HANDLE
        assert calls.run(0x1000, 8, 8, 8, 1.0, buf, 8, buf, 8, 0.0, t, 8, Stream()) == sgemm.ERR_BAD_HANDLE
        assert calls.run_ex(None, 0, 1, 8, 8, 8, 1.0, buf, 8, 0, buf, 8, 0, 0.0, t, 8, 0, 1, 0) == \
            sgemm.ERR_BAD_HANDLE
    with pytest.raises(sgemm.SgemmError):
        sgemm.sgemm_run(bogus, 8, 8, 8, 1.0, t, 8, t, 8, 0.0, t, 8, 0)
    with pytest.raises(sgemm.SgemmError):
        sgemm.sgemm_run_ex(bogus, 0, 0, 8, 8, 8, 1.0, t, 8, 0, t, 8, 0, 0.0, t, 8, 0, 1, 0)


def test_marshalling_module_rejects_malformed_arguments(lib):
    """Wrong argument counts, values that do not fit a C int and objects that
    are no buffers raise Python exceptions before the library is called."""
    calls = sgemm.calls_module()
    assert calls is not None, build.calls_build_error
    with pytest.raises(TypeError):
        calls.run(None, 8, 8, 8)
    with pytest.raises(TypeError):
        calls.run_ex(None, 0, 0, 8, 8, 8)
    with pytest.raises(OverflowError):
        calls.run(None, 1 << 40, 8, 8, 1.0, 0, 8, 0, 8, 0.0, 0, 8, 0)
    with pytest.raises((TypeError, AttributeError)):
        calls.run(None, 8, 8, 8, 1.0, object(), 8, 0, 8, 0.0, 0, 8, 0)
    with pytest.raises(TypeError):
        calls.run(None, 8, 8, 8, "one", 0, 8, 0, 8, 0.0, 0, 8, 0)
