/*
 * Argument marshalling for the two enqueue calls of the Python binding
 * (sgemm_run, sgemm_run_ex) through the CPython C API.  The binding's other
 * calls go through ctypes; these two are on the per-call path, where
 * ctypes' generic conversion of a dozen arguments costs a few microseconds
 * -- as much as a small GEMM takes on the GPU.  Nothing here computes: each
 * function converts Python ints, floats, buffers (ints or objects with a
 * data_ptr() method, such as torch tensors) and streams (ints, objects with
 * a cuda_stream attribute, or None for the caller's current stream) into C
 * values and calls the C ABI function of the library that the binding
 * loaded, found with dlopen / dlsym on the same path.  Built with the host
 * compiler next to the library; the binding uses ctypes when it is absent.
 */
#define PY_SSIZE_T_CLEAN
#include <Python.h>

#include <dlfcn.h>
#include <limits.h>

typedef int (*run_fn)(void *, int, int, int, float, const float *, int, const float *, int, float, float *, int,
                      void *);
typedef int (*run_ex_fn)(void *, int, int, int, int, int, float, const float *, int, long long, const float *, int,
                         long long, float, float *, int, long long, int, void *);

static run_fn g_run = NULL;
static run_ex_fn g_run_ex = NULL;
static PyObject *g_current_stream = NULL; /* callable returning the current stream as an int */
static PyObject *g_data_ptr = NULL, *g_cuda_stream = NULL, *g_value = NULL, *g_array_interface = NULL;

static int as_int(PyObject *o, int *out) {
    const long v = PyLong_AsLong(o);
    if (v == -1 && PyErr_Occurred()) return -1;
    if (v < INT_MIN || v > INT_MAX) {
        PyErr_SetString(PyExc_OverflowError, "argument does not fit in a C int");
        return -1;
    }
    *out = (int)v;
    return 0;
}

static int as_ll(PyObject *o, long long *out) {
    const long long v = PyLong_AsLongLong(o);
    if (v == -1 && PyErr_Occurred()) return -1;
    *out = v;
    return 0;
}

static int as_float(PyObject *o, float *out) {
    const double v = PyFloat_AsDouble(o);
    if (v == -1.0 && PyErr_Occurred()) return -1;
    *out = (float)v;
    return 0;
}

/* An address: None, an int, an object with data_ptr() (torch tensors), or an
 * object with the array interface (numpy arrays). */
static int as_ptr(PyObject *o, void **out) {
    if (o == Py_None) {
        *out = NULL;
        return 0;
    }
    if (PyLong_Check(o)) {
        *out = PyLong_AsVoidPtr(o);
        return PyErr_Occurred() ? -1 : 0;
    }
    PyObject *r = PyObject_CallMethodNoArgs(o, g_data_ptr);
    if (r == NULL) {
        if (!PyErr_ExceptionMatches(PyExc_AttributeError)) return -1;
        PyErr_Clear();
        PyObject *ai = PyObject_GetAttr(o, g_array_interface);
        if (ai == NULL) return -1;
        PyObject *data = PyDict_Check(ai) ? PyDict_GetItemString(ai, "data") : NULL; /* borrowed */
        PyObject *addr = (data != NULL && PyTuple_Check(data) && PyTuple_GET_SIZE(data) > 0)
                             ? PyTuple_GET_ITEM(data, 0) : NULL;                     /* borrowed */
        if (addr == NULL) {
            Py_DECREF(ai);
            PyErr_SetString(PyExc_TypeError, "not a buffer address");
            return -1;
        }
        *out = PyLong_AsVoidPtr(addr);
        Py_DECREF(ai);
        return PyErr_Occurred() ? -1 : 0;
    }
    *out = PyLong_AsVoidPtr(r);
    Py_DECREF(r);
    return PyErr_Occurred() ? -1 : 0;
}

/* The handle: a ctypes.c_void_p (its value), an int or None. */
static int as_handle(PyObject *o, void **out) {
    if (o == Py_None || PyLong_Check(o)) return as_ptr(o, out);
    PyObject *v = PyObject_GetAttr(o, g_value);
    if (v == NULL) return -1;
    const int rc = as_ptr(v, out);
    Py_DECREF(v);
    return rc;
}

/* The stream: an int, an object with cuda_stream, or None (the current one). */
static int as_stream(PyObject *o, void **out) {
    if (PyLong_Check(o)) return as_ptr(o, out);
    PyObject *s = (o == Py_None) ? PyObject_CallNoArgs(g_current_stream) : PyObject_GetAttr(o, g_cuda_stream);
    if (s == NULL) return -1;
    const int rc = as_ptr(s, out);
    Py_DECREF(s);
    return rc;
}

/* init(library_path, current_stream): bind the C ABI functions of the loaded library. */
static PyObject *py_init(PyObject *self, PyObject *args) {
    (void)self;
    const char *path;
    PyObject *cur;
    if (!PyArg_ParseTuple(args, "sO", &path, &cur)) return NULL;
    void *lib = dlopen(path, RTLD_NOW);
    if (lib == NULL) {
        PyErr_Format(PyExc_OSError, "dlopen(%s) failed: %s", path, dlerror());
        return NULL;
    }
    g_run = (run_fn)dlsym(lib, "sgemm_run");
    g_run_ex = (run_ex_fn)dlsym(lib, "sgemm_run_ex");
    if (g_run == NULL || g_run_ex == NULL) {
        PyErr_SetString(PyExc_OSError, "the library exports no sgemm_run / sgemm_run_ex");
        return NULL;
    }
    Py_XDECREF(g_current_stream);
    Py_INCREF(cur);
    g_current_stream = cur;
    Py_RETURN_NONE;
}

/* run(h, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream) -> status */
static PyObject *py_run(PyObject *self, PyObject *const *a, Py_ssize_t n) {
    (void)self;
    if (n != 13) {
        PyErr_SetString(PyExc_TypeError, "run takes 13 arguments");
        return NULL;
    }
    if (g_run == NULL) {
        PyErr_SetString(PyExc_RuntimeError, "init was not called");
        return NULL;
    }
    void *h, *A, *B, *C, *stream;
    int M, N, K, lda, ldb, ldc;
    float alpha, beta;
    if (as_handle(a[0], &h) || as_int(a[1], &M) || as_int(a[2], &N) || as_int(a[3], &K) ||
        as_float(a[4], &alpha) || as_ptr(a[5], &A) || as_int(a[6], &lda) || as_ptr(a[7], &B) ||
        as_int(a[8], &ldb) || as_float(a[9], &beta) || as_ptr(a[10], &C) || as_int(a[11], &ldc) ||
        as_stream(a[12], &stream))
        return NULL;
    return PyLong_FromLong(g_run(h, M, N, K, alpha, (const float *)A, lda, (const float *)B, ldb, beta, (float *)C,
                                 ldc, stream));
}

/* run_ex(h, transA, transB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB,
 *        beta, C, ldc, strideC, batch, stream) -> status */
static PyObject *py_run_ex(PyObject *self, PyObject *const *a, Py_ssize_t n) {
    (void)self;
    if (n != 19) {
        PyErr_SetString(PyExc_TypeError, "run_ex takes 19 arguments");
        return NULL;
    }
    if (g_run_ex == NULL) {
        PyErr_SetString(PyExc_RuntimeError, "init was not called");
        return NULL;
    }
    void *h, *A, *B, *C, *stream;
    int tA, tB, M, N, K, lda, ldb, ldc, batch;
    long long sA, sB, sC;
    float alpha, beta;
    if (as_handle(a[0], &h) || as_int(a[1], &tA) || as_int(a[2], &tB) || as_int(a[3], &M) || as_int(a[4], &N) ||
        as_int(a[5], &K) || as_float(a[6], &alpha) || as_ptr(a[7], &A) || as_int(a[8], &lda) ||
        as_ll(a[9], &sA) || as_ptr(a[10], &B) || as_int(a[11], &ldb) || as_ll(a[12], &sB) ||
        as_float(a[13], &beta) || as_ptr(a[14], &C) || as_int(a[15], &ldc) || as_ll(a[16], &sC) ||
        as_int(a[17], &batch) || as_stream(a[18], &stream))
        return NULL;
    return PyLong_FromLong(g_run_ex(h, tA, tB, M, N, K, alpha, (const float *)A, lda, sA, (const float *)B, ldb, sB,
                                    beta, (float *)C, ldc, sC, batch, stream));
}

static PyMethodDef kMethods[] = {
    {"init", py_init, METH_VARARGS, "init(library_path, current_stream): bind the library's enqueue calls"},
    {"run", (PyCFunction)(void (*)(void))py_run, METH_FASTCALL, "sgemm_run through the C ABI; returns the status"},
    {"run_ex", (PyCFunction)(void (*)(void))py_run_ex, METH_FASTCALL,
     "sgemm_run_ex through the C ABI; returns the status"},
    {NULL, NULL, 0, NULL}};

static struct PyModuleDef kModule = {PyModuleDef_HEAD_INIT, "_sgemm_calls", NULL, -1, kMethods, NULL, NULL, NULL,
                                     NULL};

PyMODINIT_FUNC PyInit__sgemm_calls(void) {
    g_data_ptr = PyUnicode_InternFromString("data_ptr");
    g_cuda_stream = PyUnicode_InternFromString("cuda_stream");
    g_value = PyUnicode_InternFromString("value");
    g_array_interface = PyUnicode_InternFromString("__array_interface__");
    if (g_data_ptr == NULL || g_cuda_stream == NULL || g_value == NULL || g_array_interface == NULL) return NULL;
    return PyModule_Create(&kModule);
}
