/*
 * Argument marshalling for the compute entry points of libsgemm_gb300.so,
 * as a CPython extension: each function parses its Python ints and floats
 * with one PyArg_ParseTuple and calls the C ABI through a pointer that the
 * package hands over from the library it loaded (bind), so both routes reach
 * the same library instance.  ctypes spends about 0.2 us per argument on the
 * same conversions; these calls take a fraction of a microsecond.  Nothing
 * here computes: every step of the product runs in the library's kernels.
 * Pointers and streams arrive as unsigned integers (0 = null).
 */
#define PY_SSIZE_T_CLEAN
#include <Python.h>
#include <stdint.h>

#include "sgemm_gb300.h"

#define P(x) ((void *)(uintptr_t)(x))

static __typeof__(&sgemm_f32) f_sgemm_f32;
static __typeof__(&sgemm_f32_strided_batched) f_sgemm_f32_strided_batched;
static __typeof__(&sgemm_f32_ex) f_sgemm_f32_ex;
static __typeof__(&sgemm_f32_ex_strided_batched) f_sgemm_f32_ex_strided_batched;
static __typeof__(&sgemm_f32_tf32x3_ex) f_sgemm_f32_tf32x3_ex;
static __typeof__(&sgemm_f32_splitk) f_sgemm_f32_splitk;
static __typeof__(&sgemm_f32_streamk) f_sgemm_f32_streamk;
static __typeof__(&sgemm_f32_tf32x3) f_sgemm_f32_tf32x3;
static __typeof__(&sgemm_f32_tf32x3_strided_batched) f_sgemm_f32_tf32x3_strided_batched;
static __typeof__(&sgemm_f32_tf32) f_sgemm_f32_tf32;
static __typeof__(&sgemm_f32_tf32_strided_batched) f_sgemm_f32_tf32_strided_batched;
static __typeof__(&sgemm_f32_tf32x3_noalloc) f_sgemm_f32_tf32x3_noalloc;

/* Not bound yet: raise instead of calling a null pointer. */
static int unbound(const void *fn) {
    if (fn != NULL) return 0;
    PyErr_SetString(PyExc_RuntimeError, "_calls.bind() has not been called");
    return 1;
}

/* M, N, K, A, lda, B, ldb, C, ldc, transA, transB, stream */
static PyObject *py_sgemm_f32(PyObject *self, PyObject *args) {
    long long M, N, K, lda, ldb, ldc;
    unsigned long long A, B, C, s;
    int tA, tB;
    (void)self;
    if (unbound((const void *)f_sgemm_f32)) return NULL;
    if (!PyArg_ParseTuple(args, "LLLKLKLKLiiK", &M, &N, &K, &A, &lda, &B, &ldb, &C, &ldc, &tA,
                          &tB, &s))
        return NULL;
    return PyLong_FromLong(f_sgemm_f32(M, N, K, P(A), lda, P(B), ldb, P(C), ldc, tA, tB, P(s)));
}

/* M, N, K, A, lda, strideA, B, ldb, strideB, C, ldc, strideC, batch, transA,
 * transB, stream */
static PyObject *py_sgemm_f32_strided_batched(PyObject *self, PyObject *args) {
    long long M, N, K, lda, sA, ldb, sB, ldc, sC, batch;
    unsigned long long A, B, C, s;
    int tA, tB;
    (void)self;
    if (unbound((const void *)f_sgemm_f32_strided_batched)) return NULL;
    if (!PyArg_ParseTuple(args, "LLLKLLKLLKLLLiiK", &M, &N, &K, &A, &lda, &sA, &B, &ldb, &sB, &C,
                          &ldc, &sC, &batch, &tA, &tB, &s))
        return NULL;
    return PyLong_FromLong(f_sgemm_f32_strided_batched(M, N, K, P(A), lda, sA, P(B), ldb, sB, P(C),
                                                       ldc, sC, batch, tA, tB, P(s)));
}

/* M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bias, transA, transB, stream */
static PyObject *py_sgemm_f32_ex(PyObject *self, PyObject *args) {
    long long M, N, K, lda, ldb, ldc;
    unsigned long long A, B, C, bias, s;
    float alpha, beta;
    int tA, tB;
    (void)self;
    if (unbound((const void *)f_sgemm_f32_ex)) return NULL;
    if (!PyArg_ParseTuple(args, "LLLfKLKLfKLKiiK", &M, &N, &K, &alpha, &A, &lda, &B, &ldb, &beta,
                          &C, &ldc, &bias, &tA, &tB, &s))
        return NULL;
    return PyLong_FromLong(f_sgemm_f32_ex(M, N, K, alpha, P(A), lda, P(B), ldb, beta, P(C), ldc,
                                          P(bias), tA, tB, P(s)));
}

/* M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc, strideC,
 * bias, batch, transA, transB, stream */
static PyObject *py_sgemm_f32_ex_strided_batched(PyObject *self, PyObject *args) {
    long long M, N, K, lda, sA, ldb, sB, ldc, sC, batch;
    unsigned long long A, B, C, bias, s;
    float alpha, beta;
    int tA, tB;
    (void)self;
    if (unbound((const void *)f_sgemm_f32_ex_strided_batched)) return NULL;
    if (!PyArg_ParseTuple(args, "LLLfKLLKLLfKLLKLiiK", &M, &N, &K, &alpha, &A, &lda, &sA, &B, &ldb,
                          &sB, &beta, &C, &ldc, &sC, &bias, &batch, &tA, &tB, &s))
        return NULL;
    return PyLong_FromLong(f_sgemm_f32_ex_strided_batched(M, N, K, alpha, P(A), lda, sA, P(B), ldb,
                                                          sB, beta, P(C), ldc, sC, P(bias), batch,
                                                          tA, tB, P(s)));
}

/* M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bias, transA, transB,
 * workspace, workspace_bytes, stream */
static PyObject *py_sgemm_f32_tf32x3_ex(PyObject *self, PyObject *args) {
    long long M, N, K, lda, ldb, ldc;
    unsigned long long A, B, C, bias, ws, wsb, s;
    float alpha, beta;
    int tA, tB;
    (void)self;
    if (unbound((const void *)f_sgemm_f32_tf32x3_ex)) return NULL;
    if (!PyArg_ParseTuple(args, "LLLfKLKLfKLKiiKKK", &M, &N, &K, &alpha, &A, &lda, &B, &ldb, &beta,
                          &C, &ldc, &bias, &tA, &tB, &ws, &wsb, &s))
        return NULL;
    return PyLong_FromLong(f_sgemm_f32_tf32x3_ex(M, N, K, alpha, P(A), lda, P(B), ldb, beta, P(C),
                                                 ldc, P(bias), tA, tB, P(ws), (uint64_t)wsb,
                                                 P(s)));
}

/* M, N, K, A, lda, B, ldb, C, ldc, transA, transB, splits, workspace,
 * workspace_bytes, stream */
static PyObject *py_sgemm_f32_splitk(PyObject *self, PyObject *args) {
    long long M, N, K, lda, ldb, ldc;
    unsigned long long A, B, C, ws, wsb, s;
    int tA, tB, splits;
    (void)self;
    if (unbound((const void *)f_sgemm_f32_splitk)) return NULL;
    if (!PyArg_ParseTuple(args, "LLLKLKLKLiiiKKK", &M, &N, &K, &A, &lda, &B, &ldb, &C, &ldc, &tA,
                          &tB, &splits, &ws, &wsb, &s))
        return NULL;
    return PyLong_FromLong(f_sgemm_f32_splitk(M, N, K, P(A), lda, P(B), ldb, P(C), ldc, tA, tB,
                                              splits, P(ws), (uint64_t)wsb, P(s)));
}

/* The entries shaped M, N, K, A, lda, B, ldb, C, ldc, transA, transB,
 * workspace, workspace_bytes, stream: sgemm_f32_streamk, sgemm_f32_tf32x3,
 * sgemm_f32_tf32. */
#define WS_ENTRY(name)                                                                          \
    static PyObject *py_##name(PyObject *self, PyObject *args) {                               \
        long long M, N, K, lda, ldb, ldc;                                                      \
        unsigned long long A, B, C, ws, wsb, s;                                                \
        int tA, tB;                                                                            \
        (void)self;                                                                            \
        if (unbound((const void *)f_##name)) return NULL;                                      \
        if (!PyArg_ParseTuple(args, "LLLKLKLKLiiKKK", &M, &N, &K, &A, &lda, &B, &ldb, &C,      \
                              &ldc, &tA, &tB, &ws, &wsb, &s))                                   \
            return NULL;                                                                       \
        return PyLong_FromLong(f_##name(M, N, K, P(A), lda, P(B), ldb, P(C), ldc, tA, tB,      \
                                        P(ws), (uint64_t)wsb, P(s)));                          \
    }
WS_ENTRY(sgemm_f32_streamk)
WS_ENTRY(sgemm_f32_tf32x3)
WS_ENTRY(sgemm_f32_tf32)

/* The strided-batched tensor entries: M, N, K, A, lda, strideA, B, ldb,
 * strideB, C, ldc, strideC, batch, transA, transB, workspace,
 * workspace_bytes, stream. */
#define WS_BATCHED_ENTRY(name)                                                                  \
    static PyObject *py_##name(PyObject *self, PyObject *args) {                               \
        long long M, N, K, lda, sA, ldb, sB, ldc, sC, batch;                                   \
        unsigned long long A, B, C, ws, wsb, s;                                                \
        int tA, tB;                                                                            \
        (void)self;                                                                            \
        if (unbound((const void *)f_##name)) return NULL;                                      \
        if (!PyArg_ParseTuple(args, "LLLKLLKLLKLLLiiKKK", &M, &N, &K, &A, &lda, &sA, &B, &ldb, \
                              &sB, &C, &ldc, &sC, &batch, &tA, &tB, &ws, &wsb, &s))           \
            return NULL;                                                                       \
        return PyLong_FromLong(f_##name(M, N, K, P(A), lda, sA, P(B), ldb, sB, P(C), ldc, sC,  \
                                        batch, tA, tB, P(ws), (uint64_t)wsb, P(s)));           \
    }
WS_BATCHED_ENTRY(sgemm_f32_tf32x3_strided_batched)
WS_BATCHED_ENTRY(sgemm_f32_tf32_strided_batched)

/* M, N, K, A, lda, B, ldb, C, ldc, transA, transB, stream */
static PyObject *py_sgemm_f32_tf32x3_noalloc(PyObject *self, PyObject *args) {
    long long M, N, K, lda, ldb, ldc;
    unsigned long long A, B, C, s;
    int tA, tB;
    (void)self;
    if (unbound((const void *)f_sgemm_f32_tf32x3_noalloc)) return NULL;
    if (!PyArg_ParseTuple(args, "LLLKLKLKLiiK", &M, &N, &K, &A, &lda, &B, &ldb, &C, &ldc, &tA,
                          &tB, &s))
        return NULL;
    return PyLong_FromLong(f_sgemm_f32_tf32x3_noalloc(M, N, K, P(A), lda, P(B), ldb, P(C), ldc, tA,
                                                      tB, P(s)));
}

/* bind({name: address}): the entry points' addresses in the loaded library.
 * Every name above must be present. */
static PyObject *py_bind(PyObject *self, PyObject *args) {
    PyObject *table;
    (void)self;
    if (!PyArg_ParseTuple(args, "O!", &PyDict_Type, &table)) return NULL;
#define BIND(name)                                                                              \
    do {                                                                                       \
        PyObject *v = PyDict_GetItemString(table, #name);                                      \
        if (v == NULL) {                                                                       \
            PyErr_SetString(PyExc_KeyError, #name);                                            \
            return NULL;                                                                       \
        }                                                                                      \
        unsigned long long a = PyLong_AsUnsignedLongLong(v);                                   \
        if (PyErr_Occurred()) return NULL;                                                     \
        f_##name = (__typeof__(f_##name))(uintptr_t)a;                                         \
    } while (0)
    BIND(sgemm_f32);
    BIND(sgemm_f32_strided_batched);
    BIND(sgemm_f32_ex);
    BIND(sgemm_f32_ex_strided_batched);
    BIND(sgemm_f32_tf32x3_ex);
    BIND(sgemm_f32_splitk);
    BIND(sgemm_f32_streamk);
    BIND(sgemm_f32_tf32x3);
    BIND(sgemm_f32_tf32x3_strided_batched);
    BIND(sgemm_f32_tf32);
    BIND(sgemm_f32_tf32_strided_batched);
    BIND(sgemm_f32_tf32x3_noalloc);
#undef BIND
    Py_RETURN_NONE;
}

#define ENTRY(name) {#name, py_##name, METH_VARARGS, NULL}
static PyMethodDef methods[] = {
    {"bind", py_bind, METH_VARARGS, "bind({name: address}) of the loaded library's entry points"},
    ENTRY(sgemm_f32),
    ENTRY(sgemm_f32_strided_batched),
    ENTRY(sgemm_f32_ex),
    ENTRY(sgemm_f32_ex_strided_batched),
    ENTRY(sgemm_f32_tf32x3_ex),
    ENTRY(sgemm_f32_splitk),
    ENTRY(sgemm_f32_streamk),
    ENTRY(sgemm_f32_tf32x3),
    ENTRY(sgemm_f32_tf32x3_strided_batched),
    ENTRY(sgemm_f32_tf32),
    ENTRY(sgemm_f32_tf32_strided_batched),
    ENTRY(sgemm_f32_tf32x3_noalloc),
    {NULL, NULL, 0, NULL},
};

static struct PyModuleDef module = {PyModuleDef_HEAD_INIT, "_calls",
                                    "Argument marshalling for libsgemm_gb300.so", -1, methods};

PyMODINIT_FUNC PyInit__calls(void) { return PyModule_Create(&module); }
