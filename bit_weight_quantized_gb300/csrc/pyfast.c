/* pyfast.c -- a CPython extension that calls the library's 14-argument
 * matmul entry points (qmm_gemv, qmm_gemm, qmm_gemv_tile16: same signature)
 * through a function address, so that the Python binding's hot calls skip
 * ctypes' per-argument conversion.  It does no arithmetic and no checks
 * beyond argument parsing; the binding falls back to ctypes when this module
 * is not built.  Built by build.py next to libqmm.so. */
#define PY_SSIZE_T_CLEAN
#include <Python.h>
#include <stdint.h>

typedef int (*qmm_call14)(const void *, int, const uint8_t *, int, int, const void *, const uint8_t *,
                          int, void *, int, int, int, int, void *);

static int as_u64(PyObject *o, unsigned long long *v)
{
    if (o == Py_None) {
        *v = 0;
        return 0;
    }
    *v = PyLong_AsUnsignedLongLong(o);
    return (*v == (unsigned long long)-1 && PyErr_Occurred()) ? -1 : 0;
}

static int as_int(PyObject *o, int *v)
{
    long t = PyLong_AsLong(o);
    if (t == -1 && PyErr_Occurred())
        return -1;
    if (t < INT32_MIN || t > INT32_MAX) {
        PyErr_SetString(PyExc_OverflowError, "argument does not fit in a C int");
        return -1;
    }
    *v = (int)t;
    return 0;
}

/* call14(fn, x, x_dtype, packed, bits, group, scales, zeros, zero_const, y,
 *        y_dtype, M, N, K, stream) -> status.  Pointers are ints or None. */
static PyObject *call14(PyObject *self, PyObject *const *args, Py_ssize_t nargs)
{
    (void)self;
    if (nargs != 15) {
        PyErr_SetString(PyExc_TypeError, "call14 takes 15 arguments");
        return NULL;
    }
    unsigned long long fn, x, packed, scales, zeros, y, stream;
    int xdt, bits, group, zc, ydt, M, N, K;
    if (as_u64(args[0], &fn) || as_u64(args[1], &x) || as_int(args[2], &xdt) || as_u64(args[3], &packed) ||
        as_int(args[4], &bits) || as_int(args[5], &group) || as_u64(args[6], &scales) ||
        as_u64(args[7], &zeros) || as_int(args[8], &zc) || as_u64(args[9], &y) || as_int(args[10], &ydt) ||
        as_int(args[11], &M) || as_int(args[12], &N) || as_int(args[13], &K) || as_u64(args[14], &stream))
        return NULL;
    if (!fn) {
        PyErr_SetString(PyExc_ValueError, "null function address");
        return NULL;
    }
    const int st = ((qmm_call14)(uintptr_t)fn)((const void *)(uintptr_t)x, xdt, (const uint8_t *)(uintptr_t)packed,
                                               bits, group, (const void *)(uintptr_t)scales,
                                               (const uint8_t *)(uintptr_t)zeros, zc, (void *)(uintptr_t)y, ydt, M,
                                               N, K, (void *)(uintptr_t)stream);
    return PyLong_FromLong(st);
}

static PyMethodDef methods[] = {
    {"call14", (PyCFunction)(void (*)(void))call14, METH_FASTCALL,
     "call14(fn, x, x_dtype, packed, bits, group, scales, zeros, zero_const, y, y_dtype, M, N, K, stream)"},
    {NULL, NULL, 0, NULL},
};

static struct PyModuleDef module = {PyModuleDef_HEAD_INIT, "_qmmfast", NULL, -1, methods,
                                    NULL, NULL, NULL, NULL};

PyMODINIT_FUNC PyInit__qmmfast(void) { return PyModule_Create(&module); }
