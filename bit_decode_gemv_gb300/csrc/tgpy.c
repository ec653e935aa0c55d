/* tgpy.c -- a CPython call path to tg_gemv_i8 for the eager per-token loop.
 *
 * The Python binding marshals arguments through ctypes; for the one call a
 * decode loop makes per weight matrix and token, ctypes' per-argument
 * conversion is a large part of the host cost. This module takes the same
 * six arguments as plain integers (addresses of the layout, the weights, x
 * and y; M; the stream handle) and calls the library function directly.
 * It links against the in-tree libtg.so (rpath $ORIGIN), so it shares the
 * library's state with the ctypes path. It is optional: without it the
 * binding uses ctypes.
 */
#define PY_SSIZE_T_CLEAN
#include <Python.h>
#include <stdint.h>

#include "tg.h"

static PyObject *py_gemv_i8(PyObject *self, PyObject *const *args, Py_ssize_t nargs)
{
    (void)self;
    if (nargs != 6) {
        PyErr_SetString(PyExc_TypeError, "gemv_i8(layout, w, x, M, y, stream) takes 6 integer arguments");
        return NULL;
    }
    unsigned long long addr[6];
    long long m = 0;
    for (Py_ssize_t i = 0; i < 6; i++) {
        if (i == 3) {
            m = PyLong_AsLongLong(args[i]);
        } else {
            addr[i] = PyLong_AsUnsignedLongLong(args[i]);
        }
        if (PyErr_Occurred())
            return NULL;
    }
    const int r = tg_gemv_i8((const tg_layout *)(uintptr_t)addr[0], (const void *)(uintptr_t)addr[1],
                             (const int8_t *)(uintptr_t)addr[2], (int64_t)m, (int64_t *)(uintptr_t)addr[4],
                             (void *)(uintptr_t)addr[5]);
    return PyLong_FromLong(r);
}

static PyMethodDef tgpy_methods[] = {
    {"gemv_i8", (PyCFunction)(void (*)(void))py_gemv_i8, METH_FASTCALL,
     "tg_gemv_i8 with every argument an integer (addresses, M, stream); returns the tg_status."},
    {NULL, NULL, 0, NULL},
};

static struct PyModuleDef tgpy_module = {PyModuleDef_HEAD_INIT, "_tgpy", NULL, -1, tgpy_methods,
                                         NULL, NULL, NULL, NULL};

PyMODINIT_FUNC PyInit__tgpy(void) { return PyModule_Create(&tgpy_module); }
