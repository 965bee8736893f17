/* A CPython extension that forwards the product entry points of the C-ABI
 * (sbgemm, sbgemm_ex) with their arguments converted straight from Python
 * objects.  Argument marshalling only: the functions it calls are the
 * library's own, whose addresses the Python binding hands over once with
 * bind(), so the library instance is the one the binding loaded.
 *
 * Why: a ctypes call converts each of the twenty arguments through its
 * argtypes, which measured about 2.5 us per call on an Arm server core,
 * more than the library's whole host side (checks, plan, launch: 2 us); a
 * latency-bound product such as a 64 x 48 x 32 one pays that on every
 * launch.  Here the conversion is one PyLong_AsLongLong / PyFloat_AsDouble
 * per argument.
 *
 * Pointers are Python ints (0 or None for NULL), strides and sizes ints (or
 * objects with __index__), alpha a float.  Each call returns the library's
 * status as an int; a bad argument type raises TypeError or OverflowError. */
#define PY_SSIZE_T_CLEAN
#include <Python.h>
#include <stdint.h>

#include "sbgemm.h"

typedef int (*ex_fn)(const float*, int64_t, int64_t, int64_t, const float*, int64_t, int64_t, int64_t,
                     float*, int64_t, int64_t, int64_t, int64_t, int64_t, int64_t, int64_t, float, int,
                     void*, const sbgemm_options*);
typedef int (*plain_fn)(const float*, int64_t, int64_t, int64_t, const float*, int64_t, int64_t, int64_t,
                        float*, int64_t, int64_t, int64_t, int64_t, int64_t, int64_t, int64_t, float, int,
                        void*);

static ex_fn g_ex = NULL;
static plain_fn g_plain = NULL;

static int as_ptr(PyObject* o, void** out) {
    if (o == Py_None) {
        *out = NULL;
        return 1;
    }
    *out = PyLong_AsVoidPtr(o);
    return !(*out == NULL && PyErr_Occurred());
}

static int as_i64(PyObject* o, int64_t* out) {
    const long long v = PyLong_AsLongLong(o);
    if (v == -1 && PyErr_Occurred()) return 0;
    *out = (int64_t)v;
    return 1;
}

/* The twelve operand arguments and the four sizes shared by both calls. */
typedef struct {
    void *A, *B, *C;
    int64_t s[9];
    int64_t M, N, K, batch;
    float alpha;
    int accumulate;
    void* stream;
} Call;

static int parse_common(PyObject* const* args, Call* c) {
    void** ptr[3] = {&c->A, &c->B, &c->C};
    for (int op = 0; op < 3; ++op) {
        if (!as_ptr(args[4 * op], ptr[op])) return 0;
        for (int k = 0; k < 3; ++k)
            if (!as_i64(args[4 * op + 1 + k], &c->s[3 * op + k])) return 0;
    }
    if (!as_i64(args[12], &c->M) || !as_i64(args[13], &c->N) || !as_i64(args[14], &c->K) ||
        !as_i64(args[15], &c->batch))
        return 0;
    const double alpha = PyFloat_AsDouble(args[16]);
    if (alpha == -1.0 && PyErr_Occurred()) return 0;
    c->alpha = (float)alpha;
    const int acc = PyObject_IsTrue(args[17]);
    if (acc < 0) return 0;
    c->accumulate = acc;
    return as_ptr(args[18], &c->stream);
}

static PyObject* fc_bind(PyObject* self, PyObject* const* args, Py_ssize_t nargs) {
    (void)self;
    if (nargs != 2) {
        PyErr_SetString(PyExc_TypeError, "bind(sbgemm_ex address, sbgemm address)");
        return NULL;
    }
    void *ex = NULL, *plain = NULL;
    if (!as_ptr(args[0], &ex) || !as_ptr(args[1], &plain)) return NULL;
    g_ex = (ex_fn)ex;
    g_plain = (plain_fn)plain;
    Py_RETURN_NONE;
}

/* sbgemm_ex(A, rsA, csA, bsA, B, rsB, csB, bsB, C, rsC, csC, bsC, M, N, K,
 *           batch, alpha, accumulate, stream, options address) -> status */
static PyObject* fc_sbgemm_ex(PyObject* self, PyObject* const* args, Py_ssize_t nargs) {
    (void)self;
    if (nargs != 20) {
        PyErr_SetString(PyExc_TypeError, "sbgemm_ex takes 20 arguments");
        return NULL;
    }
    if (!g_ex) {
        PyErr_SetString(PyExc_RuntimeError, "the library is not bound");
        return NULL;
    }
    Call c;
    void* opt = NULL;
    if (!parse_common(args, &c) || !as_ptr(args[19], &opt)) return NULL;
    int st;
    Py_BEGIN_ALLOW_THREADS
    st = g_ex((const float*)c.A, c.s[0], c.s[1], c.s[2], (const float*)c.B, c.s[3], c.s[4], c.s[5],
              (float*)c.C, c.s[6], c.s[7], c.s[8], c.M, c.N, c.K, c.batch, c.alpha, c.accumulate,
              c.stream, (const sbgemm_options*)opt);
    Py_END_ALLOW_THREADS
    return PyLong_FromLong(st);
}

/* sbgemm(A, rsA, csA, bsA, B, rsB, csB, bsB, C, rsC, csC, bsC, M, N, K,
 *        batch, alpha, accumulate, stream) -> status */
static PyObject* fc_sbgemm(PyObject* self, PyObject* const* args, Py_ssize_t nargs) {
    (void)self;
    if (nargs != 19) {
        PyErr_SetString(PyExc_TypeError, "sbgemm takes 19 arguments");
        return NULL;
    }
    if (!g_plain) {
        PyErr_SetString(PyExc_RuntimeError, "the library is not bound");
        return NULL;
    }
    Call c;
    if (!parse_common(args, &c)) return NULL;
    int st;
    Py_BEGIN_ALLOW_THREADS
    st = g_plain((const float*)c.A, c.s[0], c.s[1], c.s[2], (const float*)c.B, c.s[3], c.s[4], c.s[5],
                 (float*)c.C, c.s[6], c.s[7], c.s[8], c.M, c.N, c.K, c.batch, c.alpha, c.accumulate,
                 c.stream);
    Py_END_ALLOW_THREADS
    return PyLong_FromLong(st);
}

static PyMethodDef kMethods[] = {
    {"bind", (PyCFunction)(void (*)(void))fc_bind, METH_FASTCALL, "bind the library's entry points"},
    {"sbgemm_ex", (PyCFunction)(void (*)(void))fc_sbgemm_ex, METH_FASTCALL, "sbgemm_ex; returns the status"},
    {"sbgemm", (PyCFunction)(void (*)(void))fc_sbgemm, METH_FASTCALL, "sbgemm; returns the status"},
    {NULL, NULL, 0, NULL},
};

static struct PyModuleDef kModule = {PyModuleDef_HEAD_INIT, "_fastcall", NULL, -1, kMethods,
                                     NULL, NULL, NULL, NULL};

PyMODINIT_FUNC PyInit__fastcall(void) { return PyModule_Create(&kModule); }
