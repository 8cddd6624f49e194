/*
 * _fastcall: a minimal CPython extension that calls moe_finalize_ex of the
 * loaded libmoe_finalize.so.  ctypes converts each of the call's twenty
 * arguments through its generic machinery on every call, which costs more
 * host time than the decode-size kernel takes on the GPU.  Here call_now
 * converts them directly, and pack/call go further for repeated calls: the
 * arguments are packed once into a C struct (a capsule) and each call passes
 * only the stream.  It does no computation and no checking beyond what the
 * C ABI itself does.
 */
#define PY_SSIZE_T_CLEAN
#include <Python.h>
#include <stdint.h>
#include <stdlib.h>

typedef int (*finalize_ex_fn)(const void *permuted_out, int64_t P, const int32_t *idx_map,
                              const void *weights, int wkind, float routed_scale,
                              const void *shared_out, const void *residual, const void *gamma,
                              float eps, void *out, void *residual_out, void *norm_out, int T,
                              int K, int H, int splits_hint, int threads_hint, unsigned flags,
                              void *stream);

typedef struct {
    finalize_ex_fn fn;
    const void *permuted_out;
    int64_t P;
    const int32_t *idx_map;
    const void *weights;
    int wkind;
    float routed_scale;
    const void *shared_out, *residual, *gamma;
    float eps;
    void *out, *residual_out, *norm_out;
    int T, K, H, splits, threads;
    unsigned flags;
} bound_call;

static const char *kCapsule = "moe_finalize_bound_call";

static void free_bound(PyObject *cap) {
    free(PyCapsule_GetPointer(cap, kCapsule));
}

static void *as_ptr(PyObject *o) {
    return o == Py_None ? NULL : PyLong_AsVoidPtr(o);
}

/* Converts the twenty positional arguments (fn_address, permuted_out, P,
 * idx_map, weights, wkind, routed_scale, shared_out, residual, gamma, eps,
 * out, residual_out, norm_out, T, K, H, splits, threads, flags) into `b`.
 * Pointers are ints (or None), as tensor.data_ptr() gives them.  Returns 0,
 * or -1 with a Python error set. */
static int parse_call(PyObject *const *a, bound_call *b) {
    b->fn = (finalize_ex_fn)as_ptr(a[0]);
    b->permuted_out = as_ptr(a[1]);
    b->P = (int64_t)PyLong_AsLongLong(a[2]);
    b->idx_map = (const int32_t *)as_ptr(a[3]);
    b->weights = as_ptr(a[4]);
    b->wkind = (int)PyLong_AsLong(a[5]);
    b->routed_scale = (float)PyFloat_AsDouble(a[6]);
    b->shared_out = as_ptr(a[7]);
    b->residual = as_ptr(a[8]);
    b->gamma = as_ptr(a[9]);
    b->eps = (float)PyFloat_AsDouble(a[10]);
    b->out = as_ptr(a[11]);
    b->residual_out = as_ptr(a[12]);
    b->norm_out = as_ptr(a[13]);
    b->T = (int)PyLong_AsLong(a[14]);
    b->K = (int)PyLong_AsLong(a[15]);
    b->H = (int)PyLong_AsLong(a[16]);
    b->splits = (int)PyLong_AsLong(a[17]);
    b->threads = (int)PyLong_AsLong(a[18]);
    b->flags = (unsigned)PyLong_AsUnsignedLong(a[19]);
    if (PyErr_Occurred()) return -1;
    if (!b->fn) {
        PyErr_SetString(PyExc_ValueError, "null function pointer");
        return -1;
    }
    return 0;
}

static int enqueue(const bound_call *b, void *stream) {
    return b->fn(b->permuted_out, b->P, b->idx_map, b->weights, b->wkind, b->routed_scale,
                 b->shared_out, b->residual, b->gamma, b->eps, b->out, b->residual_out,
                 b->norm_out, b->T, b->K, b->H, b->splits, b->threads, b->flags, stream);
}

/* pack(<the twenty arguments>) -> capsule holding them */
static PyObject *pack(PyObject *self, PyObject *const *args, Py_ssize_t nargs) {
    (void)self;
    if (nargs != 20) {
        PyErr_SetString(PyExc_TypeError, "pack takes 20 arguments");
        return NULL;
    }
    bound_call *b = (bound_call *)calloc(1, sizeof(bound_call));
    if (!b) return PyErr_NoMemory();
    if (parse_call(args, b) != 0) {
        free(b);
        return NULL;
    }
    return PyCapsule_New(b, kCapsule, free_bound);
}

/* call_now(<the twenty arguments>, stream_handle) -> status of one
 * moe_finalize_ex call, with nothing kept */
static PyObject *call_now(PyObject *self, PyObject *const *args, Py_ssize_t nargs) {
    (void)self;
    if (nargs != 21) {
        PyErr_SetString(PyExc_TypeError, "call_now takes 21 arguments");
        return NULL;
    }
    bound_call b;
    if (parse_call(args, &b) != 0) return NULL;
    void *stream = as_ptr(args[20]);
    if (PyErr_Occurred()) return NULL;
    return PyLong_FromLong(enqueue(&b, stream));
}

/* call(capsule, stream_handle) -> status of moe_finalize_ex */
static PyObject *call(PyObject *self, PyObject *const *args, Py_ssize_t nargs) {
    (void)self;
    if (nargs != 2) {
        PyErr_SetString(PyExc_TypeError, "call(capsule, stream)");
        return NULL;
    }
    bound_call *b = (bound_call *)PyCapsule_GetPointer(args[0], kCapsule);
    if (!b) return NULL;
    void *stream = as_ptr(args[1]);
    if (PyErr_Occurred()) return NULL;
    return PyLong_FromLong(enqueue(b, stream));
}

static PyMethodDef methods[] = {
    {"pack", (PyCFunction)(void (*)(void))pack, METH_FASTCALL,
     "Pack a moe_finalize_ex call into a capsule."},
    {"call", (PyCFunction)(void (*)(void))call, METH_FASTCALL,
     "Enqueue a packed call on a stream; returns the status."},
    {"call_now", (PyCFunction)(void (*)(void))call_now, METH_FASTCALL,
     "Enqueue one moe_finalize_ex call from its arguments; returns the status."},
    {NULL, NULL, 0, NULL},
};

static struct PyModuleDef module = {PyModuleDef_HEAD_INIT, "_fastcall", NULL, -1, methods,
                                    NULL, NULL, NULL, NULL};

PyMODINIT_FUNC PyInit__fastcall(void) { return PyModule_Create(&module); }
