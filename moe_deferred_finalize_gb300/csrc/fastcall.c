/*
 * _fastcall: a minimal CPython extension that replays a pre-marshalled
 * moe_finalize_ex call.  ctypes converts every one of the call's twenty
 * arguments on every call, which costs more host time than the decode-size
 * kernel takes on the GPU; here the arguments are packed once into a C
 * struct (a capsule) and each call passes only the stream.  It does no
 * computation and no checking beyond what the C ABI itself does: the
 * function pointer is moe_finalize_ex of the loaded libmoe_finalize.so.
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

/* pack(fn_address, permuted_out, P, idx_map, weights, wkind, routed_scale,
 *      shared_out, residual, gamma, eps, out, residual_out, norm_out,
 *      T, K, H, splits, threads, flags) -> capsule
 * Pointers are ints (or None), as ctypes' c_void_p(...).value gives them. */
static PyObject *pack(PyObject *self, PyObject *args) {
    (void)self;
    PyObject *fn, *x, *idx, *w, *sh, *res, *g, *out, *ro, *no;
    long long P;
    int wkind, T, K, H, splits, threads;
    unsigned int flags;
    double scale, eps;
    if (!PyArg_ParseTuple(args, "OOLOOidOOOdOOOiiiiiI", &fn, &x, &P, &idx, &w, &wkind, &scale,
                          &sh, &res, &g, &eps, &out, &ro, &no, &T, &K, &H, &splits, &threads,
                          &flags))
        return NULL;
    bound_call *b = (bound_call *)calloc(1, sizeof(bound_call));
    if (!b) return PyErr_NoMemory();
    b->fn = (finalize_ex_fn)as_ptr(fn);
    b->permuted_out = as_ptr(x);
    b->P = (int64_t)P;
    b->idx_map = (const int32_t *)as_ptr(idx);
    b->weights = as_ptr(w);
    b->wkind = wkind;
    b->routed_scale = (float)scale;
    b->shared_out = as_ptr(sh);
    b->residual = as_ptr(res);
    b->gamma = as_ptr(g);
    b->eps = (float)eps;
    b->out = as_ptr(out);
    b->residual_out = as_ptr(ro);
    b->norm_out = as_ptr(no);
    b->T = T;
    b->K = K;
    b->H = H;
    b->splits = splits;
    b->threads = threads;
    b->flags = flags;
    if (PyErr_Occurred() || !b->fn) {
        free(b);
        if (!PyErr_Occurred()) PyErr_SetString(PyExc_ValueError, "null function pointer");
        return NULL;
    }
    return PyCapsule_New(b, kCapsule, free_bound);
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
    int st = b->fn(b->permuted_out, b->P, b->idx_map, b->weights, b->wkind, b->routed_scale,
                   b->shared_out, b->residual, b->gamma, b->eps, b->out, b->residual_out,
                   b->norm_out, b->T, b->K, b->H, b->splits, b->threads, b->flags, stream);
    return PyLong_FromLong(st);
}

static PyMethodDef methods[] = {
    {"pack", pack, METH_VARARGS, "Pack a moe_finalize_ex call into a capsule."},
    {"call", (PyCFunction)(void (*)(void))call, METH_FASTCALL,
     "Enqueue a packed call on a stream; returns the status."},
    {NULL, NULL, 0, NULL},
};

static struct PyModuleDef module = {PyModuleDef_HEAD_INIT, "_fastcall", NULL, -1, methods,
                                    NULL, NULL, NULL, NULL};

PyMODINIT_FUNC PyInit__fastcall(void) { return PyModule_Create(&module); }
