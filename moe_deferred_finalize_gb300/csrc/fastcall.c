/*
 * _fastcall: a minimal CPython extension that calls moe_finalize_ex of the
 * loaded libmoe_finalize.so.  ctypes converts each of the call's twenty
 * arguments through its generic machinery on every call, which costs more
 * host time than the decode-size kernel takes on the GPU.  Here call_now
 * converts them directly, and pack/call go further for repeated calls: the
 * arguments are packed once into a C struct (a capsule) and each call passes
 * only the stream.  checked_call does the Python binding's argument checks
 * on DLPack descriptions of the tensors before calling.  Nothing here
 * computes anything of the finalize.
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

/* ---------------------------------------------------------------------------
 * checked_call: the checks of the Python binding, done here on DLPack
 * descriptions of the tensors (one capsule per tensor, as torch's
 * to_dlpack() makes them), then one moe_finalize_ex call.  Reading a
 * tensor's device, dtype, shape, strides and address costs one DLPack
 * export instead of six attribute lookups.
 *
 * The structures below are the DLPack interchange format (DLTensor inside a
 * DLManagedTensor, capsule name "dltensor"): a public interface that any
 * consumer has to lay out the same way.  The capsules are only read; each
 * one's own destructor releases its tensor.
 */
typedef struct {
    int32_t device_type;
    int32_t device_id;
} dl_device;

typedef struct {
    uint8_t code;
    uint8_t bits;
    uint16_t lanes;
} dl_dtype;

typedef struct {
    void *data;
    dl_device device;
    int32_t ndim;
    dl_dtype dtype;
    int64_t *shape;
    int64_t *strides;
    uint64_t byte_offset;
} dl_tensor;

typedef struct {
    dl_tensor t;
    void *manager_ctx;
    void (*deleter)(void *self);
} dl_managed;

enum { DL_INT = 0, DL_FLOAT = 2, DL_BFLOAT = 4 };
enum { DL_CUDA = 2 };

/* a tensor description; NULL for None (or on error, with a Python error) */
static const dl_tensor *described(PyObject *cap) {
    if (cap == Py_None) return NULL;
    dl_managed *m = (dl_managed *)PyCapsule_GetPointer(cap, "dltensor");
    return m ? &m->t : NULL;
}

/* 1 when t is a dense row-major array on CUDA device `dev` of element type
 * (code, bits), with ndim dimensions; its sizes go to dims */
static int dense(const dl_tensor *t, int dev, uint8_t code, uint8_t bits, int ndim,
                 int64_t *dims) {
    if (!t || t->device.device_type != DL_CUDA || t->device.device_id != dev) return 0;
    if (t->dtype.code != code || t->dtype.bits != bits || t->dtype.lanes != 1) return 0;
    if (t->ndim != ndim) return 0;
    int64_t stride = 1;
    for (int d = ndim - 1; d >= 0; --d) {
        dims[d] = t->shape[d];
        if (t->strides && t->shape[d] != 1 && t->strides[d] != stride) return 0;
        stride *= t->shape[d];
    }
    return 1;
}

static void *address(const dl_tensor *t) {
    return t ? (void *)((char *)t->data + t->byte_offset) : NULL;
}

/* checked_call(fn_address, wkind, weight_code, weight_bits, routed_scale,
 *              eps, device, splits, threads, flags, stream, permuted_out,
 *              idx_map, weights, shared_out, residual, gamma, out,
 *              residual_out, norm_out) -> status
 * The last nine are DLPack capsules or None.  Returns moe_finalize_ex's
 * status, or -1 when a tensor fails the binding's checks (wrong device,
 * dtype, rank, shape or layout, or a missing or extra tensor): the caller
 * then runs its own checks to report which. */
static PyObject *checked_call(PyObject *self, PyObject *const *a, Py_ssize_t nargs) {
    (void)self;
    if (nargs != 20) {
        PyErr_SetString(PyExc_TypeError, "checked_call takes 20 arguments");
        return NULL;
    }
    finalize_ex_fn fn = (finalize_ex_fn)as_ptr(a[0]);
    const int wkind = (int)PyLong_AsLong(a[1]);
    const uint8_t wcode = (uint8_t)PyLong_AsLong(a[2]);
    const uint8_t wbits = (uint8_t)PyLong_AsLong(a[3]);
    const float scale = (float)PyFloat_AsDouble(a[4]);
    const float eps = (float)PyFloat_AsDouble(a[5]);
    const int dev = (int)PyLong_AsLong(a[6]);
    const int splits = (int)PyLong_AsLong(a[7]);
    const int threads = (int)PyLong_AsLong(a[8]);
    const unsigned flags = (unsigned)PyLong_AsUnsignedLong(a[9]);
    void *stream = as_ptr(a[10]);
    if (PyErr_Occurred()) return NULL;
    if (!fn) {
        PyErr_SetString(PyExc_ValueError, "null function pointer");
        return NULL;
    }
    const dl_tensor *t[9];
    for (int i = 0; i < 9; ++i) {
        t[i] = described(a[11 + i]);
        if (PyErr_Occurred()) return NULL;
    }
    const dl_tensor *x = t[0], *idx = t[1], *w = t[2], *sh = t[3], *res = t[4], *gam = t[5],
                    *out = t[6], *rout = t[7], *nout = t[8];
    int64_t xd[2], id[2], d2[2], d1[1];
    int ok = dense(x, dev, DL_BFLOAT, 16, 2, xd) && dense(idx, dev, DL_INT, 32, 2, id) &&
             dense(w, dev, wcode, wbits, 2, d2) && d2[0] == id[0] && d2[1] == id[1] &&
             dense(sh, dev, DL_BFLOAT, 16, 2, d2) && d2[0] == id[0] && d2[1] == xd[1];
    const int norm = res != NULL;
    if (ok && (norm != (gam != NULL) || norm != (rout != NULL) || norm != (nout != NULL) ||
               (!norm && !out)))
        ok = 0;
    const dl_tensor *rows[4] = {res, out, rout, nout};
    for (int i = 0; ok && i < 4; ++i)
        if (rows[i])
            ok = dense(rows[i], dev, DL_BFLOAT, 16, 2, d2) && d2[0] == id[0] && d2[1] == xd[1];
    if (ok && gam) ok = dense(gam, dev, DL_BFLOAT, 16, 1, d1) && d1[0] == xd[1];
    if (ok && (xd[1] > 0x7FFFFFFF || id[0] > 0x7FFFFFFF || id[1] > 0x7FFFFFFF)) ok = 0;
    if (!ok) return PyLong_FromLong(-1);
    return PyLong_FromLong(fn(address(x), xd[0], (const int32_t *)address(idx), address(w),
                              wkind, scale, address(sh), address(res), address(gam), eps,
                              address(out), address(rout), address(nout), (int)id[0],
                              (int)id[1], (int)xd[1], splits, threads, flags, stream));
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
    {"checked_call", (PyCFunction)(void (*)(void))checked_call, METH_FASTCALL,
     "Check DLPack-described tensors and enqueue one moe_finalize_ex call."},
    {NULL, NULL, 0, NULL},
};

static struct PyModuleDef module = {PyModuleDef_HEAD_INIT, "_fastcall", NULL, -1, methods,
                                    NULL, NULL, NULL, NULL};

PyMODINIT_FUNC PyInit__fastcall(void) { return PyModule_Create(&module); }
