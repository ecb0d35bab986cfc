/*
 * fastcall.c -- a CPython extension that makes one prepared dpred_flush_bucket
 * call with less host overhead than ctypes.
 *
 * A training loop flushes the same buckets every step with the same
 * arguments.  ctypes converts all seventeen arguments on every call (about
 * 1.3 us); here they are converted once, by prepare(), into a C struct kept in
 * a capsule, and flush() passes them on together with the per-call stream and
 * probe.  call() makes one unprepared call from plain integers, for the
 * binding's flush_bucket.  The function called is the library's own dpred_flush_bucket, whose
 * address the Python binding hands over (the library is loaded once, by the
 * binding, so the plan cache and the error state are the ones every other
 * call uses).  This module adds no arithmetic: argument marshalling only.
 * It is optional: where it cannot be built (no Python headers), the binding
 * makes the same call through ctypes.
 */
#define PY_SSIZE_T_CLEAN
#include <Python.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "dpred.h"

typedef int (*flush_fn)(int32_t, int32_t, void*, int64_t, const dpred_task*, int32_t, const int32_t*, int32_t,
                        int32_t, void* const*, int32_t, int32_t, int32_t, dpred_probe*, void*, size_t, void*);

typedef struct {
    flush_fn fn;
    int32_t world, in_dt, n_tasks, n_params, out_dt, pre_div, rto, flags;
    void* grads;
    int64_t ld;
    const dpred_task* tasks;
    const int32_t* owner;
    void* const* dst;
    void* workspace;
    size_t workspace_bytes;
} Prepared;

static const char* kCapsule = "dpred.prepared_flush";

static void release(PyObject* cap) { free(PyCapsule_GetPointer(cap, kCapsule)); }

/* prepare(fn, world, in_dt, grads, ld, tasks, n_tasks, owner, n_params, out_dt, dst, pre_div,
 *         reduce_to_owner, flags, workspace, workspace_bytes) -> capsule
 * Pointers are integer addresses (0 = NULL); the caller keeps the memory behind
 * them alive for as long as the capsule is used. */
static PyObject* prepare(PyObject* self, PyObject* args) {
    (void)self;
    unsigned long long fn, grads, tasks, owner, dst, ws, ws_bytes;
    long long ld;
    int world, in_dt, n_tasks, n_params, out_dt, pre_div, rto, flags;
    if (!PyArg_ParseTuple(args, "KiiKLKiKiiKiiiKK", &fn, &world, &in_dt, &grads, &ld, &tasks, &n_tasks, &owner,
                          &n_params, &out_dt, &dst, &pre_div, &rto, &flags, &ws, &ws_bytes))
        return NULL;
    if (!fn) {
        PyErr_SetString(PyExc_ValueError, "null function address");
        return NULL;
    }
    Prepared* p = (Prepared*)malloc(sizeof(Prepared));
    if (!p) return PyErr_NoMemory();
    p->fn = (flush_fn)(uintptr_t)fn;
    p->world = world;
    p->in_dt = in_dt;
    p->grads = (void*)(uintptr_t)grads;
    p->ld = (int64_t)ld;
    p->tasks = (const dpred_task*)(uintptr_t)tasks;
    p->n_tasks = n_tasks;
    p->owner = (const int32_t*)(uintptr_t)owner;
    p->n_params = n_params;
    p->out_dt = out_dt;
    p->dst = (void* const*)(uintptr_t)dst;
    p->pre_div = pre_div;
    p->rto = rto;
    p->flags = flags;
    p->workspace = (void*)(uintptr_t)ws;
    p->workspace_bytes = (size_t)ws_bytes;
    PyObject* cap = PyCapsule_New(p, kCapsule, release);
    if (!cap) free(p);
    return cap;
}

/* The interpreter lock is released around the library call, as ctypes does:
 * a plan that needs workspace copies it to the device, which can block. */
static int call(const Prepared* p, dpred_probe* probe, PyObject* stream_arg) {
    const unsigned long long stream = PyLong_AsUnsignedLongLong(stream_arg);
    if (stream == (unsigned long long)-1 && PyErr_Occurred()) return INT32_MIN;
    int rc;
    Py_BEGIN_ALLOW_THREADS
    rc = p->fn(p->world, p->in_dt, p->grads, p->ld, p->tasks, p->n_tasks, p->owner, p->n_params, p->out_dt, p->dst,
               p->pre_div, p->rto, p->flags, probe, p->workspace, p->workspace_bytes, (void*)(uintptr_t)stream);
    Py_END_ALLOW_THREADS
    return rc;
}

/* flush(capsule, stream) -> status code of dpred_flush_bucket */
static PyObject* flush(PyObject* self, PyObject* const* args, Py_ssize_t nargs) {
    (void)self;
    if (nargs != 2) {
        PyErr_SetString(PyExc_TypeError, "flush(prepared, stream)");
        return NULL;
    }
    const Prepared* p = (const Prepared*)PyCapsule_GetPointer(args[0], kCapsule);
    if (!p) return NULL;
    const int rc = call(p, NULL, args[1]);
    return rc == INT32_MIN ? NULL : PyLong_FromLong(rc);
}

/* The probe counters of one call as (status, flush_index, tasks, reduced_elems,
 * owner_tasks, owner_elems, [kept_elems of each rank]). */
static PyObject* probe_tuple(int rc, const dpred_probe* probe, int world) {
    const int w = world < 0 ? 0 : (world > DPRED_MAX_WORLD ? DPRED_MAX_WORLD : world);
    PyObject* kept = PyList_New(w);
    if (!kept) return NULL;
    for (int r = 0; r < w; ++r) {
        PyObject* v = PyLong_FromLongLong(probe->kept_elems[r]);
        if (!v) {
            Py_DECREF(kept);
            return NULL;
        }
        PyList_SET_ITEM(kept, r, v);
    }
    return Py_BuildValue("(iLLLLLN)", rc, (long long)probe->flush_index, (long long)probe->tasks,
                         (long long)probe->reduced_elems, (long long)probe->owner_tasks, (long long)probe->owner_elems,
                         kept);
}

/* flush_probed(capsule, stream, flush_index)
 *   -> (status, flush_index, tasks, reduced_elems, owner_tasks, owner_elems, [kept_elems of each rank])
 * The counters live on this call's stack, so concurrent calls share nothing. */
static PyObject* flush_probed(PyObject* self, PyObject* const* args, Py_ssize_t nargs) {
    (void)self;
    if (nargs != 3) {
        PyErr_SetString(PyExc_TypeError, "flush_probed(prepared, stream, flush_index)");
        return NULL;
    }
    const Prepared* p = (const Prepared*)PyCapsule_GetPointer(args[0], kCapsule);
    if (!p) return NULL;
    dpred_probe probe;
    memset(&probe, 0, sizeof probe);
    probe.flush_index = PyLong_AsLongLong(args[2]);
    if (probe.flush_index == -1 && PyErr_Occurred()) return NULL;
    const int rc = call(p, &probe, args[1]);
    if (rc == INT32_MIN) return NULL;
    return probe_tuple(rc, &probe, p->world);
}

/* call(fn, world, in_dt, grads, ld, tasks, n_tasks, owner, n_params, out_dt, dst, pre_div,
 *      reduce_to_owner, flags, workspace, workspace_bytes, stream, flush_index)
 * One unprepared dpred_flush_bucket call; addresses are integers (0 = NULL).
 * flush_index None: no probe, returns the status code; an integer: returns the
 * probe tuple of flush_probed. */
static PyObject* call_once(PyObject* self, PyObject* const* args, Py_ssize_t nargs) {
    (void)self;
    if (nargs != 18) {
        PyErr_SetString(PyExc_TypeError, "call() takes 18 arguments");
        return NULL;
    }
    /* addresses and the workspace size are unsigned; the other arguments are
     * signed and reach the library as ctypes would pass them */
    static const int kUnsigned[16] = {1, 0, 0, 1, 0, 1, 0, 1, 0, 0, 1, 0, 0, 0, 1, 1};
    unsigned long long u[16];
    for (int i = 0; i < 16; ++i) {
        if (kUnsigned[i]) {
            u[i] = PyLong_AsUnsignedLongLong(args[i]);
        } else {
            const long long v = PyLong_AsLongLong(args[i]);
            u[i] = (unsigned long long)v;
        }
        if (u[i] == (unsigned long long)-1 && PyErr_Occurred()) return NULL;
    }
    if (!u[0]) {
        PyErr_SetString(PyExc_ValueError, "null function address");
        return NULL;
    }
    Prepared p;
    p.fn = (flush_fn)(uintptr_t)u[0];
    p.world = (int32_t)u[1];
    p.in_dt = (int32_t)u[2];
    p.grads = (void*)(uintptr_t)u[3];
    p.ld = (int64_t)u[4];
    p.tasks = (const dpred_task*)(uintptr_t)u[5];
    p.n_tasks = (int32_t)u[6];
    p.owner = (const int32_t*)(uintptr_t)u[7];
    p.n_params = (int32_t)u[8];
    p.out_dt = (int32_t)u[9];
    p.dst = (void* const*)(uintptr_t)u[10];
    p.pre_div = (int32_t)u[11];
    p.rto = (int32_t)u[12];
    p.flags = (int32_t)u[13];
    p.workspace = (void*)(uintptr_t)u[14];
    p.workspace_bytes = (size_t)u[15];
    if (args[17] == Py_None) {
        const int rc = call(&p, NULL, args[16]);
        return rc == INT32_MIN ? NULL : PyLong_FromLong(rc);
    }
    dpred_probe probe;
    memset(&probe, 0, sizeof probe);
    probe.flush_index = PyLong_AsLongLong(args[17]);
    if (probe.flush_index == -1 && PyErr_Occurred()) return NULL;
    const int rc = call(&p, &probe, args[16]);
    if (rc == INT32_MIN) return NULL;
    return probe_tuple(rc, &probe, p.world);
}

static PyMethodDef kMethods[] = {
    {"prepare", prepare, METH_VARARGS, "Convert one dpred_flush_bucket call's arguments once."},
    {"flush", (PyCFunction)(void (*)(void))flush, METH_FASTCALL, "Make a prepared dpred_flush_bucket call."},
    {"flush_probed", (PyCFunction)(void (*)(void))flush_probed, METH_FASTCALL,
     "Make a prepared dpred_flush_bucket call and return its probe counters."},
    {"call", (PyCFunction)(void (*)(void))call_once, METH_FASTCALL, "Make one unprepared dpred_flush_bucket call."},
    {NULL, NULL, 0, NULL},
};

static struct PyModuleDef kModule = {PyModuleDef_HEAD_INIT, "_fastcall", NULL, -1, kMethods, NULL, NULL, NULL, NULL};

PyMODINIT_FUNC PyInit__fastcall(void) { return PyModule_Create(&kModule); }
