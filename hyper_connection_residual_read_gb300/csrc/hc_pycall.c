/* Python call path of the read entry points: hc_read and hc_read_path called from
 * CPython with the arguments converted in C, instead of through ctypes' per-call
 * argument conversion. Marshalling only: the module holds no arithmetic of the read
 * and links nothing; it calls the library's own entry points, whose addresses the
 * binding hands over once (bind) from the library it has loaded, so that both call
 * paths always enter the same library.
 *
 * A pointer argument is None (NULL), an int (the address) or any object with a
 * data_ptr() method (a torch tensor). The return value is the entry point's status
 * code; the binding turns a non-zero code into an exception.
 */
#define PY_SSIZE_T_CLEAN
#include <Python.h>
#include <limits.h>
#include <stdint.h>

typedef int (*read_fn)(int, void*, void*, void*, void*, void*, void*, void*, void*, void*,
                       void*);
typedef int (*read_path_fn)(int, int, void*, void*, void*, void*, void*, void*, void*, void*,
                            void*, void*);

static read_fn p_read = NULL;
static read_path_fn p_read_path = NULL;
static PyObject* s_data_ptr = NULL; /* interned "data_ptr" */

/* The address an argument stands for; -1 with an exception set on failure. */
static int to_ptr(PyObject* o, void** out) {
    if (o == Py_None) {
        *out = NULL;
        return 0;
    }
    if (PyLong_Check(o)) {
        *out = PyLong_AsVoidPtr(o);
        return (*out == NULL && PyErr_Occurred()) ? -1 : 0;
    }
    PyObject* v = PyObject_CallMethodNoArgs(o, s_data_ptr);
    if (v == NULL) return -1;
    *out = PyLong_AsVoidPtr(v);
    Py_DECREF(v);
    return (*out == NULL && PyErr_Occurred()) ? -1 : 0;
}

/* An int argument of the entry point (token count, path): -1 with an exception set if
 * it is not an int or does not fit in a C int (rather than truncating it into one that
 * the library's range checks would accept). */
static int to_int(PyObject* o, int* out) {
    const long v = PyLong_AsLong(o);
    if (v == -1 && PyErr_Occurred()) return -1;
    if (v < INT_MIN || v > INT_MAX) {
        PyErr_SetString(PyExc_OverflowError, "argument out of the range of a C int");
        return -1;
    }
    *out = (int)v;
    return 0;
}

/* bind(addr_hc_read, addr_hc_read_path) */
static PyObject* py_bind(PyObject* self, PyObject* const* args, Py_ssize_t n) {
    (void)self;
    if (n != 2) {
        PyErr_SetString(PyExc_TypeError, "bind takes 2 addresses");
        return NULL;
    }
    void* a = PyLong_AsVoidPtr(args[0]);
    void* b = PyLong_AsVoidPtr(args[1]);
    if (PyErr_Occurred()) return NULL;
    p_read = (read_fn)a;
    p_read_path = (read_path_fn)b;
    Py_RETURN_NONE;
}

/* read(tokens, R, P, w_norm, W_down, W_up, Rmix, out_f32, out_bf16, out_fp16, stream) */
static PyObject* py_read(PyObject* self, PyObject* const* args, Py_ssize_t n) {
    (void)self;
    if (n != 11) {
        PyErr_SetString(PyExc_TypeError, "read takes 11 arguments");
        return NULL;
    }
    if (p_read == NULL) {
        PyErr_SetString(PyExc_RuntimeError, "read: not bound to a library");
        return NULL;
    }
    int tokens;
    if (to_int(args[0], &tokens) != 0) return NULL;
    void* p[10];
    for (int i = 0; i < 10; ++i)
        if (to_ptr(args[1 + i], &p[i]) != 0) return NULL;
    const int rc = p_read(tokens, p[0], p[1], p[2], p[3], p[4], p[5], p[6], p[7], p[8], p[9]);
    return PyLong_FromLong(rc);
}

/* read_path(path, tokens, R, P, w_norm, W_down, W_up, Rmix, out_f32, out_bf16, out_fp16,
 * stream) */
static PyObject* py_read_path(PyObject* self, PyObject* const* args, Py_ssize_t n) {
    (void)self;
    if (n != 12) {
        PyErr_SetString(PyExc_TypeError, "read_path takes 12 arguments");
        return NULL;
    }
    if (p_read_path == NULL) {
        PyErr_SetString(PyExc_RuntimeError, "read_path: not bound to a library");
        return NULL;
    }
    int path, tokens;
    if (to_int(args[0], &path) != 0 || to_int(args[1], &tokens) != 0) return NULL;
    void* p[10];
    for (int i = 0; i < 10; ++i)
        if (to_ptr(args[2 + i], &p[i]) != 0) return NULL;
    const int rc = p_read_path(path, tokens, p[0], p[1], p[2], p[3], p[4], p[5], p[6], p[7], p[8],
                               p[9]);
    return PyLong_FromLong(rc);
}

static PyMethodDef methods[] = {
    {"bind", (PyCFunction)(void (*)(void))py_bind, METH_FASTCALL, "bind the entry points"},
    {"read", (PyCFunction)(void (*)(void))py_read, METH_FASTCALL, "hc_read"},
    {"read_path", (PyCFunction)(void (*)(void))py_read_path, METH_FASTCALL, "hc_read_path"},
    {NULL, NULL, 0, NULL},
};

static struct PyModuleDef module = {PyModuleDef_HEAD_INIT, "_hcpycall", NULL, -1, methods,
                                    NULL, NULL, NULL, NULL};

PyMODINIT_FUNC PyInit__hcpycall(void) {
    s_data_ptr = PyUnicode_InternFromString("data_ptr");
    if (s_data_ptr == NULL) return NULL;
    return PyModule_Create(&module);
}
