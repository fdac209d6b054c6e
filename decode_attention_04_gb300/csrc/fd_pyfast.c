// CPython entries for the per-call public functions fd_decode_attn,
// fd_decode_attn_ex, fd_decode_attn_fp8 and fd_decode_attn_fp8_ex: argument
// marshalling only (device addresses, the plan's host address and sizes as
// Python integers in, the library's status code out). They save the
// generic ctypes conversion on the host path of every call; the package falls
// back to ctypes when this module was not built.
#define PY_SSIZE_T_CLEAN
#include <Python.h>

#include "fd_decode_attn.h"

static PyObject* py_decode_attn(PyObject* self, PyObject* args) {
  unsigned long long q, k, v, out, lens, stream;
  int B, NH, NKV, HS, capacity, window;
  double scale;
  (void)self;
  if (!PyArg_ParseTuple(args, "KKKKKiiiiiidK", &q, &k, &v, &out, &lens, &B, &NH, &NKV, &HS, &capacity, &window,
                        &scale, &stream))
    return NULL;
  const int rc = fd_decode_attn((const void*)(uintptr_t)q, (const void*)(uintptr_t)k, (const void*)(uintptr_t)v,
                                (void*)(uintptr_t)out, (const int*)(uintptr_t)lens, B, NH, NKV, HS, capacity, window,
                                (float)scale, (fd_stream_t)(uintptr_t)stream);
  return PyLong_FromLong(rc);
}

static PyObject* py_decode_attn_fp8(PyObject* self, PyObject* args) {
  unsigned long long q, k8, v8, ks, vs, out, lens, stream;
  int B, NH, NKV, HS, capacity, window;
  double scale;
  (void)self;
  if (!PyArg_ParseTuple(args, "KKKKKKKiiiiiidK", &q, &k8, &v8, &ks, &vs, &out, &lens, &B, &NH, &NKV, &HS, &capacity,
                        &window, &scale, &stream))
    return NULL;
  const int rc = fd_decode_attn_fp8((const void*)(uintptr_t)q, (const void*)(uintptr_t)k8, (const void*)(uintptr_t)v8,
                                    (const float*)(uintptr_t)ks, (const float*)(uintptr_t)vs, (void*)(uintptr_t)out,
                                    (const int*)(uintptr_t)lens, B, NH, NKV, HS, capacity, window, (float)scale,
                                    (fd_stream_t)(uintptr_t)stream);
  return PyLong_FromLong(rc);
}

static PyObject* py_decode_attn_ex(PyObject* self, PyObject* args) {
  unsigned long long plan, ws, ws_bytes, out32, q, k, v, out, lens, stream;
  int B, NH, NKV, HS, capacity, window;
  double scale;
  (void)self;
  if (!PyArg_ParseTuple(args, "KKKKKKKKKiiiiiidK", &plan, &ws, &ws_bytes, &out32, &q, &k, &v, &out, &lens, &B, &NH,
                        &NKV, &HS, &capacity, &window, &scale, &stream))
    return NULL;
  const int rc = fd_decode_attn_ex((const fd_plan_t*)(uintptr_t)plan, (void*)(uintptr_t)ws, (size_t)ws_bytes,
                                   (float*)(uintptr_t)out32, (const void*)(uintptr_t)q, (const void*)(uintptr_t)k,
                                   (const void*)(uintptr_t)v, (void*)(uintptr_t)out, (const int*)(uintptr_t)lens, B, NH,
                                   NKV, HS, capacity, window, (float)scale, (fd_stream_t)(uintptr_t)stream);
  return PyLong_FromLong(rc);
}

static PyObject* py_decode_attn_fp8_ex(PyObject* self, PyObject* args) {
  unsigned long long plan, ws, ws_bytes, out32, q, k8, v8, ks, vs, out, lens, stream;
  int B, NH, NKV, HS, capacity, window;
  double scale;
  (void)self;
  if (!PyArg_ParseTuple(args, "KKKKKKKKKKKiiiiiidK", &plan, &ws, &ws_bytes, &out32, &q, &k8, &v8, &ks, &vs, &out,
                        &lens, &B, &NH, &NKV, &HS, &capacity, &window, &scale, &stream))
    return NULL;
  const int rc = fd_decode_attn_fp8_ex(
      (const fd_plan_t*)(uintptr_t)plan, (void*)(uintptr_t)ws, (size_t)ws_bytes, (float*)(uintptr_t)out32,
      (const void*)(uintptr_t)q, (const void*)(uintptr_t)k8, (const void*)(uintptr_t)v8, (const float*)(uintptr_t)ks,
      (const float*)(uintptr_t)vs, (void*)(uintptr_t)out, (const int*)(uintptr_t)lens, B, NH, NKV, HS, capacity,
      window, (float)scale, (fd_stream_t)(uintptr_t)stream);
  return PyLong_FromLong(rc);
}

static PyMethodDef kMethods[] = {
    {"decode_attn_ex", py_decode_attn_ex, METH_VARARGS, "fd_decode_attn_ex; returns the status code"},
    {"decode_attn_fp8_ex", py_decode_attn_fp8_ex, METH_VARARGS, "fd_decode_attn_fp8_ex; returns the status code"},
    {"decode_attn", py_decode_attn, METH_VARARGS, "fd_decode_attn; returns the status code"},
    {"decode_attn_fp8", py_decode_attn_fp8, METH_VARARGS, "fd_decode_attn_fp8; returns the status code"},
    {NULL, NULL, 0, NULL}};

static struct PyModuleDef kModule = {PyModuleDef_HEAD_INIT, "_fdfast", NULL, -1, kMethods, NULL, NULL, NULL, NULL};

PyMODINIT_FUNC PyInit__fdfast(void) { return PyModule_Create(&kModule); }
