/*
 * _pkvfast: low-overhead Python entry points for the per-step calls of
 * libpagedkv.so (paged_decode, paged_decode_step, paged_decode_attention,
 * kv_append).  Argument marshalling only: each function parses plain Python
 * integers and floats (addresses as integers, the CUDA stream as an
 * integer) and calls the C ABI function of the same name, returning its
 * status.  The ctypes binding marshals the same calls about 10 us slower
 * per call, which bounds a Python loop of small decode steps.
 */
#define PY_SSIZE_T_CLEAN
#include <Python.h>

#include <stddef.h>
#include <stdint.h>

#include "paged_kv.h"

#define PTR(x) ((void*)(uintptr_t)(x))

static PyObject* fast_paged_decode(PyObject* self, PyObject* args)
{
    unsigned long long out, q, k_new, v_new, k_cache, v_cache, bt, ctx, chunks, seq_chunk, ws,
        ws_bytes, stream;
    int out_dtype, kv_dtype, num_blocks, max_blocks, num_seqs, hq, hkv, d, num_chunks;
    float k_scale, v_scale, scale;
    unsigned int flags;
    (void)self;
    if (!PyArg_ParseTuple(args, "KiKKKKKiffiKiKiiiifKKiIKKK", &out, &out_dtype, &q, &k_new,
                          &v_new, &k_cache, &v_cache, &kv_dtype, &k_scale, &v_scale,
                          &num_blocks, &bt, &max_blocks, &ctx, &num_seqs, &hq, &hkv, &d, &scale,
                          &chunks, &seq_chunk, &num_chunks, &flags, &ws, &ws_bytes, &stream))
        return NULL;
    int rc;
    Py_BEGIN_ALLOW_THREADS
    rc = paged_decode(PTR(out), out_dtype, PTR(q), PTR(k_new), PTR(v_new), PTR(k_cache),
                      PTR(v_cache), kv_dtype, k_scale, v_scale, num_blocks,
                      (const int32_t*)PTR(bt), max_blocks, (const int32_t*)PTR(ctx), num_seqs,
                      hq, hkv, d, scale, (const int32_t*)PTR(chunks),
                      (const int32_t*)PTR(seq_chunk), num_chunks, flags, PTR(ws),
                      (size_t)ws_bytes, PTR(stream));
    Py_END_ALLOW_THREADS
    return PyLong_FromLong(rc);
}

static PyObject* fast_paged_decode_step(PyObject* self, PyObject* args)
{
    unsigned long long out, q, k_new, v_new, k_cache, v_cache, bt, ctx, ws, ws_bytes, stream;
    int out_dtype, kv_dtype, num_blocks, max_blocks, num_seqs, hq, hkv, d;
    float k_scale, v_scale, scale;
    (void)self;
    if (!PyArg_ParseTuple(args, "KiKKKKKiffiKiKiiiifKKK", &out, &out_dtype, &q, &k_new, &v_new,
                          &k_cache, &v_cache, &kv_dtype, &k_scale, &v_scale, &num_blocks, &bt,
                          &max_blocks, &ctx, &num_seqs, &hq, &hkv, &d, &scale, &ws, &ws_bytes,
                          &stream))
        return NULL;
    int rc;
    Py_BEGIN_ALLOW_THREADS
    rc = paged_decode_step(PTR(out), out_dtype, PTR(q), PTR(k_new), PTR(v_new), PTR(k_cache),
                           PTR(v_cache), kv_dtype, k_scale, v_scale, num_blocks,
                           (const int32_t*)PTR(bt), max_blocks, (const int32_t*)PTR(ctx),
                           num_seqs, hq, hkv, d, scale, PTR(ws), (size_t)ws_bytes, PTR(stream));
    Py_END_ALLOW_THREADS
    return PyLong_FromLong(rc);
}

static PyObject* fast_paged_decode_attention(PyObject* self, PyObject* args)
{
    unsigned long long out, q, k_cache, v_cache, bt, ctx, ws, ws_bytes, stream;
    int out_dtype, kv_dtype, num_blocks, max_blocks, num_seqs, hq, hkv, d;
    float k_scale, v_scale, scale;
    (void)self;
    if (!PyArg_ParseTuple(args, "KiKKKiffiKiKiiiifKKK", &out, &out_dtype, &q, &k_cache,
                          &v_cache, &kv_dtype, &k_scale, &v_scale, &num_blocks, &bt,
                          &max_blocks, &ctx, &num_seqs, &hq, &hkv, &d, &scale, &ws, &ws_bytes,
                          &stream))
        return NULL;
    int rc;
    Py_BEGIN_ALLOW_THREADS
    rc = paged_decode_attention(PTR(out), out_dtype, PTR(q), PTR(k_cache), PTR(v_cache),
                                kv_dtype, k_scale, v_scale, num_blocks,
                                (const int32_t*)PTR(bt), max_blocks, (const int32_t*)PTR(ctx),
                                num_seqs, hq, hkv, d, scale, PTR(ws), (size_t)ws_bytes,
                                PTR(stream));
    Py_END_ALLOW_THREADS
    return PyLong_FromLong(rc);
}

static PyObject* fast_kv_append(PyObject* self, PyObject* args)
{
    unsigned long long k, v, k_cache, v_cache, slots, stream;
    int num_tokens, hkv, d, num_blocks, kv_dtype;
    float k_scale, v_scale;
    (void)self;
    if (!PyArg_ParseTuple(args, "KKKKKiiiiiffK", &k, &v, &k_cache, &v_cache, &slots,
                          &num_tokens, &hkv, &d, &num_blocks, &kv_dtype, &k_scale, &v_scale,
                          &stream))
        return NULL;
    int rc;
    Py_BEGIN_ALLOW_THREADS
    rc = kv_append(PTR(k), PTR(v), PTR(k_cache), PTR(v_cache), (const int64_t*)PTR(slots),
                   num_tokens, hkv, d, num_blocks, kv_dtype, k_scale, v_scale, PTR(stream));
    Py_END_ALLOW_THREADS
    return PyLong_FromLong(rc);
}

static PyMethodDef methods[] = {
    {"paged_decode", fast_paged_decode, METH_VARARGS, "paged_decode of libpagedkv (26 args)"},
    {"paged_decode_step", fast_paged_decode_step, METH_VARARGS,
     "paged_decode_step of libpagedkv (22 args)"},
    {"paged_decode_attention", fast_paged_decode_attention, METH_VARARGS,
     "paged_decode_attention of libpagedkv (20 args)"},
    {"kv_append", fast_kv_append, METH_VARARGS, "kv_append of libpagedkv (13 args)"},
    {NULL, NULL, 0, NULL}};

static struct PyModuleDef module = {PyModuleDef_HEAD_INIT, "_pkvfast",
                                    "Low-overhead entry points of libpagedkv.", -1, methods,
                                    NULL, NULL, NULL, NULL};

PyMODINIT_FUNC PyInit__pkvfast(void) { return PyModule_Create(&module); }
