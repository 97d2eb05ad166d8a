"""The C-ABI library builds, loads without a GPU and exports every entry point
that include/paged_kv.h declares; its host-only functions agree with the
pages' worked numbers and with the oracle."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "paged_kv.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^(?:const\s+char\s*\*|int64_t|int|void|size_t)\s+\**\s*(\w+)\s*\(",
                       src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib_path():
    import __graft_entry__
    return __graft_entry__.build_native()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("kv_bytes", "kv_cache_alloc", "kv_append", "paged_decode_attention",
                     "kv_step", "kv_seq_add", "kv_seq_fork", "kv_seq_free", "kv_alloc_destroy",
                     "kv_copy_blocks", "paged_decode_workspace_bytes", "kv_slot_mapping"):
        assert required in names


def test_library_exports_every_declared_symbol(lib_path):
    L = ctypes.CDLL(lib_path)
    for name in declared_functions():
        assert hasattr(L, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True,
                         text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing


def test_binding_loads_and_reports_version(lib_path):
    import paged_kv_cache_21_gb300 as pk
    assert pk.version().startswith("pagedkv")
    assert os.path.samefile(pk.native_library_path(), lib_path)


def test_product_kv_bytes_matches_worked_examples(lib_path, golden):
    import paged_kv_cache_21_gb300 as pk
    for layers, batch, heads, seq, d, nbytes, expected in golden("kv_bytes_examples.txt"):
        assert pk.kv_bytes(layers, batch, heads, seq, d, nbytes) == expected
    with pytest.raises(ValueError):
        pk.kv_bytes(-1, 1, 1, 1, 1, 1)
    with pytest.raises(ValueError):
        pk.kv_bytes(1 << 30, 1 << 30, 1 << 30, 1, 1, 2)        # int64 overflow


def test_product_slot_mapping_matches_oracle(lib_path, golden):
    import paged_kv_cache_21_gb300 as pk
    rows = golden("slot_mapping_example.txt")
    pos = np.array([r[0] for r in rows], dtype=np.int64)
    bt = np.tile(np.array([[7, 2, 9]], dtype=np.int32), (len(pos), 1))
    np.testing.assert_array_equal(pk.slot_mapping(bt, pos), [r[1] for r in rows])
    rng = np.random.default_rng(0)
    n, mb = 500, 40
    bt = rng.integers(0, 100000, size=(n, mb)).astype(np.int32)
    pos = rng.integers(0, mb * 16, size=n)
    np.testing.assert_array_equal(pk.slot_mapping(bt, pos),
                                  oracle.slot_mapping(bt, np.arange(n), pos))
    assert pk.slot_mapping(bt[:1], np.array([-1]))[0] == -1
    with pytest.raises(pk.KVError):
        pk.slot_mapping(bt[:1], np.array([mb * 16]))


def test_gpu_entry_points_reject_bad_arguments_without_a_gpu(lib_path):
    import paged_kv_cache_21_gb300 as pk
    L = pk._lib
    # shape checks happen before any CUDA call
    assert L.kv_append(None, None, None, None, None, 4, 0, 128, 10, 0, 1.0, 1.0, None) == \
        pk.KV_ERR_INVALID_ARG
    assert L.kv_append(None, None, None, None, None, 4, 8, 100, 10, 0, 1.0, 1.0, None) == \
        pk.KV_ERR_UNSUPPORTED
    assert L.paged_decode_attention(None, 0, None, None, None, 0, 1.0, 1.0, 1, None, 1, None,
                                    1, 32, 8, 96, 0.1, None, 0, None) == pk.KV_ERR_UNSUPPORTED
    # group sizes: 17 and 34 have no even split into sub-groups of <= 16 rows,
    # 256 exceeds the largest split; 16, 24 and 128 pass the shape checks
    # (and then fail on the NULL buffers, still before any CUDA call)
    for hq, hkv, want in ((51, 3, pk.KV_ERR_UNSUPPORTED), (68, 2, pk.KV_ERR_UNSUPPORTED),
                          (256, 1, pk.KV_ERR_UNSUPPORTED), (48, 3, pk.KV_ERR_INVALID_ARG),
                          (48, 2, pk.KV_ERR_INVALID_ARG), (128, 1, pk.KV_ERR_INVALID_ARG)):
        assert L.paged_decode_attention(None, 0, None, None, None, 0, 1.0, 1.0, 1, None, 1, None,
                                        1, hq, hkv, 128, 0.1, None, 0, None) == want, (hq, hkv)
    assert L.paged_decode_attention(None, 0, None, None, None, 0, 1.0, 1.0, 1, None, 1, None,
                                    1, 30, 8, 128, 0.1, None, 0, None) == pk.KV_ERR_INVALID_ARG
    assert L.paged_decode_attention(None, 0, None, None, None, 0, 1.0, 1.0, 1, None, 1, None,
                                    0, 32, 8, 128, 0.1, None, 0, None) == pk.KV_OK


def test_measurement_hooks_reject_bad_arguments_without_a_gpu(lib_path):
    import paged_kv_cache_21_gb300 as pk
    L = pk._lib
    sink = ctypes.c_void_p(64)
    # kv_read_ceiling: no buffer, no bytes, a size or an address off 16 bytes
    assert L.kv_read_ceiling(None, 4096, sink, None) == pk.KV_ERR_INVALID_ARG
    assert L.kv_read_ceiling(ctypes.c_void_p(4096), 0, sink, None) == pk.KV_ERR_INVALID_ARG
    assert L.kv_read_ceiling(ctypes.c_void_p(4096), 4100, sink, None) == pk.KV_ERR_INVALID_ARG
    assert L.kv_read_ceiling(ctypes.c_void_p(4104), 4096, sink, None) == pk.KV_ERR_INVALID_ARG
    assert L.kv_read_ceiling(ctypes.c_void_p(4096), 4096, None, None) == pk.KV_ERR_INVALID_ARG
    # paged_decode_timed shares paged_decode's shape checks (head_dim 96)
    assert L.paged_decode_timed(None, 0, None, None, None, None, None, 0, 1.0, 1.0, 1, None, 1,
                                None, 1, 32, 8, 96, 0.1, None, None, 0, 0, None, 0, None, None,
                                None, None) == pk.KV_ERR_UNSUPPORTED


def test_fast_call_module_marshals_only(lib_path):
    """The CPython-API module, when built, exposes the four per-step calls
    and checks only the argument list (a wrong one fails before any call)."""
    import paged_kv_cache_21_gb300 as pk
    if not pk.fast_path():
        pytest.skip("no Python headers here: the ctypes binding serves every call")
    import paged_kv_cache_21_gb300._pkvfast as fast
    for name, n in (("paged_decode", 26), ("paged_decode_step", 22),
                    ("paged_decode_attention", 20), ("kv_append", 13)):
        fn = getattr(fast, name)
        with pytest.raises(TypeError):
            fn(*([0] * (n - 1)))
        with pytest.raises(TypeError):
            fn(*([0] * (n + 1)))
    # the module links the library the ctypes handle loaded, not a copy
    out = subprocess.run(["ldd", fast.__file__], capture_output=True, text=True).stdout
    assert "libpagedkv.so" in out and os.path.dirname(lib_path) in out
