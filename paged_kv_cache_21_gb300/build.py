"""Build ``libpagedkv.so`` in-tree for sm_103a.

Each CUDA translation unit is compiled by its own nvcc process (in parallel),
the host allocator by g++, and everything is linked with nvcc into
``paged_kv_cache_21_gb300/libpagedkv.so`` (CUDA runtime linked statically).
Objects go to ``paged_kv_cache_21_gb300/_build/``.  A target is rebuilt when
any source or header is newer than it.
"""
import concurrent.futures as cf
import glob
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libpagedkv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]
CXX_FLAGS = ["-O2", "-fPIC", "-std=c++17", "-Wall", "-Wextra", "-I", INCLUDE, "-I", CSRC]


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src, extra_flags=(), verbose_ptxas=False):
    os.makedirs(BUILD, exist_ok=True)
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    if not _stale(obj, [src] + _headers() + [__file__]):
        return obj, ""
    if src.endswith(".cu"):
        cmd = [_nvcc()] + NVCC_FLAGS + list(extra_flags) + ["-c", src, "-o", obj]
        if verbose_ptxas:
            cmd += ["-Xptxas", "-v"]
    else:
        cmd = ["g++"] + CXX_FLAGS + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("compile failed: %s\n%s\n%s" % (" ".join(cmd), r.stdout, r.stderr))
    return obj, r.stderr


def build(force=False, verbose_ptxas=False, jobs=None):
    """Compile and link the library; returns its path."""
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    if force and os.path.isdir(BUILD):
        for f in glob.glob(os.path.join(BUILD, "*.o")):
            os.remove(f)
    jobs = jobs or min(len(sources), os.cpu_count() or 4)
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose_ptxas=verbose_ptxas), sources))
    objs = [o for o, _ in results]
    if verbose_ptxas:
        for _, log in results:
            if log:
                print(log)
    if force or _stale(LIB, objs):
        tmp = LIB + ".tmp.%d" % os.getpid()
        cmd = [_nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed: %s\n%s\n%s" % (" ".join(cmd), r.stdout, r.stderr))
        os.replace(tmp, LIB)
    build_fast(force=force)
    return LIB


PYEXT_SRC = os.path.join(PKG, "pyext", "pkvfast.c")


def build_fast(force=False):
    """Compile the CPython-API module ``_pkvfast`` (the per-step calls without
    ctypes marshalling) against ``libpagedkv.so``; returns its path, or None
    where this Python has no headers (the ctypes binding then serves every
    call)."""
    import sysconfig
    inc = sysconfig.get_paths().get("include")
    if not inc or not os.path.exists(os.path.join(inc, "Python.h")):
        return None
    out = os.path.join(PKG, "_pkvfast" + sysconfig.get_config_var("EXT_SUFFIX"))
    if not force and not _stale(out, [PYEXT_SRC, LIB, __file__] + _headers()):
        return out
    tmp = out + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-shared", "-fPIC", "-Wall", "-Wextra", "-I", inc, "-I", INCLUDE,
           PYEXT_SRC, "-o", tmp, "-L", PKG, "-l:libpagedkv.so", "-Wl,-rpath,$ORIGIN"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        # optional: the ctypes binding serves every call without it
        import sys
        print("warning: _pkvfast not built (%s):\n%s" % (" ".join(cmd), r.stderr),
              file=sys.stderr)
        return None
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
