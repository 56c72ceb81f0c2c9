"""Build libpattn.so in-tree for sm_103a with nvcc.

Each .cu file is compiled to an object in parallel, then linked into
``paged_varlen_attention_attn_gb300/_build/libpattn.so``.  One -gencode only
(compute_103a -> sm_103a); -lineinfo keeps ncu's source attribution.

``build_wait_test()`` compiles the same sources with PATTN_WAIT_TEST into
``_build/wait_test/libpattn_wait_test.so``: a library that only the tests
load, whose bounded waits give up after 10 ms instead of 2 s and which exports
``pattn_test_set_wait_skip`` so a test can make one wait run out.
"""
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libpattn.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(
        os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h"))


WAIT_TEST_DIR = os.path.join(OUT_DIR, "wait_test")
WAIT_TEST_LIB = os.path.join(WAIT_TEST_DIR, "libpattn_wait_test.so")


def up_to_date(lib=LIB):
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force=False, verbose=False, extra_flags=(), lib=LIB):
    """Compile (if stale) and return the path of libpattn.so."""
    if not force and up_to_date(lib):
        return lib
    out_dir = os.path.dirname(lib)
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    flags = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                    "-I", INCLUDE, "-I", CSRC] + list(extra_flags)
    if verbose:
        flags += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.basename(src) + ".o")
        r = subprocess.run([nvcc, "-c", src, "-o", obj] + flags,
                           capture_output=True, text=True)
        return src, obj, r

    objs = []
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        for src, obj, r in ex.map(compile_one, _sources()):
            if r.returncode != 0 or verbose:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {os.path.basename(src)}")
            objs.append(obj)
    tmp = lib + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart"],
                       capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError(f"link of {os.path.basename(lib)} failed")
    os.replace(tmp, lib)
    return lib


def build_wait_test(force=False):
    """The wait-test library (tests only): short wait limit, skip hook."""
    return build(force=force, extra_flags=("-DPATTN_WAIT_TEST",), lib=WAIT_TEST_LIB)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
