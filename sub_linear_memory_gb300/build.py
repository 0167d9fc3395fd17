"""Build ``libslim_attn.so`` in-tree with nvcc for sm_103a (no torch extension
machinery: the library is a plain C ABI).  Translation units compile in
parallel; the link step uses the static CUDA runtime."""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIB = os.path.join(HERE, "libslim_attn.so")
OBJDIR = os.path.join(HERE, "_build")
# -DSLIM_DEBUG: device-side bounds checks that record SLIM_ERR_BOUNDS, and every
# call waits for its work and reports device-side errors itself
DEBUG_LIB = os.path.join(HERE, "libslim_attn_debug.so")
DEBUG_OBJDIR = os.path.join(HERE, "_build_debug")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE]


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    files = sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "slim_attn.h"))
    return files


def up_to_date(lib=LIB):
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps() + [__file__])


def build(force=False, verbose=False, extra_flags=(), debug=False):
    """Compile and link the library (the release build, or with debug=True the
    -DSLIM_DEBUG variant libslim_attn_debug.so); skips an up-to-date target."""
    lib, objdir = (DEBUG_LIB, DEBUG_OBJDIR) if debug else (LIB, OBJDIR)
    if debug:
        extra_flags = tuple(extra_flags) + ("-DSLIM_DEBUG",)
    if not force and up_to_date(lib):
        return lib
    nvcc = os.environ.get("NVCC", "nvcc")
    os.makedirs(objdir, exist_ok=True)
    procs, objs = [], []
    for src in sources():
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmd = [nvcc, *ARCH, *FLAGS, *extra_flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, pr in procs:
        out, _ = pr.communicate()
        if pr.returncode != 0:
            failed.append((src, out.decode(errors="replace")))
        elif verbose and out:
            print(out.decode(errors="replace"), file=sys.stderr)
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join("%s:\n%s" % f for f in failed))
    tmp = lib + ".tmp%d" % os.getpid()
    subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"], check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
