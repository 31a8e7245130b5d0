"""Build libfattn.so in-tree with nvcc for sm_103a (no cmake, no torch extension),
and the host-only libfattn_host.so with g++.

Each .cu under csrc/ compiles to an object in parallel; the objects link into
online_softmax_08_gb300/libfattn.so with the static CUDA runtime.  The host
library (csrc/host_attn.cpp, OpenMP) compiles at the same time.
"""
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD_DIR = os.path.join(os.path.dirname(HERE), "_build")
LIB = os.path.join(HERE, "libfattn.so")
HOST_LIB = os.path.join(HERE, "libfattn_host.so")
HOST_SRC = os.path.join(CSRC, "host_attn.cpp")
# -ffp-contract=fast: each "a * b + c" statement becomes one fused multiply-add
HOST_FLAGS = ["-O3", "-std=c++17", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=fast",
              "-Wno-psabi", "-I", INCLUDE]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", INCLUDE]


def nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _stale(obj, deps):
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def _host_cmd(out):
    cxx = os.environ.get("CXX", "g++")
    return [cxx] + HOST_FLAGS + [HOST_SRC, "-o", out]


def build_host(force=False, verbose=False):
    """Compile csrc/host_attn.cpp into libfattn_host.so; returns its path."""
    header = os.path.join(INCLUDE, "fattn_host.h")
    if force or _stale(HOST_LIB, [HOST_SRC, header, __file__]):
        tmp = HOST_LIB + ".tmp.%d" % os.getpid()
        cmd = _host_cmd(tmp)
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        subprocess.run(cmd, check=True)
        os.replace(tmp, HOST_LIB)
    return HOST_LIB


def build(force=False, verbose=False, extra_flags=()):
    """Compile every csrc/*.cu and link libfattn.so, and build libfattn_host.so;
    returns the path of libfattn.so."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    host_proc = None
    host_tmp = HOST_LIB + ".tmp.%d" % os.getpid()
    if force or _stale(HOST_LIB, [HOST_SRC, os.path.join(INCLUDE, "fattn_host.h"), __file__]):
        host_proc = subprocess.Popen(_host_cmd(host_tmp), stdout=subprocess.PIPE,
                                     stderr=subprocess.STDOUT)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(INCLUDE, "fattn.h")]
    procs, objs = [], []
    for src in sources:
        obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + headers + [__file__]):
            cmd = [nvcc()] + ARCH + FLAGS + list(extra_flags) + ["-c", src, "-o", obj]
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                stderr=subprocess.STDOUT)))
    failed = []
    for src, pr in procs:
        out, _ = pr.communicate()
        if pr.returncode != 0 or verbose:
            sys.stderr.write(out.decode(errors="replace"))
        if pr.returncode != 0:
            failed.append(src)
    if host_proc is not None:
        # the host library is independent of the CUDA one: a failure to build it
        # is reported and leaves libfattn.so alone (its own tests then fail)
        out, _ = host_proc.communicate()
        if host_proc.returncode != 0 or verbose:
            sys.stderr.write(out.decode(errors="replace"))
        if host_proc.returncode != 0:
            sys.stderr.write("warning: %s did not build\n" % HOST_LIB)
        else:
            os.replace(host_tmp, HOST_LIB)
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    if force or procs or _stale(LIB, objs):
        tmp = LIB + ".tmp.%d" % os.getpid()
        cmd = [nvcc()] + ARCH + ["-shared", "-Xcompiler", "-fPIC", "-o", tmp] + objs
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
