"""Builds lib/libds4moe.so in-tree: CUDA sources with nvcc for sm_103a, the host quantisers
with g++ (no fused multiply-add, so the packed bytes are reproducible), all in parallel."""
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB_DIR = os.path.join(HERE, "lib")
OBJ_DIR = os.path.join(LIB_DIR, "obj")
LIB_PATH = os.path.join(LIB_DIR, "libds4moe.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _sources():
    cu = sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))
    cpp = sorted(f for f in os.listdir(CSRC) if f.endswith(".cpp"))
    return cu, cpp


def _stale(out, deps):
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose=False, force=False):
    """Compile every translation unit (in parallel) and link the shared library."""
    nvcc = _nvcc()
    os.makedirs(OBJ_DIR, exist_ok=True)
    cu, cpp = _sources()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers.append(os.path.join(os.path.dirname(HERE), "include", "ds4moe.h"))
    jobs, objs = [], []
    for f in cu:
        src = os.path.join(CSRC, f)
        obj = os.path.join(OBJ_DIR, f + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + headers):
            cmd = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                   "-Xptxas", "-warn-spills", "-c", src, "-o", obj]
            jobs.append((cmd, f))
    for f in cpp:
        src = os.path.join(CSRC, f)
        obj = os.path.join(OBJ_DIR, f + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + headers):
            cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-ffp-contract=off", "-fno-fast-math", "-pthread",
                   "-c", src, "-o", obj]
            jobs.append((cmd, f))
    procs = [(subprocess.Popen(c, stdout=subprocess.PIPE, stderr=subprocess.STDOUT), f) for c, f in jobs]
    failed = []
    for p, f in procs:
        out, _ = p.communicate()
        if verbose or p.returncode:
            print(out.decode(errors="replace"))
        if p.returncode:
            failed.append(f)
    if failed:
        raise RuntimeError("compilation failed: %s" % ", ".join(failed))
    if force or jobs or _stale(LIB_PATH, objs):
        tmp = LIB_PATH + ".%d.tmp" % os.getpid()
        subprocess.check_call([nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lpthread"])
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    build(verbose=True)
