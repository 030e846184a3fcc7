"""Build libetmoe.so (the CUDA path) in-tree for sm_103a with nvcc.

Each translation unit compiles in parallel; the shared object links the CUDA
runtime statically and fetches the driver's tensor-map encoder at run time,
so it loads (and exports its symbols) on machines without a GPU too.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libetmoe.so")
SOURCES = ["etmoe_api.cu", "moe_kernel.cu", "splitk_kernel.cu", "mlp_kernel.cu"]
HEADERS = ["et_device.cuh", "et_gemm.cuh", "et_layout.h"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libetmoe")
    return p


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          out_dir: str = None, defines=()) -> str:
    """Compile (what is stale, or everything with force) into out_dir (default:
    the in-tree _build) and link libetmoe.so there; returns its path.
    `defines` adds -D flags (e.g. "ET_FIXED_T=1": a build specialised for one
    token count, used only to time the per-batch-size build alternative)."""
    out_dir = out_dir or OUT_DIR
    lib = os.path.join(out_dir, "libetmoe.so")
    os.makedirs(out_dir, exist_ok=True)
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "etmoe.h")]
    objs = []
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(out_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + hdrs):
            cmd = [nvcc()] + ARCH + NVCC_FLAGS + (["-Xptxas", "-v"] if ptxas_info else []) + \
                ["-D" + d for d in defines] + ["-c", s, "-o", o]
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    def crashed(r):  # the compiler died of a signal (not a compile error)
        return r.returncode < 0 or "Segmentation fault" in r.stderr or r.returncode >= 128

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            results = list(ex.map(run, jobs))
        for cmd, r in results:
            # the device front end has died of a signal now and then on both
            # hosts, on sources that build on the next attempt: build the unit
            # again, alone, a few times
            for _ in range(3):
                if r.returncode == 0 or not crashed(r):
                    break
                cmd, r = run(cmd)
            if verbose or ptxas_info or r.returncode != 0:
                sys.stdout.write(r.stdout)
                sys.stderr.write(r.stderr)
            if r.returncode != 0:
                raise RuntimeError("nvcc failed: " + " ".join(cmd))
    if force or jobs or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-lpthread"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stderr)
            raise RuntimeError("link failed: " + " ".join(cmd))
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
