"""Build libmxq.so (the sm_103a quantization library) in-tree.

Each .cu file under csrc/ is compiled to an object in parallel, then linked
into fp4_quantization_gb300/libmxq.so.  One -gencode (sm_103a), no cmake, so
a build takes seconds on either host (x86-64 here, aarch64 next to the GPU).
"""
import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmxq.so")

# (source, extra nvcc flags, object): mx_kernels.cu is built twice, for the
# row-major and the tiled scale layouts.
UNITS = [
    ("mxq_api.cu", [], "mxq_api.o"),
    ("mx_kernels.cu", [], "mx_kernels.o"),
    ("mx_kernels.cu", ["-DMXQ_TILED_SCALES=1"], "mx_kernels_tiled.o"),
    ("nvfp4_kernels.cu", [], "nvfp4_kernels.o"),
    ("mxq_noalloc.cu", [], "mxq_noalloc.o"),
    ("mxq_host.cu", [], "mxq_host.o"),
]
SOURCES = sorted({src for src, _, _ in UNITS})

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "--expt-relaxed-constexpr",
    "-I", INCLUDE, "-I", CSRC,
]


def _nvcc():
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmxq.so")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "mxq.h"))
    files.append(os.path.abspath(__file__))
    return files


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile and link libmxq.so unless it is newer than every source."""
    if not force and os.path.exists(LIB):
        newest = max(os.path.getmtime(f) for f in _deps())
        if os.path.getmtime(LIB) >= newest:
            return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    # Optional -D overrides of the launch configuration (tuning builds).
    extra += os.environ.get("MXQ_NVCC_DEFINES", "").split()

    def compile_one(unit):
        src, flags, obj_name = unit
        obj = os.path.join(BUILD_DIR, obj_name)
        cmd = [nvcc, *NVCC_FLAGS, *flags, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(UNITS)) as pool:
        results = list(pool.map(compile_one, UNITS))
    if verbose or ptxas_verbose:
        for _, log in results:
            if log.strip():
                print(log, file=sys.stderr)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-o", tmp,
           *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv))
