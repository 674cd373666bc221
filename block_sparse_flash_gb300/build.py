"""Builds libsplash.so in-tree (block_sparse_flash_gb300/_build/) with nvcc for
sm_103a.  Translation units are compiled in parallel and linked into one
shared library; nothing is installed outside the repository."""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libsplash.so")
# (source, object, defines): attention_fwd.cu is compiled once per pattern
# mode, so that its kernel instantiations build in parallel
SOURCES = [("api.cu", "api", []), ("mask_info.cu", "mask_info", []),
           ("attention_fwd.cu", "attention_fwd", ["-DSPLASH_FWD_PM=0"]),
           ("attention_fwd.cu", "attention_fwd_band", ["-DSPLASH_FWD_PM=1"]),
           ("attention_fwd.cu", "attention_fwd_band_seg", ["-DSPLASH_FWD_PM=2"]),
           ("attention_bwd.cu", "attention_bwd", []), ("host_pipeline.cu", "host_pipeline", [])]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _newest_input():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "splash.h"),
                                                               os.path.abspath(__file__)]
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    """Compiles (if stale) and returns the path of libsplash.so."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _newest_input():
        return LIB
    nvcc = _nvcc()

    def compile_one(entry):
        src, name, defines = entry
        obj = os.path.join(OUT_DIR, name + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *defines, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    v = "-v" in sys.argv
    print(build(force="--force" in sys.argv, verbose=v, extra=["-Xptxas", "-v"] if v else []))
