"""Build libkvd.so (the decode library) and libkvd_inputs.so (the device-side
input generator) in-tree, with nvcc for sm_103a only.

Translation units compile in parallel; a stamp of the sources, headers and
flags skips the build when nothing changed. Set KVD_PTXAS_VERBOSE=1 to see
register and shared-memory use per kernel.
"""
import concurrent.futures
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")

LIB_SOURCES = ["api.cu", "append.cu", "decode_simt.cu", "noalloc.cu",
               "decode_mma.cu", "decode_wide.cu", "decode_latent_tc.cu",
               "decode_gather_tc.cu",
               "indexer.cu", "block_pool.cu"]
INPUTS_SOURCES = ["inputs_fill.cu"]
LIB = os.path.join(PKG, "libkvd.so")
INPUTS_LIB = os.path.join(PKG, "libkvd_inputs.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc",
                 shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put it on PATH)")


def flags():
    f = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                "-I", INCLUDE, "-I", CSRC]
    if os.environ.get("KVD_PTXAS_VERBOSE"):
        f += ["-Xptxas", "-v"]
    return f


def _stamp(sources):
    h = hashlib.sha256()
    h.update(" ".join(flags()).encode())
    files = sorted(set(sources) | {n for n in os.listdir(CSRC)
                                   if n.endswith((".h", ".cuh"))})
    for name in files:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    with open(os.path.join(INCLUDE, "kvd.h"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()


def _compile(src):
    obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), "-c", os.path.join(CSRC, src), "-o", obj] + flags()
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def _link(objs, out):
    tmp = out + ".tmp"
    cmd = [nvcc(), "-shared", "-o", tmp] + objs + ARCH
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed for {out}:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)


def build(force=False, verbose=False):
    """Compile and link both libraries; returns their paths."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    stamp_file = os.path.join(BUILD_DIR, "stamp")
    stamp = _stamp(LIB_SOURCES + INPUTS_SOURCES)
    if (not force and os.path.exists(LIB) and os.path.exists(INPUTS_LIB)
            and os.path.exists(stamp_file)
            and open(stamp_file).read() == stamp):
        return LIB, INPUTS_LIB
    sources = LIB_SOURCES + INPUTS_SOURCES
    with concurrent.futures.ThreadPoolExecutor(len(sources)) as ex:
        results = dict(zip(sources, ex.map(_compile, sources)))
    if verbose or os.environ.get("KVD_PTXAS_VERBOSE"):
        for src in sources:
            if results[src][1].strip():
                sys.stderr.write(f"--- {src}\n{results[src][1]}")
    _link([results[s][0] for s in LIB_SOURCES], LIB)
    _link([results[s][0] for s in INPUTS_SOURCES], INPUTS_LIB)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return LIB, INPUTS_LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
    print(LIB)
    print(INPUTS_LIB)
