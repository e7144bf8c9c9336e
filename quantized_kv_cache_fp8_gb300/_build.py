"""Build libkvq.so in-tree with nvcc for sm_103a (GB300)."""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libkvq.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                 "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]
# translation unit -> extra flags.  The codecs are byte-exact: no implicit fusion of a
# multiply and an add (every fma the methods specify is explicit in the source).
UNITS = {
    "kvq_api.cu": [],
    "kvq_codec.cu": ["--fmad=false"],
    "kvq_decode.cu": [],
    "kvq_decode_tc.cu": [],
    "kvq_decode_tc16.cu": [],
    "kvq_decode_tcf8.cu": [],
    "kvq_decode_mma.cu": [],
    "kvq_noalloc.cu": [],
    "kvq_q4_decode.cu": [],
    "kvq_persist.cu": [],
}


def _sources():
    return [os.path.join(CSRC, u) for u in UNITS]


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = _sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")]
    deps.append(os.path.join(INCLUDE, "kvq.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    objs = []
    cmds = []
    for unit, extra in UNITS.items():
        obj = os.path.join(OUT_DIR, unit.replace(".cu", ".o"))
        objs.append(obj)
        cmds.append([NVCC, *COMMON, *extra, "-c", os.path.join(CSRC, unit), "-o", obj])
    with cf.ThreadPoolExecutor(max_workers=len(cmds)) as ex:
        futs = [ex.submit(subprocess.run, c, capture_output=True, text=True) for c in cmds]
        for c, f in zip(cmds, futs):
            r = f.result()
            if verbose or r.returncode != 0:
                print(" ".join(c))
                print(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {c[-3]}")
    tmp = LIB + f".tmp{os.getpid()}"
    link = [NVCC, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        print(" ".join(link))
        print(r.stdout + r.stderr)
        raise RuntimeError("link of libkvq.so failed")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
